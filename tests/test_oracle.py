"""Pins of the CPU oracle against things other than itself.

Each check is chosen so that a plausible mistake in the oracle (a dropped
decay, a pre-update read, a wrong head map, a transposed state, a sign error in
the delta, a wrong chunk restart) fails at least one of them:

  * a hand-worked example (tests/golden/hand_worked_2tok.txt);
  * brute force with explicit K x K transition matrices, in two forms;
  * closed forms: beta = 0 (pure decay), g = 0 / beta = 1 / orthonormal keys
    (exact overwrite), KDA with a channel-constant gate == scalar gate,
    GVA == MHA with repeated key heads, varlen == separate calls;
  * the chunked WY form == the tokenwise form (chunk 1, 7, 16, 64; g = -2);
  * a contraction bound;
  * negative controls that must fail.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_37_gb300 import workloads
from tests.conftest import read_golden


def rel_l2(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.linalg.norm((x - y).ravel()) / max(np.linalg.norm(y.ravel()), 1e-300))


def _golden_inputs(gd, channel):
    q = np.array(gd["q"]).reshape(2, 1, 2)
    k = np.array(gd["k"]).reshape(2, 1, 2)
    v = np.array(gd["v"]).reshape(2, 1, 2)
    beta = np.array(gd["beta"]).reshape(2, 1)
    s0 = np.array(gd["s0"]).reshape(1, 1, 2, 2)
    if channel:
        gk = np.log(np.array(gd["decay_channel"])).reshape(2, 1, 2)
        return dict(q=q, k=k, v=v, beta=beta, initial_state=s0, gk=gk)
    g = np.log(np.array(gd["decay_scalar"])).reshape(2, 1)
    return dict(q=q, k=k, v=v, beta=beta, initial_state=s0, g=g)


@pytest.mark.parametrize("channel", [False, True])
def test_hand_worked_example(channel):
    gd = read_golden("hand_worked_2tok.txt")
    inp = _golden_inputs(gd, channel)
    tag = "channel" if channel else "scalar"
    cu = [0, 2]
    o, sf = oracle.tokenwise(cu_seqlens=cu, scale=1.0, **inp)
    np.testing.assert_allclose(o.ravel(), gd[f"o_{tag}"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sf.ravel(), gd[f"s_final_{tag}"], rtol=0, atol=1e-12)
    oc, sfc = oracle.chunked(cu_seqlens=cu, scale=1.0, chunk=64, **inp)
    np.testing.assert_allclose(oc.ravel(), gd[f"o_{tag}"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sfc.ravel(), gd[f"s_final_{tag}"], rtol=0, atol=1e-12)
    ob, sb, closed = oracle.bruteforce(inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0],
                                       inp["beta"][:, 0],
                                       g=None if channel else inp["g"][:, 0],
                                       gk=inp["gk"][:, 0] if channel else None,
                                       initial_state=inp["initial_state"][0, 0], scale=1.0)
    np.testing.assert_allclose(ob.ravel(), gd[f"o_{tag}"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(closed.ravel(), gd[f"s_final_{tag}"], rtol=0, atol=1e-12)


def test_hand_worked_negative_control_pre_update():
    gd = read_golden("hand_worked_2tok.txt")
    inp = _golden_inputs(gd, False)
    o, _ = oracle.tokenwise(cu_seqlens=[0, 2], scale=1.0, variant=oracle.READ_PRE_UPDATE, **inp)
    np.testing.assert_allclose(o[1, 0], gd["o2_pre_update_scalar"], atol=1e-12)
    assert np.abs(o[1, 0] - np.array(gd["o_scalar"][2:])).max() > 0.1


def _rand_case(rng, T, Hk, Hv, K, V, gate="g", g_lo=-0.5, h0=True, beta_hi=1.0):
    q = rng.standard_normal((T, Hk, K))
    k = rng.standard_normal((T, Hk, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, V))
    beta = rng.uniform(0, beta_hi, (T, Hv))
    d = dict(q=q, k=k, v=v, beta=beta)
    if gate == "g":
        d["g"] = rng.uniform(g_lo, 0, (T, Hv))
    else:
        d["gk"] = rng.uniform(g_lo, 0, (T, Hv, K))
    d["initial_state"] = rng.standard_normal((1, Hv, V, K)) if h0 else None
    return d


@pytest.mark.parametrize("gate", ["g", "gk"])
@pytest.mark.parametrize("T,K,V", [(1, 2, 3), (3, 4, 4), (4, 3, 2)])
def test_bruteforce_agrees(gate, T, K, V):
    rng = np.random.default_rng(100 + T * 10 + K)
    d = _rand_case(rng, T, 1, 1, K, V, gate=gate)
    o, sf = oracle.tokenwise(cu_seqlens=[0, T], scale=0.7, **d)
    ob, sb, closed = oracle.bruteforce(d["q"][:, 0], d["k"][:, 0], d["v"][:, 0], d["beta"][:, 0],
                                       g=d["g"][:, 0] if gate == "g" else None,
                                       gk=d["gk"][:, 0] if gate == "gk" else None,
                                       initial_state=d["initial_state"][0, 0], scale=0.7)
    np.testing.assert_allclose(o[:, 0], ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sf[0, 0], sb, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sf[0, 0], closed, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("gate", ["g", "gk"])
def test_beta_zero_is_pure_decay(gate):
    rng = np.random.default_rng(7)
    T, K, V = 9, 5, 6
    d = _rand_case(rng, T, 1, 1, K, V, gate=gate, g_lo=-1.0)
    d["beta"][:] = 0.0
    o, sf = oracle.tokenwise(cu_seqlens=[0, T], scale=0.5, **d)
    S0 = d["initial_state"][0, 0]
    gam = np.cumsum(d["g"][:, 0], 0)[:, None] * np.ones(K) if gate == "g" else np.cumsum(d["gk"][:, 0], 0)
    for t in range(T):
        St = S0 * np.exp(gam[t])[None, :]
        np.testing.assert_allclose(o[t, 0], 0.5 * St @ d["q"][t, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(sf[0, 0], S0 * np.exp(gam[-1])[None, :], rtol=1e-12)


def test_orthonormal_overwrite():
    """g = 0, beta = 1, orthonormal keys, S_0 = 0: S_n = sum_j v_j k_j^T exactly
    and S_t k_j = v_j for every j <= t."""
    rng = np.random.default_rng(8)
    K, V, n = 8, 5, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:, :n].T.copy()                       # n orthonormal rows
    q = rng.standard_normal((n, 1, K))
    v = rng.standard_normal((n, 1, V))
    d = dict(q=q, k=keys[:, None, :], v=v, beta=np.ones((n, 1)), g=np.zeros((n, 1)))
    o, sf = oracle.tokenwise(cu_seqlens=[0, n], scale=1.3, **d)
    S = np.einsum("jv,jk->vk", v[:, 0], keys)
    np.testing.assert_allclose(sf[0, 0], S, rtol=1e-12, atol=1e-13)
    for t in range(n):
        expect = 1.3 * sum((keys[j] @ q[t, 0]) * v[j, 0] for j in range(t + 1))
        np.testing.assert_allclose(o[t, 0], expect, rtol=1e-12, atol=1e-13)
    # the full-state recall property after the last token
    for j in range(n):
        np.testing.assert_allclose(sf[0, 0] @ keys[j], v[j, 0], atol=1e-12)


def test_kda_with_constant_channels_equals_scalar_gate():
    rng = np.random.default_rng(9)
    T, K, V, H = 20, 6, 4, 2
    d = _rand_case(rng, T, H, H, K, V, gate="g", g_lo=-1.0)
    o1, s1 = oracle.tokenwise(cu_seqlens=[0, T], scale=0.4, **d)
    gk = np.repeat(d.pop("g")[:, :, None], K, axis=2)
    o2, s2 = oracle.tokenwise(cu_seqlens=[0, T], scale=0.4, gk=gk, **d)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(s1, s2, rtol=1e-13, atol=1e-14)


def test_gva_equals_mha_with_repeated_heads():
    rng = np.random.default_rng(10)
    T, K, V, Hk, Hv = 11, 4, 4, 2, 6
    d = _rand_case(rng, T, Hk, Hv, K, V)
    o1, s1 = oracle.tokenwise(cu_seqlens=[0, T], scale=0.3, **d)
    rep = Hv // Hk
    d2 = dict(d, q=np.repeat(d["q"], rep, axis=1), k=np.repeat(d["k"], rep, axis=1))
    o2, s2 = oracle.tokenwise(cu_seqlens=[0, T], scale=0.3, **d2)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(s1, s2, rtol=1e-13, atol=1e-14)
    # the wrong map (h % Hk) differs from h // (Hv/Hk)
    o3, _ = oracle.tokenwise(cu_seqlens=[0, T], scale=0.3, variant=oracle.HEAD_MOD, **d)
    assert rel_l2(o3, o1) > 1e-2


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(11)
    lens = [3, 1, 7, 5]
    T = sum(lens)
    K, V, H = 4, 3, 2
    d = _rand_case(rng, T, H, H, K, V, h0=False)
    h0 = rng.standard_normal((len(lens), H, V, K))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, sf = oracle.tokenwise(cu_seqlens=cu, scale=0.6, initial_state=h0,
                             **{k_: v_ for k_, v_ in d.items() if k_ != "initial_state"})
    for b in range(len(lens)):
        sl = slice(cu[b], cu[b + 1])
        ob, sb = oracle.tokenwise(q=d["q"][sl], k=d["k"][sl], v=d["v"][sl], g=d["g"][sl],
                                  beta=d["beta"][sl], initial_state=h0[b:b + 1],
                                  cu_seqlens=[0, lens[b]], scale=0.6)
        np.testing.assert_allclose(o[sl], ob, rtol=1e-14, atol=0)
        np.testing.assert_allclose(sf[b], sb[0], rtol=1e-14, atol=0)


@pytest.mark.parametrize("gate", ["g", "gk"])
def test_segment_state_map_is_affine(gate):
    """The reading the chunk-parallel scan rests on: over any run of tokens the
    state map is affine in the start state, S_end = S_start P + B ([V][K]
    layout), with P the run from the identity with v = 0 and B the run from
    zero; composing two segments that way gives the one-pass final state."""
    rng = np.random.default_rng(21)
    K = V = 6
    T1, T2 = 9, 13
    d = _rand_case(rng, T1 + T2, 1, 2, K, V, gate=gate, g_lo=-0.7, h0=False)
    h0 = rng.standard_normal((1, 2, V, K))
    full = {k_: v_ for k_, v_ in d.items() if k_ != "initial_state"}
    _, s_full = oracle.tokenwise(cu_seqlens=[0, T1 + T2], scale=0.5, initial_state=h0, **full)

    def run(sl, start, zero_v=False):
        seg = {k_: v_[sl] for k_, v_ in full.items()}
        if zero_v:
            seg["v"] = np.zeros_like(seg["v"])
        n = sl.stop - sl.start
        return oracle.tokenwise(cu_seqlens=[0, n], scale=0.5, initial_state=start, **seg)[1]

    eye = np.broadcast_to(np.eye(K), (1, 2, K, K)).copy()
    s_mid = h0
    for sl in (slice(0, T1), slice(T1, T1 + T2)):
        P = run(sl, eye, zero_v=True)
        B = run(sl, None)
        direct = run(sl, s_mid)
        composed = np.einsum("nhvm,nhmk->nhvk", s_mid, P) + B
        np.testing.assert_allclose(composed, direct, rtol=1e-12, atol=1e-12)
        s_mid = composed
    np.testing.assert_allclose(s_mid, s_full, rtol=1e-12, atol=1e-12)
    # P depends on the keys, gates and betas but not on v
    P1 = run(slice(0, T1), eye, zero_v=True)
    d2 = dict(full, v=rng.standard_normal(full["v"].shape))
    seg = {k_: v_[:T1] for k_, v_ in d2.items()}
    seg["v"] = np.zeros_like(seg["v"])
    P2 = oracle.tokenwise(cu_seqlens=[0, T1], scale=0.5, initial_state=eye, **seg)[1]
    np.testing.assert_array_equal(P1, P2)
    # a wrong composition order (P S instead of S P) is caught
    wrong = np.einsum("nhvm,nhmk->nhvk", P1, h0)
    assert rel_l2(wrong + run(slice(0, T1), None), run(slice(0, T1), h0)) > 1e-3


@pytest.mark.parametrize("gate,g_lo", [("g", -0.05), ("g", -2.0), ("gk", -0.1), ("gk", -2.0)])
@pytest.mark.parametrize("chunk", [1, 7, 16, 64])
def test_chunked_equals_tokenwise(gate, g_lo, chunk):
    rng = np.random.default_rng(12)
    lens = [65, 1, 63, 130]
    T = sum(lens)
    K, V, Hk, Hv = 8, 6, 1, 2
    d = _rand_case(rng, T, Hk, Hv, K, V, gate=gate, g_lo=g_lo, h0=False)
    d["initial_state"] = rng.standard_normal((len(lens), Hv, V, K))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o1, s1 = oracle.tokenwise(cu_seqlens=cu, scale=0.35, **d)
    o2, s2 = oracle.chunked(cu_seqlens=cu, scale=0.35, chunk=chunk, **d)
    assert np.isfinite(o2).all() and np.isfinite(s2).all()
    assert rel_l2(o2, o1) <= 1e-12
    assert rel_l2(s2, s1) <= 1e-12


def test_chunked_gate_minus_two_stays_finite_at_full_chunk():
    """g = -2 per token gives a prefix of -128 over a 64-token chunk; an
    exp(-prefix) formulation would overflow past token ~45 (cuLA PR #113 review)."""
    rng = np.random.default_rng(13)
    T, K, V = 128, 8, 8
    d = _rand_case(rng, T, 1, 1, K, V, gate="g")
    d["g"][:] = -2.0
    o1, s1 = oracle.tokenwise(cu_seqlens=[0, T], scale=1.0, **d)
    o2, s2 = oracle.chunked(cu_seqlens=[0, T], scale=1.0, chunk=64, **d)
    assert np.isfinite(o2).all()
    assert rel_l2(o2, o1) <= 1e-12 and rel_l2(s2, s1) <= 1e-12


def test_contraction_bound():
    """beta in [0,1], |k| = 1: (I - beta k k^T) has spectral norm <= 1, so
    |S_t|_F <= exp(g_t) |S_{t-1}|_F + beta_t |v_t|."""
    rng = np.random.default_rng(14)
    T, K, V = 40, 6, 5
    d = _rand_case(rng, T, 1, 1, K, V, g_lo=-0.3)
    prev = np.linalg.norm(d["initial_state"])
    for t in range(1, T + 1):
        _, s = oracle.tokenwise(q=d["q"][:t], k=d["k"][:t], v=d["v"][:t], g=d["g"][:t],
                                beta=d["beta"][:t], initial_state=d["initial_state"],
                                cu_seqlens=[0, t], scale=1.0)
        cur = np.linalg.norm(s)
        bound = math.exp(d["g"][t - 1, 0]) * prev + d["beta"][t - 1, 0] * np.linalg.norm(d["v"][t - 1, 0])
        assert cur <= bound * (1 + 1e-12)
        prev = cur


def test_negative_controls_fail_parity():
    """The planted mistakes must break the parity bounds the GPU is held to."""
    rng = np.random.default_rng(15)
    T, K, V, Hk, Hv = 32, 8, 8, 2, 4
    d = _rand_case(rng, T, Hk, Hv, K, V, g_lo=-0.2)
    o, s = oracle.tokenwise(cu_seqlens=[0, T], scale=0.4, **d)
    for variant in (oracle.READ_PRE_UPDATE, oracle.HEAD_MOD, oracle.TRANSPOSED):
        ob, sb = oracle.tokenwise(cu_seqlens=[0, T], scale=0.4, variant=variant, **d)
        assert rel_l2(ob, o) > 5e-3 or rel_l2(sb, s) > 1e-4, variant
    ob, _ = oracle.tokenwise(cu_seqlens=[0, T], scale=0.4, variant=oracle.READ_PRE_UPDATE, **d)
    assert rel_l2(ob, o) > 5e-3


def test_pool_decode_and_verify_match_tokenwise():
    """Decode at T=1 and verify's per-token states are the tokenwise recurrence
    started from the gathered pool slot; padding rows are never touched."""
    case = workloads.pool_case(21, [3, 1, 4, 2], 2, 4, 8, 6, num_slots=6,
                               pool_dtype=torch.float32, pad_count=1, commit=True,
                               steps=5, ibuf_rows=5)
    o, pout, ib = oracle.pool(case.q, case.k, case.v, case.g, case.beta, case.pool,
                              case.state_indices, case.cu_seqlens, scale=case.scale,
                              commit=True, steps=5, ibuf_rows=5)
    pin = case.pool.double().numpy()
    cu = case.cu_seqlens.numpy()
    for b in range(case.N):
        slot = int(case.state_indices[b])
        sl = slice(cu[b], cu[b + 1])
        if slot < 0:
            assert np.isnan(o[sl]).all() and np.isnan(ib[b]).all()
            continue
        L = cu[b + 1] - cu[b]
        for t in range(1, L + 1):
            ot, st = oracle.tokenwise(q=case.q[cu[b]:cu[b] + t], k=case.k[cu[b]:cu[b] + t],
                                      v=case.v[cu[b]:cu[b] + t], g=case.g[cu[b]:cu[b] + t],
                                      beta=case.beta[cu[b]:cu[b] + t],
                                      initial_state=pin[slot:slot + 1], cu_seqlens=[0, t],
                                      scale=case.scale)
            np.testing.assert_allclose(ib[b, t - 1], st[0], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(o[sl], ot, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(pout[slot], st[0], rtol=1e-13, atol=1e-15)
        assert np.isnan(ib[b, L:]).all()
    untouched = set(range(case.pool.shape[0])) - {int(s) for s in case.state_indices if s >= 0}
    for s in untouched:
        assert np.array_equal(pout[s], pin[s])


def test_pool_channel_gate_matches_tokenwise():
    """Per-key-channel gates in decode / verify: each per-token state and the
    committed state are the tokenwise recurrence (with gk) from the gathered
    slot; the padding row stays untouched."""
    case = workloads.pool_case(23, [2, 3, 1], 1, 2, 6, 5, num_slots=5, pool_dtype=torch.float32,
                               pad_count=1, commit=True, steps=3, ibuf_rows=3, channel_gate=True,
                               g_range=(-1.5, 0.0))
    assert case.g.shape == (case.T, 2, 6)
    o, pout, ib = oracle.pool(case.q, case.k, case.v, case.g, case.beta, case.pool, case.state_indices,
                              case.cu_seqlens, scale=case.scale, commit=True, steps=3, ibuf_rows=3)
    pin = case.pool.double().numpy()
    cu = case.cu_seqlens.numpy()
    for b in range(case.N):
        slot = int(case.state_indices[b])
        sl = slice(cu[b], cu[b + 1])
        if slot < 0:
            assert np.isnan(o[sl]).all() and np.isnan(ib[b]).all()
            continue
        L = cu[b + 1] - cu[b]
        for t in range(1, L + 1):
            ot, st = oracle.tokenwise(q=case.q[cu[b]:cu[b] + t], k=case.k[cu[b]:cu[b] + t],
                                      v=case.v[cu[b]:cu[b] + t], gk=case.g[cu[b]:cu[b] + t],
                                      beta=case.beta[cu[b]:cu[b] + t], initial_state=pin[slot:slot + 1],
                                      cu_seqlens=[0, t], scale=case.scale)
            np.testing.assert_allclose(ib[b, t - 1], st[0], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(o[sl], ot, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(pout[slot], st[0], rtol=1e-13, atol=1e-15)


def test_pool_channel_constant_gate_equals_scalar_gate():
    """A per-channel gate that is the same on every key channel is the scalar gate."""
    case = workloads.pool_case(24, [3, 2], 2, 4, 8, 4, num_slots=4, pool_dtype=torch.float32,
                               commit=True, steps=3, ibuf_rows=2)
    gk = case.g[:, :, None].expand(-1, -1, 8).contiguous()
    kw = dict(scale=case.scale, commit=True, steps=3, ibuf_rows=2)
    o1, p1, i1 = oracle.pool(case.q, case.k, case.v, case.g, case.beta, case.pool, case.state_indices,
                             case.cu_seqlens, **kw)
    o2, p2, i2 = oracle.pool(case.q, case.k, case.v, gk, case.beta, case.pool, case.state_indices,
                             case.cu_seqlens, **kw)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(p1, p2)
    np.testing.assert_array_equal(i1, i2)


def test_pool_no_commit_leaves_pool():
    case = workloads.pool_case(22, [2, 2], 1, 2, 4, 4, num_slots=3, pool_dtype=torch.float32,
                               commit=False, steps=2, ibuf_rows=2)
    _, pout, _ = oracle.pool(case.q, case.k, case.v, case.g, case.beta, case.pool,
                             case.state_indices, case.cu_seqlens, scale=case.scale,
                             commit=False, steps=2, ibuf_rows=2)
    assert np.array_equal(pout, case.pool.double().numpy())


def test_gated_rmsnorm_hand_example_and_invariants():
    """Decode output epilogue rmsnorm(o) * w * sigmoid(gate): a hand-worked row,
    unit RMS with w = 1 and an open gate, scale invariance at eps = 0, and the
    gate at 0 halving the output."""
    # row (3, 4): mean square 12.5; eps 0.5 -> divisor sqrt(13) ; w (2, 1); gate 0 -> 1/2
    y = oracle.gated_rmsnorm(np.array([[[3.0, 4.0]]]), np.array([2.0, 1.0]), np.zeros((1, 1, 2)), 0.5)
    np.testing.assert_allclose(y[0, 0], [3.0 / math.sqrt(13.0), 2.0 / math.sqrt(13.0)], rtol=1e-15)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 2, 16))
    open_gate = np.full_like(x, 50.0)
    y1 = oracle.gated_rmsnorm(x, np.ones(16), open_gate, 0.0)
    np.testing.assert_allclose(np.mean(y1 * y1, axis=-1), 1.0, rtol=1e-12)
    y2 = oracle.gated_rmsnorm(7.5 * x, np.ones(16), open_gate, 0.0)
    np.testing.assert_allclose(y2, y1, rtol=1e-12)
    y3 = oracle.gated_rmsnorm(x, np.ones(16), np.zeros_like(x), 0.0)
    np.testing.assert_allclose(y3, 0.5 * y1, rtol=1e-12)


def test_gating_closed_forms():
    # a + dt_bias = 0 -> softplus = ln 2; b = 0 -> sigmoid = 1/2
    a = np.array([[0.0, 25.0, -3.0]])
    dt = np.array([0.0, 0.0, 1.0])
    A_log = np.array([0.0, math.log(2.0), 0.0])
    b = np.array([[0.0, 100.0, -2.0]])
    g, beta = oracle.gating(a, dt, A_log, b)
    assert g[0, 0] == pytest.approx(-math.log(2.0), rel=1e-15)
    assert g[0, 1] == pytest.approx(-2.0 * 25.0, rel=1e-15)       # threshold branch: x > 20 -> x
    assert g[0, 2] == pytest.approx(-math.log1p(math.exp(-2.0)), rel=1e-15)
    assert beta[0, 0] == 0.5 and beta[0, 1] == pytest.approx(1.0)
    assert beta[0, 2] == pytest.approx(1.0 / (1.0 + math.exp(2.0)), rel=1e-15)
    g2, beta2 = oracle.gating(a, dt, A_log, b, neg_eigval=True)
    np.testing.assert_array_equal(g2, g)
    np.testing.assert_allclose(beta2, 2 * beta, rtol=0)


def test_l2norm():
    rng = np.random.default_rng(16)
    x = rng.standard_normal((5, 3, 16))
    y = oracle.l2norm(x, eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=-1, keepdims=True), x, rtol=1e-14)
    z = oracle.l2norm(np.full((1, 4), 0.5), eps=1e-6)      # sum x^2 = 1
    np.testing.assert_allclose(z, 0.5 / math.sqrt(1.0 + 1e-6), rtol=1e-15)
