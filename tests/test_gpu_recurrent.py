"""GPU parity of the recurrent decode / verify kernel against the CPU oracle,
through the C ABI.  Slot indexing, padding skips, ragged boundaries and every
region the call must not write are checked bit for bit."""
import numpy as np
import pytest
import torch

import gated_delta_rule_37_gb300 as gdr
import oracle
from gated_delta_rule_37_gb300 import workloads
from tests.gpu_util import Guarded, bits_equal, check_out, check_state, sentinel_like

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load()


def run_case(case, *, flags, with_ibuf, gated=False):
    dev = DEV
    pool = Guarded(case.pool.shape, case.pool.dtype, dev, fill_bytes=case.pool)
    o_init = sentinel_like((case.T, case.v.shape[1], case.v.shape[2]), case.q.dtype)
    o = Guarded(o_init.shape, case.q.dtype, dev, fill_bytes=o_init)
    ib = None
    if with_ibuf:
        ib_shape = (case.ibuf_rows, case.steps) + tuple(case.pool.shape[1:])
        ib_init = sentinel_like(ib_shape, case.pool.dtype)
        ib = Guarded(ib_shape, case.pool.dtype, dev, fill_bytes=ib_init)
    if case.norm is not None:
        nw, nz = case.norm["weight"].to(dev), case.norm["gate"].to(dev)
        gdr.recurrent_fwd_norm(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.g.to(dev), case.beta.to(dev),
                               pool.view, case.state_indices.to(dev), case.cu_seqlens.to(dev), nw, nz,
                               eps=case.norm["eps"], scale=case.scale, flags=flags, o=o.view,
                               intermediate_states=ib.view if ib else None)
    elif gated:
        r = {n: t.to(dev) for n, t in case.raw.items()}
        gdr.recurrent_fwd_gated(case.q.to(dev), case.k.to(dev), case.v.to(dev), r["a"], r["b"], r["A_log"],
                                r["dt_bias"], pool.view, case.state_indices.to(dev), case.cu_seqlens.to(dev),
                                scale=case.scale, flags=flags, o=o.view, intermediate_states=ib.view if ib else None)
    else:
        gdr.recurrent_fwd(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.g.to(dev), case.beta.to(dev),
                          pool.view, case.state_indices.to(dev), case.cu_seqlens.to(dev), scale=case.scale,
                          flags=flags, o=o.view, intermediate_states=ib.view if ib else None)
    torch.cuda.synchronize()
    assert pool.guards_intact() and o.guards_intact() and (ib is None or ib.guards_intact())
    return pool, o, ib, o_init


def _o_init(case):
    """The sentinel run_case fills o with."""
    return sentinel_like((case.T, case.v.shape[1], case.v.shape[2]), case.q.dtype)


def check_case(case, pool, o, ib, o_init, *, commit):
    ro, rpool, rib = oracle.pool(case.q, case.k, case.v, case.g, case.beta, case.pool, case.state_indices,
                                 case.cu_seqlens, scale=case.scale, commit=commit, steps=case.steps,
                                 ibuf_rows=case.ibuf_rows)
    if case.norm is not None:  # padding rows of ro stay NaN
        ro = oracle.gated_rmsnorm(ro, case.norm["weight"], case.norm["gate"], case.norm["eps"])
    cu = case.cu_seqlens.tolist()
    idx = case.state_indices.tolist()
    valid_rows = [b for b in range(case.N) if idx[b] >= 0]
    ov = o.view.cpu()
    tok_valid = np.zeros(case.T, dtype=bool)
    for b in valid_rows:
        tok_valid[cu[b]:cu[b + 1]] = True
    # outputs of valid tokens vs the oracle; padding rows keep the sentinel bits
    if tok_valid.any():
        check_out(ov[torch.from_numpy(tok_valid)], ro[tok_valid], "o")
    assert bits_equal(ov[torch.from_numpy(~tok_valid)], o_init[torch.from_numpy(~tok_valid)])
    pv = pool.view.cpu()
    used = sorted(idx[b] for b in valid_rows)
    if commit and used:
        check_state(pv[used], rpool[used], "pool (committed slots)")
    untouched = [s for s in range(case.pool.shape[0]) if not (commit and s in set(used))]
    assert bits_equal(pv[untouched], case.pool[untouched]), "pool slots that must stay untouched changed"
    if ib is not None:
        ibv = ib.view.cpu()
        sentinel = sentinel_like(ibv.shape[2:], ibv.dtype)
        for b in range(case.ibuf_rows):
            L = cu[b + 1] - cu[b] if b < case.N else 0
            if b < case.N and idx[b] >= 0 and L > 0:
                check_state(ibv[b, :L], rib[b, :L], f"ibuf row {b}")
                rest = range(L, case.steps)
            else:
                rest = range(case.steps)
            for t in rest:
                assert bits_equal(ibv[b, t], sentinel), f"ibuf row {b} step {t} written"


def test_decode_fp32_pool_full_size():
    """256 single-token sequences, Hk 16 / Hv 32, K = V = 128, fp32 pool of 513
    slots, 26 padding rows, committed in place."""
    case = workloads.decode_fp32_pool()
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=False)
    check_case(case, pool, o, ib, o_init, commit=True)


def test_verify_bf16_pool_full_size():
    """64 sequences of 1..12 accepted tokens, bf16 pool, per-token states into
    [65, 12, 32, 128, 128], pool not committed."""
    case = workloads.verify_bf16_pool()
    pool, o, ib, o_init = run_case(case, flags=0, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=False)


def test_verify_with_padding_rows():
    case = workloads.verify_bf16_pool(pad_count=7)
    pool, o, ib, o_init = run_case(case, flags=0, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=False)


def test_channel_gate_decode_full_size():
    """Per-key-channel gates (tokenspeed PR #834's KDA decode): the decode
    workload with gk [T, Hv, K], fp32 pool committed in place."""
    case = workloads.decode_kda_fp32_pool()
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=False)
    check_case(case, pool, o, ib, o_init, commit=True)


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("dtype,pool_dtype", [(torch.bfloat16, torch.float32), (torch.float32, torch.float32),
                                              (torch.bfloat16, torch.bfloat16)])
def test_channel_gate_small_cases(K, dtype, pool_dtype):
    """Ragged verify with per-channel gates, GVA 2, padding row, per-token
    states and commit."""
    lens = [1, 7, 0, 12, 4]
    case = workloads.pool_case(41 + K, lens, 2, 4, K, K, 7, dtype=dtype, pool_dtype=pool_dtype, pad_count=1,
                               commit=True, steps=12, ibuf_rows=6, g_range=(-2.0, 0.0), channel_gate=True)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=True)


def test_channel_gate_constant_matches_scalar_gate():
    """A per-channel gate equal on every key channel gives the scalar-gate
    result (up to rounding order)."""
    case = workloads.pool_case(45, [3, 5, 1], 2, 4, 128, 128, 5, pool_dtype=torch.float32, commit=True,
                               steps=5, ibuf_rows=3)
    pool_a, o_a, ib_a, _ = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    import dataclasses
    chan = dataclasses.replace(case, g=case.g[:, :, None].expand(-1, -1, 128).contiguous())
    pool_b, o_b, ib_b, _ = run_case(chan, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_out(o_b.view.cpu(), o_a.view.cpu().double().numpy(), "o")
    check_state(pool_b.view.cpu(), pool_a.view.cpu().double().numpy(), "pool")
    cu = case.cu_seqlens.tolist()
    for b in range(case.N):
        L = cu[b + 1] - cu[b]
        check_state(ib_b.view[b, :L].cpu(), ib_a.view[b, :L].cpu().double().numpy(), f"ibuf row {b}")
    # and both against the oracle, the per-channel one on its own per-channel gates
    check_case(case, pool_a, o_a, ib_a, _o_init(case), commit=True)
    check_case(chan, pool_b, o_b, ib_b, _o_init(chan), commit=True)


def test_output_norm_decode_full_size():
    """Gated RMSNorm output epilogue (tokenspeed PR #834) fused into decode:
    the decode workload, rows normalised over V, scaled by the weight and the
    sigmoid of the gate; padding rows untouched."""
    case = workloads.decode_fp32_pool_norm()
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=False)
    check_case(case, pool, o, ib, o_init, commit=True)


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("channel", [False, True])
def test_output_norm_small_cases(K, channel):
    """Ragged verify with the epilogue: per-token states, commit, padding,
    scalar or per-channel gates."""
    lens = [1, 5, 0, 9]
    case = workloads.pool_case(61 + K, lens, 2, 4, K, K, 6, pool_dtype=torch.bfloat16, pad_count=1, commit=True,
                               steps=9, ibuf_rows=4, channel_gate=channel)
    case.norm = workloads.output_norm(62, case.T, 4, K, eps=1e-4)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=True)


def _with_oracle_gates(case, neg_eigval=False):
    """The case with g and beta formed from its raw projections by the oracle (fp64)."""
    import dataclasses
    r = case.raw
    g, beta = oracle.gating(r["a"], r["dt_bias"], r["A_log"], r["b"], neg_eigval=neg_eigval)
    return dataclasses.replace(case, g=torch.from_numpy(g), beta=torch.from_numpy(beta))


def test_gated_verify_full_size():
    """In-kernel gating (FlashQLA's in-kernel gating commit) on the verify
    workload: gates formed from raw a, b, A_log, dt_bias inside the kernel."""
    case = workloads.verify_bf16_pool_raw_gates()
    pool, o, ib, o_init = run_case(case, flags=0, with_ibuf=True, gated=True)
    check_case(_with_oracle_gates(case), pool, o, ib, o_init, commit=False)


@pytest.mark.parametrize("neg_eigval", [False, True])
@pytest.mark.parametrize("dtype,pool_dtype", [(torch.bfloat16, torch.float32), (torch.float32, torch.bfloat16)])
def test_gated_small_cases(neg_eigval, dtype, pool_dtype):
    lens = [1, 6, 0, 3, 12]
    case = workloads.pool_case(51, lens, 2, 4, 128, 128, 7, dtype=dtype, pool_dtype=pool_dtype, pad_count=1,
                               commit=True, steps=12, ibuf_rows=5)
    case.raw = workloads.raw_gates(52, case.T, 4, dtype=dtype)
    flags = gdr.GDR_COMMIT | (gdr.GDR_NEG_EIGVAL if neg_eigval else 0)
    pool, o, ib, o_init = run_case(case, flags=flags, with_ibuf=True, gated=True)
    check_case(_with_oracle_gates(case, neg_eigval), pool, o, ib, o_init, commit=True)


def _unnormalised(case, seed):
    """The case with each q / k row rescaled by a random factor in [0.25, 4]
    (rounded to the input dtype): inputs for the in-kernel normalisation."""
    gen = torch.Generator().manual_seed(seed)
    out = []
    for x in (case.q, case.k):
        f = torch.exp(torch.empty(x.shape[:2] + (1,)).uniform_(-1.386, 1.386, generator=gen))
        out.append((x.float() * f).to(x.dtype))
    return out


def _with_oracle_l2norm(case):
    """The case with q and k normalised by the oracle (x / sqrt(sum x^2 + 1e-6), fp64)."""
    import dataclasses
    return dataclasses.replace(case, q=torch.from_numpy(oracle.l2norm(case.q, 1e-6)),
                               k=torch.from_numpy(oracle.l2norm(case.k, 1e-6)))


@pytest.mark.parametrize("pool_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gated_with_qk_l2norm_ragged(dtype, pool_dtype):
    """The in-kernel gating and the in-kernel q / k normalisation in one verify
    launch (FlashQLA's in-kernel gating commit forms both inside the kernel):
    ragged 1..40-token sequences (windows of every fill, one empty sequence),
    padding rows, per-token states, the pool committed."""
    lens = torch.randint(1, 41, (9,), generator=torch.Generator().manual_seed(91)).tolist() + [0]
    case = workloads.pool_case(92, lens, 2, 4, 128, 128, 12, dtype=dtype, pool_dtype=pool_dtype, pad_count=2,
                               commit=True, steps=40, ibuf_rows=10)
    case.raw = workloads.raw_gates(93, case.T, 4, dtype=dtype)
    case.q, case.k = _unnormalised(case, 94)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT | gdr.GDR_QK_L2NORM, with_ibuf=True, gated=True)
    check_case(_with_oracle_l2norm(_with_oracle_gates(case)), pool, o, ib, o_init, commit=True)


def test_gated_with_qk_l2norm_decode():
    """Gating and normalisation in the kernel on single-token calls (inputs
    read straight from global memory), fp32 pool committed, padding rows."""
    case = workloads.pool_case(95, [1] * 24, 2, 4, 128, 128, 30, pool_dtype=torch.float32, pad_count=3,
                               commit=True)
    case.raw = workloads.raw_gates(96, case.T, 4)
    case.q, case.k = _unnormalised(case, 97)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT | gdr.GDR_QK_L2NORM, with_ibuf=False, gated=True)
    check_case(_with_oracle_l2norm(_with_oracle_gates(case)), pool, o, ib, o_init, commit=True)


def test_gated_with_qk_l2norm_verify_full_size():
    """The raw-gate verify workload (64 sequences of 1..12 tokens, bf16 pool,
    per-token states) with un-normalised q / k normalised in the kernel."""
    case = workloads.verify_bf16_pool_raw_gates()
    case.q, case.k = _unnormalised(case, 98)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_QK_L2NORM, with_ibuf=True, gated=True)
    check_case(_with_oracle_l2norm(_with_oracle_gates(case)), pool, o, ib, o_init, commit=False)


@pytest.mark.parametrize("Hk,Hv", [(4, 4), (2, 8), (1, 4)])       # MHA, GVA 4, MQA
@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("dtype,pool_dtype", [(torch.bfloat16, torch.float32), (torch.float32, torch.float32),
                                              (torch.bfloat16, torch.bfloat16)])
def test_small_cases(Hk, Hv, K, dtype, pool_dtype):
    lens = [1, 8, 3, 0, 12, 5]
    case = workloads.pool_case(31 + K + Hk, lens, Hk, Hv, K, K, 9, dtype=dtype, pool_dtype=pool_dtype,
                               pad_count=1, commit=True, steps=12, ibuf_rows=7, g_range=(-1.0, 0.0))
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=True)


def test_gate_endpoints_and_slot_zero():
    """g = 0 and g = -2 (adversarial decay), beta at 0 and 1; slot 0 valid."""
    case = workloads.pool_case(41, [4, 4, 4], 2, 4, 128, 128, 3, pool_dtype=torch.float32,
                               commit=True, steps=4, ibuf_rows=3)
    case.g[:4] = 0.0
    case.g[4:8] = -2.0
    case.beta[8:10] = 0.0
    case.beta[10:12] = 1.0
    case.state_indices = torch.tensor([0, 2, 1], dtype=torch.int32)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=True)


def test_qk_l2norm_flag():
    """GDR_QK_L2NORM normalises q and k rows in the kernel (x rsqrt(sum x^2 + 1e-6))."""
    case = workloads.pool_case(42, [2, 5, 1], 2, 4, 128, 128, 4, dtype=torch.float32,
                               pool_dtype=torch.float32, commit=True)
    gen = torch.Generator().manual_seed(5)
    case.q = torch.randn(case.q.shape, generator=gen) * 3.0
    case.k = torch.randn(case.k.shape, generator=gen) * 0.5
    pool, o, _, _ = run_case(case, flags=gdr.GDR_COMMIT | gdr.GDR_QK_L2NORM, with_ibuf=False)
    qn = torch.from_numpy(oracle.l2norm(case.q, 1e-6))
    kn = torch.from_numpy(oracle.l2norm(case.k, 1e-6))
    ro, rpool, _ = oracle.pool(qn, kn, case.v, case.g, case.beta, case.pool, case.state_indices,
                               case.cu_seqlens, scale=case.scale, commit=True)
    check_out(o.view.cpu(), ro, "o")
    used = sorted(int(s) for s in case.state_indices if s >= 0)
    check_state(pool.view.cpu()[used], rpool[used], "pool")


def test_decode_equals_chunk_path_at_one_token():
    """Decode at T = 1 and the chunked prefill at T = 1 give the same state."""
    case = workloads.pool_case(43, [1, 1, 1, 1], 2, 4, 128, 128, 4, pool_dtype=torch.float32, commit=True)
    case.state_indices = torch.arange(4, dtype=torch.int32)
    pool, o, _, _ = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=False)
    oc, sc = gdr.chunk_fwd(case.q.to(DEV), case.k.to(DEV), case.v.to(DEV), case.beta.to(DEV),
                           case.cu_seqlens.to(DEV), g=case.g.to(DEV), initial_state=case.pool.to(DEV),
                           scale=case.scale)
    torch.cuda.synchronize()
    check_state(pool.view.cpu(), sc.cpu().double().numpy(), "decode vs chunk state")
    check_out(o.view.cpu(), oc.float().cpu().double().numpy(), "decode vs chunk o")
    # and both against the oracle's tokenwise recurrence from the same states
    ro, rs = oracle.tokenwise(case.q, case.k, case.v, case.beta, case.cu_seqlens, g=case.g,
                              initial_state=case.pool[:4], scale=case.scale)
    check_state(sc.cpu(), rs, "chunk path final state vs oracle")
    check_state(pool.view.cpu(), rs, "decode pool vs oracle")
    check_out(oc.cpu(), ro, "chunk path o vs oracle")
    check_out(o.view.cpu(), ro, "decode o vs oracle")


def test_deterministic_repeat():
    case = workloads.verify_bf16_pool()
    outs = []
    for _ in range(3):
        pool, o, ib, _ = run_case(case, flags=0, with_ibuf=True)
        outs.append((o.view.cpu(), ib.view.cpu()))
    for o2, ib2 in outs[1:]:
        assert bits_equal(o2, outs[0][0]) and bits_equal(ib2, outs[0][1])


def test_validate_flag_rejects_bad_content():
    case = workloads.pool_case(44, [2, 3], 2, 4, 128, 128, 4, pool_dtype=torch.float32, commit=True,
                               steps=3, ibuf_rows=2)
    dev = DEV
    args = [case.q.to(dev), case.k.to(dev), case.v.to(dev), case.g.to(dev), case.beta.to(dev)]
    pool = case.pool.to(dev)
    ib = torch.zeros((2, 3) + tuple(case.pool.shape[1:]), device=dev)
    bad_idx = torch.tensor([1, 1], dtype=torch.int32, device=dev)          # duplicate slot
    with pytest.raises(gdr.GdrError) as e:
        gdr.recurrent_fwd(*args, pool, bad_idx, case.cu_seqlens.to(dev), flags=gdr.GDR_COMMIT | gdr.GDR_VALIDATE,
                          intermediate_states=ib)
    assert e.value.code == 6 and "duplicate" in str(e.value)
    g_bad = case.g.clone()
    g_bad[0, 0] = 0.5                                                   # gate > 0
    args[3] = g_bad.to(dev)
    with pytest.raises(gdr.GdrError):
        gdr.recurrent_fwd(*args, pool, case.state_indices.to(dev), case.cu_seqlens.to(dev),
                          flags=gdr.GDR_VALIDATE, intermediate_states=ib)
    assert torch.equal(pool.cpu(), case.pool)                            # nothing launched


def test_cuda_graph_replay_equals_eager():
    case = workloads.verify_bf16_pool()
    dev = DEV
    ins = [t.to(dev) for t in (case.q, case.k, case.v, case.g, case.beta)]
    pool = case.pool.to(dev)
    idx, cu = case.state_indices.to(dev), case.cu_seqlens.to(dev)
    o = torch.empty(case.T, 32, 128, dtype=torch.bfloat16, device=dev)
    ib = torch.zeros((65, 12, 32, 128, 128), dtype=torch.bfloat16, device=dev)
    gdr.recurrent_fwd(*ins, pool, idx, cu, scale=case.scale, flags=0, o=o, intermediate_states=ib)
    torch.cuda.synchronize()
    o_e, ib_e = o.clone(), ib.clone()
    o.zero_()
    ib.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gdr.recurrent_fwd(*ins, pool, idx, cu, scale=case.scale, flags=0, o=o, intermediate_states=ib,
                              stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert bits_equal(o, o_e) and bits_equal(ib, ib_e)


# Multi-token calls stage each window of up to 16 tokens' inputs in shared
# memory; sequences of 17, 33 and 40 tokens cross one to two window edges.
LONG_LENS = [1, 17, 40, 0, 33, 16]


@pytest.mark.parametrize("mode", ["scalar", "channel", "gated", "norm", "norm_channel"])
@pytest.mark.parametrize("K", [64, 128])
def test_multi_window_sequences(mode, K):
    dtype = torch.float32 if K == 64 else torch.bfloat16
    pool_dtype = torch.bfloat16 if mode.startswith("norm") else torch.float32
    case = workloads.pool_case(71 + K, LONG_LENS, 2, 4, K, K, 8, dtype=dtype, pool_dtype=pool_dtype, pad_count=1,
                               commit=True, steps=40, ibuf_rows=6, g_range=(-0.5, 0.0),
                               channel_gate=mode in ("channel", "norm_channel"))
    if mode.startswith("norm"):
        case.norm = workloads.output_norm(72, case.T, 4, K, dtype=dtype, eps=1e-4)
    if mode == "gated":
        case.raw = workloads.raw_gates(73, case.T, 4, dtype=dtype)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True, gated=mode == "gated")
    check_case(_with_oracle_gates(case) if mode == "gated" else case, pool, o, ib, o_init, commit=True)


def test_multi_window_qk_l2norm():
    """GDR_QK_L2NORM on the staged path: q and k normalised once per window."""
    case = workloads.pool_case(74, LONG_LENS, 2, 4, 128, 128, 8, dtype=torch.float32, pool_dtype=torch.float32,
                               commit=True)
    gen = torch.Generator().manual_seed(6)
    case.q = torch.randn(case.q.shape, generator=gen) * 3.0
    case.k = torch.randn(case.k.shape, generator=gen) * 0.5
    pool, o, _, _ = run_case(case, flags=gdr.GDR_COMMIT | gdr.GDR_QK_L2NORM, with_ibuf=False)
    qn = torch.from_numpy(oracle.l2norm(case.q, 1e-6))
    kn = torch.from_numpy(oracle.l2norm(case.k, 1e-6))
    ro, rpool, _ = oracle.pool(qn, kn, case.v, case.g, case.beta, case.pool, case.state_indices,
                               case.cu_seqlens, scale=case.scale, commit=True)
    check_out(o.view.cpu(), ro, "o")
    used = sorted(int(s) for s in case.state_indices if s >= 0)
    check_state(pool.view.cpu()[used], rpool[used], "pool")


@pytest.mark.parametrize("mode", ["scalar", "channel", "norm"])
def test_direct_path_multi_token_sequence(mode):
    """A call with as many tokens as sequences reads its inputs straight from
    global memory; a 3-token sequence beside two empty ones still runs every
    token in order."""
    case = workloads.pool_case(75, [3, 0, 0, 1], 2, 4, 128, 128, 5, pool_dtype=torch.float32, commit=True,
                               steps=3, ibuf_rows=4, channel_gate=mode == "channel")
    if mode == "norm":
        case.norm = workloads.output_norm(76, case.T, 4, 128, eps=1e-4)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=True)


@pytest.mark.parametrize("mode", ["scalar", "channel", "gated"])
def test_multi_token_wide_blocks(mode):
    """Enough (sequence, head) units for the 128-row blocks of multi-token
    calls (80 x 4 = 320, two per SM): ragged 1..40-token sequences, so windows
    of every fill, and padding rows; the pool is committed (the per-token
    states of these block sizes are covered by the full-size verify tests)."""
    lens = torch.randint(1, 41, (80,), generator=torch.Generator().manual_seed(77)).tolist()
    case = workloads.pool_case(78, lens, 2, 4, 128, 128, 90, pool_dtype=torch.bfloat16, pad_count=3, commit=True,
                               g_range=(-0.5, 0.0), channel_gate=mode == "channel")
    if mode == "gated":
        case.raw = workloads.raw_gates(79, case.T, 4)
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=False, gated=mode == "gated")
    check_case(_with_oracle_gates(case) if mode == "gated" else case, pool, o, ib, o_init, commit=True)


def test_multi_token_beyond_longest_first_limit():
    """1500 multi-token sequences (more than the 1024 a call ranks longest
    first, so the CTAs take them in index order): 1..4 tokens each, padding
    rows, bf16 pool committed, per-token states."""
    lens = torch.randint(1, 5, (1500,), generator=torch.Generator().manual_seed(81)).tolist()
    case = workloads.pool_case(82, lens, 1, 2, 128, 128, 1600, pool_dtype=torch.bfloat16, pad_count=40, commit=True,
                               steps=4, ibuf_rows=1500, g_range=(-0.5, 0.0))
    pool, o, ib, o_init = run_case(case, flags=gdr.GDR_COMMIT, with_ibuf=True)
    check_case(case, pool, o, ib, o_init, commit=True)
