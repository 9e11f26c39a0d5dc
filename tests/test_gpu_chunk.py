"""GPU parity of the chunked prefill against the CPU oracle, through the C ABI:
the three prefill workloads at full size (the long KDA one on sampled heads),
small ragged / GVA / tail / adversarial-decay cases, contract checks."""
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


def run_gpu(case, flags=0, guarded=True):
    dev = DEV
    T, Hv, V, K, N = case.T, case.v.shape[1], case.v.shape[2], case.q.shape[2], case.N
    o = Guarded((T, Hv, V), case.q.dtype, dev)
    sf = Guarded((N, Hv, V, K), torch.float32, dev)
    ins = dict(g=case.g.to(dev) if case.g is not None else None,
               gk=case.gk.to(dev) if case.gk is not None else None,
               initial_state=case.initial_state.to(dev) if case.initial_state is not None else None)
    q, k, v, beta = case.q.to(dev), case.k.to(dev), case.v.to(dev), case.beta.to(dev)
    snap = [t.clone() for t in (q, k, v, beta)]
    gdr.chunk_fwd(q, k, v, beta, case.cu_seqlens.to(dev), scale=case.scale, flags=flags, o=o.view,
                  final_state=sf.view, **ins)
    torch.cuda.synchronize()
    assert gdr.device_status() == 0, "a bounded device wait gave up"
    assert o.guards_intact() and sf.guards_intact(), "write outside the output buffers"
    for a, b in zip((q, k, v, beta), snap):
        assert bits_equal(a, b), "an input was modified"
    return o.view, sf.view


def oracle_ref(case, heads=None):
    if heads is None:
        return oracle.tokenwise(case.q, case.k, case.v, case.beta, case.cu_seqlens, g=case.g, gk=case.gk,
                                initial_state=case.initial_state, scale=case.scale)
    Hk, Hv = case.q.shape[1], case.v.shape[1]
    kh = [h // (Hv // Hk) for h in heads]
    sl = lambda t: None if t is None else t[:, heads]
    return oracle.tokenwise(case.q[:, kh], case.k[:, kh], case.v[:, heads], case.beta[:, heads],
                            case.cu_seqlens, g=sl(case.g), gk=sl(case.gk),
                            initial_state=None if case.initial_state is None else case.initial_state[:, heads],
                            scale=case.scale)


def test_tiny_fp32_prefill_full_size():
    """1 sequence T=128 (2 chunks), 2 heads, K=V=64, fp32, scale 1/8."""
    case = workloads.tiny_fp32_prefill()
    o, sf = run_gpu(case)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_varlen_bf16_prefill_full_size():
    """4 sequences {65,1000,2048,3000}, H=16, K=V=128, bf16, g ~ U[-2,0], h0."""
    case = workloads.varlen_bf16_prefill()
    o, sf = run_gpu(case)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_kda_long_prefill_full_size_sampled_heads():
    """T=32768, Hk 16 / Hv 32, per-channel gk ~ U[-0.1,0]; the oracle runs the
    whole sequence for 4 sampled value-heads (both heads of one key head, and
    two others), every token of those heads is compared."""
    case = workloads.kda_long_prefill()
    o, sf = run_gpu(case, guarded=True)
    heads = [0, 1, 17, 30]
    ro, rs = oracle_ref(case, heads)
    check_out(o[:, heads].cpu(), ro, "o (sampled heads)")
    check_state(sf[:, heads].cpu(), rs, "final state (sampled heads)")


CASES = [
    # (lens, Hk, Hv, gate, g_range, h0, dtype, K)
    ([1], 2, 2, "g", (-0.05, 0.0), False, torch.bfloat16, 128),
    ([65, 1], 2, 2, "g", (-1.0, 0.0), True, torch.bfloat16, 128),
    ([65, 63], 2, 2, "g", (-2.0, 0.0), True, torch.bfloat16, 128),
    ([1024], 1, 1, "g", (-0.5, 0.0), False, torch.bfloat16, 128),
    ([1] * 32, 2, 2, "g", (-1.0, 0.0), True, torch.bfloat16, 128),
    ([1, 63, 65, 2], 2, 4, "g", (-2.0, 0.0), True, torch.bfloat16, 128),     # GVA 2
    ([4], 1, 4, "g", (-1.0, 0.0), True, torch.bfloat16, 128),                # GVA 4 with init
    ([65, 1, 129, 63], 1, 4, "gk", (-0.3, 0.0), True, torch.bfloat16, 128),  # KDA GVA 4
    ([200, 7], 2, 4, "gk", (-2.0, 0.0), False, torch.bfloat16, 128),         # KDA adversarial
    ([100, 28], 2, 2, "g", (-1.0, 0.0), True, torch.float32, 64),
    ([65, 1, 130, 64], 2, 4, "g", (-2.0, 0.0), True, torch.bfloat16, 64),   # bf16, 64 channels: tensor cores
    ([130, 7, 64], 1, 2, "gk", (-0.5, 0.0), True, torch.bfloat16, 64),      # KDA, 64 channels
    ([130, 3], 1, 2, "gk", (-0.5, 0.0), True, torch.float32, 128),
]


@pytest.mark.parametrize("lens,Hk,Hv,gate,g_range,h0,dtype,K", CASES)
def test_small_cases(lens, Hk, Hv, gate, g_range, h0, dtype, K):
    case = workloads.chunk_case(51 + sum(lens) % 97, lens, Hk, Hv, K, K, dtype=dtype, gate=gate,
                                g_range=g_range, h0_std=0.1 if h0 else None)
    o, sf = run_gpu(case)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


@pytest.mark.parametrize("gate", ["g", "gk"])
def test_gate_minus_two_everywhere(gate):
    """g = -2 on every token: a prefix of -128 per 64-token chunk; every
    exponential must stay an in-chunk difference (finite results)."""
    case = workloads.chunk_case(61, [128, 64, 33], 2, 2, 128, 128, gate=gate, h0_std=0.1)
    if gate == "g":
        case.g[:] = -2.0
    else:
        case.gk[:] = -2.0
    o, sf = run_gpu(case)
    assert torch.isfinite(o.float()).all() and torch.isfinite(sf).all()
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


@pytest.mark.parametrize("g_range", [(-0.3, 0.0), (-4.0, 0.0)])
def test_channel_gate_every_chunk_length(g_range):
    """Per-key-channel gates on sequences of every length 1..64 (so a chunk of
    every fill, each pivot of the in-chunk pairs falling inside and beyond the
    chunk end), behind 65- and 128-token sequences, GVA 2, with an initial
    state; decays up to -4 per token and channel."""
    lens = [65] + list(range(1, 65)) + [128]
    case = workloads.chunk_case(63 + int(-g_range[0]), lens, 1, 2, 128, 128, gate="gk", g_range=g_range, h0_std=0.1)
    o, sf = run_gpu(case)
    assert torch.isfinite(o.float()).all() and torch.isfinite(sf).all()
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_gate_zero_and_beta_endpoints():
    case = workloads.chunk_case(62, [70, 64], 2, 2, 128, 128, h0_std=0.1)
    case.g[:40] = 0.0
    case.beta[:20] = 0.0
    case.beta[20:60] = 1.0
    o, sf = run_gpu(case)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_channel_gate_zero_and_beta_endpoints():
    """Per-channel gates with no decay at all: tokens on which no channel
    decays (chunks of decay span 0) and channels that never decay, with beta
    at 0 and at 1, GVA 2 and an initial state."""
    case = workloads.chunk_case(65, [70, 64, 130], 1, 2, 128, 128, gate="gk", g_range=(-0.5, 0.0), h0_std=0.1)
    case.gk[:40] = 0.0
    case.gk[:, :, :16] = 0.0
    case.beta[:20] = 0.0
    case.beta[20:60] = 1.0
    o, sf = run_gpu(case)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_qk_l2norm_flag():
    case = workloads.chunk_case(63, [90, 40], 2, 4, 128, 128, dtype=torch.float32, h0_std=0.1)
    gen = torch.Generator().manual_seed(3)
    case.q = torch.randn(case.q.shape, generator=gen) * 2.0
    case.k = torch.randn(case.k.shape, generator=gen) * 0.7
    o, sf = run_gpu(case, flags=gdr.GDR_QK_L2NORM)
    qn = torch.from_numpy(oracle.l2norm(case.q, 1e-6))
    kn = torch.from_numpy(oracle.l2norm(case.k, 1e-6))
    ro, rs = oracle.tokenwise(qn, kn, case.v, case.beta, case.cu_seqlens, g=case.g,
                              initial_state=case.initial_state, scale=case.scale)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_position_independence():
    """A sequence's result does not depend on where it sits in the packed batch."""
    a = workloads.chunk_case(64, [100, 37, 70], 1, 2, 128, 128, h0_std=0.1)
    o1, s1 = run_gpu(a)
    perm = [2, 0, 1]
    cu = a.cu_seqlens.tolist()
    segs = [slice(cu[i], cu[i + 1]) for i in range(3)]
    b = workloads.ChunkCase(name="perm", q=torch.cat([a.q[segs[i]] for i in perm]),
                            k=torch.cat([a.k[segs[i]] for i in perm]), v=torch.cat([a.v[segs[i]] for i in perm]),
                            beta=torch.cat([a.beta[segs[i]] for i in perm]),
                            g=torch.cat([a.g[segs[i]] for i in perm]),
                            cu_seqlens=torch.tensor([0, 70, 170, 207], dtype=torch.int32),
                            scale=a.scale, initial_state=a.initial_state[perm])
    o2, s2 = run_gpu(b)
    for j, i in enumerate(perm):
        assert bits_equal(s2[j], s1[i])
        cb = b.cu_seqlens.tolist()
        assert bits_equal(o2[cb[j]:cb[j + 1]], o1[segs[i]])


def test_deterministic_repeat():
    case = workloads.varlen_bf16_prefill()
    o1, s1 = run_gpu(case)
    o1, s1 = o1.clone(), s1.clone()
    for _ in range(2):
        o2, s2 = run_gpu(case)
        assert bits_equal(o2, o1) and bits_equal(s2, s1)


def test_validate_flag():
    case = workloads.chunk_case(65, [10, 20], 1, 1, 128, 128)
    dev = DEV
    g = case.g.clone()
    g[3, 0] = float("inf")
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_fwd(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.beta.to(dev),
                      case.cu_seqlens.to(dev), g=g.to(dev), flags=gdr.GDR_VALIDATE)
    assert e.value.code == 6
    bad_cu = torch.tensor([0, 20, 10], dtype=torch.int32, device=dev)
    with pytest.raises(gdr.GdrError):
        gdr.chunk_fwd(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.beta.to(dev), bad_cu,
                      g=case.g.to(dev), flags=gdr.GDR_VALIDATE)


@pytest.mark.parametrize("n_seqs", [3, 70])
@pytest.mark.parametrize("defect", ["decreasing", "last_not_T", "first_not_zero"])
def test_malformed_cu_seqlens_writes_nothing(n_seqs, defect):
    """Without GDR_VALIDATE a malformed cu_seqlens is found on the device and
    no output is written (3 sequences: the prep forms the chunk metadata
    itself; 70: the metadata kernel does)."""
    case = workloads.chunk_case(67, [40] * n_seqs, 1, 2, 128, 128, gate="g", h0_std=0.1)
    cu = case.cu_seqlens.clone()
    if defect == "decreasing":
        cu[1], cu[2] = cu[2].item(), cu[1].item()
    elif defect == "last_not_T":
        cu[-1] -= 5
    else:
        cu[0] = 1
    dev = DEV
    o = Guarded(tuple(case.v.shape), case.q.dtype, dev, fill_bytes=sentinel_like(case.v.shape, case.q.dtype))
    sf_shape = (case.N, 2, 128, 128)
    sf = Guarded(sf_shape, torch.float32, dev, fill_bytes=sentinel_like(sf_shape, torch.float32))
    gdr.chunk_fwd(case.q.to(dev), case.k.to(dev), case.v.to(dev), case.beta.to(dev), cu.to(dev), g=case.g.to(dev),
                  initial_state=case.initial_state.to(dev), scale=case.scale, o=o.view, final_state=sf.view)
    torch.cuda.synchronize()
    assert gdr.device_status() == 0
    assert o.guards_intact() and sf.guards_intact()
    assert bits_equal(o.view, sentinel_like(case.v.shape, case.q.dtype))
    assert bits_equal(sf.view, sentinel_like(sf_shape, torch.float32))


def test_cuda_graph_replay_equals_eager():
    case = workloads.varlen_bf16_prefill()
    dev = DEV
    q, k, v, beta = (t.to(dev) for t in (case.q, case.k, case.v, case.beta))
    g, h0, cu = case.g.to(dev), case.initial_state.to(dev), case.cu_seqlens.to(dev)
    o = torch.empty_like(v)
    sf = torch.empty_like(h0)
    ws = torch.empty(gdr.chunk_workspace_size(case.N, case.T, 16, 16, 128, 128, gate_kind=0, dtype=0),
                     dtype=torch.uint8, device=dev)
    gdr.chunk_fwd(q, k, v, beta, cu, g=g, initial_state=h0, scale=case.scale, o=o, final_state=sf, workspace=ws)
    torch.cuda.synchronize()
    o_e, s_e = o.clone(), sf.clone()
    o.zero_()
    sf.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gdr.chunk_fwd(q, k, v, beta, cu, g=g, initial_state=h0, scale=case.scale, o=o, final_state=sf,
                          workspace=ws, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert bits_equal(o, o_e) and bits_equal(sf, s_e)


def test_gating_kernel():
    T, Hv = 300, 8
    gen = torch.Generator().manual_seed(66)
    a = torch.randn(T, Hv, generator=gen) * 8
    a[0, 0] = 30.0                       # threshold branch
    b = torch.randn(T, Hv, generator=gen) * 3
    dt = torch.randn(Hv, generator=gen)
    A_log = torch.randn(Hv, generator=gen) * 0.5
    for flags, neg in ((0, False), (gdr.GDR_NEG_EIGVAL, True)):
        g, beta = gdr.gating_fwd(a.to(DEV), dt.to(DEV), A_log.to(DEV), b.to(DEV), flags=flags)
        torch.cuda.synchronize()
        rg, rb = oracle.gating(a, dt, A_log, b, neg_eigval=neg)
        np.testing.assert_allclose(g.cpu().double().numpy(), rg, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(beta.cpu().double().numpy(), rb, rtol=1e-5, atol=1e-6)


def test_most_sequences_per_call():
    """65535 sequences in one call, the most the tensor-core path accepts (one
    grid row per sequence): mostly one token, some spanning one, two and four
    chunks, in a shuffled order.  A sample of the sequences (every long one and
    a random set of short ones) is checked against the oracle, computed on each
    sequence alone; every output row must be finite."""
    gen = torch.Generator().manual_seed(64)
    lens = [1] * 65400 + [64] * 100 + [65] * 20 + [200] * 15
    lens = [lens[i] for i in torch.randperm(len(lens), generator=gen).tolist()]
    case = workloads.chunk_case(64, lens, 1, 1, 128, 128, gate="g", g_range=(-1.0, 0.0))
    dev = DEV
    q, k, v, beta, g = (t.to(dev) for t in (case.q, case.k, case.v, case.beta, case.g))
    o, sf = gdr.chunk_fwd(q, k, v, beta, case.cu_seqlens.to(dev), g=g, scale=case.scale)
    torch.cuda.synchronize()
    assert gdr.device_status() == 0
    assert torch.isfinite(o.float()).all()
    cu = case.cu_seqlens.tolist()
    longs = [b for b in range(case.N) if cu[b + 1] - cu[b] > 1]
    shorts = torch.randperm(case.N, generator=gen)[:64].tolist()
    for b in longs + shorts:
        sl = slice(cu[b], cu[b + 1])
        ro, rs = oracle.tokenwise(case.q[sl], case.k[sl], case.v[sl], case.beta[sl], [0, cu[b + 1] - cu[b]],
                                  g=case.g[sl], scale=case.scale)
        check_out(o[sl].cpu(), ro, f"o of sequence {b}")
        check_state(sf[b:b + 1].cpu(), rs, f"final state of sequence {b}")


def test_bf16_64_channels_run_on_the_tensor_cores():
    """bf16 heads of 64 channels take the tensor-core kernels (128-channel
    tiles, upper half zero), not the CUDA-core ones; GDR_CHUNK_SCAN is ignored
    for them (bit-identical results); the in-library q/k normalisation too."""
    case = workloads.chunk_case(65, [300, 40, 129], 2, 4, 64, 64, gate="g", g_range=(-1.0, 0.0), h0_std=0.1)
    gdr.profile_read()
    gdr.profile_enable(True)
    o, sf = run_gpu(case)
    o, sf = o.clone(), sf.clone()
    o2, s2 = run_gpu(case, flags=gdr.GDR_CHUNK_SCAN)
    torch.cuda.synchronize()
    gdr.profile_enable(False)
    names = set(gdr.profile_read())
    assert {"chunk_prep", "chunk_chain"} <= names, names
    assert not names & {"chunk_intra", "chunk_state", "chunk_out", "chunk_seg_scan"}, names
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")
    assert bits_equal(o, o2) and bits_equal(sf, s2)

    gen = torch.Generator().manual_seed(66)
    case.q = (torch.randn(case.q.shape, generator=gen) * 2.0).to(torch.bfloat16)
    case.k = (torch.randn(case.k.shape, generator=gen) * 0.7).to(torch.bfloat16)
    o3, s3 = run_gpu(case, flags=gdr.GDR_QK_L2NORM)
    # the library stores the normalised rows in the input type: the oracle runs on them rounded to bf16
    qn = torch.from_numpy(oracle.l2norm(case.q, 1e-6)).to(torch.bfloat16)
    kn = torch.from_numpy(oracle.l2norm(case.k, 1e-6)).to(torch.bfloat16)
    ro3, rs3 = oracle.tokenwise(qn, kn, case.v, case.beta, case.cu_seqlens, g=case.g,
                                initial_state=case.initial_state, scale=case.scale)
    check_out(o3.cpu(), ro3, "o (in-library q/k normalisation)")
    check_state(s3.cpu(), rs3, "final state (in-library q/k normalisation)")


def test_state_error_matches_the_split_model():
    """The kernels' final-state error against the oracle is the one the CPU
    model of their bf16 hi / lo split products predicts (within 3x): no
    rounding beyond the modelled split terms, on weak and strong decays."""
    from tests.test_split_terms import ALL_TERMS, _cases, model_final_states, rel_l2
    for name, case in _cases().items():
        _, sf = run_gpu(case)
        _, rs = oracle_ref(case)
        rs = np.asarray(rs)
        e_gpu = rel_l2(sf.cpu().double().numpy(), rs)
        e_model = rel_l2(model_final_states(case, ALL_TERMS), rs)
        print(f"{name}: GPU {e_gpu:.2e}, model {e_model:.2e}")
        assert e_gpu <= 3 * e_model, f"{name}: GPU {e_gpu:.2e} against the model's {e_model:.2e}"


def test_channel_gate_single_and_level_pivot_chunks():
    """Per-channel gates whose chunks fall on both sides of the single-pivot
    limit (a decay span of 2^64 over a chunk on some channel): chunks of
    small decays, of large decays (-2 per token), and chunks with spans just
    below and just above the limit, in one call with GVA, ragged lengths and
    an initial state."""
    lens = [130, 257, 64, 70, 5]
    case = workloads.chunk_case(71, lens, 1, 2, 128, 128, gate="gk", g_range=(-0.05, 0.0), h0_std=0.1)
    gk = case.gk
    ln2 = float(np.log(2.0))
    # a chunk's span is the decay after its first token: 63 tokens of a 64-token chunk
    gk[130:200] *= 40.0                        # up to -2 per token: spans far above the limit
    gk[387:451] = -60.0 * ln2 / 64.0           # the 64-token sequence: 2^59 on half the channels,
    gk[387:451, :, 64:] = -66.0 * ln2 / 64.0   # 2^65 on the others (just above the limit)
    gk[451:515] = -64.5 * ln2 / 64.0           # a whole chunk at 2^63.5 (just below)
    o, sf = run_gpu(case)
    assert torch.isfinite(o.float()).all() and torch.isfinite(sf).all()
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")
