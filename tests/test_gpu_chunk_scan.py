"""GPU parity of the chunk-parallel scan (GDR_CHUNK_SCAN) against the CPU
oracle, through the C ABI: the long few-head workload at full size, ragged
multi-sequence cases whose segments end inside a sequence, on a partial chunk
and exactly on a segment boundary, per-channel gates, GVA, and agreement with
the one-pass chain on the same inputs."""
import numpy as np
import pytest
import torch

import gated_delta_rule_37_gb300 as gdr
import oracle
from gated_delta_rule_37_gb300 import workloads
from tests.gpu_util import bits_equal, check_out, check_state, rel_l2
from tests.test_gpu_chunk import oracle_ref, run_gpu

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SCAN = gdr.GDR_CHUNK_SCAN


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load()


def test_long_few_heads_full_size():
    """T=32768, Hk = Hv = 4, g ~ U[-0.1,0], h0: every token and the final state
    of every head against the oracle."""
    case = workloads.long_few_heads_prefill()
    o, sf = run_gpu(case, flags=SCAN)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


SCAN_CASES = [
    # (lens, Hk, Hv, gate, g_range, h0); the library picks the segment length
    # (4 to 7 chunks at these sizes): 2 to 13 segments per sequence
    ([4096], 1, 1, "g", (-0.5, 0.0), True),                 # 13 segments
    ([512], 1, 1, "g", (-0.3, 0.0), True),                  # 2 segments: the scan forms no product
    ([1536], 1, 1, "g", (-0.05, 0.0), False),               # the last segment ends on its boundary
    ([1500, 65, 3000, 1], 1, 2, "g", (-0.3, 0.0), True),    # partial chunks, one-segment sequences
    ([1030, 2], 2, 4, "g", (-2.0, 0.0), True),              # GVA, adversarial decay
    ([2100, 700], 1, 2, "gk", (-0.3, 0.0), False),          # per-channel gates
    ([1100], 2, 4, "gk", (-0.05, 0.0), True),               # per-channel gates, GVA, h0
]


@pytest.mark.parametrize("lens,Hk,Hv,gate,g_range,h0", SCAN_CASES)
def test_scan_small_cases(lens, Hk, Hv, gate, g_range, h0):
    case = workloads.chunk_case(71 + sum(lens) % 89, lens, Hk, Hv, 128, 128, dtype=torch.bfloat16, gate=gate,
                                g_range=g_range, h0_std=0.1 if h0 else None)
    o, sf = run_gpu(case, flags=SCAN)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_scan_agrees_with_one_pass_chain():
    """The same inputs with and without the scan: both within the parity bound
    of the oracle, and close to each other (the scan only reassociates fp32
    state arithmetic)."""
    case = workloads.chunk_case(77, [3000, 900], 2, 2, 128, 128, dtype=torch.bfloat16, gate="g",
                                g_range=(-0.2, 0.0), h0_std=0.1)
    o1, s1 = run_gpu(case)
    o2, s2 = run_gpu(case, flags=SCAN)
    assert rel_l2(s2.cpu().numpy(), s1.cpu().numpy()) <= 1e-4
    assert rel_l2(o2.float().cpu().numpy(), o1.float().cpu().numpy()) <= 5e-3
    ro, rs = oracle.tokenwise(case.q, case.k, case.v, case.beta, case.cu_seqlens, g=case.g,
                              initial_state=case.initial_state, scale=case.scale)
    for o, sf, what in ((o1, s1, "one pass"), (o2, s2, "scan")):
        check_out(o.cpu(), ro, f"o ({what}) vs oracle")
        check_state(sf.cpu(), rs, f"final state ({what}) vs oracle")


def test_scan_deterministic_and_graph_safe():
    """Two scan calls give bit-identical results, and a CUDA-graph replay of the
    call equals the eager call."""
    case = workloads.chunk_case(78, [2500], 1, 2, 128, 128, dtype=torch.bfloat16, gate="g",
                                g_range=(-0.2, 0.0), h0_std=0.1)
    q, k, v, beta = (t.to(DEV) for t in (case.q, case.k, case.v, case.beta))
    g, h0, cu = case.g.to(DEV), case.initial_state.to(DEV), case.cu_seqlens.to(DEV)
    T, Hv = case.T, case.v.shape[1]
    need = gdr.chunk_workspace_size(case.N, T, 1, Hv, 128, 128, gate_kind=0, dtype=0, flags=SCAN)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(2):
        o = torch.empty(T, Hv, 128, dtype=torch.bfloat16, device=DEV)
        sf = torch.empty(case.N, Hv, 128, 128, dtype=torch.float32, device=DEV)
        gdr.chunk_fwd(q, k, v, beta, cu, g=g, initial_state=h0, scale=case.scale, flags=SCAN, o=o,
                      final_state=sf, workspace=ws)
        outs.append((o, sf))
    torch.cuda.synchronize()
    assert bits_equal(outs[0][0], outs[1][0]) and bits_equal(outs[0][1], outs[1][1])
    og = torch.empty_like(outs[0][0])
    sg = torch.empty_like(outs[0][1])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gdr.chunk_fwd(q, k, v, beta, cu, g=g, initial_state=h0, scale=case.scale, flags=SCAN, o=og,
                          final_state=sg, workspace=ws, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert bits_equal(og, outs[0][0]) and bits_equal(sg, outs[0][1])


def test_scan_gate_minus_two_everywhere():
    """g = -2 on every token: every segment transition decays to (nearly) zero
    and every exponential stays an in-chunk difference."""
    case = workloads.chunk_case(81, [1300, 700], 1, 2, 128, 128, gate="g", h0_std=0.1)
    case.g[:] = -2.0
    o, sf = run_gpu(case, flags=SCAN)
    assert torch.isfinite(o.float()).all() and torch.isfinite(sf).all()
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_scan_many_ragged_sequences():
    """40 sequences of 1..700 tokens: one to several segments each, the
    segment table spanning many sequences."""
    gen = torch.Generator().manual_seed(82)
    lens = torch.randint(1, 701, (40,), generator=gen).tolist()
    case = workloads.chunk_case(82, lens, 1, 2, 128, 128, gate="g", g_range=(-0.3, 0.0), h0_std=0.1)
    o, sf = run_gpu(case, flags=SCAN)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")


def test_scan_with_qk_l2norm():
    """GDR_CHUNK_SCAN together with in-library q / k normalisation (bf16): the
    oracle runs on the normalised rows rounded to bf16 as the library stores them."""
    case = workloads.chunk_case(83, [2100, 300], 1, 2, 128, 128, gate="g", g_range=(-0.2, 0.0), h0_std=0.1)
    gen = torch.Generator().manual_seed(84)
    q = (torch.randn(case.q.shape, generator=gen) * 2.0).to(torch.bfloat16)
    k = (torch.randn(case.k.shape, generator=gen) * 0.7).to(torch.bfloat16)
    case.q, case.k = q, k
    o, sf = run_gpu(case, flags=SCAN | gdr.GDR_QK_L2NORM)

    def norm_bf16(x):
        xf = x.float()
        return (xf * torch.rsqrt((xf * xf).sum(-1, keepdim=True) + 1e-6)).to(torch.bfloat16)

    ref = workloads.ChunkCase(name="normed", q=norm_bf16(q), k=norm_bf16(k), v=case.v, beta=case.beta, g=case.g,
                              cu_seqlens=case.cu_seqlens, scale=case.scale, initial_state=case.initial_state)
    ro, rs = oracle_ref(ref)
    check_out(o.cpu(), ro, "o")
    check_state(sf.cpu(), rs, "final state")



@pytest.mark.parametrize("trial", range(6))
def test_random_configurations(trial):
    """Seeded random shapes through the tensor-core path, with and without the
    scan: 1-6 sequences of 1-1500 tokens, GVA 1 or 2, scalar or per-channel
    gates, with or without h0."""
    rng = np.random.default_rng(900 + trial)
    n = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(1, 1501, n)]
    Hk = int(rng.integers(1, 3))
    Hv = Hk * int(rng.integers(1, 3))
    gate = "g" if rng.random() < 0.6 else "gk"
    lo = float(rng.choice([-2.0, -0.5, -0.05]))
    h0 = trial % 3 != 0
    flags = SCAN if trial % 2 == 0 else 0
    case = workloads.chunk_case(910 + trial, lens, Hk, Hv, 128, 128, dtype=torch.bfloat16, gate=gate,
                                g_range=(lo, 0.0), h0_std=0.1 if h0 else None)
    o, sf = run_gpu(case, flags=flags)
    ro, rs = oracle_ref(case)
    check_out(o.cpu(), ro, f"o (trial {trial}: lens {lens}, Hk {Hk}, Hv {Hv}, {gate}, flags {flags})")
    check_state(sf.cpu(), rs, f"final state (trial {trial})")
