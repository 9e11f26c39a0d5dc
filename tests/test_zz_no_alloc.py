"""The no-allocation chunked prefill (gdr_chunk_fwd_noalloc).

It serves callers that cannot allocate device memory -- an engine whose arena
already owns the GPU's memory, a plugin without an allocator, a latency-bound
loop that cannot take cudaMalloc's implicit synchronisation -- by running on a
fixed scratch array inside the library instead of a caller workspace.

This file is collected last on purpose: the scratch array is shared process
state, and the test must pass both alone in a fresh process and after every
other test has run.  It calls the entry point twice in a row, on two problems
of different sizes, through the C ABI, and checks each result against the
workspace entry point gdr_chunk_fwd on the same inputs, with the same
tolerances the other parity tests use.
"""
import pytest
import torch

import gated_delta_rule_37_gb300 as gdr
from gated_delta_rule_37_gb300 import workloads
from tests.gpu_util import bits_equal, check_out, check_state

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(case):
    d = dict(g=case.g.to(DEV) if case.g is not None else None,
             gk=case.gk.to(DEV) if case.gk is not None else None,
             initial_state=case.initial_state.to(DEV) if case.initial_state is not None else None)
    return (case.q.to(DEV), case.k.to(DEV), case.v.to(DEV), case.beta.to(DEV), case.cu_seqlens.to(DEV)), d


def test_noalloc_matches_workspace_entry_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdr.load()
    cases = [workloads.chunk_case(71, [65, 130, 7], 2, 4, 128, 128, gate="g", g_range=(-2.0, 0.0), h0_std=0.1),
             workloads.chunk_case(72, [200, 1, 64], 1, 2, 128, 128, gate="gk", g_range=(-0.5, 0.0))]
    refs = []
    for c in cases:
        pos, kw = _inputs(c)
        o, s = gdr.chunk_fwd(*pos, scale=c.scale, **kw)
        refs.append((o.clone(), s.clone()))
    torch.cuda.synchronize()
    # outputs preallocated by the caller; the two no-alloc calls run back to back
    outs = []
    for c in cases:
        o = torch.full((c.T, c.v.shape[1], c.v.shape[2]), float("nan"), dtype=c.q.dtype, device=DEV)
        s = torch.full((c.N, c.v.shape[1], c.v.shape[2], c.q.shape[2]), float("nan"), device=DEV)
        outs.append((o, s, _inputs(c)))
    for (o, s, (pos, kw)), c in zip(outs, cases):
        gdr.chunk_fwd_noalloc(*pos, scale=c.scale, o=o, final_state=s, **kw)
    torch.cuda.synchronize()
    for (o, s, _), (o_ref, s_ref) in zip(outs, refs):
        check_out(o.cpu(), o_ref.float().cpu().double().numpy(), "o (no-alloc vs workspace entry)")
        check_state(s.cpu(), s_ref.cpu().double().numpy(), "final state (no-alloc vs workspace entry)")


def test_noalloc_rejects_problem_larger_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = workloads.kda_long_prefill(T=8192)
    need = gdr.chunk_workspace_size(c.N, c.T, 16, 32, 128, 128, gate_kind=gdr.GDR_GATE_CHANNEL, dtype=0)
    assert need > gdr.NOALLOC_WORKSPACE_BYTES
    o = torch.empty(c.T, 32, 128, dtype=torch.bfloat16, device=DEV)
    pos, kw = _inputs(c)
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_fwd_noalloc(*pos, scale=c.scale, o=o, **kw)
    assert e.value.code == 3 and "static scratch" in str(e.value)


def test_scan_no_alloc_entry():
    """The scan through the no-allocation entry point equals the workspace entry bit for bit."""
    case = workloads.chunk_case(85, [3000, 200], 1, 2, 128, 128, gate="g", g_range=(-0.2, 0.0), h0_std=0.1)
    need = gdr.chunk_workspace_size(case.N, case.T, 1, 2, 128, 128, gate_kind=0, dtype=0, flags=gdr.GDR_CHUNK_SCAN)
    assert need <= 64 << 20
    q, k, v, beta = (t.to(DEV) for t in (case.q, case.k, case.v, case.beta))
    g, h0, cu = case.g.to(DEV), case.initial_state.to(DEV), case.cu_seqlens.to(DEV)
    o1, s1 = gdr.chunk_fwd(q, k, v, beta, cu, g=g, initial_state=h0, scale=case.scale, flags=gdr.GDR_CHUNK_SCAN)
    o2 = torch.empty_like(o1)
    s2 = torch.empty_like(s1)
    gdr.chunk_fwd_noalloc(q, k, v, beta, cu, g=g, initial_state=h0, scale=case.scale, flags=gdr.GDR_CHUNK_SCAN, o=o2,
                          final_state=s2)
    torch.cuda.synchronize()
    assert bits_equal(o1, o2) and bits_equal(s1, s2)
