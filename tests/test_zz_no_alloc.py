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
import os
import subprocess
import sys

import numpy as np
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


def _largest_tokens_that_fit(N, Hk, Hv, gate_kind):
    """(T, need(T), need(T + 64)): the largest multiple of 64 tokens whose
    workspace fits the no-alloc scratch, with its size and the next one's."""
    def need(T):
        return gdr.chunk_workspace_size(N, T, Hk, Hv, 128, 128, gate_kind=gate_kind, dtype=gdr.GDR_BF16)
    lo, hi = 64, 64
    while need(hi) <= gdr.NOALLOC_WORKSPACE_BYTES:
        lo, hi = hi, 2 * hi
    while hi - lo > 64:
        mid = (lo + hi) // 2 // 64 * 64
        if need(mid) <= gdr.NOALLOC_WORKSPACE_BYTES:
            lo = mid
        else:
            hi = mid
    return lo, need(lo), need(lo + 64)


def test_noalloc_runs_at_its_limit_and_rejects_just_above_it():
    """The largest problem that fits the scratch runs (and matches the
    workspace entry); 64 more tokens are rejected before anything runs."""
    T, n_fit, n_over = _largest_tokens_that_fit(1, 4, 4, gdr.GDR_GATE_SCALAR)
    assert n_fit <= gdr.NOALLOC_WORKSPACE_BYTES < n_over
    case = workloads.chunk_case(86, [T], 4, 4, 128, 128, gate="g", g_range=(-1.0, 0.0), h0_std=0.1)
    pos, kw = _inputs(case)
    o_ref, s_ref = gdr.chunk_fwd(*pos, scale=case.scale, **kw)
    o, s = torch.empty_like(o_ref), torch.empty_like(s_ref)
    gdr.chunk_fwd_noalloc(*pos, scale=case.scale, o=o, final_state=s, **kw)
    torch.cuda.synchronize()
    assert bits_equal(o, o_ref) and bits_equal(s, s_ref)
    big = workloads.chunk_case(87, [T + 64], 4, 4, 128, 128, gate="g", g_range=(-1.0, 0.0))
    pos, kw = _inputs(big)
    ob = torch.full((big.T, 4, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_fwd_noalloc(*pos, scale=big.scale, o=ob, **kw)
    torch.cuda.synchronize()
    assert e.value.code == 3 and "static scratch" in str(e.value)
    assert bool((ob == 7.0).all())


def test_noalloc_calls_allocate_no_device_memory():
    """After a first call (which may load the library's device code), two more
    calls leave the device's free memory exactly where it was."""
    case = workloads.chunk_case(88, [300, 64, 5], 2, 4, 128, 128, gate="gk", g_range=(-0.5, 0.0), h0_std=0.1)
    pos, kw = _inputs(case)
    o = torch.empty(case.T, 4, 128, dtype=torch.bfloat16, device=DEV)
    s = torch.empty(case.N, 4, 128, 128, device=DEV)
    gdr.chunk_fwd_noalloc(*pos, scale=case.scale, o=o, final_state=s, **kw)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        gdr.chunk_fwd_noalloc(*pos, scale=case.scale, o=o, final_state=s, **kw)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"


# A child process with no torch CUDA state: it allocates with the CUDA
# runtime directly, runs the workspace entry and the no-alloc entry, resets
# the device (which tears down its context and with it the scratch array's
# mapping), and runs the no-alloc entry again on fresh buffers.  The scratch
# address must be looked up again in the new context.
_RESET_CHILD = r"""
import ctypes, os, sys
import numpy as np

lib = ctypes.CDLL(sys.argv[1])
try:
    rt = ctypes.CDLL("libcudart.so.13", mode=os.RTLD_NOLOAD)
except OSError:
    rt = ctypes.CDLL("libcudart.so.13")
d = np.load(sys.argv[2])
P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
rt.cudaMalloc.argtypes = [ctypes.POINTER(P), SZ]
rt.cudaMemcpy.argtypes = [P, P, SZ, I]
lib.gdr_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I, I, P, P, P, SZ, P]
lib.gdr_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I, I, P, P, P]
lib.gdr_chunk_workspace_size.argtypes = [I, I64, I, I, I, I, I, I, I, ctypes.POINTER(SZ)]
lib.gdr_last_error.restype = ctypes.c_char_p
N, T, Hk, Hv, D = (int(x) for x in d["dims"])
scale = float(d["scale"])

def chk(rc, what):
    if rc != 0:
        raise SystemExit(f"{what}: status {rc} {lib.gdr_last_error()}")

def upload(a):
    p = P()
    chk(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
    chk(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, 1), "cudaMemcpy H2D")
    return p

def alloc(nbytes):
    p = P()
    chk(rt.cudaMalloc(ctypes.byref(p), nbytes), "cudaMalloc")
    return p

def download(p, like):
    out = np.empty_like(like)
    chk(rt.cudaMemcpy(out.ctypes.data, p, out.nbytes, 2), "cudaMemcpy D2H")
    return out

o_like = np.empty((T, Hv, D), dtype=np.uint16)
s_like = np.empty((N, Hv, D, D), dtype=np.float32)

def buffers():
    ins = [upload(np.ascontiguousarray(d[n])) for n in ("q", "k", "v", "g", "beta", "h0", "cu")]
    return ins, alloc(o_like.nbytes), alloc(s_like.nbytes)

def args(ins):
    q, k, v, g, beta, h0, cu = ins
    return (q, k, v, g, None, beta, h0, cu, N, T, Hk, Hv, D, D, scale, 0, 0)

chk(rt.cudaSetDevice(0), "cudaSetDevice")
ins, o, s = buffers()
need = SZ(0)
chk(lib.gdr_chunk_workspace_size(N, T, Hk, Hv, D, D, 0, 0, 0, ctypes.byref(need)), "workspace size")
ws = alloc(need.value)
chk(lib.gdr_chunk_fwd(*args(ins), o, s, ws, need.value, None), "gdr_chunk_fwd")
o_ref, s_ref = download(o, o_like), download(s, s_like)

def bf16(u):
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

def same(o_got, s_got, what):
    a, b = bf16(o_got), bf16(o_ref)
    e_o = np.linalg.norm(a - b) / np.linalg.norm(b)
    m_o = np.abs(a - b).max()
    e_s = np.linalg.norm(s_got.astype(np.float64) - s_ref) / np.linalg.norm(s_ref)
    if not (e_o <= 5e-3 and m_o <= 3e-2 and e_s <= 1e-4):
        raise SystemExit(f"{what}: o rel-L2 {e_o:.3e} max-abs {m_o:.3e}, state rel-L2 {e_s:.3e}")

chk(lib.gdr_chunk_fwd_noalloc(*args(ins), o, s, None), "gdr_chunk_fwd_noalloc")
same(download(o, o_like), download(s, s_like), "before the reset")
chk(rt.cudaDeviceReset(), "cudaDeviceReset")
chk(rt.cudaSetDevice(0), "cudaSetDevice after the reset")
ins, o, s = buffers()
chk(lib.gdr_chunk_fwd_noalloc(*args(ins), o, s, None), "gdr_chunk_fwd_noalloc after the reset")
chk(rt.cudaDeviceSynchronize(), "synchronize after the reset")
same(download(o, o_like), download(s, s_like), "after the reset")
print("ok")
"""


def test_noalloc_after_device_reset(tmp_path):
    """The no-alloc entry point stays correct after cudaDeviceReset: the
    scratch array's address belongs to the context and is looked up again."""
    case = workloads.chunk_case(89, [130, 64, 7], 2, 4, 128, 128, gate="g", g_range=(-1.0, 0.0), h0_std=0.1)
    f = tmp_path / "inputs.npz"
    np.savez(f, q=case.q.view(torch.int16).numpy(), k=case.k.view(torch.int16).numpy(),
             v=case.v.view(torch.int16).numpy(), beta=case.beta.view(torch.int16).numpy(),
             g=case.g.numpy(), h0=case.initial_state.numpy(), cu=case.cu_seqlens.numpy(),
             dims=np.array([case.N, case.T, 2, 4, 128]), scale=np.array(case.scale))
    r = subprocess.run([sys.executable, "-c", _RESET_CHILD, gdr.LIB_PATH, str(f)], capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, CUDA_VISIBLE_DEVICES=os.environ.get("CUDA_VISIBLE_DEVICES",
                                                                                            "0").split(",")[0]))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
