"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol include/gdr.h declares, sizes its workspace, and rejects bad
arguments before touching the device (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import gated_delta_rule_37_gb300 as gdr
from gated_delta_rule_37_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdr.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "gdr.h")).read()
    return sorted(set(re.findall(r"GDR_API\s+[\w\s\*]*?\b(gdr_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(gdr.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", gdr.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gdr_\w+)", out))
    assert set(_declared()) == exported


def test_version_and_clean_error(lib):
    assert lib.gdr_version() == 100


def test_workspace_size(lib):
    n1 = gdr.chunk_workspace_size(4, 6113, 16, 16, 128, 128, gate_kind=0, dtype=0)
    n2 = gdr.chunk_workspace_size(4, 6113, 16, 16, 128, 128, gate_kind=0, dtype=0, flags=gdr.GDR_QK_L2NORM)
    assert n1 > 0 and n2 > n1
    assert n1 % 256 == 0
    # capacity bound: ceil(T/64) + N chunks, so more sequences never shrink it
    assert gdr.chunk_workspace_size(8, 6113, 16, 16, 128, 128, gate_kind=0, dtype=0) >= n1


def test_workspace_size_chunk_scan(lib):
    """GDR_CHUNK_SCAN adds, per segment and value head, a K x K transition and
    a V x K offset (fp32) on the tensor-core path, at least one segment per
    sequence; other shapes ignore the flag."""
    S = gdr.GDR_CHUNK_SCAN
    for N, T, Hv in [(1, 32768, 4), (4, 6113, 16), (3, 100, 1)]:
        n0 = gdr.chunk_workspace_size(N, T, Hv, Hv, 128, 128, gate_kind=0, dtype=0)
        n1 = gdr.chunk_workspace_size(N, T, Hv, Hv, 128, 128, gate_kind=0, dtype=0, flags=S)
        assert n1 % 256 == 0
        assert n1 - n0 >= 2 * (N + 1) * Hv * 128 * 128 * 4
        # at most one segment per chunk of the capacity ceil(T / 64) + N, plus N
        segs_max = -(-T // 64) + 2 * N
        assert n1 - n0 <= 2 * segs_max * Hv * 128 * 128 * 4 + 16 * segs_max + 4 * (N + 1) + 3 * 256
    assert gdr.chunk_workspace_size(1, 4096, 1, 1, 64, 64, gate_kind=0, dtype=0, flags=S) == \
        gdr.chunk_workspace_size(1, 4096, 1, 1, 64, 64, gate_kind=0, dtype=0)
    assert gdr.chunk_workspace_size(1, 4096, 1, 1, 128, 128, gate_kind=0, dtype=1, flags=S) == \
        gdr.chunk_workspace_size(1, 4096, 1, 1, 128, 128, gate_kind=0, dtype=1)


@pytest.mark.parametrize("args,code", [
    (dict(Hk=3, Hv=4), 1),               # Hv not a multiple of Hk
    (dict(K=96, V=96), 2),               # unsupported head dim
    (dict(K=128, V=64), 2),              # K != V
    (dict(dtype=7), 2),                  # bad dtype
    (dict(gate_kind=5), 1),
])
def test_workspace_size_rejects(lib, args, code):
    base = dict(N=1, T=64, Hk=2, Hv=4, K=128, V=128, gate_kind=0, dtype=0)
    base.update(args)
    out = ctypes.c_size_t(0)
    rc = lib.gdr_chunk_workspace_size(base["N"], base["T"], base["Hk"], base["Hv"], base["K"], base["V"],
                                      base["gate_kind"], base["dtype"], 0, ctypes.byref(out))
    assert rc == code
    assert lib.gdr_last_error().decode()


def _chunk_call(lib, **kw):
    P = ctypes.c_void_p
    a = dict(q=P(16), k=P(32), v=P(48), g=P(64), gk=None, beta=P(80), h0=None, cu=P(96), N=1, T=64,
             Hk=2, Hv=4, K=128, V=128, scale=0.1, dtype=0, flags=0, o=P(112), hT=None,
             ws=P(256), ws_bytes=1 << 40, stream=None)
    a.update(kw)
    return lib.gdr_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["gk"], a["beta"], a["h0"], a["cu"], a["N"],
                             a["T"], a["Hk"], a["Hv"], a["K"], a["V"], a["scale"], a["dtype"], a["flags"],
                             a["o"], a["hT"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(g=None), 1),                                  # neither g nor gk
    (dict(gk=ctypes.c_void_p(128)), 1),                 # both g and gk
    (dict(q=None), 1),                                  # null input
    (dict(q=ctypes.c_void_p(17)), 1),                   # misaligned
    (dict(ws=ctypes.c_void_p(272)), 1),                 # workspace not 256-aligned
    (dict(ws_bytes=1024), 3),                           # workspace too small
    (dict(flags=0x4), 1),                               # commit is not a prefill flag
    (dict(flags=0x40), 1),                              # unknown flag
    (dict(K=64, V=128), 2),
    (dict(N=0, T=64), 1),                               # tokens without sequences
])
def test_chunk_fwd_rejects_before_launch(lib, kw, code):
    assert _chunk_call(lib, **kw) == code
    assert lib.gdr_last_error().decode()


def test_chunk_scan_rejects_segment_capacity_above_grid_limit(lib):
    """GDR_CHUNK_SCAN launches one CTA row per segment of capacity; more than
    65535 of them is rejected before anything runs."""
    N = 65535
    rc = _chunk_call(lib, N=N, T=64 * N, Hk=1, Hv=1, flags=gdr.GDR_CHUNK_SCAN)
    assert rc == 2
    assert "segment capacity" in lib.gdr_last_error().decode()


def test_chunk_fwd_empty_is_ok_without_device(lib):
    assert _chunk_call(lib, N=0, T=0) == 0


def _rec_call(lib, **kw):
    P = ctypes.c_void_p
    a = dict(q=P(16), k=P(32), v=P(48), g=P(64), beta=P(80), pool=P(96), pool_dtype=1, num_slots=8,
             idx=P(112), cu=P(128), N=4, T=4, Hk=2, Hv=4, K=128, V=128, scale=0.1, dtype=0, flags=4,
             o=P(144), ibuf=None, steps=0, stream=None)
    a.update(kw)
    return lib.gdr_recurrent_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["pool"], a["pool_dtype"],
                                 a["num_slots"], a["idx"], a["cu"], a["N"], a["T"], a["Hk"], a["Hv"], a["K"],
                                 a["V"], a["scale"], a["dtype"], a["flags"], a["o"], a["ibuf"], a["steps"],
                                 a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(pool_dtype=3), 2),
    (dict(num_slots=0), 1),
    (dict(ibuf=ctypes.c_void_p(160), steps=0), 1),
    (dict(idx=None), 1),
    (dict(pool=ctypes.c_void_p(100)), 1),               # misaligned pool
    (dict(flags=0x2), 1),                               # neg-eigval is a gating flag
    (dict(Hk=3), 1),
])
def test_recurrent_fwd_rejects_before_launch(lib, kw, code):
    assert _rec_call(lib, **kw) == code


def test_recurrent_fwd_empty_is_ok(lib):
    assert _rec_call(lib, N=0, T=0) == 0


def _gated_call(lib, **kw):
    P = ctypes.c_void_p
    a = dict(q=P(16), k=P(32), v=P(48), a=P(64), b=P(80), A_log=P(96), dt_bias=P(112), pool=P(128), pool_dtype=1,
             num_slots=8, idx=P(144), cu=P(160), N=4, T=4, Hk=2, Hv=4, K=128, V=128, scale=0.1, dtype=0, flags=4,
             o=P(176), ibuf=None, steps=0, stream=None)
    a.update(kw)
    return lib.gdr_recurrent_fwd_gated(a["q"], a["k"], a["v"], a["a"], a["b"], a["A_log"], a["dt_bias"], a["pool"],
                                       a["pool_dtype"], a["num_slots"], a["idx"], a["cu"], a["N"], a["T"], a["Hk"],
                                       a["Hv"], a["K"], a["V"], a["scale"], a["dtype"], a["flags"], a["o"], a["ibuf"],
                                       a["steps"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(flags=0x10), 1),                              # per-channel gates are not formed from raw projections
    (dict(A_log=None), 1),
    (dict(b=None), 1),
    (dict(pool_dtype=3), 2),
    (dict(K=96, V=96), 2),
])
def test_recurrent_fwd_gated_rejects_before_launch(lib, kw, code):
    assert _gated_call(lib, **kw) == code


def test_recurrent_fwd_gated_empty_is_ok(lib):
    assert _gated_call(lib, N=0, T=0) == 0


def test_recurrent_fwd_norm_rejects_before_launch(lib):
    P = ctypes.c_void_p
    base = [P(16), P(32), P(48), P(64), P(80), P(96), 1, 8, P(112), P(128), 4, 4, 2, 4, 128, 128, 0.1, 0, 4]
    tail = [P(176), None, 0, None]
    assert lib.gdr_recurrent_fwd_norm(*base, None, P(144), 1e-6, *tail) == 1        # no weight
    assert lib.gdr_recurrent_fwd_norm(*base, P(160), None, 1e-6, *tail) == 1        # no gate
    assert lib.gdr_recurrent_fwd_norm(*base, P(160), P(144), -1.0, *tail) == 1      # negative eps
    assert lib.gdr_recurrent_fwd_norm(*base[:10], 0, 0, *base[12:], P(160), P(144), 1e-6, *tail) == 0  # empty


def test_gating_rejects(lib):
    P = ctypes.c_void_p
    assert lib.gdr_gating_fwd(P(16), P(32), P(48), P(64), 4, 0, 0, 0, P(80), P(96), None) == 1
    assert lib.gdr_gating_fwd(P(16), P(32), P(48), P(64), 4, 2, 9, 0, P(80), P(96), None) == 2
    assert lib.gdr_gating_fwd(P(16), P(32), P(48), P(64), 0, 2, 0, 0, P(80), P(96), None) == 0


def test_noalloc_rejects_oversized_problem_before_touching_the_device(lib):
    P = ctypes.c_void_p
    # 1M tokens x 32 heads needs far more scratch than the library's static array
    rc = lib.gdr_chunk_fwd_noalloc(P(16), P(32), P(48), P(64), None, P(80), None, P(96), 1, 1 << 20,
                                   16, 32, 128, 128, 0.1, 0, 0, P(112), None, None)
    assert rc == 3
    assert "static scratch" in lib.gdr_last_error().decode()


def test_noalloc_limit_matches_header_and_rejects_exactly_above_it(lib):
    """The binding's NOALLOC_WORKSPACE_BYTES is the header's
    GDR_NOALLOC_WORKSPACE_BYTES, and the size check rejects a problem exactly
    when its workspace exceeds it (host-side: the call that fits goes on and
    fails later only for want of a device here)."""
    src = open(os.path.join(ROOT, "include", "gdr.h")).read()
    m = re.search(r"#define\s+GDR_NOALLOC_WORKSPACE_BYTES\s+\((\d+)ull\s*<<\s*(\d+)\)", src)
    assert m, "GDR_NOALLOC_WORKSPACE_BYTES not found in gdr.h"
    assert int(m.group(1)) << int(m.group(2)) == gdr.NOALLOC_WORKSPACE_BYTES

    def need(T):
        return gdr.chunk_workspace_size(1, T, 4, 4, 128, 128, gate_kind=0, dtype=0)
    T = 64
    while need(T + 64) <= gdr.NOALLOC_WORKSPACE_BYTES:
        T += 64
    P = ctypes.c_void_p

    def call(T):
        return lib.gdr_chunk_fwd_noalloc(P(16), P(32), P(48), P(64), None, P(80), None, P(96), 1, T,
                                         4, 4, 128, 128, 0.1, 0, 0, P(112), None, None)
    assert need(T) <= gdr.NOALLOC_WORKSPACE_BYTES < need(T + 64)
    assert call(T + 64) == 3 and "static scratch" in lib.gdr_last_error().decode()
    import torch
    if not torch.cuda.is_available():
        assert call(T) != 3
