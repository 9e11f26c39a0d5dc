"""GB300 (sm_103a) gated delta rule forward: thin Python binding of libgdr.so.

Every step of the computation runs in the library's CUDA kernels; this module
only marshals torch tensors (device memory, streams) into the C ABI declared in
``include/gdr.h`` and raises on a non-zero status.  There is no CPU fallback:
if ``libgdr.so`` is missing or no CUDA device is present, calls fail loudly.

Entry points (same names as the C ABI, without the ``gdr_`` prefix):
  chunk_fwd           chunked prefill          -> o, final_state
  recurrent_fwd       slot-indexed decode / verify (pool in place, ibuf)
  gating_fwd          g, beta from raw projections
  chunk_workspace_size
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr.so")

GDR_BF16, GDR_F32 = 0, 1
GDR_GATE_SCALAR, GDR_GATE_CHANNEL = 0, 1
GDR_QK_L2NORM, GDR_NEG_EIGVAL, GDR_COMMIT, GDR_VALIDATE, GDR_CHANNEL_GATE = 0x1, 0x2, 0x4, 0x8, 0x10
GDR_CHUNK_SCAN = 0x20
CHUNK = 64

STATUS = {0: "GDR_OK", 1: "GDR_ERR_INVALID_ARG", 2: "GDR_ERR_UNSUPPORTED", 3: "GDR_ERR_WORKSPACE",
          4: "GDR_ERR_LAUNCH", 5: "GDR_ERR_DEVICE_TIMEOUT", 6: "GDR_ERR_VALIDATION"}

# every symbol include/gdr.h declares
EXPORTED = ("gdr_chunk_workspace_size", "gdr_chunk_fwd", "gdr_chunk_fwd_noalloc", "gdr_recurrent_fwd",
            "gdr_recurrent_fwd_gated", "gdr_recurrent_fwd_norm", "gdr_gating_fwd",
            "gdr_last_error", "gdr_get_device_status", "gdr_selftest_bounded_wait", "gdr_profile_enable",
            "gdr_profile_read",
            "gdr_version")

_lib = None


class GdrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def load(path: str | None = None):
    """Load libgdr.so (built in-tree by ``build.build()``); raises if missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libgdr.so not found at {p}: build it with gated_delta_rule_37_gb300.build.build()")
    lib = ctypes.CDLL(p)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.gdr_chunk_workspace_size.argtypes = [I, I64, I, I, I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.gdr_chunk_workspace_size.restype = I
    lib.gdr_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I, I, P, P, P, SZ, P]
    lib.gdr_chunk_fwd.restype = I
    lib.gdr_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, I64, I, I, I, I, F, I, I, P, P, P]
    lib.gdr_chunk_fwd_noalloc.restype = I
    lib.gdr_recurrent_fwd.argtypes = [P, P, P, P, P, P, I, I, P, P, I, I64, I, I, I, I, F, I, I, P, P, I, P]
    lib.gdr_recurrent_fwd.restype = I
    lib.gdr_recurrent_fwd_gated.argtypes = [P, P, P, P, P, P, P, P, I, I, P, P, I, I64, I, I, I, I, F, I, I, P, P, I, P]
    lib.gdr_recurrent_fwd_gated.restype = I
    lib.gdr_recurrent_fwd_norm.argtypes = [P, P, P, P, P, P, I, I, P, P, I, I64, I, I, I, I, F, I, I, P, P, F, P, P, I,
                                           P]
    lib.gdr_recurrent_fwd_norm.restype = I
    lib.gdr_gating_fwd.argtypes = [P, P, P, P, I64, I, I, I, P, P, P]
    lib.gdr_gating_fwd.restype = I
    lib.gdr_last_error.argtypes = []
    lib.gdr_last_error.restype = ctypes.c_char_p
    lib.gdr_get_device_status.argtypes = [P, ctypes.POINTER(I)]
    lib.gdr_get_device_status.restype = I
    lib.gdr_selftest_bounded_wait.argtypes = [P]
    lib.gdr_selftest_bounded_wait.restype = I
    lib.gdr_profile_enable.argtypes = [I]
    lib.gdr_profile_enable.restype = I
    lib.gdr_profile_read.argtypes = [I, ctypes.c_char_p, SZ, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.gdr_profile_read.restype = I
    lib.gdr_version.argtypes = []
    lib.gdr_version.restype = I
    if path is None:
        _lib = lib
    return lib


def _check(code: int):
    if code != 0:
        raise GdrError(code, load().gdr_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDR_BF16
    if t.dtype == torch.float32:
        return GDR_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libgdr must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libgdr must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def chunk_workspace_size(N: int, T: int, Hk: int, Hv: int, K: int, V: int, *, gate_kind: int,
                         dtype: int, flags: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(load().gdr_chunk_workspace_size(N, T, Hk, Hv, K, V, gate_kind, dtype, flags, ctypes.byref(out)))
    return out.value


def chunk_fwd(q, k, v, beta, cu_seqlens, *, g=None, gk=None, initial_state=None, scale=None,
              flags: int = 0, o=None, final_state=None, output_final_state: bool = True,
              workspace=None, stream=None):
    """Chunked prefill.  q,k [T,Hk,K]; v [T,Hv,V]; g [T,Hv] fp32 or gk [T,Hv,K]
    fp32; beta [T,Hv]; initial_state [N,Hv,V,K] fp32 or None; cu_seqlens [N+1]
    int32 (device).  Returns (o, final_state or None)."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty(T, Hv, V, dtype=q.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, Hv, V, K, dtype=torch.float32, device=q.device)
    gate_kind = GDR_GATE_SCALAR if g is not None else GDR_GATE_CHANNEL
    need = chunk_workspace_size(N, T, Hk, Hv, K, V, gate_kind=gate_kind, dtype=dt, flags=flags)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(load().gdr_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gk), _ptr(beta),
                                _ptr(initial_state), _ptr(cu_seqlens), N, T, Hk, Hv, K, V,
                                float(scale), dt, flags, _ptr(o), _ptr(final_state),
                                _ptr(workspace), workspace.numel(), _stream(stream)))
    return o, final_state


NOALLOC_WORKSPACE_BYTES = 64 << 20


def chunk_fwd_noalloc(q, k, v, beta, cu_seqlens, *, g=None, gk=None, initial_state=None, scale=None,
                      flags: int = 0, o, final_state=None, stream=None):
    """Chunked prefill through gdr_chunk_fwd_noalloc: no workspace argument and
    no device allocation inside the call (the library's fixed scratch array of
    NOALLOC_WORKSPACE_BYTES is used).  For callers that cannot allocate device
    memory; they pass preallocated outputs ``o`` (and ``final_state``).  Calls
    that overlap on the GPU share the scratch and must be serialised."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    _check(load().gdr_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gk), _ptr(beta),
                                        _ptr(initial_state), _ptr(cu_seqlens), N, T, Hk, Hv, K, V,
                                        float(scale), _dtype_code(q), flags, _ptr(o), _ptr(final_state),
                                        _stream(stream)))
    return o, final_state


def recurrent_fwd(q, k, v, g, beta, state_pool, state_indices, cu_seqlens, *, scale=None,
                  flags: int = GDR_COMMIT, o=None, intermediate_states=None, stream=None):
    """Slot-indexed decode / verify.  ``g`` is the scalar log-decay [T, Hv] or
    the per-key-channel one [T, Hv, K] (sets GDR_CHANNEL_GATE).  The pool is
    updated in place only with GDR_COMMIT; ``intermediate_states`` [rows, steps,
    Hv, V, K] (pool dtype) receives per-token states.  Returns o."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    if g.dim() == 3:
        if tuple(g.shape) != (T, Hv, K):
            raise ValueError("a per-channel gate must be [T, Hv, K]")
        flags |= GDR_CHANNEL_GATE
    if scale is None:
        scale = K ** -0.5
    if o is None:
        o = torch.empty(T, Hv, V, dtype=q.dtype, device=q.device)
    steps = 0
    if intermediate_states is not None:
        if intermediate_states.dim() != 5 or intermediate_states.shape[0] < N:
            raise ValueError("intermediate_states must be [rows >= N, steps, Hv, V, K]")
        if intermediate_states.dtype != state_pool.dtype:
            raise TypeError("intermediate_states must have the pool dtype")
        steps = intermediate_states.shape[1]
    _check(load().gdr_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool),
                                    _dtype_code(state_pool), state_pool.shape[0], _ptr(state_indices),
                                    _ptr(cu_seqlens), N, T, Hk, Hv, K, V, float(scale), _dtype_code(q),
                                    flags, _ptr(o), _ptr(intermediate_states), steps, _stream(stream)))
    return o


def recurrent_fwd_norm(q, k, v, g, beta, state_pool, state_indices, cu_seqlens, norm_weight, norm_gate, *,
                       eps: float = 1e-6, scale=None, flags: int = GDR_COMMIT, o=None, intermediate_states=None,
                       stream=None):
    """recurrent_fwd with the gated RMSNorm output epilogue: each value row x of
    o becomes x / sqrt(mean(x^2) + eps) * norm_weight * sigmoid(norm_gate).
    norm_weight [V] fp32; norm_gate [T, Hv, V] (q's dtype).  Returns o."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    if g.dim() == 3:
        flags |= GDR_CHANNEL_GATE
    if o is None:
        o = torch.empty(T, Hv, V, dtype=q.dtype, device=q.device)
    steps = 0
    if intermediate_states is not None:
        steps = intermediate_states.shape[1]
    if norm_gate.dtype != q.dtype or tuple(norm_gate.shape) != (T, Hv, V):
        raise ValueError("norm_gate must be [T, Hv, V] in q's dtype")
    _check(load().gdr_recurrent_fwd_norm(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool),
                                         _dtype_code(state_pool), state_pool.shape[0], _ptr(state_indices),
                                         _ptr(cu_seqlens), N, T, Hk, Hv, K, V, float(scale), _dtype_code(q), flags,
                                         _ptr(norm_weight), _ptr(norm_gate), float(eps), _ptr(o),
                                         _ptr(intermediate_states), steps, _stream(stream)))
    return o


def recurrent_fwd_gated(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, cu_seqlens, *, scale=None,
                        flags: int = GDR_COMMIT, o=None, intermediate_states=None, stream=None):
    """recurrent_fwd with the gates formed in the kernel from the raw
    projections: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b) (x2
    with GDR_NEG_EIGVAL).  a, b [T, Hv] (q's dtype); A_log, dt_bias [Hv] fp32.
    Returns o."""
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    if o is None:
        o = torch.empty(T, Hv, V, dtype=q.dtype, device=q.device)
    steps = 0
    if intermediate_states is not None:
        if intermediate_states.dim() != 5 or intermediate_states.shape[0] < N:
            raise ValueError("intermediate_states must be [rows >= N, steps, Hv, V, K]")
        if intermediate_states.dtype != state_pool.dtype:
            raise TypeError("intermediate_states must have the pool dtype")
        steps = intermediate_states.shape[1]
    if a.dtype != q.dtype or b.dtype != q.dtype:
        raise TypeError("a and b must have q's dtype")
    _check(load().gdr_recurrent_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                          _ptr(state_pool), _dtype_code(state_pool), state_pool.shape[0],
                                          _ptr(state_indices), _ptr(cu_seqlens), N, T, Hk, Hv, K, V, float(scale),
                                          _dtype_code(q), flags, _ptr(o), _ptr(intermediate_states), steps,
                                          _stream(stream)))
    return o


def gating_fwd(a, dt_bias, A_log, b, *, flags: int = 0, g=None, beta=None, stream=None):
    """g = -exp(A_log) softplus(a + dt_bias) (fp32), beta = sigmoid(b) (x2 with
    GDR_NEG_EIGVAL).  a, b [T, Hv]; dt_bias, A_log [Hv] fp32."""
    T, Hv = a.shape
    if g is None:
        g = torch.empty(T, Hv, dtype=torch.float32, device=a.device)
    if beta is None:
        beta = torch.empty(T, Hv, dtype=a.dtype, device=a.device)
    _check(load().gdr_gating_fwd(_ptr(a), _ptr(dt_bias), _ptr(A_log), _ptr(b), T, Hv, _dtype_code(a),
                                 flags, _ptr(g), _ptr(beta), _stream(stream)))
    return g, beta


def device_status(stream=None) -> int:
    """Synchronise and read/clear the library's device error word."""
    w = ctypes.c_int(0)
    code = load().gdr_get_device_status(_stream(stream), ctypes.byref(w))
    if code not in (0, 5):
        _check(code)
    return w.value


def profile_enable(on: bool = True):
    """Bracket every library kernel launch with CUDA events on its stream."""
    _check(load().gdr_profile_enable(1 if on else 0))


def profile_read(max_kernels: int = 32):
    """{kernel name: (total device ms, launches)} since the previous read."""
    names = ctypes.create_string_buffer(4096)
    ms = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_int * max_kernels)()
    n = ctypes.c_int(0)
    _check(load().gdr_profile_read(max_kernels, names, 4096, ms, cnt, ctypes.byref(n)))
    keys = [k for k in names.value.decode().split(",") if k]
    return {keys[i]: (ms[i], cnt[i]) for i in range(n.value)}
