"""Oracle for the gated delta rule forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is a plain, slow, fp64 CPU statement
of what the GPU path computes and shares no code with it (the GPU library lives
in ``gated_delta_rule_37_gb300/csrc`` and is never imported from here).

Contents
  * ``tokenwise``   -- the recurrence itself, token by token (C, fp64).
  * ``chunked``     -- the chunked WY form of the same recurrence (C, fp64),
                       the independent second statement.
  * ``pool``        -- slot-indexed decode / multi-step verify (C, fp64).
  * ``bruteforce``  -- explicit K x K transition matrices (numpy, tiny sizes).
  * ``gating``, ``l2norm`` -- the optional input preparation (C, fp64).
  * ``gated_rmsnorm`` -- the optional output epilogue of decode (numpy, fp64):
                       rmsnorm(o) * w * sigmoid(gate) over each value row
                       (tokenspeed PR #834, fused gated-norm epilogue commit).

Recurrence per value-head (state S in R^{V x K}, V-major):
  S~ = exp(g_t) S_{t-1};  n_t = beta_t (v_t - S~ k_t);  S_t = S~ + n_t k_t^T;
  o_t = scale * S_t q_t  (post-update read).
Sources: FlashQLA PR #1 (fused recurrent GDN decode + DFlash verify), core
decode-kernel and paged-verify commits; attention-gym PR #344 (inter-chunk
state h of the chunked form, 64-token chunks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

# negative-control switches (must match the C source)
READ_PRE_UPDATE = 1
HEAD_MOD = 2
TRANSPOSED = 4


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_tokenwise.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, D, I, P, P, I]
        lib.oracle_tokenwise.restype = I
        lib.oracle_chunked.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, D, I, P, P, I]
        lib.oracle_chunked.restype = I
        lib.oracle_pool.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, D, I, P, P, I, I]
        lib.oracle_pool.restype = I
        lib.oracle_gating.argtypes = [P, P, P, P, ctypes.c_int64, I, I, P, P]
        lib.oracle_gating.restype = None
        lib.oracle_l2norm.argtypes = [P, ctypes.c_int64, I, D, P]
        lib.oracle_l2norm.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _f64(x):
    """Exact fp64 upcast of an input (torch tensor or numpy array)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cu64(cu):
    if hasattr(cu, "detach"):
        cu = cu.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int64))


def tokenwise(q, k, v, beta, cu_seqlens, *, g=None, gk=None, initial_state=None, scale,
              variant: int = 0, nthreads: int = 0):
    """Tokenwise recurrence.  Shapes: q,k [T,Hk,K]; v [T,Hv,V]; g [T,Hv] or gk
    [T,Hv,K]; beta [T,Hv]; initial_state [N,Hv,V,K] or None.
    Returns (o [T,Hv,V], final_state [N,Hv,V,K]) in fp64."""
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    g, gk, s0 = _f64(g), _f64(gk), _f64(initial_state)
    cu = _cu64(cu_seqlens)
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = len(cu) - 1
    o = np.zeros((T, Hv, V))
    sf = np.zeros((N, Hv, V, K))
    rc = _load().oracle_tokenwise(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gk), _ptr(beta),
                                  _ptr(s0), _ptr(cu), N, Hk, Hv, K, V, float(scale), int(variant),
                                  _ptr(o), _ptr(sf), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_tokenwise rejected its arguments")
    return o, sf


def chunked(q, k, v, beta, cu_seqlens, *, g=None, gk=None, initial_state=None, scale,
            chunk: int = 64, nthreads: int = 0):
    """Chunked WY form (independent second statement).  Same contract as
    :func:`tokenwise`."""
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    g, gk, s0 = _f64(g), _f64(gk), _f64(initial_state)
    cu = _cu64(cu_seqlens)
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = len(cu) - 1
    o = np.zeros((T, Hv, V))
    sf = np.zeros((N, Hv, V, K))
    rc = _load().oracle_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gk), _ptr(beta),
                                _ptr(s0), _ptr(cu), N, Hk, Hv, K, V, float(scale), int(chunk),
                                _ptr(o), _ptr(sf), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_chunked rejected its arguments")
    return o, sf


def pool(q, k, v, g, beta, pool_state, state_indices, cu_seqlens, *, scale, commit: bool,
         steps: int = 0, ibuf_rows: int = 0, o_init=None, ibuf_init=None, nthreads: int = 0):
    """Slot-indexed decode / verify.  ``g`` is the scalar log-decay [T, Hv] or
    the per-key-channel one [T, Hv, K].  Returns (o, pool_out, ibuf) in fp64,
    where rows that the method leaves untouched keep ``o_init`` / ``ibuf_init``
    (NaN when not given) and the input pool content."""
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    gk = g if g.ndim == 3 else None
    if gk is not None:
        g = np.zeros(g.shape[:2])
    pin = _f64(pool_state)
    pout = pin.copy()
    idx = state_indices
    if hasattr(idx, "detach"):
        idx = idx.detach().cpu().numpy()
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    cu = _cu64(cu_seqlens)
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = len(cu) - 1
    num_slots = pin.shape[0]
    o = np.full((T, Hv, V), np.nan) if o_init is None else _f64(o_init).copy()
    ib = None
    if steps > 0:
        ib = (np.full((ibuf_rows, steps, Hv, V, K), np.nan) if ibuf_init is None
              else _f64(ibuf_init).copy())
    rc = _load().oracle_pool(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gk), _ptr(beta), _ptr(pin), _ptr(pout),
                             _ptr(idx), _ptr(cu), N, num_slots, Hk, Hv, K, V, float(scale),
                             int(bool(commit)), _ptr(o), _ptr(ib), int(steps), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_pool rejected its arguments")
    return o, pout, ib


def gating(a, dt_bias, A_log, b, *, neg_eigval: bool = False):
    """g = -exp(A_log) softplus(a + dt_bias); beta = sigmoid(b) (x2 with neg_eigval)."""
    a, dt_bias, A_log, b = _f64(a), _f64(dt_bias), _f64(A_log), _f64(b)
    T, Hv = a.shape
    g = np.zeros((T, Hv))
    beta = np.zeros((T, Hv))
    _load().oracle_gating(_ptr(a), _ptr(dt_bias), _ptr(A_log), _ptr(b), T, Hv, int(neg_eigval),
                          _ptr(g), _ptr(beta))
    return g, beta


def l2norm(x, eps: float = 1e-6):
    """Row-wise x / sqrt(sum x^2 + eps) over the last axis."""
    x = _f64(x)
    D = x.shape[-1]
    y = np.zeros_like(x)
    _load().oracle_l2norm(_ptr(x), x.size // D, D, float(eps), _ptr(y))
    return y


def gated_rmsnorm(o, weight, gate, eps: float):
    """The decode output epilogue: each value row x = o[t, h, :] becomes
    x / sqrt(mean(x^2) + eps) * weight * sigmoid(gate[t, h, :]).  o, gate
    [T, Hv, V]; weight [V]."""
    x = _f64(o)
    w = _f64(weight)
    z = _f64(gate)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w * (1.0 / (1.0 + np.exp(-z)))


def bruteforce(q, k, v, beta, *, g=None, gk=None, initial_state=None, scale):
    """One sequence, tiny sizes: explicit transitions
    P_t = D_t (I - beta_t k_t k_t^T) with D_t = exp(g_t) I (or diag(exp(gk_t))),
    S_t = S_{t-1} P_t + beta_t v_t k_t^T, o_t = scale S_t q_t.
    Also returns the unrolled closed form of the final state,
    S_T = S_0 prod_t P_t + sum_t beta_t v_t k_t^T prod_{s>t} P_s.
    Shapes: q,k [T,K]; v [T,V]; g [T] or gk [T,K]; beta [T]; state [V,K]."""
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    T, K = q.shape
    V = v.shape[1]
    S0 = np.zeros((V, K)) if initial_state is None else _f64(initial_state)
    Ps = []
    for t in range(T):
        d = np.exp(_f64(gk)[t]) if gk is not None else np.full(K, np.exp(_f64(g)[t]))
        Ps.append(np.diag(d) @ (np.eye(K) - beta[t] * np.outer(k[t], k[t])))
    S = S0.copy()
    o = np.zeros((T, V))
    for t in range(T):
        S = S @ Ps[t] + beta[t] * np.outer(v[t], k[t])
        o[t] = scale * S @ q[t]
    prod_all = np.eye(K)
    for t in range(T):
        prod_all = prod_all @ Ps[t]
    closed = S0 @ prod_all
    for t in range(T):
        tail = np.eye(K)
        for s in range(t + 1, T):
            tail = tail @ Ps[s]
        closed = closed + beta[t] * np.outer(v[t], k[t]) @ tail
    return o, S, closed
