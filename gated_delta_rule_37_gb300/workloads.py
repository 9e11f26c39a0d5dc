"""Seeded synthetic inputs for the gated delta rule forward pass.

This module only draws random numbers and shapes them into the layouts the
library takes; it holds none of the method's arithmetic and imports neither the
GPU library nor the oracle, so both sides can be fed the same bits.

Layouts (token-major, packed variable-length, batch folded into tokens):
  q, k      [T, Hk, K]          v        [T, Hv, V]
  g         [T, Hv]   fp32      gk       [T, Hv, K] fp32
  beta      [T, Hv]             states   [N, Hv, V, K] fp32 (V-major)
  cu_seqlens [N+1] int32        pool     [num_slots, Hv, V, K]
  state_indices [N] int32 (-1 = padding)
  ibuf      [rows, steps, Hv, V, K] (pool dtype)

Value recipe (shared by every workload): q, k ~ N(0, 1) per element, then each
head row scaled to unit l2 norm in fp32 and rounded to the input dtype;
v ~ N(0, 1); beta = sigmoid(N(0, 1)); gates uniform in the stated range.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import math

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    # input shaping only: rows of N(0,1) draws rescaled to unit length
    return x / x.pow(2).sum(-1, keepdim=True).sqrt()


def _uniform(gen, shape, lo, hi):
    return torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo


@dataclass
class ChunkCase:
    """Inputs of one chunked-prefill call (CPU tensors)."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor
    scale: float
    g: torch.Tensor | None = None
    gk: torch.Tensor | None = None
    initial_state: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def N(self):
        return self.cu_seqlens.numel() - 1

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def dims(self):
        return dict(Hk=self.q.shape[1], Hv=self.v.shape[1], K=self.q.shape[2], V=self.v.shape[2])


def chunk_case(seed: int, lens, Hk: int, Hv: int, K: int, V: int, *, dtype=torch.bfloat16,
               gate: str = "g", g_range=(-0.05, 0.0), h0_std: float | None = None,
               scale: float | None = None, name: str = "chunk") -> ChunkCase:
    gen = _gen(seed)
    lens = [int(x) for x in lens]
    T = sum(lens)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(lens, dtype=torch.int32).cumsum(0)
    q = _unit_rows(torch.randn(T, Hk, K, generator=gen)).to(dtype)
    k = _unit_rows(torch.randn(T, Hk, K, generator=gen)).to(dtype)
    v = torch.randn(T, Hv, V, generator=gen).to(dtype)
    beta = torch.sigmoid(torch.randn(T, Hv, generator=gen)).to(dtype)
    g = gk = None
    if gate == "g":
        g = _uniform(gen, (T, Hv), *g_range)
    elif gate == "gk":
        gk = _uniform(gen, (T, Hv, K), *g_range)
    else:
        raise ValueError(gate)
    h0 = None
    if h0_std is not None:
        h0 = torch.randn(len(lens), Hv, V, K, generator=gen) * h0_std
    if scale is None:
        scale = K ** -0.5
    return ChunkCase(name=name, q=q, k=k, v=v, beta=beta, cu_seqlens=cu, scale=float(scale),
                     g=g, gk=gk, initial_state=h0, meta=dict(lens=lens, seed=seed))


@dataclass
class PoolCase:
    """Inputs of one slot-indexed decode / verify call (CPU tensors)."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    pool: torch.Tensor
    state_indices: torch.Tensor
    cu_seqlens: torch.Tensor
    scale: float
    commit: bool
    steps: int = 0
    ibuf_rows: int = 0
    meta: dict = field(default_factory=dict)
    raw: dict | None = None  # raw gate projections a, b [T, Hv], A_log, dt_bias [Hv]
    norm: dict | None = None  # output epilogue: weight [V] fp32, gate [T, Hv, V], eps

    @property
    def N(self):
        return self.cu_seqlens.numel() - 1

    @property
    def T(self):
        return self.q.shape[0]


def pool_case(seed: int, lens, Hk: int, Hv: int, K: int, V: int, num_slots: int, *,
              dtype=torch.bfloat16, pool_dtype=torch.float32, g_range=(-1.0, 0.0),
              pad_count: int = 0, commit: bool = True, steps: int = 0, ibuf_rows: int = 0,
              pool_std: float = 0.1, scale: float | None = None, channel_gate: bool = False,
              name: str = "pool") -> PoolCase:
    """``channel_gate``: g is a per-key-channel log-decay [T, Hv, K] instead of
    the scalar [T, Hv]."""
    gen = _gen(seed)
    lens = [int(x) for x in lens]
    N = len(lens)
    T = sum(lens)
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(lens, dtype=torch.int32).cumsum(0)
    q = _unit_rows(torch.randn(T, Hk, K, generator=gen)).to(dtype)
    k = _unit_rows(torch.randn(T, Hk, K, generator=gen)).to(dtype)
    v = torch.randn(T, Hv, V, generator=gen).to(dtype)
    beta = torch.sigmoid(torch.randn(T, Hv, generator=gen)).to(dtype)
    g = _uniform(gen, (T, Hv, K) if channel_gate else (T, Hv), *g_range)
    pool = (torch.randn(num_slots, Hv, V, K, generator=gen) * pool_std).to(pool_dtype)
    idx = torch.randperm(num_slots, generator=gen)[:N].to(torch.int32)
    if pad_count:
        pad_at = torch.randperm(N, generator=gen)[:pad_count]
        idx[pad_at] = -1
    if scale is None:
        scale = K ** -0.5
    return PoolCase(name=name, q=q, k=k, v=v, g=g, beta=beta, pool=pool, state_indices=idx,
                    cu_seqlens=cu, scale=float(scale), commit=commit, steps=steps,
                    ibuf_rows=ibuf_rows, meta=dict(lens=lens, seed=seed))


# ----------------------------------------------------------------------------
# The five reference workloads (sizes of the pages' workloads: GVA Hk16/Hv32,
# K = V = 128, T = 12 verify, 64-token chunks).
# ----------------------------------------------------------------------------

def tiny_fp32_prefill() -> ChunkCase:
    """1 sequence, T=128 (2 chunks), 2 heads, K=V=64, fp32, g ~ U[-0.05,0]."""
    return chunk_case(0, [128], 2, 2, 64, 64, dtype=torch.float32, gate="g",
                      g_range=(-0.05, 0.0), scale=1.0 / 8.0, name="tiny_fp32_T128_H2_D64")


def varlen_bf16_prefill() -> ChunkCase:
    """4 sequences {65,1000,2048,3000}, H=16, K=V=128, bf16, g ~ U[-2,0], h0 ~ N(0,0.1)."""
    return chunk_case(1, [65, 1000, 2048, 3000], 16, 16, 128, 128, dtype=torch.bfloat16,
                      gate="g", g_range=(-2.0, 0.0), h0_std=0.1,
                      name="varlen_bf16_N4_T6113_H16_D128")


def kda_long_prefill(T: int = 32768) -> ChunkCase:
    """1 sequence T=32768, Hk=16, Hv=32, K=V=128, bf16, per-channel gk ~ U[-0.1,0]."""
    return chunk_case(2, [T], 16, 32, 128, 128, dtype=torch.bfloat16, gate="gk",
                      g_range=(-0.1, 0.0), name=f"kda_bf16_T{T}_Hk16_Hv32_D128")


def long_few_heads_prefill(T: int = 32768, Hv: int = 4) -> ChunkCase:
    """1 sequence T=32768 with few heads (Hk = Hv = 4, one tensor-parallel
    eighth of a 32-head layer), K=V=128, bf16, g ~ U[-0.1,0] (the long-context
    decay range), h0 ~ N(0,0.1): the shape the chunk-parallel scan is for."""
    return chunk_case(8, [T], Hv, Hv, 128, 128, dtype=torch.bfloat16, gate="g",
                      g_range=(-0.1, 0.0), h0_std=0.1, name=f"long_gdn_bf16_T{T}_H{Hv}_D128")


def decode_fp32_pool() -> PoolCase:
    """256 single-token sequences, Hk=16, Hv=32, K=V=128, fp32 pool of 513 slots,
    26 of 256 indices padding, committed in place."""
    return pool_case(3, [1] * 256, 16, 32, 128, 128, 513, pool_dtype=torch.float32,
                     g_range=(-1.0, 0.0), pad_count=26, commit=True,
                     name="decode_B256_Hk16_Hv32_D128_fp32pool")


def decode_kda_fp32_pool() -> PoolCase:
    """The decode workload with per-key-channel gates: 256 single-token
    sequences, Hk=16, Hv=32, K=V=128, gk ~ U[-1,0] [T, Hv, K], fp32 pool of 513
    slots, 26 padding indices, committed in place."""
    return pool_case(5, [1] * 256, 16, 32, 128, 128, 513, pool_dtype=torch.float32,
                     g_range=(-1.0, 0.0), pad_count=26, commit=True, channel_gate=True,
                     name="decode_kda_B256_Hk16_Hv32_D128_fp32pool")


def verify_bf16_pool(pad_count: int = 0) -> PoolCase:
    """64 sequences with accepted lengths U{1..12}, bf16 pool of 65 slots,
    per-token states into a [65, 12, Hv, V, K] bf16 buffer, no commit."""
    gen = _gen(4)
    lens = torch.randint(1, 13, (64,), generator=gen).tolist()
    return pool_case(4, lens, 16, 32, 128, 128, 65, pool_dtype=torch.bfloat16,
                     g_range=(-1.0, 0.0), pad_count=pad_count, commit=False, steps=12,
                     ibuf_rows=65, name="verify_B64_T1to12_Hk16_Hv32_D128_bf16pool")


def raw_gates(seed: int, T: int, Hv: int, dtype=torch.bfloat16) -> dict:
    """Raw gate projections for the in-kernel gating path: a, b ~ N(0, 1) in
    the input dtype; A_log = log U[1, 16]; dt_bias = log(expm1(dt)) with
    log dt ~ U[log 1e-3, log 1e-1] (a Mamba-style initialisation; the pages do
    not state one), both fp32 [Hv]."""
    gen = _gen(seed)
    a = torch.randn(T, Hv, generator=gen).to(dtype)
    b = torch.randn(T, Hv, generator=gen).to(dtype)
    A_log = torch.log(_uniform(gen, (Hv,), 1.0, 16.0))
    dt = torch.exp(_uniform(gen, (Hv,), math.log(1e-3), math.log(1e-1)))
    dt_bias = torch.log(torch.expm1(dt))
    return dict(a=a, b=b, A_log=A_log.float(), dt_bias=dt_bias.float())


def verify_bf16_pool_raw_gates() -> PoolCase:
    """The verify workload with its gates given as raw projections (the
    in-kernel gating path) in ``raw``; the case's own g and beta are not used
    by that path."""
    case = verify_bf16_pool()
    case.raw = raw_gates(6, case.T, case.v.shape[1])
    case.name = "verify_gated_B64_T1to12_Hk16_Hv32_D128_bf16pool"
    return case


def output_norm(seed: int, T: int, Hv: int, V: int, dtype=torch.bfloat16, eps: float = 1e-6) -> dict:
    """Inputs of the gated RMSNorm output epilogue: weight ~ U[0.5, 1.5] fp32
    [V], gate ~ N(0, 1) [T, Hv, V] in the input dtype, eps 1e-6 (our choice;
    the pages do not state the model's value)."""
    gen = _gen(seed)
    return dict(weight=_uniform(gen, (V,), 0.5, 1.5).float(), gate=torch.randn(T, Hv, V, generator=gen).to(dtype),
                eps=eps)


def decode_fp32_pool_norm() -> PoolCase:
    """The decode workload with the gated RMSNorm output epilogue fused."""
    case = decode_fp32_pool()
    case.norm = output_norm(7, case.T, case.v.shape[1], case.v.shape[2])
    case.name = "decode_norm_B256_Hk16_Hv32_D128_fp32pool"
    return case
