"""Helpers for the GPU parity tests (comparison metrics, guarded buffers)."""
import numpy as np
import torch

# parity bounds: bf16 outputs rel-L2 <= 5e-3 and max-abs <= 3e-2;
# fp32 states rel-L2 <= 1e-4; fp32 outputs rel-L2 <= 1e-4 (the same bound as
# the fp32 state: fp32 arithmetic with bf16-split tensor-core products keeps
# the relative error near 1e-5, so 1e-4 leaves a 10x margin).
BF16_REL, BF16_ABS = 5e-3, 3e-2
F32_REL = 1e-4

GUARD = 4096  # bytes of redzone on each side of a guarded buffer
PATTERN = 0xA5


def rel_l2(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.linalg.norm((x - y).ravel()) / max(np.linalg.norm(y.ravel()), 1e-300))


def max_abs(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.abs(x - y).max()) if x.size else 0.0


def check_out(got: torch.Tensor, ref, what: str):
    """Compare a GPU output (bf16 or fp32) with an fp64 oracle array."""
    g = got.detach().float().cpu().numpy()
    e = rel_l2(g, ref)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    if got.dtype == torch.bfloat16:
        m = max_abs(g, ref)
        assert e <= BF16_REL and m <= BF16_ABS, f"{what}: rel-L2 {e:.3e} max-abs {m:.3e}"
    else:
        assert e <= F32_REL, f"{what}: rel-L2 {e:.3e}"
    return e


def check_state(got: torch.Tensor, ref, what: str):
    """fp32 states: rel-L2 <= 1e-4.  bf16 states (pools, per-token states):
    rel-L2 <= 5e-3 and max-abs <= 3e-2, the bounds of every bf16 result."""
    g = got.detach().float().cpu().numpy()
    e = rel_l2(g, ref)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    if got.dtype == torch.float32:
        assert e <= F32_REL, f"{what}: rel-L2 {e:.3e} > {F32_REL}"
    else:
        m = max_abs(g, ref)
        assert e <= BF16_REL and m <= BF16_ABS, f"{what}: rel-L2 {e:.3e} max-abs {m:.3e}"
    return e


class Guarded:
    """A device buffer with byte-pattern redzones on both sides."""

    def __init__(self, shape, dtype, device, fill_bytes=None):
        self.shape = tuple(shape)
        self.dtype = dtype
        esz = torch.empty(0, dtype=dtype).element_size()
        self.n = int(np.prod(shape)) if len(shape) else 1
        nbytes = self.n * esz
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        body = self.raw[GUARD:GUARD + nbytes]
        if fill_bytes is not None:
            body.copy_(fill_bytes.reshape(-1).view(torch.uint8).to(device))
        self.view = body.view(dtype).view(self.shape)

    def guards_intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[-GUARD:]
        return bool((head == PATTERN).all().item() and (tail == PATTERN).all().item())


def sentinel_like(shape, dtype):
    """A CPU tensor of a recognisable bit pattern (a quiet NaN) of the dtype."""
    if dtype == torch.bfloat16:
        return torch.full(shape, 0x7FC1, dtype=torch.int16).view(torch.bfloat16)
    return torch.full(shape, 0x7FC00123, dtype=torch.int32).view(torch.float32)


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    a = a.detach().cpu().contiguous()
    b = b.detach().cpu().contiguous()
    return a.shape == b.shape and torch.equal(a.view(torch.uint8), b.view(torch.uint8))
