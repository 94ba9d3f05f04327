"""Shared helpers for the GPU parity tests (test infrastructure).

Builds the library once per session, moves tensors between host and device,
and permutes plain row-major scales into the GEMM's tiled scale layout with the
byte-offset formula documented in include/fp4.h.
"""

import numpy as np
import torch

_built = False


def lib():
    global _built
    if not _built:
        from fp4_block_scaled_amax_gb300 import build
        build.build()
        _built = True
    from fp4_block_scaled_amax_gb300 import fp4
    return fp4


def dev(a, dtype=None):
    t = torch.as_tensor(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def f32(x_bf16: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float32 numpy array holding the same values (oracle input)."""
    return x_bf16.float().cpu().numpy()


def mma_offsets(rows: int, nb: int) -> np.ndarray:
    """Byte offset of scale (r, b) in the tiled layout: [rows, nb] int64."""
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(nb, dtype=np.int64)[None, :]
    return ((r >> 7) * (nb >> 2) + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3)


def to_mma(scales: np.ndarray) -> np.ndarray:
    rows, nb = scales.shape
    out = np.zeros(rows * nb, dtype=np.uint8)
    out[mma_offsets(rows, nb).reshape(-1)] = scales.reshape(-1)
    return out


def from_mma(flat: np.ndarray, rows: int, nb: int) -> np.ndarray:
    return np.asarray(flat).reshape(-1)[mma_offsets(rows, nb)]
