"""16 x 16 random Hadamard transform before quantization (oracle; test infrastructure only).

The "UE5M3 FP4 Block Scaling ..." blog (section "Что сделали") describes the
randomized Hadamard transform, which spreads outliers before quantization,
and drops it from the UE5M3 recipe; the post on "INT v.s. FP: A Comprehensive
Study of Fine-Grained Low-bit Quantization Formats" (quant_prune_distill
channel page, section "Метод") uses Hadamard rotations to make weights and
activations closer to Gaussian.  Readings fixed here:

* per 16-element block along the blocked dimension, x' = 1/4 * H16 * (s . x),
  H16 the Sylvester Hadamard matrix (H[i, j] = (-1)^popcount(i & j)) and s the
  per-tensor sign vector: s[j] = -1 iff bit j of the 16-bit mask is set;
* computed in float32 by the fast Walsh-Hadamard transform: for h = 1, 2, 4, 8
  every pair (i, i + h) with i & h == 0 becomes (a + b, a - b), each a single
  float32 operation; then every value times 0.25 (exact);
* the quantizer then runs on these float32 values (global amax included).

1/4 * H16 * diag(s) is orthogonal, so two operands transformed with the same
mask along K keep their product.
"""

from __future__ import annotations

import numpy as np


def sign_vector(mask: int) -> np.ndarray:
    return np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)], dtype=np.float32)


def hadamard16() -> np.ndarray:
    """The Sylvester Hadamard matrix H16 (float64, entries +-1)."""
    i = np.arange(16)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 1, -1.0, 1.0)


def rht16(x: np.ndarray, mask: int) -> np.ndarray:
    """Float32 transform of every 16-element block along the last axis."""
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    if shape[-1] % 16:
        raise ValueError("the last dimension must be a multiple of 16")
    v = (x.reshape(-1, 16) * sign_vector(mask)[None, :]).astype(np.float32)
    h = 1
    while h < 16:
        for i in range(16):
            if i & h == 0:
                a = v[:, i].copy()
                b = v[:, i + h].copy()
                v[:, i] = a + b
                v[:, i + h] = a - b
        h *= 2
    return (v * np.float32(0.25)).astype(np.float32).reshape(shape)
