"""Seeded synthetic inputs shaped like the source pages' workloads.

This module only draws random numbers and rounds them to bf16; it holds none of
the quantization method's arithmetic.  The CUDA path (through the binding) and
the CPU oracle (in the tests) consume the identical bf16 bytes it returns.

Workloads (the pages train on datasets that are not used here; these seeded
tensors stand in for them with the same shapes and value distributions):

1. NVFP4 round trip + GEMM: A [128, 256], B [256, 256], N(0, 1) with 1 % of
   entries multiplied by 50; seed 0.
2. 350M-parameter Llama-like MLP linear: X [8192, 1024] N(0, 1) times a
   per-channel std drawn log-uniform in [0.1, 10]; W [4096, 1024] N(0, 0.02).
3. Llama-2-7B MLP linear, forward and backward: X [16384, 4096] N(0, 1) with
   0.5 % of entries multiplied by 100; W [11008, 4096] N(0, 0.02);
   dY [16384, 11008] Laplace(0, 1e-4).
4. Nemotron-H-8B-like two-linear stack: W1 [21504, 4096], W2 [4096, 21504]
   N(0, 0.02); per step t: X_t [32768, 4096] = 1.02^t N(0, 1) and
   dY_t [32768, 4096] = 1.02^t Laplace(0, 1e-4).
5. Weight-only decode: W_up [18944, 3584], W_down [3584, 18944] N(0, 0.02);
   x [b, K] N(0, 1) for b in {1, 8, 64}.

Every shape can be shrunk with `scale` (rows and columns divided by it, kept
multiples of 256) for parity tests that the oracle finishes in seconds.
"""

from __future__ import annotations

import numpy as np
import torch

SEEDS = {1: 0, 2: 2, 3: 3, 4: 4, 5: 5}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32/float64 numpy array -> contiguous bf16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal(shape, seed, stream, std=1.0, outlier_p=0.0, outlier_mult=1.0, chunk_rows=2048):
    """bf16 N(0, std^2) with a Bernoulli(outlier_p) fraction multiplied by outlier_mult."""
    rng = _rng(seed, stream)
    R, C = shape
    out = torch.empty((R, C), dtype=torch.bfloat16)
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        z = rng.standard_normal((r1 - r0, C), dtype=np.float32)
        if std != 1.0:
            z *= np.float32(std)
        if outlier_p > 0:
            m = rng.random((r1 - r0, C), dtype=np.float32) < outlier_p
            z[m] *= np.float32(outlier_mult)
        out[r0:r1] = to_bf16(z)
    return out


def laplace(shape, seed, stream, scale=1.0, mult=1.0, chunk_rows=2048):
    rng = _rng(seed, stream)
    R, C = shape
    out = torch.empty((R, C), dtype=torch.bfloat16)
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        z = rng.laplace(0.0, scale, (r1 - r0, C)) * mult
        out[r0:r1] = to_bf16(z)
    return out


def _dim(n: int, scale: int) -> int:
    if scale == 1:
        return n
    return max(256, (n // scale) // 256 * 256)


def config1():
    s = SEEDS[1]
    return {"A": normal((128, 256), s, 0, outlier_p=0.01, outlier_mult=50.0),
            "B": normal((256, 256), s, 1, outlier_p=0.01, outlier_mult=50.0)}


def config2(scale: int = 1):
    s = SEEDS[2]
    M, N, K = _dim(8192, scale), _dim(4096, scale), _dim(1024, scale)
    rng = _rng(s, 0)
    sig = (10.0 ** rng.uniform(-1.0, 1.0, K)).astype(np.float32)
    z = _rng(s, 1).standard_normal((M, K), dtype=np.float32) * sig[None, :]
    return {"X": to_bf16(z), "W": normal((N, K), s, 2, std=0.02)}


def config3(scale: int = 1):
    s = SEEDS[3]
    M, N, K = _dim(16384, scale), _dim(11008, scale), _dim(4096, scale)
    return {"X": normal((M, K), s, 0, outlier_p=0.005, outlier_mult=100.0),
            "W": normal((N, K), s, 1, std=0.02),
            "dY": laplace((M, N), s, 2, scale=1e-4)}


def config4_weights(scale: int = 1):
    s = SEEDS[4]
    H, F = _dim(4096, scale), _dim(21504, scale)
    return {"W1": normal((F, H), s, 0, std=0.02), "W2": normal((H, F), s, 1, std=0.02)}


def config4_step(t: int, scale: int = 1):
    s = SEEDS[4]
    M, H = _dim(32768, scale), _dim(4096, scale)
    g = 1.02 ** t
    return {"X": normal((M, H), s, 1000 + 2 * t, std=g),
            "dY": laplace((M, H), s, 1001 + 2 * t, scale=1e-4, mult=g)}


def config4_step_device(t: int, device, scale: int = 1):
    """Config-4 inputs of step t drawn on the device (torch's CUDA Philox
    generator, seeded per step and tensor): X_t = 1.02^t N(0, 1) and
    dY_t = 1.02^t Laplace(0, 1e-4), both [32768, 4096] bf16 at full size.
    The 100-step sequence is too large to draw on the host in reasonable
    time; the oracle reads these bytes back from the device."""
    s = SEEDS[4]
    M, H = _dim(32768, scale), _dim(4096, scale)
    mult = 1.02 ** t
    gx = torch.Generator(device=device)
    gx.manual_seed(s * 1_000_003 + 2 * t)
    x = torch.randn((M, H), generator=gx, device=device, dtype=torch.float32)
    x.mul_(mult)
    gd = torch.Generator(device=device)
    gd.manual_seed(s * 1_000_003 + 2 * t + 1)
    # Laplace(0, b) by the inverse CDF of u ~ U(-1/2, 1/2): -b sign(u) log(1 - 2|u|)
    u = torch.rand((M, H), generator=gd, device=device, dtype=torch.float32).sub_(0.5)
    d = torch.log1p(u.abs().mul_(-2.0).clamp_(min=-1.0 + 2.0 ** -24)).mul_(u.sign()).mul_(-1e-4 * mult)
    return {"X": x.to(torch.bfloat16), "dY": d.to(torch.bfloat16)}


def config5(batch: int, scale: int = 1):
    s = SEEDS[5]
    F, H = _dim(18944, scale), _dim(3584, scale)
    return {"W_up": normal((F, H), s, 0, std=0.02),
            "W_down": normal((H, F), s, 1, std=0.02),
            "x_up": normal((batch, H), s, 10 + batch),
            "x_down": normal((batch, F), s, 20 + batch)}
