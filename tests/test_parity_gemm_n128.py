"""GEMM output widths that are a multiple of 128 but not of 256 (through the C ABI).

Output tiles are 256 columns wide; with N % 256 == 128 the last tile's upper
half reads zero-filled code rows and stores nothing.  Checked against the
oracle's float64 GEMM (bound 1e-5 * sum|a||b| + 1e-6, bf16 adding one
rounding) on both GEMM kernels (CTA pairs for M % 256 == 0, single CTAs
otherwise) and all three tensor-core scale formats; a sentinel-filled margin
beyond column N (ldc > N) must stay untouched.  The quantizing epilogue at
such a width equals fp4_gemm (bf16) + fp4_quantize byte for byte.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import dev, f32, host, lib, to_mma

pytestmark = pytest.mark.gpu


def _ops(fmt, M, N, K, seed):
    A = synth.normal((M, K), seed, 0, outlier_p=0.01, outlier_mult=50.0)
    B = synth.normal((N, K), seed, 1, std=0.02)
    qa, qb = Q.quantize(f32(A), fmt), Q.quantize(f32(B), fmt)
    out = []
    for q in (qa, qb):
        sc, t = q["scales"], None
        if fmt == "UE5M3":
            t = Q.ue5m3_shift(sc)
            sc, exact = Q.ue5m3_reencode_e4m3(sc, t)
            assert exact
        out.append((dev(q["codes"]), dev(to_mma(sc)), torch.tensor([q["amax"]], device="cuda"),
                    None if t is None else torch.tensor([t], dtype=torch.int32, device="cuda")))
    return qa, qb, out


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
@pytest.mark.parametrize("M", [256, 384], ids=["pairs", "single"])
@pytest.mark.parametrize("N", [128, 384, 640])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_n_multiple_of_128(fmt, M, N, out):
    fp4 = lib()
    K = 512
    qa, qb, ((ac, as_, ga, ta), (bc, bs, gb, tb)) = _ops(fmt, M, N, K, 40 + N)
    bf16 = out == "bf16"
    ldc = N + 128
    dt = torch.bfloat16 if bf16 else torch.float32
    C = torch.full((M, ldc), float("nan"), dtype=dt, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm(ac, as_, bc, bs, ga, gb, ta, tb, M, N, K, fmt, fp4.FP4_OUT_BF16 if bf16 else fp4.FP4_OUT_F32, C,
                 ldc=ldc, dev_status=st)
    assert int(host(st)[0]) == 0
    got = host(C.float())
    assert np.isnan(got[:, N:]).all(), "a store landed beyond column N"
    Cr, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], fmt)
    bound = Gm.gemm_bound(S) + (np.abs(Cr) * 2.0 ** -8 if bf16 else 0)
    err = np.abs(got[:, :N] - Cr)
    assert (err <= bound).all(), f"worst ratio {np.max(err / bound):.3g}"


@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_quantizing_epilogue_n_multiple_of_128(rounding):
    fp4 = lib()
    M, N, K = 256, 384, 512
    _, _, ((ac, as_, ga, ta), (bc, bs, gb, tb)) = _ops("E4M3", M, N, K, 77)
    rnd = fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE
    g_out = torch.tensor([0.5], device="cuda")
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * N // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm_quantize(ac, as_, bc, bs, ga, gb, None, None, M, N, K, "E4M3", g_out, rnd, 9, fp4.FP4_SFLAYOUT_MMA,
                          codes, scales, amax, st)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp4.fp4_gemm(ac, as_, bc, bs, ga, gb, None, None, M, N, K, "E4M3", fp4.FP4_OUT_BF16, C, dev_status=st)
    c2 = torch.empty_like(codes)
    s2 = torch.empty_like(scales)
    a2 = torch.zeros(1, device="cuda")
    fp4.fp4_quantize(C, "E4M3", rnd, 9, g_out, False, fp4.FP4_SFLAYOUT_MMA, c2, s2, a2, st)
    assert int(host(st)[0]) == 0
    assert np.array_equal(host(codes), host(c2))
    assert np.array_equal(host(scales), host(s2))
    assert host(amax)[0] == host(a2)[0]
