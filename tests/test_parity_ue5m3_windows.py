"""GPU UE5M3 scale windows and the multi-pass UE5M3 GEMM vs the oracle
(through the C ABI).

Tensors whose block magnitudes spread over 2^-30 .. 1 give UE5M3 scales
spanning more than one E4M3 window: fp4_ue5m3_to_e4m3 then reports
FP4_ERR_UE5M3_RANGE, while fp4_ue5m3_windows splits them exactly and
fp4_gemm_ue5m3_windows sums the window-pair GEMMs (float32 output, within the
GEMM bound of the oracle's UE5M3 GEMM).
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import dev, f32, host, lib, to_mma

pytestmark = pytest.mark.gpu


def spread(shape, seed, lo):
    """bf16 tensor whose 16-element blocks are scaled by 2^U(lo, 0)."""
    rng = np.random.default_rng(seed)
    R, C = shape
    x = rng.standard_normal((R, C)) * np.repeat(2.0 ** rng.uniform(lo, 0, (R, C // 16)), 16, axis=1)
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


def gpu_windows(scales_flat):
    fp4 = lib()
    n = scales_flat.size
    t = torch.zeros(3, dtype=torch.int32, device="cuda")
    nw = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(3 * n, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_ue5m3_windows(dev(scales_flat), t, nw, out, st)
    assert int(host(st)[0]) == 0
    return t, nw, out


def test_windows_bit_exact_every_code():
    rng = np.random.default_rng(50)
    for top in (0xFE, 0xA7, 0x3C):
        codes = np.arange(top + 1, dtype=np.uint8)
        codes = np.concatenate([codes, rng.integers(0, top + 1, 4000).astype(np.uint8)])
        t, nw, out = gpu_windows(codes)
        tr, outr, nr = Q.ue5m3_windows(codes)
        assert list(host(t)) == tr and int(host(nw)[0]) == nr
        assert np.array_equal(host(out).reshape(3, -1), outr)
    # all-zero scales: one window, shifts from t = 0
    t, nw, out = gpu_windows(np.zeros(64, dtype=np.uint8))
    assert list(host(t)) == [0, -14, -28] and int(host(nw)[0]) == 1 and not host(out).any()


def run_windowed(A, B, n_expect, stale=1.0):
    # stale: the stored amax of A is its max / stale (scales above 448, up to
    # UE5M3's largest value, as between refreshes)
    fp4 = lib()
    ga_v = float(np.max(np.abs(f32(A)))) / stale
    qa, qb = Q.quantize(f32(A), "UE5M3", global_amax=ga_v), Q.quantize(f32(B), "UE5M3")
    M, K, N = A.shape[0], A.shape[1], B.shape[0]
    sa, sb = to_mma(qa["scales"]), to_mma(qb["scales"])
    # the single shift is not exact on these tensors
    _, exact_a = Q.ue5m3_reencode_e4m3(qa["scales"], Q.ue5m3_shift(qa["scales"]))
    assert exact_a is (n_expect == 1)
    tA, nA, wA = gpu_windows(sa)
    tB, nB, wB = gpu_windows(sb)
    assert int(host(nA)[0]) == Q.ue5m3_windows(qa["scales"])[2] == n_expect
    ga = torch.tensor([ga_v], dtype=torch.float32, device="cuda")
    gb = torch.tensor([qb["amax"]], dtype=torch.float32, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm_ue5m3_windows(dev(qa["codes"]), wA, tA, nA, dev(qb["codes"]), wB, tB, nB, ga, gb, M, N, K, C,
                               dev_status=st)
    assert int(host(st)[0]) == 0
    Cr, S = Gm.gemm_ref(qa["codes"], qa["scales"], ga_v, qb["codes"], qb["scales"], qb["amax"], "UE5M3")
    got = host(C)
    err = np.abs(got - Cr)
    assert (err <= Gm.gemm_bound(S)).all(), f"worst ratio {np.max(err / Gm.gemm_bound(S)):.3g}"
    return qa, qb, ga_v, got


@pytest.mark.parametrize("M", [512, 384])  # CTA pairs; single CTAs (odd number of 128-row tiles)
def test_windowed_gemm_three_by_two_windows(M):
    # A: block scales from UE5M3's largest (stale amax, 256x small) down to its
    # smallest, three windows; B: fresh amax, 17 binades, two windows
    A = spread((M, 1024), 51, -31)
    B = spread((512, 1024), 52, -17)
    run_windowed(A, B, 3, stale=256.0)


def test_windowed_gemm_one_window_equals_the_plain_ue5m3_gemm():
    fp4 = lib()
    A = synth.normal((256, 512), 53, 0, outlier_p=0.01, outlier_mult=50.0)
    B = synth.normal((256, 512), 53, 1, std=0.02)
    qa, qb, ga_v, got = run_windowed(A, B, 1)
    M, K, N = 256, 512, 256
    out = []
    for q in (qa, qb):
        t = torch.zeros(1, dtype=torch.int32, device="cuda")
        e4 = torch.empty(q["scales"].size, dtype=torch.uint8, device="cuda")
        fp4.fp4_ue5m3_to_e4m3(dev(to_mma(q["scales"])), t, e4)
        out.append((t, e4))
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ga = torch.tensor([ga_v], dtype=torch.float32, device="cuda")
    gb = torch.tensor([qb["amax"]], dtype=torch.float32, device="cuda")
    fp4.fp4_gemm(dev(qa["codes"]), out[0][1], dev(qb["codes"]), out[1][1], ga, gb, out[0][0], out[1][0], M, N, K,
                 "UE5M3", fp4.FP4_OUT_F32, C)
    assert np.array_equal(host(C), got)  # the (0, 0) pass alone, bit for bit
