"""The persistent TMA-fed dual / transposed quantizer against the oracle (through the C ABI).

fp4_quantize_dual and fp4_quantize(transpose = 1) with the tiled scale
layout and M, K multiples of 128 run on the persistent kernel that streams
128 x 128 tiles through a TMA ring.  Codes and scales must equal the oracle's
bit for bit ("NVFP4 vs MXFP" post, "Метод"; rounding per the review of
Intel's FP4 paper, "Стохастическая квантизация"), with:
  * 13 x 12 = 156 tiles, more than one per CTA on 152 SMs (the persistent loop
    and both staging buffers are exercised);
  * rows of edge values: zeros, -0.0, exact E2M1 ties, bf16 subnormals,
    a 3e4 outlier, and column blocks of the same;
  * E4M3, UE5M3 and E1M6 scales; RNE and stochastic rounding on either
    output; fresh and stale (below the data) global amax;
  * the max|x| and UE5M3 shift by-products.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import quantize as Q
from gpu_util import dev, f32, from_mma, host, lib

pytestmark = pytest.mark.gpu

M, K = 1664, 1536


def _input():
    x = f32(synth.normal((M, K), 61, 0, outlier_p=0.01, outlier_mult=50.0))
    x[0, :] = 0.0
    x[1, :] = -0.0
    x[2, :16] = [6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -6, -5, -3.5, -2.5, -1.75, -1.25, -0.75, -0.25]
    x[3, :] = 9.2e-41  # bf16 subnormal
    x[4, 7] = 3e4
    x[:, 130] = 0.0  # a zero column: its transposed blocks are zero blocks
    x[16:32, 131] = 9.2e-41
    x[32:48, 132] = np.array([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -6, -5, -3.5, -2.5, -1.75, -1.25, -0.75,
                              -0.25], np.float32) * 2.0
    return synth.to_bf16(x)


@pytest.fixture(scope="module")
def data():
    xb = _input()
    return xb, f32(xb)


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E1M6"])
@pytest.mark.parametrize("rr,rc", [("rne", "rne"), ("rne", "sr"), ("sr", "sr")])
@pytest.mark.parametrize("stale", [False, True], ids=["fresh", "stale"])
def test_dual(data, fmt, rr, rc, stale):
    fp4 = lib()
    xb, xf = data
    g = np.float32(np.max(np.abs(xf)))
    # stale: a stored amax 4x below the data without the 3e4 outlier (E4M3 scales saturate, UE5M3 not)
    g_used = np.float32(np.max(np.abs(xf[5:])) / 4) if stale else g
    xd = dev(xb)
    cr = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sr = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
    cc = torch.empty((K, M // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = torch.zeros(2, dtype=torch.int32, device="cuda") if fmt == "UE5M3" else None
    rnd = {"rne": fp4.FP4_ROUND_RNE, "sr": fp4.FP4_ROUND_STOCHASTIC}
    gt = torch.tensor([g_used], dtype=torch.float32, device="cuda")
    fp4.fp4_quantize_dual(xd, fmt, rnd[rr], 101, rnd[rc], 102, gt, fp4.FP4_SFLAYOUT_MMA, cr, sr, cc, sc, amax, st,
                          ue5m3_shift_out=t)
    ref_r = Q.quantize(xf, fmt, rr, 101, global_amax=g_used)
    ref_c = Q.quantize(xf, fmt, rc, 102, global_amax=g_used, transpose=True)
    assert int(host(st)[0]) == 0
    assert np.array_equal(from_mma(host(sr), M, K // 16), ref_r["scales"]), "row scales"
    assert np.array_equal(from_mma(host(sc), K, M // 16), ref_c["scales"]), "transposed scales"
    for got, want, what in ((host(cr), ref_r["codes"], "row"), (host(cc), ref_c["codes"], "transposed")):
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{what} codes: {len(bad)} bytes differ, first at {bad[0].tolist()}"
    assert float(host(amax)[0]) == float(g)
    if t is not None:
        assert host(t).tolist() == [Q.ue5m3_shift(ref_r["scales"]), Q.ue5m3_shift(ref_c["scales"])]


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3"])
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_transposed_only(data, fmt, rounding):
    fp4 = lib()
    xb, xf = data
    xd = dev(xb)
    cc = torch.empty((K, M // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    t = torch.zeros(1, dtype=torch.int32, device="cuda") if fmt == "UE5M3" else None
    fp4.fp4_quantize(xd, fmt, fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE, 9, None, True,
                     fp4.FP4_SFLAYOUT_MMA, cc, sc, amax, ue5m3_shift_out=t)
    ref = Q.quantize(xf, fmt, rounding, 9, transpose=True)
    assert np.array_equal(from_mma(host(sc), K, M // 16), ref["scales"])
    assert np.array_equal(host(cc), ref["codes"])
    assert float(host(amax)[0]) == float(ref["amax"])
    if t is not None:
        assert int(host(t)[0]) == Q.ue5m3_shift(ref["scales"])


def test_repeated_calls_identical(data):
    # the same call twice (and after a call on another tensor) gives the same bytes
    fp4 = lib()
    xb, _ = data
    xd = dev(xb)
    other = dev(synth.normal((256, 384), 62, 0))
    outs = []
    for rep in range(2):
        cr = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        sr = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
        cc = torch.empty((K, M // 2), dtype=torch.uint8, device="cuda")
        sc = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
        g = torch.zeros(1, dtype=torch.float32, device="cuda")
        fp4.fp4_quantize_dual(xd, "E4M3", fp4.FP4_ROUND_STOCHASTIC, 5, fp4.FP4_ROUND_STOCHASTIC, 6, None,
                              fp4.FP4_SFLAYOUT_MMA, cr, sr, cc, sc, g)
        outs.append([host(v) for v in (cr, sr, cc, sc)])
        o = [torch.empty((256, 192), dtype=torch.uint8, device="cuda"), torch.empty(6144, dtype=torch.uint8,
                                                                                     device="cuda"),
             torch.empty((384, 128), dtype=torch.uint8, device="cuda"), torch.empty(6144, dtype=torch.uint8,
                                                                                     device="cuda")]
        fp4.fp4_quantize_dual(other, "E4M3", 0, 0, 0, 0, None, fp4.FP4_SFLAYOUT_MMA, *o, torch.zeros(1, device="cuda"))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
