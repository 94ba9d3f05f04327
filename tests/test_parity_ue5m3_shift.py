"""UE5M3 shift as a quantizer by-product, and the one-pass re-encode (through the C ABI).

"UE5M3 FP4 Block Scaling ..." blog, section "Ограничения": UE5M3 ran through
software emulation on a tensor-core path that takes another scale format.
Reading fixed here: t = e_max - 7, e_max the largest unbiased exponent among a
tensor's scale values (0 when all are zero), every scale re-encoded as the
E4M3 code of s * 2^-t.

* fp4_quantize / fp4_quantize_dual with ue5m3_shift_out give the oracle's t
  for the row and the transposed scales (fresh amax, a stale amax 256x below
  the data, an all-zero tensor, ragged shapes, RNE and SR), while their codes
  and scales stay bit-exact;
* fp4_ue5m3_reencode(t) equals the oracle's re-encode and equals
  fp4_ue5m3_to_e4m3 (which finds t itself) byte for byte, shift included;
* a GEMM fed by the by-product path equals the GEMM fed by fp4_ue5m3_to_e4m3.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import quantize as Q
from gpu_util import dev, f32, from_mma, host, lib

pytestmark = pytest.mark.gpu


def _inputs():
    X = synth.normal((320, 512), 31, 0, outlier_p=0.01, outlier_mult=50.0)  # ragged: 320 rows
    Y = synth.normal((256, 384), 31, 1, std=0.02)
    Z = torch.zeros((64, 96), dtype=torch.bfloat16)
    return [("X", X), ("Y", Y), ("zeros", Z)]


@pytest.mark.parametrize("rounding", ["rne", "sr"])
@pytest.mark.parametrize("stale", [False, True], ids=["fresh", "stale"])
def test_shift_by_product_rows_and_cols(rounding, stale):
    fp4 = lib()
    rnd = fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE
    for name, x in _inputs():
        xf = f32(x)
        M, K = xf.shape
        g = np.float32(np.max(np.abs(xf)))
        if stale:
            g = np.float32(g / 256)
        gt = torch.tensor([g], dtype=torch.float32, device="cuda")
        xd = dev(x)
        for transpose in (False, True):
            rows, cols = (K, M) if transpose else (M, K)
            codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
            scales = torch.empty(rows * cols // 16, dtype=torch.uint8, device="cuda")
            t = torch.full((1,), 99, dtype=torch.int32, device="cuda")
            fp4.fp4_quantize(xd, "UE5M3", rnd, 7, gt, transpose, fp4.FP4_SFLAYOUT_PLAIN, codes, scales,
                             ue5m3_shift_out=t)
            ref = Q.quantize(xf, "UE5M3", rounding, 7, global_amax=g, transpose=transpose)
            assert np.array_equal(host(codes), ref["codes"]), (name, transpose)
            assert np.array_equal(host(scales).reshape(rows, -1), ref["scales"]), (name, transpose)
            assert int(host(t)[0]) == Q.ue5m3_shift(ref["scales"]), (name, transpose)
        # dual: both shifts from one read (the tiled scale layout where the shape allows it)
        mma = M % 128 == 0 and K % 128 == 0
        cr = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        sr = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
        cc = torch.empty((K, M // 2), dtype=torch.uint8, device="cuda")
        sc = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
        t2 = torch.full((2,), 99, dtype=torch.int32, device="cuda")
        fp4.fp4_quantize_dual(xd, "UE5M3", rnd, 7, rnd, 8, gt, fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN,
                              cr, sr, cc, sc, ue5m3_shift_out=t2)
        ra = Q.quantize(xf, "UE5M3", rounding, 7, global_amax=g)
        rb = Q.quantize(xf, "UE5M3", rounding, 8, global_amax=g, transpose=True)
        got_r = from_mma(host(sr), M, K // 16) if mma else host(sr).reshape(M, -1)
        got_c = from_mma(host(sc), K, M // 16) if mma else host(sc).reshape(K, -1)
        assert np.array_equal(host(cr), ra["codes"]) and np.array_equal(got_r, ra["scales"]), name
        assert np.array_equal(host(cc), rb["codes"]) and np.array_equal(got_c, rb["scales"]), name
        assert host(t2).tolist() == [Q.ue5m3_shift(ra["scales"]), Q.ue5m3_shift(rb["scales"])], name


def test_reencode_with_known_shift_equals_both_paths():
    fp4 = lib()
    rng = np.random.default_rng(5)
    # scales inside one E4M3 window (exact) and a spread that is not (range error)
    for lo, hi, exact in ((0x60, 0xB8, True), (0x08, 0xF0, False)):
        s = rng.integers(lo, hi, 4096).astype(np.uint8)
        s[::17] = 0
        t_ref = Q.ue5m3_shift(s)
        e4_ref, ex = Q.ue5m3_reencode_e4m3(s, t_ref)
        assert ex == exact
        sd = dev(s)
        t = torch.tensor([t_ref], dtype=torch.int32, device="cuda")
        out = torch.empty_like(sd)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4.fp4_ue5m3_reencode(sd, t, out, st)
        t2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        out2 = torch.empty_like(sd)
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4.fp4_ue5m3_to_e4m3(sd, t2, out2, st2)
        assert int(host(t2)[0]) == t_ref
        assert np.array_equal(host(out), host(out2))
        if exact:
            assert np.array_equal(host(out), e4_ref)
            assert int(host(st)[0]) == 0
        else:
            assert int(host(st)[0]) == fp4.FP4_ERR_UE5M3_RANGE
            assert int(host(st2)[0]) == fp4.FP4_ERR_UE5M3_RANGE


def test_gemm_from_by_product_shift():
    fp4 = lib()
    M, N, K = 256, 384, 512
    A = dev(synth.normal((M, K), 33, 0, outlier_p=0.01, outlier_mult=50.0))
    B = dev(synth.normal((N, K), 33, 1, std=0.02))
    outs = []
    for by_product in (True, False):
        ops = []
        for x, R in ((A, M), (B, N)):
            codes = torch.empty((R, K // 2), dtype=torch.uint8, device="cuda")
            scales = torch.empty(R * K // 16, dtype=torch.uint8, device="cuda")
            amax = torch.zeros(1, device="cuda")
            t = torch.zeros(1, dtype=torch.int32, device="cuda")
            e4 = torch.empty_like(scales)
            if by_product:
                fp4.fp4_quantize(x, "UE5M3", fp4.FP4_ROUND_RNE, 0, None, False, fp4.FP4_SFLAYOUT_MMA, codes, scales,
                                 amax, ue5m3_shift_out=t)
                fp4.fp4_ue5m3_reencode(scales, t, e4)
            else:
                fp4.fp4_quantize(x, "UE5M3", fp4.FP4_ROUND_RNE, 0, None, False, fp4.FP4_SFLAYOUT_MMA, codes, scales,
                                 amax)
                fp4.fp4_ue5m3_to_e4m3(scales, t, e4)
            ops.append((codes, e4, amax, t))
        (ac, ae, ag, at), (bc, be, bg, bt) = ops
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4.fp4_gemm(ac, ae, bc, be, ag, bg, at, bt, M, N, K, "UE5M3", fp4.FP4_OUT_F32, C, dev_status=st)
        assert int(host(st)[0]) == 0
        outs.append(host(C))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
