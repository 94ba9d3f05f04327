"""GEMM with a quantizing epilogue (fp4_gemm_quantize) through the C ABI.

The epilogue writes what fp4_quantize makes of the bf16 GEMM output under a
stored global amax ("UE5M3 FP4 Block Scaling ..." blog, section "Что
сделали": the tensor maximum refreshed every 50 steps, the stored value used
in between), so the next layer's input is quantized where it is produced.

* Identity with the two-call path on the GPU: codes, scales and the amax
  by-product equal fp4_quantize(bf16 output of fp4_gemm) bit for bit (both
  paths' parts are checked against the oracle elsewhere); the dual form's
  column blocks equal fp4_quantize(transpose = 1) of the same bf16 output.
* Against the oracle: the oracle's quantization of bf16(C_oracle) agrees on
  all but a few code nibbles (float32 vs float64 summation order can move the
  bf16 output by one ulp), and every disagreeing element moves by at most one
  grid step.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import dev, f32, from_mma, host, lib, to_mma

pytestmark = pytest.mark.gpu


def operands(fmt, M, N, K, seed):
    A = synth.normal((M, K), seed, 0, outlier_p=0.01, outlier_mult=50.0)
    B = synth.normal((N, K), seed, 1, std=0.02)
    qa, qb = Q.quantize(f32(A), fmt), Q.quantize(f32(B), fmt)
    dev_ops = []
    tv = []
    for q in (qa, qb):
        sc = to_mma(q["scales"])
        t = None
        if fmt == "UE5M3":
            t = Q.ue5m3_shift(q["scales"])
            sc_e4, exact = Q.ue5m3_reencode_e4m3(q["scales"], t)
            assert exact
            sc = to_mma(sc_e4)
        dev_ops.append((dev(q["codes"]), dev(sc), torch.tensor([q["amax"]], device="cuda"),
                        None if t is None else torch.tensor([t], dtype=torch.int32, device="cuda")))
    return qa, qb, dev_ops


def fused(dev_ops, M, N, K, fmt, g_out, rnd, seed, mma):
    fp4 = lib()
    (ac, as_, ga, ta), (bc, bs, gb, tb) = dev_ops
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * N // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm_quantize(ac, as_, bc, bs, ga, gb, ta, tb, M, N, K, fmt, torch.tensor([g_out], device="cuda"),
                          rnd, seed, fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax, st)
    assert int(host(st)[0]) == 0
    return codes, scales, amax


def unfused(dev_ops, M, N, K, fmt, g_out, rnd, seed, mma):
    fp4 = lib()
    (ac, as_, ga, ta), (bc, bs, gb, tb) = dev_ops
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm(ac, as_, bc, bs, ga, gb, ta, tb, M, N, K, fmt, fp4.FP4_OUT_BF16, C, dev_status=st)
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * N // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    fp4.fp4_quantize(C, "E4M3", rnd, seed, torch.tensor([g_out], device="cuda"), False,
                     fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax, st)
    assert int(host(st)[0]) == 0
    return codes, scales, amax, C


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
@pytest.mark.parametrize("rounding", ["rne", "sr"])
@pytest.mark.parametrize("mma", [False, True])
def test_fused_equals_two_calls(fmt, rounding, mma):
    fp4 = lib()
    M, N, K = 512, 768, 1024
    _, _, ops = operands(fmt, M, N, K, 41)
    rnd = fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE
    # a stored amax below the true one (stale) and a fresh-looking one
    _, _, _, C = unfused(ops, M, N, K, fmt, 1.0, rnd, 7, mma)
    g_true = float(C.float().abs().max())
    for g_out in (g_true, g_true / 3):
        fc, fs, fa = fused(ops, M, N, K, fmt, g_out, rnd, 7, mma)
        uc, us, ua, _ = unfused(ops, M, N, K, fmt, g_out, rnd, 7, mma)
        assert torch.equal(fc, uc)
        assert torch.equal(fs, us)
        assert float(fa) == float(ua) == g_true


def test_fused_against_the_oracle():
    fp4 = lib()
    M, N, K = 512, 512, 1024
    qa, qb, ops = operands("E4M3", M, N, K, 43)
    C, _ = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], "E4M3")
    Cb = torch.from_numpy(C.astype(np.float32)).to(torch.bfloat16).float().numpy()
    g_out = float(np.max(np.abs(Cb)))
    ref = Q.quantize(Cb, "E4M3", "sr", 9, global_amax=g_out)
    fc, fs, _ = fused(ops, M, N, K, "E4M3", g_out, fp4.FP4_ROUND_STOCHASTIC, 9, True)
    codes = host(fc)
    scales = from_mma(host(fs), M, N // 16)
    assert np.mean(scales != ref["scales"]) < 1e-3
    n_got, n_ref = Q.unpack(codes), Q.unpack(ref["codes"])
    assert np.mean(n_got != n_ref) < 2e-3
    # where they differ, the dequantized values are neighbours on the grid
    d_got = Q.dequantize_f64(codes, scales, "E4M3", g_out)
    d_ref = Q.dequantize_f64(ref["codes"], ref["scales"], "E4M3", g_out)
    step = np.repeat(Q.scale_values(scales, "E4M3"), 16, axis=1) * 2.0 / float(Q.global_encode_scale(g_out, "E4M3"))
    same_scale = np.repeat(scales == ref["scales"], 16, axis=1)
    assert np.all(np.abs(d_got - d_ref)[same_scale] <= step[same_scale] + 1e-30)


def fused_dual(dev_ops, M, N, K, fmt, g_out, r_row, seed_row, r_col, seed_col, mma, rows=True):
    fp4 = lib()
    (ac, as_, ga, ta), (bc, bs, gb, tb) = dev_ops
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda") if rows else None
    scales = torch.empty(M * N // 16, dtype=torch.uint8, device="cuda") if rows else None
    tcodes = torch.empty((N, M // 2), dtype=torch.uint8, device="cuda")
    tscales = torch.empty(M * N // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm_quantize_dual(ac, as_, bc, bs, ga, gb, ta, tb, M, N, K, fmt, torch.tensor([g_out], device="cuda"),
                               r_row, seed_row, r_col, seed_col,
                               fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, codes, scales, tcodes,
                               tscales, amax, st)
    assert int(host(st)[0]) == 0
    return codes, scales, tcodes, tscales, amax


def quantize_t(C, g_out, rnd, seed, mma):
    # fp4_quantize of C's columns (transpose = 1): codes [N, M/2]
    fp4 = lib()
    M, N = C.shape
    codes = torch.empty((N, M // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * N // 16, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_quantize(C, "E4M3", rnd, seed, torch.tensor([g_out], device="cuda"), True,
                     fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, codes, scales, None, st)
    assert int(host(st)[0]) == 0
    return codes, scales


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
@pytest.mark.parametrize("rounding", [("rne", "sr"), ("sr", "rne"), ("sr", "sr")])
@pytest.mark.parametrize("mma", [False, True])
def test_fused_dual_equals_two_calls(fmt, rounding, mma):
    # row blocks == fp4_quantize(bf16 C), column blocks == fp4_quantize(bf16 C,
    # transpose = 1), each with its own rounding and seed, one stored amax
    fp4 = lib()
    M, N, K = 512, 768, 1024
    _, _, ops = operands(fmt, M, N, K, 45)
    r_row, r_col = (fp4.FP4_ROUND_STOCHASTIC if r == "sr" else fp4.FP4_ROUND_RNE for r in rounding)
    _, _, _, C = unfused(ops, M, N, K, fmt, 1.0, r_row, 5, mma)
    g_true = float(C.float().abs().max())
    for g_out in (g_true, g_true / 3):
        fc, fs, ftc, fts, fa = fused_dual(ops, M, N, K, fmt, g_out, r_row, 5, r_col, 6, mma)
        uc, us, ua, _ = unfused(ops, M, N, K, fmt, g_out, r_row, 5, mma)
        utc, uts = quantize_t(C, g_out, r_col, 6, mma)
        assert torch.equal(fc, uc) and torch.equal(fs, us)
        assert torch.equal(ftc, utc) and torch.equal(fts, uts)
        assert float(fa) == float(ua) == g_true
        # the transposed output alone (row outputs NULL) is the same
        _, _, otc, ots, oa = fused_dual(ops, M, N, K, fmt, g_out, r_row, 5, r_col, 6, mma, rows=False)
        assert torch.equal(otc, utc) and torch.equal(ots, uts)
        assert float(oa) == g_true


def test_fused_dual_ragged_last_tile():
    # N % 256 == 128: the last output tile is half; its missing half writes nothing
    fp4 = lib()
    M, N, K = 512, 640, 512
    _, _, ops = operands("E4M3", M, N, K, 46)
    _, _, _, C = unfused(ops, M, N, K, "E4M3", 1.0, fp4.FP4_ROUND_RNE, 0, True)
    g = float(C.float().abs().max())
    fc, fs, ftc, fts, _ = fused_dual(ops, M, N, K, "E4M3", g, fp4.FP4_ROUND_RNE, 0, fp4.FP4_ROUND_STOCHASTIC, 3, True)
    utc, uts = quantize_t(C, g, fp4.FP4_ROUND_STOCHASTIC, 3, True)
    assert torch.equal(ftc, utc) and torch.equal(fts, uts)


def test_fused_transposed_against_the_oracle():
    # the column blocks against the oracle's transposed quantization of
    # bf16(C_oracle), as the row blocks are checked above
    fp4 = lib()
    M, N, K = 512, 512, 1024
    qa, qb, ops = operands("E4M3", M, N, K, 47)
    C, _ = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], "E4M3")
    Cb = torch.from_numpy(C.astype(np.float32)).to(torch.bfloat16).float().numpy()
    g_out = float(np.max(np.abs(Cb)))
    ref = Q.quantize(Cb, "E4M3", "sr", 11, global_amax=g_out, transpose=True)
    _, _, ftc, fts, _ = fused_dual(ops, M, N, K, "E4M3", g_out, fp4.FP4_ROUND_RNE, 0, fp4.FP4_ROUND_STOCHASTIC, 11,
                                   False, rows=False)
    codes = host(ftc)
    scales = host(fts).reshape(N, M // 16)
    assert codes.shape == ref["codes"].shape
    assert np.mean(scales != ref["scales"]) < 1e-3
    assert np.mean(Q.unpack(codes) != Q.unpack(ref["codes"])) < 2e-3
    d_got = Q.dequantize_f64(codes, scales, "E4M3", g_out)
    d_ref = Q.dequantize_f64(ref["codes"], ref["scales"], "E4M3", g_out)
    step = np.repeat(Q.scale_values(scales, "E4M3"), 16, axis=1) * 2.0 / float(Q.global_encode_scale(g_out, "E4M3"))
    same_scale = np.repeat(scales == ref["scales"], 16, axis=1)
    assert np.all(np.abs(d_got - d_ref)[same_scale] <= step[same_scale] + 1e-30)


def test_fused_rejects_single_cta_shapes():
    fp4 = lib()
    M, N, K = 384, 256, 256
    _, _, ops = operands("E4M3", M, N, K, 44)
    with pytest.raises(fp4.Fp4Error) as e:
        fused(ops, M, N, K, "E4M3", 1.0, fp4.FP4_ROUND_RNE, 0, False)
    assert e.value.status == fp4.FP4_ERR_UNSUPPORTED
