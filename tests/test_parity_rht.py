"""16 x 16 random Hadamard transform + row quantization vs the oracle (through the C ABI).

"UE5M3 FP4 Block Scaling ..." blog, section "Что сделали" (the randomized
transform that spreads outliers before quantization); post on "INT v.s. FP: A
Comprehensive Study of Fine-Grained Low-bit Quantization Formats", section
"Метод" (Hadamard rotations before MX/NV FP or INT quantization).  Codes and
scales bit-exact, the fresh amax of the transformed tensor exact, and the FP4
GEMM of two operands transformed with the same mask within the GEMM bound of
the oracle's.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from oracle import rht as R
from gpu_util import dev, f32, from_mma, host, lib, to_mma

pytestmark = pytest.mark.gpu

MASK = 0xB38D
FMTS = ["E4M3", "UE5M3", "E8M0", "NVINT4", "MXINT4"]


def gpu_rht(x_bf16, fmt, rounding, seed, g=None, mma=False, mask=MASK):
    fp4 = lib()
    x = dev(x_bf16)
    M, K = x.shape
    G = Q.group_size(fmt)
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * K // G, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt = None if g is None else torch.tensor([g], dtype=torch.float32, device="cuda")
    fp4.fp4_quantize_rht(x, fmt, fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE, seed, mask, gt,
                         fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax, st)
    sc = host(scales)
    sc = from_mma(sc, M, K // G) if mma else sc.reshape(M, K // G)
    assert int(host(st)[0]) == 0
    return host(codes), sc, float(host(amax)[0])


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_rht_rows_bit_exact(fmt, rounding):
    x = synth.normal((256, 512), 31, 0, outlier_p=0.01, outlier_mult=50.0)
    xf = f32(x)
    ref = Q.quantize(xf, fmt, rounding, 17, rht_mask=MASK)
    c, s, a = gpu_rht(x, fmt, rounding, 17, mma=True)
    assert a == np.float32(ref["amax"]) == np.float32(np.max(np.abs(R.rht16(xf, MASK))))
    assert np.array_equal(s, ref["scales"])
    assert np.array_equal(c, ref["codes"])
    # stored (stale) amax, plain scale layout, another mask
    g = float(ref["amax"]) / 4
    ref2 = Q.quantize(xf, fmt, rounding, 18, global_amax=g, rht_mask=0x0F0F)
    c2, s2, _ = gpu_rht(x, fmt, rounding, 18, g=g, mask=0x0F0F)
    assert np.array_equal(s2, ref2["scales"]) and np.array_equal(c2, ref2["codes"])


def test_rht_config2_input():
    # the 350M MLP input recipe (per-column sigma log-uniform in [0.1, 10]) at 1/8 size
    x = synth.config2(scale=8)["X"]
    for fmt in ("E4M3", "NVINT4"):
        ref = Q.quantize(f32(x), fmt, "rne", 0, rht_mask=MASK)
        c, s, _ = gpu_rht(x, fmt, "rne", 0)
        assert np.array_equal(c, ref["codes"]) and np.array_equal(s, ref["scales"])


def test_gemm_on_transformed_operands():
    fp4 = lib()
    X = synth.normal((512, 1024), 32, 0, outlier_p=0.01, outlier_mult=50.0)
    W = synth.normal((512, 1024), 32, 1, std=0.02)
    qa = Q.quantize(f32(X), "E4M3", rht_mask=MASK)
    qb = Q.quantize(f32(W), "E4M3", rht_mask=MASK)
    C, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], "E4M3")
    ac, as_, aa = gpu_rht(X, "E4M3", "rne", 0, mma=True)
    bc, bs, ba = gpu_rht(W, "E4M3", "rne", 0, mma=True)
    assert np.array_equal(ac, qa["codes"]) and np.array_equal(bc, qb["codes"])
    Cg = torch.empty((512, 512), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ga = torch.tensor([aa], device="cuda")
    gb = torch.tensor([ba], device="cuda")
    fp4.fp4_gemm(dev(ac), dev(to_mma(as_)), dev(bc), dev(to_mma(bs)), ga, gb, None, None, 512, 512, 1024, "E4M3",
                 fp4.FP4_OUT_F32, Cg, dev_status=st)
    assert int(host(st)[0]) == 0
    got = host(Cg)
    assert (np.abs(got - C) <= Gm.gemm_bound(S)).all()
    exact = f32(X).astype(np.float64) @ f32(W).T.astype(np.float64)
    assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < 0.2


def gpu_dual_rht(x_bf16, fmt, r_row, s_row, r_col, s_col, g=None, mma=True, mask=MASK):
    fp4 = lib()
    x = dev(x_bf16)
    M, K = x.shape
    G = Q.group_size(fmt)
    u8 = dict(dtype=torch.uint8, device="cuda")
    cr, sr = torch.empty((M, K // 2), **u8), torch.empty(M * K // G, **u8)
    cc, sc = torch.empty((K, M // 2), **u8), torch.empty(M * K // G, **u8)
    ar, ac = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    R_ = {"rne": fp4.FP4_ROUND_RNE, "sr": fp4.FP4_ROUND_STOCHASTIC}
    gr = gc = None
    if g is not None:
        gr, gc = (torch.tensor([v], device="cuda") for v in g)
    fp4.fp4_quantize_dual_rht(x, fmt, R_[r_row], s_row, R_[r_col], s_col, mask, gr, gc,
                              fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, cr, sr, cc, sc, ar, ac, st)
    assert int(host(st)[0]) == 0
    fix = (lambda v, R, C: from_mma(host(v), R, C)) if mma else (lambda v, R, C: host(v).reshape(R, C))
    return (host(cr), fix(sr, M, K // G), host(cc), fix(sc, K, M // G), float(host(ar)[0]), float(host(ac)[0]))


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
@pytest.mark.parametrize("rr,rc", [("rne", "sr"), ("sr", "sr"), ("rne", "rne")])
def test_dual_rht_bit_exact(fmt, rr, rc):
    # 192 x 544: three 64-row tiles; four 128-column tiles and a 32-column tail
    x = synth.normal((192, 544), 33, 0, outlier_p=0.01, outlier_mult=50.0)
    xf = f32(x)
    ref_r = Q.quantize(xf, fmt, rr, 101, rht_mask=MASK)
    ref_c = Q.quantize(xf, fmt, rc, 102, transpose=True, rht_mask=MASK)
    cr, sr, cc, sc, ar, ac = gpu_dual_rht(x, fmt, rr, 101, rc, 102, mma=False)
    assert ar == np.float32(ref_r["amax"]) and ac == np.float32(ref_c["amax"])
    assert np.array_equal(sr, ref_r["scales"]) and np.array_equal(cr, ref_r["codes"])
    assert np.array_equal(sc, ref_c["scales"]) and np.array_equal(cc, ref_c["codes"])


def test_dual_rht_stored_amax_and_tiled_scales():
    x = synth.normal((256, 512), 34, 0, outlier_p=0.01, outlier_mult=50.0)
    xf = f32(x)
    g = (float(np.max(np.abs(R.rht16(xf, MASK)))) / 2, float(np.max(np.abs(R.rht16(xf.T, MASK)))) / 3)
    ref_r = Q.quantize(xf, "E4M3", "rne", 0, global_amax=g[0], rht_mask=MASK)
    ref_c = Q.quantize(xf, "E4M3", "sr", 7, global_amax=g[1], transpose=True, rht_mask=MASK)
    cr, sr, cc, sc, ar, ac = gpu_dual_rht(x, "E4M3", "rne", 0, "sr", 7, g=g, mma=True)
    assert np.array_equal(sr, ref_r["scales"]) and np.array_equal(cr, ref_r["codes"])
    assert np.array_equal(sc, ref_c["scales"]) and np.array_equal(cc, ref_c["codes"])
    assert ar == np.float32(np.max(np.abs(R.rht16(xf, MASK))))
    assert ac == np.float32(np.max(np.abs(R.rht16(xf.T, MASK))))


def test_fwd_dgrad_wgrad_with_the_transform():
    # the Llama-2 7B MLP recipe at 1/8 size: every GEMM operand transformed along
    # its reduction dimension with the same mask; results within the bound of
    # the oracle's and close to the untransformed products
    fp4 = lib()
    d = synth.config3(scale=8)  # M 2048, N 1280, K 512
    X, W, dY = d["X"], d["W"], d["dY"]
    q = {}
    for name, x, rr, rc in (("X", X, "rne", "sr"), ("W", W, "rne", "rne"), ("dY", dY, "sr", "sr")):
        cr, sr, cc, sc, ar, ac = gpu_dual_rht(x, "E4M3", rr, 11, rc, 12, mma=True)
        xf = f32(x)
        ref_r = Q.quantize(xf, "E4M3", rr, 11, rht_mask=MASK)
        ref_c = Q.quantize(xf, "E4M3", rc, 12, transpose=True, rht_mask=MASK)
        assert np.array_equal(cr, ref_r["codes"]) and np.array_equal(cc, ref_c["codes"])
        q[name] = ((cr, sr, ar), (cc, sc, ac), ref_r, ref_c)
    checks = [("fwd", q["X"][0], q["W"][0], q["X"][2], q["W"][2], f32(X) @ f32(W).T),
              ("dgrad", q["dY"][0], q["W"][1], q["dY"][2], q["W"][3], f32(dY) @ f32(W)),
              ("wgrad", q["dY"][1], q["X"][1], q["dY"][3], q["X"][3], f32(dY).T @ f32(X))]
    for what, (ac_, as_, aa), (bc, bs, ba), ra, rb, exact in checks:
        M, N, K = ac_.shape[0], bc.shape[0], ac_.shape[1] * 2
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4.fp4_gemm(dev(ac_), dev(to_mma(as_)), dev(bc), dev(to_mma(bs)), torch.tensor([aa], device="cuda"),
                     torch.tensor([ba], device="cuda"), None, None, M, N, K, "E4M3", fp4.FP4_OUT_F32, C, dev_status=st)
        assert int(host(st)[0]) == 0
        Cr, S = Gm.gemm_ref(ra["codes"], ra["scales"], ra["amax"], rb["codes"], rb["scales"], rb["amax"], "E4M3")
        got = host(C)
        assert (np.abs(got - Cr) <= Gm.gemm_bound(S)).all(), what
        exact = exact.astype(np.float64)
        assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < 0.25, what
