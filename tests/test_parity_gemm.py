"""GPU block-scaled FP4 GEMM vs the oracle's float64 GEMM (through the C ABI).

The GPU GEMM gets the ORACLE's codes and scales (scales permuted on the host
into the tiled layout), so this isolates the GEMM from the quantizer.  Bound:
|C_gpu - C| <= 1e-5 * sum_k |a||b| + 1e-6 (float32 output); bf16 output adds
one bf16 rounding, 2^-8 |C|.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import dev, f32, host, lib, to_mma

pytestmark = pytest.mark.gpu


def oracle_q(x_bf16, fmt, rounding="rne", seed=0, transpose=False):
    return Q.quantize(f32(x_bf16), fmt, rounding, seed, transpose=transpose)


def gpu_gemm(qa, qb, fmt, out="f32", tA=None, tB=None, sa=None, sb=None):
    fp4 = lib()
    M, K = qa["codes"].shape[0], qa["codes"].shape[1] * 2
    N = qb["codes"].shape[0]
    sa = qa["scales"] if sa is None else sa
    sb = qb["scales"] if sb is None else sb
    C = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ga = torch.tensor([qa["amax"]], dtype=torch.float32, device="cuda")
    gb = torch.tensor([qb["amax"]], dtype=torch.float32, device="cuda")
    ta = None if tA is None else torch.tensor([tA], dtype=torch.int32, device="cuda")
    tb = None if tB is None else torch.tensor([tB], dtype=torch.int32, device="cuda")
    fp4.fp4_gemm(dev(qa["codes"]), dev(to_mma(sa)), dev(qb["codes"]), dev(to_mma(sb)), ga, gb, ta, tb, M, N, K,
                 fmt, fp4.FP4_OUT_F32 if out == "f32" else fp4.FP4_OUT_BF16, C, dev_status=st)
    assert int(host(st)[0]) == 0
    return host(C.float())


def check_bound(Cg, C, S, bf16=False):
    bound = Gm.gemm_bound(S)
    if bf16:
        bound = bound + np.abs(C) * 2.0 ** -8
    err = np.abs(Cg - C)
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} entries out of bound; worst ratio {np.max(err / bound):.3g}"


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_config1_nvfp4(out):
    d = synth.config1()
    qa, qb = oracle_q(d["A"], "E4M3"), oracle_q(d["B"], "E4M3")
    C, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], "E4M3")
    check_bound(gpu_gemm(qa, qb, "E4M3", out), C, S, bf16=out == "bf16")


def test_exact_mxfp4_integer_case():
    # E2M1 values on blocks whose maximum is 4: scale 1, every partial sum an
    # integer multiple of 1/4 below 2^24 -> the float32 result is exact.
    rng = np.random.default_rng(12)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, -0.5, -1, -1.5, -2, -3, -4])
    A = rng.choice(grid, (256, 512)).astype(np.float32)
    B = rng.choice(grid, (256, 512)).astype(np.float32)
    A[:, ::32] = 4.0
    B[:, ::32] = -4.0
    qa, qb = Q.quantize(A, "E8M0"), Q.quantize(B, "E8M0")
    C, _ = Gm.gemm_ref(qa["codes"], qa["scales"], 0, qb["codes"], qb["scales"], 0, "E8M0")
    Cg = gpu_gemm(qa, qb, "E8M0")
    assert np.array_equal(Cg, C.astype(np.float32))


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
def test_multi_tile_persistent(fmt):
    # 2560 x 2048 x 512: 160 output tiles, more than one per CTA on 152 SMs
    A = synth.normal((2560, 512), 21, 0, outlier_p=0.01, outlier_mult=50.0)
    B = synth.normal((2048, 512), 21, 1, std=0.02)
    qa, qb = oracle_q(A, fmt), oracle_q(B, fmt)
    C, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], fmt)
    if fmt == "UE5M3":
        tA, tB = Q.ue5m3_shift(qa["scales"]), Q.ue5m3_shift(qb["scales"])
        sa, ea = Q.ue5m3_reencode_e4m3(qa["scales"], tA)
        sb, eb = Q.ue5m3_reencode_e4m3(qb["scales"], tB)
        assert ea and eb
        Cg = gpu_gemm(qa, qb, fmt, tA=tA, tB=tB, sa=sa, sb=sb)
    else:
        Cg = gpu_gemm(qa, qb, fmt)
    check_bound(Cg, C, S)


def test_ue5m3_reencode_matches_oracle():
    fp4 = lib()
    x = synth.normal((256, 1024), 22, 0, outlier_p=0.01, outlier_mult=50.0)
    for g_scale in (1.0, 1 / 8):  # fresh amax and an 8x stale one
        g = float(x.float().abs().max()) * g_scale
        q = Q.quantize(f32(x), "UE5M3", global_amax=g)
        t_ref = Q.ue5m3_shift(q["scales"])
        e_ref, exact = Q.ue5m3_reencode_e4m3(q["scales"], t_ref)
        t = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty(q["scales"].size, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4.fp4_ue5m3_to_e4m3(dev(q["scales"].reshape(-1)), t, out, st)
        assert int(host(t)[0]) == t_ref
        assert np.array_equal(host(out), e_ref.reshape(-1))
        assert int(host(st)[0]) == (0 if exact else fp4.FP4_ERR_UE5M3_RANGE)


def test_config2_formats_scaled():
    d = synth.config2(scale=4)  # 2048 x 1024 x 256
    for fmt in ("E4M3", "UE5M3", "E8M0"):
        qx, qw = oracle_q(d["X"], fmt), oracle_q(d["W"], fmt)
        C, S = Gm.gemm_ref(qx["codes"], qx["scales"], qx["amax"], qw["codes"], qw["scales"], qw["amax"], fmt)
        if fmt == "UE5M3":
            tA, tB = Q.ue5m3_shift(qx["scales"]), Q.ue5m3_shift(qw["scales"])
            sa, _ = Q.ue5m3_reencode_e4m3(qx["scales"], tA)
            sb, _ = Q.ue5m3_reencode_e4m3(qw["scales"], tB)
            Cg = gpu_gemm(qx, qw, fmt, tA=tA, tB=tB, sa=sa, sb=sb)
        else:
            Cg = gpu_gemm(qx, qw, fmt)
        check_bound(Cg, C, S)


def test_config3_fwd_dgrad_wgrad_scaled():
    d = synth.config3(scale=8)  # M 2048, N 1280, K 512
    X, W, dY = d["X"], d["W"], d["dY"]
    qX = oracle_q(X, "E4M3")
    qW = oracle_q(W, "E4M3")
    qWt = oracle_q(W, "E4M3", transpose=True)
    qXt = oracle_q(X, "E4M3", "sr", 1236, transpose=True)
    qdY = oracle_q(dY, "E4M3", "sr", 1234)
    qdYt = oracle_q(dY, "E4M3", "sr", 1235, transpose=True)
    for a, b in [(qX, qW), (qdY, qWt), (qdYt, qXt)]:
        C, S = Gm.gemm_ref(a["codes"], a["scales"], a["amax"], b["codes"], b["scales"], b["amax"], "E4M3")
        check_bound(gpu_gemm(a, b, "E4M3", "bf16"), C, S, bf16=True)


@pytest.mark.parametrize("fmt", ["E4M3", "E8M0"])
def test_long_k_plan(fmt):
    # long K on CTA pairs (M = 256: one 256-row pair tile)
    A = synth.normal((256, 8192), 23, 0, outlier_p=0.01, outlier_mult=50.0)
    B = synth.normal((512, 8192), 23, 1, std=0.02)
    qa, qb = oracle_q(A, fmt), oracle_q(B, fmt)
    C, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], fmt)
    check_bound(gpu_gemm(qa, qb, fmt), C, S)
    check_bound(gpu_gemm(qa, qb, fmt, "bf16"), C, S, bf16=True)


@pytest.mark.parametrize("fmt,K", [("E4M3", 512), ("E8M0", 512), ("E4M3", 8192), ("E8M0", 8192)])
def test_single_cta_tiles(fmt, K):
    # M = 384 is an odd number of 128-row tiles, so the GEMM runs one CTA per
    # 128 x 256 tile instead of CTA pairs on 256 x 256 tiles (K >= 8192: the
    # 4-stage ring with 16-byte output blocks)
    A = synth.normal((384, K), 24, 0, outlier_p=0.01, outlier_mult=50.0)
    B = synth.normal((512, K), 24, 1, std=0.02)
    qa, qb = oracle_q(A, fmt), oracle_q(B, fmt)
    C, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], fmt)
    check_bound(gpu_gemm(qa, qb, fmt), C, S)
    check_bound(gpu_gemm(qa, qb, fmt, "bf16"), C, S, bf16=True)
