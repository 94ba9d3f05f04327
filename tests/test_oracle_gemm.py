"""Pins of the oracle's reference GEMM and GEMV (CPU only)."""

import numpy as np

from oracle import gemm as Gm
from oracle import quantize as Q
from test_oracle_quantize import bf16, _data


def test_gemm_matches_triple_loop_tiny():
    A = _data(10, (8, 64))
    B = _data(11, (6, 64))
    for fmt in ("E4M3", "UE5M3", "E8M0"):
        qa, qb = Q.quantize(A, fmt), Q.quantize(B, fmt)
        C, S = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], fmt)
        dA = Q.dequantize_f64(qa["codes"], qa["scales"], fmt, qa["amax"])
        dB = Q.dequantize_f64(qb["codes"], qb["scales"], fmt, qb["amax"])
        Cl = Gm.gemm_triple_loop(dA, dB)
        assert np.allclose(C, Cl, rtol=1e-12, atol=1e-12)
        assert np.all(S >= np.abs(C) - 1e-9)


def test_gemm_all_ones_closed_form():
    K = 512
    A = np.ones((4, K), dtype=np.float32)
    B = np.ones((3, K), dtype=np.float32)
    qa, qb = Q.quantize(A, "E4M3"), Q.quantize(B, "E4M3")
    C, _ = Gm.gemm_ref(qa["codes"], qa["scales"], 1.0, qb["codes"], qb["scales"], 1.0, "E4M3")
    assert np.all(C == K)


def test_gemm_exact_integer_special_case():
    # MXFP4 blocks whose maximum is 4 have scale 1, so the dequantized operands are
    # the E2M1 values themselves; twice each value is an integer, so 4*C equals an
    # exact integer matrix product.
    rng = np.random.default_rng(12)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, -0.5, -1, -1.5, -2, -3, -4])
    A = rng.choice(grid, (16, 128)).astype(np.float32)
    B = rng.choice(grid, (8, 128)).astype(np.float32)
    A[:, ::32] = 4.0
    B[:, ::32] = -4.0
    qa, qb = Q.quantize(A, "E8M0"), Q.quantize(B, "E8M0")
    C, _ = Gm.gemm_ref(qa["codes"], qa["scales"], 0, qb["codes"], qb["scales"], 0, "E8M0")
    Ai = (2 * A).astype(np.int64)
    Bi = (2 * B).astype(np.int64)
    assert np.array_equal((4 * C).astype(np.int64), Ai @ Bi.T)
    assert np.array_equal(4 * C, (Ai @ Bi.T).astype(np.float64))


def test_gemv_one_hot_picks_column():
    W = _data(13, (32, 64))
    qw = Q.quantize(W, "E4M3")
    dW = Q.dequantize_f64(qw["codes"], qw["scales"], "E4M3", qw["amax"])
    x = np.zeros((2, 64), dtype=np.float32)
    x[0, 5] = 1.0
    x[1, 63] = -2.0
    y, S = Gm.gemv_ref(qw["codes"], qw["scales"], qw["amax"], x)
    assert np.array_equal(y[0], dW[:, 5])
    assert np.array_equal(y[1], -2.0 * dW[:, 63])


def test_bound_shape():
    S = np.array([0.0, 1.0, 1e6])
    assert np.allclose(Gm.gemm_bound(S), [1e-6, 1e-5 + 1e-6, 10.000001])
