"""Pins of the oracle's 16 x 16 random Hadamard transform (CPU only)."""

import numpy as np
import torch

from oracle import gemm as Gm
from oracle import quantize as Q
from oracle import rht as R


def bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


MASK = 0b1011001110001101


def test_hadamard_matrix_is_sylvester_and_orthogonal():
    H = R.hadamard16()
    assert np.array_equal(H @ H.T, 16 * np.eye(16))
    H2 = np.array([[1, 1], [1, -1]])
    S = H2
    for _ in range(3):
        S = np.kron(S, H2)
    assert np.array_equal(H, S)


def test_one_hot_closed_form():
    s = R.sign_vector(MASK)
    for j in range(16):
        x = np.zeros((1, 16), np.float32)
        x[0, j] = 1.0
        got = R.rht16(x, MASK)[0]
        want = 0.25 * s[j] * R.hadamard16()[:, j]
        assert np.array_equal(got, want.astype(np.float32))


def test_equals_matrix_product_exactly_on_integers():
    rng = np.random.default_rng(0)
    x = rng.integers(-50, 51, (64, 48)).astype(np.float32)  # every partial sum exact in float32
    T = 0.25 * R.hadamard16() @ np.diag(R.sign_vector(MASK).astype(np.float64))
    want = (x.reshape(-1, 16).astype(np.float64) @ T.T).reshape(x.shape)
    assert np.array_equal(R.rht16(x, MASK).astype(np.float64), want)


def test_inverse_exact_on_integers():
    rng = np.random.default_rng(1)
    x = rng.integers(-100, 101, (32, 32)).astype(np.float32)
    y = R.rht16(x, MASK)
    back = (R.rht16(y, 0) * R.sign_vector(MASK)[None, :].repeat(2, 0).reshape(1, 32)).astype(np.float32)
    assert np.array_equal(back, x)


def test_matches_matrix_product_within_float32_rounding():
    rng = np.random.default_rng(2)
    x = bf16(rng.standard_normal((256, 128)) * np.exp(rng.standard_normal((256, 128))))
    T = 0.25 * R.hadamard16() @ np.diag(R.sign_vector(MASK).astype(np.float64))
    want = (x.reshape(-1, 16).astype(np.float64) @ T.T).reshape(x.shape)
    scale = (np.abs(x.reshape(-1, 16)).astype(np.float64) @ np.abs(T.T)).reshape(x.shape)
    assert np.all(np.abs(R.rht16(x, MASK) - want) <= 4 * 2.0 ** -24 * scale + 1e-30)


def test_product_preserved_along_k():
    rng = np.random.default_rng(3)
    X = bf16(rng.standard_normal((64, 256)))
    W = bf16(rng.standard_normal((48, 256)))
    C = X.astype(np.float64) @ W.T.astype(np.float64)
    Ct = R.rht16(X, MASK).astype(np.float64) @ R.rht16(W, MASK).T.astype(np.float64)
    S = np.abs(X).astype(np.float64) @ np.abs(W).T.astype(np.float64)
    assert np.all(np.abs(Ct - C) <= 1e-5 * S)


def test_outlier_is_spread_and_quantization_improves():
    # one large outlier per block: after the transform it is spread over the
    # 16 values of the block, and NVINT4's error drops (the INT post's point)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((512, 256)).astype(np.float32)
    x[:, ::16] *= 40.0
    x = bf16(x)
    xt = R.rht16(x, MASK)
    assert np.abs(xt).max() < 0.5 * np.abs(x).max()

    def rel_err(fmt, mask):
        ref = R.rht16(x, mask) if mask is not None else x
        q = Q.quantize(x, fmt, rht_mask=mask)
        d = Q.dequantize_f64(q["codes"], q["scales"], fmt, q["amax"])
        return np.linalg.norm(d - ref) / np.linalg.norm(ref)

    assert rel_err("NVINT4", MASK) < rel_err("NVINT4", None)


def test_quantize_with_transform_uses_transformed_amax():
    rng = np.random.default_rng(5)
    x = bf16(rng.standard_normal((32, 64)))
    q = Q.quantize(x, "E4M3", rht_mask=MASK)
    assert q["amax"] == np.float32(np.max(np.abs(R.rht16(x, MASK))))
    q2 = Q.quantize(R.rht16(x, MASK), "E4M3")
    assert np.array_equal(q["codes"], q2["codes"]) and np.array_equal(q["scales"], q2["scales"])


def test_gemm_on_transformed_operands_approximates_the_product():
    rng = np.random.default_rng(6)
    X = bf16(rng.standard_normal((128, 512)))
    W = bf16(rng.standard_normal((128, 512)) * 0.02)
    qa = Q.quantize(X, "E4M3", rht_mask=MASK)
    qb = Q.quantize(W, "E4M3", rht_mask=MASK)
    C, _ = Gm.gemm_ref(qa["codes"], qa["scales"], qa["amax"], qb["codes"], qb["scales"], qb["amax"], "E4M3")
    exact = X.astype(np.float64) @ W.T.astype(np.float64)
    assert np.linalg.norm(C - exact) / np.linalg.norm(exact) < 0.2


def test_transposed_transform_runs_along_m():
    rng = np.random.default_rng(7)
    x = bf16(rng.standard_normal((64, 32)))
    q = Q.quantize(x, "E4M3", transpose=True, rht_mask=MASK)
    q2 = Q.quantize(R.rht16(x.T, MASK), "E4M3")
    assert np.array_equal(q["codes"], q2["codes"]) and np.array_equal(q["scales"], q2["scales"])
    assert q["amax"] == np.float32(np.max(np.abs(R.rht16(x.T, MASK))))


def test_wgrad_product_preserved_with_transposed_transforms():
    # dW = dY^T X: both operands transformed along M (the reduction dimension)
    rng = np.random.default_rng(8)
    dY = bf16(rng.standard_normal((256, 48)))
    X = bf16(rng.standard_normal((256, 64)))
    exact = dY.T.astype(np.float64) @ X.astype(np.float64)
    got = R.rht16(dY.T, MASK).astype(np.float64) @ R.rht16(X.T, MASK).T.astype(np.float64)
    S = np.abs(dY.T).astype(np.float64) @ np.abs(X).astype(np.float64)
    assert np.all(np.abs(got - exact) <= 1e-5 * S)
