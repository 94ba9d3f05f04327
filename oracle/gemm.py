"""Reference GEMM / GEMV over dequantized FP4 operands (oracle; test infrastructure only).

The block-scaled FP4 GEMM of the pages ("NVFP4 vs MXFP" post, quant_prune_distill
#486, section "Метод": low-precision scales with an efficient kernel path; "UE5M3
FP4 Block Scaling ..." blog, section "Что сделали": every eligible linear layer
in FP4, forward and backward) computes, for quantized A [M, K] and B [N, K]
(both with their blocks along K),

    C[m, n] = sum_k  dA[m, k] * dB[n, k]

where dA, dB are the dequantized values e2m1 * s_b / s_enc.  This module forms
dA, dB in float64 and multiplies them with a library matmul (float64), and gives
the tolerance bound a float32-accumulating implementation must meet:

    |C_impl - C| <= 1e-5 * sum_k |dA[m,k]| |dB[n,k]| + 1e-6.

The weight-only linear (quant_prune_distill #574, section "Метод": weights in
NVFP4, activations left untouched) is y[b, n] = sum_k dW[n, k] * x[b, k] with x
the bf16 activations.
"""

from __future__ import annotations

import numpy as np

from .quantize import dequantize_f64

REL_TOL = 1e-5
ABS_TOL = 1e-6


def gemm_ref(Aq, As, ga, Bq, Bs, gb, fmt: str):
    """(C, S): float64 C = dA @ dB^T and S = |dA| @ |dB|^T."""
    dA = dequantize_f64(Aq, As, fmt, ga)
    dB = dequantize_f64(Bq, Bs, fmt, gb)
    return dA @ dB.T, np.abs(dA) @ np.abs(dB).T


def gemm_ref_rows(Aq, As, ga, Bq, Bs, gb, fmt: str, rows, cols=None):
    """C and S restricted to the given output rows (and columns)."""
    rows = np.asarray(rows)
    dA = dequantize_f64(Aq[rows], As[rows], fmt, ga)
    if cols is None:
        dB = dequantize_f64(Bq, Bs, fmt, gb)
    else:
        cols = np.asarray(cols)
        dB = dequantize_f64(Bq[cols], Bs[cols], fmt, gb)
    return dA @ dB.T, np.abs(dA) @ np.abs(dB).T


def gemm_bound(S: np.ndarray) -> np.ndarray:
    return REL_TOL * S + ABS_TOL


def gemv_ref(Wq, Ws, gw, x: np.ndarray, fmt: str = "E4M3"):
    """(y, S) for y[b, n] = sum_k dW[n, k] x[b, k] (x float32 holding bf16 values)."""
    dW = dequantize_f64(Wq, Ws, fmt, gw)
    x64 = np.asarray(x, dtype=np.float64)
    return x64 @ dW.T, np.abs(x64) @ np.abs(dW).T


def gemm_triple_loop(dA: np.ndarray, dB: np.ndarray) -> np.ndarray:
    """Plain triple loop over float64 values, for tiny shapes only."""
    M, K = dA.shape
    N = dB.shape[0]
    C = np.zeros((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(dA[m, k]) * float(dB[n, k])
            C[m, n] = acc
    return C
