"""Full-size parity in the benchmark's launch configuration (through the C ABI).

Runs one step of bench.LinearStep on the Llama-2-7B MLP workload
(M = 16384, K = 4096, N = 11008) exactly as bench.py times it, then checks
sampled outputs against the oracle:
  * fresh amaxes: exact;
  * row and transposed quantizations of X, W and dY: sampled rows and columns,
    codes and scales bit-exact (Philox indices in the output layout);
  * forward, dgrad and wgrad GEMMs (bf16 out): sampled output rows against the
    oracle's float64 GEMM over the oracle's own quantization of the operands.
"""

import numpy as np
import pytest
import torch

from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import from_mma, lib

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def step():
    lib()
    import bench
    d = bench.make_inputs()
    s = bench.LinearStep(d, torch.device("cuda", 0))
    s.run()
    torch.cuda.synchronize()
    assert int(s.status.item()) == 0
    return bench, d, s


def _rows(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, k)]))


def test_amax_exact(step):
    _, d, s = step
    a = s.amax.cpu().numpy()
    for j, name in enumerate(["X", "W", "dY"]):
        assert a[j] == np.float32(d[name].float().abs().max().item()), name


@pytest.mark.parametrize("name,rr,seed_r,rc,seed_c", [("X", "rne", 0, "sr", 1236), ("W", "rne", 0, "rne", 0),
                                                      ("dY", "sr", 1234, "sr", 1235)])
def test_quantizer_sampled(step, name, rr, seed_r, rc, seed_c):
    _, d, s = step
    x = d[name]
    R, C = x.shape
    g = float(x.float().abs().max())
    cr, sr, cc, sc = (t.cpu().numpy() for t in s.q[name])
    srow = from_mma(sr, R, C // 16)
    scol = from_mma(sc, C, R // 16)
    for r in _rows(R, 6, 1):
        codes, scales = Q.quantize_rows(x[r:r + 1].float().numpy(), "E4M3", rr, seed_r, g, row0=int(r))
        assert np.array_equal(cr[r], codes[0]) and np.array_equal(srow[r], scales[0]), (name, "row", r)
    for c in _rows(C, 6, 2):
        col = x[:, c].float().numpy()[None, :]
        codes, scales = Q.quantize_rows(col, "E4M3", rc, seed_c, g, row0=int(c))
        assert np.array_equal(cc[c], codes[0]) and np.array_equal(scol[c], scales[0]), (name, "col", c)


def _check_rows(Cg, a, b, rows):
    C, S = Gm.gemm_ref_rows(a["codes"], a["scales"], a["amax"], b["codes"], b["scales"], b["amax"], "E4M3", rows)
    got = Cg[rows].float().cpu().numpy()
    bound = Gm.gemm_bound(S) + np.abs(C) * 2.0 ** -8
    err = np.abs(got - C)
    assert (err <= bound).all(), f"worst ratio {np.max(err / bound):.3g}"


def test_gemms_sampled_rows(step):
    _, d, s = step
    X, W, dY = (d[k].float().numpy() for k in ("X", "W", "dY"))
    M, N = dY.shape
    qW = Q.quantize(W, "E4M3", "rne", 0, chunk_rows=512)
    qWt = Q.quantize(W, "E4M3", "rne", 0, transpose=True, chunk_rows=512)
    qXt = Q.quantize(X, "E4M3", "sr", 1236, transpose=True, chunk_rows=256)
    rows_m = _rows(M, 10, 3)
    rows_n = _rows(N, 10, 4)
    # forward Y = X W^T: sampled token rows of Q(X)
    g_X = np.float32(np.max(np.abs(X)))
    qX_rows = np.zeros((M, X.shape[1] // 2), np.uint8)
    sX_rows = np.zeros((M, X.shape[1] // 16), np.uint8)
    for r in rows_m:
        c, sc = Q.quantize_rows(X[r:r + 1], "E4M3", "rne", 0, g_X, row0=int(r))
        qX_rows[r], sX_rows[r] = c[0], sc[0]
    _check_rows(s.Y, {"codes": qX_rows, "scales": sX_rows, "amax": g_X}, qW, rows_m)
    # dgrad dX = dY W: rows of Q(dY) on the sampled tokens, B = Q(W^T)
    g_dY = np.float32(np.max(np.abs(dY)))
    qdY_rows = np.zeros((M, N // 2), np.uint8)
    sdY_rows = np.zeros((M, N // 16), np.uint8)
    for r in rows_m:
        c, sc = Q.quantize_rows(dY[r:r + 1], "E4M3", "sr", 1234, g_dY, row0=int(r))
        qdY_rows[r], sdY_rows[r] = c[0], sc[0]
    _check_rows(s.dX, {"codes": qdY_rows, "scales": sdY_rows, "amax": g_dY}, qWt, rows_m)
    # wgrad dW = dY^T X: sampled rows of Q(dY^T) (columns of dY), B = Q(X^T)
    qdYt_rows = np.zeros((N, M // 2), np.uint8)
    sdYt_rows = np.zeros((N, M // 16), np.uint8)
    for c in rows_n:
        cd, sc = Q.quantize_rows(dY[:, c][None, :], "E4M3", "sr", 1235, g_dY, row0=int(c))
        qdYt_rows[c], sdYt_rows[c] = cd[0], sc[0]
    _check_rows(s.dW, {"codes": qdYt_rows, "scales": sdYt_rows, "amax": g_dY}, qXt, rows_n)


def test_gemv_sampled(step):
    _, d, s = step
    W = d["W"].float().numpy()
    qw = Q.quantize(W, "E4M3", "rne", 0)
    x = d["x_dec"].float().numpy()
    y, S = Gm.gemv_ref(qw["codes"], qw["scales"], qw["amax"], x)
    got = s.yg.float().cpu().numpy()
    bound = Gm.gemm_bound(S) + np.abs(y) * 2.0 ** -8
    assert (np.abs(got - y) <= bound).all()


# ---------------------------------------------------------------------------
# 350M-parameter MLP linear (8192 x 4096 x 1024) at full size, three formats
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
def test_config2_fullsize(fmt):
    from fp4_block_scaled_amax_gb300 import synth
    from gpu_util import dev, host, to_mma
    fp4 = lib()
    d = synth.config2()
    X, W = d["X"], d["W"]
    M, K = X.shape
    N = W.shape[0]
    G = Q.group_size(fmt)
    out = {}
    for name, x in (("X", X), ("W", W)):
        R = x.shape[0]
        codes = torch.empty((R, K // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty(R * K // G, dtype=torch.uint8, device="cuda")
        amax = torch.zeros(1, dtype=torch.float32, device="cuda")
        fp4.fp4_quantize(dev(x), fmt, fp4.FP4_ROUND_RNE, 0, None, False, fp4.FP4_SFLAYOUT_MMA, codes, scales, amax)
        ref = Q.quantize(x.float().numpy(), fmt, "rne", 0)
        assert np.array_equal(host(codes), ref["codes"]), (fmt, name)
        assert np.array_equal(from_mma(host(scales), R, K // G), ref["scales"]), (fmt, name)
        out[name] = (codes, scales, amax, ref)
    (xc, xs, xa, qx), (wc, ws, wa, qw) = out["X"], out["W"]
    ta = tb = None
    if fmt == "UE5M3":
        ta, tb = torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")
        xs2, ws2 = torch.empty_like(xs), torch.empty_like(ws)
        fp4.fp4_ue5m3_to_e4m3(xs, ta, xs2)
        fp4.fp4_ue5m3_to_e4m3(ws, tb, ws2)
        xs, ws = xs2, ws2
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_gemm(xc, xs, wc, ws, xa, wa, ta, tb, M, N, K, fmt, fp4.FP4_OUT_F32, C, dev_status=st)
    assert int(host(st)[0]) == 0
    rows = _rows(M, 24, 5)
    Cr, S = Gm.gemm_ref_rows(qx["codes"], qx["scales"], qx["amax"], qw["codes"], qw["scales"], qw["amax"], fmt, rows)
    got = host(C)[rows]
    assert (np.abs(got - Cr) <= Gm.gemm_bound(S)).all()


# ---------------------------------------------------------------------------
# Weight-only decode (Qwen2.5-7B-like MLP shapes) at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wname", ["W_up", "W_down"])
def test_config5_fullsize(wname):
    from fp4_block_scaled_amax_gb300 import synth
    from gpu_util import dev, host
    fp4 = lib()
    W = synth.config5(1)[wname]
    N, K = W.shape
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(N * K // 16, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    fp4.fp4_quantize(dev(W), "E4M3", fp4.FP4_ROUND_RNE, 0, None, False, fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax)
    ref = Q.quantize(W.float().numpy(), "E4M3", "rne", 0, chunk_rows=2048)
    assert np.array_equal(host(codes), ref["codes"])
    assert np.array_equal(host(scales).reshape(N, -1), ref["scales"])
    for b in (1, 8, 64):
        xk = "x_up" if wname == "W_up" else "x_down"
        x = synth.config5(b)[xk]
        y = torch.empty((b, N), dtype=torch.bfloat16, device="cuda")
        fp4.fp4_gemv_w4a16(codes, scales, amax, dev(x), b, N, K, fp4.FP4_OUT_BF16, y)
        yr, S = Gm.gemv_ref(ref["codes"], ref["scales"], ref["amax"], x.float().numpy())
        got = host(y.float())
        bound = Gm.gemm_bound(S) + np.abs(yr) * 2.0 ** -8
        assert (np.abs(got - yr) <= bound).all(), (wname, b)


# ---------------------------------------------------------------------------
# 16 x 16 random Hadamard transform on the dual quantizer at full size
# ---------------------------------------------------------------------------

def test_dual_rht_fullsize_sampled(step):
    from oracle import rht as R
    from gpu_util import host
    bench, d, s = step
    fp4 = s.fp4
    mask = bench.RHT_MASK
    x = d["dY"]
    M, K = x.shape
    cr, srs, cc, scs = (torch.empty_like(t) for t in s.q["dY"])
    amax = torch.zeros(2, dtype=torch.float32, device=s.dY.device)
    st = torch.zeros(1, dtype=torch.int32, device=s.dY.device)
    SR = fp4.FP4_ROUND_STOCHASTIC
    fp4.fp4_quantize_dual_rht(s.dY, "E4M3", SR, 1234, SR, 1235, mask, None, None, fp4.FP4_SFLAYOUT_MMA,
                              cr, srs, cc, scs, amax[0:1], amax[1:2], st)
    a = host(amax)
    assert int(host(st)[0]) == 0
    xf = x.float().numpy()
    rows_t = R.rht16(xf, mask)                 # blocks along K
    g_row = np.float32(np.max(np.abs(rows_t)))
    assert a[0] == g_row
    cols_t = R.rht16(np.ascontiguousarray(xf.T), mask)  # blocks along M, one row per column of dY
    del xf
    g_col = np.float32(np.max(np.abs(cols_t)))
    assert a[1] == g_col
    cr, srs, cc, scs = host(cr), host(srs), host(cc), host(scs)
    srow, scol = from_mma(srs, M, K // 16), from_mma(scs, K, M // 16)
    for r in _rows(M, 8, 6):
        codes, scales = Q.quantize_rows(rows_t[r:r + 1], "E4M3", "sr", 1234, g_row, row0=int(r))
        assert np.array_equal(cr[r], codes[0]) and np.array_equal(srow[r], scales[0]), ("row", r)
    for c in _rows(K, 8, 7):
        codes, scales = Q.quantize_rows(cols_t[c:c + 1], "E4M3", "sr", 1235, g_col, row0=int(c))
        assert np.array_equal(cc[c], codes[0]) and np.array_equal(scol[c], scales[0]), ("col", c)


# ---------------------------------------------------------------------------
# Quantizing epilogue and UE5M3 windows at the forward GEMM's full size
# ---------------------------------------------------------------------------

def test_gemm_quantize_epilogue_fullsize_identical(step):
    # fp4_gemm_quantize == fp4_gemm (bf16 Y) followed by fp4_quantize of Y's rows,
    # byte for byte, with Y's stored amax (RNE and SR)
    bench, d, s = step
    fp4 = s.fp4
    M, N, K = bench.M_TOK, bench.N_FFN, bench.K_HID
    qX, qW = s.q["X"], s.q["W"]
    aX, aW = s.amax[0:1], s.amax[1:2]
    dev = s.Y.device
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", fp4.FP4_OUT_BF16, Y)
    gY = Y.float().abs().max().reshape(1)
    for rnd, seed in ((fp4.FP4_ROUND_RNE, 0), (fp4.FP4_ROUND_STOCHASTIC, 77)):
        c1, s1 = torch.empty((M, N // 2), dtype=torch.uint8, device=dev), torch.empty(M * N // 16, dtype=torch.uint8,
                                                                                     device=dev)
        c2, s2 = torch.empty_like(c1), torch.empty_like(s1)
        fp4.fp4_quantize(Y, "E4M3", rnd, seed, gY, False, fp4.FP4_SFLAYOUT_MMA, c1, s1, None)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        fp4.fp4_gemm_quantize(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", gY, rnd, seed,
                              fp4.FP4_SFLAYOUT_MMA, c2, s2, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(c1, c2) and torch.equal(s1, s2), rnd


def test_gemm_quantize_dual_epilogue_fullsize_identical(step):
    # fp4_gemm_quantize_dual on the forward GEMM: row blocks == fp4_quantize(Y),
    # column blocks == fp4_quantize(Y, transpose = 1), byte for byte
    bench, d, s = step
    fp4 = s.fp4
    M, N, K = bench.M_TOK, bench.N_FFN, bench.K_HID
    qX, qW = s.q["X"], s.q["W"]
    aX, aW = s.amax[0:1], s.amax[1:2]
    dev = s.Y.device
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", fp4.FP4_OUT_BF16, Y)
    gY = Y.float().abs().max().reshape(1)
    RNE, SR, MMA = fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC, fp4.FP4_SFLAYOUT_MMA
    rc, rs = torch.empty((M, N // 2), dtype=torch.uint8, device=dev), torch.empty(M * N // 16, dtype=torch.uint8,
                                                                                 device=dev)
    tc, ts = torch.empty((N, M // 2), dtype=torch.uint8, device=dev), torch.empty_like(rs)
    fp4.fp4_quantize(Y, "E4M3", RNE, 0, gY, False, MMA, rc, rs, None)
    fp4.fp4_quantize(Y, "E4M3", SR, 91, gY, True, MMA, tc, ts, None)
    fc, fs, ftc, fts = torch.empty_like(rc), torch.empty_like(rs), torch.empty_like(tc), torch.empty_like(ts)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    fp4.fp4_gemm_quantize_dual(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", gY, RNE, 0, SR, 91,
                               MMA, fc, fs, ftc, fts, amax, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(fc, rc) and torch.equal(fs, rs)
    assert torch.equal(ftc, tc) and torch.equal(fts, ts)
    assert float(amax) == float(gY)


def test_ue5m3_windows_fullsize_one_window_identical(step):
    # X and W quantized with UE5M3 scales (fresh amaxes) fit one window: the window
    # GEMM equals the single-shift GEMM bit for bit at 16384 x 11008 x 4096
    bench, d, s = step
    fp4 = s.fp4
    M, N, K = bench.M_TOK, bench.N_FFN, bench.K_HID
    dev = s.Y.device
    i32 = dict(dtype=torch.int32, device=dev)
    ops = []
    for x, a in ((s.X, s.amax[0:1]), (s.W, s.amax[1:2])):
        R = x.shape[0]
        codes = torch.empty((R, K // 2), dtype=torch.uint8, device=dev)
        sc = torch.empty(R * K // 16, dtype=torch.uint8, device=dev)
        fp4.fp4_quantize(x, "UE5M3", fp4.FP4_ROUND_RNE, 0, a, False, fp4.FP4_SFLAYOUT_MMA, codes, sc, None)
        t, e4 = torch.zeros(1, **i32), torch.empty_like(sc)
        fp4.fp4_ue5m3_to_e4m3(sc, t, e4)
        tw, nw, win = torch.zeros(3, **i32), torch.zeros(1, **i32), torch.empty(3 * sc.numel(), dtype=torch.uint8,
                                                                             device=dev)
        fp4.fp4_ue5m3_windows(sc, tw, nw, win)
        ops.append((codes, a, t, e4, tw, nw, win))
    (xc, xa, xt, xe, xtw, xn, xw), (wc, wa, wt, we, wtw, wn, ww) = ops
    C1 = torch.empty((M, N), dtype=torch.float32, device=dev)
    C2 = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    fp4.fp4_gemm(xc, xe, wc, we, xa, wa, xt, wt, M, N, K, "UE5M3", fp4.FP4_OUT_F32, C1)
    st = torch.zeros(1, **i32)
    fp4.fp4_gemm_ue5m3_windows(xc, xw, xtw, xn, wc, ww, wtw, wn, xa, wa, M, N, K, C2, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(xn.item()) == 1 and int(wn.item()) == 1
    assert torch.equal(C1, C2)
