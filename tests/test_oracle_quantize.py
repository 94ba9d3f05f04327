"""Pins of the oracle's quantizer (CPU only): closed forms, invariants, statistics."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import philox as P
from oracle import quantize as Q
from oracle.amax import AmaxState


def bf16(a):
    """Round float values to bf16 and return them as float32 (input preparation only)."""
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_global_encode_scale_closed_forms():
    assert Q.global_encode_scale(2688.0, "E4M3") == 1.0
    assert Q.global_encode_scale(1.0, "E4M3") == 2688.0
    assert Q.global_encode_scale(1.0, "UE5M3") == 2688.0
    assert Q.global_encode_scale(1.0, "E1M6") == np.float32(23.8125)
    assert Q.global_encode_scale(0.0, "E4M3") == 1.0
    assert Q.global_encode_scale(1e-45, "E4M3") == np.finfo(np.float32).max
    assert Q.global_encode_scale(123.0, "E8M0") == 1.0
    assert Q.global_encode_scale(3.0, "E4M3") == np.float32(896.0)
    with pytest.raises(Q.NonFiniteAmax):
        Q.global_encode_scale(float("inf"), "E4M3")
    with pytest.raises(Q.NonFiniteAmax):
        Q.global_encode_scale(float("nan"), "UE5M3")


def test_all_ones_block_closed_form():
    # x = 1 everywhere, fresh amax 1: s_enc = 2688, s_real = 448 -> code 0x7E, y = 6 -> code 7
    x = np.ones((4, 64), dtype=np.float32)
    q = Q.quantize(x, "E4M3")
    assert np.all(q["scales"] == 0x7E)
    assert np.all(q["codes"] == 0x77)
    assert np.array_equal(Q.dequantize(q["codes"], q["scales"], "E4M3", 1.0), x)
    # negative ones: sign bit set in both nibbles
    q = Q.quantize(-x, "E4M3")
    assert np.all(q["codes"] == 0xFF)


def test_mxfp4_closed_form():
    # block max 4.0 -> floor(log2 4) - 2 = 0 -> code 127, s_b = 1, y = x
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 4.0
    x[0, 1:9] = [0.5, 1, 1.5, 2, 3, -4, -6, 0.25]
    q = Q.quantize(x, "E8M0")
    assert q["scales"][0, 0] == 127
    codes = Q.unpack(q["codes"])[0]
    assert list(codes[:9]) == [6, 1, 2, 3, 4, 5, 0xE, 0xF, 0]
    # block max 100 -> floor(log2 100) = 6 -> code 131, s_b = 16, y = 6.25 -> 6
    x[0, 0] = 100.0
    q = Q.quantize(x, "E8M0")
    assert q["scales"][0, 0] == 131
    assert Q.unpack(q["codes"])[0][0] == 7


def test_nibble_order_and_signed_zero():
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 0] = 6.0
    x[0, 1] = -0.0
    x[0, 2] = -1e-3   # rounds to zero, keeps its sign
    x[0, 3] = 3.0
    q = Q.quantize(x, "E4M3", global_amax=6.0)
    assert q["codes"][0, 0] == (0x7 | (0x8 << 4))
    assert q["codes"][0, 1] == (0x8 | (0x5 << 4))


def test_zero_and_flushed_blocks():
    x = np.zeros((2, 32), dtype=np.float32)
    x[1, :16] = -1e-6          # block amax far below the global amax: scale flushes to 0
    x[1, 16] = 1.0
    q = Q.quantize(x, "E4M3")
    assert np.all(q["scales"][0] == 0)
    assert q["scales"][1, 0] == 0
    assert np.all(Q.unpack(q["codes"])[1, :16] == 0x8)
    assert np.all(Q.unpack(q["codes"])[0] == 0)


def _data(seed, shape, outliers=0.01):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    m = rng.random(shape) < outliers
    x[m] *= 50
    return bf16(x)


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
def test_block_max_code_invariant(fmt):
    # Every block whose scale is non-zero and not subnormal contains |code| = 6
    # (E4M3/UE5M3: scale rounding error <= 1/16 puts y_max above 5) or
    # |code| in {4, 6} (E8M0: y_max in [4, 8)).
    x = _data(0, (256, 512))
    q = Q.quantize(x, fmt)
    G = Q.group_size(fmt)
    mag = (Q.unpack(q["codes"]) & 7).reshape(256, 512 // G, G).max(axis=2)
    s = Q.scale_values(q["scales"], fmt)
    if fmt == "E8M0":
        assert np.all(np.isin(mag, [6, 7]))
    else:
        normal = s >= {"E4M3": 2.0 ** -6, "UE5M3": 2.0 ** -14}[fmt]
        assert normal.mean() > 0.99
        assert np.all(mag[normal] == 7)


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
def test_requantize_fixed_point(fmt):
    # quantize(bf16(dequantize(q))) == q under the same global amax, on blocks with
    # a normal scale
    x = _data(1, (128, 512))
    q = Q.quantize(x, fmt)
    xd = bf16(Q.dequantize(q["codes"], q["scales"], fmt, q["amax"]))
    q2 = Q.quantize(xd, fmt, global_amax=q["amax"])
    G = Q.group_size(fmt)
    s = Q.scale_values(q["scales"], fmt)
    normal = s >= {"E4M3": 2.0 ** -6, "UE5M3": 2.0 ** -14, "E8M0": 0}[fmt]
    assert np.array_equal(q2["scales"][normal], q["scales"][normal])
    c1 = Q.unpack(q["codes"]).reshape(128, -1, G)[normal]
    c2 = Q.unpack(q2["codes"]).reshape(128, -1, G)[normal]
    assert np.array_equal(c1, c2)


def test_ue5m3_equals_e4m3_where_e4m3_normal():
    x = _data(2, (256, 256))
    a = Q.quantize(x, "E4M3")
    b = Q.quantize(x, "UE5M3")
    sa = Q.scale_values(a["scales"], "E4M3")
    sb = Q.scale_values(b["scales"], "UE5M3")
    normal = (sa >= 2.0 ** -6) & (sa < 448)
    assert normal.mean() > 0.99
    assert np.array_equal(sa[normal], sb[normal])
    ca = Q.unpack(a["codes"]).reshape(256, -1, 16)[normal]
    cb = Q.unpack(b["codes"]).reshape(256, -1, 16)[normal]
    assert np.array_equal(ca, cb)


def test_stale_amax_e4m3_saturates_ue5m3_absorbs():
    # stored amax 4x below the true one ("UE5M3 ..." blog, "Что сделали": the tensor
    # maximum is refreshed once every 50 steps; large values must not be clipped)
    x = _data(3, (64, 256))
    g = float(np.max(np.abs(x))) / 4
    a = Q.quantize(x, "E4M3", global_amax=g)
    b = Q.quantize(x, "UE5M3", global_amax=g)
    assert np.any(Q.scale_values(a["scales"], "E4M3") == 448.0)
    assert np.all(Q.scale_values(b["scales"], "UE5M3") < 114688.0)
    ea = np.abs(Q.dequantize(a["codes"], a["scales"], "E4M3", g) - x).max()
    eb = np.abs(Q.dequantize(b["codes"], b["scales"], "UE5M3", g) - x).max()
    assert eb < ea / 4


def test_e1m6_narrow_range_direction():
    # gonzo_ML #3986, "Форматы FP4": of the scale-format sweep only E1M6, the one
    # with the narrowest range, fails.  Under the global scale a block flushes to
    # zero when its scale rounds below half the smallest positive scale:
    #   E1M6: 3.96875 * a_b / g < 1/64   (a_b/g < 1/254)
    #   E4M3: 448 * a_b / g < 2^-10      (a_b/g < 2.2e-6)
    #   UE5M3: 448 * a_b / g < 2^-18     (a_b/g < 8.5e-9)
    # Rows whose scale spans four decades cross only E1M6's threshold.
    rng = np.random.default_rng(2)
    row_sig = 10.0 ** rng.uniform(-4, 0, 512)
    x = bf16(rng.standard_normal((512, 1024)) * row_sig[:, None])
    flushed = {}
    for fmt in ("E4M3", "UE5M3", "E1M6"):
        q = Q.quantize(x, fmt)
        blk_nonzero = np.abs(x).reshape(512, -1, 16).max(axis=2) > 0
        flushed[fmt] = float(np.mean((q["scales"] == 0) & blk_nonzero))
    assert flushed["E4M3"] == 0 and flushed["UE5M3"] == 0
    a_b = np.abs(x).reshape(512, -1, 16).max(axis=2)
    expect = float(np.mean(a_b / np.abs(x).max() < 1 / 254.5))
    assert flushed["E1M6"] > 0.1
    assert abs(flushed["E1M6"] - expect) < 0.01


def test_sr_rule_exact_thresholds():
    # y = 0.25 lies half-way between 0 and 0.5: up iff r < 32768
    ay = np.array([0.25, 0.25, 0.5, 0.5, 2.5, 2.5, 6.5], dtype=np.float32)
    r = np.array([32767, 32768, 0, 65535, 32767, 32768, 0], dtype=np.uint32)
    assert list(Q._round_sr(ay, r)) == [1, 0, 1, 1, 5, 4, 7]
    # on-grid values never move
    grid = np.repeat(F.E2M1_MAGNITUDES.astype(np.float32), 5)
    rr = np.tile(np.array([0, 1, 30000, 65534, 65535], dtype=np.uint32), 8)
    assert np.array_equal(Q._round_sr(grid, rr), np.repeat(np.arange(8), 5))


@pytest.mark.parametrize("y", [0.30078125, 0.8125, 1.1015625, 2.75, 4.5, 5.96875])
def test_sr_unbiased_4sigma(y):
    # MXFP4 block with max 4.0 has s_b = 1 and r_b = 1, so the element reaching the
    # rounder is x itself; 10^6 draws of SR(y) must average to y within 4 sigma
    # (gonzo_ML #3986, "Стохастическая квантизация": stochastic rounding reduces bias).
    n_blocks = 32258  # 31 draws per block -> ~10^6
    x = np.full((n_blocks, 32), y, dtype=np.float32)
    x[:, 0] = 4.0 if y <= 4 else 6.0
    q = Q.quantize(x, "E8M0", rounding="sr", seed=1234)
    s = Q.scale_values(q["scales"], "E8M0")
    assert np.all(s == 1.0)
    vals = F.e2m1_decode(Q.unpack(q["codes"]))[:, 1:].reshape(-1)
    lo = F.E2M1_MAGNITUDES[F.e2m1_floor_magnitude(np.array([y]))[0]]
    hi = F.E2M1_MAGNITUDES[F.e2m1_floor_magnitude(np.array([y]))[0] + 1]
    assert set(np.unique(vals)) <= {lo, hi}
    f = (y - lo) / (hi - lo)
    sigma = np.sqrt(f * (1 - f)) * (hi - lo) / np.sqrt(vals.size)
    assert abs(vals.mean() - y) < 4 * sigma
    assert abs(np.mean(vals == hi) - f) < 4 * np.sqrt(f * (1 - f) / vals.size)


def test_sr_depends_only_on_seed_and_index():
    x = _data(4, (64, 128))
    a = Q.quantize(x, "E4M3", rounding="sr", seed=77)
    b = Q.quantize(x, "E4M3", rounding="sr", seed=77, chunk_rows=7)
    c = Q.quantize(x, "E4M3", rounding="sr", seed=78)
    assert np.array_equal(a["codes"], b["codes"])
    assert not np.array_equal(a["codes"], c["codes"])
    r1 = Q.quantize(x, "E4M3", rounding="rne", seed=1)
    r2 = Q.quantize(x, "E4M3", rounding="rne", seed=2)
    assert np.array_equal(r1["codes"], r2["codes"])


def test_amax_refresh_every_50_steps():
    st = AmaxState(period=50)
    rng = np.random.default_rng(0)
    seen = []
    for t in range(101):
        x = (rng.standard_normal((8, 32)) * 1.02 ** t).astype(np.float32)
        g = st.amax_for_step(t, x)
        seen.append(g)
        if t in (0, 50, 100):
            assert g == np.max(np.abs(x))
        else:
            assert g == seen[t - 1]


def test_ue5m3_reencode_exact_for_fresh_amax():
    x = _data(5, (128, 256))
    q = Q.quantize(x, "UE5M3")
    t = Q.ue5m3_shift(q["scales"])
    assert t == 1  # fresh amax puts the largest scale at 448 (exponent 8)
    codes, exact = Q.ue5m3_reencode_e4m3(q["scales"], t)
    assert exact
    assert np.array_equal(F.CODECS["E4M3"].decode(codes) * 2.0 ** t,
                          Q.scale_values(q["scales"], "UE5M3"))


# ---------------------------------------------------------------------------
# Rest of the group-16 scale-format sweep (E2M5, E3M4, E5M2, E6M1, E7M0)
# ---------------------------------------------------------------------------

SWEEP_MIN_NORMAL = {"E2M5": 1.0, "E3M4": 2.0 ** -2, "E5M2": 2.0 ** -14, "E6M1": 2.0 ** -30, "E7M0": 2.0 ** -62}
# largest element magnitude code of a block with a normal scale: the scale's
# relative rounding error (at most 2^-(m+1)) bounds y_max = 6 s_real / s_b from below
SWEEP_MAX_CODES = {"E2M5": {7}, "E3M4": {7}, "E5M2": {7}, "E6M1": {6, 7}, "E7M0": {6, 7}}


@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
def test_sweep_global_scale_closed_forms(fmt):
    st = {"E2M5": 7.875, "E3M4": 31.0, "E5M2": 114688.0, "E6M1": 1.5 * 2.0 ** 32, "E7M0": 2.0 ** 64}[fmt]
    assert Q.SCALE_TARGET[fmt] == st
    assert Q.global_encode_scale(6 * st, fmt) == 1.0
    assert Q.global_encode_scale(1.0, fmt) == np.float32(6 * st)


@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
def test_sweep_amax_block_takes_the_top_code(fmt):
    # with the fresh amax, the block that holds it has s_real = S_T (up to one
    # float32 rounding), i.e. the largest finite scale code, and its largest
    # element becomes 6
    x = _data(2, (64, 256))
    q = Q.quantize(x, fmt)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert q["scales"][r, c // 16] == 0x7F
    assert (Q.unpack(q["codes"])[r, c] & 7) == 7


@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
def test_sweep_block_max_code_invariant(fmt):
    x = _data(0, (256, 512))
    q = Q.quantize(x, fmt)
    mag = (Q.unpack(q["codes"]) & 7).reshape(256, 32, 16).max(axis=2)
    normal = Q.scale_values(q["scales"], fmt) >= SWEEP_MIN_NORMAL[fmt]
    assert normal.any()
    assert np.all(np.isin(mag[normal], list(SWEEP_MAX_CODES[fmt])))


@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
def test_sweep_requantize_fixed_point(fmt):
    x = _data(1, (128, 512))
    q = Q.quantize(x, fmt)
    xd = bf16(Q.dequantize(q["codes"], q["scales"], fmt, q["amax"]))
    q2 = Q.quantize(xd, fmt, global_amax=q["amax"])
    # blocks with a normal scale whose largest element is 6: their re-derived
    # s_real is s_b exactly (a block topped by 4 re-derives (4/6) s_b, which a
    # coarse format may round to another code)
    top6 = (Q.unpack(q["codes"]) & 7).reshape(128, -1, 16).max(axis=2) == 7
    keep = (Q.scale_values(q["scales"], fmt) >= SWEEP_MIN_NORMAL[fmt]) & top6
    assert keep.any()
    assert np.array_equal(q2["scales"][keep], q["scales"][keep])
    c1 = Q.unpack(q["codes"]).reshape(128, -1, 16)[keep]
    c2 = Q.unpack(q2["codes"]).reshape(128, -1, 16)[keep]
    assert np.array_equal(c1, c2)


# ---------------------------------------------------------------------------
# INT4 element grids: NVINT4 (E4M3 scales, group 16), MXINT4 (E8M0, group 32)
# ---------------------------------------------------------------------------

def test_int4_closed_forms():
    x = np.ones((4, 64), dtype=np.float32)
    # NVINT4, fresh amax 1: s_enc = 7 * 448, s_real = 448 -> 0x7E, y = 7 -> nibble 0x7
    q = Q.quantize(x, "NVINT4")
    assert q["s_enc"] == np.float32(3136.0)
    assert np.all(q["scales"] == 0x7E) and np.all(q["codes"] == 0x77)
    q = Q.quantize(-x, "NVINT4")
    assert np.all(q["codes"] == 0x99)  # -7 in two's complement
    # MXINT4: integers with block maximum 4 keep scale 2^0 and their own values
    rng = np.random.default_rng(3)
    xi = rng.integers(-4, 5, (8, 64)).astype(np.float32)
    xi[:, ::32] = 4.0
    q = Q.quantize(xi, "MXINT4")
    assert np.all(q["scales"] == 127)
    assert np.array_equal(Q.element_values(Q.unpack(q["codes"]), "MXINT4"), xi)
    assert np.array_equal(Q.dequantize(q["codes"], q["scales"], "MXINT4", 0), xi)


def test_int4_rne_ties_and_no_negative_zero():
    # one NVINT4 block with amax 7 and g = 7: s_enc = 448, s_b = 448, r = 1 -> y = x
    x = np.array([[7, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, -0.25, -0.0, 6.5, -6.5, 4.5, 5.5, 0.75, -7]],
                 dtype=np.float32)
    q = Q.quantize(x, "NVINT4")
    assert q["scales"][0, 0] == 0x7E
    got = Q.element_values(Q.unpack(q["codes"]), "NVINT4")[0]
    assert np.array_equal(got, [7, 0, 2, 2, 0, -2, -2, 4, 0, 0, 6, -6, 4, 6, 1, -7])
    nib = Q.unpack(q["codes"])[0]
    assert nib[8] == 0 and nib[9] == 0  # -0.25 and -0.0 give code 0 (two's complement has no -0)


@pytest.mark.parametrize("fmt,mags", [("NVINT4", {7}), ("MXINT4", {4, 5, 6, 7})])
def test_int4_block_max_invariant(fmt, mags):
    x = _data(0, (256, 512))
    q = Q.quantize(x, fmt)
    G = Q.group_size(fmt)
    mag = np.abs(Q.element_values(Q.unpack(q["codes"]), fmt)).reshape(256, 512 // G, G).max(axis=2)
    s = Q.scale_values(q["scales"], fmt)
    normal = s >= (2.0 ** -6 if fmt == "NVINT4" else 0)
    assert normal.mean() > 0.99
    assert np.all(np.isin(mag[normal], list(mags)))


@pytest.mark.parametrize("y", [0.30078125, 1.8125, 3.5, 6.40625])
def test_int4_sr_unbiased_4sigma(y):
    n = 1 << 20
    r16 = P.sr_bits16(99, np.arange(n, dtype=np.uint64))
    v = Q._int_round_sr(np.full(n, y, dtype=np.float32), r16).astype(np.float64)
    lo = np.floor(y)
    p = y - lo
    sigma = np.sqrt(p * (1 - p) / n)
    assert abs(v.mean() - y) < 4 * sigma + 1e-12
    assert set(np.unique(v)) <= {lo, lo + 1}


# ---------------------------------------------------------------------------
# UE5M3 scales split into E4M3 windows (the multi-pass UE5M3 GEMM)
# ---------------------------------------------------------------------------

def _ue5m3_codes_of(values):
    c = F.CODECS["UE5M3"].encode(np.asarray(values, dtype=np.float64))
    assert np.array_equal(F.CODECS["UE5M3"].decode(c), values)
    return c


def test_ue5m3_windows_reconstruct_every_code():
    rng = np.random.default_rng(40)
    for top in (0xFE, 0xC3, 0x80, 0x41):  # different largest scales
        codes = np.arange(top + 1, dtype=np.uint8)
        rng.shuffle(codes)
        t, out, n = Q.ue5m3_windows(codes)
        v = F.CODECS["UE5M3"].decode(codes)
        rec = sum(F.CODECS["E4M3"].decode(out[k]) * 2.0 ** t[k] for k in range(3))
        assert np.array_equal(rec, v)
        assert np.array_equal((out > 0).sum(axis=0), (v > 0).astype(int))  # one window per nonzero scale
        assert t == [t[0], t[0] - 14, t[0] - 28] and t[0] == Q.ue5m3_shift(codes)
        # every window's E4M3 values are normal (or zero): exponents -6 .. 7
        for k in range(3):
            d = F.CODECS["E4M3"].decode(out[k])
            nz = d[d > 0]
            assert nz.size == 0 or (nz.min() >= 2.0 ** -6 and nz.max() < 2.0 ** 8)


def test_ue5m3_windows_single_window_is_the_single_shift():
    rng = np.random.default_rng(41)
    v = 2.0 ** rng.integers(-5, 9, 500) * rng.choice([1, 1.125, 1.5, 1.875], 500)  # 13 binades
    codes = _ue5m3_codes_of(v)
    t, out, n = Q.ue5m3_windows(codes)
    ref, exact = Q.ue5m3_reencode_e4m3(codes, Q.ue5m3_shift(codes))
    assert n == 1 and exact and np.array_equal(out[0], ref) and not out[1:].any()


@pytest.mark.parametrize("low,n", [(-13, 1), (-14, 2), (-27, 2), (-28, 3), (-33, 3)])
def test_ue5m3_window_count_closed_form(low, n):
    # largest scale 2^16, smallest 2^(16 + low): window of the smallest = floor(-low / 14)
    v = np.array([2.0 ** 16, 2.0 ** (16 + low), 0.0, 2.0 ** 16])
    t, out, nw = Q.ue5m3_windows(_ue5m3_codes_of(v))
    assert nw == n and t[0] == 16 - 7
    assert out[n - 1][1] != 0 and out[0][2] == 0


def test_windowed_gemm_equals_the_ue5m3_gemm():
    from oracle import gemm as Gm
    rng = np.random.default_rng(42)
    M, N, K = 24, 40, 128
    Aq = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    Bq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    As = _ue5m3_codes_of(2.0 ** rng.integers(-17, 17, (M, K // 16)) * 1.0)
    Bs = _ue5m3_codes_of(2.0 ** rng.integers(-10, 17, (N, K // 16)) * 1.5 / 1.5)
    ga, gb = 3.0, 0.25
    C, S = Gm.gemm_ref(Aq, As, ga, Bq, Bs, gb, "UE5M3")
    ta, wa, na = Q.ue5m3_windows(As)
    tb, wb, nb = Q.ue5m3_windows(Bs)
    assert na == 3 and nb == 2
    Cw = sum(Gm.gemm_ref(Aq, wa[i], ga, Bq, wb[j], gb, "E4M3")[0] * 2.0 ** (ta[i] + tb[j])
             for i in range(na) for j in range(nb))
    assert np.allclose(Cw, C, rtol=1e-12, atol=1e-12 * S.max())
