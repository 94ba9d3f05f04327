"""GPU quantizer vs the CPU oracle: codes and scales bit-exact (through the C ABI)."""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import formats as F
from oracle import philox as P
from oracle import quantize as Q
from gpu_util import dev, f32, from_mma, host, lib

pytestmark = pytest.mark.gpu

FMTS = ["E4M3", "UE5M3", "E8M0", "E1M6"]


def gpu_quant(x_bf16, fmt, rounding, seed, g=None, transpose=False, mma=False):
    fp4 = lib()
    x = dev(x_bf16)
    M, K = x.shape
    rows, cols = (K, M) if transpose else (M, K)
    G = Q.group_size(fmt)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows * cols // G,), dtype=torch.uint8, device="cuda")
    amax_out = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt = None if g is None else torch.tensor([g], dtype=torch.float32, device="cuda")
    fp4.fp4_quantize(x, fmt, fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE, seed, gt,
                     transpose, fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax_out, st)
    sc = host(scales)
    sc = from_mma(sc, rows, cols // G) if mma else sc.reshape(rows, cols // G)
    return host(codes), sc, float(host(amax_out)[0]), int(host(st)[0])


def check(x_bf16, fmt, rounding, seed, g=None, transpose=False, mma=False):
    c, s, a, st = gpu_quant(x_bf16, fmt, rounding, seed, g, transpose, mma)
    ref = Q.quantize(f32(x_bf16), fmt, rounding, seed, global_amax=g, transpose=transpose)
    assert st == 0
    assert np.array_equal(s, ref["scales"]), "scales differ"
    if not np.array_equal(c, ref["codes"]):
        bad = np.argwhere(c != ref["codes"])
        r, k = bad[0]
        raise AssertionError(f"{len(bad)} code bytes differ, first at {r},{k}: gpu {c[r, k]:#x} oracle "
                             f"{ref['codes'][r, k]:#x}")
    assert a == np.float32(ref["amax"])


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_rows_config1_shapes(fmt, rounding):
    d = synth.config1()
    check(d["A"], fmt, rounding, 1234)
    check(d["B"], fmt, rounding, 99)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_transposed_ragged(fmt, rounding):
    # 96 x 800: three 32-row tiles, a ragged fourth 256-column tile
    x = synth.normal((96, 800), 7, 0, outlier_p=0.01, outlier_mult=50.0)
    check(x, fmt, rounding, 5, transpose=True)
    check(x, fmt, rounding, 5, transpose=False)


@pytest.mark.parametrize("fmt", ["E4M3", "UE5M3", "E8M0"])
def test_mma_layout_and_stale_amax(fmt):
    x = synth.normal((256, 512), 8, 0, outlier_p=0.01, outlier_mult=50.0)
    g = float(x.float().abs().max()) / 3  # stale: true max 3x the stored one
    check(x, fmt, "rne", 0, g=g, mma=True)
    check(x, fmt, "sr", 3, g=g, transpose=True, mma=True)


def test_dual_matches_two_single_calls():
    fp4 = lib()
    for fmt in FMTS:
        G = Q.group_size(fmt)
        x = synth.normal((160, 544), 9, 0, outlier_p=0.01, outlier_mult=50.0)
        M, K = x.shape
        xd = dev(x)
        cr, sr = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda"), torch.empty(M * K // G, dtype=torch.uint8, device="cuda")
        cc, sc = torch.empty((K, M // 2), dtype=torch.uint8, device="cuda"), torch.empty(M * K // G, dtype=torch.uint8, device="cuda")
        amax = torch.zeros(1, dtype=torch.float32, device="cuda")
        fp4.fp4_quantize_dual(xd, fmt, fp4.FP4_ROUND_RNE, 11, fp4.FP4_ROUND_STOCHASTIC, 12, None,
                              fp4.FP4_SFLAYOUT_PLAIN, cr, sr, cc, sc, amax)
        ref_r = Q.quantize(f32(x), fmt, "rne", 11)
        ref_c = Q.quantize(f32(x), fmt, "sr", 12, transpose=True)
        assert np.array_equal(host(cr), ref_r["codes"]) and np.array_equal(host(sr).reshape(M, -1), ref_r["scales"])
        assert np.array_equal(host(cc), ref_c["codes"]) and np.array_equal(host(sc).reshape(K, -1), ref_c["scales"])
        assert float(host(amax)[0]) == ref_r["amax"]


def test_edge_cases():
    # zeros, a single outlier, exact E2M1 ties, bf16 subnormals, -0.0
    M, K = 64, 256
    x = np.zeros((M, K), dtype=np.float32)
    x[1, 0] = 1e30
    x[2, :16] = [6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, -6, -5, -3.5, -2.5, -1.75, -1.25, -0.75, -0.25]
    x[3, :] = -0.0
    x[4, :] = 9.2e-41  # bf16 subnormal
    x[5, :32] = np.linspace(-1, 1, 32)
    x[6, 5] = -3.0
    xb = synth.to_bf16(x)
    for fmt in FMTS:
        for rnd in ("rne", "sr"):
            check(xb, fmt, rnd, 77)
            check(xb, fmt, rnd, 77, g=6.0)
            check(xb, fmt, rnd, 77, transpose=True)


def test_amax_n_equals_single_calls():
    # three tensors in one launch (one strided, one empty) against max |x| and fp4_amax
    fp4 = lib()
    big = dev(synth.normal((384, 1040), 12, 0, outlier_p=0.01, outlier_mult=50.0))
    xs = [dev(synth.laplace((1000, 256), 12, 1, scale=1e-4)), big[:, :1024], dev(torch.zeros((0, 64)).bfloat16())]
    out = torch.full((3,), -1.0, dtype=torch.float32, device="cuda")
    fp4.fp4_amax_n(xs, out)
    got = host(out)
    for i, x in enumerate(xs):
        want = float(x.float().abs().max()) if x.numel() else 0.0
        one = torch.zeros(1, dtype=torch.float32, device="cuda")
        fp4.fp4_amax(x, one)
        assert got[i] == np.float32(want) == host(one)[0], i


def test_nonfinite_stored_amax_reports_status():
    x = synth.normal((32, 64), 1, 0)
    _, _, _, st = gpu_quant(x, "E4M3", "rne", 0, g=float("inf"))
    assert st == lib().FP4_ERR_NONFINITE


def test_empty_tensor_is_noop():
    fp4 = lib()
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((0, 32), dtype=torch.uint8, device="cuda")
    s = torch.empty((0,), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, device="cuda")
    fp4.fp4_quantize(x, "E4M3", 0, 0, g, False, 0, c, s)
    torch.cuda.synchronize()


def test_scale_encoder_conformance():
    # every scale code boundary: midpoints, codes, and a dense sweep of float32 values
    fp4 = lib()
    for fmt in ["E4M3", "UE5M3", "E1M6"]:
        codec = F.CODECS[fmt]
        v = codec.vals
        mids = (v[1:] + v[:-1]) / 2
        rng = np.random.default_rng(0)
        sweep = np.exp(rng.uniform(np.log(v[1] / 8), np.log(v[-1] * 4), 2_000_000))
        s = np.concatenate([v, mids, np.nextafter(mids.astype(np.float32), 0), np.nextafter(mids.astype(np.float32), np.inf),
                            sweep, [0.0, np.inf, 3.4e38]]).astype(np.float32)
        codes = torch.empty(len(s), dtype=torch.uint8, device="cuda")
        dec = torch.empty(len(s), dtype=torch.float32, device="cuda")
        fp4.fp4_encode_scales(dev(s), fmt, codes, dec)
        want = codec.encode(s.astype(np.float64))
        assert np.array_equal(host(codes), want), fmt
        assert np.array_equal(host(dec), codec.decode(want).astype(np.float32)), fmt
    # E8M0 takes block amaxes
    a = np.concatenate([np.exp(np.random.default_rng(1).uniform(-85, 85, 100000)), [0, 1e-45, 4.0, 8.0]]).astype(np.float32)
    codes = torch.empty(len(a), dtype=torch.uint8, device="cuda")
    dec = torch.empty(len(a), dtype=torch.float32, device="cuda")
    fp4.fp4_encode_scales(dev(a), "E8M0", codes, dec)
    want, wv = Q.block_scales(a, np.float32(1), "E8M0")
    assert np.array_equal(host(codes), want)
    assert np.array_equal(host(dec), wv)


def test_philox_matches_oracle_10M():
    fp4 = lib()
    n = 10_000_000
    for seed, start in [(1234, 0), (0xDEADBEEFCAFEF00D, (1 << 35) - 4096)]:
        out = torch.empty(n, dtype=torch.int16, device="cuda")
        fp4.fp4_philox_bits16(seed, start, n, out)
        got = host(out).view(np.uint16)
        idx = np.arange(start, start + n, dtype=np.uint64)
        want = np.concatenate([P.sr_bits16(seed, idx[i:i + 1_000_000]) for i in range(0, n, 1_000_000)])
        assert np.array_equal(got.astype(np.uint32), want)


# ---------------------------------------------------------------------------
# The rest of the group-16 scale-format sweep (row quantization only)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_sweep_formats_rows(fmt, rounding):
    # the 350M-parameter MLP input recipe (per-column sigma log-uniform in
    # [0.1, 10]) at 1/8 size, plain and tiled scale layouts, fresh and stale amax
    x = synth.config2(scale=8)["X"]
    check(x, fmt, rounding, 77)
    check(x, fmt, rounding, 78, mma=True)
    check(x, fmt, rounding, 79, g=float(x.float().abs().max()) / 5)


@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
def test_sweep_formats_dequantize(fmt):
    fp4 = lib()
    x = synth.config2(scale=8)["X"]
    M, K = x.shape
    ref = Q.quantize(f32(x), fmt, "rne", 0)
    g = torch.tensor([ref["amax"]], dtype=torch.float32, device="cuda")
    out = torch.empty((M, K), dtype=torch.float32, device="cuda")
    fp4.fp4_dequantize(dev(ref["codes"]), dev(ref["scales"].reshape(-1)), fp4.FP4_SFLAYOUT_PLAIN, M, K, fmt, g,
                       fp4.FP4_OUT_F32, out)
    assert np.array_equal(host(out), Q.dequantize(ref["codes"], ref["scales"], fmt, ref["amax"]))


@pytest.mark.parametrize("fmt", Q.SWEEP_FORMATS)
def test_sweep_formats_encode_every_code(fmt):
    # every non-negative code's value, its neighbours' midpoints and values just
    # around them encode as the oracle's nearest-even, saturating rule does
    fp4 = lib()
    vals = F.CODECS[fmt].vals
    mids = (vals[1:] + vals[:-1]) / 2
    probe = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                            np.nextafter(mids.astype(np.float32), np.float32(np.inf)), [vals[-1] * 2, 3e38]])
    probe = probe.astype(np.float32)
    s = torch.from_numpy(probe).cuda()
    codes = torch.empty(probe.size, dtype=torch.uint8, device="cuda")
    dec = torch.empty(probe.size, dtype=torch.float32, device="cuda")
    fp4.fp4_encode_scales(s, fmt, codes, dec)
    want = F.CODECS[fmt].encode(probe)
    assert np.array_equal(host(codes), want)
    assert np.array_equal(host(dec), F.CODECS[fmt].decode(want).astype(np.float32))


@pytest.mark.parametrize("fmt", ["NVINT4", "MXINT4"])
@pytest.mark.parametrize("rounding", ["rne", "sr"])
def test_int4_grids_rows(fmt, rounding):
    x = synth.config2(scale=8)["X"]
    check(x, fmt, rounding, 81)
    check(x, fmt, rounding, 82, mma=True)
    check(x, fmt, rounding, 83, g=float(x.float().abs().max()) / 5)
    y = synth.normal((128, 512), 10, 0, outlier_p=0.01, outlier_mult=50.0)
    check(y, fmt, rounding, 84)


@pytest.mark.parametrize("fmt", ["NVINT4", "MXINT4"])
def test_int4_grids_dequantize(fmt):
    fp4 = lib()
    x = synth.config2(scale=8)["X"]
    M, K = x.shape
    ref = Q.quantize(f32(x), fmt, "sr", 5)
    g = torch.tensor([ref["amax"]], dtype=torch.float32, device="cuda")
    out = torch.empty((M, K), dtype=torch.float32, device="cuda")
    fp4.fp4_dequantize(dev(ref["codes"]), dev(ref["scales"].reshape(-1)), fp4.FP4_SFLAYOUT_PLAIN, M, K, fmt, g,
                       fp4.FP4_OUT_F32, out)
    assert np.array_equal(host(out), Q.dequantize(ref["codes"], ref["scales"], fmt, ref["amax"]))
