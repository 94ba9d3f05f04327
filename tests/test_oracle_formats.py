"""Pins of the oracle's number formats (CPU only)."""

import math

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quantize as Q
from golden_io import rows


def test_e2m1_table_matches_golden():
    for code, val in rows("e2m1_values.txt"):
        c = int(code, 16)
        v = float(val)
        got = F.E2M1.decode_code(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (code, got, v)
    assert np.array_equal(F.E2M1_MAGNITUDES, [0, 0.5, 1, 1.5, 2, 3, 4, 6])


def test_e2m1_rne_ties_golden():
    for y, code in rows("e2m1_rne_ties.txt"):
        assert F.e2m1_rne_magnitude(np.array([float(y)]))[0] == int(code), y


def test_e2m1_encode_decode_identity_and_bruteforce():
    # every magnitude encodes to itself
    assert np.array_equal(F.e2m1_rne_magnitude(F.E2M1_MAGNITUDES), np.arange(8))
    # brute force: nearest of the 8 magnitudes by exhaustive comparison, ties -> even code
    rng = np.random.default_rng(7)
    ys = np.concatenate([rng.uniform(0, 8, 20000), np.arange(0, 7.01, 0.125)])
    got = F.e2m1_rne_magnitude(ys)
    for y, g in zip(ys, got):
        d = [abs(y - v) for v in F.E2M1_MAGNITUDES]
        best = min(d)
        cands = [c for c in range(8) if d[c] == best]
        want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        assert g == want, (y, g, want)


def test_e2m1_floor():
    assert list(F.e2m1_floor_magnitude(np.array([0, 0.49, 0.5, 0.99, 1, 5.9, 6, 100]))) == \
        [0, 0, 1, 1, 2, 6, 7, 7]


@pytest.mark.parametrize("name", ["E4M3", "UE5M3", "E8M0", "E1M6"])
def test_scale_format_extremes_golden(name):
    rec = {r[0]: r[1:] for r in rows("scale_format_extremes.txt")}[name]
    fmt = {"E4M3": F.E4M3, "UE5M3": F.UE5M3, "E8M0": F.E8M0, "E1M6": F.E1M6}[name]
    t = fmt.table()
    assert t[int(rec[0], 16)] == float(rec[1])
    assert np.nanmax(t) == float(rec[1])
    assert t[int(rec[2], 16)] == float(rec[3])
    pos = t[(t > 0) & ~np.isnan(t)]
    assert pos.min() == float(rec[3])
    nans = set() if rec[4] == "-" else {int(c, 16) for c in rec[4].split(",")}
    assert set(np.nonzero(np.isnan(t))[0].tolist()) == nans


def test_all_256_codes_each_scale_format():
    for fmt in (F.E4M3, F.UE5M3, F.E8M0, F.E1M6):
        t = fmt.table()
        assert len(t) == 256
        nn = fmt.nonneg_codes()
        vals = t[nn]
        assert np.all(np.diff(vals) > 0), fmt.name  # monotone on non-negative finite codes
    # UE5M3 has no sign bit: no code decodes negative ("UE5M3 ..." blog, "Что сделали")
    t = F.UE5M3.table()
    assert np.all((t >= 0) | np.isnan(t))
    # E8M0 is a pure power of two ("NVFP4 vs MXFP" post, item 2: scale ops are shifts)
    t = F.E8M0.table()
    for c in range(255):
        assert t[c] == 2.0 ** (c - 127)


def test_e4m3_and_e8m0_decode_match_torch():
    # independent library decoders: torch's float8_e4m3fn and float8_e8m0fnu
    u = torch.arange(256, dtype=torch.uint8)
    te = u.view(torch.float8_e4m3fn).float().double().numpy()
    oe = F.E4M3.table()
    assert np.array_equal(np.isnan(te), np.isnan(oe))
    ok = ~np.isnan(oe)
    assert np.array_equal(te[ok], oe[ok])
    te8 = u.view(torch.float8_e8m0fnu).float().double().numpy()
    o8 = F.E8M0.table()
    assert np.array_equal(np.isnan(te8), np.isnan(o8))
    assert np.array_equal(te8[~np.isnan(o8)], o8[~np.isnan(o8)])


@pytest.mark.parametrize("name", ["E4M3", "UE5M3", "E1M6", "E2M5", "E3M4", "E5M2", "E6M1", "E7M0"])
def test_scale_encode_roundtrip_and_bruteforce(name):
    codec = F.CODECS[name]
    # encode(decode(c)) == c for every finite non-negative code
    assert np.array_equal(codec.encode(codec.vals), codec.codes.astype(np.uint8))
    # brute-force nearest over all codes on random and midpoint values
    rng = np.random.default_rng(1)
    top = codec.vals[-1]
    mids = (codec.vals[1:] + codec.vals[:-1]) / 2
    v = np.concatenate([rng.uniform(0, top * 1.2, 3000),
                        np.exp(rng.uniform(np.log(codec.vals[1] / 4), np.log(top), 3000)),
                        mids, [0.0, top * 10]]).astype(np.float32).astype(np.float64)
    got = codec.encode(v)
    vals, codes = codec.vals, codec.codes
    for x, g in zip(v, got):
        d = np.abs(vals - x)
        best = d.min()
        c = codes[d == best]
        want = c[0] if len(c) == 1 else c[c % 2 == 0][0]
        assert g == want, (name, x, g, want)


def test_e4m3_encode_matches_torch_in_range():
    # torch's float32 -> float8_e4m3fn conversion rounds to nearest even; compare in range
    rng = np.random.default_rng(3)
    v = np.concatenate([np.exp(rng.uniform(np.log(2.0 ** -11), np.log(448.0), 50000)),
                        (F.CODECS["E4M3"].vals[1:] + F.CODECS["E4M3"].vals[:-1]) / 2]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.CODECS["E4M3"].encode(v)
    assert np.array_equal(got, want)


def test_storage_bits_per_param_golden():
    for fmt, group, bits in rows("storage_bits.txt"):
        assert Q.group_size(fmt) == int(group)
        R, C = 64, 1024
        cb, sb = Q.storage_bytes(R, C, fmt)
        assert (cb + sb) * 8 / (R * C) == float(bits)
