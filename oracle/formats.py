"""Element and block-scale number formats (oracle; test infrastructure only).

Formats named on the pages:

* E2M1, the FP4 element ("NVFP4 vs MXFP" post, quant_prune_distill #486,
  section "Метод", item 1: NVFP4 is FP4 E2M1).  Value set
  +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E4M3, the NVFP4 block scale (same post and item).
* E8M0, the MXFP4 block scale: a pure power of two, so scale operations are
  bit shifts (same post, item 2).
* UE5M3, an unsigned 8-bit scale whose bits all go to a 5-bit exponent and a
  3-bit fraction, never negative ("UE5M3 FP4 Block Scaling ..." blog,
  section "Что сделали").
* E1M6 ... E8M0 at group 16, the scale-format sweep of the FP4 training review
  (gonzo_ML #3986, section "Форматы FP4"); E1M6 has the narrowest range.

Readings taken where the pages are silent (each is one fixed choice):

* Generic ExMy rule: one sign bit unless the format is unsigned, exponent bias
  2^(E-1)-1 unless stated, IEEE-style subnormals at exponent field 0, every
  code finite except the NaN codes the format names; no infinities.
* E4M3 is the OCP FP8 "FN" variant: bias 7, subnormals m*2^-9, max 448, only
  S.1111.111 is NaN.
* UE5M3: bias 15, subnormals m/8*2^-14, 0xFF is NaN (never produced), max
  finite 0xFE = 1.75*2^16 = 114688.
* E8M0: bias 127, value 2^(c-127), 0xFF is NaN, no zero and no subnormals.
* E1M6: bias 0, subnormals m/32, all codes finite, max 3.96875.
* Encoding a block scale is round-to-nearest with ties to the even code,
  saturating at the largest finite code (the scale never becomes NaN).
"""

from __future__ import annotations

import dataclasses

import numpy as np

# ---------------------------------------------------------------------------
# Generic ExMy decoder
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class ExMy:
    """A small floating-point format with `ebits` exponent and `mbits` mantissa bits."""

    name: str
    ebits: int
    mbits: int
    bias: int
    signed: bool
    nan_codes: tuple = ()
    power_of_two_only: bool = False  # E8M0: value 2^(e-bias) for every code, no zero

    @property
    def nbits(self) -> int:
        return int(self.signed) + self.ebits + self.mbits

    def decode_code(self, code: int) -> float:
        """Value of one code as a Python float (exact: every value fits in binary64)."""
        if code in self.nan_codes:
            return float("nan")
        m = code & ((1 << self.mbits) - 1)
        e = (code >> self.mbits) & ((1 << self.ebits) - 1)
        neg = self.signed and (code >> (self.ebits + self.mbits)) & 1
        if self.power_of_two_only:
            mag = 2.0 ** (e - self.bias)
        elif e == 0:  # subnormal: no implicit leading one, exponent 1-bias
            mag = (m / (1 << self.mbits)) * 2.0 ** (1 - self.bias)
        else:
            mag = (1.0 + m / (1 << self.mbits)) * 2.0 ** (e - self.bias)
        return -mag if neg else mag

    def table(self) -> np.ndarray:
        """float64 value of every code 0 .. 2^nbits-1 (NaN for NaN codes)."""
        return np.array([self.decode_code(c) for c in range(1 << self.nbits)], dtype=np.float64)

    def nonneg_codes(self) -> np.ndarray:
        """Finite codes with a clear sign bit, in code order."""
        limit = 1 << (self.ebits + self.mbits)
        return np.array([c for c in range(limit) if c not in self.nan_codes], dtype=np.int64)

    def max_finite(self) -> float:
        t = self.table()
        return float(np.nanmax(t))


E2M1 = ExMy("E2M1", ebits=2, mbits=1, bias=1, signed=True)
E4M3 = ExMy("E4M3", ebits=4, mbits=3, bias=7, signed=True, nan_codes=(0x7F, 0xFF))
UE5M3 = ExMy("UE5M3", ebits=5, mbits=3, bias=15, signed=False, nan_codes=(0xFF,))
E8M0 = ExMy("E8M0", ebits=8, mbits=0, bias=127, signed=False, nan_codes=(0xFF,), power_of_two_only=True)
E1M6 = ExMy("E1M6", ebits=1, mbits=6, bias=0, signed=True)

# The rest of the gonzo_ML #3986 sweep at group 16 (generic rule, no NaN codes).
SWEEP = {
    "E1M6": E1M6,
    "E2M5": ExMy("E2M5", ebits=2, mbits=5, bias=1, signed=True),
    "E3M4": ExMy("E3M4", ebits=3, mbits=4, bias=3, signed=True),
    "E4M3": E4M3,
    "E5M2": ExMy("E5M2", ebits=5, mbits=2, bias=15, signed=True),
    "E6M1": ExMy("E6M1", ebits=6, mbits=1, bias=31, signed=True),
    "E7M0": ExMy("E7M0", ebits=7, mbits=0, bias=63, signed=True),
}

# E2M1 magnitudes indexed by the 3-bit magnitude code.
E2M1_MAGNITUDES = np.array([E2M1.decode_code(c) for c in range(8)], dtype=np.float64)

# ---------------------------------------------------------------------------
# Block-scale encoding: nearest finite non-negative code, ties to even code,
# saturating at the largest finite code.
# ---------------------------------------------------------------------------


class ScaleCodec:
    """Round-to-nearest-even, saturating encoder for a non-negative scale format."""

    def __init__(self, fmt: ExMy):
        self.fmt = fmt
        codes = fmt.nonneg_codes()
        vals = np.array([fmt.decode_code(int(c)) for c in codes], dtype=np.float64)
        # Non-negative codes of every format here are ordered by value; the
        # neighbour search below relies on it.
        assert np.all(np.diff(vals) > 0), f"{fmt.name}: non-negative codes not monotone"
        self.codes = codes
        self.vals = vals
        self.table = fmt.table()

    def encode(self, v: np.ndarray) -> np.ndarray:
        """Codes (uint8) of non-negative float values `v` (float32 or float64).

        The nearest representable value wins; at an exact tie the even code wins;
        anything above the largest finite value gives the largest finite code.
        """
        v = np.asarray(v, dtype=np.float64)
        if np.any(~(v >= 0)):
            raise ValueError("scale values must be non-negative and not NaN")
        n = len(self.vals)
        hi = np.searchsorted(self.vals, v, side="left")  # first value >= v
        hi_c = np.minimum(hi, n - 1)
        lo_c = np.maximum(hi - 1, 0)
        d_hi = np.abs(self.vals[hi_c] - v)
        d_lo = np.abs(v - self.vals[lo_c])
        code_hi = self.codes[hi_c]
        code_lo = self.codes[lo_c]
        pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (code_lo % 2 == 0))
        out = np.where(pick_lo, code_lo, code_hi)
        out = np.where(hi >= n, self.codes[-1], out)  # beyond the max: saturate
        return out.astype(np.uint8)

    def decode(self, codes: np.ndarray) -> np.ndarray:
        """float64 values of codes."""
        return self.table[np.asarray(codes, dtype=np.int64)]


CODECS = {name: ScaleCodec(f) for name, f in
          [("E4M3", E4M3), ("UE5M3", UE5M3), ("E1M6", E1M6)] + list(SWEEP.items())}

# ---------------------------------------------------------------------------
# E2M1 element rounding
# ---------------------------------------------------------------------------


def e2m1_rne_magnitude(a: np.ndarray) -> np.ndarray:
    """3-bit magnitude code of |y| rounded to the nearest E2M1 value.

    Ties go to the even code, values above 6 saturate to 6 (code 7).  `a` holds
    non-negative magnitudes (float32 or float64; compared exactly).
    """
    a = np.asarray(a, dtype=np.float64)
    mags = E2M1_MAGNITUDES
    hi = np.searchsorted(mags, a, side="left")
    hi_c = np.minimum(hi, 7)
    lo_c = np.maximum(hi - 1, 0)
    d_hi = np.abs(mags[hi_c] - a)
    d_lo = np.abs(a - mags[lo_c])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo_c % 2 == 0))
    out = np.where(pick_lo, lo_c, hi_c)
    out = np.where(hi > 7, 7, out)
    return out.astype(np.uint8)


def e2m1_floor_magnitude(a: np.ndarray) -> np.ndarray:
    """3-bit code of the largest E2M1 magnitude <= a (a >= 0), 7 for a >= 6."""
    a = np.asarray(a, dtype=np.float64)
    return (np.searchsorted(E2M1_MAGNITUDES, a, side="right") - 1).astype(np.uint8)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of 4-bit E2M1 codes (bit 3 is the sign)."""
    codes = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAGNITUDES[codes & 7]
    return np.where(codes & 8, -mag, mag)


# ---------------------------------------------------------------------------
# fp32 bit helpers
# ---------------------------------------------------------------------------


def f32_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def f32_sign_bit(x: np.ndarray) -> np.ndarray:
    """1 where the float32 sign bit is set (including -0.0)."""
    return (f32_bits(x) >> 31).astype(np.uint8)


def f32_floor_log2_biased(a: np.ndarray) -> np.ndarray:
    """Biased fp32 exponent field of a (0 for zero and subnormals).

    For a normal positive float32 a this is floor(log2(a)) + 127, read from the
    bits, with no transcendental call.
    """
    return ((f32_bits(a) >> 23) & 0xFF).astype(np.int64)
