"""Two-level block-scaled FP4 quantizer (oracle; test infrastructure only).

What it follows:

* Block scaling with a per-block scale stored in low precision: "NVFP4 vs MXFP"
  post (quant_prune_distill #486, section "Метод": small groups with a shared
  scale, scales stored in low precision; NVFP4 = E2M1, group 16, E4M3 scale;
  MXFP4 = group 32, E8M0 scale).
* A per-16-element block scale and a whole-tensor maximum that may be stale
  between refreshes: "UE5M3 FP4 Block Scaling ..." blog, section "Что сделали".
* Nearest rounding for forward weights/activations, stochastic rounding (up or
  down, with a probability set by the distance to the neighbouring grid point)
  for backward tensors: gonzo_ML #3986, section "Стохастическая квантизация".

The pages print no formula; the steps below are the readings fixed for this
implementation (all float32 operations are single IEEE binary32 operations with
round-to-nearest-even; G is the group size):

1. Global encode scale  s_enc = f32(f32(6 * S_T) / g), g the stored tensor amax,
   S_T = 448 for E4M3 and UE5M3, otherwise the scale format's largest finite
   value (3.96875 for E1M6; 7.875, 31, 114688, 1.5*2^32 and 2^64 for the rest
   of the sweep E2M5, E3M4, E5M2, E6M1, E7M0); g == 0 -> 1; an overflow ->
   FLT_MAX.  E8M0 (MXFP4) uses no global scale: s_enc = 1.
2. Block amax a_b = max |x| over G consecutive elements along the last axis.
3. Block scale: s_real = f32(f32(a_b / 6) * s_enc), code = nearest scale code
   (ties to even code, saturating), s_b = value of code.
   E8M0 instead: code = clamp(floor(log2 a_b) - 2 + 127, 0, 254), the
   exponent read from the float32 bits (a_b == 0 -> 0); s_b = 2^(code-127).
4. Elements: if s_b == 0 every element becomes a signed zero; otherwise
   r_b = f32(s_enc / s_b), y = f32(x * r_b), and |y| is rounded to E2M1:
   nearest with ties to the even code (saturating at 6), or stochastically:
   with lo <= |y| < hi the neighbouring grid values, f = (|y|-lo)/(hi-lo), a
   16-bit draw r rounds up iff r < f * 2^16 (|y| >= 6 gives 6).
   The sign bit of each code is the sign bit of x (so -0.0 gives code 0x8).
5. Packing: byte j holds element 2j in its low nibble, element 2j+1 in its high
   nibble.  Scales: one byte per block, row-major [R, C/G].
6. Dequantization: f32(f32(e2m1 * s_b) / s_enc).

INT element grids (post on "INT v.s. FP: A Comprehensive Study of Fine-Grained
Low-bit Quantization Formats", quant_prune_distill channel page, section
"Метод": NVINT4 = groups of 16 with E4M3 scales, MXINT4 = groups of 32 with
E8M0 scales, on an INT grid instead of the FP one).  Readings fixed here: the grid is the
integers -7..7, stored as a 4-bit two's-complement nibble (no negative zero);
every "6" above becomes 7 (s_enc = f32(f32(7 * 448) / g) for NVINT4, s_real =
f32(f32(a_b / 7) * s_enc)); MXINT4's E8M0 block exponent is floor(log2 a_b) - 2
(2 = floor(log2 7)); rounding is nearest with ties to even, or stochastic with
the same 16-bit rule (up iff r < 65536 * frac(|y|)); |y| >= 7 gives 7.
"""

from __future__ import annotations

import numpy as np

from . import formats as F
from .philox import sr_bits16
from .rht import rht16

GROUP = {"E4M3": 16, "UE5M3": 16, "E1M6": 16, "E8M0": 32, "NVINT4": 16, "MXINT4": 32}
# INT4 element grid: the scale codec each INT format uses, and the element maximum
INT_SCALE = {"NVINT4": "E4M3", "MXINT4": "E8M0"}
SCALE_TARGET = {"E4M3": 448.0, "UE5M3": 448.0, "E1M6": 3.96875}
# the rest of the group-16 scale-format sweep (gonzo_ML #3986, "Форматы FP4"):
# generic ExMy scales, target = the format's largest finite value
SWEEP_FORMATS = ("E2M5", "E3M4", "E5M2", "E6M1", "E7M0")
for _name in SWEEP_FORMATS:
    GROUP[_name] = 16
    SCALE_TARGET[_name] = F.SWEEP[_name].max_finite()
SCALE_TARGET["NVINT4"] = 448.0


def is_int(fmt: str) -> bool:
    return fmt in INT_SCALE


def elem_max(fmt: str) -> float:
    """Largest element magnitude of the format's grid: 6 (E2M1) or 7 (INT4)."""
    return 7.0 if is_int(fmt) else 6.0


def scale_codec_name(fmt: str) -> str:
    return INT_SCALE.get(fmt, fmt)
FLT_MAX = np.float32(np.finfo(np.float32).max)


class NonFiniteAmax(ValueError):
    pass


def group_size(fmt: str) -> int:
    return GROUP[fmt]


def storage_bytes(rows: int, cols: int, fmt: str) -> tuple:
    """(code bytes, scale bytes) of an [rows, cols] tensor: 4 bits per element
    plus one 8-bit scale per group."""
    g = GROUP[fmt]
    if cols % g:
        raise ValueError("cols must be a multiple of the group size")
    return rows * cols // 2, rows * cols // g


def global_encode_scale(g, fmt: str) -> np.float32:
    """Step 1: the per-tensor float32 encode scale from the stored amax g."""
    if scale_codec_name(fmt) == "E8M0":
        return np.float32(1.0)
    g = np.float32(g)
    if not np.isfinite(g):
        raise NonFiniteAmax(f"global amax {g} is not finite")
    if g == 0:
        return np.float32(1.0)
    with np.errstate(over="ignore"):
        s = np.float32(np.float32(elem_max(fmt)) * np.float32(SCALE_TARGET[fmt])) / g
    if np.isinf(s):
        s = FLT_MAX
    return np.float32(s)


def block_scales(a_b: np.ndarray, s_enc: np.float32, fmt: str):
    """Step 3: scale codes (uint8) and their float32 values from block amaxes."""
    a_b = np.asarray(a_b, dtype=np.float32)
    emax = np.float32(elem_max(fmt))
    fmt = scale_codec_name(fmt)
    if fmt == "E8M0":
        e = F.f32_floor_log2_biased(a_b)  # floor(log2 a_b) + 127 for normals
        code = np.where(e > 0, e - 2, 0)
        code = np.clip(code, 0, 254).astype(np.uint8)
        s_b = np.ldexp(np.float32(1.0), code.astype(np.int32) - 127).astype(np.float32)
        return code, s_b
    s_real = np.float32(a_b / emax) * s_enc
    s_real = s_real.astype(np.float32)
    codec = F.CODECS[fmt]
    code = codec.encode(s_real)
    s_b = codec.decode(code).astype(np.float32)
    return code, s_b


def _round_rne(ay: np.ndarray) -> np.ndarray:
    return F.e2m1_rne_magnitude(ay)


def _round_sr(ay: np.ndarray, r16: np.ndarray) -> np.ndarray:
    """Stochastic E2M1 rounding of magnitudes ay (float32) with 16-bit draws r16."""
    ay64 = ay.astype(np.float64)
    lo_c = F.e2m1_floor_magnitude(ay64).astype(np.int64)
    sat = lo_c >= 7
    lo_c = np.minimum(lo_c, 6)
    lo = F.E2M1_MAGNITUDES[lo_c]
    hi = F.E2M1_MAGNITUDES[lo_c + 1]
    thresh = (ay64 - lo) / (hi - lo) * 65536.0  # exact: power-of-two step
    up = r16.astype(np.float64) < thresh
    out = lo_c + up.astype(np.int64)
    out = np.where(sat, 7, out)
    return out.astype(np.uint8)


def _int_round_rne(ay: np.ndarray) -> np.ndarray:
    """INT4 magnitude: nearest integer, ties to even, saturating at 7."""
    return np.minimum(np.rint(ay.astype(np.float64)), 7).astype(np.int64)


def _int_round_sr(ay: np.ndarray, r16: np.ndarray) -> np.ndarray:
    """INT4 magnitude by stochastic rounding with 16-bit draws (|y| >= 7 -> 7)."""
    ay64 = ay.astype(np.float64)
    lo = np.floor(ay64)
    up = r16.astype(np.float64) < (ay64 - lo) * 65536.0
    return np.minimum(lo + up, 7).astype(np.int64)


def quantize_rows(x: np.ndarray, fmt: str, rounding: str, seed: int, g,
                  row0: int = 0):
    """Quantize row blocks of a float32 array x [R, C] (bf16 values).

    Returns (codes [R, C/2] uint8, scales [R, C/G] uint8).  `row0` is the
    output-layout row index of x[0] (for Philox indices when x is a slab).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    G = GROUP[fmt]
    if C % G:
        raise ValueError("C must be a multiple of the group size")
    s_enc = global_encode_scale(g, fmt)
    xb = x.reshape(R, C // G, G)
    a_b = np.max(np.abs(xb), axis=2)
    scode, s_b = block_scales(a_b, s_enc, fmt)
    zero_blk = s_b == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r_b = np.where(zero_blk, np.float32(0), s_enc / np.where(zero_blk, np.float32(1), s_b))
    r_b = r_b.astype(np.float32)
    y = (xb * r_b[:, :, None]).astype(np.float32)
    ay = np.abs(y).reshape(R, C)
    if rounding == "rne":
        mag = _int_round_rne(ay) if is_int(fmt) else _round_rne(ay)
    elif rounding == "sr":
        idx = (np.arange(R, dtype=np.uint64)[:, None] + np.uint64(row0)) * np.uint64(C) \
            + np.arange(C, dtype=np.uint64)[None, :]
        r16 = sr_bits16(seed, idx)
        mag = _int_round_sr(ay, r16) if is_int(fmt) else _round_sr(ay, r16)
    else:
        raise ValueError(rounding)
    mag = np.where(np.repeat(zero_blk, G, axis=1), 0, mag)
    if is_int(fmt):
        # two's complement nibble of sign(x) * mag (no negative zero)
        q = (np.where(F.f32_sign_bit(x) == 1, -mag, mag) & 0xF).astype(np.uint8)
    else:
        q = mag.astype(np.uint8) | (F.f32_sign_bit(x) << 3)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, scode


def quantize(x: np.ndarray, fmt: str = "E4M3", rounding: str = "rne", seed: int = 0,
             global_amax=None, transpose: bool = False, chunk_rows: int = 1024, rht_mask=None):
    """Quantize x [M, K] (float32 holding bf16 values).

    global_amax None -> the fresh amax of x.  transpose=True quantizes x^T
    (blocks along the original rows; output layout [K, M], Philox indices in
    that layout).  rht_mask: apply the 16 x 16 random Hadamard transform with
    this sign mask to every 16-element block along the blocked dimension first
    (K for rows, M for transpose=True); the amax is then the transformed
    tensor's.  Returns dict(codes, scales, amax, s_enc).
    """
    x = np.asarray(x, dtype=np.float32)
    if rht_mask is not None:
        # transform along the blocked dimension: K for rows, M for the transposed output
        x = rht16(x.T, rht_mask).T if transpose else rht16(x, rht_mask)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    g = amax if global_amax is None else np.float32(global_amax)
    src = x.T if transpose else x
    R, C = src.shape
    G = GROUP[fmt]
    codes = np.empty((R, C // 2), dtype=np.uint8)
    scales = np.empty((R, C // G), dtype=np.uint8)
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        codes[r0:r1], scales[r0:r1] = quantize_rows(src[r0:r1], fmt, rounding, seed, g, row0=r0)
    return {"codes": codes, "scales": scales, "amax": amax,
            "s_enc": global_encode_scale(g, fmt)}


def unpack(codes: np.ndarray) -> np.ndarray:
    """[R, C/2] packed bytes -> [R, C] 4-bit codes (step 5 inverted)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


def element_values(codes: np.ndarray, fmt: str) -> np.ndarray:
    """float64 values of 4-bit element codes: E2M1, or two's-complement INT4."""
    codes = np.asarray(codes, dtype=np.int64)
    if is_int(fmt):
        return np.where(codes >= 8, codes - 16, codes).astype(np.float64)
    return F.e2m1_decode(codes)


def scale_values(scales: np.ndarray, fmt: str) -> np.ndarray:
    """float64 values of scale codes."""
    fmt = scale_codec_name(fmt)
    if fmt == "E8M0":
        return np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    return F.CODECS[fmt].decode(scales)


def dequantize(codes, scales, fmt: str, global_amax) -> np.ndarray:
    """Step 6: float32 f32(f32(e2m1 * s_b) / s_enc)."""
    s_enc = global_encode_scale(global_amax, fmt)
    G = GROUP[fmt]
    e = element_values(unpack(codes), fmt).astype(np.float32)
    s_b = np.repeat(scale_values(scales, fmt).astype(np.float32), G, axis=1)
    return ((e * s_b).astype(np.float32) / s_enc).astype(np.float32)


def dequantize_f64(codes, scales, fmt: str, global_amax) -> np.ndarray:
    """float64 e2m1 * s_b / s_enc: the operand values of the reference GEMM."""
    s_enc = float(global_encode_scale(global_amax, fmt))
    G = GROUP[fmt]
    e = element_values(unpack(codes), fmt)
    s_b = np.repeat(scale_values(scales, fmt), G, axis=1)
    return e * s_b / s_enc


# ---------------------------------------------------------------------------
# UE5M3 emulation on an E4M3 scale path ("UE5M3 ..." blog, section
# "Ограничения": UE5M3 ran through software emulation because the tensor-core
# path takes another block-scale format).  Reading fixed here: per tensor,
# t = e_max - 7 with e_max the largest unbiased exponent among the tensor's
# scale values; every scale s is re-encoded as the E4M3 value s * 2^-t, which
# must be exact; the GEMM multiplies its result by 2^(tA + tB).
# ---------------------------------------------------------------------------


def ue5m3_shift(scales: np.ndarray) -> int:
    v = scale_values(scales, "UE5M3")
    vmax = float(np.max(v)) if v.size else 0.0
    if vmax == 0.0:
        return 0
    _, e = np.frexp(vmax)  # vmax = m * 2^e with m in [0.5, 1)
    return int(e) - 1 - 7


def ue5m3_reencode_e4m3(scales: np.ndarray, t: int):
    """(E4M3 codes, all_exact) for UE5M3 scale codes shifted by 2^-t."""
    v = scale_values(scales, "UE5M3") * (2.0 ** -t)
    codec = F.CODECS["E4M3"]
    code = codec.encode(v)
    exact = bool(np.all(codec.decode(code) == v))
    return code, exact


# ---------------------------------------------------------------------------
# UE5M3 scales wider than one E4M3 window ("UE5M3 ..." blog, section
# "Ограничения", the same software emulation).  Reading fixed here: with
# e(s) = floor(log2 s) for every nonzero scale value and e_max the largest,
# scale s belongs to window w = floor((e_max - e(s)) / 14), and window w is
# re-encoded as E4M3 with the shift t_w = e_max - 7 - 14 w (window 0 is the
# single shift above).  Inside a window e(s) - t_w lies in [-6, 7], the normal
# E4M3 exponents, and a UE5M3 value has at most 4 significant bits, so every
# re-encode is exact.  UE5M3 values span 2^-17 .. 1.75 * 2^16, so three
# windows always suffice.  A GEMM over UE5M3 operands is then the sum, over
# window pairs (wa, wb), of the E4M3 GEMMs with every other window's scales
# set to zero, each multiplied by 2^(t_wa + t_wb).
# ---------------------------------------------------------------------------

UE5M3_WINDOW_BINADES = 14
UE5M3_MAX_WINDOWS = 3


def ue5m3_windows(scales: np.ndarray):
    """(shifts t_w for w = 0..2, E4M3 codes per window [3, *scales.shape],
    number of windows in use)."""
    v = scale_values(scales, "UE5M3")
    nz = v > 0
    t0 = ue5m3_shift(scales)
    e_max = t0 + 7
    e = np.zeros(v.shape, dtype=np.int64)
    e[nz] = np.frexp(v[nz])[1].astype(np.int64) - 1
    w = np.where(nz, (e_max - e) // UE5M3_WINDOW_BINADES, -1)
    shifts = [e_max - 7 - UE5M3_WINDOW_BINADES * k for k in range(UE5M3_MAX_WINDOWS)]
    codec = F.CODECS["E4M3"]
    out = np.zeros((UE5M3_MAX_WINDOWS,) + v.shape, dtype=np.uint8)
    for k in range(UE5M3_MAX_WINDOWS):
        sel = w == k
        out[k][sel] = codec.encode(v[sel] * (2.0 ** -shifts[k]))
    n_windows = int(w.max()) + 1 if nz.any() else 1
    return shifts, out, n_windows
