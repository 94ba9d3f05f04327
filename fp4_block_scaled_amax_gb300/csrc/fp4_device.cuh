// Device building blocks of the FP4 block-scaled quantizer (sm_103a).
//
// Method sources (web pages, cited by title and section):
//   "NVFP4 vs MXFP" post (quant_prune_distill #486), "Метод": E2M1 elements,
//     group 16 with an E4M3 scale (NVFP4), group 32 with an E8M0 power-of-two
//     scale (MXFP4).
//   "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining" (rit.work
//     blog), "Что сделали": unsigned 5-exponent/3-fraction block scale.
//   Review of Intel's FP4 training paper (gonzo_ML #3986), "Форматы FP4"
//     (E1M6 .. E8M0 scale sweep) and "Стохастическая квантизация" (nearest
//     rounding forward, stochastic rounding backward).
//
// Every float32 step of the method is a single correctly rounded operation
// (__fmul_rn / __fdiv_rn / __fadd_rn), so no fused multiply-add or reciprocal
// approximation changes a result; the integer steps work on IEEE bit fields.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "../../include/fp4.h"

namespace fp4dev {

// ---------------------------------------------------------------------------
// Status word (first error wins)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

// ---------------------------------------------------------------------------
// bf16 helpers: a 32-bit word holds element 2j in its low half, 2j+1 high.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max |x| over the two bf16 halves of each word, kept as packed non-negative
// bf16 (sign bit cleared, so the packed max is the magnitude max).
__device__ __forceinline__ uint32_t absmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 m = __hmax2(x, y);
  return *reinterpret_cast<uint32_t*>(&m);
}
// max(|a|, |b|) per bf16 half; the sign bits of the result are the XOR of the
// inputs' signs and are cleared by the caller once at the end.
__device__ __forceinline__ uint32_t absmax2_xs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Packed magnitude maxima of n words (each half separately), sign bits clear.
__device__ __forceinline__ uint32_t absmax_words2(const uint32_t* w, int n) {
  uint32_t m = w[0];
#pragma unroll
  for (int i = 1; i < n; ++i) m = absmax2_xs(m, w[i]);
  return m & 0x7FFF7FFFu;
}
__device__ __forceinline__ float absmax_words(const uint32_t* w, int n) {
  const uint32_t m = absmax_words2(w, n);
  return fmaxf(bf16_lo(m), bf16_hi(m));
}

// ---------------------------------------------------------------------------
// Scale formats.  Generic small float with EB exponent bits, MB mantissa bits,
// bias BIAS, IEEE-style subnormals; MAXCODE is the largest finite
// non-negative code.  Encoding: nearest value, ties to the even code,
// saturating at MAXCODE.
// ---------------------------------------------------------------------------
template <int MB, int BIAS>
__device__ __forceinline__ float exmy_decode(uint32_t code) {
  const uint32_t e = code >> MB, m = code & ((1u << MB) - 1u);
  if (e == 0) {
    // m * 2^(1-BIAS-MB): an exact product of a small integer and a power of two
    return __fmul_rn((float)m, __uint_as_float((uint32_t)(127 + 1 - BIAS - MB) << 23));
  }
  return __uint_as_float(((e + 127u - (uint32_t)BIAS) << 23) | (m << (23 - MB)));
}

template <int MB, int BIAS, uint32_t MAXCODE>
__device__ __forceinline__ uint32_t exmy_encode_rne_sat(float s) {
  const float maxv = exmy_decode<MB, BIAS>(MAXCODE);
  if (!(s < maxv)) return MAXCODE;  // also +Inf
  const uint32_t b = __float_as_uint(s);
  const int e = (int)(b >> 23) - 127;
  if (e >= 1 - BIAS) {
    // normal in the target: round the 23-bit fraction to MB bits, ties to even;
    // a carry out of the fraction moves into the exponent field by itself
    constexpr int SH = 23 - MB;
    const uint32_t lsb = (b >> SH) & 1u;
    const uint32_t r = (b + ((1u << (SH - 1)) - 1u) + lsb) >> SH;
    return r - ((uint32_t)(127 - BIAS) << MB);
  }
  // subnormal in the target: count of 2^(1-BIAS-MB) steps, nearest even integer
  const float t = __fmul_rn(s, __uint_as_float((uint32_t)(127 + BIAS + MB - 1) << 23));
  return (uint32_t)__float2int_rn(t);
}

// Format tags, matching fp4_scale_fmt.
enum : int {
  SF_E4M3 = FP4_SF_E4M3,
  SF_UE5M3 = FP4_SF_UE5M3,
  SF_E8M0 = FP4_SF_E8M0,
  SF_E1M6 = FP4_SF_E1M6,
  SF_E2M5 = FP4_SF_E2M5,
  SF_E3M4 = FP4_SF_E3M4,
  SF_E5M2 = FP4_SF_E5M2,
  SF_E6M1 = FP4_SF_E6M1,
  SF_E7M0 = FP4_SF_E7M0,
  SF_NVINT4 = FP4_SF_NVINT4,
  SF_MXINT4 = FP4_SF_MXINT4
};

// Element grid of a format: E2M1 (largest magnitude 6) or, for NVINT4 and
// MXINT4, the integers -7..7 as two's-complement nibbles (largest 7).
template <int FMT> struct Elem { static constexpr bool INT4 = false; };
template <> struct Elem<SF_NVINT4> { static constexpr bool INT4 = true; };
template <> struct Elem<SF_MXINT4> { static constexpr bool INT4 = true; };
template <int FMT> __host__ __device__ constexpr float elem_max() { return Elem<FMT>::INT4 ? 7.0f : 6.0f; }
// Power-of-two (E8M0) block scales without a global scale: MXFP4 and MXINT4
template <int FMT> __host__ __device__ constexpr bool e8m0_scales() { return FMT == SF_E8M0 || FMT == SF_MXINT4; }

template <int FMT> struct ScaleFmt;
// E4M3 (FN) nearest-even with saturation to 448 is the hardware conversion;
// it equals exmy_encode_rne_sat<3, 7, 0x7E> for every non-negative input.
__device__ __forceinline__ uint32_t e4m3_encode_hw(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
  return (uint32_t)(r & 0xFFu);
}
template <> struct ScaleFmt<SF_E4M3> {
  static constexpr int G = 16;
  static constexpr float SIX_ST = 2688.0f;  // 6 * 448
  __device__ static uint32_t encode(float s) { return e4m3_encode_hw(s); }
  __device__ static float decode(uint32_t c) { return exmy_decode<3, 7>(c); }
};
template <> struct ScaleFmt<SF_UE5M3> {
  static constexpr int G = 16;
  static constexpr float SIX_ST = 2688.0f;  // 6 * 448
  __device__ static uint32_t encode(float s) { return exmy_encode_rne_sat<3, 15, 0xFEu>(s); }
  __device__ static float decode(uint32_t c) { return exmy_decode<3, 15>(c); }
};
template <> struct ScaleFmt<SF_E1M6> {
  static constexpr int G = 16;
  static constexpr float SIX_ST = 23.8125f;  // 6 * 3.96875
  __device__ static uint32_t encode(float s) { return exmy_encode_rne_sat<6, 0, 0x7Fu>(s); }
  __device__ static float decode(uint32_t c) { return exmy_decode<6, 0>(c); }
};
// The rest of the group-16 sweep: signed ExMy with bias 2^(E-1)-1, no NaN;
// the non-negative codes run up to 0x7F, and the global-scale target S_T is
// the largest finite value.
template <int MB, int BIAS, int SIX_ST_BITS>
struct SweepScale {
  static constexpr int G = 16;
  __device__ static float six_st() { return __uint_as_float((uint32_t)SIX_ST_BITS); }
  __device__ static uint32_t encode(float s) { return exmy_encode_rne_sat<MB, BIAS, 0x7Fu>(s); }
  __device__ static float decode(uint32_t c) { return exmy_decode<MB, BIAS>(c); }
};
// 6 * S_T as float32 bits: 47.25, 186, 688128, 9 * 2^32, 1.5 * 2^66
template <> struct ScaleFmt<SF_E2M5> : SweepScale<5, 1, 0x423D0000> {};
template <> struct ScaleFmt<SF_E3M4> : SweepScale<4, 3, 0x433A0000> {};
template <> struct ScaleFmt<SF_E5M2> : SweepScale<2, 15, 0x49280000> {};
template <> struct ScaleFmt<SF_E6M1> : SweepScale<1, 31, 0x51100000> {};
template <> struct ScaleFmt<SF_E7M0> : SweepScale<0, 63, 0x60C00000> {};

template <> struct ScaleFmt<SF_E8M0> {
  static constexpr int G = 32;
  static constexpr float SIX_ST = 0.0f;  // unused: no global scale
  // code = clamp(floor(log2 a) - 2 + 127, 0, 254), the exponent read from the bits
  __device__ static uint32_t encode_from_amax(float a) {
    const int e = (int)(__float_as_uint(a) >> 23);
    int c = e > 0 ? e - 2 : 0;
    c = c < 0 ? 0 : (c > 254 ? 254 : c);
    return (uint32_t)c;
  }
  __device__ static float decode(uint32_t c) {
    return c > 0 ? __uint_as_float(c << 23) : __uint_as_float(0x00400000u);  // 2^-127
  }
};

// NVINT4: E4M3 scales with the numerator f32(7 * 448); MXINT4: E8M0 scales.
template <> struct ScaleFmt<SF_NVINT4> : ScaleFmt<SF_E4M3> {
  static constexpr float SIX_ST = 3136.0f;  // 7 * 448: the INT4 grid tops out at 7
};
template <> struct ScaleFmt<SF_MXINT4> : ScaleFmt<SF_E8M0> {};

// f32(emax * S_T), the numerator of s_enc (SIX_ST: "6 * S_T" for E2M1 grids,
// 7 * S_T for NVINT4).
template <int FMT>
__device__ __forceinline__ float six_st_of() {
  if constexpr (FMT >= SF_E2M5 && FMT <= SF_E7M0) return ScaleFmt<FMT>::six_st();
  else return ScaleFmt<FMT>::SIX_ST;
}

// Per-tensor encode scale from the stored amax g.
template <int FMT>
__device__ __forceinline__ float global_encode_scale(float g, int32_t* status) {
  if (e8m0_scales<FMT>()) return 1.0f;
  if (!(fabsf(g) <= 3.402823466e38f)) {  // Inf or NaN
    set_status(status, FP4_ERR_NONFINITE);
    return 1.0f;
  }
  if (g == 0.0f) return 1.0f;
  const float s = __fdiv_rn(six_st_of<FMT>(), g);
  return (s > 3.402823466e38f) ? 3.402823466e38f : s;
}

struct BlockScale {
  uint32_t code;
  float r;  // element multiplier s_enc / s_b (0 when s_b == 0)
};

// Element multiplier of a scale code: s_enc / s_b (0 when s_b == 0).
template <int FMT>
__device__ __forceinline__ float code_multiplier(uint32_t code, float s_enc) {
  const float s_b = ScaleFmt<FMT>::decode(code);
  return (s_b == 0.0f) ? 0.0f : __fdiv_rn(s_enc, s_b);
}

// f32(a / D) for D = 6 or 7 and a block maximum a that is a bf16 value (at
// most 8 significant bits): q0 = f32(a * f32(1/D)), the exact residual
// a - D q0 by one fma, and q0 + residual * f32(1/D) by another equal the
// correctly rounded quotient for every 8-bit significand (checked
// exhaustively); the binade only scales the result while it stays normal, so
// small a takes the division itself.
template <int D>
__device__ __forceinline__ float div_small_exact(float a) {
  static_assert(D == 6 || D == 7, "divisor");
  if (!(a >= 7.8886091e-31f)) return __fdiv_rn(a, (float)D);  // below 2^-100 (and zero)
  const float c = D == 6 ? __uint_as_float(0x3E2AAAABu) : __uint_as_float(0x3E124925u);  // f32(1/D)
  const float q0 = __fmul_rn(a, c);
  const float res = __fmaf_rn(-(float)D, q0, a);
  return __fmaf_rn(res, c, q0);
}

// Block scale with the multiplier looked up in a per-CTA table of all codes.
// BF16_AMAX: a_b is a bf16 value (the block maximum of bf16 inputs), so the
// division by the grid maximum takes div_small_exact.
template <int FMT, bool BF16_AMAX = false>
__device__ __forceinline__ BlockScale block_scale_tab(float a_b, float s_enc, const float* rtab) {
  BlockScale out;
  if constexpr (e8m0_scales<FMT>()) {
    out.code = ScaleFmt<SF_E8M0>::encode_from_amax(a_b);
  } else {
    const float a6 = BF16_AMAX ? div_small_exact<(int)elem_max<FMT>()>(a_b) : __fdiv_rn(a_b, elem_max<FMT>());
    out.code = ScaleFmt<FMT>::encode(__fmul_rn(a6, s_enc));
  }
  out.r = rtab[out.code];
  return out;
}

template <int FMT, bool BF16_AMAX = false>
__device__ __forceinline__ BlockScale block_scale(float a_b, float s_enc) {
  BlockScale out;
  float s_b;
  if constexpr (e8m0_scales<FMT>()) {
    out.code = ScaleFmt<SF_E8M0>::encode_from_amax(a_b);
    s_b = ScaleFmt<SF_E8M0>::decode(out.code);
  } else {
    const float a6 = BF16_AMAX ? div_small_exact<(int)elem_max<FMT>()>(a_b) : __fdiv_rn(a_b, elem_max<FMT>());
    const float s_real = __fmul_rn(a6, s_enc);
    out.code = ScaleFmt<FMT>::encode(s_real);
    s_b = ScaleFmt<FMT>::decode(out.code);
  }
  out.r = (s_b == 0.0f) ? 0.0f : __fdiv_rn(s_enc, s_b);
  return out;
}

// ---------------------------------------------------------------------------
// E2M1 element rounding
// ---------------------------------------------------------------------------
// Round-to-nearest-even with saturation, two values into one byte: `lo` in the
// low nibble, `hi` in the high nibble (cvt.rn.satfinite.e2m1x2.f32 puts its
// first source in the upper nibble).
__device__ __forceinline__ uint32_t e2m1x2_rne(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Stochastic rounding of one value with a 16-bit draw R (reading R8): with
// lo <= |y| < hi the neighbouring grid values, round up iff
// R < 65536 * (|y| - lo) / (hi - lo); |y| >= 6 gives 6.  Returns the rounded
// grid value with the sign of x (the caller converts exact grid values to
// codes).  It is a carry into the grid-step bit of z = |y| * 2^-126:
//  * for 1 <= |y| < 8, z is normal and exact, and the E2M1 step is 2^(e-1)
//    with e the binary exponent of |y|, i.e. bit 22 of the float32 pattern
//    of z; f = (|y| - lo)/step is the 22-bit field m below it over 2^22, and
//    "R < 65536 f" is "m > 64 R" (R is an integer), i.e. m + (2^22 - 1 - 64 R)
//    carries into bit 22.  So adding d = 0x3FFFFF - 64 R and clearing the 22
//    low bits gives lo or hi; a carry out of the mantissa moves into the
//    exponent by itself (1.5 -> 2, 3 -> 4, 6 -> 8, which the saturating
//    conversion maps to 6);
//  * below 1, z is subnormal: its pattern is the integer |y| * 2^23 rounded
//    up (the product is rounded toward +inf), so bit 22 is again the step
//    0.5 and the same carry applies; rounding up keeps the decision exact,
//    as the threshold lo + 64 R * 2^-23 lies on that grid and a value rounded
//    up exceeds it iff the value itself does; 0.5 + 0.5 carries into the
//    exponent field and gives 1 * 2^-126, the normal pattern of 1;
//  * |y| = 0 stays 0; +Inf stays +Inf.
// Multiplying back by 2^126 is exact on the grid values.  d is computed by
// the caller from the draw (sr_d_lo / sr_d_hi).
__device__ __forceinline__ float e2m1_sr_value(float x, float r, uint32_t d) {
  const float ay = __fmul_rn(fabsf(x), r);
  float z;
  asm("mul.rp.f32 %0, %1, 0f00800000;" : "=f"(z) : "f"(ay));  // ay * 2^-126, subnormals kept
  const float q = __uint_as_float((__float_as_uint(z) + d) & 0xFFC00000u);
  const float m = __fmul_rn(q, 0x1p126f);  // exact: * 2^126
  return __uint_as_float(__float_as_uint(m) | (__float_as_uint(x) & 0x80000000u));
}
// The carry constant d = 0x3FFFFF - 64 R of the low and the high 16-bit draw
// R of a Philox word (one multiply-add each).
__device__ __forceinline__ uint32_t sr_d_lo(uint32_t w) { return (w & 0xFFFFu) * 0xFFFFFFC0u + 0x3FFFFFu; }
__device__ __forceinline__ uint32_t sr_d_hi(uint32_t w) { return (w >> 16) * 0xFFFFFFC0u + 0x3FFFFFu; }
// INT4 grid (integers -7..7, two's-complement nibble): nearest with ties to
// even after clamping to [-7, 7]; adding 1.5 * 2^23 rounds to an integer in
// float32 and leaves it in the low mantissa bits.
__device__ __forceinline__ uint32_t int4_rne(float y) {
  const float yc = fminf(fmaxf(y, -7.0f), 7.0f);
  return (__float_as_uint(__fadd_rn(yc, 12582912.0f)) - 0x4B400000u) & 0xFu;
}
// INT4 stochastic rounding: ceil(min(|y|, 7) - r * 2^-16) with the sign of x.
// The grid step is 1, so the argument of e2m1_sr_value holds with z = |y|:
// near an integer n in 1..6 the float32 difference is off by at least
// ulp(z) >= 2^-21 > ulp(n)/2, and below 1 it is exact.  -0 becomes code 0.
__device__ __forceinline__ uint32_t int4_sr(float x, float r, uint32_t rbits) {
  const float ay = fminf(__fmul_rn(fabsf(x), r), 7.0f);
  const float rho = __fsub_rn(__uint_as_float(rbits), 1.0f);  // r * 2^-23
  const float t = __fmaf_rn(-rho, 128.0f, ay);                 // ay - r * 2^-16, one rounding
  const float c = __fsub_rn(__fadd_ru(t, 12582912.0f), 12582912.0f);
  const float v = __uint_as_float(__float_as_uint(c) | (__float_as_uint(x) & 0x80000000u));
  return (__float_as_uint(__fadd_rn(v, 12582912.0f)) - 0x4B400000u) & 0xFu;
}

// 1 + r * 2^-23 (float32 bits 0x3F800000 | r) for the low and high 16-bit
// halves r of a Philox word (the INT4 grid's stochastic rounding): one byte
// permute each.
__device__ __forceinline__ uint32_t sr_rbits_lo(uint32_t w) { return __byte_perm(w, 0x3F800000u, 0x7610u); }
__device__ __forceinline__ uint32_t sr_rbits_hi(uint32_t w) { return __byte_perm(w, 0x3F800000u, 0x7632u); }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of
// (c0,c1,c2,c3) -> (hi(M1*c2)^c1^k0, lo(M1*c2), hi(M0*c0)^c3^k1, lo(M0*c0)),
// the key advanced by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
// The ten round keys of a seed (key = (seed low, seed high), advanced by the
// Weyl constants), computed once per thread where it draws many times.
struct PhiloxKey {
  uint32_t k0[10], k1[10];
  __device__ __forceinline__ explicit PhiloxKey(uint64_t seed) {
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      k0[i] = a;
      k1[i] = b;
      a += 0x9E3779B9u;
      b += 0xBB67AE85u;
    }
  }
};
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const PhiloxKey& key) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    c0 = (uint32_t)(p1 >> 32) ^ c1 ^ key.k0[i];
    c1 = (uint32_t)p1;
    c2 = (uint32_t)(p0 >> 32) ^ c3 ^ key.k1[i];
    c3 = (uint32_t)p0;
  }
  return make_uint4(c0, c1, c2, c3);
}
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    // one 32 x 32 -> 64-bit multiply gives both halves of each product
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    c0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    c1 = (uint32_t)p1;
    c2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c3 = (uint32_t)p0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// The 8 draws of output indices 8*blk .. 8*blk+7: element j takes word j/2,
// low half for even j, high half for odd j.
__device__ __forceinline__ uint4 sr_draws8(uint64_t seed, uint64_t blk) {
  return philox4x32_10((uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u, (uint32_t)seed,
                       (uint32_t)(seed >> 32));
}
__device__ __forceinline__ uint4 sr_draws8(const PhiloxKey& key, uint64_t blk) {
  return philox4x32_10((uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u, key);
}
// A block index below 2^32 (a tensor of fewer than 2^35 elements): the
// counter's second word is a literal zero, which removes a multiply from the
// second round and an xor from the first.
__device__ __forceinline__ uint4 sr_draws8(const PhiloxKey& key, uint32_t blk) {
  return philox4x32_10(blk, 0u, 0u, 0u, key);
}
// Where the draws of 16 consecutive elements start: an element index (a
// multiple of 8), or SrIdx32, the block index itself when it fits 32 bits.
struct SrIdx32 {
  uint32_t blk;
};
__device__ __forceinline__ uint64_t sr_block(uint64_t idx0, int h) { return (idx0 >> 3) + (uint64_t)h; }
__device__ __forceinline__ uint32_t sr_block(SrIdx32 i, int h) { return i.blk + (uint32_t)h; }
__device__ __forceinline__ uint32_t draw16(const uint4& w, int j) {
  const uint32_t v = (j >> 1) == 0 ? w.x : (j >> 1) == 1 ? w.y : (j >> 1) == 2 ? w.z : w.w;
  return (j & 1) ? (v >> 16) : (v & 0xFFFFu);
}

// ---------------------------------------------------------------------------
// Quantize 16 bf16 values (8 words, element order = word order, low half
// first) with block multiplier r into 8 bytes of packed codes.
// Philox indices of the 16 elements start at idx0 (a multiple of 8).
// ---------------------------------------------------------------------------
// Four pairs (lo in the low nibble of each byte) -> one 32-bit word, byte 0
// from the first pair.
__device__ __forceinline__ uint32_t e2m1x8_rne(const float* y) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  return r;
}

template <bool SR, bool INT4 = false, class KEY = uint64_t, class IDX = uint64_t>
__device__ __forceinline__ uint2 quant16(const uint32_t* w, float r, const KEY& seed, IDX idx0) {
  if constexpr (INT4) {
    uint32_t nib[16];
    if constexpr (!SR) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        nib[2 * i] = int4_rne(__fmul_rn(bf16_lo(w[i]), r));
        nib[2 * i + 1] = int4_rne(__fmul_rn(bf16_hi(w[i]), r));
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 d = sr_draws8(seed, sr_block(idx0, h));
        const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          nib[8 * h + 2 * i] = int4_sr(bf16_lo(w[4 * h + i]), r, sr_rbits_lo(dw[i]));
          nib[8 * h + 2 * i + 1] = int4_sr(bf16_hi(w[4 * h + i]), r, sr_rbits_hi(dw[i]));
        }
      }
    }
    uint2 out = make_uint2(0u, 0u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      out.x |= nib[i] << (4 * i);
      out.y |= nib[8 + i] << (4 * i);
    }
    return out;
  }
  float y[16];
  if constexpr (!SR) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[2 * i] = __fmul_rn(bf16_lo(w[i]), r);
      y[2 * i + 1] = __fmul_rn(bf16_hi(w[i]), r);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 d = sr_draws8(seed, sr_block(idx0, h));
      const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t wi = w[4 * h + i];
        y[8 * h + 2 * i] = e2m1_sr_value(bf16_lo(wi), r, sr_d_lo(dw[i]));
        y[8 * h + 2 * i + 1] = e2m1_sr_value(bf16_hi(wi), r, sr_d_hi(dw[i]));
      }
    }
  }
  return make_uint2(e2m1x8_rne(y), e2m1x8_rne(y + 8));
}

// quant16 of one column of a 16-row block held as 16 words, each a row's
// pair of neighbouring columns: HI selects the high (odd) column.
template <bool SR, bool HI, class KEY = uint64_t, class IDX = uint64_t>
__device__ __forceinline__ uint2 quant16_col(const uint32_t (&v)[16], float r, const KEY& seed, IDX idx0) {
  float y[16];
  if constexpr (!SR) {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(HI ? bf16_hi(v[i]) : bf16_lo(v[i]), r);
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 d = sr_draws8(seed, sr_block(idx0, h));
      const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t a = v[8 * h + 2 * i], b = v[8 * h + 2 * i + 1];
        y[8 * h + 2 * i] = e2m1_sr_value(HI ? bf16_hi(a) : bf16_lo(a), r, sr_d_lo(dw[i]));
        y[8 * h + 2 * i + 1] = e2m1_sr_value(HI ? bf16_hi(b) : bf16_lo(b), r, sr_d_hi(dw[i]));
      }
    }
  }
  return make_uint2(e2m1x8_rne(y), e2m1x8_rne(y + 8));
}

// ---------------------------------------------------------------------------
// 16 x 16 random Hadamard transform of one block held as 16 floats:
// x' = 1/4 * H16 * (s . x), s[j] = -1 iff bit j of mask is set; the fast
// Walsh-Hadamard butterflies for h = 1, 2, 4, 8, each add and subtract one
// float32 operation, then the exact scaling by 1/4.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void rht16(float (&v)[16], uint32_t mask) {
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((mask >> j) & 1u) << 31));
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// quant16 for 16 float32 inputs (the transformed block).
template <bool SR, bool INT4>
__device__ __forceinline__ uint2 quant16f(const float (&v)[16], float r, uint64_t seed, uint64_t idx0) {
  if constexpr (INT4) {
    uint32_t nib[16];
    if constexpr (!SR) {
#pragma unroll
      for (int i = 0; i < 16; ++i) nib[i] = int4_rne(__fmul_rn(v[i], r));
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 d = sr_draws8(seed, (idx0 >> 3) + h);
        const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          nib[8 * h + 2 * i] = int4_sr(v[8 * h + 2 * i], r, sr_rbits_lo(dw[i]));
          nib[8 * h + 2 * i + 1] = int4_sr(v[8 * h + 2 * i + 1], r, sr_rbits_hi(dw[i]));
        }
      }
    }
    uint2 out = make_uint2(0u, 0u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      out.x |= nib[i] << (4 * i);
      out.y |= nib[8 + i] << (4 * i);
    }
    return out;
  }
  float y[16];
  if constexpr (!SR) {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(v[i], r);
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 d = sr_draws8(seed, (idx0 >> 3) + h);
      const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        y[8 * h + 2 * i] = e2m1_sr_value(v[8 * h + 2 * i], r, sr_d_lo(dw[i]));
        y[8 * h + 2 * i + 1] = e2m1_sr_value(v[8 * h + 2 * i + 1], r, sr_d_hi(dw[i]));
      }
    }
  }
  return make_uint2(e2m1x8_rne(y), e2m1x8_rne(y + 8));
}

// Byte offset of scale (row r, block b) in the tiled MMA scale layout with nb
// blocks per row: 128-row x 4-block atoms of 512 bytes, row-major over atoms;
// inside an atom row r sits at (r%32)*16 + ((r/32)%4)*4, block b at b%4.
__device__ __forceinline__ int64_t mma_sf_offset(int64_t r, int64_t b, int64_t nb) {
  return ((r >> 7) * (nb >> 2) + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}

}  // namespace fp4dev
