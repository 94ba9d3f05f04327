// Weight-only NVFP4 linear for small batches (sm_103a), HBM-bound.
//
// Weight-only NVFP4 post (quant_prune_distill #574): weights in NVFP4,
// activations untouched (section "Метод"); the speed-up comes from a
// memory-bound kernel for small-batch generation (section "Эксперименты").
//
//   y[b, n] = (1 / s_enc) * sum_k (e2m1[n, k] * s_b[n, k/16]) * x[b, k]
//
// W streams once from HBM: 0.5 B of codes + 1/16 B of scale per weight.  Each
// warp turns its codes into bf16 A-fragments in registers (e2m1 * s_b is exact
// in bf16: at most 6 significant bits, exponent in [-10, 12]) and multiplies
// them with the bf16 activations on the tensor cores (mma.sync m16n8k16,
// float32 accumulation).  The batch is the MMA's N dimension (8 per tile).
//
// Two forms.  K % 256 == 0 (any batch up to 64) takes the TMA-fed kernel
// further down: weights, scales and activations stream through a shared-memory
// ring and are shared by all warps of a CTA.  Other K take the register-fed
// kernel right below.
//
// Register-fed form.  k permutation: inside a 128-wide k chunk, lane q of a quad (q = lane % 4)
// supplies at MMA step s the fragment positions {2q, 2q+1, 2q+8, 2q+9} from
// the actual columns 32q + 4s + {0, 1, 2, 3}.  A and B use the same map, so the
// sum over positions is the sum over k, while each lane reads 16 contiguous
// code bytes and 64 contiguous activation bytes per chunk.
//
// CTA = 16 weight rows x WARPS warps splitting K; partial sums meet in shared
// memory.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "async_sm103.cuh"
#include "device_cache.h"
#include "fp4_device.cuh"
#include "launch.h"

namespace {

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Four E2M1 codes (16 bits, element 0 in the low nibble) -> two bf16x2 words.
// Magnitude bytes come from two 8-entry byte tables through PRMT.
__device__ __forceinline__ void e2m1x4_to_bf16x4(uint32_t c16, uint32_t& w01, uint32_t& w23) {
  // bf16 of {0, 0.5, 1, 1.5, 2, 3, 4, 6}: high bytes 00 3F 3F 3F 40 40 40 40,
  // low bytes 00 00 80 C0 00 40 80 C0
  const uint32_t sel = c16 & 0x7777u;
  uint32_t lo, hi;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0xC0800000u), "r"(0xC0804000u), "r"(sel));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x3F3F3F00u), "r"(0x40404040u), "r"(sel));
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(lo), "r"(hi), "r"(0x5140u));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b) : "r"(lo), "r"(hi), "r"(0x7362u));
  w01 = a | ((c16 & 0x8u) << 12) | ((c16 & 0x80u) << 24);
  w23 = b | ((c16 & 0x800u) << 4) | ((c16 & 0x8000u) << 16);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t s2) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&s2);
  __nv_bfloat162 r = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// E4M3 scale code -> bf16 bits replicated in both halves (exact).
__device__ __forceinline__ uint32_t e4m3_to_bf16x2(uint32_t c) {
  const float v = fp4dev::ScaleFmt<fp4dev::SF_E4M3>::decode(c);
  const uint32_t h = __float_as_uint(v) >> 16;  // exact: <= 4 significant bits
  return h | (h << 16);
}

// Loads of one 128-wide k chunk for one lane: 16 code bytes and 2 scale bytes
// of its two weight rows, and its 32 activations of each batch row it feeds.
template <int NT>
struct Chunk {
  uint4 w0, w1;
  uint32_t s0, s1;
  uint4 xb[NT][4];
};

template <int NT>
__device__ __forceinline__ void load_chunk(Chunk<NT>& ch, const uint8_t* __restrict__ Wq,
                                           const uint8_t* __restrict__ Ws, const uint16_t* __restrict__ x,
                                           int64_t r0, int64_t r1, bool v0, bool v1, int64_t k0, int64_t K,
                                           int batch, int g) {
  const bool kin = k0 < K;  // K % 32 == 0: a lane's 32 columns are all in or all out
  ch.w0 = ch.w1 = make_uint4(0, 0, 0, 0);
  ch.s0 = ch.s1 = 0;
  if (kin && v0) {
    ch.w0 = ld_stream16(Wq + r0 * (K / 2) + k0 / 2);
    ch.s0 = *reinterpret_cast<const uint16_t*>(Ws + r0 * (K / 16) + k0 / 16);
  }
  if (kin && v1) {
    ch.w1 = ld_stream16(Wq + r1 * (K / 2) + k0 / 2);
    ch.s1 = *reinterpret_cast<const uint16_t*>(Ws + r1 * (K / 16) + k0 / 16);
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int b = t * 8 + g;
#pragma unroll
    for (int i = 0; i < 4; ++i) ch.xb[t][i] = make_uint4(0, 0, 0, 0);
    if (kin && b < batch) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)b * K + k0);
#pragma unroll
      for (int i = 0; i < 4; ++i) ch.xb[t][i] = __ldg(src + i);
    }
  }
}

template <int NT>
__device__ __forceinline__ void mma_chunk(float (&acc)[NT][4], const Chunk<NT>& ch) {
  const uint32_t sc0[2] = {e4m3_to_bf16x2(ch.s0 & 0xFFu), e4m3_to_bf16x2(ch.s0 >> 8)};
  const uint32_t sc1[2] = {e4m3_to_bf16x2(ch.s1 & 0xFFu), e4m3_to_bf16x2(ch.s1 >> 8)};
  const uint32_t cw0[4] = {ch.w0.x, ch.w0.y, ch.w0.z, ch.w0.w};
  const uint32_t cw1[4] = {ch.w1.x, ch.w1.y, ch.w1.z, ch.w1.w};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t c0 = (cw0[s >> 1] >> (16 * (s & 1))) & 0xFFFFu;
    const uint32_t c1 = (cw1[s >> 1] >> (16 * (s & 1))) & 0xFFFFu;
    uint32_t a0, a2, a1, a3;
    e2m1x4_to_bf16x4(c0, a0, a2);
    e2m1x4_to_bf16x4(c1, a1, a3);
    a0 = bf16x2_mul(a0, sc0[s >> 2]);
    a2 = bf16x2_mul(a2, sc0[s >> 2]);
    a1 = bf16x2_mul(a1, sc1[s >> 2]);
    a3 = bf16x2_mul(a3, sc1[s >> 2]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint4 xv = ch.xb[t][s >> 1];
      const uint32_t b0 = (s & 1) ? xv.z : xv.x;
      const uint32_t b1 = (s & 1) ? xv.w : xv.y;
      mma_bf16_16816(acc[t], a0, a1, a2, a3, b0, b1);
    }
  }
}

constexpr int MAX_WARPS = 16;

template <int NT>
__global__ void __launch_bounds__(NT <= 2 ? 512 : 256) k_gemv_w4a16(const uint8_t* __restrict__ Wq, const uint8_t* __restrict__ Ws,
                                                     const float* __restrict__ gw, const uint16_t* __restrict__ x,
                                                     int batch, int64_t N, int64_t K, bool bf16_out,
                                                     void* __restrict__ y) {
  // partial sums [warp][row][batch]; 16 warps x 16 rows x 32 (NT <= 4) or
  // 8 warps x 16 x 64 (NT = 8): 32 KB either way
  __shared__ float red[MAX_WARPS * 16 * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * 16;
  const int64_t r0 = n0 + g, r1 = n0 + g + 8;
  const bool v0 = r0 < N, v1 = r1 < N;
  const int64_t nchunk_total = (K + 127) / 128;
  const int64_t per = (nchunk_total + nwarps - 1) / nwarps;
  const int64_t c_begin = warp * per;
  const int64_t c_end = min(nchunk_total, c_begin + per);

  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

  if constexpr (NT <= 2) {
    // software pipeline: the next chunk's loads are in flight during this chunk's MMAs
    Chunk<NT> cur, nxt;
    if (c_begin < c_end) load_chunk<NT>(cur, Wq, Ws, x, r0, r1, v0, v1, c_begin * 128 + 32 * q, K, batch, g);
    for (int64_t c = c_begin; c < c_end; ++c) {
      if (c + 1 < c_end) load_chunk<NT>(nxt, Wq, Ws, x, r0, r1, v0, v1, (c + 1) * 128 + 32 * q, K, batch, g);
      mma_chunk<NT>(acc, cur);
      cur = nxt;
    }
  } else {
    // larger batches: 32 MMAs per chunk hide the load latency; one buffer keeps
    // the activations in registers without spilling
    for (int64_t c = c_begin; c < c_end; ++c) {
      Chunk<NT> cur;
      load_chunk<NT>(cur, Wq, Ws, x, r0, r1, v0, v1, c * 128 + 32 * q, K, batch, g);
      mma_chunk<NT>(acc, cur);
    }
  }
  // D fragment: (row g, cols 2q, 2q+1) and (row g+8, cols 2q, 2q+1)
  constexpr int BW = 8 * NT;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    red[(warp * 16 + g) * BW + t * 8 + 2 * q] = acc[t][0];
    red[(warp * 16 + g) * BW + t * 8 + 2 * q + 1] = acc[t][1];
    red[(warp * 16 + g + 8) * BW + t * 8 + 2 * q] = acc[t][2];
    red[(warp * 16 + g + 8) * BW + t * 8 + 2 * q + 1] = acc[t][3];
  }
  __syncthreads();
  const float s_enc = fp4dev::global_encode_scale<fp4dev::SF_E4M3>(__ldg(gw), nullptr);
  for (int i = threadIdx.x; i < 16 * BW; i += blockDim.x) {
    const int r = i / BW, b = i % BW;
    const int64_t n = n0 + r;
    if (n >= N || b >= batch) continue;
    float v = 0.0f;
    for (int w = 0; w < nwarps; ++w) v = __fadd_rn(v, red[(w * 16 + r) * BW + b]);
    v = __fdiv_rn(v, s_enc);
    if (bf16_out) static_cast<__nv_bfloat16*>(y)[(int64_t)b * N + n] = __float2bfloat16_rn(v);
    else static_cast<float*>(y)[(int64_t)b * N + n] = v;
  }
}


// ---------------------------------------------------------------------------
// TMA-fed form: K % 256 == 0, batch up to 64 (NT tiles of 8 rows)
// ---------------------------------------------------------------------------
// One CTA per group of T 16-row tiles (T chosen so the groups cover the SMs
// in about one wave).  Warp 0 streams stages of SC = 128 * WPT columns into a
// shared-memory ring with cp.async.bulk.tensor: the T*16 code rows (128-byte
// boxes, 128-byte swizzle), their SC/16 scale bytes per row, and the eight
// activation rows of the same columns (64-column boxes, 128-byte swizzle; rows
// >= batch, code rows >= N and columns >= K arrive as zeros).  Each 16-row
// tile has WPT consumer warps, one per 128-column slice of the stage; a lane
// reads one code word (8 columns) of each of its two rows per pair of MMAs.
//
// Pairing: the code word's nibbles n0..n7 become four bf16x2 registers
// (n_i, n_{i+4}).  Bits (e1 e0 m) of a nibble at bf16 bits 8..6 are the E2M1
// value times 2^-126 exactly (e = 0 lands on a bf16 subnormal), with the sign
// at bit 15: isolating nibbles i and i+4 and multiplying by 2^6 + 2^12 puts
// both fields in place at once (the two shifted copies do not overlap), and
// one AND clears the rest.  One bf16x2 multiply by the block scale times
// 2^118 gives e2m1 * s_b * 2^-8, exact (<= 6 significant bits, normal).  The
// activations are paired the same way, (x_i, x_{i+4}), with one PRMT per
// register, so each MMA's k positions are the same columns on both sides.
// Word order: lane q takes its four words starting at word q (mod 4), which
// keeps the 16-byte activation loads and the code loads free of bank
// conflicts.  The 2^-8 folds into the final division by s_enc.

constexpr int TV_MAX_TILES = 8;  // 16-row tiles per CTA
constexpr int TV_MAX_STAGES = 32;
constexpr int TV_RING_BUDGET = 200 * 1024;
constexpr int TV_SMEM_MAX = 227 * 1024;  // dynamic shared memory per CTA on sm_103a

// WPT consumer warps per 16-row tile; NT batch tiles of 8 rows (the MMA's N)
template <int WPT, int NT>
struct TvLayout {
  static constexpr int SC = 128 * WPT;     // columns per stage
  static constexpr int SB = SC / 16;       // scale bytes per row per stage
  static constexpr int CODE_BOXES = SC / 256;
  static constexpr int X_BOXES = SC / 64;  // 64-column activation boxes of 8 * NT rows
  static constexpr uint32_t X_BOX_BYTES = 1024u * NT;
  __host__ __device__ static constexpr uint32_t code_box_bytes(int T) { return 2048u * T; }
  __host__ __device__ static constexpr uint32_t code_bytes(int T) { return CODE_BOXES * code_box_bytes(T); }
  __host__ __device__ static constexpr uint32_t x_bytes() { return X_BOX_BYTES * X_BOXES; }
  __host__ __device__ static constexpr uint32_t stage_bytes(int T) {
    return code_bytes(T) + x_bytes() + ((16u * SB * T + 1023u) & ~1023u);
  }
};

// Code word (nibbles n0..n7, n0 lowest) -> bf16x2 (n_i, n_{i+4}) * 2^-126.
__device__ __forceinline__ void e2m1x8_pairs(uint32_t v, uint32_t (&r)[4]) {
  constexpr uint32_t M = 0x81C081C0u;  // bf16 bits 8..6 and 15 of both halves
  const uint32_t v2 = v >> 8;
  r[0] = ((v & 0x000F000Fu) * 4160u) & M;
  r[1] = ((v & 0x00F000F0u) * 260u) & M;
  r[2] = ((v2 & 0x000F000Fu) * 4160u) & M;
  r[3] = ((v2 & 0x00F000F0u) * 260u) & M;
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two E4M3 scale codes per row (sa: row A, sb: row B; low byte = block 2j)
// -> bf16x2 of (value * 2^118) for each row and block, in both halves.  A
// code shifted to bf16 bits 11..4 is value * 2^-120 exactly (E4M3 subnormals
// land on bf16 subnormals); two exact multiplies by 2^119.
__device__ __forceinline__ void e4m3_scales_bf16x2(uint32_t sa, uint32_t sb, uint32_t (&sA)[2],
                                                   uint32_t (&sB)[2]) {
  const uint32_t both = sa | (sb << 16);
  constexpr uint32_t TWO119 = 0x7B007B00u;  // bf16x2 (2^119, 2^119)
  const uint32_t lo = mul_bf16x2(mul_bf16x2((both & 0x00FF00FFu) << 4, TWO119), TWO119);
  const uint32_t hi = mul_bf16x2(mul_bf16x2((both >> 4) & 0x0FF00FF0u, TWO119), TWO119);
  sA[0] = prmt(lo, lo, 0x1010u);
  sB[0] = prmt(lo, lo, 0x3232u);
  sA[1] = prmt(hi, hi, 0x1010u);
  sB[1] = prmt(hi, hi, 0x3232u);
}

// MMA without side effects, so the compiler may schedule the next step's
// shared-memory loads ahead of it.
__device__ __forceinline__ void mma_bf16_16816_pure(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                    uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Every lane waits; the warp proceeds only if all lanes saw the phase.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status) {
  const bool ok = fp4async::wait_bounded(bar, parity, abort_flag, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Wait, without recording an error, for a phase that should already be
// complete (copies issued before an abort); gives up after DRAIN_CYCLES.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!fp4async::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > fp4async::DRAIN_CYCLES) return;
  }
}

// Prefetch of a tensor-map tile into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

template <int WPT, int NT>
__global__ void __launch_bounds__(NT == 1 ? 32 * (1 + 4 * 6) : 32 * (1 + 2 * 8))
    k_gemv_w4a16_tma(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                     const __grid_constant__ CUtensorMap tm_x, const float* __restrict__ gw, int batch, int N,
                     int nk_total, int T, int S, int ksplit, bool bf16_out, void* __restrict__ y, int32_t* status) {
  using namespace fp4async;
  using L = TvLayout<WPT, NT>;
  constexpr int BW = 8 * NT;  // batch columns per tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t stage_bytes = L::stage_bytes(T);
  const uint32_t code_bytes = L::code_bytes(T);
  const uint32_t code_box = L::code_box_bytes(T);
  const int nwarps = WPT * T;
  float* const red = reinterpret_cast<float*>(base_ptr + S * stage_bytes);  // [WPT*T][16][BW]
  const uint32_t bars = base + S * stage_bytes + (uint32_t)nwarps * 16 * BW * 4;  // full[S], empty[S]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // split K: the ksplit CTAs of a cluster share the tiles and each takes a
  // contiguous run of the K stages; rank 0 sums the partial results
  uint32_t rank = 0;
  if (ksplit > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int n0 = (blockIdx.x / ksplit) * 16 * T;
  const int it0 = (int)(((int64_t)nk_total * rank) / ksplit);
  const int nk = (int)(((int64_t)nk_total * (rank + 1)) / ksplit) - it0;

  // a GEMV launched after this one may start its CTAs as these exit (they
  // wait for this grid before they read its activations)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 8 * (S + s), nwarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_codes)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_scales)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      const uint32_t tx = code_bytes + L::x_bytes() + 16u * L::SB * T;
      // The weights do not depend on a preceding kernel: those of the first
      // two stages are prefetched into L2 while it may still be running
      // (programmatic dependent launch); then every stage loads as usual,
      // codes, activations and scales, once that kernel has completed.  (A
      // deeper prefetch queues ahead of the real loads when nothing precedes.)
      const int pre = nk < 2 ? nk : 2;
      for (int it = 0; it < pre; ++it) {
        const int gs = it0 + it;
#pragma unroll
        for (int i = 0; i < L::CODE_BOXES; ++i) tma_prefetch_l2_2d(&tm_codes, gs * (L::SC / 2) + 128 * i, n0);
        tma_prefetch_l2_2d(&tm_scales, gs * L::SB, n0);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int issued = 0;
      for (int it = 0, s = 0, ph = 0; it < nk; ++it) {
        if (it >= S && !wait_bounded(bars + 8 * (S + s), ph ^ 1, &abort_flag, status)) break;
        const uint32_t full = bars + 8 * s;
        const uint32_t st = base + s * stage_bytes;
        mbar_expect_tx(full, tx);
        const int gs = it0 + it;  // the stage's place along K
#pragma unroll
        for (int i = 0; i < L::CODE_BOXES; ++i)
          tma_load_2d(st + code_box * i, &tm_codes, full, gs * (L::SC / 2) + 128 * i, n0);
#pragma unroll
        for (int i = 0; i < L::X_BOXES; ++i)
          tma_load_2d(st + code_bytes + L::X_BOX_BYTES * i, &tm_x, full, gs * L::SC + 64 * i, 0);
        tma_load_2d(st + code_bytes + L::x_bytes(), &tm_scales, full, gs * L::SB, n0);
        issued = it + 1;
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      // no copy may still be landing when the CTA exits
      for (int it = issued > S ? issued - S : 0; it < issued; ++it) wait_drain(bars + 8 * (it % S), (it / S) & 1);
    }
  } else {
    // everything these warps read or write follows the preceding kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int cw = warp - 1, t = cw / WPT, qt = cw % WPT;
    const int g = lane >> 2, q = lane & 3;
    const int j = 4 * qt + q;  // the lane's 32-column chunk of the stage
    const uint32_t rowA = 16u * t + g;
    uint32_t code_off[4], x_off[4];
    bool upper[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int w = (s + q) & 3;
      code_off[s] = (uint32_t)(j >> 3) * code_box + rowA * 128u + ((uint32_t)((j & 7) ^ g) << 4) + 4u * w;
      x_off[s] = code_bytes + (uint32_t)(j >> 1) * L::X_BOX_BYTES + g * 128u + ((uint32_t)((4 * (j & 1) + w) ^ g) << 4);
      upper[s] = (w >> 1) != 0;
    }
    const uint32_t sc_off = code_bytes + L::x_bytes() + rowA * L::SB + 2u * j;
    // NT == 1: two accumulator chains (even and odd MMAs); NT > 1: one chain per batch tile
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    float acc[NT][4];
#pragma unroll
    for (int t8 = 0; t8 < NT; ++t8) acc[t8][0] = acc[t8][1] = acc[t8][2] = acc[t8][3] = 0.f;
    for (int it = 0, s = 0, ph = 0; it < nk; ++it) {
      if (!wait_warp(bars + 8 * s, ph, &abort_flag, status)) break;
      const uint8_t* st = base_ptr + s * stage_bytes;
      uint32_t scA[2], scB[2];
      e4m3_scales_bf16x2(*reinterpret_cast<const uint16_t*>(st + sc_off),
                         *reinterpret_cast<const uint16_t*>(st + sc_off + 8 * L::SB), scA, scB);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t va = *reinterpret_cast<const uint32_t*>(st + code_off[k]);
        const uint32_t vb = *reinterpret_cast<const uint32_t*>(st + code_off[k] + 8 * 128);
        uint32_t ra[4], rb[4];
        e2m1x8_pairs(va, ra);
        e2m1x8_pairs(vb, rb);
        const uint32_t sA = upper[k] ? scA[1] : scA[0], sB = upper[k] ? scB[1] : scB[0];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ra[i] = mul_bf16x2(ra[i], sA);
          rb[i] = mul_bf16x2(rb[i], sB);
        }
        if constexpr (NT == 1) {
          const uint4 xv = *reinterpret_cast<const uint4*>(st + x_off[k]);
          mma_bf16_16816_pure(acc0, ra[0], rb[0], ra[1], rb[1], prmt(xv.x, xv.z, 0x5410u), prmt(xv.x, xv.z, 0x7632u));
          mma_bf16_16816_pure(acc1, ra[2], rb[2], ra[3], rb[3], prmt(xv.y, xv.w, 0x5410u), prmt(xv.y, xv.w, 0x7632u));
        } else {
          // batch tile t8 is activation rows 8*t8 + g: 8 rows (1 KB) further into the box
#pragma unroll
          for (int t8 = 0; t8 < NT; ++t8) {
            const uint4 xv = *reinterpret_cast<const uint4*>(st + x_off[k] + 1024u * t8);
            mma_bf16_16816_pure(acc[t8], ra[0], rb[0], ra[1], rb[1], prmt(xv.x, xv.z, 0x5410u),
                                prmt(xv.x, xv.z, 0x7632u));
            mma_bf16_16816_pure(acc[t8], ra[2], rb[2], ra[3], rb[3], prmt(xv.y, xv.w, 0x5410u),
                                prmt(xv.y, xv.w, 0x7632u));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (S + s));
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
    float* rw = red + (size_t)cw * 16 * BW;
    if constexpr (NT == 1) {
      rw[g * 8 + 2 * q] = acc0[0] + acc1[0];
      rw[g * 8 + 2 * q + 1] = acc0[1] + acc1[1];
      rw[(g + 8) * 8 + 2 * q] = acc0[2] + acc1[2];
      rw[(g + 8) * 8 + 2 * q + 1] = acc0[3] + acc1[3];
    } else {
#pragma unroll
      for (int t8 = 0; t8 < NT; ++t8) {
        rw[g * BW + 8 * t8 + 2 * q] = acc[t8][0];
        rw[g * BW + 8 * t8 + 2 * q + 1] = acc[t8][1];
        rw[(g + 8) * BW + 8 * t8 + 2 * q] = acc[t8][2];
        rw[(g + 8) * BW + 8 * t8 + 2 * q + 1] = acc[t8][3];
      }
    }
  }
  __syncthreads();
  if (ksplit > 1) {
    // every CTA's partial sums are in its shared memory before rank 0 reads them
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  if (rank == 0) {
    const float s_enc = fp4dev::global_encode_scale<fp4dev::SF_E4M3>(__ldg(gw), nullptr);
    const int rows = 16 * T;
    for (int i = threadIdx.x; i < rows * BW; i += blockDim.x) {
      const int b = i / rows, r = i % rows;
      const int n = n0 + r;
      if (n >= N || b >= batch) continue;
      const int t = r >> 4, rr = r & 15;
      const float* p = red + ((size_t)(WPT * t) * 16 + rr) * BW + b;
      float v = 0.0f;
#pragma unroll
      for (int k = 0; k < WPT; ++k) v = __fadd_rn(v, p[k * 16 * BW]);
      // the other ranks' partial sums, in rank order (a fixed summation order)
      for (int q = 1; q < ksplit; ++q) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(q));
#pragma unroll
        for (int k = 0; k < WPT; ++k) {
          float pv;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pv) : "r"(remote + 4u * k * 16 * BW));
          v = __fadd_rn(v, pv);
        }
      }
      v = __fdiv_rn(__fmul_rn(v, 256.0f), s_enc);
      if (bf16_out) static_cast<__nv_bfloat16*>(y)[(int64_t)b * N + n] = __float2bfloat16_rn(v);
      else static_cast<float*>(y)[(int64_t)b * N + n] = v;
    }
  }
  if (ksplit > 1) {
    // no CTA leaves while rank 0 may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
}

bool make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz,
              CUtensorMapL2promotion l2) {
  auto fn = fp4async::encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() { return fp4lib::current_sm_count(); }

template <int WPT, int NT>
cudaError_t launch_tma_t(const fp4lib::GemvArgs& a, int T, int ksplit, cudaStream_t st) {
  using L = TvLayout<WPT, NT>;
  const int64_t tiles = (a.N + 15) / 16;
  const int64_t ctas = (tiles + T - 1) / T * ksplit;
  const int nk_total = (int)((a.K + L::SC - 1) / L::SC);
  const int nk = (nk_total + ksplit - 1) / ksplit;  // the most stages one CTA streams
  const size_t red_bytes = (size_t)WPT * T * 16 * 8 * NT * 4;
  // batch <= 8: a 200 KB ring; larger batches: what fits beside the reduction buffer
  const size_t budget =
      NT == 1 ? (size_t)TV_RING_BUDGET : (size_t)TV_SMEM_MAX - 1024 - red_bytes - 16 * TV_MAX_STAGES;
  int S = (int)(budget / L::stage_bytes(T));
  if (S > TV_MAX_STAGES) S = TV_MAX_STAGES;
  if (S > nk) S = nk;
  if (S < 1) return cudaErrorNotSupported;
  const size_t smem = 1024 + (size_t)S * L::stage_bytes(T) + red_bytes + 16u * S;
  CUtensorMap mc, ms, mx;
  if (!make_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wq, a.K / 2, a.N, a.K / 2, 128, 16 * T,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Ws, a.K / 16, a.N, a.K / 16, L::SB, 16 * T,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.batch, a.K * 2, 64, 8 * NT,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorNotSupported;
  // once per device: allow the most dynamic shared memory this instance can
  // have there (the opt-in limit less its static shared memory)
  static fp4lib::DeviceInts smem_allowed;
  cudaError_t e = cudaSuccess;
  const int allowed = smem_allowed.get([&] {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa{};
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaFuncGetAttributes(&fa, k_gemv_w4a16_tma<WPT, NT>)) != cudaSuccess)
      return 0;
    const int n = optin - (int)fa.sharedSizeBytes;
    e = cudaFuncSetAttribute(k_gemv_w4a16_tma<WPT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, n);
    return e == cudaSuccess ? n : 0;
  });
  if (e != cudaSuccess) return e;
  if (allowed <= 0 || smem > (size_t)allowed) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  // programmatic dependent launch: the kernel may start while the preceding
  // kernel in the stream finishes (it waits for it before reading x)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)ksplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(32 * (1 + WPT * T), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = ksplit > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_w4a16_tma<WPT, NT>, mc, ms, mx, a.gw, (int)a.batch, (int)a.N, nk_total, T, S,
                            ksplit, a.bf16_out, a.y, a.status);
}

// Returns cudaErrorNotSupported (before launching anything) when the shape or
// the tensor-map encoder rules the TMA-fed form out.  Four warps per tile
// (512-column stages) up to six tiles per CTA, two beyond.
cudaError_t launch_gemv_tma(const fp4lib::GemvArgs& a, cudaStream_t st) {
  if (a.batch > 64 || a.K % 256 != 0 || a.N > (int64_t)1 << 30 || a.K > (int64_t)1 << 30)
    return cudaErrorNotSupported;
  const int64_t tiles = (a.N + 15) / 16;
  const int sms = sm_count();
  // tiles per CTA and K split: the fewest split ways whose CTAs cover at least
  // 90 % of the SMs (a split needs at least 4 stages per CTA), else the best
  int T = 1, ksplit = 1;
  double best = -1.0;
  for (int s = 1; s <= 4; s *= 2) {
    int t = (int)((tiles * s + sms - 1) / sms);
    t = t < 1 ? 1 : t;
    if (t > TV_MAX_TILES) continue;
    const int64_t stages = a.K / 256;  // 256-column stages at the least
    if (s > 1 && stages < 4 * s) continue;
    const double cover = (double)(((tiles + t - 1) / t) * s) / sms;
    if (cover > best + 0.02) {
      best = cover;
      T = t;
      ksplit = s;
    }
    if (cover >= 0.9) break;
  }
  // eight batch tiles of 8 rows: 512-column stages (four warps per tile) when a CTA holds few tiles,
  // 256-column stages (two warps per tile) otherwise
  if (a.batch > 8) return T <= 3 ? launch_tma_t<4, 8>(a, T, ksplit, st) : launch_tma_t<2, 8>(a, T, ksplit, st);
  return T <= 6 ? launch_tma_t<4, 1>(a, T, ksplit, st) : launch_tma_t<2, 1>(a, T, ksplit, st);
}

}  // namespace

namespace fp4lib {

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st) {
  cudaError_t e = launch_gemv_umma(a, st);  // batch > 8: tensor-memory accumulation
  if (e != cudaErrorNotSupported) return e;
  e = launch_gemv_tma(a, st);
  if (e != cudaErrorNotSupported) return e;
  // register-fed form: 16 weight rows per CTA; enough warps per CTA (split K) to put about 16
  // warps on each of the GPU's SMs in a single wave
  const int64_t ctas = (a.N + 15) / 16;
  const int sms = fp4lib::current_sm_count();
  const int64_t kchunks = (a.K + 127) / 128;
  int64_t warps = (int64_t)sms * 16 / ctas;
  warps = warps < 4 ? 4 : (warps > MAX_WARPS ? MAX_WARPS : warps);
  if (warps > kchunks) warps = kchunks < 1 ? 1 : kchunks;
  const int nt = (int)((a.batch + 7) / 8);
  if (nt > 2 && warps > 8) warps = 8;  // the larger batch tiles launch with at most 256 threads
  const unsigned grid = (unsigned)ctas;
  const unsigned threads = (unsigned)(32 * warps);
  const auto* x = static_cast<const uint16_t*>(a.x);
  const int b = (int)a.batch;
  if (nt == 1) k_gemv_w4a16<1><<<grid, threads, 0, st>>>(a.Wq, a.Ws, a.gw, x, b, a.N, a.K, a.bf16_out, a.y);
  else if (nt == 2) k_gemv_w4a16<2><<<grid, threads, 0, st>>>(a.Wq, a.Ws, a.gw, x, b, a.N, a.K, a.bf16_out, a.y);
  else if (nt <= 4) k_gemv_w4a16<4><<<grid, threads, 0, st>>>(a.Wq, a.Ws, a.gw, x, b, a.N, a.K, a.bf16_out, a.y);
  else k_gemv_w4a16<8><<<grid, threads, 0, st>>>(a.Wq, a.Ws, a.gw, x, b, a.N, a.K, a.bf16_out, a.y);
  return cudaGetLastError();
}

}  // namespace fp4lib
