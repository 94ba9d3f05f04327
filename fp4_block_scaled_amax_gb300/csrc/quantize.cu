// FP4 block-scaled quantizer kernels for sm_103a (HBM-bound).
//
// What they compute (web pages, cited by title and section):
//   "NVFP4 vs MXFP" post (quant_prune_distill #486), "Метод": per-block scale
//     stored in low precision (E4M3 / group 16, E8M0 / group 32), elements in
//     FP4 E2M1, scale handling fused into the kernel.
//   "UE5M3 FP4 Block Scaling ..." (rit.work blog), "Что сделали": UE5M3 block
//     scale per 16 elements; the tensor maximum may be a stored (stale) value.
//   gonzo_ML #3986, "Стохастическая квантизация": nearest rounding for forward
//     weights/activations, stochastic rounding for backward tensors.
//
// Kernels:
//   k_amax            max|x| of a bf16 matrix (fresh global amax), 2 B/elem read.
//   k_amax_n          the same for up to eight matrices in one launch.
//   k_quant_rows      blocks along K; one thread per 16 elements straight from
//                     two 128-bit loads; 2 + 0.5 + 1/G B per element.
//   k_quant_dual_tma  persistent dual (row + transposed) quantizer over 128 x
//                     128 tiles loaded by TMA into a 4-stage ring; transposed
//                     codes and both scale layouts staged and stored by TMA /
//                     bulk copies (MMA scale layout, G = 16, M and K multiples
//                     of 128): 2 + 2 * (0.5 + 1/16) B per element.
//   k_quant_tile      64 x 128 tile staged in shared memory; writes the
//                     transposed quantization (blocks along M) and, in the dual
//                     form, the row quantization from the same read:
//                     2 + 2 * (0.5 + 1/G) B per element (the other layouts
//                     and formats).
//   k_dequant         codes + scales -> float32 / bf16.
//   k_ue5m3_*         UE5M3 -> shifted E4M3 re-encode for the tensor-core path,
//                     the shift from the quantizers' largest scale code, and
//                     the multi-window split of wide UE5M3 scales.
//   k_encode_scales, k_philox_bits16   conformance helpers (same device code).
#include <cstdint>
#include <cuda_runtime.h>

#include "async_sm103.cuh"
#include "device_cache.h"
#include "fp4_device.cuh"
#include "launch.h"

using namespace fp4dev;

namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void atomic_max_nonneg(float* dst, float v) {
  // non-negative IEEE floats order like their bit patterns
  atomicMax(reinterpret_cast<unsigned int*>(dst), __float_as_uint(v));
}

// ---------------------------------------------------------------------------
// K0: global amax
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_amax(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                              int64_t ldx, float* __restrict__ out) {
  const int64_t per_row = K / 8;  // 16-byte chunks per row
  const int64_t total = M * per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const bool dense = ldx == K;  // rows back to back: one flat array, no index division
  uint32_t m = 0;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  auto addr = [&](int64_t c) -> const uint16_t* {
    if (dense) return x + c * 8;
    const int64_t r = c / per_row;
    return x + r * ldx + (c - r * per_row) * 8;
  };
  // eight independent 16-byte loads in flight per thread, the last round
  // guarded, so the tail costs one memory latency rather than one per chunk
  for (; i < total; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = i + u * stride < total ? ld_stream(addr(i + u * stride)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      m = absmax2_xs(m, v[u].x);
      m = absmax2_xs(m, v[u].y);
      m = absmax2_xs(m, v[u].z);
      m = absmax2_xs(m, v[u].w);
    }
  }
  m &= 0x7FFF7FFFu;  // the packed maxima carry XOR-ed signs
  float a = fmaxf(bf16_lo(m), bf16_hi(m));
  unsigned int ab = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(a));
  __shared__ unsigned int warp_max[8];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = ab;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned int v = threadIdx.x < (blockDim.x >> 5) ? warp_max[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(out), v);
  }
}

// Several tensors in one launch: CTA b works on tensor i with
// cta_begin[i] <= b < cta_begin[i + 1] (CTA counts in proportion to size).
struct AmaxN {
  const uint16_t* x[fp4lib::AMAX_N_MAX];
  int64_t M[fp4lib::AMAX_N_MAX], K[fp4lib::AMAX_N_MAX], ldx[fp4lib::AMAX_N_MAX];
  int cta_begin[fp4lib::AMAX_N_MAX + 1];
  int n;
};

// 128-thread CTAs (at most 64 registers a thread, 8 K a CTA): one fits on an
// SM beside a persistent dual quantizer, whose 576 threads of 96 registers
// leave 10 K, so that an amax pass launched on another stream runs in the
// quantizer's spare resources.
constexpr int AMAXN_THREADS = 128;
__global__ void __launch_bounds__(AMAXN_THREADS, 8) k_amax_n(const __grid_constant__ AmaxN a, float* __restrict__ out) {
  int i = 0;
  while (i + 1 < a.n && (int)blockIdx.x >= a.cta_begin[i + 1]) ++i;
  const int b = (int)blockIdx.x - a.cta_begin[i], nb = a.cta_begin[i + 1] - a.cta_begin[i];
  const int64_t K = a.K[i], ldx = a.ldx[i];
  const int64_t per_row = K / 8;
  const int64_t total = a.M[i] * per_row;
  const int64_t stride = (int64_t)nb * blockDim.x;
  const bool dense = ldx == K;
  const uint16_t* x = a.x[i];
  uint32_t m = 0;
  auto addr = [&](int64_t c) -> const uint16_t* {
    if (dense) return x + c * 8;
    const int64_t r = c / per_row;
    return x + r * ldx + (c - r * per_row) * 8;
  };
  for (int64_t c = (int64_t)b * blockDim.x + threadIdx.x; c < total; c += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = c + u * stride < total ? ld_stream(addr(c + u * stride)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      m = absmax2_xs(m, v[u].x);
      m = absmax2_xs(m, v[u].y);
      m = absmax2_xs(m, v[u].z);
      m = absmax2_xs(m, v[u].w);
    }
  }
  m &= 0x7FFF7FFFu;
  const float am = fmaxf(bf16_lo(m), bf16_hi(m));
  unsigned int ab = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(am));
  __shared__ unsigned int warp_max[8];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = ab;
  __syncthreads();
  if (threadIdx.x < 32) {
    unsigned int v = threadIdx.x < (blockDim.x >> 5) ? warp_max[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(out + i), v);
  }
}

// ---------------------------------------------------------------------------
// K1: row quantizer (blocks along K)
// ---------------------------------------------------------------------------
template <int FMT, bool SR, bool MMA, bool AMAX>
__global__ void __launch_bounds__(256) k_quant_rows(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                    int64_t ldx, const float* __restrict__ gptr,
                                                    uint64_t seed, uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ scales,
                                                    float* __restrict__ amax_out, int32_t* status,
                                                    uint32_t* __restrict__ sf_max) {
  constexpr int G = ScaleFmt<FMT>::G;
  const int64_t per_row = K / 16;
  const int64_t chunk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = chunk < M * per_row;
  const unsigned mask = __ballot_sync(0xFFFFFFFFu, valid);
  if (!valid) return;
  const float s_enc = global_encode_scale<FMT>(
      __ldg(gptr), (blockIdx.x == 0 && threadIdx.x == 0) ? status : nullptr);
  const int64_t row = chunk / per_row;
  const int64_t c16 = chunk - row * per_row;
  const uint16_t* src = x + row * ldx + c16 * 16;
  const uint4 v0 = ld_stream(src), v1 = ld_stream(src + 8);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float a = absmax_words(w, 8);
  if constexpr (AMAX) {
    const unsigned int am = __reduce_max_sync(mask, __float_as_uint(a));
    if ((threadIdx.x & 31) == (unsigned)(__ffs(mask) - 1)) atomicMax(reinterpret_cast<unsigned int*>(amax_out), am);
  }
  if constexpr (G == 32) a = fmaxf(a, __shfl_xor_sync(mask, a, 1));
  const BlockScale bs = block_scale<FMT, true>(a, s_enc);
  const uint2 q = quant16<SR, Elem<FMT>::INT4>(w, bs.r, seed, (uint64_t)(row * K + c16 * 16));
  *reinterpret_cast<uint2*>(codes + row * (K / 2) + c16 * 8) = q;
  if constexpr (FMT == SF_UE5M3) {
    if (sf_max != nullptr) {
      // UE5M3 codes order like their values: the largest code gives e_max
      const unsigned int mc = __reduce_max_sync(mask, bs.code);
      if ((threadIdx.x & 31) == (unsigned)(__ffs(mask) - 1)) atomicMax(sf_max, mc);
    }
  }
  if (G == 16 || (c16 & 1) == 0) {
    const int64_t b = c16 * 16 / G;
    const int64_t nb = K / G;
    const int64_t off = MMA ? mma_sf_offset(row, b, nb) : row * nb + b;
    scales[off] = (uint8_t)bs.code;
  }
}

// ---------------------------------------------------------------------------
// K2/K3: tile quantizer (transposed output, plus the row output when DUAL)
// ---------------------------------------------------------------------------
// A CTA stages a 64-row x 128-column bf16 tile in shared memory.  Row pass:
// each thread quantizes two 16-element chunks straight from its loads.
// Column pass: thread t takes column t/2 and the 32-row half t%2, so two
// neighbouring lanes write one whole 32-byte sector of the transposed output.
// Columns are stored XOR-swizzled by the half (bit 4 of the column index
// flips for rows 32..63), which keeps the column pass free of bank conflicts.
// The element multipliers s_enc / s_b of all 256 scale codes are computed
// once per CTA into a shared table (the same correctly rounded division).
constexpr int TILE_M = 64;
constexpr int TILE_K = 128;

__device__ __forceinline__ int tile_col(int r, int c) { return c ^ (((r >> 5) & 1) << 4); }

template <int FMT, bool DUAL, bool ROW_SR, bool COL_SR, bool MMA, bool AMAX>
__global__ void __launch_bounds__(256) k_quant_tile(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx, const float* __restrict__ gptr,
    uint64_t seed_row, uint64_t seed_col, uint8_t* __restrict__ codes_row, uint8_t* __restrict__ scales_row,
    uint8_t* __restrict__ codes_col, uint8_t* __restrict__ scales_col, float* __restrict__ amax_out,
    int32_t* status, uint32_t* __restrict__ sf_max_row, uint32_t* __restrict__ sf_max_col) {
  constexpr int G = ScaleFmt<FMT>::G;
  __shared__ __align__(16) uint16_t tile[TILE_M][TILE_K];
  __shared__ float rtab[256];
  // blockIdx.x walks M fastest so neighbouring CTAs write neighbouring
  // sectors of each transposed-output row
  const int64_t m0 = (int64_t)blockIdx.x * TILE_M;
  const int64_t k0 = (int64_t)blockIdx.y * TILE_K;
  const float s_enc = global_encode_scale<FMT>(
      __ldg(gptr), (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) ? status : nullptr);

  // ---- load 64 x 128 (two 16-element chunks per thread, all loads first) ----
  uint32_t w[2][8];
  bool valid[2];
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int j = threadIdx.x + 256 * it;  // chunk id in the tile: 8 chunks per row
    const int r = j >> 3, cc = j & 7;
    const int64_t col = k0 + cc * 16;
    // K % 32 == 0 keeps a G=32 pair valid together; M % 32 == 0 makes a
    // 32-row half all valid or all not
    valid[it] = col < K && m0 + r < M;
    if (valid[it]) {
      const uint16_t* src = x + (m0 + r) * ldx + col;
      const uint4 v0 = ld_stream(src), v1 = ld_stream(src + 8);
      w[it][0] = v0.x; w[it][1] = v0.y; w[it][2] = v0.z; w[it][3] = v0.w;
      w[it][4] = v1.x; w[it][5] = v1.y; w[it][6] = v1.z; w[it][7] = v1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[it][i] = 0u;
    }
  }
  rtab[threadIdx.x] = code_multiplier<FMT>(threadIdx.x, s_enc);
  __syncthreads();
  float amax_local = 0.0f;
  uint32_t maxc_row = 0;  // largest row scale code (UE5M3 shift by-product)
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int j = threadIdx.x + 256 * it;
    const int r = j >> 3, cc = j & 7;
    uint4* dst = reinterpret_cast<uint4*>(&tile[r][tile_col(r, cc * 16)]);
    dst[0] = make_uint4(w[it][0], w[it][1], w[it][2], w[it][3]);
    dst[1] = make_uint4(w[it][4], w[it][5], w[it][6], w[it][7]);
    float a = absmax_words(w[it], 8);
    amax_local = fmaxf(amax_local, a);
    if constexpr (DUAL) {
      if constexpr (G == 32) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
      if (valid[it]) {
        const int64_t row = m0 + r, col = k0 + cc * 16;
        const BlockScale bs = block_scale_tab<FMT, true>(a, s_enc, rtab);
        const uint2 q = quant16<ROW_SR>(w[it], bs.r, seed_row, (uint64_t)(row * K + col));
        *reinterpret_cast<uint2*>(codes_row + row * (K / 2) + col / 2) = q;
        maxc_row = max(maxc_row, bs.code);
        if (G == 16 || (cc & 1) == 0) {
          const int64_t b = col / G;
          const int64_t nb = K / G;
          scales_row[MMA ? mma_sf_offset(row, b, nb) : row * nb + b] = (uint8_t)bs.code;
        }
      }
    }
  }
  if constexpr (AMAX) {
    const unsigned int am = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_local));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(amax_out), am);
  }
  if constexpr (DUAL && FMT == SF_UE5M3) {
    if (sf_max_row != nullptr) {
      const unsigned int mc = __reduce_max_sync(0xFFFFFFFFu, maxc_row);
      if ((threadIdx.x & 31) == 0) atomicMax(sf_max_row, mc);
    }
  }
  __syncthreads();

  // ---- column pass: thread t owns column k0 + t/2, rows m0 + 32*(t%2) .. +31 ----
  const int cl = threadIdx.x >> 1, h = threadIdx.x & 1;
  const int64_t c = k0 + cl;
  const int64_t rbase = m0 + 32 * h;
  const unsigned cmask = __ballot_sync(0xFFFFFFFFu, c < K && rbase < M);
  if (c >= K || rbase >= M) return;
  const int pc = cl ^ (h << 4);
  uint32_t v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    v[i] = (uint32_t)tile[32 * h + 2 * i][pc] | ((uint32_t)tile[32 * h + 2 * i + 1][pc] << 16);
  const uint64_t idx0 = (uint64_t)(c * M + rbase);
  uint2 q0, q1;
  uint32_t sc0, sc1 = 0;
  if constexpr (G == 16) {
    const BlockScale b0 = block_scale_tab<FMT, true>(absmax_words(v, 8), s_enc, rtab);
    const BlockScale b1 = block_scale_tab<FMT, true>(absmax_words(v + 8, 8), s_enc, rtab);
    q0 = quant16<COL_SR>(v, b0.r, seed_col, idx0);
    q1 = quant16<COL_SR>(v + 8, b1.r, seed_col, idx0 + 16);
    sc0 = b0.code;
    sc1 = b1.code;
  } else {
    const BlockScale b0 = block_scale_tab<FMT, true>(absmax_words(v, 16), s_enc, rtab);
    q0 = quant16<COL_SR>(v, b0.r, seed_col, idx0);
    q1 = quant16<COL_SR>(v + 8, b0.r, seed_col, idx0 + 16);
    sc0 = b0.code;
  }
  *reinterpret_cast<uint4*>(codes_col + c * (M / 2) + rbase / 2) = make_uint4(q0.x, q0.y, q1.x, q1.y);
  if constexpr (FMT == SF_UE5M3) {
    if (sf_max_col != nullptr) {
      const unsigned int mc = __reduce_max_sync(cmask, max(sc0, sc1));
      if ((threadIdx.x & 31) == (unsigned)(__ffs(cmask) - 1)) atomicMax(sf_max_col, mc);
    }
  }
  const int64_t nb = M / G;
  const int64_t b = rbase / G;
  if constexpr (G == 16) {
    // blocks b, b+1 (b even) are adjacent bytes in both layouts
    const int64_t off = MMA ? mma_sf_offset(c, b, nb) : c * nb + b;
    *reinterpret_cast<uint16_t*>(scales_col + off) = (uint16_t)(sc0 | (sc1 << 8));
  } else {
    scales_col[MMA ? mma_sf_offset(c, b, nb) : c * nb + b] = (uint8_t)sc0;
  }
}

// ---------------------------------------------------------------------------
// K3': persistent TMA-fed dual / transposed quantizer (tiled scale layout)
// ---------------------------------------------------------------------------
// One CTA per SM walks 128 x 128 tiles of x (M fastest).  Warp 0 streams
// each tile into a 4-stage ring of 32 KB stages with two TMA loads (64-column
// boxes, 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8));
// sixteen consumer warps quantize it; warp 17 writes the staged outputs.
//   row pass   thread (warp w, lane l) takes row 8w + l % 8 and the 16-column
//              chunks 4j + l / 8 (j = 0, 1): two 16-byte loads each, eight
//              lanes on eight rows of one chunk (no bank conflict); its 8 code
//              bytes go straight to global memory (the four chunks of a row in
//              one instruction fill a 32-byte sector);
//   col pass   warp w takes box w / 8 and rows 16 (w % 8) .. +15; lane l reads
//              the 32-bit word of columns 2l, 2l + 1 in each of the 16 rows
//              (a whole 128-byte row per instruction) and quantizes both
//              columns' 16-row blocks;
// the transposed codes (128 output rows x 64 bytes, 64-byte swizzle: chunk j
// of row c at j ^ ((c / 2) % 4)) and both scale sets (for a 128 x 128 tile,
// the row scales of rows m0.. and the transposed scales of columns k0.. are
// each two whole 512-byte atoms of the tiled layout, contiguous in memory)
// are staged in shared memory and written by one TMA tensor store and two
// bulk copies.  Staging is double-buffered.  Every wait is bounded.  The
// Philox block indices (element index / 8) are 32-bit: a tensor of 2^35
// elements or more takes k_quant_tile instead.
constexpr int QD_T = 128;                    // tile rows = tile columns
constexpr int QD_STAGES = 4;
constexpr int QD_CONSUMERS = 16;             // warps
constexpr int QD_THREADS = 32 * (QD_CONSUMERS + 2);
constexpr int QD_STAGE_BYTES = QD_T * QD_T * 2;  // 32 KB of bf16
constexpr int QD_COLC_BYTES = QD_T * QD_T / 2;   // 8 KB of transposed codes
constexpr int QD_SF_BYTES = QD_T * QD_T / 16;    // 1 KB of scales per layout
constexpr int QD_STG_BYTES = QD_COLC_BYTES + 2 * QD_SF_BYTES;
constexpr int QD_SMEM_STAGES = 0;
constexpr int QD_SMEM_STG = QD_SMEM_STAGES + QD_STAGES * QD_STAGE_BYTES;
constexpr int QD_SMEM_RTAB = QD_SMEM_STG + 2 * QD_STG_BYTES;
constexpr int QD_SMEM_BAR = QD_SMEM_RTAB + 256 * 4;
constexpr int QD_SMEM_TOTAL = QD_SMEM_BAR + 8 * (2 * QD_STAGES + 4) + 16;
constexpr int QD_SMEM_LAUNCH = QD_SMEM_TOTAL + 1024;  // base aligned up to 1024
static_assert(QD_SMEM_STG % 1024 == 0 && QD_STG_BYTES % 1024 == 0, "swizzled buffers need 1024-byte alignment");

struct QdParams {
  const float* gptr;
  uint64_t seed_row, seed_col;
  int64_t M, K;
  uint8_t* codes_row;
  uint8_t* scales_row;
  uint8_t* scales_col;
  float* amax_out;
  int32_t* status;
  uint32_t* sf_max_row;
  uint32_t* sf_max_col;
};

__device__ __forceinline__ void qd_tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void qd_bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
// The tiles t = t0, t0 + stride, ... of a grid with m_tiles tiles per column
// (M fastest), walked without a division per tile.
struct TileWalk {
  int mt, kt, dm, dk, m_tiles;
  __device__ __forceinline__ TileWalk(int t0, int stride, int m_tiles_)
      : mt(t0 % m_tiles_), kt(t0 / m_tiles_), dm(stride % m_tiles_), dk(stride / m_tiles_), m_tiles(m_tiles_) {}
  __device__ __forceinline__ void next() {
    mt += dm;
    kt += dk;
    if (mt >= m_tiles) {
      mt -= m_tiles;
      ++kt;
    }
  }
};

// scale (row r, block b) of a 128-row x 8-block tile inside its two atoms
__device__ __forceinline__ int qd_sf_off(int r, int b) { return (b >> 2) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3); }

template <int FMT, bool DO_ROW, bool ROW_SR, bool COL_SR, bool AMAX>
__global__ void __launch_bounds__(QD_THREADS, 1)
    k_quant_dual_tma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_ccol,
                     QdParams p) {
  using namespace fp4async;
  static_assert(ScaleFmt<FMT>::G == 16, "16-element blocks only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  float* rtab = reinterpret_cast<float*>(smem + QD_SMEM_RTAB);
  const uint32_t bar_full = sbase + QD_SMEM_BAR;
  const uint32_t bar_empty = bar_full + 8 * QD_STAGES;
  const uint32_t bar_stg_full = bar_empty + 8 * QD_STAGES;  // [2]
  const uint32_t bar_stg_free = bar_stg_full + 16;          // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + QD_SMEM_BAR + 8 * (2 * QD_STAGES + 4));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (int)(p.M / QD_T), k_tiles = (int)(p.K / QD_T);
  const int ntiles = m_tiles * k_tiles;
  const float s_enc =
      global_encode_scale<FMT>(__ldg(p.gptr), (blockIdx.x == 0 && threadIdx.x == 0) ? p.status : nullptr);
  if (threadIdx.x < 256) rtab[threadIdx.x] = code_multiplier<FMT>(threadIdx.x, s_enc);
  if (threadIdx.x == 0) {
    for (int s = 0; s < QD_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, QD_CONSUMERS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_stg_full + 8 * b, QD_CONSUMERS);
      mbar_init(bar_stg_free + 8 * b, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      int it = 0;
      TileWalk tw(blockIdx.x, gridDim.x, m_tiles);
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it, tw.next()) {
        const int s = it % QD_STAGES;
        if (it >= QD_STAGES &&
            !wait_bounded(bar_empty + 8 * s, ((it / QD_STAGES) - 1) & 1, abort_flag, p.status))
          break;
        if (*abort_flag) break;
        const int m0 = tw.mt * QD_T, k0 = tw.kt * QD_T;
        const uint32_t fb = bar_full + 8 * s, dst = sbase + QD_SMEM_STAGES + s * QD_STAGE_BYTES;
        mbar_expect_tx(fb, QD_STAGE_BYTES);
        tma_load_2d(dst, &tm_x, fb, k0, m0);
        tma_load_2d(dst + QD_STAGE_BYTES / 2, &tm_x, fb, k0 + 64, m0);
      }
    }
  } else if (warp <= QD_CONSUMERS) {
    // ------------------------------ consumers -----------------------------
    const int cw = warp - 1;
    float amax_local = 0.0f;
    uint32_t maxc_row = 0, maxc_col = 0;
    // row pass: row 8 cw + l % 8, chunks 4 j + l / 8
    const int rr = 8 * cw + (lane & 7), rq = lane >> 3;
    // col pass: box cw / 8, row block cw % 8, columns 2 l, 2 l + 1 of the box
    const int cbox = cw >> 3, crb = cw & 7;
    const PhiloxKey key_row(p.seed_row), key_col(p.seed_col);
    int it = 0;
    TileWalk tw(blockIdx.x, gridDim.x, m_tiles);
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it, tw.next()) {
      const int s = it % QD_STAGES, b = it & 1;
      const int m0 = tw.mt * QD_T, k0 = tw.kt * QD_T;
      if (!wait_lane0(bar_full + 8 * s, (it / QD_STAGES) & 1, abort_flag, p.status, lane)) break;
      if ((it >> 1) > 0 && !wait_lane0(bar_stg_free + 8 * b, ((it >> 1) - 1) & 1, abort_flag, p.status, lane))
        break;
      const uint8_t* stage = smem + QD_SMEM_STAGES + s * QD_STAGE_BYTES;
      uint8_t* stg = smem + QD_SMEM_STG + b * QD_STG_BYTES;
      uint8_t* stg_colc = stg;
      uint8_t* stg_sfr = stg + QD_COLC_BYTES;
      uint8_t* stg_sfc = stg_sfr + QD_SF_BYTES;
      if constexpr (DO_ROW) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 4 * j + rq;  // 16-column chunk of the tile
          const uint8_t* row = stage + j * (QD_STAGE_BYTES / 2) + rr * 128;
          const uint4 v0 = *reinterpret_cast<const uint4*>(row + (((2 * rq) ^ (rr & 7)) << 4));
          const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((2 * rq + 1) ^ (rr & 7)) << 4));
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          const float a = absmax_words(w, 8);
          amax_local = fmaxf(amax_local, a);
          const BlockScale bs = block_scale_tab<FMT, true>(a, s_enc, rtab);
          maxc_row = max(maxc_row, bs.code);
          const int64_t grow = m0 + rr, gcol = k0 + 16 * c;
          const uint2 q = quant16<ROW_SR>(
              w, bs.r, key_row, SrIdx32{(uint32_t)grow * (uint32_t)(p.K >> 3) + (uint32_t)(gcol >> 3)});
          *reinterpret_cast<uint2*>(p.codes_row + grow * (p.K / 2) + gcol / 2) = q;
          stg_sfr[qd_sf_off(rr, c)] = (uint8_t)bs.code;
        }
      }
      {
        uint32_t v[16];
        const uint8_t* box = stage + cbox * (QD_STAGE_BYTES / 2);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = 16 * crb + i;
          v[i] = *reinterpret_cast<const uint32_t*>(box + r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4);
        }
        const uint32_t am2 = absmax_words2(v, 16);  // both columns' block maxima
        const float a_lo = bf16_lo(am2), a_hi = bf16_hi(am2);
        if constexpr (!DO_ROW) amax_local = fmaxf(amax_local, fmaxf(a_lo, a_hi));
        const BlockScale b0 = block_scale_tab<FMT, true>(a_lo, s_enc, rtab);
        const BlockScale b1 = block_scale_tab<FMT, true>(a_hi, s_enc, rtab);
        maxc_col = max(maxc_col, max(b0.code, b1.code));
        const int c0 = 64 * cbox + 2 * lane;  // tile column of the low half
        // Philox blocks of output elements (k0 + c0) M + m0 + 16 crb and the next row of the output
        const uint32_t blk0 = (uint32_t)(k0 + c0) * (uint32_t)(p.M >> 3) + (uint32_t)((m0 + 16 * crb) >> 3);
        const uint2 q0 = quant16_col<COL_SR, false>(v, b0.r, key_col, SrIdx32{blk0});
        const uint2 q1 = quant16_col<COL_SR, true>(v, b1.r, key_col, SrIdx32{blk0 + (uint32_t)(p.M >> 3)});
        // staged transposed codes: output row c, bytes 8 crb .. +7 (64-byte swizzle)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = c0 + h;
          *reinterpret_cast<uint2*>(stg_colc + c * 64 + (((crb >> 1) ^ ((c >> 1) & 3)) << 4) + (crb & 1) * 8) =
              h ? q1 : q0;
        }
        stg_sfc[qd_sf_off(c0, crb)] = (uint8_t)b0.code;
        stg_sfc[qd_sf_off(c0 + 1, crb)] = (uint8_t)b1.code;
      }
      // the stage may refill; the staged outputs go to the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_empty + 8 * s);
        mbar_arrive(bar_stg_full + 8 * b);
      }
    }
    if constexpr (AMAX) {
      const unsigned int am = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_local));
      if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), am);
    }
    if constexpr (FMT == SF_UE5M3) {
      if (DO_ROW && p.sf_max_row != nullptr) {
        const unsigned int mc = __reduce_max_sync(0xFFFFFFFFu, maxc_row);
        if (lane == 0) atomicMax(p.sf_max_row, mc);
      }
      if (p.sf_max_col != nullptr) {
        const unsigned int mc = __reduce_max_sync(0xFFFFFFFFu, maxc_col);
        if (lane == 0) atomicMax(p.sf_max_col, mc);
      }
    }
  } else {
    // ------------------------------ storer --------------------------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_ccol)) : "memory");
      int it = 0;
      TileWalk tw(blockIdx.x, gridDim.x, m_tiles);
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it, tw.next()) {
        const int b = it & 1;
        if (!wait_bounded(bar_stg_full + 8 * b, (it >> 1) & 1, abort_flag, p.status)) break;
        const int m0 = tw.mt * QD_T, k0 = tw.kt * QD_T;
        const uint32_t stg = sbase + QD_SMEM_STG + b * QD_STG_BYTES;
        qd_tma_store_2d(&tm_ccol, stg, m0 / 2, k0);
        if (DO_ROW)
          qd_bulk_store(p.scales_row + ((int64_t)(m0 / QD_T) * (p.K / 64) + k0 / 64) * 512, stg + QD_COLC_BYTES,
                        QD_SF_BYTES);
        qd_bulk_store(p.scales_col + ((int64_t)(k0 / QD_T) * (p.M / 64) + m0 / 64) * 512,
                      stg + QD_COLC_BYTES + QD_SF_BYTES, QD_SF_BYTES);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        // the staging buffer is free once these copies have read it
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        mbar_arrive(bar_stg_free + 8 * b);
      }
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
  }
  __syncwarp();
  __syncthreads();
  drain_after_abort(abort_flag);
}

// ---------------------------------------------------------------------------
// K4: dequantize
// ---------------------------------------------------------------------------
__device__ __forceinline__ float e2m1_value(uint32_t n) {
  const uint32_t m = n & 7u;
  float v = (m < 2u) ? (m == 1u ? 0.5f : 0.0f)
                     : __uint_as_float(((126u + (m >> 1)) << 23) | ((m & 1u) << 22));
  return (n & 8u) ? -v : v;
}

template <int FMT, bool MMA, bool BF16>
__global__ void __launch_bounds__(256) k_dequant(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                                 int64_t M, int64_t K, const float* __restrict__ gptr,
                                                 void* __restrict__ out) {
  constexpr int G = ScaleFmt<FMT>::G;
  const int64_t per_row = K / 16;
  const int64_t chunk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (chunk >= M * per_row) return;
  const float s_enc = global_encode_scale<FMT>(__ldg(gptr), nullptr);
  const int64_t row = chunk / per_row, c16 = chunk - row * per_row;
  const int64_t b = c16 * 16 / G, nb = K / G;
  const uint32_t code = scales[MMA ? mma_sf_offset(row, b, nb) : row * nb + b];
  const float s_b = ScaleFmt<FMT>::decode(code);
  const uint2 q = *reinterpret_cast<const uint2*>(codes + row * (K / 2) + c16 * 8);
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = i < 8 ? q.x : q.y;
    const uint32_t n = (word >> (4 * (i & 7))) & 0xFu;
    const float e = Elem<FMT>::INT4 ? (float)((int)n - ((int)n & 8) * 2) : e2m1_value(n);
    v[i] = __fdiv_rn(__fmul_rn(e, s_b), s_enc);
  }
  if constexpr (BF16) {
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + row * K + c16 * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row * K + c16 * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// ---------------------------------------------------------------------------
// K8: UE5M3 -> E4M3 re-encode with a per-tensor power-of-two shift
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_ue5m3_maxcode(const uint8_t* __restrict__ s, int64_t n, int32_t* acc) {
  unsigned int m = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    m = max(m, (unsigned int)s[i]);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m > 0) atomicMax(reinterpret_cast<unsigned int*>(acc), m);
}

// t = e_max - 7 from the largest UE5M3 code (codes order like their values)
__device__ __forceinline__ int ue5m3_shift_from_maxcode(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  if (e > 0) return (int)e - 15 - 7;
  if (m == 0) return 0;
  return (31 - __clz(m)) - 17 - 7;  // m * 2^-17, floor(log2 m) in 0..2
}

// FROM_CODE: *tword holds the largest UE5M3 code (the shift follows from it);
// otherwise *tword is the shift t itself.
template <bool FROM_CODE>
__global__ void __launch_bounds__(256) k_ue5m3_reencode(const uint8_t* __restrict__ s, int64_t n,
                                                        const int32_t* tword, uint8_t* __restrict__ out,
                                                        int32_t* status) {
  const int t = FROM_CODE ? ue5m3_shift_from_maxcode((uint32_t)__ldg(tword)) : (int)__ldg(tword);
  // 2^-t as a float (|t| <= 26)
  const float scale = __uint_as_float((uint32_t)(127 - t) << 23);
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = __fmul_rn(ScaleFmt<SF_UE5M3>::decode(s[i]), scale);  // exact
    const uint32_t c = ScaleFmt<SF_E4M3>::encode(v);
    bad |= ScaleFmt<SF_E4M3>::decode(c) != v;
    out[i] = (uint8_t)c;
  }
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) set_status(status, FP4_ERR_UE5M3_RANGE);
}

// n words, each the largest UE5M3 code of a scale set, become its shift t
__global__ void k_ue5m3_finalize(int32_t* t_inout, int n) {
  if ((int)threadIdx.x < n) t_inout[threadIdx.x] = ue5m3_shift_from_maxcode((uint32_t)t_inout[threadIdx.x]);
}

// UE5M3 scales wider than one E4M3 window: with e_max the largest exponent
// (t_0 = e_max - 7), scale s with exponent e goes to window
// w = (e_max - e) / 14 and is re-encoded as E4M3 of s * 2^-(t_0 - 14 w), which
// is exact (e - t_w lies in -6..7 and s has at most 4 significant bits).
// out holds UE5M3_WINDOWS arrays of n codes; other windows get code 0.
constexpr int UE5M3_WINDOWS = 3;
constexpr int UE5M3_WINDOW_BINADES = 14;

__global__ void __launch_bounds__(256) k_ue5m3_windows(const uint8_t* __restrict__ s, int64_t n,
                                                       const int32_t* maxcode, uint8_t* __restrict__ out,
                                                       int32_t* wmax, int32_t* status) {
  const int e_max = ue5m3_shift_from_maxcode((uint32_t)__ldg(maxcode)) + 7;
  int top = 0;
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = ScaleFmt<SF_UE5M3>::decode(s[i]);
    uint8_t c[UE5M3_WINDOWS] = {0, 0, 0};
    if (v > 0.0f) {
      const int e = (int)((__float_as_uint(v) >> 23) & 0xFFu) - 127;  // UE5M3 values are normal floats
      const int w = (e_max - e) / UE5M3_WINDOW_BINADES;
      const int t = e_max - 7 - UE5M3_WINDOW_BINADES * w;
      const float u = __fmul_rn(v, __uint_as_float((uint32_t)(127 - t) << 23));  // exact
      const uint32_t code = ScaleFmt<SF_E4M3>::encode(u);
      bad |= w >= UE5M3_WINDOWS || ScaleFmt<SF_E4M3>::decode(code) != u;
      if (w < UE5M3_WINDOWS) c[w] = (uint8_t)code;
      top = max(top, w + 1);
    }
#pragma unroll
    for (int k = 0; k < UE5M3_WINDOWS; ++k) out[k * n + i] = c[k];
  }
  top = __reduce_max_sync(0xFFFFFFFFu, top);
  if ((threadIdx.x & 31) == 0 && top > 0) atomicMax(wmax, top);
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) set_status(status, FP4_ERR_UE5M3_RANGE);
}

// t_out[0] held the largest code; n_out the number of windows in use (0 for
// an all-zero tensor)
__global__ void k_ue5m3_windows_finalize(int32_t* t_out, int32_t* n_out) {
  const int t0 = ue5m3_shift_from_maxcode((uint32_t)t_out[0]);
#pragma unroll
  for (int k = 0; k < UE5M3_WINDOWS; ++k) t_out[k] = t0 - UE5M3_WINDOW_BINADES * k;
  *n_out = max(*n_out, 1);
}

// ---------------------------------------------------------------------------
// Conformance helpers
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void __launch_bounds__(256) k_encode_scales(const float* __restrict__ s, int64_t n, uint8_t* codes,
                                                       float* decoded) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint32_t c;
  if constexpr (e8m0_scales<FMT>()) c = ScaleFmt<SF_E8M0>::encode_from_amax(s[i]);
  else c = ScaleFmt<FMT>::encode(s[i]);
  codes[i] = (uint8_t)c;
  decoded[i] = ScaleFmt<FMT>::decode(c);
}

__global__ void __launch_bounds__(256) k_philox_bits16(uint64_t seed, uint64_t start, int64_t n, uint16_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint64_t idx = start + (uint64_t)i;
  const uint4 d = sr_draws8(seed, idx >> 3);
  out[i] = (uint16_t)draw16(d, (int)(idx & 7));
}

inline unsigned grid_for(int64_t items, int per_block = 256) {
  return (unsigned)((items + per_block - 1) / per_block);
}

}  // namespace

// ===========================================================================
// Launchers (called by the C ABI after argument checks)
// ===========================================================================
namespace fp4lib {

cudaError_t launch_amax(const void* x, int64_t M, int64_t K, int64_t ldx, float* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  if (M == 0 || K == 0) return cudaSuccess;
  const int64_t chunks = M * (K / 8);
  int64_t blocks = (chunks + 255) / 256;
  const int64_t cap = 152 * 8;
  if (blocks > cap) blocks = cap;
  k_amax<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(x), M, K, ldx, out);
  return cudaGetLastError();
}

cudaError_t launch_amax_n(int n, const void* const* x, const int64_t* M, const int64_t* K, const int64_t* ldx,
                          float* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * n, st);
  if (e != cudaSuccess || n == 0) return e;
  AmaxN a{};
  a.n = n;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) total += M[i] * (K[i] / 8);
  if (total == 0) return cudaSuccess;
  // as many threads as one fp4_amax launch, shared out by size (at least one CTA each)
  const int64_t cap = 152 * 8 * (256 / AMAXN_THREADS);
  int64_t blocks_total = (total + AMAXN_THREADS - 1) / AMAXN_THREADS;
  if (blocks_total > cap) blocks_total = cap;
  int begin = 0;
  for (int i = 0; i < n; ++i) {
    a.x[i] = static_cast<const uint16_t*>(x[i]);
    a.M[i] = M[i];
    a.K[i] = K[i];
    a.ldx[i] = ldx[i];
    a.cta_begin[i] = begin;
    const int64_t chunks = M[i] * (K[i] / 8);
    int64_t nb = (chunks * blocks_total + total - 1) / total;
    nb = nb < 1 ? 1 : nb;
    begin += (int)nb;
  }
  a.cta_begin[n] = begin;
  k_amax_n<<<(unsigned)begin, AMAXN_THREADS, 0, st>>>(a, out);
  return cudaGetLastError();
}

template <int FMT, bool SR, bool MMA, bool AMAX>
static void rows_t(const QuantArgs& a, cudaStream_t st) {
  const int64_t chunks = a.M * (a.K / 16);
  if (chunks == 0) return;
  k_quant_rows<FMT, SR, MMA, AMAX><<<grid_for(chunks), 256, 0, st>>>(
      static_cast<const uint16_t*>(a.x), a.M, a.K, a.ldx, a.gptr, a.seed_row, a.codes_row, a.scales_row,
      a.amax_out, a.status, a.sf_max_row);
}

template <int FMT, bool DUAL, bool RSR, bool CSR, bool MMA, bool AMAX>
static void tile_t(const QuantArgs& a, cudaStream_t st) {
  if (a.M == 0 || a.K == 0) return;
  dim3 grid((unsigned)((a.M + TILE_M - 1) / TILE_M), (unsigned)((a.K + TILE_K - 1) / TILE_K));
  k_quant_tile<FMT, DUAL, RSR, CSR, MMA, AMAX><<<grid, 256, 0, st>>>(
      static_cast<const uint16_t*>(a.x), a.M, a.K, a.ldx, a.gptr, a.seed_row, a.seed_col, a.codes_row,
      a.scales_row, a.codes_col, a.scales_col, a.amax_out, a.status, a.sf_max_row, a.sf_max_col);
}

// The TMA-fed dual / transposed quantizer: 16-element blocks, tiled scale
// layout, M and K multiples of 128.  cudaErrorNotSupported (before any
// launch) sends the call to k_quant_tile instead.
template <int FMT, bool DO_ROW, bool RSR, bool CSR, bool AM>
static cudaError_t dual_tma_t(const QuantArgs& a, cudaStream_t st) {
  auto fn = fp4async::encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  CUtensorMap mx, mc;
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    cuuint64_t strides[1] = {(cuuint64_t)(a.ldx * 2)};
    cuuint32_t box[2] = {64u, (cuuint32_t)QD_T};
    cuuint32_t estr[2] = {1u, 1u};
    if (fn(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)(a.M / 2), (cuuint64_t)a.K};
    cuuint64_t strides[1] = {(cuuint64_t)(a.M / 2)};
    cuuint32_t box[2] = {64u, (cuuint32_t)QD_T};
    cuuint32_t estr[2] = {1u, 1u};
    if (fn(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.codes_col, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
  }
  auto kern = k_quant_dual_tma<FMT, DO_ROW, RSR, CSR, AM>;
  static fp4lib::DeviceInts attr_set;
  cudaError_t e = cudaSuccess;
  attr_set.get([&] {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QD_SMEM_LAUNCH);
    return e == cudaSuccess ? 1 : 0;
  });
  if (e != cudaSuccess) return e;
  QdParams p{};
  p.gptr = a.gptr;
  p.seed_row = a.seed_row;
  p.seed_col = a.seed_col;
  p.M = a.M;
  p.K = a.K;
  p.codes_row = a.codes_row;
  p.scales_row = a.scales_row;
  p.scales_col = a.scales_col;
  p.amax_out = a.amax_out;
  p.status = a.status;
  p.sf_max_row = a.sf_max_row;
  p.sf_max_col = a.sf_max_col;
  const int64_t tiles = (a.M / QD_T) * (a.K / QD_T);
  const int sms = fp4lib::current_sm_count();
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  kern<<<grid, QD_THREADS, QD_SMEM_LAUNCH, st>>>(mx, mc, p);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t dispatch_dual_tma(const QuantArgs& a, cudaStream_t st) {
  if constexpr (ScaleFmt<FMT>::G != 16 || Elem<FMT>::INT4) {
    return cudaErrorNotSupported;
  } else {
    if (!a.mma || a.M % QD_T != 0 || a.K % QD_T != 0 || a.M == 0 || a.K == 0) return cudaErrorNotSupported;
    // the kernel's Philox block indices (element index / 8) are 32-bit
    if ((a.M >> 3) * a.K > (int64_t)0xFFFFFFFF) return cudaErrorNotSupported;
    const bool amax = a.amax_by_product;
    if (a.mode == QuantArgs::DUAL) {
#define DT_CASE(RS, CS, AM) \
  if (a.row_sr == RS && a.col_sr == CS && amax == AM) return dual_tma_t<FMT, true, RS, CS, AM>(a, st);
      DT_CASE(false, false, false) DT_CASE(false, false, true) DT_CASE(false, true, false) DT_CASE(false, true, true)
      DT_CASE(true, false, false) DT_CASE(true, false, true) DT_CASE(true, true, false) DT_CASE(true, true, true)
#undef DT_CASE
    } else if (a.mode == QuantArgs::COLS) {
      if (a.col_sr && amax) return dual_tma_t<FMT, false, false, true, true>(a, st);
      if (a.col_sr) return dual_tma_t<FMT, false, false, true, false>(a, st);
      if (amax) return dual_tma_t<FMT, false, false, false, true>(a, st);
      return dual_tma_t<FMT, false, false, false, false>(a, st);
    }
    return cudaErrorNotSupported;
  }
}

// runtime -> template dispatch
template <int FMT>
static void dispatch_fmt(const QuantArgs& a, cudaStream_t st) {
  const bool amax = a.amax_by_product;
  if (a.mode == QuantArgs::ROWS) {
#define ROWS_CASE(SR, MMA, AM) \
  if (a.row_sr == SR && a.mma == MMA && amax == AM) return rows_t<FMT, SR, MMA, AM>(a, st);
    ROWS_CASE(false, false, false) ROWS_CASE(false, false, true) ROWS_CASE(false, true, false)
    ROWS_CASE(false, true, true) ROWS_CASE(true, false, false) ROWS_CASE(true, false, true)
    ROWS_CASE(true, true, false) ROWS_CASE(true, true, true)
#undef ROWS_CASE
  } else {
    const bool dual = a.mode == QuantArgs::DUAL;
#define TILE_CASE(D, RS, CS, MMA, AM)                                                           \
  if (dual == D && (!D || a.row_sr == RS) && a.col_sr == CS && a.mma == MMA && amax == AM) \
    return tile_t<FMT, D, RS, CS, MMA, AM>(a, st);
#define TILE_CASES(D, RS) \
  TILE_CASE(D, RS, false, false, false) TILE_CASE(D, RS, false, false, true) \
  TILE_CASE(D, RS, false, true, false) TILE_CASE(D, RS, false, true, true)   \
  TILE_CASE(D, RS, true, false, false) TILE_CASE(D, RS, true, false, true)   \
  TILE_CASE(D, RS, true, true, false) TILE_CASE(D, RS, true, true, true)
    TILE_CASES(false, false) TILE_CASES(true, false) TILE_CASES(true, true)
#undef TILE_CASES
#undef TILE_CASE
  }
}

// The rest of the scale-format sweep: row quantization only.
template <int FMT>
static cudaError_t dispatch_rows_only(const QuantArgs& a, cudaStream_t st) {
  if (a.mode != QuantArgs::ROWS) return cudaErrorNotSupported;
  const bool amax = a.amax_by_product;
#define ROWS_CASE(SR, MMA, AM) \
  if (a.row_sr == SR && a.mma == MMA && amax == AM) rows_t<FMT, SR, MMA, AM>(a, st);
  ROWS_CASE(false, false, false) ROWS_CASE(false, false, true) ROWS_CASE(false, true, false)
  ROWS_CASE(false, true, true) ROWS_CASE(true, false, false) ROWS_CASE(true, false, true)
  ROWS_CASE(true, true, false) ROWS_CASE(true, true, true)
#undef ROWS_CASE
  return cudaSuccess;
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st) {
  cudaError_t e = cudaErrorNotSupported;
  if (a.mode != QuantArgs::ROWS) {
    switch (a.fmt) {
      case FP4_SF_E4M3: e = dispatch_dual_tma<SF_E4M3>(a, st); break;
      case FP4_SF_UE5M3: e = dispatch_dual_tma<SF_UE5M3>(a, st); break;
      case FP4_SF_E1M6: e = dispatch_dual_tma<SF_E1M6>(a, st); break;
      default: break;
    }
    if (e != cudaErrorNotSupported) return e;
  }
  e = cudaSuccess;
  switch (a.fmt) {
    case FP4_SF_E4M3: dispatch_fmt<SF_E4M3>(a, st); break;
    case FP4_SF_UE5M3: dispatch_fmt<SF_UE5M3>(a, st); break;
    case FP4_SF_E8M0: dispatch_fmt<SF_E8M0>(a, st); break;
    case FP4_SF_E1M6: dispatch_fmt<SF_E1M6>(a, st); break;
    case FP4_SF_E2M5: e = dispatch_rows_only<SF_E2M5>(a, st); break;
    case FP4_SF_E3M4: e = dispatch_rows_only<SF_E3M4>(a, st); break;
    case FP4_SF_E5M2: e = dispatch_rows_only<SF_E5M2>(a, st); break;
    case FP4_SF_E6M1: e = dispatch_rows_only<SF_E6M1>(a, st); break;
    case FP4_SF_E7M0: e = dispatch_rows_only<SF_E7M0>(a, st); break;
    case FP4_SF_NVINT4: e = dispatch_rows_only<SF_NVINT4>(a, st); break;
    case FP4_SF_MXINT4: e = dispatch_rows_only<SF_MXINT4>(a, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, bool mma, int64_t M, int64_t K,
                              int fmt, const float* gptr, bool bf16, void* out, cudaStream_t st) {
  const int64_t chunks = M * (K / 16);
  if (chunks == 0) return cudaSuccess;
  const unsigned g = grid_for(chunks);
#define DQ(F)                                                                                           \
  if (mma && bf16) k_dequant<F, true, true><<<g, 256, 0, st>>>(codes, scales, M, K, gptr, out);         \
  else if (mma) k_dequant<F, true, false><<<g, 256, 0, st>>>(codes, scales, M, K, gptr, out);           \
  else if (bf16) k_dequant<F, false, true><<<g, 256, 0, st>>>(codes, scales, M, K, gptr, out);          \
  else k_dequant<F, false, false><<<g, 256, 0, st>>>(codes, scales, M, K, gptr, out);
  switch (fmt) {
    case FP4_SF_E4M3: DQ(SF_E4M3) break;
    case FP4_SF_UE5M3: DQ(SF_UE5M3) break;
    case FP4_SF_E8M0: DQ(SF_E8M0) break;
    case FP4_SF_E1M6: DQ(SF_E1M6) break;
    case FP4_SF_E2M5: DQ(SF_E2M5) break;
    case FP4_SF_E3M4: DQ(SF_E3M4) break;
    case FP4_SF_E5M2: DQ(SF_E5M2) break;
    case FP4_SF_E6M1: DQ(SF_E6M1) break;
    case FP4_SF_E7M0: DQ(SF_E7M0) break;
    case FP4_SF_NVINT4: DQ(SF_NVINT4) break;
    case FP4_SF_MXINT4: DQ(SF_MXINT4) break;
    default: return cudaErrorInvalidValue;
  }
#undef DQ
  return cudaGetLastError();
}

cudaError_t launch_ue5m3_to_e4m3(const uint8_t* in, int64_t n, int32_t* t_out, uint8_t* out, int32_t* status,
                                 cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(t_out, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    k_ue5m3_maxcode<<<(unsigned)blocks, 256, 0, st>>>(in, n, t_out);
    k_ue5m3_reencode<true><<<(unsigned)blocks, 256, 0, st>>>(in, n, t_out, out, status);
  }
  k_ue5m3_finalize<<<1, 32, 0, st>>>(t_out, 1);
  return cudaGetLastError();
}

cudaError_t launch_ue5m3_reencode(const uint8_t* in, int64_t n, const int32_t* t, uint8_t* out, int32_t* status,
                                  cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  k_ue5m3_reencode<false><<<(unsigned)blocks, 256, 0, st>>>(in, n, t, out, status);
  return cudaGetLastError();
}

cudaError_t launch_ue5m3_finalize(int32_t* words, int n, cudaStream_t st) {
  k_ue5m3_finalize<<<1, 32, 0, st>>>(words, n);
  return cudaGetLastError();
}

cudaError_t launch_ue5m3_windows(const uint8_t* in, int64_t n, int32_t* t_out, int32_t* n_out, uint8_t* out,
                                 int32_t* status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(t_out, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(n_out, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    k_ue5m3_maxcode<<<(unsigned)blocks, 256, 0, st>>>(in, n, t_out);
    k_ue5m3_windows<<<(unsigned)blocks, 256, 0, st>>>(in, n, t_out, out, n_out, status);
  }
  k_ue5m3_windows_finalize<<<1, 1, 0, st>>>(t_out, n_out);
  return cudaGetLastError();
}

cudaError_t launch_encode_scales(const float* s, int64_t n, int fmt, uint8_t* codes, float* decoded,
                                 cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const unsigned g = grid_for(n);
  switch (fmt) {
    case FP4_SF_E4M3: k_encode_scales<SF_E4M3><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_UE5M3: k_encode_scales<SF_UE5M3><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E8M0: k_encode_scales<SF_E8M0><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E1M6: k_encode_scales<SF_E1M6><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E2M5: k_encode_scales<SF_E2M5><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E3M4: k_encode_scales<SF_E3M4><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E5M2: k_encode_scales<SF_E5M2><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E6M1: k_encode_scales<SF_E6M1><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_E7M0: k_encode_scales<SF_E7M0><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_NVINT4: k_encode_scales<SF_NVINT4><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    case FP4_SF_MXINT4: k_encode_scales<SF_MXINT4><<<g, 256, 0, st>>>(s, n, codes, decoded); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_philox_bits16(uint64_t seed, uint64_t start, int64_t n, uint16_t* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  k_philox_bits16<<<grid_for(n), 256, 0, st>>>(seed, start, n, out);
  return cudaGetLastError();
}

}  // namespace fp4lib
