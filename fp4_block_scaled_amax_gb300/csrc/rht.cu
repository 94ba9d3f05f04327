// 16 x 16 random Hadamard transform fused into the row quantizer (sm_103a).
//
// "UE5M3 FP4 Block Scaling ..." blog, section "Что сделали": the randomized
// Hadamard transform spreads outliers before quantization (and the UE5M3
// recipe drops it); post on "INT v.s. FP: A Comprehensive Study of
// Fine-Grained Low-bit Quantization Formats" (quant_prune_distill channel
// page), section "Метод": Hadamard rotations make weights and activations
// closer to Gaussian before MX/NV FP or INT quantization.
//
// Every 16-element block along K becomes x' = 1/4 * H16 * (s . x) (float32
// fast Walsh-Hadamard butterflies, fp4dev::rht16), and the method of
// fp4_quantize then runs on x': block amax, scale, element rounding, packing.
// The global amax is max |x'| over the tensor.
//   k_amax_rht        fresh global amax of the transformed tensor (blocks along K).
//   k_amax_rht_cols   the same with the transform along M (transposed layout).
//   k_quant_rows_rht  one thread per 16 elements: two 128-bit loads, the
//                     transform in registers, quantization, one 8-byte store.
//   k_quant_dual_rht  64 x 128 tile staged in shared memory: rows transformed
//                     along K, the transposed output along M (16-row blocks),
//                     each quantized under its own global amax.
#include <cstdint>
#include <cuda_runtime.h>

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

// 16 bf16 values of one block (two 16-byte loads) -> 16 floats
__device__ __forceinline__ void load_block(const uint16_t* src, float (&v)[16]) {
  const uint4 a = ld_stream(src), b = ld_stream(src + 8);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

__device__ __forceinline__ float absmax16(const float (&v)[16]) {
  float a = fabsf(v[0]);
#pragma unroll
  for (int i = 1; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
  return a;
}

__global__ void __launch_bounds__(256) k_amax_rht(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                  uint32_t mask, float* __restrict__ out) {
  const int64_t per_row = K / 16;
  const int64_t n = M * per_row;
  float m = 0.0f;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = c / per_row, c16 = c - row * per_row;
    float v[16];
    load_block(x + row * ldx + c16 * 16, v);
    rht16(v, mask);
    m = fmaxf(m, absmax16(v));
  }
  // non-negative floats order like their bit patterns
  const unsigned int am = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(out), am);
}

template <int FMT, bool SR, bool MMA, bool AMAX>
__global__ void __launch_bounds__(256) k_quant_rows_rht(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                        int64_t ldx, uint32_t mask, const float* __restrict__ gptr,
                                                        uint64_t seed, uint8_t* __restrict__ codes,
                                                        uint8_t* __restrict__ scales, float* __restrict__ amax_out,
                                                        int32_t* status) {
  constexpr int G = ScaleFmt<FMT>::G;
  const int64_t per_row = K / 16;
  const int64_t chunk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = chunk < M * per_row;
  const unsigned vmask = __ballot_sync(0xFFFFFFFFu, valid);
  if (!valid) return;
  const float s_enc = global_encode_scale<FMT>(__ldg(gptr), (blockIdx.x == 0 && threadIdx.x == 0) ? status : nullptr);
  const int64_t row = chunk / per_row;
  const int64_t c16 = chunk - row * per_row;
  float v[16];
  load_block(x + row * ldx + c16 * 16, v);
  rht16(v, mask);
  float a = absmax16(v);
  if constexpr (AMAX) {
    const unsigned int am = __reduce_max_sync(vmask, __float_as_uint(a));
    if ((threadIdx.x & 31) == (unsigned)(__ffs(vmask) - 1)) atomicMax(reinterpret_cast<unsigned int*>(amax_out), am);
  }
  if constexpr (G == 32) a = fmaxf(a, __shfl_xor_sync(vmask, a, 1));
  const BlockScale bs = block_scale<FMT>(a, s_enc);
  const uint2 q = quant16f<SR, Elem<FMT>::INT4>(v, bs.r, seed, (uint64_t)(row * K + c16 * 16));
  *reinterpret_cast<uint2*>(codes + row * (K / 2) + c16 * 8) = q;
  if (G == 16 || (c16 & 1) == 0) {
    const int64_t b = c16 * 16 / G;
    const int64_t nb = K / G;
    scales[MMA ? mma_sf_offset(row, b, nb) : row * nb + b] = (uint8_t)bs.code;
  }
}

// max |x'| with the transform along M: unit u = (16-row block u / K, column
// u % K); neighbouring threads read neighbouring columns of each row.
__global__ void __launch_bounds__(256) k_amax_rht_cols(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                       int64_t ldx, uint32_t mask, float* __restrict__ out) {
  const int64_t n = (M / 16) * K;
  float m = 0.0f;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rb = u / K, c = u - rb * K;
    const uint16_t* src = x + rb * 16 * ldx + c;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float((uint32_t)__ldg(src + i * ldx) << 16);
    rht16(v, mask);
    m = fmaxf(m, absmax16(v));
  }
  const unsigned int am = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned int*>(out), am);
}

constexpr int TILE_M = 64;
constexpr int TILE_K = 128;
// 32-row halves of the tile use column-swizzled halves (no bank conflicts in
// the column pass)
__device__ __forceinline__ int tile_col(int r, int c) { return c ^ (((r >> 5) & 1) << 4); }

// Row (transform along K) and transposed (transform along M) quantization of a
// 64 x 128 tile; the transposed output's blocks are 16 rows (one transform) or
// 32 rows (two transforms, one scale) long.  M % 32 == 0, K % 32 == 0.
template <int FMT, bool RSR, bool CSR, bool MMA, bool AMAX>
__global__ void __launch_bounds__(256) k_quant_dual_rht(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx, uint32_t mask,
    const float* __restrict__ g_row, const float* __restrict__ g_col, uint64_t seed_row, uint64_t seed_col,
    uint8_t* __restrict__ codes_row, uint8_t* __restrict__ scales_row, uint8_t* __restrict__ codes_col,
    uint8_t* __restrict__ scales_col, float* __restrict__ amax_row_out, float* __restrict__ amax_col_out,
    int32_t* status) {
  constexpr int G = ScaleFmt<FMT>::G;
  __shared__ __align__(16) uint16_t tile[TILE_M][TILE_K];
  const int64_t m0 = (int64_t)blockIdx.x * TILE_M;
  const int64_t k0 = (int64_t)blockIdx.y * TILE_K;
  const bool first = blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
  const float se_row = global_encode_scale<FMT>(__ldg(g_row), first ? status : nullptr);
  const float se_col = global_encode_scale<FMT>(__ldg(g_col), first ? status : nullptr);

  uint32_t w[2][8];
  bool valid[2];
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int j = threadIdx.x + 256 * it;
    const int r = j >> 3, cc = j & 7;
    const int64_t col = k0 + cc * 16;
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
  float amax_row = 0.0f;
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int j = threadIdx.x + 256 * it;
    const int r = j >> 3, cc = j & 7;
    uint4* dst = reinterpret_cast<uint4*>(&tile[r][tile_col(r, cc * 16)]);
    dst[0] = make_uint4(w[it][0], w[it][1], w[it][2], w[it][3]);
    dst[1] = make_uint4(w[it][4], w[it][5], w[it][6], w[it][7]);
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(w[it][i]);
      v[2 * i + 1] = bf16_hi(w[it][i]);
    }
    rht16(v, mask);
    float a = absmax16(v);
    amax_row = fmaxf(amax_row, a);
    if constexpr (G == 32) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    if (valid[it]) {
      const int64_t row = m0 + r, col = k0 + cc * 16;
      const BlockScale bs = block_scale<FMT>(a, se_row);
      const uint2 q = quant16f<RSR, false>(v, bs.r, seed_row, (uint64_t)(row * K + col));
      *reinterpret_cast<uint2*>(codes_row + row * (K / 2) + col / 2) = q;
      if (G == 16 || (cc & 1) == 0) {
        const int64_t b = col / G, nb = K / G;
        scales_row[MMA ? mma_sf_offset(row, b, nb) : row * nb + b] = (uint8_t)bs.code;
      }
    }
  }
  __syncthreads();

  // ---- transposed output: thread t owns column k0 + t/2, rows m0 + 32*(t%2) .. +31 ----
  const int cl = threadIdx.x >> 1, h = threadIdx.x & 1;
  const int64_t c = k0 + cl;
  const int64_t rbase = m0 + 32 * h;
  float amax_col = 0.0f;
  if (c < K && rbase < M) {
    const int pc = cl ^ (h << 4);
    float f0[16], f1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      f0[i] = __uint_as_float((uint32_t)tile[32 * h + i][pc] << 16);
      f1[i] = __uint_as_float((uint32_t)tile[32 * h + 16 + i][pc] << 16);
    }
    rht16(f0, mask);
    rht16(f1, mask);
    const float a0 = absmax16(f0), a1 = absmax16(f1);
    amax_col = fmaxf(a0, a1);
    const uint64_t idx0 = (uint64_t)(c * M + rbase);
    uint2 q0, q1;
    uint32_t sc0, sc1 = 0;
    if constexpr (G == 16) {
      const BlockScale b0 = block_scale<FMT>(a0, se_col);
      const BlockScale b1 = block_scale<FMT>(a1, se_col);
      q0 = quant16f<CSR, false>(f0, b0.r, seed_col, idx0);
      q1 = quant16f<CSR, false>(f1, b1.r, seed_col, idx0 + 16);
      sc0 = b0.code;
      sc1 = b1.code;
    } else {
      const BlockScale b0 = block_scale<FMT>(amax_col, se_col);
      q0 = quant16f<CSR, false>(f0, b0.r, seed_col, idx0);
      q1 = quant16f<CSR, false>(f1, b0.r, seed_col, idx0 + 16);
      sc0 = b0.code;
    }
    *reinterpret_cast<uint4*>(codes_col + c * (M / 2) + rbase / 2) = make_uint4(q0.x, q0.y, q1.x, q1.y);
    const int64_t nb = M / G, b = rbase / G;
    if constexpr (G == 16) {
      const int64_t off = MMA ? mma_sf_offset(c, b, nb) : c * nb + b;
      *reinterpret_cast<uint16_t*>(scales_col + off) = (uint16_t)(sc0 | (sc1 << 8));
    } else {
      scales_col[MMA ? mma_sf_offset(c, b, nb) : c * nb + b] = (uint8_t)sc0;
    }
  }
  if constexpr (AMAX) {
    const unsigned int ar = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_row));
    const unsigned int ac = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_col));
    if ((threadIdx.x & 31) == 0) {
      atomicMax(reinterpret_cast<unsigned int*>(amax_row_out), ar);
      atomicMax(reinterpret_cast<unsigned int*>(amax_col_out), ac);
    }
  }
}

unsigned grid_for(int64_t n) { return (unsigned)((n + 255) / 256); }

template <int FMT>
cudaError_t dispatch_dual(const fp4lib::DualRhtArgs& a, cudaStream_t st) {
  if (a.M == 0 || a.K == 0) return cudaSuccess;
  dim3 grid((unsigned)((a.M + TILE_M - 1) / TILE_M), (unsigned)((a.K + TILE_K - 1) / TILE_K));
#define DUAL_CASE(RS, CS, MMA, AM)                                                                             \
  if (a.row_sr == RS && a.col_sr == CS && a.mma == MMA && a.amax_by_product == AM) {                         \
    k_quant_dual_rht<FMT, RS, CS, MMA, AM><<<grid, 256, 0, st>>>(                                            \
        static_cast<const uint16_t*>(a.x), a.M, a.K, a.ldx, a.mask, a.g_row, a.g_col, a.seed_row, a.seed_col, \
        a.codes_row, a.scales_row, a.codes_col, a.scales_col, a.amax_row_out, a.amax_col_out, a.status);      \
    return cudaGetLastError();                                                                                 \
  }
#define DUAL_CASES(RS, CS) DUAL_CASE(RS, CS, false, false) DUAL_CASE(RS, CS, false, true) \
  DUAL_CASE(RS, CS, true, false) DUAL_CASE(RS, CS, true, true)
  DUAL_CASES(false, false) DUAL_CASES(false, true) DUAL_CASES(true, false) DUAL_CASES(true, true)
#undef DUAL_CASES
#undef DUAL_CASE
  return cudaErrorInvalidValue;
}

template <int FMT>
cudaError_t dispatch(const fp4lib::QuantArgs& a, uint32_t mask, cudaStream_t st) {
  const int64_t chunks = a.M * (a.K / 16);
  if (chunks == 0) return cudaSuccess;
#define RHT_CASE(SR, MMA, AM)                                                                                  \
  if (a.row_sr == SR && a.mma == MMA && a.amax_by_product == AM) {                                            \
    k_quant_rows_rht<FMT, SR, MMA, AM><<<grid_for(chunks), 256, 0, st>>>(                                    \
        static_cast<const uint16_t*>(a.x), a.M, a.K, a.ldx, mask, a.gptr, a.seed_row, a.codes_row,            \
        a.scales_row, a.amax_out, a.status);                                                                   \
    return cudaGetLastError();                                                                                 \
  }
  RHT_CASE(false, false, false) RHT_CASE(false, false, true) RHT_CASE(false, true, false)
  RHT_CASE(false, true, true) RHT_CASE(true, false, false) RHT_CASE(true, false, true)
  RHT_CASE(true, true, false) RHT_CASE(true, true, true)
#undef RHT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

namespace fp4lib {

cudaError_t launch_amax_rht(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t mask, float* out,
                            cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t chunks = M * (K / 16);
  if (chunks == 0) return cudaSuccess;
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  k_amax_rht<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(x), M, K, ldx, mask, out);
  return cudaGetLastError();
}

cudaError_t launch_amax_rht_cols(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t mask, float* out,
                                 cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t units = (M / 16) * K;
  if (units == 0) return cudaSuccess;
  int64_t blocks = (units + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  k_amax_rht_cols<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(x), M, K, ldx, mask, out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_dual_rht(const DualRhtArgs& a, cudaStream_t st) {
  switch (a.fmt) {
    case FP4_SF_E4M3: return dispatch_dual<SF_E4M3>(a, st);
    case FP4_SF_UE5M3: return dispatch_dual<SF_UE5M3>(a, st);
    case FP4_SF_E8M0: return dispatch_dual<SF_E8M0>(a, st);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_quantize_rht(const QuantArgs& a, uint32_t mask, cudaStream_t st) {
  switch (a.fmt) {
    case FP4_SF_E4M3: return dispatch<SF_E4M3>(a, mask, st);
    case FP4_SF_UE5M3: return dispatch<SF_UE5M3>(a, mask, st);
    case FP4_SF_E8M0: return dispatch<SF_E8M0>(a, mask, st);
    case FP4_SF_NVINT4: return dispatch<SF_NVINT4>(a, mask, st);
    case FP4_SF_MXINT4: return dispatch<SF_MXINT4>(a, mask, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fp4lib
