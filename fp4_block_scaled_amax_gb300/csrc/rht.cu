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
//   k_amax_rht        fresh global amax of the transformed tensor.
//   k_quant_rows_rht  one thread per 16 elements: two 128-bit loads, the
//                     transform in registers, quantization, one 8-byte store.
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

unsigned grid_for(int64_t n) { return (unsigned)((n + 255) / 256); }

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
