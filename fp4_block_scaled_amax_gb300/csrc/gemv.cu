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
// k permutation: inside a 128-wide k chunk, lane q of a quad (q = lane % 4)
// supplies at MMA step s the fragment positions {2q, 2q+1, 2q+8, 2q+9} from
// the actual columns 32q + 4s + {0, 1, 2, 3}.  A and B use the same map, so the
// sum over positions is the sum over k, while each lane reads 16 contiguous
// code bytes and 64 contiguous activation bytes per chunk.
//
// CTA = 16 weight rows x WARPS warps splitting K; partial sums meet in shared
// memory.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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

}  // namespace

namespace fp4lib {

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st) {
  // 16 weight rows per CTA; enough warps per CTA (split K) to put about 16
  // warps on each of the GPU's SMs in a single wave
  const int64_t ctas = (a.N + 15) / 16;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
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
