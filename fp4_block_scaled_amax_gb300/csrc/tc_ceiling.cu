// Tensor-core ceiling of this GPU, per SM and per clock: a standalone
// measurement program (not part of libfp4.so).
//
// Each CTA (one per SM) streams R tcgen05.mma instructions of one form back
// to back from a single warp (one elected lane issues, warp-uniform operands,
// no waits between them), commits once and waits (bounded) for the commit;
// SM cycles from clock64 over that span give FLOP per clock per SM.  Forms:
//   bf16   kind::f16, bf16 x bf16 -> f32, M = 128, N = 256, K = 16 (cta_group::1)
//   nvf4   kind::mxf4nvf4 scale_vec::4X (E2M1, ue4m3 scales per 16), the CTA
//          pair (cta_group::2), M = 256, N = 256, K = 64: the FP4 GEMM's MMA
//   mxf4   kind::mxf4nvf4 scale_vec::2X (E2M1, ue8m0 scales per 32),
//          cta_group::1, M = 128, N = 256, K = 64
// Operands are constant (bf16 1.0, E2M1 1.0, scale 1.0); the MMA's speed
// does not depend on them.  Prints one JSON line.
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "async_sm103.cuh"

namespace {

using namespace fp4async;

constexpr int R_MMAS = 2048;
constexpr int SMEM_BYTES = 120 * 1024;  // keeps one CTA per SM
constexpr long long WAIT_CYCLES = 2000000000LL;

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // 8 rows x 128 bytes between core groups
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fill_tmem(uint32_t tmem, int warp, uint32_t col, uint32_t v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
      "%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(tmem + ((uint32_t)(32 * warp) << 16) + col),
      "r"(v)
      : "memory");
}

// FORM 0: bf16 (cta_group::1); 1: nvf4 pair (cta_group::2); 2: mxf4 (cta_group::1)
template <int FORM>
__global__ void __launch_bounds__(128, 1) k_ceiling(long long* cycles, int* ok_out) {
  constexpr bool PAIR = FORM == 1;
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t rank = 0;
  if (PAIR) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const uint32_t fill = FORM == 0 ? 0x3F803F80u : 0x22222222u;  // bf16 1.0 pairs / E2M1 1.0 nibbles
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = fill;
  const uint32_t sa = smem_u32(sm), sb = sa + 16384, bar = sa + 65536;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 65536 + 64);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    if (PAIR) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(512)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(512)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (PAIR) cl_sync();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *slot;
  // scale factors in columns 256..319 (ue4m3 1.0 = 0x38, ue8m0 1.0 = 0x7F)
  const uint32_t sfv = FORM == 2 ? 0x7F7F7F7Fu : 0x38383838u;
  fill_tmem(tmem, warp, 256, sfv);
  fill_tmem(tmem, warp, 288, sfv);
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (PAIR) cl_sync();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  if (warp == 0 && rank == 0) {
    const long long t0 = clock64();
    for (int i = 0; i < R_MMAS; i += 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t acc = (i > 0 || j > 0) ? 1u : 0u;
        const uint64_t ad = sw128_desc(sa + 32 * j), bd = sw128_desc(sb + 32 * j);
        if constexpr (FORM == 0) {
          constexpr uint32_t ID = (1u << 4) | (1u << 7) | (1u << 10) | (256u >> 3 << 17) | (128u >> 4 << 24);
          asm volatile(
              "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
              "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(ID), "r"(acc)
              : "memory");
        } else if constexpr (FORM == 1) {
          constexpr uint32_t ID = (1u << 7) | (1u << 10) | (256u >> 3 << 17) | (256u >> 4 << 24);
          asm volatile(
              "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
              "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
              "p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(ID), "r"(tmem + 256 + 4 * j), "r"(tmem + 272 + 8 * j), "r"(acc)
              : "memory");
        } else {
          constexpr uint32_t ID = (1u << 7) | (1u << 10) | (256u >> 3 << 17) | (1u << 23) | (128u >> 4 << 24);
          asm volatile(
              "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
              "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], "
              "p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(ID), "r"(tmem + 256 + 4 * (j >> 1)), "r"(tmem + 272 + 8 * (j >> 1)), "r"(acc)
              : "memory");
        }
      }
    }
    if (PAIR) {
      asm volatile(
          "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
          "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
              bar),
          "h"((uint16_t)3)
          : "memory");
    } else {
      asm volatile(
          "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
          "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
          : "memory");
    }
    int got = 0;
    if (lane == 0) {
      for (long long t = clock64(); clock64() - t < WAIT_CYCLES;)
        if (mbar_try_wait(bar, 0)) {
          got = 1;
          break;
        }
    }
    const long long t1 = clock64();
    if (lane == 0) {
      const int unit = PAIR ? blockIdx.x / 2 : blockIdx.x;
      cycles[unit] = t1 - t0;
      ok_out[unit] = got;
    }
  } else if (PAIR && warp == 0 && rank == 1) {
    // the peer keeps its tensor memory until the pair's commit has landed
    if (lane == 0) {
      for (long long t = clock64(); clock64() - t < WAIT_CYCLES;)
        if (mbar_try_wait(bar, 0)) break;
    }
    __syncwarp();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (PAIR) cl_sync();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// Median FLOP per clock per SM over the CTAs (pairs) of the last of three launches; < 0 on error.
template <int FORM>
double measure(int sms, double flop_per_mma_per_sm) {
  const bool pair = FORM == 1;
  const int ctas = pair ? sms / 2 * 2 : sms;
  const int units = pair ? ctas / 2 : ctas;
  long long* d_cyc = nullptr;
  int* d_ok = nullptr;
  if (cudaMalloc(&d_cyc, sizeof(long long) * units) != cudaSuccess ||
      cudaMalloc(&d_ok, sizeof(int) * units) != cudaSuccess)
    return -1.0;
  double result = -1.0;
  if (cudaFuncSetAttribute(k_ceiling<FORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess) {
    bool launched = true;
    for (int rep = 0; rep < 3 && launched; ++rep) {
      if (pair) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(ctas, 1, 1);
        cfg.blockDim = dim3(128, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        launched = cudaLaunchKernelEx(&cfg, k_ceiling<FORM>, d_cyc, d_ok) == cudaSuccess;
      } else {
        k_ceiling<FORM><<<ctas, 128, SMEM_BYTES>>>(d_cyc, d_ok);
        launched = cudaGetLastError() == cudaSuccess;
      }
      launched = launched && cudaDeviceSynchronize() == cudaSuccess;
    }
    if (launched) {
      long long* cyc = new long long[units];
      int* ok = new int[units];
      cudaMemcpy(cyc, d_cyc, sizeof(long long) * units, cudaMemcpyDeviceToHost);
      cudaMemcpy(ok, d_ok, sizeof(int) * units, cudaMemcpyDeviceToHost);
      bool all_ok = true;
      for (int i = 0; i < units; ++i) all_ok = all_ok && ok[i] == 1;
      if (all_ok) {
        // median by partial selection sort (a few hundred entries)
        for (int i = 0; i <= units / 2; ++i)
          for (int j = i + 1; j < units; ++j)
            if (cyc[j] < cyc[i]) {
              const long long t = cyc[i];
              cyc[i] = cyc[j];
              cyc[j] = t;
            }
        result = flop_per_mma_per_sm * R_MMAS / (double)cyc[units / 2];
      }
      delete[] cyc;
      delete[] ok;
    }
  }
  cudaFree(d_cyc);
  cudaFree(d_ok);
  return result;
}

}  // namespace

int main() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const double bf16 = measure<0>(sms, 2.0 * 128 * 256 * 16);
  const double nvf4 = measure<1>(sms, 2.0 * 128 * 256 * 64);  // each SM computes its 128 rows of the pair's M = 256
  const double mxf4 = measure<2>(sms, 2.0 * 128 * 256 * 64);
  const bool ok = bf16 > 0 && nvf4 > 0 && mxf4 > 0;
  printf("{\"sms\": %d, \"mmas_per_cta\": %d, \"bf16_flop_per_clk_sm\": %.1f, \"nvf4_pair_flop_per_clk_sm\": %.1f, "
         "\"mxf4_flop_per_clk_sm\": %.1f, \"ok\": %s}\n",
         sms, R_MMAS, bf16, nvf4, mxf4, ok ? "true" : "false");
  return ok ? 0 : 1;
}
