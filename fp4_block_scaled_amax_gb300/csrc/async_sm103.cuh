// Asynchronous-copy plumbing shared by the sm_103a kernels: mbarriers with
// bounded waits, 2-D TMA tile loads, and the host-side tensor-map encoder.
//
// Every wait is bounded: after WAIT_LIMIT_CYCLES the waiting thread raises
// its CTA's abort flag and records FP4_ERR_TIMEOUT in the status word, so a
// lost copy ends the kernel with an error instead of a hang.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fp4_device.cuh"

namespace fp4async {

constexpr long long WAIT_LIMIT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz
// After an abort, copies issued before it may still be landing in shared
// memory (or completing on a barrier); the CTA waits this long (~10 ms, far
// beyond a copy's latency) before it exits (and, where it holds tensor
// memory, before it frees it).
constexpr long long DRAIN_CYCLES = 20000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait.  Returns false (and raises the CTA's abort flag and the status
// word) if the phase does not complete within the limit or another role has
// already aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
      *abort_flag = 1;
      fp4dev::set_status(status, FP4_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void drain_after_abort(volatile int* abort_flag) {
  if (threadIdx.x == 0 && *abort_flag) {
    const long long t0 = clock64();
    while (clock64() - t0 < DRAIN_CYCLES) {
    }
  }
  __syncthreads();
}

// Bounded wait by lane 0 of a converged warp; the outcome is broadcast so the
// warp stays converged.
__device__ __forceinline__ bool wait_lane0(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                                           int lane) {
  int ok = 0;
  if (lane == 0) ok = wait_bounded(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// ---- TMA / bulk copies ----------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// The driver's tensor-map encoder (one entry point for every device; the
// function-local static is initialised once, thread-safely).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace fp4async
