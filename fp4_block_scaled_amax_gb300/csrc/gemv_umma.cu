// Weight-only NVFP4 linear for batches of 9 to 64 on the sm_103a tcgen05
// tensor cores (weight-only NVFP4 post, quant_prune_distill #574: weights in
// NVFP4, activations untouched, section "Метод").
//
//   y[b, n] = (1 / s_enc) * sum_k (e2m1[n, k] * s_b[n, k/16]) * x[b, k]
//
// At batch 64 the weight stream is a contraction of about 200 FLOP per byte,
// so the expansion of the codes, not the MMA, decides the speed.  The expanded
// weights never touch shared memory: they go from registers to tensor memory
// and the MMA reads its A operand there.  A CTA owns 128 weight rows and a run
// of K:
//   warp 0     TMA: per 256-column stage the codes (128 rows x 128 bytes,
//              128-byte swizzle), the scales (128 rows x 16 bytes) and the
//              activations (four 64-column boxes of 64 rows, 128-byte
//              swizzle; rows past the batch read as zero) into a 4-stage ring;
//   warp 1     allocates 512 tensor-memory columns (a 64-column float32
//              accumulator and three 128-column A slots); per stage, after one
//              wait, an elected lane issues sixteen tcgen05.mma.kind::f16 with
//              A in tensor memory (M = 128 weight rows, N = 64 batch rows,
//              K = 16, bf16 operands) back to back and commits the A slot and
//              the stage back to their producers.  The warp runs the loop in
//              step with warp-uniform values and keeps the bursts long: a wait
//              between short bursts of MMAs costs far more than the MMAs;
//   warps 2-9  expand the codes of each stage into bf16 weights,
//              e2m1 * s_b * 2^-8 exactly, one weight row per thread (the row
//              is the tensor-memory lane its warp may write), and store them
//              with tcgen05.st; then four of them drain the accumulator.
// Tall K splits over a cluster of CTAs that reduce their float32 partial
// products through distributed shared memory (rank 0 adds them in rank
// order and writes y).  Every wait is bounded.
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

using namespace fp4async;

// Prefetch of a tensor-map tile into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

constexpr int UM_ROWS = 128;     // weight rows per CTA (the MMA's M)
constexpr int UM_BATCH = 64;     // batch rows of the MMA (its N); smaller batches read zeros
constexpr int UM_KSTAGE = 256;   // columns per TMA stage
constexpr int UM_STAGES = 4;
constexpr int UM_ASLOTS = 3;     // tensor-memory A slots of one stage (256 columns of K) each
constexpr int UM_DECODERS = 8;   // warps
constexpr int UM_THREADS = 32 * (2 + UM_DECODERS);
constexpr int UM_CODE_BYTES = UM_ROWS * UM_KSTAGE / 2;      // 16 KB
constexpr int UM_SCALE_BYTES = UM_ROWS * UM_KSTAGE / 16;    // 2 KB
constexpr int UM_XBOX_BYTES = UM_BATCH * 64 * 2;            // 8 KB: 64 rows x 64 columns
constexpr int UM_X_BYTES = 4 * UM_XBOX_BYTES;               // 32 KB
constexpr int UM_STAGE_BYTES = UM_CODE_BYTES + UM_X_BYTES + UM_SCALE_BYTES;  // 50 KB
constexpr int UM_SMEM_RING = 0;
constexpr int UM_SMEM_BAR = UM_SMEM_RING + UM_STAGES * UM_STAGE_BYTES;
constexpr int UM_NBARS = 2 * UM_STAGES + 2 * UM_ASLOTS + 1;
constexpr int UM_SMEM_TOTAL = UM_SMEM_BAR + 8 * UM_NBARS + 16;
constexpr int UM_SMEM_LAUNCH = UM_SMEM_TOTAL + 1024;
// tensor memory: the float32 accumulator in columns 0..63, then the A slots
// of 128 columns (128 lanes = weight rows; a column holds two bf16 of K, the
// even one low)
constexpr uint32_t UM_TMEM_COLS = 512;
constexpr uint32_t UM_ACOL0 = 64, UM_ASLOT_COLS = 128;
static_assert(UM_ACOL0 + UM_ASLOTS * UM_ASLOT_COLS <= UM_TMEM_COLS, "tensor-memory slots");
static_assert(UM_STAGE_BYTES % 1024 == 0, "swizzled buffers need 1024-byte alignment");
static_assert(UM_SMEM_LAUNCH <= 232448, "shared memory over the sm_103a per-CTA limit");
// the float32 partial products [128 rows][64 batch] of a split-K rank reuse the ring
static_assert(UM_ROWS * UM_BATCH * 4 <= UM_STAGES * UM_STAGE_BYTES, "reduction buffer");

// Shared-memory matrix descriptor (start address, leading/stride byte offsets
// in 16-byte units, version 1 at bit 46, layout 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t um_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // 8 rows x 128 bytes between core groups
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor of kind::f16: float32 accumulator (bits 4-5 = 1),
// bf16 A and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t UM_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(UM_BATCH >> 3) << 17) |
                              ((uint32_t)(UM_ROWS >> 4) << 24);

// D (tensor memory) += A (tensor memory) * B (shared-memory descriptor),
// issued by one lane that the converged warp elects
__device__ __forceinline__ void um_mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xFFFFFFFF;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(UM_IDESC), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void um_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xFFFFFFFF;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void um_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void um_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ uint32_t um_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t um_mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Eight E2M1 codes (one word, element 0 in the low nibble) -> four bf16x2
// words in natural order, (0, 1), (2, 3), (4, 5), (6, 7), each value
// e2m1 * 2^-126 exactly.  The low and high nibbles are split into two byte
// planes; a byte permute then places byte j of each plane 16 bits apart with
// zero bytes between them (the sign-replicate mode of a byte whose top bit is
// clear), and the multiply by 2^6 + 2^12 puts each nibble's magnitude bits at
// bf16 bits 8..6 and its sign at bit 15.
__device__ __forceinline__ void um_e2m1x8(uint32_t v, uint32_t (&r)[4]) {
  constexpr uint32_t M = 0x81C081C0u;
  const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // bytes: lo[j], 0, hi[j], 0
    const uint32_t t = um_prmt(lo, hi, 0x8480u + 0x1111u * (uint32_t)j);
    r[j] = (t * 4160u) & M;
  }
}
// E4M3 scale code -> bf16 of value * 2^118 in both halves (exact): the code
// shifted to bf16 bits 11..4 is value * 2^-120; two exact multiplies by 2^119.
__device__ __forceinline__ uint32_t um_scale_bf16x2(uint32_t c) {
  constexpr uint32_t TWO119 = 0x7B007B00u;
  const uint32_t h = (c & 0xFFu) << 4;
  return um_mul_bf16x2(um_mul_bf16x2(h | (h << 16), TWO119), TWO119);
}

// 32 columns of the warp's tensor-memory lane quarter into registers (waits for them)
__device__ __forceinline__ void um_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct UmParams {
  const float* gw;
  int batch, N, nk_total;  // nk_total: 256-column stages along K
  int ksplit;
  bool bf16_out;
  void* y;
  int32_t* status;
};

__global__ void __launch_bounds__(UM_THREADS, 1)
    k_gemv_w4a16_umma(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                      const __grid_constant__ CUtensorMap tm_x, UmParams p) {
  // a GEMV launched after this one may start its CTAs as these exit (they
  // wait for this grid before they read its activations)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + UM_SMEM_BAR;         // [S] TMA stage landed
  const uint32_t bar_empty = bar_full + 8 * UM_STAGES;   // [S] MMAs of the stage done
  const uint32_t bar_done = bar_empty + 8 * UM_STAGES;   // [A] slot decoded
  const uint32_t bar_free = bar_done + 8 * UM_ASLOTS;    // [A] MMAs of the slot done
  const uint32_t bar_acc = bar_free + 8 * UM_ASLOTS;     // accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + UM_SMEM_BAR + 8 * UM_NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + UM_SMEM_BAR + 8 * UM_NBARS + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t rank = 0;
  if (p.ksplit > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int n0 = (blockIdx.x / p.ksplit) * UM_ROWS;
  const int it0 = (int)(((int64_t)p.nk_total * rank) / p.ksplit);
  const int nk = (int)(((int64_t)p.nk_total * (rank + 1)) / p.ksplit) - it0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < UM_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < UM_ASLOTS; ++a) {
      mbar_init(bar_done + 8 * a, UM_DECODERS);
      mbar_init(bar_free + 8 * a, 1);
    }
    mbar_init(bar_acc, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(UM_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  um_fence_before();
  __syncthreads();
  um_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything the warps other than the producer read or write follows the
  // preceding kernel (the producer waits after prefetching weights)
  if (warp != 0) asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ------------------------------ TMA producer --------------------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_codes)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_scales)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
      // the weights of the first two stages stream into L2 while a preceding
      // kernel may still run (programmatic dependent launch); every stage then
      // loads as usual once it has completed
      for (int it = 0; it < nk && it < 2; ++it) {
        tma_prefetch_l2_2d(&tm_codes, (it0 + it) * (UM_KSTAGE / 2), n0);
        tma_prefetch_l2_2d(&tm_scales, (it0 + it) * (UM_KSTAGE / 16), n0);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int it = 0; it < nk; ++it) {
        const int s = it % UM_STAGES;
        if (it >= UM_STAGES &&
            !wait_bounded(bar_empty + 8 * s, ((it / UM_STAGES) - 1) & 1, abort_flag, p.status))
          break;
        if (*abort_flag) break;
        const int gs = it0 + it;
        const uint32_t fb = bar_full + 8 * s, st = sbase + UM_SMEM_RING + s * UM_STAGE_BYTES;
        mbar_expect_tx(fb, UM_STAGE_BYTES);
        tma_load_2d(st, &tm_codes, fb, gs * (UM_KSTAGE / 2), n0);
#pragma unroll
        for (int i = 0; i < 4; ++i) tma_load_2d(st + UM_CODE_BYTES + i * UM_XBOX_BYTES, &tm_x, fb, gs * UM_KSTAGE + 64 * i, 0);
        tma_load_2d(st + UM_CODE_BYTES + UM_X_BYTES, &tm_scales, fb, gs * (UM_KSTAGE / 16), n0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    // The decoders arrive on a slot only after they saw the stage's TMA
    // barrier complete, so their arrival also orders the activations that the
    // MMA reads: one wait per stage.
    bool ok = true;
    for (int it = 0; it < nk; ++it) {
      const int s = it % UM_STAGES, a = it % UM_ASLOTS;
      if (!wait_lane0(bar_done + 8 * a, (it / UM_ASLOTS) & 1, abort_flag, p.status, lane)) {
        ok = false;
        break;
      }
      um_fence_after();
      const uint32_t xs = sbase + UM_SMEM_RING + s * UM_STAGE_BYTES + UM_CODE_BYTES;
      const uint32_t acol = tmem + UM_ACOL0 + a * UM_ASLOT_COLS;
#pragma unroll
      for (int j = 0; j < 16; ++j) {  // K = 16 per MMA: 8 A columns; 32 bytes of a 64-column x box row
        const uint64_t bd = um_desc(xs + (j >> 2) * UM_XBOX_BYTES + 32 * (j & 3));
        um_mma_ts_elect(tmem, acol + 8 * j, bd, (it > 0 || j > 0) ? 1u : 0u);
      }
      um_commit_elect(bar_free + 8 * a);   // the A slot may be decoded into again
      um_commit_elect(bar_empty + 8 * s);  // the stage's activations are read
    }
    if (ok) um_commit_elect(bar_acc);
    __syncwarp();
  } else {
    // ------------------------------ decoders, then the epilogue -----------
    // thread: weight row r (the tensor-memory lane quarter of its warp), K
    // columns 128 h + 64 hh .. + 63 of each stage, h = 0, 1
    const int hh = (warp - 2) >> 2, r = 32 * (warp & 3) + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + UM_ACOL0 + 32 * hh;
    for (int it = 0; it < nk; ++it) {
      const int s = it % UM_STAGES, a = it % UM_ASLOTS;
      if (!wait_lane0(bar_full + 8 * s, (it / UM_STAGES) & 1, abort_flag, p.status, lane)) break;
      if (it >= UM_ASLOTS &&
          !wait_lane0(bar_free + 8 * a, ((it / UM_ASLOTS) - 1) & 1, abort_flag, p.status, lane))
        break;
      um_fence_after();
      const uint8_t* st = smem + UM_SMEM_RING + s * UM_STAGE_BYTES;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        // 16-byte code chunks 4 h + 2 hh and + 1 of the row's 128 bytes (128-byte swizzle)
        const uint8_t* crow = st + r * 128;
        const int c0 = 4 * h + 2 * hh;
        const uint4 w0 = *reinterpret_cast<const uint4*>(crow + ((c0 ^ (r & 7)) << 4));
        const uint4 w1 = *reinterpret_cast<const uint4*>(crow + (((c0 + 1) ^ (r & 7)) << 4));
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(st + UM_CODE_BYTES + UM_X_BYTES + r * 16 + 8 * h + 4 * hh);
        const uint32_t cw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t o[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {  // 16 columns per block scale
          const uint32_t s2 = um_scale_bf16x2(sc >> (8 * g));
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t rr[4];
            um_e2m1x8(cw[2 * g + u], rr);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[8 * g + 4 * u + i] = um_mul_bf16x2(rr[i], s2);
          }
        }
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
            "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(lane_base + a * UM_ASLOT_COLS + 64 * h),
            "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7]), "r"(o[8]),
            "r"(o[9]), "r"(o[10]), "r"(o[11]), "r"(o[12]), "r"(o[13]), "r"(o[14]), "r"(o[15]), "r"(o[16]),
            "r"(o[17]), "r"(o[18]), "r"(o[19]), "r"(o[20]), "r"(o[21]), "r"(o[22]), "r"(o[23]), "r"(o[24]),
            "r"(o[25]), "r"(o[26]), "r"(o[27]), "r"(o[28]), "r"(o[29]), "r"(o[30]), "r"(o[31])
            : "memory");
      }
      // the stores are complete before the MMA issuer learns of them
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      um_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_done + 8 * a);
    }
  }
  // ---- epilogue: warps 2..5 hold tensor-memory lane quarters 2, 3, 0, 1 ----
  const bool epi = warp >= 2 && warp < 6;
  const int row = 32 * (warp & 3) + lane;  // weight row within the CTA (epilogue warps)
  float v[UM_BATCH];
  if (epi) {
    const bool have = wait_bounded(bar_acc, 0, abort_flag, p.status);
    if (have) {
      um_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t rg[32];
        um_ld32(taddr + 32 * hb, rg);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * hb + i] = __uint_as_float(rg[i]);
      }
    } else {
#pragma unroll
      for (int b = 0; b < UM_BATCH; ++b) v[b] = 0.0f;
    }
    um_fence_before();
    if (p.ksplit > 1) {
      // this rank's partial products in its shared memory (the ring is idle once the
      // accumulator is complete), [batch][row]: consecutive lanes, consecutive words
      float* part = reinterpret_cast<float*>(smem + UM_SMEM_RING);
#pragma unroll
      for (int b = 0; b < UM_BATCH; ++b) part[b * UM_ROWS + row] = v[b];
    }
  }
  if (p.ksplit > 1) {
    // every thread of every rank: the partial products are in place before rank 0 reads them
    __syncthreads();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  if (epi && rank == 0) {
    const float* part = reinterpret_cast<const float*>(smem + UM_SMEM_RING);
    for (int q = 1; q < p.ksplit; ++q) {
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(part)), "r"(q));
#pragma unroll
      for (int b = 0; b < UM_BATCH; ++b) {
        float pv;
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pv) : "r"(remote + 4u * (b * UM_ROWS + row)));
        v[b] = __fadd_rn(v[b], pv);
      }
    }
    const float s_enc = fp4dev::global_encode_scale<fp4dev::SF_E4M3>(__ldg(p.gw), nullptr);
    const int n = n0 + row;
    if (n < p.N) {
#pragma unroll
      for (int b = 0; b < UM_BATCH; ++b) {
        if (b < p.batch) {
          const float o = __fdiv_rn(__fmul_rn(v[b], 256.0f), s_enc);
          if (p.bf16_out) static_cast<__nv_bfloat16*>(p.y)[(int64_t)b * p.N + n] = __float2bfloat16_rn(o);
          else static_cast<float*>(p.y)[(int64_t)b * p.N + n] = o;
        }
      }
    }
  }
  if (p.ksplit > 1) {
    // no rank leaves while rank 0 may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  // ------------------------------ teardown --------------------------------
  um_fence_before();
  __syncthreads();
  drain_after_abort(abort_flag);
  if (warp == 1) {
    um_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(UM_TMEM_COLS) : "memory");
  }
}

bool um_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace fp4lib {

// Batches of 9..64 with K a multiple of 256; cudaErrorNotSupported (nothing
// launched) otherwise, or when the tensor-map encoder refuses the shapes.
cudaError_t launch_gemv_umma(const GemvArgs& a, cudaStream_t st) {
  if (a.batch <= 8 || a.batch > UM_BATCH || a.K % UM_KSTAGE != 0 || a.N > (int64_t)1 << 30 ||
      a.K > (int64_t)1 << 30)
    return cudaErrorNotSupported;
  CUtensorMap mc, ms, mx;
  if (!um_map(&mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wq, a.K / 2, a.N, a.K / 2, 128, UM_ROWS, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !um_map(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Ws, a.K / 16, a.N, a.K / 16, 16, UM_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !um_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.K, a.batch, a.K * 2, 64, UM_BATCH, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorNotSupported;
  static DeviceInts attr_set;
  cudaError_t e = cudaSuccess;
  attr_set.get([&] {
    e = cudaFuncSetAttribute(k_gemv_w4a16_umma, cudaFuncAttributeMaxDynamicSharedMemorySize, UM_SMEM_LAUNCH);
    return e == cudaSuccess ? 1 : 0;
  });
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.N + UM_ROWS - 1) / UM_ROWS;
  const int nk_total = (int)(a.K / UM_KSTAGE);
  const int sms = current_sm_count();
  // K split: the most ways (up to 8, at least 4 stages each) that keep one wave
  int ksplit = 1;
  for (int s = 2; s <= 8; ++s)
    if (tiles * s <= sms && nk_total >= 4 * s) ksplit = s;
  UmParams p{};
  p.gw = a.gw;
  p.batch = (int)a.batch;
  p.N = (int)a.N;
  p.nk_total = nk_total;
  p.ksplit = ksplit;
  p.bf16_out = a.bf16_out;
  p.y = a.y;
  p.status = a.status;
  cudaLaunchConfig_t cfg = {};
  // programmatic dependent launch, as for the TMA-fed form
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)ksplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(tiles * ksplit), 1, 1);
  cfg.blockDim = dim3(UM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = UM_SMEM_LAUNCH;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = ksplit > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_w4a16_umma, mc, ms, mx, p);
}

}  // namespace fp4lib
