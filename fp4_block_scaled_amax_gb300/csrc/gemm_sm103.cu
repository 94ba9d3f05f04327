// Block-scaled FP4 GEMM on the sm_103a tcgen05 tensor cores.
//
// Computes, for packed E2M1 operands A [M, K], B [N, K] (blocks along K) and
// their block scales ("NVFP4 vs MXFP" post, quant_prune_distill #486, section
// "Метод"; every eligible linear in FP4 for forward and backward: "UE5M3 FP4
// Block Scaling ..." blog, section "Что сделали"):
//
//   C[m, n] = alpha * sum_k (qa * sa)(qb * sb),   float32 accumulation,
//   alpha   = f32(1 / f32(s_encA * s_encB)) * 2^(tA + tB).
//
// NVFP4 (E4M3 scales, 16-element blocks) runs as kind::mxf4nvf4 with
// scale_vec::4X and ue4m3 scales; MXFP4 (E8M0, 32-element blocks) as
// scale_vec::2X with ue8m0 scales.  UE5M3 has no tensor-core scale type; its
// scales arrive re-encoded as E4M3 of s * 2^-t (exact) and 2^(tA + tB) folds
// into alpha (the software emulation of the "UE5M3 ..." blog, "Ограничения").
//
// Two forms share the roles below.  When M is a multiple of 256, clusters of
// two CTAs run cta_group::2 MMAs on 256 x 256 output tiles (k_gemm_fp4_pair):
// each SM holds half of the B tile, so it streams A + B/2 per K step.
// Otherwise one CTA per SM runs 128 x 256 tiles (k_gemm_fp4).  N is a
// multiple of 128: a half last tile reads zero-filled code rows (the TMA's
// out-of-range fill) and stores nothing past N.
//
// Kernel structure (one CTA per SM, persistent over 128 x 256 output tiles,
// 23 warps):
//   warp 0       code producer: A/B code tiles (128-byte swizzle) by
//                cp.async.bulk.tensor into a 3- or 4-stage shared-memory ring;
//   warp 1       allocates tensor memory; one lane issues the 4 tcgen05.mma of
//                each 256-wide K step once its scales sit in tensor memory and
//                its codes in shared memory; tcgen05.commit frees the stage
//                (and, after the last K step, hands the accumulator over);
//   warp 2       scale producer: the K step's scale atoms by cp.async.bulk into
//                a separate 4-slot ring that runs ahead of the code ring (a slot
//                frees as soon as the scale writers have read it);
//   warps 3-6    scale writers, one per 32-lane quarter of tensor memory: each
//                lane reads its row of every 512-byte scale atom from shared
//                memory and, once the MMAs of K step k - STAGES have released
//                the stage's tensor-memory columns, writes it with tcgen05.st
//                into the replicated layout the MMA reads (row r's scales in
//                column r/32 of lane r%32 of every quarter), off the MMA's
//                critical path;
//   warps 7-22   epilogue: each warp drains 32 rows x 64 columns of the
//                float32 accumulator with tcgen05.ld, releases the tensor
//                memory at once (the next tile's MMAs overlap the rest), scales,
//                converts and stages 32-row blocks of 16-byte rows (long K: 512
//                bytes per warp, which leaves room for a 4-stage ring) or
//                64-byte rows (2 KB) in shared memory, and writes them with TMA
//                bulk-tensor stores.  With a quantized output
//                (fp4_gemm_quantize[_dual], CTA pairs) the warp instead
//                quantizes bf16(acc * alpha): row blocks from its registers,
//                column blocks (the layout of C^T) after passing the values
//                through its 2 KB staging buffer.
// Every mbarrier wait is bounded: on expiry the CTA records FP4_ERR_TIMEOUT in
// the status word and winds down instead of spinning.  Once aborted, the
// producers issue no further copies, and the CTA waits a fixed ~10 ms for
// copies already in flight before it frees its tensor memory and exits.
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

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;  // FP4 elements per K step = 128 bytes per row
constexpr int A_BYTES = BM * BK / 2;   // 16 KB
constexpr int B_BYTES = BN * BK / 2;   // 32 KB
constexpr int SFA_MAX = BM * BK / 16;  // 2 KB (NVFP4); MXFP4 uses half
constexpr int SFB_MAX = BN * BK / 16;  // 4 KB

constexpr int NUM_SF_WARPS = 4;
constexpr int NUM_EPI_WARPS = 16;
constexpr int SF_PRODUCER_WARP = 2;
constexpr int FIRST_SF_WARP = 3;
constexpr int SF_SLOTS = 4;  // scale ring depth
constexpr int FIRST_EPI_WARP = FIRST_SF_WARP + NUM_SF_WARPS;
constexpr int NUM_THREADS = 32 * (FIRST_EPI_WARP + NUM_EPI_WARPS);
constexpr int EPI_COLS = BN / (NUM_EPI_WARPS / 4);  // 64 accumulator columns per epilogue warp

// Shared-memory plan of one configuration: S stages of the code/scale ring
// and, per epilogue warp, one 32-row output block with OB-byte rows (OB = 64:
// 64-byte-swizzled blocks; OB = 16: plain 512-byte blocks).  Short K (an
// output-heavy GEMM) wants wide blocks; long K wants the deeper ring.
template <int S, int OB, int BB = B_BYTES>
struct Plan {
  static constexpr int STAGES = S;
  static constexpr int OUT_ROW_BYTES = OB;
  static constexpr int STAGE_BYTES = 32 * OB;
  static constexpr int B_STAGE = BB;  // B code bytes per stage (half the tile for a CTA pair)
  static constexpr int SMEM_A = 0;
  static constexpr int SMEM_B = SMEM_A + S * A_BYTES;
  static constexpr int SMEM_SFA = SMEM_B + S * BB;
  static constexpr int SMEM_SFB = SMEM_SFA + SF_SLOTS * SFA_MAX;
  static constexpr int SMEM_OUT = SMEM_SFB + SF_SLOTS * SFB_MAX;
  static constexpr int SMEM_BAR = SMEM_OUT + NUM_EPI_WARPS * STAGE_BYTES;
  static constexpr int SMEM_TOTAL = SMEM_BAR + 256;
  static constexpr int SMEM_LAUNCH = SMEM_TOTAL + 1024;  // room to align the base to 1024
  // tensor memory columns: accumulator 0..255, then per stage 16 columns of
  // A scales (4 K64 steps x 4) and 32 of B scales (4 K64 steps x 2 halves x 4)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TMEM_SFA = 256;
  static constexpr uint32_t TMEM_SFB = TMEM_SFA + 16 * S;
  static_assert(SMEM_OUT % 1024 == 0, "output staging must stay 1024-byte aligned");
  static_assert(SMEM_LAUNCH <= 232448, "shared memory over the sm_103a per-CTA limit");
  static_assert(TMEM_SFB + 32 * S <= TMEM_COLS, "tensor memory budget");
};
using PlanShortK = Plan<3, 64>;
using PlanLongK = Plan<4, 16>;
// CTA pair: each CTA holds half of B, so five stages fit beside wide output blocks
using PlanPair = Plan<5, 64, B_BYTES / 2>;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
// The same store, added element-wise to what the destination holds (float32
// add for a float32 map): the later passes of a multi-pass GEMM.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ---- tcgen05 --------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// Shared-memory matrix descriptor: start address, leading/stride byte offsets
// (16-byte units), fixed version field 1 at bit 46, layout type at bits 61-63
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1) at bits
// 7-9 and 10-12, K-major both, N>>3 at bits 17-22, scale type at bit 23
// (0 = ue4m3, 1 = ue8m0), M>>4 at bits 24-28, scale-factor ids 0.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool ue8m0) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
         ((uint32_t)(m >> 4) << 24);
}

template <bool MX>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (MX) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  }
}

// ---- CTA pair (cta_group::2) ----------------------------------------------
// Address of the same shared-memory object in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose byte count completes on the
// mbarrier at cluster address `bar`, which may sit in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Block-scaled FP4 MMA of the CTA pair (M = 256), and the commit that arrives
// on the mbarrier at `bar` in both CTAs once the pair's prior tcgen05
// operations have completed; each issued by one elected lane of a converged
// warp (the warp's operands stay warp-uniform).
template <bool MX>
__device__ __forceinline__ void tc_mma_pair_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (MX) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %6, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  }
}
__device__ __forceinline__ void tc_commit_pair_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          bar),
      "h"((uint16_t)3)
      : "memory");
}
#define TC_LD32(taddr, r)                                                                                          \
  asm volatile(                                                                                                    \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18," \
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                               \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),            \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),      \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),    \
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])     \
      : "r"(taddr))

// N consecutive tensor-memory columns of this warp's 32 lanes <- N registers
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

struct Params {
  const uint8_t* As;
  const uint8_t* Bs;
  const float* ga;
  const float* gb;
  const int32_t* tA;
  const int32_t* tB;
  int M, N, K;
  int32_t* status;
  // quantized output (pair kernel with QOUT): see fp4lib::GemmArgs
  uint8_t* q_codes;
  uint8_t* q_scales;
  const float* q_g;
  float* q_amax_out;
  uint64_t q_seed;
  int q_sr, q_mma;
  uint8_t* qt_codes;  // column blocks (nullable; q_codes may then be null)
  uint8_t* qt_scales;
  uint64_t qt_seed;
  int qt_sr;
  // multi-pass GEMM (UE5M3 scale windows): add to C instead of storing it, and
  // skip the launch when window wa of A or wb of B is unused (device counts)
  int accumulate;
  const int32_t* wcount_a;
  const int32_t* wcount_b;
  int wa, wb;
};

// True when this launch is a multi-pass GEMM pass over an unused window.
__device__ __forceinline__ bool skip_pass(const Params& p) {
  return p.wcount_a != nullptr && (p.wa >= __ldg(p.wcount_a) || p.wb >= __ldg(p.wcount_b));
}

// Epilogue of one warp: 32 accumulator rows (row0.., one per lane) x 64
// columns held in r, scaled by alpha, converted, staged in shared memory as
// 32-row blocks of PL::OUT_ROW_BYTES-byte rows and written by TMA stores.
template <bool BF16, class PL>
__device__ __forceinline__ void store_block(const uint32_t (&r)[2][32], float alpha, uint8_t* stage_buf,
                                            uint32_t stage_addr, const CUtensorMap* tmap_c, int row0, int col0,
                                            int lane, bool accumulate) {
  constexpr int OB = PL::OUT_ROW_BYTES;
  constexpr int BLK_COLS = OB / (BF16 ? 2 : 4);  // columns per staged row
  constexpr int VECS = OB / 16;                  // 16-byte vectors per staged row
#pragma unroll
  for (int b = 0; b < EPI_COLS / BLK_COLS; ++b) {
    uint32_t w[4 * VECS];
    if constexpr (BF16) {
#pragma unroll
      for (int i = 0; i < 2 * VECS * 2; ++i) {
        const int c = BLK_COLS * b + 2 * i;
        const float x0 = __fmul_rn(__uint_as_float(r[c >> 5][c & 31]), alpha);
        const float x1 = __fmul_rn(__uint_as_float(r[c >> 5][(c & 31) + 1]), alpha);
        const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4 * VECS; ++i) {
        const int c = BLK_COLS * b + i;
        w[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[c >> 5][c & 31]), alpha));
      }
    }
    // the previous block's store must have read the staging buffer
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    // row `lane`; with 64-byte rows, 16-byte chunk v goes to chunk
    // v ^ ((lane >> 1) & 3), the 64-byte swizzle the output map declares
#pragma unroll
    for (int v = 0; v < VECS; ++v) {
      const int pc = VECS == 4 ? (v ^ ((lane >> 1) & 3)) : v;
      *reinterpret_cast<uint4*>(stage_buf + lane * OB + pc * 16) =
          make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      if (accumulate) tma_reduce_add_2d(tmap_c, stage_addr, col0 + BLK_COLS * b, row0);
      else tma_store_2d(tmap_c, stage_addr, col0 + BLK_COLS * b, row0);
      bulk_commit();
    }
  }
}

// Quantizing epilogue of one warp: rows row0 .. row0 + 31 (row0 + lane in
// this lane) x 64 columns from col0 of bf16(acc * alpha), the values the
// other epilogue would store, quantized as fp4_quantize would (E4M3 scales,
// block amax, scale, RNE or Philox SR at output-layout indices):
//  * row blocks (p.q_codes): 16 columns of the lane's row, indices
//    row * N + col; 32 code bytes and 4 scale bytes per lane;
//  * column blocks (p.qt_codes), the layout of C^T: 16 rows of one column,
//    indices col * M + row.  The warp's 32 x 64 values pass through its
//    2 KB staging buffer 32 columns at a time (row-major, 64 bytes a row,
//    16-byte chunks XOR-swizzled by row); lane l then holds columns 2 (l % 16)
//    and + 1 of rows 16 (l / 16) .. + 15 and quantizes both 16-row blocks.
__device__ __forceinline__ void quant_epilogue(const uint32_t (&r)[2][32], float alpha, const Params& p, int row0,
                                               int lane, int col0, float s_enc_out, float& amax_local,
                                               uint8_t* stage) {
  const int row = row0 + lane;
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int c = 2 * i;
    const float x0 = __fmul_rn(__uint_as_float(r[c >> 5][c & 31]), alpha);
    const float x1 = __fmul_rn(__uint_as_float(r[c >> 5][(c & 31) + 1]), alpha);
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  if (p.q_codes != nullptr) {
    uint32_t q[8];
    uint32_t sc = 0;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      const uint32_t* wb = w + 8 * blk;
      const float a = fp4dev::absmax_words(wb, 8);
      amax_local = fmaxf(amax_local, a);
      const fp4dev::BlockScale bs = fp4dev::block_scale<fp4dev::SF_E4M3, true>(a, s_enc_out);
      const uint64_t idx0 = (uint64_t)row * (uint64_t)p.N + (uint64_t)(col0 + 16 * blk);
      const uint2 qq = p.q_sr ? fp4dev::quant16<true>(wb, bs.r, p.q_seed, idx0)
                              : fp4dev::quant16<false>(wb, bs.r, p.q_seed, idx0);
      q[2 * blk] = qq.x;
      q[2 * blk + 1] = qq.y;
      sc |= bs.code << (8 * blk);
    }
    uint4* dst = reinterpret_cast<uint4*>(p.q_codes + (int64_t)row * (p.N / 2) + col0 / 2);
    dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
    dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
    const int64_t nb = p.N / 16, b = col0 / 16;
    const int64_t off = p.q_mma ? fp4dev::mma_sf_offset(row, b, nb) : (int64_t)row * nb + b;
    *reinterpret_cast<uint32_t*>(p.q_scales + off) = sc;
  } else {
    amax_local = fmaxf(amax_local, fp4dev::absmax_words(w, 32));
  }
  if (p.qt_codes == nullptr) return;
  const int cp = lane & 15, rb = lane >> 4;
  const int m = row0 + 16 * rb;  // first row of this lane's blocks
  const int64_t mh = p.M / 2, nbt = p.M / 16, bt = m / 16;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    __syncwarp();  // the previous half's reads are done
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(stage + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(w[16 * hh + 4 * j], w[16 * hh + 4 * j + 1], w[16 * hh + 4 * j + 2], w[16 * hh + 4 * j + 3]);
    __syncwarp();
    uint32_t v[16];  // rows m .. m + 15, columns (2 cp, 2 cp + 1) of this half
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int rr = 16 * rb + i;
      v[i] = *reinterpret_cast<const uint32_t*>(stage + rr * 64 + (((cp >> 2) ^ ((rr >> 1) & 3)) << 4) + (cp & 3) * 4);
    }
    const uint32_t am2 = fp4dev::absmax_words2(v, 16);
    const fp4dev::BlockScale b0 = fp4dev::block_scale<fp4dev::SF_E4M3, true>(fp4dev::bf16_lo(am2), s_enc_out);
    const fp4dev::BlockScale b1 = fp4dev::block_scale<fp4dev::SF_E4M3, true>(fp4dev::bf16_hi(am2), s_enc_out);
    const int n = col0 + 32 * hh + 2 * cp;  // the low column; its C^T row
    const uint64_t i0 = (uint64_t)n * (uint64_t)p.M + (uint64_t)m;
    const uint2 q0 = p.qt_sr ? fp4dev::quant16_col<true, false>(v, b0.r, p.qt_seed, i0)
                             : fp4dev::quant16_col<false, false>(v, b0.r, p.qt_seed, i0);
    const uint2 q1 = p.qt_sr ? fp4dev::quant16_col<true, true>(v, b1.r, p.qt_seed, i0 + (uint64_t)p.M)
                             : fp4dev::quant16_col<false, true>(v, b1.r, p.qt_seed, i0 + (uint64_t)p.M);
    *reinterpret_cast<uint2*>(p.qt_codes + (int64_t)n * mh + m / 2) = q0;
    *reinterpret_cast<uint2*>(p.qt_codes + (int64_t)(n + 1) * mh + m / 2) = q1;
    p.qt_scales[p.q_mma ? fp4dev::mma_sf_offset(n, bt, nbt) : (int64_t)n * nbt + bt] = (uint8_t)b0.code;
    p.qt_scales[p.q_mma ? fp4dev::mma_sf_offset(n + 1, bt, nbt) : (int64_t)(n + 1) * nbt + bt] = (uint8_t)b1.code;
  }
  __syncwarp();
}

// Epilogue scale of the accumulator: alpha = 1 / (s_encA * s_encB), times
// 2^(tA + tB) for UE5M3 (1 for MXFP4).
template <int FMT>
__device__ __forceinline__ float epilogue_alpha(const Params& p) {
  float alpha = 1.0f;
  if constexpr (FMT != fp4dev::SF_E8M0) {
    constexpr int SFMT = FMT == fp4dev::SF_UE5M3 ? fp4dev::SF_E4M3 : FMT;
    const float sa = fp4dev::global_encode_scale<SFMT>(__ldg(p.ga), nullptr);
    const float sb = fp4dev::global_encode_scale<SFMT>(__ldg(p.gb), nullptr);
    alpha = __fdiv_rn(1.0f, __fmul_rn(sa, sb));
    if (FMT == fp4dev::SF_UE5M3) alpha = ldexpf(alpha, __ldg(p.tA) + __ldg(p.tB));
  }
  return alpha;
}

template <int FMT, bool BF16, class PL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_fp4(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
               const __grid_constant__ CUtensorMap tmap_c, Params p) {
  constexpr bool MX = FMT == fp4dev::SF_E8M0;
  constexpr int ATOMS = MX ? 2 : 4;         // 512-byte scale atoms per 128 rows per K step
  constexpr int SFA_BYTES = 512 * ATOMS;    // scales of one K step for 128 rows
  constexpr int SFB_HALF = SFA_BYTES;       // per 128 rows of B
  constexpr uint32_t IDESC = make_idesc(BM, BN, MX);
  constexpr int STAGES = PL::STAGES;
  constexpr int SMEM_A = PL::SMEM_A, SMEM_B = PL::SMEM_B, SMEM_SFA = PL::SMEM_SFA, SMEM_SFB = PL::SMEM_SFB;
  constexpr int SMEM_OUT = PL::SMEM_OUT, SMEM_BAR = PL::SMEM_BAR, STAGE_BYTES = PL::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = PL::TMEM_COLS, TMEM_SFA = PL::TMEM_SFA, TMEM_SFB = PL::TMEM_SFB;

  if (skip_pass(p)) return;  // uniform: before any barrier, cluster sync or tensor memory
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  // barriers: full[S] (codes landed), sf[S] (scales written to tensor
  // memory), empty[S] (stage's MMAs done), sfd_full[F] / sfd_empty[F] (scale
  // ring slot landed / read), acc_full, acc_empty
  const uint32_t bar_full = sbase + SMEM_BAR;
  const uint32_t bar_sf = bar_full + 8 * STAGES;
  const uint32_t bar_empty = bar_sf + 8 * STAGES;
  const uint32_t bar_sfd_full = bar_empty + 8 * STAGES;
  const uint32_t bar_sfd_empty = bar_sfd_full + 8 * SF_SLOTS;
  const uint32_t bar_acc_full = bar_sfd_empty + 8 * SF_SLOTS;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  constexpr int BAR_BYTES = 8 * (3 * STAGES + 2 * SF_SLOTS + 2);
  static_assert(BAR_BYTES + 16 <= 256, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_BAR + BAR_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_BAR + BAR_BYTES + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = p.M / BM, n_tiles = (p.N + BN - 1) / BN;  // N % 128 == 0: the last tile may be half
  const int m_groups = m_tiles;
  const int num_units = m_groups * n_tiles;
  const int cluster_id = blockIdx.x, num_clusters = gridDim.x;
  const int k_steps = p.K / BK;
  const int64_t sf_row_stride = (int64_t)(p.K / (MX ? 32 : 16)) / 4 * 512;  // bytes per 128-row slab

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_sf + 8 * s, NUM_SF_WARPS);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int s = 0; s < SF_SLOTS; ++s) {
      mbar_init(bar_sfd_full + 8 * s, 1);
      mbar_init(bar_sfd_empty + 8 * s, NUM_SF_WARPS);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, NUM_EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cluster_id; u < num_units && ok; u += num_clusters) {
        const int mt = u % m_groups, nt = u / m_groups;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status) || *abort_flag) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_expect_tx(fb, A_BYTES + B_BYTES);
          tma_load_2d(sbase + SMEM_A + stage * A_BYTES, &tmap_a, fb, ks * (BK / 2), mt * BM);
          tma_load_2d(sbase + SMEM_B + stage * B_BYTES, &tmap_b, fb, ks * (BK / 2), nt * BN);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int iter = 0;
      for (int u = cluster_id; u < num_units && ok; u += num_clusters, ++iter) {
        if (iter > 0) {
          if (!wait_bounded(bar_acc_empty, acc_phase ^ 1u, abort_flag, p.status)) break;
          tc_fence_after();
        }
        for (int ks = 0; ks < k_steps; ++ks) {
          // scales in tensor memory, then the code tiles in shared memory
          if (!wait_bounded(bar_sf + 8 * stage, phase, abort_flag, p.status) ||
              !wait_bounded(bar_full + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + TMEM_SFA + 16 * stage;
          const uint32_t sfb_t = tmem_base + TMEM_SFB + 32 * stage;
          const uint32_t a_smem = sbase + SMEM_A + stage * A_BYTES;
          const uint32_t b_smem = sbase + SMEM_B + stage * B_BYTES;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // K step j: 64 elements = 32 bytes into each 128-byte swizzled row
            const uint64_t ad = smem_desc(a_smem + 32 * j, 0, 1024, 2);
            const uint64_t bd = smem_desc(b_smem + 32 * j, 0, 1024, 2);
            uint32_t idesc = IDESC;
            uint32_t sfa_col = sfa_t + 4 * j, sfb_col = sfb_t + 8 * j;
            if constexpr (MX) {
              // two K steps share an atom; the second reads bytes 2-3 of each cell
              sfa_col = sfa_t + 4 * (j >> 1);
              sfb_col = sfb_t + 8 * (j >> 1);
              const uint32_t id = (j & 1) ? 2u : 0u;
              idesc |= (id << 29) | (id << 4);
            }
            tc_mma<MX>(tmem_base, ad, bd, idesc, sfa_col, sfb_col, (ks > 0 || j > 0) ? 1u : 0u);
          }
          // stage (smem and its scale columns) free once these finish
          tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(bar_acc_full);
        acc_phase ^= 1u;
      }
    }
    __syncwarp();
  } else if (warp == SF_PRODUCER_WARP) {
    // ------------------------------ scale producer ------------------------
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cluster_id; u < num_units && ok; u += num_clusters) {
        const int mt = u % m_groups, nt = u / m_groups;
        // a half tile past N (N % 256 == 128) reads the first half's scales:
        // its code rows are zero-filled, so any finite scale gives 0
        const int b_hi = (2 * nt + 1) * 128 < p.N ? 2 * nt + 1 : 2 * nt;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(bar_sfd_empty + 8 * slot, phase ^ 1u, abort_flag, p.status) || *abort_flag) {
            ok = false;
            break;
          }
          const uint32_t sb = bar_sfd_full + 8 * slot;
          mbar_expect_tx(sb, SFA_BYTES + 2 * SFB_HALF);
          // scales of this K step: SFA_BYTES contiguous bytes per 128-row slab
          bulk_load(sbase + SMEM_SFA + slot * SFA_MAX, p.As + mt * sf_row_stride + (int64_t)ks * SFA_BYTES,
                    SFA_BYTES, sb);
          bulk_load(sbase + SMEM_SFB + slot * SFB_MAX, p.Bs + (2 * nt) * sf_row_stride + (int64_t)ks * SFB_HALF,
                    SFB_HALF, sb);
          bulk_load(sbase + SMEM_SFB + slot * SFB_MAX + SFB_HALF,
                    p.Bs + b_hi * sf_row_stride + (int64_t)ks * SFB_HALF, SFB_HALF, sb);
          if (++slot == SF_SLOTS) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < FIRST_EPI_WARP) {
    // ------------------------------ scale writers -------------------------
    // Lane i of the warp serving quarter q writes, for every 512-byte atom
    // (rows 0..127 x 4 blocks), the atom's 16-byte row i -- the scales of rows
    // i, i+32, i+64, i+96 -- into 4 consecutive columns of lane 32q+i.
    const int quarter = warp & 3;
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    for (int u = cluster_id; u < num_units; u += num_clusters) {
      bool ok = true;
      for (int ks = 0; ks < k_steps; ++ks) {
        if (!wait_bounded(bar_sfd_full + 8 * slot, sphase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* sfa = smem + SMEM_SFA + slot * SFA_MAX + 16 * lane;
        const uint8_t* sfb = smem + SMEM_SFB + slot * SFB_MAX + 16 * lane;
        uint32_t va[4 * ATOMS], vb[8 * ATOMS];
#pragma unroll
        for (int j = 0; j < ATOMS; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sfa + 512 * j);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sfb + 512 * j);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sfb + SFB_HALF + 512 * j);
          va[4 * j + 0] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
          vb[8 * j + 0] = b0.x; vb[8 * j + 1] = b0.y; vb[8 * j + 2] = b0.z; vb[8 * j + 3] = b0.w;
          vb[8 * j + 4] = b1.x; vb[8 * j + 5] = b1.y; vb[8 * j + 6] = b1.z; vb[8 * j + 7] = b1.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfd_empty + 8 * slot);  // the scale slot may refill
        // this stage's tensor-memory columns are free once the MMAs of K step
        // k - STAGES have completed (their commit to empty[stage])
        if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t lane_base = tmem_base + ((uint32_t)(32 * quarter) << 16);
        if constexpr (ATOMS == 4) {
          tc_st16(lane_base + TMEM_SFA + 16 * stage, va);
          tc_st32(lane_base + TMEM_SFB + 32 * stage, vb);
        } else {
          tc_st8(lane_base + TMEM_SFA + 16 * stage, va);
          tc_st16(lane_base + TMEM_SFB + 32 * stage, vb);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sf + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++slot == SF_SLOTS) {
          slot = 0;
          sphase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int ew = warp - FIRST_EPI_WARP;  // 0..15
    const int quarter = warp & 3;          // tensor-memory lanes this warp may access
    const int cblk = ew >> 2;              // 64-column block of the accumulator
    const float alpha = epilogue_alpha<FMT>(p);
    uint8_t* stage_buf = smem + SMEM_OUT + ew * STAGE_BYTES;
    const uint32_t stage_addr = smem_u32(stage_buf);
    uint32_t acc_phase = 0;
    for (int u = cluster_id; u < num_units; u += num_clusters) {
      const int mt = u % m_groups, nt = u / m_groups;
      if (!wait_bounded(bar_acc_full, acc_phase, abort_flag, p.status)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      uint32_t r[2][32];
      const uint32_t t0 = tmem_base + ((uint32_t)(32 * quarter) << 16) + EPI_COLS * cblk;
      TC_LD32(t0, r[0]);
      TC_LD32(t0 + 32, r[1]);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty);
      // 64-column slabs at or past N (a half tile) hold no output
      if (nt * BN + EPI_COLS * cblk < p.N)
        store_block<BF16, PL>(r, alpha, stage_buf, stage_addr, &tmap_c, mt * BM + 32 * quarter,
                              nt * BN + EPI_COLS * cblk, lane, p.accumulate != 0);
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }

  // ------------------------------ teardown --------------------------------
  tc_fence_before();
  __syncthreads();
  drain_after_abort(abort_flag);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// CTA-pair form: a cluster of 2 CTAs computes a 256 x 256 output tile with
// cta_group::2 MMAs (M = 256).  CTA r (r = 0, 1) holds rows 128r..128r+127 of
// the A tile and of the B tile in its shared memory and rows 128r.. of the
// accumulator in its tensor memory; the MMA of the even CTA reads both CTAs'
// operands, so each SM streams A + B/2 per K step instead of A + B.  Roles
// as in k_gemm_fp4, with the pair's hand-offs:
//   * both producers' TMA loads complete on the even CTA's full[] barrier,
//     whose expect_tx covers both CTAs' bytes;
//   * the even CTA's MMA thread waits for full[] and for sf[] (scale writers
//     of both CTAs), issues the MMAs and commits to empty[] / acc_full in both
//     CTAs at once;
//   * each CTA's scale writers fill its own tensor memory: its 128 rows of A
//     scales and all 256 rows of B scales (each SM applies the B scales of
//     the whole tile to its half of the product);
//   * both CTAs' epilogue warps drain their own accumulator rows and release
//     them on the even CTA's acc_empty.
template <int FMT, bool BF16, class PL, bool QOUT = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_fp4_pair(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_c, Params p) {
  constexpr bool MX = FMT == fp4dev::SF_E8M0;
  constexpr int ATOMS = MX ? 2 : 4;
  constexpr int SFA_BYTES = 512 * ATOMS;
  constexpr int SFB_HALF = SFA_BYTES;
  constexpr int PM = 2 * BM;  // rows of the pair's output tile
  constexpr int B_STAGE = PL::B_STAGE;
  static_assert(B_STAGE == B_BYTES / 2, "each CTA holds half of the B tile");
  constexpr uint32_t IDESC = make_idesc(PM, BN, MX);
  constexpr int STAGES = PL::STAGES;
  constexpr int SMEM_A = PL::SMEM_A, SMEM_B = PL::SMEM_B, SMEM_SFA = PL::SMEM_SFA, SMEM_SFB = PL::SMEM_SFB;
  constexpr int SMEM_OUT = PL::SMEM_OUT, SMEM_BAR = PL::SMEM_BAR, STAGE_BYTES = PL::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = PL::TMEM_COLS, TMEM_SFA = PL::TMEM_SFA, TMEM_SFB = PL::TMEM_SFB;

  if (skip_pass(p)) return;  // uniform: before any barrier, cluster sync or tensor memory
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + SMEM_BAR;
  const uint32_t bar_sf = bar_full + 8 * STAGES;
  const uint32_t bar_empty = bar_sf + 8 * STAGES;
  const uint32_t bar_sfd_full = bar_empty + 8 * STAGES;
  const uint32_t bar_sfd_empty = bar_sfd_full + 8 * SF_SLOTS;
  const uint32_t bar_acc_full = bar_sfd_empty + 8 * SF_SLOTS;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  constexpr int BAR_BYTES = 8 * (3 * STAGES + 2 * SF_SLOTS + 2);
  static_assert(BAR_BYTES + 16 <= 256, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_BAR + BAR_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_BAR + BAR_BYTES + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();  // 0: issues the MMAs; 1: its peer
  const bool leader = crank == 0;
  const int m_pairs = p.M / PM, n_tiles = (p.N + BN - 1) / BN;  // N % 128 == 0: the last tile may be half
  // units walk N fastest: the clusters of one round share a few 256-row
  // blocks of A and sweep B, which keeps a round's operands within L2 even
  // when A alone approaches its size (dgrad, wgrad)
  const int num_units = m_pairs * n_tiles;
  const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
  const int k_steps = p.K / BK;
  const int64_t sf_row_stride = (int64_t)(p.K / (MX ? 32 : 16)) / 4 * 512;  // bytes per 128-row slab
  // the even CTA's barriers that the peer signals, as cluster addresses
  const uint32_t lead_full = mapa_shared(bar_full, 0);
  const uint32_t lead_acc_empty = mapa_shared(bar_acc_empty, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // one arrival with the expected bytes of both CTAs' code tiles, plus one
      // per scale-writer warp of both CTAs
      mbar_init(bar_full + 8 * s, 1 + 2 * NUM_SF_WARPS);
      mbar_init(bar_sf + 8 * s, 1);  // unused in the pair form
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int s = 0; s < SF_SLOTS; ++s) {
      mbar_init(bar_sfd_full + 8 * s, 1);
      mbar_init(bar_sfd_empty + 8 * s, NUM_SF_WARPS);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 2 * NUM_EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    // one warp of each CTA of the pair allocates, together, the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers and tensor memory exist before any cross-CTA traffic
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) {
    // the MMA addresses the peer's tensor memory with the even CTA's column base
    uint32_t peer_base;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer_base) : "r"(mapa_shared(smem_u32(tmem_slot), crank ^ 1u)));
    if (peer_base != tmem_base) {
      *abort_flag = 1;
      fp4dev::set_status(p.status, FP4_ERR_CUDA);
    }
  }
  __syncthreads();
  const bool run = *abort_flag == 0;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0 && run) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cluster_id; u < num_units && ok; u += num_clusters) {
        const int mp = u / n_tiles, nt = u % n_tiles;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status) || *abort_flag) {
            ok = false;
            break;
          }
          if (leader) mbar_expect_tx(bar_full + 8 * stage, 2 * (A_BYTES + B_STAGE));
          const uint32_t fb = lead_full + 8 * stage;
          tma_load_2d_pair(sbase + SMEM_A + stage * A_BYTES, &tmap_a, fb, ks * (BK / 2), mp * PM + BM * (int)crank);
          tma_load_2d_pair(sbase + SMEM_B + stage * B_STAGE, &tmap_b, fb, ks * (BK / 2),
                           nt * BN + (BN / 2) * (int)crank);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer (even CTA) -----------------
    // The whole warp runs the loop (its operands stay warp-uniform); one
    // elected lane issues each tcgen05 instruction.
    if (leader && run) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int iter = 0;
      for (int u = cluster_id; u < num_units && ok; u += num_clusters, ++iter) {
        if (iter > 0) {
          if (!wait_lane0(bar_acc_empty, acc_phase ^ 1u, abort_flag, p.status, lane)) break;
          tc_fence_after();
        }
        for (int ks = 0; ks < k_steps; ++ks) {
          // codes of both CTAs landed and both CTAs' scales written
          if (!wait_lane0(bar_full + 8 * stage, phase, abort_flag, p.status, lane)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + TMEM_SFA + 16 * stage;
          const uint32_t sfb_t = tmem_base + TMEM_SFB + 32 * stage;
          const uint32_t a_smem = sbase + SMEM_A + stage * A_BYTES;
          const uint32_t b_smem = sbase + SMEM_B + stage * B_STAGE;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = smem_desc(a_smem + 32 * j, 0, 1024, 2);
            const uint64_t bd = smem_desc(b_smem + 32 * j, 0, 1024, 2);
            uint32_t idesc = IDESC;
            uint32_t sfa_col = sfa_t + 4 * j, sfb_col = sfb_t + 8 * j;
            if constexpr (MX) {
              sfa_col = sfa_t + 4 * (j >> 1);
              sfb_col = sfb_t + 8 * (j >> 1);
              const uint32_t id = (j & 1) ? 2u : 0u;
              idesc |= (id << 29) | (id << 4);
            }
            tc_mma_pair_elect<MX>(tmem_base, ad, bd, idesc, sfa_col, sfb_col, (ks > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit_pair_elect(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_elect(bar_acc_full);
        acc_phase ^= 1u;
      }
    }
    __syncwarp();
  } else if (warp == SF_PRODUCER_WARP) {
    // ------------------------------ scale producer ------------------------
    if (lane == 0 && run) {
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cluster_id; u < num_units && ok; u += num_clusters) {
        const int mp = u / n_tiles, nt = u % n_tiles;
        const int a_slab = 2 * mp + (int)crank;
        // a half tile past N (N % 256 == 128) reads the first half's scales:
        // its code rows are zero-filled, so any finite scale gives 0
        const int b_hi = (2 * nt + 1) * 128 < p.N ? 2 * nt + 1 : 2 * nt;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!wait_bounded(bar_sfd_empty + 8 * slot, phase ^ 1u, abort_flag, p.status) || *abort_flag) {
            ok = false;
            break;
          }
          const uint32_t sb = bar_sfd_full + 8 * slot;
          mbar_expect_tx(sb, SFA_BYTES + 2 * SFB_HALF);
          bulk_load(sbase + SMEM_SFA + slot * SFA_MAX, p.As + a_slab * sf_row_stride + (int64_t)ks * SFA_BYTES,
                    SFA_BYTES, sb);
          bulk_load(sbase + SMEM_SFB + slot * SFB_MAX, p.Bs + (2 * nt) * sf_row_stride + (int64_t)ks * SFB_HALF,
                    SFB_HALF, sb);
          bulk_load(sbase + SMEM_SFB + slot * SFB_MAX + SFB_HALF,
                    p.Bs + b_hi * sf_row_stride + (int64_t)ks * SFB_HALF, SFB_HALF, sb);
          if (++slot == SF_SLOTS) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < FIRST_EPI_WARP) {
    // ------------------------------ scale writers -------------------------
    const int quarter = warp & 3;
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    for (int u = cluster_id; u < num_units && run; u += num_clusters) {
      bool ok = true;
      for (int ks = 0; ks < k_steps; ++ks) {
        if (!wait_bounded(bar_sfd_full + 8 * slot, sphase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* sfa = smem + SMEM_SFA + slot * SFA_MAX + 16 * lane;
        const uint8_t* sfb = smem + SMEM_SFB + slot * SFB_MAX + 16 * lane;
        uint32_t va[4 * ATOMS], vb[8 * ATOMS];
#pragma unroll
        for (int j = 0; j < ATOMS; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sfa + 512 * j);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sfb + 512 * j);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sfb + SFB_HALF + 512 * j);
          va[4 * j + 0] = a.x; va[4 * j + 1] = a.y; va[4 * j + 2] = a.z; va[4 * j + 3] = a.w;
          vb[8 * j + 0] = b0.x; vb[8 * j + 1] = b0.y; vb[8 * j + 2] = b0.z; vb[8 * j + 3] = b0.w;
          vb[8 * j + 4] = b1.x; vb[8 * j + 5] = b1.y; vb[8 * j + 6] = b1.z; vb[8 * j + 7] = b1.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfd_empty + 8 * slot);
        // this CTA's columns of the stage are free once the pair's MMAs of
        // K step k - STAGES have completed (their commit reaches both CTAs)
        if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t lane_base = tmem_base + ((uint32_t)(32 * quarter) << 16);
        if constexpr (ATOMS == 4) {
          tc_st16(lane_base + TMEM_SFA + 16 * stage, va);
          tc_st32(lane_base + TMEM_SFB + 32 * stage, vb);
        } else {
          tc_st8(lane_base + TMEM_SFA + 16 * stage, va);
          tc_st16(lane_base + TMEM_SFB + 32 * stage, vb);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_full + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++slot == SF_SLOTS) {
          slot = 0;
          sphase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int ew = warp - FIRST_EPI_WARP;
    const int quarter = warp & 3;
    const int cblk = ew >> 2;
    const float alpha = epilogue_alpha<FMT>(p);
    uint8_t* stage_buf = smem + SMEM_OUT + ew * STAGE_BYTES;
    const uint32_t stage_addr = smem_u32(stage_buf);
    float s_enc_out = 1.0f, amax_local = 0.0f;
    if constexpr (QOUT) s_enc_out = fp4dev::global_encode_scale<fp4dev::SF_E4M3>(__ldg(p.q_g), p.status);
    uint32_t acc_phase = 0;
    for (int u = cluster_id; u < num_units && run; u += num_clusters) {
      const int mp = u / n_tiles, nt = u % n_tiles;
      if (!wait_bounded(bar_acc_full, acc_phase, abort_flag, p.status)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      uint32_t r[2][32];
      const uint32_t t0 = tmem_base + ((uint32_t)(32 * quarter) << 16) + EPI_COLS * cblk;
      TC_LD32(t0, r[0]);
      TC_LD32(t0 + 32, r[1]);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_acc_empty);
      if (nt * BN + EPI_COLS * cblk >= p.N) continue;  // a slab past N (half tile): no output
      if constexpr (QOUT) {
        quant_epilogue(r, alpha, p, mp * PM + BM * (int)crank + 32 * quarter, lane, nt * BN + EPI_COLS * cblk,
                       s_enc_out, amax_local, stage_buf);
      } else {
        store_block<BF16, PL>(r, alpha, stage_buf, stage_addr, &tmap_c, mp * PM + BM * (int)crank + 32 * quarter,
                              nt * BN + EPI_COLS * cblk, lane, p.accumulate != 0);
      }
    }
    if constexpr (QOUT) {
      if (p.q_amax_out != nullptr) {
        // non-negative floats order like their bit patterns
        const unsigned int am = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax_local));
        if (lane == 0) atomicMax(reinterpret_cast<unsigned int*>(p.q_amax_out), am);
      }
    }
    if (lane == 0) bulk_wait0();
    __syncwarp();
  }

  // ------------------------------ teardown --------------------------------
  tc_fence_before();
  __syncthreads();
  drain_after_abort(abort_flag);
  cluster_sync_all();  // no more MMAs, TMA completions or arrivals between the two CTAs
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 2-D uint8 map over packed codes [rows, K/2 bytes] with a 128-byte x box_rows
// box and the 128-byte swizzle the MMA descriptors assume.
bool make_code_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output C [M, N] (leading dimension ldc elements): 32-row x `row_bytes`
// boxes, 64-byte swizzle for 64-byte rows, none for 16-byte rows.
bool make_out_map(CUtensorMap* map, void* base, int64_t M, int64_t N, int64_t ldc, bool bf16, int row_bytes) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)(ldc * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(row_bytes / esz), 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() { return fp4lib::current_sm_count(); }

template <int FMT, bool BF16, class PL>
cudaError_t launch_t(const fp4lib::GemmArgs& a, cudaStream_t st) {
  auto kern = k_gemm_fp4<FMT, BF16, PL>;
  constexpr int SMEM_LAUNCH = PL::SMEM_LAUNCH;
  static fp4lib::DeviceInts attr_set;  // per device: the shared-memory size is set
  cudaError_t e = cudaSuccess;
  attr_set.get([&] {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LAUNCH);
    return e == cudaSuccess ? 1 : 0;
  });
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb, mc;
  if (!make_code_map(&ma, a.Aq, a.M, a.K / 2, BM) || !make_code_map(&mb, a.Bq, a.N, a.K / 2, BN) ||
      !make_out_map(&mc, a.C, a.M, a.N, a.ldc, BF16, PL::OUT_ROW_BYTES))
    return cudaErrorInvalidValue;
  Params p{};
  p.As = a.As;
  p.Bs = a.Bs;
  p.ga = a.ga;
  p.gb = a.gb;
  p.tA = a.tA;
  p.accumulate = a.accumulate ? 1 : 0;
  p.wcount_a = a.wcount_a;
  p.wcount_b = a.wcount_b;
  p.wa = a.wa;
  p.wb = a.wb;
  p.tB = a.tB;
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.status = a.status;
  const int units = (int)((a.M / BM) * ((a.N + BN - 1) / BN));
  const int ctas = units < sm_count() ? units : sm_count();
  kern<<<(unsigned)ctas, NUM_THREADS, SMEM_LAUNCH, st>>>(ma, mb, mc, p);
  return cudaGetLastError();
}

// CTA-pair launch: clusters of 2 CTAs, one 256 x 256 output tile per cluster
// and round.
template <int FMT, bool BF16, bool QOUT = false>
cudaError_t launch_pair(const fp4lib::GemmArgs& a, cudaStream_t st) {
  using PL = PlanPair;
  auto kern = k_gemm_fp4_pair<FMT, BF16, PL, QOUT>;
  constexpr int SMEM_LAUNCH = PL::SMEM_LAUNCH;
  // per device: the shared-memory size set, then the co-resident clusters
  static fp4lib::DeviceInts max_clusters_of;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_LAUNCH;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaSuccess;
  const int max_clusters = max_clusters_of.get([&] {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LAUNCH);
    if (err != cudaSuccess) return 0;
    cfg.gridDim = dim3(sm_count() & ~1, 1, 1);
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    return err == cudaSuccess ? n : 0;
  });
  if (err != cudaSuccess) return err;
  if (max_clusters <= 0) return cudaErrorInvalidConfiguration;
  CUtensorMap ma, mb, mc;
  // with a quantized output the C map is never used; it is built over a code
  // buffer of the same size (M x N/2 bytes, either layout)
  void* cbase = QOUT ? static_cast<void*>(a.q_codes != nullptr ? a.q_codes : a.qt_codes) : a.C;
  const int64_t cn = QOUT ? a.N / 4 : a.N, cld = QOUT ? a.N / 4 : a.ldc;
  if (!make_code_map(&ma, a.Aq, a.M, a.K / 2, BM) || !make_code_map(&mb, a.Bq, a.N, a.K / 2, BN / 2) ||
      !make_out_map(&mc, cbase, a.M, cn, cld, QOUT ? true : BF16, PL::OUT_ROW_BYTES))
    return cudaErrorInvalidValue;
  Params p{};
  p.As = a.As;
  p.Bs = a.Bs;
  p.ga = a.ga;
  p.gb = a.gb;
  p.tA = a.tA;
  p.accumulate = a.accumulate ? 1 : 0;
  p.wcount_a = a.wcount_a;
  p.wcount_b = a.wcount_b;
  p.wa = a.wa;
  p.wb = a.wb;
  p.tB = a.tB;
  p.M = (int)a.M;
  p.N = (int)a.N;
  p.K = (int)a.K;
  p.status = a.status;
  p.q_codes = a.q_codes;
  p.q_scales = a.q_scales;
  p.q_g = a.q_g;
  p.q_amax_out = a.q_amax_out;
  p.q_seed = a.q_seed;
  p.q_sr = a.q_sr ? 1 : 0;
  p.q_mma = a.q_mma ? 1 : 0;
  p.qt_codes = a.qt_codes;
  p.qt_scales = a.qt_scales;
  p.qt_seed = a.qt_seed;
  p.qt_sr = a.qt_sr ? 1 : 0;
  const int units = (int)((a.M / (2 * BM)) * ((a.N + BN - 1) / BN));
  const int clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, p);
}

// CTA pairs whenever the 128-row tiles pair up; single CTAs otherwise.
template <int FMT, bool BF16>
cudaError_t launch_cm(const fp4lib::GemmArgs& a, cudaStream_t st) {
  const int64_t m_tiles = a.M / BM;
  if (m_tiles % 2 == 0) return launch_pair<FMT, BF16>(a, st);
  return a.K >= 8192 ? launch_t<FMT, BF16, PlanLongK>(a, st) : launch_t<FMT, BF16, PlanShortK>(a, st);
}

}  // namespace

namespace fp4lib {

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  if (a.N % 128 != 0) return cudaErrorNotSupported;
  if (a.qout) {
    // quantizing epilogue: CTA-pair kernel only (M a multiple of 256)
    if (a.M % (2 * BM) != 0) return cudaErrorNotSupported;
    switch (a.fmt) {
      case FP4_SF_E4M3: return launch_pair<fp4dev::SF_E4M3, true, true>(a, st);
      case FP4_SF_UE5M3: return launch_pair<fp4dev::SF_UE5M3, true, true>(a, st);
      case FP4_SF_E8M0: return launch_pair<fp4dev::SF_E8M0, true, true>(a, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.fmt) {
    case FP4_SF_E4M3: return a.bf16_out ? launch_cm<fp4dev::SF_E4M3, true>(a, st) : launch_cm<fp4dev::SF_E4M3, false>(a, st);
    case FP4_SF_UE5M3: return a.bf16_out ? launch_cm<fp4dev::SF_UE5M3, true>(a, st) : launch_cm<fp4dev::SF_UE5M3, false>(a, st);
    case FP4_SF_E8M0: return a.bf16_out ? launch_cm<fp4dev::SF_E8M0, true>(a, st) : launch_cm<fp4dev::SF_E8M0, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp4lib
