// Internal launcher interface between the C ABI (abi.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp4lib {

struct QuantArgs {
  enum Mode { ROWS, COLS, DUAL } mode;
  int fmt;
  const void* x;
  int64_t M, K, ldx;
  const float* gptr;  // device: stored global amax
  bool row_sr, col_sr, mma, amax_by_product;
  uint64_t seed_row, seed_col;
  uint8_t *codes_row, *scales_row, *codes_col, *scales_col;
  float* amax_out;
  int32_t* status;
  // UE5M3 only, nullable: atomic max of the row / transposed outputs' scale
  // codes (zeroed by the caller; launch_ue5m3_finalize turns each into t)
  uint32_t *sf_max_row, *sf_max_col;
};

cudaError_t launch_amax(const void* x, int64_t M, int64_t K, int64_t ldx, float* out, cudaStream_t st);
constexpr int AMAX_N_MAX = 8;
// the amaxes of n <= AMAX_N_MAX tensors (host arrays of their pointers and sizes) into out[0..n)
cudaError_t launch_amax_n(int n, const void* const* x, const int64_t* M, const int64_t* K, const int64_t* ldx,
                          float* out, cudaStream_t st);
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, bool mma, int64_t M, int64_t K,
                              int fmt, const float* gptr, bool bf16, void* out, cudaStream_t st);
cudaError_t launch_ue5m3_to_e4m3(const uint8_t* in, int64_t n, int32_t* t_out, uint8_t* out, int32_t* status,
                                 cudaStream_t st);
// the same re-encode with a known shift *t (device int)
cudaError_t launch_ue5m3_reencode(const uint8_t* in, int64_t n, const int32_t* t, uint8_t* out, int32_t* status,
                                  cudaStream_t st);
// words[0..n): largest UE5M3 code of a scale set -> its shift t = e_max - 7
cudaError_t launch_ue5m3_finalize(int32_t* words, int n, cudaStream_t st);
// UE5M3 scale codes -> up to three E4M3 windows (out: 3 arrays of n codes),
// shifts t_out[3], windows in use n_out[1]
cudaError_t launch_ue5m3_windows(const uint8_t* in, int64_t n, int32_t* t_out, int32_t* n_out, uint8_t* out,
                                 int32_t* status, cudaStream_t st);
cudaError_t launch_encode_scales(const float* s, int64_t n, int fmt, uint8_t* codes, float* decoded,
                                 cudaStream_t st);
cudaError_t launch_philox_bits16(uint64_t seed, uint64_t start, int64_t n, uint16_t* out, cudaStream_t st);
// 16 x 16 random Hadamard transform + row quantization (rht.cu)
cudaError_t launch_amax_rht(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t mask, float* out,
                            cudaStream_t st);
cudaError_t launch_quantize_rht(const QuantArgs& a, uint32_t mask, cudaStream_t st);
struct DualRhtArgs {
  int fmt;
  const void* x;
  int64_t M, K, ldx;
  uint32_t mask;
  const float *g_row, *g_col;  // device: stored global amaxes of the two transformed layouts
  bool row_sr, col_sr, mma, amax_by_product;
  uint64_t seed_row, seed_col;
  uint8_t *codes_row, *scales_row, *codes_col, *scales_col;
  float *amax_row_out, *amax_col_out;
  int32_t* status;
};
cudaError_t launch_amax_rht_cols(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t mask, float* out,
                                 cudaStream_t st);
cudaError_t launch_quantize_dual_rht(const DualRhtArgs& a, cudaStream_t st);

struct GemmArgs {
  const uint8_t *Aq, *As, *Bq, *Bs;
  const float *ga, *gb;
  const int32_t *tA, *tB;
  int64_t M, N, K, ldc;
  int fmt;
  bool bf16_out;
  void* C;
  int32_t* status;
  // quantized output instead of C (fp4_gemm_quantize): NVFP4 codes and scales
  // of bf16(C) in row blocks (nullable when qt_codes is given) under the
  // stored global amax q_g
  bool qout;
  uint8_t *q_codes, *q_scales;
  const float* q_g;
  float* q_amax_out;  // nullable: max |bf16(C)|
  uint64_t q_seed;
  bool q_sr, q_mma;
  // column-block output of bf16(C) (16 elements along M, codes [N, M/2]);
  // nullable, as is q_codes when this one is given
  uint8_t *qt_codes, *qt_scales;
  uint64_t qt_seed;
  bool qt_sr;
  // multi-pass GEMM over UE5M3 scale windows: add into C (float32 output),
  // and skip the launch if window wa of A or wb of B is unused
  bool accumulate;
  const int32_t *wcount_a, *wcount_b;
  int wa, wb;
};
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st);

struct GemvArgs {
  const uint8_t *Wq, *Ws;
  const float* gw;
  const void* x;
  int64_t batch, N, K;
  bool bf16_out;
  void* y;
  int32_t* status;
};
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st);
// batches of 9..64 on the tcgen05 tensor cores (gemv_umma.cu); cudaErrorNotSupported otherwise
cudaError_t launch_gemv_umma(const GemvArgs& a, cudaStream_t st);

}  // namespace fp4lib
