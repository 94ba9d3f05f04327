// C ABI of libfp4.so (declared in include/fp4.h): host-side argument checks,
// then launches on the caller's stream.  No allocation, no synchronization.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fp4.h"
#include "launch.h"

namespace {

thread_local int g_last_cuda_error = 0;

fp4_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FP4_OK;
  g_last_cuda_error = (int)e;
  // clear the runtime's per-thread last error (a non-sticky one), so that a
  // later call's launch check does not report this failure again
  (void)cudaGetLastError();
  return FP4_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_fmt(int f) { return f >= FP4_SF_E4M3 && f <= FP4_SF_MXINT4; }

// E2M5 .. E7M0 (the rest of the scale-format sweep) and the INT4 grids:
// row quantization only
bool sweep_fmt(int f) { return f >= FP4_SF_E2M5 && f <= FP4_SF_MXINT4; }

int group_of(int f) {
  if (!valid_fmt(f)) return 0;
  return (f == FP4_SF_E8M0 || f == FP4_SF_MXINT4) ? 32 : 16;
}

// Checks shared by the quantizer entry points.  rows/cols are the OUTPUT
// layout's (blocks run along cols).
fp4_status check_quant_common(const void* x, int64_t M, int64_t K, int64_t ldx, int f, int sfl, int64_t out_rows,
                              int64_t out_cols) {
  if (!valid_fmt(f) || (sfl != FP4_SFLAYOUT_PLAIN && sfl != FP4_SFLAYOUT_MMA)) return FP4_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || ldx < K) return FP4_ERR_SHAPE;
  const int G = group_of(f);
  if (out_cols % G != 0) return FP4_ERR_SHAPE;
  if (x == nullptr && M * K > 0) return FP4_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx * 2) % 16 != 0) return FP4_ERR_ALIGNMENT;
  if (sfl == FP4_SFLAYOUT_MMA && (out_rows % 128 != 0 || (out_cols / G) % 4 != 0)) return FP4_ERR_SHAPE;
  return FP4_OK;
}

fp4_status check_out(const void* codes, const void* scales) {
  if (codes == nullptr || scales == nullptr) return FP4_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(scales)) return FP4_ERR_ALIGNMENT;
  return FP4_OK;
}

// Fresh or stored global amax; sets a.gptr / a.amax_by_product / a.amax_out.
fp4_status prepare_amax(fp4lib::QuantArgs& a, const float* global_amax, float* amax_out, cudaStream_t st) {
  a.amax_out = amax_out;
  if (global_amax == nullptr) {
    if (amax_out == nullptr) return FP4_ERR_INVALID_ARG;
    fp4_status s = cuda_status(fp4lib::launch_amax(a.x, a.M, a.K, a.ldx, amax_out, st));
    if (s != FP4_OK) return s;
    a.gptr = amax_out;
    a.amax_by_product = false;
  } else {
    a.gptr = global_amax;
    a.amax_by_product = amax_out != nullptr;
    if (a.amax_by_product) {
      fp4_status s = cuda_status(cudaMemsetAsync(amax_out, 0, sizeof(float), st));
      if (s != FP4_OK) return s;
    }
  }
  return FP4_OK;
}

// UE5M3 shift by-product: zero the word(s) the quantizer maxes its scale
// codes into (n = 1 or 2 consecutive int32), before the launch.
fp4_status prepare_shift(int f, int32_t* shift_out, int n, cudaStream_t st) {
  if (shift_out == nullptr) return FP4_OK;
  if (f != FP4_SF_UE5M3) return FP4_ERR_UNSUPPORTED;
  return cuda_status(cudaMemsetAsync(shift_out, 0, n * sizeof(int32_t), st));
}

}  // namespace

extern "C" {

int fp4_group_size(fp4_scale_fmt f) { return group_of((int)f); }

fp4_status fp4_storage_bytes(int64_t rows, int64_t cols, fp4_scale_fmt f, size_t* code_bytes,
                             size_t* scale_bytes) {
  if (!valid_fmt((int)f) || code_bytes == nullptr || scale_bytes == nullptr) return FP4_ERR_INVALID_ARG;
  const int G = group_of((int)f);
  if (rows < 0 || cols < 0 || cols % G != 0) return FP4_ERR_SHAPE;
  *code_bytes = (size_t)(rows * (cols / 2));
  *scale_bytes = (size_t)(rows * (cols / G));
  return FP4_OK;
}

fp4_status fp4_amax(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, float* amax_out,
                    fp4_stream_t stream) {
  if (amax_out == nullptr) return FP4_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || ldx < K || K % 8 != 0) return FP4_ERR_SHAPE;
  if (x_bf16 == nullptr && M * K > 0) return FP4_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || (ldx * 2) % 16 != 0) return FP4_ERR_ALIGNMENT;
  return cuda_status(fp4lib::launch_amax(x_bf16, M, K, ldx, amax_out, (cudaStream_t)stream));
}

fp4_status fp4_amax_n(int n, const void* const* x_bf16, const int64_t* M, const int64_t* K, const int64_t* ldx,
                      float* amax_out, fp4_stream_t stream) {
  if (n < 0 || n > fp4lib::AMAX_N_MAX) return FP4_ERR_SHAPE;
  if (n == 0) return FP4_OK;
  if (x_bf16 == nullptr || M == nullptr || K == nullptr || ldx == nullptr || amax_out == nullptr)
    return FP4_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (M[i] < 0 || K[i] < 0 || ldx[i] < K[i] || K[i] % 8 != 0) return FP4_ERR_SHAPE;
    if (x_bf16[i] == nullptr && M[i] * K[i] > 0) return FP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16[i]) || (ldx[i] * 2) % 16 != 0) return FP4_ERR_ALIGNMENT;
  }
  return cuda_status(fp4lib::launch_amax_n(n, x_bf16, M, K, ldx, amax_out, (cudaStream_t)stream));
}

fp4_status fp4_quantize(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, fp4_scale_fmt f, fp4_rounding r,
                        uint64_t seed, const float* global_amax, int transpose, fp4_sf_layout sfl, uint8_t* codes,
                        uint8_t* scales, float* amax_out, int32_t* ue5m3_shift_out, int32_t* dev_status,
                        fp4_stream_t stream) {
  if (r != FP4_ROUND_RNE && r != FP4_ROUND_STOCHASTIC) return FP4_ERR_INVALID_ARG;
  if (transpose != 0 && transpose != 1) return FP4_ERR_INVALID_ARG;
  const int64_t out_rows = transpose ? K : M, out_cols = transpose ? M : K;
  fp4_status s = check_quant_common(x_bf16, M, K, ldx, (int)f, (int)sfl, out_rows, out_cols);
  if (s != FP4_OK) return s;
  if (transpose && sweep_fmt((int)f)) return FP4_ERR_UNSUPPORTED;
  if (transpose && (M % 32 != 0 || K % 32 != 0)) return FP4_ERR_SHAPE;
  if (M * K > 0 && (s = check_out(codes, scales)) != FP4_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  fp4lib::QuantArgs a{};
  a.mode = transpose ? fp4lib::QuantArgs::COLS : fp4lib::QuantArgs::ROWS;
  a.fmt = (int)f;
  a.x = x_bf16;
  a.M = M;
  a.K = K;
  a.ldx = ldx;
  a.mma = sfl == FP4_SFLAYOUT_MMA;
  a.status = dev_status;
  const bool sr = r == FP4_ROUND_STOCHASTIC;
  uint32_t* shift_word = reinterpret_cast<uint32_t*>(ue5m3_shift_out);
  if (transpose) {
    a.col_sr = sr;
    a.seed_col = seed;
    a.codes_col = codes;
    a.scales_col = scales;
    a.sf_max_col = shift_word;
  } else {
    a.row_sr = sr;
    a.seed_row = seed;
    a.codes_row = codes;
    a.scales_row = scales;
    a.sf_max_row = shift_word;
  }
  if ((s = prepare_shift((int)f, ue5m3_shift_out, 1, st)) != FP4_OK) return s;
  if ((s = prepare_amax(a, global_amax, amax_out, st)) != FP4_OK) return s;
  if ((s = cuda_status(fp4lib::launch_quantize(a, st))) != FP4_OK) return s;
  if (ue5m3_shift_out != nullptr) return cuda_status(fp4lib::launch_ue5m3_finalize(ue5m3_shift_out, 1, st));
  return FP4_OK;
}

fp4_status fp4_quantize_rht(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, fp4_scale_fmt f, fp4_rounding r,
                            uint64_t seed, uint32_t rht_mask, const float* global_amax, fp4_sf_layout sfl,
                            uint8_t* codes, uint8_t* scales, float* amax_out, int32_t* dev_status,
                            fp4_stream_t stream) {
  if (r != FP4_ROUND_RNE && r != FP4_ROUND_STOCHASTIC) return FP4_ERR_INVALID_ARG;
  if (rht_mask > 0xFFFFu) return FP4_ERR_INVALID_ARG;
  fp4_status s = check_quant_common(x_bf16, M, K, ldx, (int)f, (int)sfl, M, K);
  if (s != FP4_OK) return s;
  if (f != FP4_SF_E4M3 && f != FP4_SF_UE5M3 && f != FP4_SF_E8M0 && f != FP4_SF_NVINT4 && f != FP4_SF_MXINT4)
    return FP4_ERR_UNSUPPORTED;
  if (M * K > 0 && (s = check_out(codes, scales)) != FP4_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  fp4lib::QuantArgs a{};
  a.mode = fp4lib::QuantArgs::ROWS;
  a.fmt = (int)f;
  a.x = x_bf16;
  a.M = M;
  a.K = K;
  a.ldx = ldx;
  a.mma = sfl == FP4_SFLAYOUT_MMA;
  a.status = dev_status;
  a.row_sr = r == FP4_ROUND_STOCHASTIC;
  a.seed_row = seed;
  a.codes_row = codes;
  a.scales_row = scales;
  a.amax_out = amax_out;
  if (global_amax == nullptr) {
    // fresh: max |x'| of the transformed tensor first
    if (amax_out == nullptr) return FP4_ERR_INVALID_ARG;
    if ((s = cuda_status(fp4lib::launch_amax_rht(x_bf16, M, K, ldx, rht_mask, amax_out, st))) != FP4_OK) return s;
    a.gptr = amax_out;
    a.amax_by_product = false;
  } else {
    a.gptr = global_amax;
    a.amax_by_product = amax_out != nullptr;
    if (a.amax_by_product && (s = cuda_status(cudaMemsetAsync(amax_out, 0, sizeof(float), st))) != FP4_OK) return s;
  }
  return cuda_status(fp4lib::launch_quantize_rht(a, rht_mask, st));
}

fp4_status fp4_quantize_dual_rht(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, fp4_scale_fmt f,
                                 fp4_rounding r_row, uint64_t seed_row, fp4_rounding r_col, uint64_t seed_col,
                                 uint32_t rht_mask, const float* g_row, const float* g_col, fp4_sf_layout sfl,
                                 uint8_t* codes_row, uint8_t* scales_row, uint8_t* codes_col, uint8_t* scales_col,
                                 float* amax_row_out, float* amax_col_out, int32_t* dev_status,
                                 fp4_stream_t stream) {
  if ((r_row != FP4_ROUND_RNE && r_row != FP4_ROUND_STOCHASTIC) ||
      (r_col != FP4_ROUND_RNE && r_col != FP4_ROUND_STOCHASTIC) || rht_mask > 0xFFFFu)
    return FP4_ERR_INVALID_ARG;
  if ((g_row == nullptr) != (g_col == nullptr)) return FP4_ERR_INVALID_ARG;
  if ((amax_row_out == nullptr) != (amax_col_out == nullptr)) return FP4_ERR_INVALID_ARG;
  fp4_status s = check_quant_common(x_bf16, M, K, ldx, (int)f, (int)sfl, M, K);
  if (s != FP4_OK) return s;
  if ((s = check_quant_common(x_bf16, M, K, ldx, (int)f, (int)sfl, K, M)) != FP4_OK) return s;
  if (f != FP4_SF_E4M3 && f != FP4_SF_UE5M3 && f != FP4_SF_E8M0) return FP4_ERR_UNSUPPORTED;
  if (M % 32 != 0 || K % 32 != 0) return FP4_ERR_SHAPE;
  if (M * K > 0) {
    if ((s = check_out(codes_row, scales_row)) != FP4_OK) return s;
    if ((s = check_out(codes_col, scales_col)) != FP4_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  fp4lib::DualRhtArgs a{};
  a.fmt = (int)f;
  a.x = x_bf16;
  a.M = M;
  a.K = K;
  a.ldx = ldx;
  a.mask = rht_mask;
  a.row_sr = r_row == FP4_ROUND_STOCHASTIC;
  a.col_sr = r_col == FP4_ROUND_STOCHASTIC;
  a.mma = sfl == FP4_SFLAYOUT_MMA;
  a.seed_row = seed_row;
  a.seed_col = seed_col;
  a.codes_row = codes_row;
  a.scales_row = scales_row;
  a.codes_col = codes_col;
  a.scales_col = scales_col;
  a.amax_row_out = amax_row_out;
  a.amax_col_out = amax_col_out;
  a.status = dev_status;
  if (g_row == nullptr) {
    // fresh: both transformed amaxes first
    if (amax_row_out == nullptr) return FP4_ERR_INVALID_ARG;
    if ((s = cuda_status(fp4lib::launch_amax_rht(x_bf16, M, K, ldx, rht_mask, amax_row_out, st))) != FP4_OK) return s;
    if ((s = cuda_status(fp4lib::launch_amax_rht_cols(x_bf16, M, K, ldx, rht_mask, amax_col_out, st))) != FP4_OK)
      return s;
    a.g_row = amax_row_out;
    a.g_col = amax_col_out;
    a.amax_by_product = false;
  } else {
    a.g_row = g_row;
    a.g_col = g_col;
    a.amax_by_product = amax_row_out != nullptr;
    if (a.amax_by_product) {
      if ((s = cuda_status(cudaMemsetAsync(amax_row_out, 0, sizeof(float), st))) != FP4_OK) return s;
      if ((s = cuda_status(cudaMemsetAsync(amax_col_out, 0, sizeof(float), st))) != FP4_OK) return s;
    }
  }
  return cuda_status(fp4lib::launch_quantize_dual_rht(a, st));
}

fp4_status fp4_quantize_dual(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, fp4_scale_fmt f,
                             fp4_rounding r_row, uint64_t seed_row, fp4_rounding r_col, uint64_t seed_col,
                             const float* global_amax, fp4_sf_layout sfl, uint8_t* codes_row, uint8_t* scales_row,
                             uint8_t* codes_col, uint8_t* scales_col, float* amax_out, int32_t* ue5m3_shift_out,
                             int32_t* dev_status, fp4_stream_t stream) {
  if ((r_row != FP4_ROUND_RNE && r_row != FP4_ROUND_STOCHASTIC) ||
      (r_col != FP4_ROUND_RNE && r_col != FP4_ROUND_STOCHASTIC))
    return FP4_ERR_INVALID_ARG;
  fp4_status s = check_quant_common(x_bf16, M, K, ldx, (int)f, (int)sfl, M, K);
  if (s != FP4_OK) return s;
  if ((s = check_quant_common(x_bf16, M, K, ldx, (int)f, (int)sfl, K, M)) != FP4_OK) return s;
  if (sweep_fmt((int)f)) return FP4_ERR_UNSUPPORTED;
  if (M % 32 != 0 || K % 32 != 0) return FP4_ERR_SHAPE;
  if (M * K > 0) {
    if ((s = check_out(codes_row, scales_row)) != FP4_OK) return s;
    if ((s = check_out(codes_col, scales_col)) != FP4_OK) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  fp4lib::QuantArgs a{};
  a.mode = fp4lib::QuantArgs::DUAL;
  a.fmt = (int)f;
  a.x = x_bf16;
  a.M = M;
  a.K = K;
  a.ldx = ldx;
  a.mma = sfl == FP4_SFLAYOUT_MMA;
  a.status = dev_status;
  a.row_sr = r_row == FP4_ROUND_STOCHASTIC;
  a.col_sr = r_col == FP4_ROUND_STOCHASTIC;
  a.seed_row = seed_row;
  a.seed_col = seed_col;
  a.codes_row = codes_row;
  a.scales_row = scales_row;
  a.codes_col = codes_col;
  a.scales_col = scales_col;
  if (ue5m3_shift_out != nullptr) {
    a.sf_max_row = reinterpret_cast<uint32_t*>(ue5m3_shift_out);
    a.sf_max_col = reinterpret_cast<uint32_t*>(ue5m3_shift_out + 1);
  }
  if ((s = prepare_shift((int)f, ue5m3_shift_out, 2, st)) != FP4_OK) return s;
  if ((s = prepare_amax(a, global_amax, amax_out, st)) != FP4_OK) return s;
  if ((s = cuda_status(fp4lib::launch_quantize(a, st))) != FP4_OK) return s;
  if (ue5m3_shift_out != nullptr) return cuda_status(fp4lib::launch_ue5m3_finalize(ue5m3_shift_out, 2, st));
  return FP4_OK;
}

fp4_status fp4_dequantize(const uint8_t* codes, const uint8_t* scales, fp4_sf_layout sfl, int64_t M, int64_t K,
                          fp4_scale_fmt f, const float* global_amax, fp4_out_dtype od, void* out,
                          fp4_stream_t stream) {
  if (!valid_fmt((int)f) || (sfl != FP4_SFLAYOUT_PLAIN && sfl != FP4_SFLAYOUT_MMA) ||
      (od != FP4_OUT_F32 && od != FP4_OUT_BF16))
    return FP4_ERR_INVALID_ARG;
  const int G = group_of((int)f);
  if (M < 0 || K < 0 || K % G != 0) return FP4_ERR_SHAPE;
  if (sfl == FP4_SFLAYOUT_MMA && (M % 128 != 0 || (K / G) % 4 != 0)) return FP4_ERR_SHAPE;
  if (M * K == 0) return FP4_OK;
  if (codes == nullptr || scales == nullptr || out == nullptr || global_amax == nullptr) return FP4_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(out)) return FP4_ERR_ALIGNMENT;
  return cuda_status(fp4lib::launch_dequantize(codes, scales, sfl == FP4_SFLAYOUT_MMA, M, K, (int)f, global_amax,
                                               od == FP4_OUT_BF16, out, (cudaStream_t)stream));
}

fp4_status fp4_ue5m3_to_e4m3(const uint8_t* ue5m3_scales, int64_t n, int32_t* t_out, uint8_t* e4m3_out,
                             int32_t* dev_status, fp4_stream_t stream) {
  if (t_out == nullptr || n < 0) return n < 0 ? FP4_ERR_SHAPE : FP4_ERR_INVALID_ARG;
  if (n > 0 && (ue5m3_scales == nullptr || e4m3_out == nullptr)) return FP4_ERR_INVALID_ARG;
  return cuda_status(fp4lib::launch_ue5m3_to_e4m3(ue5m3_scales, n, t_out, e4m3_out, dev_status,
                                                  (cudaStream_t)stream));
}

fp4_status fp4_ue5m3_reencode(const uint8_t* ue5m3_scales, int64_t n, const int32_t* t, uint8_t* e4m3_out,
                              int32_t* dev_status, fp4_stream_t stream) {
  if (n < 0) return FP4_ERR_SHAPE;
  if (t == nullptr || (n > 0 && (ue5m3_scales == nullptr || e4m3_out == nullptr))) return FP4_ERR_INVALID_ARG;
  return cuda_status(fp4lib::launch_ue5m3_reencode(ue5m3_scales, n, t, e4m3_out, dev_status, (cudaStream_t)stream));
}

fp4_status fp4_ue5m3_windows(const uint8_t* ue5m3_scales, int64_t n, int32_t* t_out, int32_t* n_windows_out,
                             uint8_t* e4m3_out, int32_t* dev_status, fp4_stream_t stream) {
  if (n < 0) return FP4_ERR_SHAPE;
  if (t_out == nullptr || n_windows_out == nullptr) return FP4_ERR_INVALID_ARG;
  if (n > 0 && (ue5m3_scales == nullptr || e4m3_out == nullptr)) return FP4_ERR_INVALID_ARG;
  return cuda_status(fp4lib::launch_ue5m3_windows(ue5m3_scales, n, t_out, n_windows_out, e4m3_out, dev_status,
                                                  (cudaStream_t)stream));
}

fp4_status fp4_gemm_ue5m3_windows(const uint8_t* Aq, const uint8_t* As_windows, const int32_t* tA,
                                  const int32_t* nA, const uint8_t* Bq, const uint8_t* Bs_windows,
                                  const int32_t* tB, const int32_t* nB, const float* ga, const float* gb,
                                  int64_t M, int64_t N, int64_t K, float* C, int64_t ldc, int32_t* dev_status,
                                  fp4_stream_t stream) {
  if (Aq == nullptr || As_windows == nullptr || tA == nullptr || nA == nullptr || Bq == nullptr ||
      Bs_windows == nullptr || tB == nullptr || nB == nullptr || ga == nullptr || gb == nullptr || C == nullptr)
    return FP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 != 0 || N % 128 != 0 || K % 256 != 0 || ldc < N) return FP4_ERR_SHAPE;
  if (!aligned16(Aq) || !aligned16(As_windows) || !aligned16(Bq) || !aligned16(Bs_windows) || !aligned16(C) ||
      (ldc * 4) % 16 != 0)
    return FP4_ERR_ALIGNMENT;
  // one window's scale array: M*K/16 (A) or N*K/16 (B) bytes, a multiple of 16
  const int64_t a_win = M * K / 16, b_win = N * K / 16;
  fp4lib::GemmArgs a{};
  a.Aq = Aq;
  a.Bq = Bq;
  a.ga = ga;
  a.gb = gb;
  a.M = M;
  a.N = N;
  a.K = K;
  a.ldc = ldc;
  a.fmt = (int)FP4_SF_UE5M3;
  a.bf16_out = false;
  a.C = C;
  a.status = dev_status;
  a.wcount_a = nA;
  a.wcount_b = nB;
  for (int wa = 0; wa < 3; ++wa) {
    for (int wb = 0; wb < 3; ++wb) {
      a.As = As_windows + wa * a_win;
      a.Bs = Bs_windows + wb * b_win;
      a.tA = tA + wa;
      a.tB = tB + wb;
      a.wa = wa;
      a.wb = wb;
      a.accumulate = wa != 0 || wb != 0;  // window pair (0, 0) always runs and stores C
      const fp4_status s = cuda_status(fp4lib::launch_gemm(a, (cudaStream_t)stream));
      if (s != FP4_OK) return s;
    }
  }
  return FP4_OK;
}

fp4_status fp4_gemm(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs, const float* ga,
                    const float* gb, const int32_t* tA, const int32_t* tB, int64_t M, int64_t N, int64_t K,
                    fp4_scale_fmt f, fp4_gemm_layout layout, fp4_out_dtype od, void* C, int64_t ldc,
                    int32_t* dev_status, fp4_stream_t stream) {
  if (layout != FP4_LAYOUT_TN || (od != FP4_OUT_F32 && od != FP4_OUT_BF16) || !valid_fmt((int)f))
    return FP4_ERR_INVALID_ARG;
  if (f == FP4_SF_E1M6 || sweep_fmt((int)f)) return FP4_ERR_UNSUPPORTED;
  if (Aq == nullptr || As == nullptr || Bq == nullptr || Bs == nullptr || C == nullptr) return FP4_ERR_INVALID_ARG;
  if (f != FP4_SF_E8M0 && (ga == nullptr || gb == nullptr)) return FP4_ERR_INVALID_ARG;
  if (f == FP4_SF_UE5M3 && (tA == nullptr || tB == nullptr)) return FP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 != 0 || N % 128 != 0 || K % 256 != 0 || ldc < N) return FP4_ERR_SHAPE;
  const int64_t esz = od == FP4_OUT_BF16 ? 2 : 4;
  if (!aligned16(Aq) || !aligned16(As) || !aligned16(Bq) || !aligned16(Bs) || !aligned16(C) ||
      (ldc * esz) % 16 != 0)
    return FP4_ERR_ALIGNMENT;
  fp4lib::GemmArgs a{};
  a.Aq = Aq;
  a.As = As;
  a.Bq = Bq;
  a.Bs = Bs;
  a.ga = ga;
  a.gb = gb;
  a.tA = f == FP4_SF_UE5M3 ? tA : nullptr;
  a.tB = f == FP4_SF_UE5M3 ? tB : nullptr;
  a.M = M;
  a.N = N;
  a.K = K;
  a.ldc = ldc;
  a.fmt = (int)f;
  a.bf16_out = od == FP4_OUT_BF16;
  a.C = C;
  a.status = dev_status;
  return cuda_status(fp4lib::launch_gemm(a, (cudaStream_t)stream));
}

namespace {

// fp4_gemm_quantize and its dual form: row blocks (C_codes, C_scales) and/or
// column blocks (Ct_codes, Ct_scales) of bf16(C).
fp4_status gemm_quantize(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                         const float* ga, const float* gb, const int32_t* tA, const int32_t* tB, int64_t M,
                         int64_t N, int64_t K, fp4_scale_fmt f, fp4_gemm_layout layout, const float* g_out,
                         fp4_rounding r_row, uint64_t seed_row, fp4_rounding r_col, uint64_t seed_col,
                         fp4_sf_layout sfl_out, uint8_t* C_codes, uint8_t* C_scales, uint8_t* Ct_codes,
                         uint8_t* Ct_scales, float* C_amax_out, int32_t* dev_status, fp4_stream_t stream) {
  if (layout != FP4_LAYOUT_TN || !valid_fmt((int)f)) return FP4_ERR_INVALID_ARG;
  if (r_row != FP4_ROUND_RNE && r_row != FP4_ROUND_STOCHASTIC) return FP4_ERR_INVALID_ARG;
  if (r_col != FP4_ROUND_RNE && r_col != FP4_ROUND_STOCHASTIC) return FP4_ERR_INVALID_ARG;
  if (sfl_out != FP4_SFLAYOUT_PLAIN && sfl_out != FP4_SFLAYOUT_MMA) return FP4_ERR_INVALID_ARG;
  if (f == FP4_SF_E1M6 || sweep_fmt((int)f)) return FP4_ERR_UNSUPPORTED;
  if (Aq == nullptr || As == nullptr || Bq == nullptr || Bs == nullptr || g_out == nullptr)
    return FP4_ERR_INVALID_ARG;
  // each output is a pair of buffers, given together; at least one pair
  if ((C_codes == nullptr) != (C_scales == nullptr) || (Ct_codes == nullptr) != (Ct_scales == nullptr) ||
      (C_codes == nullptr && Ct_codes == nullptr))
    return FP4_ERR_INVALID_ARG;
  if (f != FP4_SF_E8M0 && (ga == nullptr || gb == nullptr)) return FP4_ERR_INVALID_ARG;
  if (f == FP4_SF_UE5M3 && (tA == nullptr || tB == nullptr)) return FP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 != 0 || N % 128 != 0 || K % 256 != 0) return FP4_ERR_SHAPE;
  if (M % 256 != 0) return FP4_ERR_UNSUPPORTED;  // the quantizing epilogue runs on CTA pairs
  if (!aligned16(Aq) || !aligned16(As) || !aligned16(Bq) || !aligned16(Bs) || !aligned16(C_codes) ||
      !aligned16(C_scales) || !aligned16(Ct_codes) || !aligned16(Ct_scales))
    return FP4_ERR_ALIGNMENT;
  cudaStream_t st = (cudaStream_t)stream;
  if (C_amax_out != nullptr) {
    fp4_status s = cuda_status(cudaMemsetAsync(C_amax_out, 0, sizeof(float), st));
    if (s != FP4_OK) return s;
  }
  fp4lib::GemmArgs a{};
  a.Aq = Aq;
  a.As = As;
  a.Bq = Bq;
  a.Bs = Bs;
  a.ga = ga;
  a.gb = gb;
  a.tA = f == FP4_SF_UE5M3 ? tA : nullptr;
  a.tB = f == FP4_SF_UE5M3 ? tB : nullptr;
  a.M = M;
  a.N = N;
  a.K = K;
  a.ldc = N;
  a.fmt = (int)f;
  a.bf16_out = true;
  a.status = dev_status;
  a.qout = true;
  a.q_codes = C_codes;
  a.q_scales = C_scales;
  a.q_g = g_out;
  a.q_amax_out = C_amax_out;
  a.q_seed = seed_row;
  a.q_sr = r_row == FP4_ROUND_STOCHASTIC;
  a.q_mma = sfl_out == FP4_SFLAYOUT_MMA;
  a.qt_codes = Ct_codes;
  a.qt_scales = Ct_scales;
  a.qt_seed = seed_col;
  a.qt_sr = r_col == FP4_ROUND_STOCHASTIC;
  return cuda_status(fp4lib::launch_gemm(a, st));
}

}  // namespace

fp4_status fp4_gemm_quantize(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                             const float* ga, const float* gb, const int32_t* tA, const int32_t* tB, int64_t M,
                             int64_t N, int64_t K, fp4_scale_fmt f, fp4_gemm_layout layout, const float* g_out,
                             fp4_rounding r_out, uint64_t seed_out, fp4_sf_layout sfl_out, uint8_t* C_codes,
                             uint8_t* C_scales, float* C_amax_out, int32_t* dev_status, fp4_stream_t stream) {
  if (C_codes == nullptr || C_scales == nullptr) return FP4_ERR_INVALID_ARG;
  return gemm_quantize(Aq, As, Bq, Bs, ga, gb, tA, tB, M, N, K, f, layout, g_out, r_out, seed_out, FP4_ROUND_RNE, 0,
                       sfl_out, C_codes, C_scales, nullptr, nullptr, C_amax_out, dev_status, stream);
}

fp4_status fp4_gemm_quantize_dual(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                                  const float* ga, const float* gb, const int32_t* tA, const int32_t* tB,
                                  int64_t M, int64_t N, int64_t K, fp4_scale_fmt f, fp4_gemm_layout layout,
                                  const float* g_out, fp4_rounding r_row, uint64_t seed_row, fp4_rounding r_col,
                                  uint64_t seed_col, fp4_sf_layout sfl_out, uint8_t* C_codes, uint8_t* C_scales,
                                  uint8_t* Ct_codes, uint8_t* Ct_scales, float* C_amax_out, int32_t* dev_status,
                                  fp4_stream_t stream) {
  return gemm_quantize(Aq, As, Bq, Bs, ga, gb, tA, tB, M, N, K, f, layout, g_out, r_row, seed_row, r_col, seed_col,
                       sfl_out, C_codes, C_scales, Ct_codes, Ct_scales, C_amax_out, dev_status, stream);
}

fp4_status fp4_gemv_w4a16(const uint8_t* Wq, const uint8_t* Ws, const float* gw, const void* x_bf16,
                          int64_t batch, int64_t N, int64_t K, fp4_out_dtype od, void* y, int32_t* dev_status,
                          fp4_stream_t stream) {
  if (od != FP4_OUT_F32 && od != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
  if (Wq == nullptr || Ws == nullptr || gw == nullptr || x_bf16 == nullptr || y == nullptr)
    return FP4_ERR_INVALID_ARG;
  if (batch < 1 || batch > 64 || N <= 0 || K <= 0 || K % 32 != 0) return FP4_ERR_SHAPE;
  if (!aligned16(Wq) || !aligned16(Ws) || !aligned16(x_bf16) || !aligned16(y)) return FP4_ERR_ALIGNMENT;
  fp4lib::GemvArgs a{};
  a.Wq = Wq;
  a.Ws = Ws;
  a.gw = gw;
  a.x = x_bf16;
  a.batch = batch;
  a.N = N;
  a.K = K;
  a.bf16_out = od == FP4_OUT_BF16;
  a.y = y;
  a.status = dev_status;
  return cuda_status(fp4lib::launch_gemv(a, (cudaStream_t)stream));
}

fp4_status fp4_encode_scales(const float* s, int64_t n, fp4_scale_fmt f, uint8_t* codes, float* decoded,
                             fp4_stream_t stream) {
  if (!valid_fmt((int)f)) return FP4_ERR_INVALID_ARG;
  if (n < 0) return FP4_ERR_SHAPE;
  if (n > 0 && (s == nullptr || codes == nullptr || decoded == nullptr)) return FP4_ERR_INVALID_ARG;
  return cuda_status(fp4lib::launch_encode_scales(s, n, (int)f, codes, decoded, (cudaStream_t)stream));
}

fp4_status fp4_philox_bits16(uint64_t seed, uint64_t start, int64_t n, uint16_t* out, fp4_stream_t stream) {
  if (n < 0) return FP4_ERR_SHAPE;
  if (n > 0 && out == nullptr) return FP4_ERR_INVALID_ARG;
  return cuda_status(fp4lib::launch_philox_bits16(seed, start, n, out, (cudaStream_t)stream));
}

const char* fp4_status_string(fp4_status s) {
  switch (s) {
    case FP4_OK: return "ok";
    case FP4_ERR_INVALID_ARG: return "invalid argument (NULL pointer or bad enum)";
    case FP4_ERR_SHAPE: return "unsupported shape";
    case FP4_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
    case FP4_ERR_UNSUPPORTED: return "combination not supported";
    case FP4_ERR_NONFINITE: return "stored global amax is not finite";
    case FP4_ERR_UE5M3_RANGE: return "UE5M3 scale not exact on the shifted E4M3 path";
    case FP4_ERR_TIMEOUT: return "bounded device wait expired";
    case FP4_ERR_CUDA: return "CUDA runtime error (see fp4_last_cuda_error)";
    default: return "unknown status";
  }
}

int fp4_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
