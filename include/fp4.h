/*
 * fp4.h -- C ABI of libfp4.so: the FP4 block-scaled linear-layer hot path on
 * GB300 (sm_103a).
 *
 * Sources of the method (web pages, cited by title and section):
 *   [NVFP4/MX]  "NVFP4 vs MXFP" post, quant_prune_distill #486, section "Метод":
 *               small groups sharing a low-precision scale; NVFP4 = FP4 E2M1,
 *               group 16, E4M3 scale (4.5 bits/param); MXFP4 = group 32, E8M0
 *               power-of-two scale (4.25 bits/param); scale handling done by an
 *               efficient kernel.
 *   [FP4-REV]   review of Intel's FP4 training paper, gonzo_ML #3986, sections
 *               "Форматы FP4" (group 16, scale formats E1M6..E8M0) and
 *               "Стохастическая квантизация" (nearest rounding forward,
 *               stochastic rounding backward).
 *   [UE5M3]     "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining"
 *               (rit.work blog), sections "Что сделали" (unsigned 5+3-bit scale
 *               per 16 elements, tensor maximum refreshed every 50 steps,
 *               stochastic rounding on backward gradients, all linears in FP4)
 *               and "Ограничения" (UE5M3 run by software emulation).
 *   [W4A16]     weight-only NVFP4 post, quant_prune_distill #574, sections
 *               "Метод" (weights only, activations untouched) and
 *               "Эксперименты" (memory-bound kernel for small batches).
 *   [INT-FP]    post on "INT v.s. FP: A Comprehensive Study of Fine-Grained
 *               Low-bit Quantization Formats" (quant_prune_distill channel page),
 *               section "Метод": MXINT4 / NVINT4 beside MXFP4 / NVFP4, the same
 *               groups and scales on an INT grid.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or synchronizes.  Every call is asynchronous on
 *     `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Matrices are row-major; `ld*` arguments are leading dimensions in
 *     elements.  bf16 is IEEE bfloat16 (2 bytes).
 *   - Argument errors are detected on the host before anything is launched and
 *     returned as an fp4_status; nothing is launched then.  A failed launch
 *     returns FP4_ERR_CUDA and fp4_last_cuda_error() gives the cudaError_t.
 *   - Conditions only the device can see (a non-finite stored amax, a UE5M3
 *     scale that the E4M3 emulation cannot hold exactly, an expired bounded
 *     wait) are written to the optional device word `dev_status` (the first
 *     non-zero fp4_status wins; the caller zeroes it).  No kernel traps.
 *   - Packed codes: byte j of a row holds element 2j in its low nibble and
 *     element 2j+1 in its high nibble; bit 3 of a nibble is the sign.
 *   - Scales: one byte per block.  FP4_SFLAYOUT_PLAIN is row-major
 *     [rows, cols/G].  FP4_SFLAYOUT_MMA is the tiled layout the GEMM reads:
 *     for scale (r, b) of a matrix with nb = cols/G blocks per row (nb % 4 ==
 *     0, rows % 128 == 0), byte offset
 *       ((r/128) * (nb/4) + b/4) * 512 + (r%32)*16 + ((r/32)%4)*4 + b%4.
 */
#ifndef FP4_H
#define FP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp4_stream_t; /* same type as cudaStream_t */

typedef enum {
  FP4_OK = 0,
  FP4_ERR_INVALID_ARG = 1, /* NULL pointer or bad enum value */
  FP4_ERR_SHAPE = 2,       /* sizes not supported (see each call) */
  FP4_ERR_ALIGNMENT = 3,   /* a pointer or leading dimension not 16-byte aligned */
  FP4_ERR_UNSUPPORTED = 4, /* valid but not implemented combination */
  FP4_ERR_NONFINITE = 5,   /* device: stored global amax is Inf or NaN */
  FP4_ERR_UE5M3_RANGE = 6, /* device: a UE5M3 scale is not exact on the E4M3 path */
  FP4_ERR_TIMEOUT = 7,     /* device: a bounded wait expired; outputs invalid */
  FP4_ERR_CUDA = 8         /* a CUDA runtime call failed; see fp4_last_cuda_error() */
} fp4_status;

/* Block-scale formats.  G = elements per block. */
typedef enum {
  FP4_SF_E4M3 = 0,  /* NVFP4: E4M3 (bias 7, max 448), G = 16   [NVFP4/MX] */
  FP4_SF_UE5M3 = 1, /* unsigned 5+3 bits (bias 15, max 114688), G = 16   [UE5M3] */
  FP4_SF_E8M0 = 2,  /* MXFP4: 2^(c-127), G = 32, no global scale   [NVFP4/MX] */
  FP4_SF_E1M6 = 3,  /* narrowest format of the sweep (max 3.96875), G = 16;
                       quantizer only, no GEMM   [FP4-REV "Форматы FP4"] */
  /* The rest of the group-16 scale-format sweep of [FP4-REV] "Форматы FP4":
   * signed ExMy scales with bias 2^(E-1)-1, IEEE-style subnormals and no NaN
   * (only their non-negative codes occur).  Row quantization (fp4_quantize
   * with transpose = 0), fp4_dequantize and fp4_encode_scales only; every
   * other call returns FP4_ERR_UNSUPPORTED for them. */
  FP4_SF_E2M5 = 4,  /* max 7.875 */
  FP4_SF_E3M4 = 5,  /* max 31 */
  FP4_SF_E5M2 = 6,  /* max 114688 */
  FP4_SF_E6M1 = 7,  /* max 1.5 * 2^32 */
  FP4_SF_E7M0 = 8,  /* max 2^64 */
  /* INT4 element grid instead of E2M1 ([INT-FP] "Метод": NV = groups of 16
   * with E4M3 scales, MX = groups of 32 with E8M0 scales): elements are the
   * integers -7..7 stored as two's-complement nibbles; every 6 of the E2M1
   * method becomes 7 (s_enc = f32(f32(7*448)/g), s_real = f32(f32(a_b/7)*s_enc),
   * E8M0 exponent floor(log2 a_b) - 2); RNE ties to even, SR as for E2M1.
   * Row quantization, fp4_dequantize and fp4_encode_scales only. */
  FP4_SF_NVINT4 = 9,
  FP4_SF_MXINT4 = 10
} fp4_scale_fmt;

typedef enum {
  FP4_ROUND_RNE = 0,       /* nearest, ties to even code, saturate at 6 */
  FP4_ROUND_STOCHASTIC = 1 /* Philox4x32-10 16-bit draws   [FP4-REV] */
} fp4_rounding;

typedef enum { FP4_SFLAYOUT_PLAIN = 0, FP4_SFLAYOUT_MMA = 1 } fp4_sf_layout;
typedef enum { FP4_OUT_F32 = 0, FP4_OUT_BF16 = 1 } fp4_out_dtype;
typedef enum { FP4_LAYOUT_TN = 0 /* A[M,K], B[N,K], both K-contiguous; C[M,N] */ } fp4_gemm_layout;

/* Elements per block of a scale format (16 or 32); 0 for an unknown format. */
int fp4_group_size(fp4_scale_fmt f);

/* Bytes of packed codes (rows*cols/2) and of scales (rows*cols/G) of an
 * [rows, cols] tensor: 4.5 bits/param for NVFP4, 4.25 for MXFP4 [NVFP4/MX].
 * FP4_ERR_SHAPE unless cols % G == 0 and rows, cols >= 0. */
fp4_status fp4_storage_bytes(int64_t rows, int64_t cols, fp4_scale_fmt f,
                             size_t* code_bytes, size_t* scale_bytes);

/* Global amax g = max |x| of a bf16 [M, K] matrix (leading dimension ldx)
 * into the device float *amax_out (overwritten; 0 for an empty matrix).
 * The per-tensor amax of [UE5M3] "Что сделали"; a caller that refreshes it
 * only every 50 steps calls this on refresh steps only. */
fp4_status fp4_amax(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                    float* amax_out, fp4_stream_t stream);

/* fp4_amax of n tensors (1 <= n <= 8; n == 0 does nothing) in one launch:
 * x_bf16[i], M[i], K[i], ldx[i] are HOST arrays describing tensor i (device
 * pointers, the same requirements as fp4_amax each), and amax_out[i] (device
 * float[n]) receives max |x_i|.  One launch for the several fresh amaxes a
 * step needs, instead of one short launch per tensor. */
fp4_status fp4_amax_n(int n, const void* const* x_bf16, const int64_t* M, const int64_t* K,
                      const int64_t* ldx, float* amax_out, fp4_stream_t stream);

/* Quantize a bf16 [M, K] matrix to FP4 codes plus block scales.
 * Method ([NVFP4/MX] "Метод", [UE5M3] "Что сделали", [FP4-REV]
 * "Стохастическая квантизация"), all float32 steps correctly rounded:
 *   s_enc = f32(f32(6*S_T) / g), S_T = 448 (E4M3, UE5M3), otherwise the
 *           scale format's largest finite value (3.96875 for E1M6);
 *           g == 0 -> 1, overflow -> FLT_MAX; E8M0: s_enc = 1;
 *   per block of G elements along K: a_b = max|x|;
 *           s_b = decode(encode_rne_sat(f32(f32(a_b/6) * s_enc)));
 *           E8M0: code = clamp(floor(log2 a_b) - 2 + 127, 0, 254);
 *   per element: y = f32(x * f32(s_enc / s_b)) (0 when s_b == 0), rounded to
 *           E2M1 by RNE or stochastically (16 Philox bits r, up iff
 *           r < 65536*(|y|-lo)/(hi-lo)); sign bit copied from x.
 *   Philox: key = seed, counter = (i/8, 0, 0) with i the element's row-major
 *           index in the OUTPUT layout, word (i/2)%4, half i%2.
 * transpose = 0: codes [M, K/2], scales per row along K.
 * transpose = 1: the result equals quantizing x^T: codes [K, M/2], blocks of
 *           G along the original rows (so dgrad/wgrad reduce over blocks).
 * global_amax: device float, the stored g (possibly stale); NULL computes a
 *           fresh g first and then requires amax_out (which receives it).
 * amax_out: nullable device float; receives max|x| of this call (the value a
 *           refresh would store).
 * ue5m3_shift_out: nullable device int32, f = UE5M3 only (other formats:
 *           FP4_ERR_UNSUPPORTED); receives t = e_max - 7 of this call's
 *           scales, e_max the largest unbiased exponent among them (0 when
 *           all are zero): the shift fp4_ue5m3_reencode and fp4_gemm take
 *           for the E4M3 tensor-core emulation ([UE5M3] "Ограничения"),
 *           found while the scales are made instead of by a second pass.
 * Requirements: M, K >= 0; the blocked dimension a multiple of G; x, codes,
 * scales 16-byte aligned and ldx*2 a multiple of 16; for transpose = 1 also
 * M % 32 == 0 and K % 32 == 0; FP4_SFLAYOUT_MMA needs the output rows % 128 == 0
 * and blocks per row % 4 == 0. */
fp4_status fp4_quantize(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                        fp4_scale_fmt f, fp4_rounding r, uint64_t seed,
                        const float* global_amax, int transpose, fp4_sf_layout sfl,
                        uint8_t* codes, uint8_t* scales, float* amax_out,
                        int32_t* ue5m3_shift_out, int32_t* dev_status, fp4_stream_t stream);

/* fp4_quantize (row layout) of the 16 x 16 random Hadamard transform of x:
 * every 16-element block along K first becomes x' = 1/4 * H16 * (s . x), H16
 * the Sylvester Hadamard matrix (H[i][j] = (-1)^popcount(i & j)), s[j] = -1
 * iff bit j of rht_mask is set, computed in float32 by the fast Walsh-Hadamard
 * butterflies (h = 1, 2, 4, 8: (a, b) -> (a + b, a - b)) and the exact 1/4;
 * the method then runs on x' (block amax, scale, rounding; the global amax g
 * is max |x'|, fresh when global_amax is NULL).  The transform is orthogonal:
 * two operands transformed with the same mask along K keep their product, so
 * fp4_gemm of such operands approximates x * w^T.  ([UE5M3] "Что сделали":
 * the randomized transform that spreads outliers, dropped from the UE5M3
 * recipe; [INT-FP] "Метод": Hadamard rotations before MX/NV FP or INT
 * quantization.)  Formats: E4M3, UE5M3, E8M0, NVINT4, MXINT4 (others:
 * FP4_ERR_UNSUPPORTED).  rht_mask < 2^16.  Other arguments and requirements
 * as fp4_quantize with transpose = 0. */
fp4_status fp4_quantize_rht(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                            fp4_scale_fmt f, fp4_rounding r, uint64_t seed, uint32_t rht_mask,
                            const float* global_amax, fp4_sf_layout sfl,
                            uint8_t* codes, uint8_t* scales, float* amax_out,
                            int32_t* dev_status, fp4_stream_t stream);

/* Row and transposed quantization with the 16 x 16 random Hadamard transform
 * of fp4_quantize_rht, from one read: the row output transforms 16-element
 * blocks along K, the transposed output (blocks along the original rows)
 * 16-row blocks along M, so fwd, dgrad and wgrad operands all see the
 * transform along their reduction dimension.  The two transformed tensors
 * have their own global amax: g_row / g_col (device floats, both or neither;
 * NULL computes both fresh, which then requires amax_row_out / amax_col_out),
 * and amax_row_out / amax_col_out (both or neither) receive this call's
 * max |x'| of each.  Formats E4M3, UE5M3, E8M0.  Needs M % 32 == 0 and
 * K % 32 == 0 besides fp4_quantize_dual's requirements. */
fp4_status fp4_quantize_dual_rht(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                 fp4_scale_fmt f, fp4_rounding r_row, uint64_t seed_row,
                                 fp4_rounding r_col, uint64_t seed_col, uint32_t rht_mask,
                                 const float* g_row, const float* g_col, fp4_sf_layout sfl,
                                 uint8_t* codes_row, uint8_t* scales_row,
                                 uint8_t* codes_col, uint8_t* scales_col,
                                 float* amax_row_out, float* amax_col_out,
                                 int32_t* dev_status, fp4_stream_t stream);

/* Row and transposed quantization of one bf16 [M, K] matrix from a single
 * read: writes exactly what fp4_quantize(transpose=0, r_row, seed_row) and
 * fp4_quantize(transpose=1, r_col, seed_col) would, with the same global amax.
 * ue5m3_shift_out: nullable device int32[2] (UE5M3 only): the shifts t of the
 * row and of the transposed scales, as fp4_quantize defines them.
 * Needs M % 32 == 0 and K % 32 == 0 besides fp4_quantize's requirements. */
fp4_status fp4_quantize_dual(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                             fp4_scale_fmt f, fp4_rounding r_row, uint64_t seed_row,
                             fp4_rounding r_col, uint64_t seed_col,
                             const float* global_amax, fp4_sf_layout sfl,
                             uint8_t* codes_row, uint8_t* scales_row,
                             uint8_t* codes_col, uint8_t* scales_col,
                             float* amax_out, int32_t* ue5m3_shift_out,
                             int32_t* dev_status, fp4_stream_t stream);

/* Dequantize codes + scales of an [M, K] tensor (blocks along K):
 * out = f32(f32(e2m1 * s_b) / s_enc) with s_enc from *global_amax as in
 * fp4_quantize; bf16 output is that float32 rounded to nearest even. */
fp4_status fp4_dequantize(const uint8_t* codes, const uint8_t* scales, fp4_sf_layout sfl,
                          int64_t M, int64_t K, fp4_scale_fmt f, const float* global_amax,
                          fp4_out_dtype od, void* out, fp4_stream_t stream);

/* UE5M3 on the E4M3 tensor-core scale path ([UE5M3] "Ограничения": UE5M3 ran
 * by software emulation).  For n UE5M3 scale codes: t = e_max - 7, with e_max
 * the largest unbiased exponent among the scale values (t = 0 if all are 0),
 * written to the device int *t_out; each scale s becomes the E4M3 code of
 * s * 2^-t in e4m3_out (same layout as the input).  A scale that is not exact
 * after the shift is encoded to nearest and raises FP4_ERR_UE5M3_RANGE in
 * dev_status.  fp4_gemm then multiplies its result by 2^(tA + tB). */
fp4_status fp4_ue5m3_to_e4m3(const uint8_t* ue5m3_scales, int64_t n, int32_t* t_out,
                             uint8_t* e4m3_out, int32_t* dev_status, fp4_stream_t stream);

/* fp4_ue5m3_to_e4m3 with the shift already known (the ue5m3_shift_out of
 * fp4_quantize / fp4_quantize_dual, device int *t): one pass over the n
 * scales, each written as the E4M3 code of s * 2^-t; a scale that is not
 * exact after the shift is encoded to nearest and raises FP4_ERR_UE5M3_RANGE
 * in dev_status. */
fp4_status fp4_ue5m3_reencode(const uint8_t* ue5m3_scales, int64_t n, const int32_t* t,
                              uint8_t* e4m3_out, int32_t* dev_status, fp4_stream_t stream);

/* UE5M3 scales wider than one E4M3 window (the same emulation, [UE5M3]
 * "Ограничения").  With e(s) = floor(log2 s) for each nonzero scale value and
 * e_max the largest: scale s belongs to window w = floor((e_max - e(s)) / 14)
 * and becomes the E4M3 code of s * 2^-t_w, t_w = e_max - 7 - 14 w, which is
 * always exact (e(s) - t_w lies in -6..7).  UE5M3 spans 2^-17 .. 1.75 * 2^16,
 * so three windows suffice.  Writes, for n scale codes (any layout):
 *   e4m3_out      3 arrays of n codes, window-major (code 0 where a scale
 *                 belongs to another window), caller-owned device memory;
 *   t_out         device int32[3], the shifts t_0, t_1, t_2;
 *   n_windows_out device int32[1], the windows in use (1 if all scales are 0).
 * Window 0 equals fp4_ue5m3_to_e4m3's output whenever that one is exact. */
fp4_status fp4_ue5m3_windows(const uint8_t* ue5m3_scales, int64_t n, int32_t* t_out,
                             int32_t* n_windows_out, uint8_t* e4m3_out, int32_t* dev_status,
                             fp4_stream_t stream);

/* UE5M3 GEMM over windowed scales: C = sum over window pairs (wa, wb) of the
 * fp4_gemm (f = UE5M3, float32 out) of A with window wa's scales and B with
 * window wb's, shifted by tA[wa], tB[wb].  Pair (0, 0) stores C; every other
 * pair adds its result into C (TMA reduce-add) or, when wa >= *nA or
 * wb >= *nB (device counts from fp4_ue5m3_windows), exits at once, so the host
 * never reads the counts.  Nine launches on the stream.  As_windows /
 * Bs_windows: fp4_ue5m3_windows outputs for A's and B's MMA-layout scales
 * (3 x M*K/16 and 3 x N*K/16 bytes).  C is float32 [M, N], ldc elements; the
 * sum of passes adds one float32 rounding per pass in use.  Shape and
 * alignment rules as fp4_gemm. */
fp4_status fp4_gemm_ue5m3_windows(const uint8_t* Aq, const uint8_t* As_windows, const int32_t* tA,
                                  const int32_t* nA, const uint8_t* Bq, const uint8_t* Bs_windows,
                                  const int32_t* tB, const int32_t* nB, const float* ga,
                                  const float* gb, int64_t M, int64_t N, int64_t K, float* C,
                                  int64_t ldc, int32_t* dev_status, fp4_stream_t stream);

/* Block-scaled FP4 GEMM (forward, dgrad and wgrad are all this call in TN form),
 * float32 accumulation on tcgen05 tensor cores:
 *   C[m, n] = alpha * sum_k (qa[m,k] * sa[m, k/G]) * (qb[n,k] * sb[n, k/G]),
 *   alpha = f32(1 / f32(s_encA * s_encB)) * 2^(tA + tB),
 * with s_enc derived from the device floats *ga, *gb exactly as the quantizer
 * does (E8M0: alpha = 1) [NVFP4/MX], [UE5M3].
 * Aq [M, K/2], Bq [N, K/2] packed codes; As, Bs scales in FP4_SFLAYOUT_MMA.
 * f = E4M3 or E8M0; f = UE5M3 takes the E4M3 scales and shifts produced by
 * fp4_ue5m3_to_e4m3 (tA, tB device ints, required; NULL for other formats).
 * C: float32 or bf16 [M, N] with leading dimension ldc (elements).
 * Requirements: M % 128 == 0, N % 128 == 0, K % 256 == 0, all > 0; pointers
 * 16-byte aligned; ldc * element size a multiple of 16.  (Output tiles are
 * 256 columns wide; with N % 256 == 128 the last tile's upper half reads
 * zero-filled code rows and stores nothing.) */
fp4_status fp4_gemm(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                    const float* ga, const float* gb, const int32_t* tA, const int32_t* tB,
                    int64_t M, int64_t N, int64_t K, fp4_scale_fmt f, fp4_gemm_layout layout,
                    fp4_out_dtype od, void* C, int64_t ldc, int32_t* dev_status,
                    fp4_stream_t stream);

/* fp4_gemm with its output quantized in the epilogue instead of stored:
 * writes exactly what fp4_quantize(bf16(C), FP4_SF_E4M3, r_out, seed_out,
 * g_out, transpose = 0, sfl_out) would make of the bf16 result of fp4_gemm
 * with the same operands, i.e. NVFP4 codes [M, N/2] and E4M3 scales of
 * 16-element blocks along N (Philox indices row * N + col), without the
 * bf16 C in memory.  Quantizing the next layer's input where it is produced
 * needs the stored global amax of C (g_out, device float), the recipe of
 * [UE5M3] "Что сделали" (tensor maximum refreshed every 50 steps, the stored
 * value used in between); C_amax_out (nullable device float) receives
 * max |bf16(C)| for the next refresh.  Requirements as fp4_gemm, and M % 256
 * == 0 (the epilogue runs on the CTA-pair kernel; FP4_ERR_UNSUPPORTED
 * otherwise). */
fp4_status fp4_gemm_quantize(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                             const float* ga, const float* gb, const int32_t* tA, const int32_t* tB,
                             int64_t M, int64_t N, int64_t K, fp4_scale_fmt f, fp4_gemm_layout layout,
                             const float* g_out, fp4_rounding r_out, uint64_t seed_out,
                             fp4_sf_layout sfl_out, uint8_t* C_codes, uint8_t* C_scales,
                             float* C_amax_out, int32_t* dev_status, fp4_stream_t stream);

/* fp4_gemm_quantize with both quantized layouts of C from the one GEMM: row
 * blocks (16 elements along N: codes [M, N/2], what fp4_quantize(bf16(C),
 * transpose = 0, r_row, seed_row) makes) and column blocks (16 elements along
 * M, the layout of C^T: codes [N, M/2], E4M3 scales of (n, m/16), Philox
 * indices n * M + m: what fp4_quantize(bf16(C), transpose = 1, r_col,
 * seed_col) makes), under the one stored global amax g_out, as
 * fp4_quantize_dual defines them.  The column layout is the operand the
 * backward pass needs along M (the next layer's wgrad takes X^T; dgrad's
 * output dX feeds the previous layer's wgrad as dX^T): [UE5M3] "Что
 * сделали" runs every linear in FP4 forward and backward.  Either pair of
 * outputs may be NULL (both pointers of a pair together), not both;
 * C_amax_out as fp4_gemm_quantize.  Requirements as fp4_gemm_quantize. */
fp4_status fp4_gemm_quantize_dual(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                                  const float* ga, const float* gb, const int32_t* tA, const int32_t* tB,
                                  int64_t M, int64_t N, int64_t K, fp4_scale_fmt f, fp4_gemm_layout layout,
                                  const float* g_out, fp4_rounding r_row, uint64_t seed_row,
                                  fp4_rounding r_col, uint64_t seed_col, fp4_sf_layout sfl_out,
                                  uint8_t* C_codes, uint8_t* C_scales, uint8_t* Ct_codes, uint8_t* Ct_scales,
                                  float* C_amax_out, int32_t* dev_status, fp4_stream_t stream);

/* Weight-only NVFP4 linear ([W4A16] "Метод"): y[b, n] = sum_k deq(W)[n, k] * x[b, k],
 * deq(W) = e2m1 * s_b / s_enc(*gw) (E4M3 scales, G = 16, FP4_SFLAYOUT_PLAIN),
 * x bf16 [batch, K] (row stride K), float32 accumulation, y [batch, N] float32
 * or bf16 (row stride N).  Requirements: 1 <= batch <= 64, N > 0, K % 32 == 0,
 * pointers 16-byte aligned.  K % 256 == 0 streams W through shared memory
 * with TMA: batches up to 8 on mma.sync, 9..64 on tcgen05 with the expanded
 * weights in tensor memory, a long K split over a thread-block cluster whose
 * CTAs add their partial sums in a fixed order (the result does not depend on
 * timing).  Its waits are bounded and a wait that expires records
 * FP4_ERR_TIMEOUT in *dev_status (optional int32 device word, first error
 * wins). */
fp4_status fp4_gemv_w4a16(const uint8_t* Wq, const uint8_t* Ws, const float* gw,
                          const void* x_bf16, int64_t batch, int64_t N, int64_t K,
                          fp4_out_dtype od, void* y, int32_t* dev_status, fp4_stream_t stream);

/* Conformance helpers (same device code paths as the quantizer):
 * fp4_encode_scales: n non-negative floats -> scale codes of format f and
 *   their decoded float values (encode as in fp4_quantize's block-scale step;
 *   E8M0 takes the values as block amaxes a_b). */
fp4_status fp4_encode_scales(const float* s, int64_t n, fp4_scale_fmt f,
                             uint8_t* codes, float* decoded, fp4_stream_t stream);

/* fp4_philox_bits16: the 16-bit stochastic-rounding draws of output indices
 *   start .. start+n-1 for `seed` (uint16 device array of n). */
fp4_status fp4_philox_bits16(uint64_t seed, uint64_t start, int64_t n, uint16_t* out,
                             fp4_stream_t stream);

const char* fp4_status_string(fp4_status s);
int fp4_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FP4_H */
