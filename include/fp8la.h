/*
 * fp8la.h -- C ABI of the GB300 (sm_103a) FP8 E4M3 quantize + scaled GEMM
 * library (libfp8la.so).
 *
 * Sources cited below (the three web pages the method comes from):
 *   [P1] "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核"
 *        (blog.hotdry.top, 2025-10-03) -- FP8 GEMM: kernel-code paragraph,
 *        scale paragraph ("此内核借鉴 CUTLASS"), optimisation parameter list
 *        ("优化参数清单"), risks paragraph ("风险考虑").
 *   [P3] "JAX 中使用 Triton 优化 Blackwell GPU 的 FP8 GEMM 内核：TMA 异步加载与
 *        Warp 级原语" (blog.hotdry.top, 2025-10-07) -- warp-specialisation
 *        paragraph ("Warp 级原语"), implementation/MoE paragraph
 *        ("要落地这些优化").
 *   [FP8] Micikevicius et al., "FP8 Formats for Deep Learning" (2022): the
 *        E4M3 encoding (bias 7, max 448, NaN = S.1111.111, no infinity).
 *
 * Conventions shared by every entry point
 *   - All data pointers are DEVICE pointers on the current CUDA device, owned
 *     by the caller.  The library allocates nothing per call and keeps no
 *     per-call state; it launches its kernels on `stream` and never
 *     synchronises (except fp8_get_device_status).  NULL `stream` means the
 *     legacy default stream.
 *   - Sizes and leading dimensions are element counts (int64).  Matrices are
 *     row-major with the given leading dimension.
 *   - E4M3 codes are stored one per byte (uint8_t).  BF16 outputs are stored
 *     as their 16-bit patterns (uint16_t).
 *   - Arguments are validated on the host before anything is launched; on an
 *     error nothing is launched and a negative fp8la_status is returned.  A
 *     failed launch returns FP8LA_ERR_CUDA.  Nothing crosses the ABI as an
 *     exception, and no kernel traps.
 *   - The first call of an entry point on a device does one-time set-up
 *     (kernel attributes, occupancy queries); make it before capturing a
 *     stream into a CUDA graph.  Later calls touch no CUDA runtime state
 *     beyond their launches, so they can be captured.
 *   - fp8_gemm launches with programmatic stream serialization: its set-up
 *     (barriers, tensor memory) may overlap the previous kernel in the
 *     stream, and it waits for that kernel to finish before reading any
 *     operand or scale.  Ordering against other streams, copies and events
 *     is unchanged.
 *   - Every wait inside a kernel is bounded in time.  A wait that runs out
 *     makes the kernel record FP8LA_ERR_DEVICE_TIMEOUT in a device status
 *     word and return early (its outputs are then undefined); read and clear
 *     the word with fp8_get_device_status.
 *   - GEMM operands are E4M3 codes: A is [M][K] (K contiguous, leading
 *     dimension lda); B is stored K-major, [N][K] (element (k, n) of the
 *     K x N matrix at B[n*ldb + k]); C is [M][N] BF16 (leading dimension
 *     ldc).  TMA needs 16-byte-aligned base pointers and strides: A and B
 *     must be 16-byte aligned with lda, ldb multiples of 16 (otherwise
 *     FP8LA_ERR_ALIGNMENT).  C needs only 2-byte alignment; when C is
 *     16-byte aligned and ldc is a multiple of 8 the kernels store whole
 *     32 x 32 blocks by TMA and 16-byte vectors, otherwise single elements.
 *     M, N, K need not be multiples of any tile.
 *     K = 0 writes C = 0; M = 0 or N = 0 does nothing.
 */
#ifndef FP8LA_H
#define FP8LA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points keep default visibility even when the library is built with
 * -fvisibility=hidden. */
#if defined(__GNUC__)
#define FP8LA_API __attribute__((visibility("default")))
#else
#define FP8LA_API
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *fp8la_stream_t;

typedef int fp8la_status;
#define FP8LA_OK                  0
#define FP8LA_ERR_INVALID_ARG    -1  /* NULL pointer, negative size, ld < width, ... */
#define FP8LA_ERR_ALIGNMENT      -2  /* pointer or stride breaks the 16-byte TMA rule */
#define FP8LA_ERR_UNSUPPORTED    -3  /* size beyond a TMA or kernel limit; no sm_10x GPU */
#define FP8LA_ERR_CUDA           -4  /* a CUDA runtime or driver call failed */
#define FP8LA_ERR_DEVICE_TIMEOUT -5  /* a bounded wait inside a kernel ran out */
#define FP8LA_ERR_DEVICE_ARG     -6  /* a kernel found a device-side argument it
                                        cannot use (m_offsets of fp8_grouped_gemm or
                                        fp8_quantize_pertensor_grouped) */

/*
 * Per-tensor E4M3 quantisation ([P1] risks paragraph: E4M3 spans +-448 and
 * needs per-tensor scaling against overflow; parameter list: scale_max=448;
 * encoding per [FP8]).
 *
 *   amax   = max |x[i][j]| over the rows x cols tensor, NaN ignored (fp32)
 *   qscale = fp32(448 / amax),   scale = fp32(amax / 448)   (IEEE division)
 *            (amax == 0 or qscale not finite: qscale = scale = 1)
 *   q[i][j] = E4M3 code of fp32(x[i][j] * qscale), round-to-nearest-even,
 *             saturating to +-448 (NaN -> 0x7F; the sign of zero is kept)
 *
 * x: fp32 [rows][ldx] (device, read); q: uint8 [rows][ldq] (device, written);
 * amax_out, scale_out: one fp32 each (device, written).  The scale stays on
 * the device so it can feed fp8_gemm by pointer with no host round trip.
 * Requires ldx >= cols, ldq >= cols.  rows == 0 or cols == 0 writes
 * amax = 0, scale = 1.  x and q must not overlap.  amax_out and scale_out
 * must be two different words (the cast reads the amax while the scale is
 * written): the same pointer for both returns FP8LA_ERR_INVALID_ARG.
 */
FP8LA_API fp8la_status fp8_quantize_pertensor(const float *x, int64_t rows, int64_t cols,
                                    int64_t ldx, uint8_t *q, int64_t ldq,
                                    float *amax_out, float *scale_out,
                                    fp8la_stream_t stream);

/*
 * FP8 formats for the *_ex entry points.  E4M3 is the method's format;
 * E5M2 ([P3] tensor-core paragraph names both; [FP8]: 1 sign, 5 exponent
 * bits with bias 15, 2 mantissa bits, IEEE-style infinities and NaNs,
 * largest finite magnitude 57344) trades precision for range.
 */
#define FP8LA_FORMAT_E4M3 0
#define FP8LA_FORMAT_E5M2 1

/*
 * fp8_quantize_pertensor for a chosen FP8 format: as above with 448
 * replaced by the format's largest finite magnitude (57344 for E5M2):
 * qscale = fp32(fmax / amax), scale = fp32(amax / fmax), saturating RNE
 * cast to the format (NaN -> 0x7F).  format: FP8LA_FORMAT_E4M3 or
 * FP8LA_FORMAT_E5M2, else FP8LA_ERR_INVALID_ARG.
 */
FP8LA_API fp8la_status fp8_quantize_pertensor_ex(const float *x, int64_t rows,
                                                 int64_t cols, int64_t ldx,
                                                 uint8_t *q, int64_t ldq,
                                                 float *amax_out,
                                                 float *scale_out,
                                                 int32_t format,
                                                 fp8la_stream_t stream);

/*
 * Delayed-scaling per-tensor quantisation: one pass over x instead of two.
 * The pages describe per-tensor scaling with the tensor's own amax
 * ([P1] risks paragraph); this variant takes the scale from an amax
 * carried over from an earlier call (typically the same tensor's amax at
 * the previous step) and records the current amax for the next call:
 *
 *   qscale = fp32(fmax / amax_prev),  scale = fp32(amax_prev / fmax)
 *            (amax_prev == 0 or qscale not finite: qscale = scale = 1)
 *   q[i][j] = code of fp32(x[i][j] * qscale), RNE, saturating to +-fmax
 *             (values beyond amax_prev land on the largest code)
 *   amax_out = max |x[i][j]|, NaN ignored
 *
 * fmax = 448 (FP8LA_FORMAT_E4M3) or 57344 (FP8LA_FORMAT_E5M2).  x: fp32
 * [rows][ldx] (device, read); q: uint8 [rows][ldq] (device, written);
 * amax_prev: one fp32 (device, read); amax_out, scale_out: one fp32 each
 * (device, written).  amax_prev, amax_out and scale_out must be three
 * different words (FP8LA_ERR_INVALID_ARG otherwise): a caller keeping a
 * history alternates two amax words between steps.  rows == 0 or cols == 0
 * writes amax_out = 0 and the scale of amax_prev.  Memory traffic: 4 bytes
 * read and 1 written per element.
 */
FP8LA_API fp8la_status fp8_quantize_pertensor_delayed(
    const float *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
    int64_t ldq, const float *amax_prev, float *amax_out, float *scale_out,
    int32_t format, fp8la_stream_t stream);

/*
 * 32x32 block E4M3 quantisation ([P3] implementation paragraph: scale
 * granularity of 32x32 blocks).  Each 32x32 tile (ragged at the right and
 * bottom edges: a tile covers only its in-range elements) is quantised
 * exactly as fp8_quantize_pertensor quantises a whole tensor, with its own
 * amax; its scale fp32(tile_amax / 448) goes to
 * scales[(i/32) * ld_scales + (j/32)].
 *
 * x: fp32 [rows][ldx]; q: uint8 [rows][ldq]; scales: fp32
 * [ceil(rows/32)][ld_scales], ld_scales >= ceil(cols/32).  All device.
 */
FP8LA_API fp8la_status fp8_quantize_blockwise_32x32(const float *x, int64_t rows,
                                          int64_t cols, int64_t ldx,
                                          uint8_t *q, int64_t ldq,
                                          float *scales, int64_t ld_scales,
                                          fp8la_stream_t stream);

/*
 * Per-tensor-scaled E4M3 GEMM ([P1] kernel-code paragraph: C tile = sum over
 * K of A tile x B tile with an FP32 accumulator; scale paragraph:
 * acc = acc * scale_a * scale_b; parameter list: E4M3 inputs, FP32
 * accumulator, BF16 output).
 *
 *   C[m][n] = bf16_rn( scale_a * scale_b * sum_k dec(A[m][k]) * dec(B[n][k]) )
 *
 * The sum is accumulated in FP32 on the tensor cores; the two scales are
 * applied once to the finished accumulator, left to right as the scale
 * paragraph writes it: fp32(fp32(acc * scale_a) * scale_b).  The scales are
 * never multiplied together, so outputs inside the FP32 range stay exact to
 * the bound even where scale_a * scale_b itself is not (two scales near
 * 1e-23, or near 1e20).  scale_a, scale_b: one fp32 each
 * (device, read at run time, e.g. fp8_quantize_pertensor's scale_out).
 * Layout and alignment rules: see the file header.
 */
FP8LA_API fp8la_status fp8_gemm(const uint8_t *A, int64_t lda, const uint8_t *B,
                      int64_t ldb, uint16_t *C, int64_t ldc, int64_t M,
                      int64_t N, int64_t K, const float *scale_a,
                      const float *scale_b, fp8la_stream_t stream);

/*
 * fp8_gemm with each operand in a chosen FP8 format (FP8LA_FORMAT_E4M3 or
 * FP8LA_FORMAT_E5M2; the two may differ): the same contraction, FP32
 * accumulation and BF16 output, decoding A with a_format and B with
 * b_format.  Other format values return FP8LA_ERR_INVALID_ARG.
 */
FP8LA_API fp8la_status fp8_gemm_ex(const uint8_t *A, int64_t lda,
                                   const uint8_t *B, int64_t ldb, uint16_t *C,
                                   int64_t ldc, int64_t M, int64_t N, int64_t K,
                                   const float *scale_a, const float *scale_b,
                                   int32_t a_format, int32_t b_format,
                                   fp8la_stream_t stream);

/*
 * Grouped per-tensor E4M3 quantisation: the per-expert operand feed of
 * fp8_grouped_gemm ([P3] implementation paragraph: the MoE grouped GEMM;
 * [P1] risks paragraph: per-tensor scaling).  Group e, the rows r in
 * [m_offsets[e], m_offsets[e+1]) of x, is quantised as fp8_quantize_pertensor
 * quantises a tensor, with its own amax:
 *
 *   amax_out[e]  = max |x[r][j]| over the group's rows, NaN ignored
 *   scale_out[e] = fp32(amax_out[e] / 448)   (amax 0 or 448/amax not finite: 1)
 *   q[r][j]      = E4M3 code of fp32(x[r][j] * fp32(448 / amax_out[e])),
 *                  round-to-nearest-even, saturating
 *
 * m_offsets: int32 [num_groups + 1] on the DEVICE, as for fp8_grouped_gemm
 * (starting at 0, non-decreasing, m_offsets[num_groups] <= rows_capacity);
 * the host never reads it, so a routing result can feed the quantiser and
 * the GEMM without a synchronisation.  Both kernels check it first: offsets
 * that break these rules make the call write no codes and no scales and
 * record FP8LA_ERR_DEVICE_ARG in the device status word
 * (fp8_get_device_status); amax_out is cleared in any case.  Groups with no
 * rows get amax 0 and scale 1.  x: fp32 [rows_capacity][ldx]; q: uint8
 * [rows_capacity][ldq] (rows at or past m_offsets[num_groups] are neither
 * read nor written); amax_out, scale_out: fp32 [num_groups], two arrays that
 * must not overlap (FP8LA_ERR_INVALID_ARG).  Requires ldx >= cols,
 * ldq >= cols, 0 <= num_groups <= 1024 (0: nothing is done),
 * rows_capacity < 2^31.
 */
FP8LA_API fp8la_status fp8_quantize_pertensor_grouped(const float *x, int32_t num_groups,
                                            const int32_t *m_offsets,
                                            int64_t rows_capacity, int64_t cols,
                                            int64_t ldx, uint8_t *q, int64_t ldq,
                                            float *amax_out, float *scale_out,
                                            fp8la_stream_t stream);

/*
 * 32x32 block-scaled E4M3 GEMM ([P3] implementation paragraph: 32x32 scale
 * blocks; warp-specialisation paragraph: one warp loads by TMA, one issues
 * the FP8 MMA, another promotes partial results on the CUDA cores).
 *
 *   C[m][n] = bf16_rn( sum_kb sa[m/32][kb] * sb[n/32][kb] * S_kb[m][n] ),
 *   S_kb[m][n] = sum_{k in [32kb, 32kb+32) and k < K} dec(A[m][k]) * dec(B[n][k])
 *
 * Each 32-wide K block's partial sum is formed on the tensor cores and then
 * promoted, multiplied by its tile-scale product, into an FP32 accumulator
 * on the CUDA cores.  The tile-scale product sa * sb is formed in FP32 (once
 * per pair of tiles, not per output), so the results meet the bound while
 * every product is a normal FP32 number; for scales amax / 448 from
 * fp8_quantize_blockwise_32x32 that is two tiles whose amax values multiply
 * to between 448^2 2^-126 (about 2.4e-33) and 448^2 2^128 (about 6.8e43).
 * sa: fp32 [ceil(M/32)][ld_sa], ld_sa >= ceil(K/32);
 * sb: fp32 [ceil(N/32)][ld_sb], ld_sb >= ceil(K/32).  All device.  The
 * scale grids are read by TMA: sa and sb must be 16-byte aligned and ld_sa,
 * ld_sb multiples of 4 (otherwise FP8LA_ERR_ALIGNMENT).
 */
FP8LA_API fp8la_status fp8_gemm_blockscaled_32x32(const uint8_t *A, int64_t lda,
                                        const uint8_t *B, int64_t ldb,
                                        uint16_t *C, int64_t ldc, int64_t M,
                                        int64_t N, int64_t K, const float *sa,
                                        int64_t ld_sa, const float *sb,
                                        int64_t ld_sb, fp8la_stream_t stream);

/*
 * Grouped per-tensor-scaled E4M3 GEMM for MoE experts, all groups in one
 * launch ([P3] implementation paragraph: for MoE the GEMM extends to a
 * grouped GEMM over the experts).
 *
 * For e in 0..num_groups-1, with rows r in [m_offsets[e], m_offsets[e+1]):
 *   C[r][n] = bf16_rn( scale_a[e] * scale_b[e] * sum_k dec(A[r][k]) * dec(B_e[n][k]) ),
 *   B_e = B + e * b_group_stride  ([N][K], K-major, leading dimension ldb).
 *
 * m_offsets: int32 [num_groups + 1] on the DEVICE, non-decreasing, starting
 * at 0, with m_offsets[num_groups] <= m_capacity; the host never reads it,
 * so routing results can feed the GEMM without a synchronisation.  The
 * kernels check it before computing anything: offsets that break these
 * rules make the call write nothing to C and record FP8LA_ERR_DEVICE_ARG in
 * the device status word (fp8_get_device_status), so a bad routing result
 * cannot write outside C.  A: [m_capacity][lda]; C: [m_capacity][ldc];
 * rows at or past m_offsets[num_groups] are neither read for any output nor
 * written.
 * Groups with no rows are skipped.  scale_a, scale_b: fp32 [num_groups]
 * (device), applied as in fp8_gemm.  b_group_stride (elements) must be a multiple of 16 and
 * >= N * ldb.  1 <= num_groups <= 1024.
 */
FP8LA_API fp8la_status fp8_grouped_gemm(int32_t num_groups, const int32_t *m_offsets,
                              int64_t m_capacity, const uint8_t *A,
                              int64_t lda, const uint8_t *B, int64_t ldb,
                              int64_t b_group_stride, uint16_t *C,
                              int64_t ldc, int64_t N, int64_t K,
                              const float *scale_a, const float *scale_b,
                              fp8la_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the current device's status
 * word.  Returns FP8LA_OK, FP8LA_ERR_DEVICE_TIMEOUT if a kernel's bounded
 * wait ran out since the last call, FP8LA_ERR_DEVICE_ARG if a kernel
 * refused a device-side argument (and no wait ran out), or FP8LA_ERR_CUDA if
 * the synchronisation or the copy failed.
 */
FP8LA_API fp8la_status fp8_get_device_status(fp8la_stream_t stream);

/*
 * Set the time limit, in nanoseconds, of every bounded wait inside the
 * library's kernels launched afterwards from this process (default 2e9,
 * i.e. 2 s; legitimate waits last microseconds).  Values < 1000 are
 * rejected with FP8LA_ERR_INVALID_ARG.
 */
FP8LA_API fp8la_status fp8la_set_wait_timeout_ns(int64_t timeout_ns);

/*
 * Diagnostic: launch one CTA of the per-tensor GEMM's pipeline on a
 * 128 x 256 x 128 problem with the producer's first TMA arrival withheld, so
 * the MMA warp's bounded wait must run out.  The kernel records
 * FP8LA_ERR_DEVICE_TIMEOUT, drains, frees its tensor memory and returns;
 * the caller checks fp8_get_device_status.  Buffers as for fp8_gemm with
 * M = 128, N = 256, K = 128.
 */
FP8LA_API fp8la_status fp8la_diag_gemm_withheld_arrival(const uint8_t *A, int64_t lda,
                                              const uint8_t *B, int64_t ldb,
                                              uint16_t *C, int64_t ldc,
                                              const float *scale_a,
                                              const float *scale_b,
                                              fp8la_stream_t stream);

/*
 * Diagnostic, as fp8la_diag_gemm_withheld_arrival, for the other GEMM
 * kernels.  kernel = FP8LA_DIAG_KERNEL_PAIR: the CTA-pair per-tensor kernel
 * (as fp8_gemm with scale_a, scale_b one fp32 each; ld_sa, ld_sb ignored;
 * M > 128), whose second CTA leaves out its first TMA loads, so the leader's
 * MMA wait and then every wait of both CTAs run out.  kernel =
 * FP8LA_DIAG_KERNEL_BLOCK32: the block-scaled kernel (arguments as
 * fp8_gemm_blockscaled_32x32), whose producer leaves out its first stage.
 * Either way the kernel records FP8LA_ERR_DEVICE_TIMEOUT, drains what it
 * issued, frees its tensor memory and returns; C is undefined.  Other
 * kernel values, or M, N, K <= 0, return FP8LA_ERR_INVALID_ARG.
 */
#define FP8LA_DIAG_KERNEL_PAIR 1
#define FP8LA_DIAG_KERNEL_BLOCK32 2
FP8LA_API fp8la_status fp8la_diag_withheld_arrival(
    int32_t kernel, const uint8_t *A, int64_t lda, const uint8_t *B,
    int64_t ldb, uint16_t *C, int64_t ldc, int64_t M, int64_t N, int64_t K,
    const float *scale_a, int64_t ld_sa, const float *scale_b, int64_t ld_sb,
    fp8la_stream_t stream);

/*
 * Choose the kernel behind fp8_gemm and fp8_grouped_gemm for calls made
 * afterwards from this process: 0 = by problem shape (default), 1 = the
 * single-CTA kernel (128 x 256 tiles), 2 = the CTA-pair kernel (256 x 256
 * tiles on two SMs, tcgen05 cta_group::2), 3 = the single-CTA kernel with
 * 128 x 128 tiles, 4 = two CTA pairs per cluster of four sharing the rows
 * of A by TMA multicast (3 and 4: fp8_gemm only; fp8_grouped_gemm treats
 * them as 0).  All
 * compute the same result within the documented bound; this exists for
 * testing and tuning.  Other values return FP8LA_ERR_INVALID_ARG.
 */
FP8LA_API fp8la_status fp8la_set_gemm_variant(int32_t variant);

/* Human-readable name of a status code (static storage). */
FP8LA_API const char *fp8la_status_string(fp8la_status status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
FP8LA_API int fp8la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8LA_H */
