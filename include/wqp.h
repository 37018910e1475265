/*
 * wqp.h - C ABI of libwqp.so: packed weight-only-quantized decode GEMV/GEMM
 * for GB300 (sm_103a).
 *
 *   C[M, N] = A[M, K] @ dequant(W)^T        (W stored per output row n)
 *
 * A is BF16 [M, K] row-major, C is BF16 [M, N] row-major, and W stays packed
 * in device memory; it is dequantised inside the dot product. Each output is
 * accumulated in FP32 and rounded once to BF16 (round to nearest even).
 *
 * Common contract of every compute entry point
 * ---------------------------------------------
 * Pointers. A, W, scales and C are DEVICE pointers that the caller owns.
 *   The library allocates no device memory, keeps no reference after the
 *   call and is safe to call from several host threads.
 * Stream. `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream). The call returns once the work is enqueued. A launch failure is
 *   returned as WQP_ERR_CUDA. A bounded wait that expires inside a kernel is
 *   recorded on the device and read with wqp_get_device_error().
 * Validation. All checks run before any CUDA call. A failed check returns
 *   WQP_ERR_INVALID_ARG and enqueues nothing. wqp_last_error() gives the
 *   reason. The checks are:
 *   - M >= 0 (M == 0 is a no-op returning WQP_OK), N >= 1, K >= 128,
 *     K % 128 == 0, K <= 1048576 and N <= 16777216;
 *   - the pointers are non-NULL;
 *   - A, W and the W4 scales are 16-byte aligned and C is 2-byte aligned;
 *   - for the strided forms, lda >= K, lda % 8 == 0 and ldc >= N.
 * Device. The library is built for sm_103a only. Any other device returns
 *   WQP_ERR_UNSUPPORTED.
 * Rows. Every compute entry accepts any M >= 0. Up to 16 rows go in one
 *   launch: every weight byte is read once for all of those rows. Larger M is
 *   served in 16-row launches on the same stream, with A and C advanced by
 *   whole rows ("w8a16_gemm_m16.rs", doc of `w8a16_gemm_m16`: callers with
 *   more rows than the M tile run it again on the next contiguous rows).
 * Numerics. A row of a batched call equals the same row computed with M = 1,
 *   bit for bit, and does not depend on the other rows. The tensor-core
 *   entries are exempt (see w8a16_gemm_tc).
 *
 * Citations are to the source pages by title and item.
 */
#ifndef WQP_H
#define WQP_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum wqp_status {
  WQP_OK = 0,
  WQP_ERR_INVALID_ARG = 1,    /* an argument failed validation; nothing ran  */
  WQP_ERR_UNSUPPORTED = 2,    /* device is not sm_103                         */
  WQP_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed         */
  WQP_ERR_DEVICE_TIMEOUT = 4  /* a kernel's bounded wait expired (see below)  */
} wqp_status;

/* Rows computed by one launch of the GEMV kernels (weights read once). */
#define WQP_MAX_M_PER_LAUNCH 16

/* ---------------------------------------------------------------- Q2_0 ---
 * Ternary Q2_0 decode GEMV.
 * Defined by "spark_model/layers/ops/gemv_q2_vec.rs": the docs of
 * `q2_0_gemv_vec` and `q2_0_gemv_vec_batchm`, and the test helper `gemv_row`:
 *   out[m, n] = sum_k a[m, k] * ((code(n, k) & 3) - 1) * d(n, k / 128)
 * The scale d is stored inline as fp16 in each block_q2_0, so there is no
 * separate scale pointer.
 * Layout. Each (row n, 128-wide K group g) is one 34-byte block, stored at
 *   byte offset (n * K/128 + g) * 34. Bytes 0..31 hold the codes: code i of
 *   the group is in bits 2*(i % 4) of byte i / 4. Bytes 32..33 hold d as
 *   little-endian fp16. There is no padding, so a row is 34 * K / 128 bytes.
 * scales: must be NULL (WQP_ERR_INVALID_ARG otherwise).
 */
int q2_gemv(const void* A, const void* W, const void* scales, void* C,
            int M, int N, int K, void* stream);

/* Q2_0 GEMV with row pitches in elements: A row m starts at A + m * lda,
 * C row m at C + m * ldc. Otherwise identical to q2_gemv. */
int q2_gemv_strided(const void* A, int lda, const void* W, void* C, int ldc,
                    int M, int N, int K, void* stream);

/* Tensor-core (tcgen05) form of q2_gemv: swap-AB, with the weight rows on
 * the 128-row MMA side and the activation rows padded to 16 on the MMA N
 * side. The codes enter the MMA as exact BF16 values c * 4^j * 2^-133 and the
 * activations as a * 2^(64 - 2j), so every product c * a is exact; each
 * 128-K group's sum of (c - 1) * a is scaled by its inline d once, in FP32.
 * Activations must satisfy |a| < 2^62 (the pre-scale stays finite).
 * Arguments and layouts are those of q2_gemv, with one more limit:
 * K % 1024 == 0, so that rows stay 16-byte aligned for the tensor-map
 * copies. Anything else gives WQP_ERR_INVALID_ARG.
 * Numerics: every product is exact and only the order of the FP32 additions
 * differs from the plain row sum, so the contract is the scalar one: within
 * 1 BF16 ULP of the FP32 row sum, or within the FP32 reordering bound
 * 8 * sqrt(K) * 2^-24 * sum_k |a * w| for outputs near zero. It is not
 * bit-identical to q2_gemv. A row does not depend on the other rows of the
 * call.
 */
int q2_gemm_tc(const void* A, const void* W, void* C, int M, int N, int K, void* stream);
int q2_gemm_tc_strided(const void* A, int lda, const void* W, void* C, int ldc,
                       int M, int N, int K, void* stream);

/* Warp-level tensor-core form of q2_gemv (mma.sync m16n8k16, BF16 operands,
 * FP32 accumulation), swap-AB with 16 weight rows by 8 activation rows per
 * MMA. Each warp decodes its own code words straight into MMA operands in
 * registers (the same exact encoding as q2_gemm_tc: c * 4^j * 2^-133 against
 * a * 2^(64 - 2j)); each 128-K block's sum of (c - 1) * a is scaled by its
 * inline d once, in FP32. The K range is split over the CTAs of a thread-block
 * cluster and the partial sums are added in rank order in shared memory.
 * Arguments, layouts and limits are those of q2_gemm_tc (K % 1024 == 0,
 * |a| < 2^62); anything else gives WQP_ERR_INVALID_ARG.
 * Shapes of at least two 64-row tiles per SM (N >= 128 * SMs) with
 * K <= 57344 run on a persistent kernel whose CTAs build their activation
 * fragments once and stream their weight tiles through a ring of raw
 * stages; one launch serves up to 16 activation rows (two column tiles), so
 * the weights are read once for all of them. Other shapes run one short CTA
 * per (tile, K range) and 8 activation rows per launch (M = 9..16 is two
 * launches). The choice depends on N and K only, never on M.
 * Numerics: the scalar contract of q2_gemm_tc. Not bit-identical to q2_gemv
 * or q2_gemm_tc. A row does not depend on the other rows of the call.
 * Device-side waits are bounded as for the other kernels (see
 * wqp_get_device_error).
 */
int q2_gemm_mma(const void* A, const void* W, void* C, int M, int N, int K, void* stream);
int q2_gemm_mma_strided(const void* A, int lda, const void* W, void* C, int ldc,
                        int M, int N, int K, void* stream);

/* ---------------------------------------------------------------- W4A16 ---
 * 4-bit E2M1 weights with E4M3 group scales (NVFP4-style) decode GEMV.
 * The family is "spark_model/layers/w4a16_gemv_tiers.rs" (module docs: the
 * batched W4A16 GEMV, and the exact-M tier rationale). The pages do not print
 * the dequant formula. The reading taken is
 *   w[n, k] = (e2m1(nibble(n, k)) * e4m3(scales[n, k / 16])) * global_scale
 * with C[m, n] = bf16(sum_k a[m, k] * w[n, k]) accumulated in FP32.
 * Layout. W is uint8 [N, K/2]: byte j of a row holds element 2j in its low
 *   nibble and element 2j+1 in its high nibble. scales is uint8 [N, K/16]
 *   of E4M3 codes (OCP FP8, bias 7).
 * w4a16_gemv uses global_scale = 1.0. w4a16_gemv_ex takes it explicitly,
 * together with the row pitches lda and ldc.
 */
int w4a16_gemv(const void* A, const void* W, const void* scales, void* C,
               int M, int N, int K, void* stream);
int w4a16_gemv_ex(const void* A, int lda, const void* W, const void* scales,
                  float global_scale, void* C, int ldc,
                  int M, int N, int K, void* stream);

/* Tensor-core (tcgen05) form of w4a16_gemv: swap-AB, with the weight rows on
 * the 128-row MMA side and the activation rows padded to 16 on the MMA N
 * side. Each e2m1 * e4m3 product is exact in BF16, so the products are
 * exact; the global scale multiplies each FP32 result once, at the store.
 * Arguments and layouts are those of w4a16_gemv / w4a16_gemv_ex, with one
 * more limit: K % 256 == 0, so that the scale rows (K/16 bytes) are
 * multiples of 16 bytes for the tensor-map copies. Anything else gives
 * WQP_ERR_INVALID_ARG.
 * Numerics: the products are exact, so the contract is the scalar one of
 * q2_gemm_tc. It is not bit-identical to w4a16_gemv. A row does not depend
 * on the other rows of the call.
 */
int w4a16_gemm_tc(const void* A, const void* W, const void* scales, void* C,
                  int M, int N, int K, void* stream);
int w4a16_gemm_tc_ex(const void* A, int lda, const void* W, const void* scales,
                     float global_scale, void* C, int ldc,
                     int M, int N, int K, void* stream);

/* Warp-level tensor-core form of w4a16_gemv (mma.sync m16n8k16, FP16
 * operands, FP32 accumulation), swap-AB with 16 weight rows by 8 activation
 * rows per MMA. Shapes of at least 1.75 64-row tiles per SM, or of more than
 * 8 K stages of 1024, run on a persistent kernel with two column tiles for
 * M = 9..16, so the weights are read once for up to 16 rows; smaller shapes
 * run one short CTA per (tile, K stage) and 8 rows per launch (M = 9..16 is
 * two launches). The choice depends on N and K only, never on M. The weight
 * operand is e2m1 * e4m3(scale), exact in
 * FP16. Each activation row is scaled per 128-K block by the power of two
 * 2^e that puts its largest magnitude in [2^14, 2^15) and rounded to FP16
 * (exact for every value of at least 2^-31 times that maximum); each block's
 * FP32 sum is multiplied by 2^-e once, and the global scale multiplies each
 * FP32 result at the store.
 * Arguments and layouts are those of w4a16_gemv / w4a16_gemv_ex, with one
 * more limit: K % 1024 == 0 (whole stages of 8 blocks for the tensor-map
 * copies). Anything else gives WQP_ERR_INVALID_ARG.
 * Numerics: the scalar contract of q2_gemm_tc. A row does not depend on the
 * other rows of the call.
 */
int w4a16_gemm_mma(const void* A, const void* W, const void* scales, void* C,
                   int M, int N, int K, void* stream);
int w4a16_gemm_mma_ex(const void* A, int lda, const void* W, const void* scales,
                      float global_scale, void* C, int ldc,
                      int M, int N, int K, void* stream);

/* ---------------------------------------------------------------- W8A16 ---
 * FP8 E4M3 weights with FP32 128x128 block scales, scalar-FMA decode GEMM.
 * Defined by "metrale_model_layers/layers/ops/w8a16_gemm_m16.rs" (doc of
 * `w8a16_gemm_m16`: weight [N, K] FP8 E4M3, block_scale [N/128, K/128] FP32;
 * module docs: the 128-K block scale is folded once per block onto an FP32
 * outer accumulator, never per element and never into BF16):
 *   C[m, n] = bf16( sum_b s[n/128, b] * sum_{k in block b} a[m, k] * e4m3(W[n, k]) )
 * Layout. W is uint8 [N, K]. scales is float [ceil(N/128), K/128] and must
 *   be 4-byte aligned.
 */
int w8a16_gemm(const void* A, const void* W, const float* scales, void* C,
               int M, int N, int K, void* stream);
int w8a16_gemm_strided(const void* A, int lda, const void* W, const float* scales,
                       void* C, int ldc, int M, int N, int K, void* stream);

/* Tensor-core (tcgen05) form of w8a16_gemm: swap-AB, with the weights on the
 * 128-row MMA side and the activation rows padded to 16 on the MMA N side.
 * Same arguments and layouts as w8a16_gemm. The kernel's M tile is 16 rows
 * ("w8a16_gemm_m16.rs", doc of `w8a16_gemm_m16`); M > 16 runs as further
 * 16-row launches.
 * Numerics ("w8a16_gemm_m16.rs", module docs): the tensor core reduces each
 * 16-K step in its own order, so the result is not bit-identical to
 * w8a16_gemm. The contract is: at most 4 BF16 ULP from the reference, or an
 * absolute error below 1e-3 * sqrt(K) * rms(a[m,:]) * max_k |w[n,k]|. The
 * block scale is still folded once per 128-K block, in FP32.
 */
int w8a16_gemm_tc(const void* A, const void* W, const float* scales, void* C,
                  int M, int N, int K, void* stream);
int w8a16_gemm_tc_strided(const void* A, int lda, const void* W, const float* scales,
                          void* C, int ldc, int M, int N, int K, void* stream);

/* Warp-level tensor-core form of w8a16_gemm (mma.sync m16n8k16, FP16
 * operands, FP32 accumulation), swap-AB as w4a16_gemm_mma. E4M3 is a subset
 * of FP16, so the weight operand is exact; the activations are scaled per
 * (row, 128-K block) by a power of two and rounded to FP16 as in
 * w4a16_gemm_mma. Each 128-K block's FP32 sum is multiplied once by its block
 * scale (and by 2^-e) and added to the FP32 accumulator, as "w8a16_gemm_m16.rs"
 * (module docs) requires.
 * Arguments and layouts are those of w8a16_gemm, with two more limits:
 * K % 1024 == 0, and scales 16-byte aligned (the tensor-map copies).
 * Anything else gives WQP_ERR_INVALID_ARG.
 * Numerics: the scalar contract of q2_gemm_tc. A row does not depend on the
 * other rows of the call.
 */
int w8a16_gemm_mma(const void* A, const void* W, const float* scales, void* C,
                   int M, int N, int K, void* stream);
int w8a16_gemm_mma_strided(const void* A, int lda, const void* W, const float* scales,
                           void* C, int ldc, int M, int N, int K, void* stream);

/* ------------------------------------------------------------ dequant ---
 * Unpack every weight to FP32: out is float [N, K] row-major, device memory,
 * 4-byte aligned. Each value is the one the GEMVs multiply by:
 *   q2:  ((code & 3) - 1) * d
 *   w4:  (e2m1 * e4m3(scale)) * global_scale
 *   w8:  e4m3(W) * s[n/128, k/128]           (one FP32 multiply)
 * These are debugging and verification aids, not part of the hot path.
 */
int q2_dequant(const void* W, float* out, int N, int K, void* stream);
int w4a16_dequant(const void* W, const void* scales, float global_scale, float* out,
                  int N, int K, void* stream);
int w8a16_dequant(const void* W, const float* scales, float* out, int N, int K, void* stream);

/* ------------------------------------------------------------ host helpers -
 * Row chunking for calls with more rows than one launch computes
 * ("gemv_q2_vec.rs", `batchm_row_chunks` and `batchm_launch_chunks`).
 * Writes up to `cap` triples (a_byte_offset, c_byte_offset, rows) into
 * `out`, for contiguous BF16 A [M, K] and C [M, N] split into chunks of at
 * most max_rows rows. Returns the number of chunks (0 when M == 0), or -1
 * for invalid arguments or when cap is too small. Host only: no CUDA call.
 */
int wqp_row_chunks(int M, int K, int N, int max_rows, long long* out, int cap);

/* Launch policy: when enabled, kernels are launched with programmatic
 * dependent launch (PDL). A kernel may then start while the previous kernel
 * on the stream is finishing. It prefetches W (and the scales) before it
 * waits for that kernel, and reads A only after the wait. So with PDL
 * enabled, W must not be written by the kernel launched just before on the
 * same stream. Off by default. The setting is process-wide. Returns the
 * previous setting. */
int wqp_set_pdl(int enable);

/* Read and clear the device error word on the current device. It makes one
 * synchronous cudaMemcpy, so it waits for the work queued before it. Returns
 * WQP_OK, WQP_ERR_DEVICE_TIMEOUT (a bounded mbarrier wait inside a kernel
 * ran out; that kernel stopped early and its C is not valid), or
 * WQP_ERR_CUDA. */
int wqp_get_device_error(void);

/* Self-test of the failure path (for tests): launches one small kernel that
 * waits, through the same bounded mbarrier wait the GEMM kernels use, on a
 * barrier nothing ever completes. After limit_us microseconds (1..10^6) of
 * wall time the wait gives up, the kernel records the timeout in the device
 * error word and returns, so the next wqp_get_device_error() reports
 * WQP_ERR_DEVICE_TIMEOUT and the context stays usable. (The GEMM kernels'
 * waits give up after 2 s.) No trap, fault or hang is involved. Returns
 * WQP_ERR_INVALID_ARG for limit_us out of range, WQP_ERR_CUDA if the launch
 * fails, else WQP_OK. */
int wqp_selftest_wait_timeout(int limit_us, void* stream);

/* Human-readable name of a status code (static string). */
const char* wqp_status_string(int status);

/* Reason for the last non-OK status returned on the calling thread (static
 * thread-local buffer; "" when none). */
const char* wqp_last_error(void);

/* ABI version of this header (increments on incompatible change). */
int wqp_abi_version(void);
#define WQP_ABI_VERSION 1

#ifdef __cplusplus
}
#endif
#endif /* WQP_H */
