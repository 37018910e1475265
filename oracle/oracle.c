/*
 * CPU oracle for the packed weight-only-quantized decode GEMV/GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library. The product path (libwqp.so and its
 * Python binding) never links, loads or calls it, and it shares no code,
 * header, table or helper with the CUDA sources.
 *
 * It is plain and slow on purpose: every output is one sequential loop over k
 * in ascending order, in the precision the source pages fix, with no
 * blocking, fusion or reordering. Build flags: -O2 -ffp-contract=off
 * -fno-fast-math, so `acc = acc + a * w` is a separately rounded multiply
 * and add (as in the Rust test oracle, which never contracts to FMA).
 * OpenMP only splits independent (m, n) outputs, so results do not depend
 * on the thread count.
 *
 * Sources (page title, item):
 *  - "spark_model/layers/ops/gemv_q2_vec.rs", test helper `gemv_row`:
 *      out[n] = sum_k a[k] * ((code(n,k) & 3) - 1) * d(n, k/128), f32
 *      accumulator, then BF16 (round to nearest even). The module docs: the
 *      Q2_0 block carries its fp16 scale inline; group = 128.
 *  - "metrale_model_layers/layers/ops/w8a16_gemm_m16.rs", module docs: the
 *      128-K block scale is folded once per block onto an FP32 outer
 *      accumulator, never per element and never into BF16; weights [N, K]
 *      FP8 E4M3 and block scales [N/128, K/128] FP32 (doc of w8a16_gemm_m16).
 *  - "spark_model/layers/w4a16_gemv_tiers.rs", module docs: the W4A16
 *      (NVFP4) batched GEMV; the pages do not print its dequant formula.
 *      Reading taken: w = (e2m1(nibble) * e4m3(group scale)) * g with one
 *      E4M3 scale per 16 K and one FP32 per-tensor scale g, per element,
 *      summed sequentially in f32 like the Q2_0 row oracle.
 *
 * Format decoders are written from the format definitions (IEEE 754 binary16,
 * bfloat16 = the upper half of binary32, OCP FP8 E4M3 with bias 7 and no
 * infinities, OCP MX E2M1 with bias 1), not from any CUDA header.
 *
 * Besides the BF16 result, every GEMV entry can return, per output, the fp64
 * sum R = sum_k a*w and the fp64 magnitude sum S = sum_k |a*w| (w the
 * element's full dequantised value including its scale); the tests derive
 * their reordering tolerance from S.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------ decoders */

/* bfloat16 -> binary32: the bf16 pattern is the upper 16 bits. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even; NaN stays NaN. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* IEEE binary16 -> binary32. */
static float f16_to_f32(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  float v;
  if (e == 0)
    v = ldexpf((float)m, -24);                   /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexpf((float)(1024 + m), e - 25);       /* (1 + m/1024) * 2^(e-15) */
  return s ? -v : v;
}

/* OCP FP8 E4M3: bias 7, S.1111.111 is NaN, no infinities. */
static float e4m3_to_f32(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 7;
  float v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexpf((float)m, -9);                    /* m/8 * 2^-6 */
  else
    v = ldexpf((float)(8 + m), e - 10);          /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* OCP MX E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. */
static float e2m1_to_f32(uint8_t nib) {
  int s = (nib >> 3) & 1;
  int e = (nib >> 1) & 3;
  int m = nib & 1;
  float v;
  if (e == 0)
    v = 0.5f * (float)m;                         /* subnormal: m/2 * 2^0 */
  else
    v = ldexpf((float)(2 + m), e - 2);           /* (1 + m/2) * 2^(e-1) */
  return s ? -v : v;
}

/* ------------------------------------------------------------ Q2_0 */

#define Q2_GROUP 128
#define Q2_BLOCK 34

/* Value of the Q2_0 weight (n, k): ((code & 3) - 1) * d. The block of
 * (n, g) starts at byte (n * K/128 + g) * 34; code i of the group sits in
 * bits 2*(i%4) of byte i/4; bytes 32..33 are d (fp16, little-endian). */
static float q2_weight(const uint8_t* W, int K, int n, int k) {
  const uint8_t* blk = W + ((size_t)n * (size_t)(K / Q2_GROUP) + (size_t)(k / Q2_GROUP)) * Q2_BLOCK;
  int i = k % Q2_GROUP;
  int code = (blk[i / 4] >> (2 * (i % 4))) & 3;
  float d = f16_to_f32((uint16_t)(blk[32] | (blk[33] << 8)));
  return (float)(code - 1) * d;
}

void oracle_q2_dequant(const uint8_t* W, int N, int K, float* out) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) out[(size_t)n * K + k] = q2_weight(W, K, n, k);
}

void oracle_q2_gemv(const uint16_t* A, const uint8_t* W, int M, int N, int K,
                    uint16_t* C, double* R, double* S) {
  long total = (long)M * N;
#pragma omp parallel for schedule(static)
  for (long mn = 0; mn < total; ++mn) {
    int m = (int)(mn / N), n = (int)(mn % N);
    float acc = 0.0f;
    double r = 0.0, s = 0.0;
    for (int k = 0; k < K; ++k) {
      float a = bf16_to_f32(A[(size_t)m * K + k]);
      float w = q2_weight(W, K, n, k);
      float p = a * w;
      acc = acc + p;
      r += (double)a * (double)w;
      s += fabs((double)a * (double)w);
    }
    C[(size_t)m * N + n] = f32_to_bf16(acc);
    if (R) R[(size_t)m * N + n] = r;
    if (S) S[(size_t)m * N + n] = s;
  }
}

/* ------------------------------------------------------------ W4 (E2M1) */

#define W4_GROUP 16

/* Value of W4 weight (n, k): (e2m1(nibble) * e4m3(scale[n, k/16])) * g.
 * Byte j of a row holds element 2j in its low nibble, 2j+1 in its high. */
static float w4_weight(const uint8_t* codes, const uint8_t* scales, float g, int K, int n, int k) {
  uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
  uint8_t nib = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
  float s = e4m3_to_f32(scales[(size_t)n * (K / W4_GROUP) + k / W4_GROUP]);
  float q = e2m1_to_f32(nib) * s;
  return q * g;
}

void oracle_w4_dequant(const uint8_t* codes, const uint8_t* scales, float g, int N, int K, float* out) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) out[(size_t)n * K + k] = w4_weight(codes, scales, g, K, n, k);
}

void oracle_w4_gemv(const uint16_t* A, const uint8_t* codes, const uint8_t* scales, float g,
                    int M, int N, int K, uint16_t* C, double* R, double* S) {
  long total = (long)M * N;
#pragma omp parallel for schedule(static)
  for (long mn = 0; mn < total; ++mn) {
    int m = (int)(mn / N), n = (int)(mn % N);
    float acc = 0.0f;
    double r = 0.0, s = 0.0;
    for (int k = 0; k < K; ++k) {
      float a = bf16_to_f32(A[(size_t)m * K + k]);
      float w = w4_weight(codes, scales, g, K, n, k);
      float p = a * w;
      acc = acc + p;
      r += (double)a * (double)w;
      s += fabs((double)a * (double)w);
    }
    C[(size_t)m * N + n] = f32_to_bf16(acc);
    if (R) R[(size_t)m * N + n] = r;
    if (S) S[(size_t)m * N + n] = s;
  }
}

/* ------------------------------------------------------------ W8 (E4M3) */

#define W8_BLOCK 128

/* Dequantised W8 weight: e4m3(w[n,k]) * s[n/128, k/128], one f32 multiply. */
void oracle_w8_dequant(const uint8_t* w, const float* bs, int N, int K, float* out) {
  int kb = K / W8_BLOCK;
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      out[(size_t)n * K + k] =
          e4m3_to_f32(w[(size_t)n * K + k]) * bs[(size_t)(n / W8_BLOCK) * kb + k / W8_BLOCK];
}

/* Per 128-K block b: inner = sum_{k in b} a * e4m3(w) (sequential, f32),
 * then acc = acc + inner * s[n/128, b] (f32). Output bf16(acc). */
void oracle_w8_gemm(const uint16_t* A, const uint8_t* w, const float* bs, int M, int N, int K,
                    uint16_t* C, double* R, double* S) {
  long total = (long)M * N;
  int kb = K / W8_BLOCK;
#pragma omp parallel for schedule(static)
  for (long mn = 0; mn < total; ++mn) {
    int m = (int)(mn / N), n = (int)(mn % N);
    float acc = 0.0f;
    double r = 0.0, s = 0.0;
    for (int b = 0; b < kb; ++b) {
      float scale = bs[(size_t)(n / W8_BLOCK) * kb + b];
      float inner = 0.0f;
      for (int k = b * W8_BLOCK; k < (b + 1) * W8_BLOCK; ++k) {
        float a = bf16_to_f32(A[(size_t)m * K + k]);
        float q = e4m3_to_f32(w[(size_t)n * K + k]);
        float p = a * q;
        inner = inner + p;
        double wd = (double)q * (double)scale;
        r += (double)a * wd;
        s += fabs((double)a * wd);
      }
      float t = inner * scale;
      acc = acc + t;
    }
    C[(size_t)m * N + n] = f32_to_bf16(acc);
    if (R) R[(size_t)m * N + n] = r;
    if (S) S[(size_t)m * N + n] = s;
  }
}

/* ------------------------------------------------------------ utilities */

/* Element decoders exposed for the pins (tables checked against the format
 * definitions and library routines). */
float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16(f); }
float oracle_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
float oracle_e4m3_to_f32(uint8_t b) { return e4m3_to_f32(b); }
float oracle_e2m1_to_f32(uint8_t n) { return e2m1_to_f32(n); }

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
