// In-register decoders for the three packed weight formats. Every decoded
// weight is exact (every Q2_0, E2M1 and E4M3 value is a BF16 and an FP32
// value; the Q2_0 FP32 decode carries a power-of-two position factor). The
// dequant kernels use the same FP32 decoders as the scalar GEMVs, so the
// bit-exact dequant tests cover the GEMV decode path too.
#pragma once
#include <cuda_fp16.h>

#include "common.cuh"

namespace wqp {

// ---------------------------------------------------------------- Q2_0
// Q2_0 block ("spark_model/layers/ops/gemv_q2_vec.rs", module docs and the
// test helper `gemv_row`): 34 bytes = 32 bytes of 2-bit codes, code i in bits
// 2*(i%4) of byte i/4, then the fp16 scale d; weight = ((code & 3) - 1) * d.

// Position factor of code j of a 16-code word: 4^j for j <= 10, 4^(j - 11)
// for j >= 11 (those fields are shifted down by 22 bits before masking).
__host__ __device__ constexpr float q2_pos_weight(int p) {
  return p <= 10 ? static_cast<float>(1u << (2 * p)) : static_cast<float>(1u << (2 * (p - 11)));
}

// FP32 decode of a 16-code word q (code j at bits 2j) with one mask per code:
// the field of code j, masked in place, read as FP32 bits is the subnormal
// c_j * q2_pos_weight(j) * 2^-149, exactly. w[i] = (w_{2i}, w_{2i+1}). A
// consumer multiplies it by the activation pre-scaled by
// 2^80 / q2_pos_weight(j) (a power of two), so every product is
// c * a * 2^-69 exactly, and accounts for the -1 of every code by starting
// each 16-code sum from -2^-69 * sum a.
__device__ __forceinline__ void q2_decode_sub(uint32_t q, float2 (&w)[8]) {
  const uint32_t q22 = q >> 22;
  float v[16];
#pragma unroll
  for (int j = 0; j < 11; ++j) v[j] = __uint_as_float(q & (3u << (2 * j)));
#pragma unroll
  for (int j = 11; j < 16; ++j) v[j] = __uint_as_float(q22 & (3u << (2 * (j - 11))));
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = make_float2(v[2 * i], v[2 * i + 1]);
}

// The 16 codes of word w (0..7) of a block that starts at a 2-byte aligned
// shared-memory address.
__device__ __forceinline__ uint32_t q2_code_word(const uint8_t* blk, int w) {
  const uint16_t* b16 = reinterpret_cast<const uint16_t*>(blk);
  return static_cast<uint32_t>(b16[2 * w]) | (static_cast<uint32_t>(b16[2 * w + 1]) << 16);
}
__device__ __forceinline__ float q2_scale(const uint8_t* blk) {
  return __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(blk)[16]));
}

// ---------------------------------------------------------------- FP8 / FP4
// Two E4M3 codes (low byte = first element) -> f16x2 (exact: E4M3 is a subset
// of binary16; NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t d;
  asm("{\n\t.reg .b16 lo;\n\tmov.b32 {lo, _}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(d)
      : "r"(two_bytes));
  return d;
}

// One byte of two E2M1 codes (low nibble = first element) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  asm("{\n\t.reg .b8 b;\n\tmov.b32 {b, _, _, _}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(d)
      : "r"(byte));
  return d;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
  __half2 v;
  *reinterpret_cast<uint32_t*>(&v) = h;
  return __half22float2(v);
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const uint32_t h = e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

// f16x2 -> bf16x2 for values whose FP32 form has a zero low half (every
// E4M3 and E2M1 value): widen exactly to FP32, then keep the upper halves.
// This avoids the FP32 -> BF16 packing conversion, which is slow.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_exact(uint32_t h) {
  const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

// Four E4M3 bytes of word x -> two bf16x2 pairs in element order.
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t x, uint32_t& p01, uint32_t& p23) {
  p01 = f16x2_to_bf16x2_exact(e4m3x2_to_f16x2(x & 0xFFFFu));
  p23 = f16x2_to_bf16x2_exact(e4m3x2_to_f16x2(x >> 16));
}

}  // namespace wqp
