// FP16 operand helpers of the warp-level FP8/W4 GEMMs (mma.sync m16n8k16,
// FP16 operands, FP32 accumulation): the MMA, the exact E4M3/E2M1 -> f16x2
// conversions, and the B fragments of power-of-two-scaled activations.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace wqp {
namespace f16op {

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// First MMA of a chain: d = A * B (zero accumulator).
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}
// (hi, lo) floats -> f16x2 (round to nearest even; exact for the scaled
// activations of at least 2^-17).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float hi, float lo) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Byte i (0..3) of x as two E2M1 codes -> f16x2 (low nibble = first element).
template <int I>
__device__ __forceinline__ uint32_t e2m1x2_byte(uint32_t x) {
  uint32_t d;
  if constexpr (I == 0)
    asm("{\n\t.reg .b8 b;\n\tmov.b32 {b, _, _, _}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "r"(x));
  else if constexpr (I == 1)
    asm("{\n\t.reg .b8 b;\n\tmov.b32 {_, b, _, _}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "r"(x));
  else if constexpr (I == 2)
    asm("{\n\t.reg .b8 b;\n\tmov.b32 {_, _, b, _}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "r"(x));
  else
    asm("{\n\t.reg .b8 b;\n\tmov.b32 {_, _, _, b}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "r"(x));
  return d;
}
// Half h (0: low, 1: high) of x as two E4M3 codes -> f16x2 (low byte first).
template <int H>
__device__ __forceinline__ uint32_t e4m3x2_half(uint32_t x) {
  uint32_t d;
  if constexpr (H == 0)
    asm("{\n\t.reg .b16 h;\n\tmov.b32 {h, _}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(d) : "r"(x));
  else
    asm("{\n\t.reg .b16 h;\n\tmov.b32 {_, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(d) : "r"(x));
  return d;
}
__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// B fragments of one block for one column tile from this thread's 32
// activations r (BF16 pairs in k order): scaled by 2^e and rounded to FP16,
// and 2^-e, where 2^e puts the block row's largest magnitude (over the 4
// lanes of the row, lanes 4g .. 4g + 3) in [2^14, 2^15).
__device__ __forceinline__ void build_bfrag_regs(const uint32_t (&r)[16], uint32_t (&bf)[16], float& inv) {
  // Largest magnitude of the block row: BF16 magnitudes order like their bits.
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) mx = __vmaxu2(mx, r[i] & 0x7FFF7FFFu);
  mx = max(mx & 0xFFFFu, mx >> 16);
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));   // the 4 lanes of row g hold its 128 activations
  const int E = static_cast<int>(mx >> 7);              // BF16 exponent field of the maximum
  const int sh = min(100, max(-113, 141 - E));           // 2^(E - 127 + sh) = 2^14
  const float scale = __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);
  inv = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
#pragma unroll
  for (int i = 0; i < 16; ++i) bf[i] = f32x2_to_f16x2(bf16hi(r[i]) * scale, bf16lo(r[i]) * scale);
}

// B fragments of one block for one column tile: the 32 activations of row
// min(g + 8 mt, M - 1) at k = kb + 32 t .. + 31 read from global memory.
__device__ __forceinline__ void build_bfrag(const uint16_t* A, int lda, int M, int kb, int mt, int g, int t4,
                                            uint32_t (&bf)[16], float& inv) {
  const int m = min(g + 8 * mt, M - 1);           // rows past M: any valid row, results unused
  const uint16_t* src = A + static_cast<size_t>(m) * lda + kb + 32 * t4;
  uint32_t r[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = ld_nc_v4(src + 8 * q);
    r[4 * q] = v.x;
    r[4 * q + 1] = v.y;
    r[4 * q + 2] = v.z;
    r[4 * q + 3] = v.w;
  }
  build_bfrag_regs(r, bf, inv);
}

}  // namespace f16op
}  // namespace wqp
