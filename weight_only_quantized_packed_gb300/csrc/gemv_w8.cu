// W8A16 scalar-FMA GEMM: FP8 E4M3 weights [N, K] with FP32 block scales
// [ceil(N/128), K/128] ("metrale_model_layers/layers/ops/w8a16_gemm_m16.rs",
// doc of `w8a16_gemm_m16`). The block scale is applied once per 16-K segment
// to that segment's FP32 partial sum, on the FP32 outer accumulator; it never
// multiplies a single element and never touches BF16 (module docs of the same
// page).
#include "decode.cuh"
#include "gemv_scalar.cuh"

namespace wqp {

struct W8Fmt {
  static constexpr int kWBytesPerRow = 1024;
  static constexpr bool kJ8 = false;
  static bool bulk_ok(int) { return true; }   // rows start at n * K, K % 128 == 0
  __device__ static uint32_t row_tile_bytes(int, int, int tg) { return 128u * tg; }
  __device__ static void issue_row_bulk(const ScalarParams& p, int n, int t, int tg, uint32_t dst,
                                        uint32_t bar, uint64_t pol) {
    bulk_g2s_stream(dst, p.W + static_cast<size_t>(n) * p.K + 1024 * t, 128u * tg, bar, pol);
  }
  __device__ static void copy_row_plain(const ScalarParams& p, int n, int t, int tg, uint8_t* dst,
                                        int lane) {
    const uint4* c = reinterpret_cast<const uint4*>(p.W + static_cast<size_t>(n) * p.K + 1024 * t);
    for (int i = lane; i < 8 * tg; i += 32) reinterpret_cast<uint4*>(dst)[i] = __ldg(c + i);
  }
  __device__ static void decode(const ScalarParams& p, int n, int t, int sg, const uint8_t* sW, Seg& g) {
    const uint4 c = *reinterpret_cast<const uint4*>(sW + 16 * sg);
    e4m3x4_to_bf16(c.x, g.p[0], g.p[1]);
    e4m3x4_to_bf16(c.y, g.p[2], g.p[3]);
    e4m3x4_to_bf16(c.z, g.p[4], g.p[5]);
    e4m3x4_to_bf16(c.w, g.p[6], g.p[7]);
    const int kb = p.K >> 7;
    g.s = __ldg(static_cast<const float*>(p.scales) + static_cast<size_t>(n >> 7) * kb + t * 8 + (sg >> 3));
  }
};

cudaError_t launch_w8a16_gemm(const GemvArgs& a, cudaStream_t s) {
  return launch_scalar_dispatch<W8Fmt, true>(a, s);
}

}  // namespace wqp
