// W8A16 scalar-FMA GEMM: FP8 E4M3 weights [N, K] with FP32 block scales
// [ceil(N/128), K/128] ("metrale_model_layers/layers/ops/w8a16_gemm_m16.rs",
// doc of `w8a16_gemm_m16`). The block scale is applied to each 16-K
// segment's FP32 partial sum on the FP32 outer accumulator. It never
// multiplies a single element and never touches BF16 (module docs of the
// same page).
#include "decode.cuh"
#include "gemv_scalar.cuh"

namespace wqp {

struct W8Fmt {
  static constexpr int kTK = 512;
  static constexpr int kWRow = 512;
  static constexpr int kW2Row = 0;
  static bool bulk_ok(int) { return true; }   // rows are K bytes, K % 128 == 0
  static cudaError_t make_maps(const GemvArgs& a, CUtensorMap* mw, CUtensorMap*) {
    const uint64_t K = static_cast<uint64_t>(a.K);
    return make_rows_map(mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, K / 4, a.N, K, kWRow / 4, kRows);
  }
  __device__ static void issue_tile(const CUtensorMap* mw, const CUtensorMap*, uint32_t dst, uint32_t,
                                    int t, int n0, uint32_t bar, uint64_t pol) {
    tc::tma_load_2d_hint(dst, mw, t * (kWRow / 4), n0, bar, pol);
  }
  __device__ static void copy_row_plain(const ScalarParams& p, int n, int t, int tg, uint8_t* dst, uint8_t*,
                                        int lane) {
    const uint4* c = reinterpret_cast<const uint4*>(p.W + static_cast<size_t>(n) * p.K + 512 * t);
    for (int i = lane; i < 8 * tg; i += 32) reinterpret_cast<uint4*>(dst)[i] = __ldg(c + i);
  }
  __device__ static constexpr float prescale(int) { return 1.0f; }
  static constexpr bool kOffset = false;
  static constexpr float kOutScale = 1.0f;
  __device__ static void decode(const ScalarParams& p, int n, int t, int sg, const uint8_t* sW, const uint8_t*,
                                Seg& g) {
    const uint4 c = *reinterpret_cast<const uint4*>(sW + 16 * sg);
    const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      g.w[2 * i] = f16x2_to_float2(e4m3x2_to_f16x2(w4[i] & 0xFFFFu));
      g.w[2 * i + 1] = f16x2_to_float2(e4m3x2_to_f16x2(w4[i] >> 16));
    }
    const int kb = p.K >> 7;
    g.s = __ldg(static_cast<const float*>(p.scales) + static_cast<size_t>(n >> 7) * kb + t * 4 + (sg >> 3));
  }
};

cudaError_t launch_w8a16_gemm(const GemvArgs& a, cudaStream_t s) {
  return launch_scalar_dispatch<W8Fmt, true>(a, s);
}

}  // namespace wqp
