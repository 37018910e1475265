// W4A16 scalar-FMA GEMV: E2M1 codes with one E4M3 scale per 16 K and one FP32
// per-tensor scale ("spark_model/layers/w4a16_gemv_tiers.rs", module docs: the
// NVFP4 batched GEMV family with one specialisation per M).
#include "decode.cuh"
#include "gemv_scalar.cuh"

namespace wqp {

struct W4Fmt {
  static constexpr int kTK = 1024;                 // 8 groups per stage
  static constexpr int kWRow = 512;                // code bytes of 1024 K
  static constexpr int kW2Row = 64;                // E4M3 scale bytes of 1024 K
  // Scale rows are K/16 bytes: a multiple of 16 iff K % 256 == 0.
  static bool bulk_ok(int K) { return K % 256 == 0; }
  static cudaError_t make_maps(const GemvArgs& a, CUtensorMap* mw, CUtensorMap* ms) {
    const uint64_t K = static_cast<uint64_t>(a.K);
    cudaError_t e = make_rows_map(mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, K / 8, a.N, K / 2, kWRow / 4, kRows);
    if (e != cudaSuccess) return e;
    return make_rows_map(ms, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.scales, K / 64, a.N, K / 16, kW2Row / 4, kRows);
  }
  __device__ static void issue_tile(const CUtensorMap* mw, const CUtensorMap* ms, uint32_t dst,
                                    uint32_t dst2, int t, int n0, uint32_t bar, uint64_t pol) {
    tc::tma_load_2d_hint(dst, mw, t * (kWRow / 4), n0, bar, pol);
    tc::tma_load_2d_hint(dst2, ms, t * (kW2Row / 4), n0, bar, pol);
  }
  __device__ static void copy_row_plain(const ScalarParams& p, int n, int t, int tg, uint8_t* dst,
                                        uint8_t* dst2, int lane) {
    const size_t K = static_cast<size_t>(p.K);
    const uint32_t* c = reinterpret_cast<const uint32_t*>(p.W + n * (K / 2) + kWRow * t);
    for (int i = lane; i < 16 * tg; i += 32) reinterpret_cast<uint32_t*>(dst)[i] = __ldg(c + i);
    const uint16_t* sc =
        reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(p.scales) + n * (K / 16) + kW2Row * t);
    for (int i = lane; i < 4 * tg; i += 32) reinterpret_cast<uint16_t*>(dst2)[i] = __ldg(sc + i);
  }
  __device__ static constexpr float prescale(int) { return 1.0f; }
  static constexpr bool kOffset = false;
  static constexpr float kOutScale = 1.0f;
  // Segment sg = K elements [16 sg, 16 sg + 16) of the tile: 8 code bytes and
  // the one E4M3 scale of that 16-group.
  __device__ static void decode(const ScalarParams& p, int, int, int sg, const uint8_t* sW,
                                const uint8_t* sW2, Seg& g) {
    const uint2 c = *reinterpret_cast<const uint2*>(sW + 8 * sg);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      g.w[i] = f16x2_to_float2(e2m1x2_to_f16x2((c.x >> (8 * i)) & 0xFFu));
      g.w[4 + i] = f16x2_to_float2(e2m1x2_to_f16x2((c.y >> (8 * i)) & 0xFFu));
    }
    g.s = e4m3_to_f32(sW2[sg]) * p.gscale;
  }
};

cudaError_t launch_w4a16_gemv(const GemvArgs& a, cudaStream_t s) {
  return W4Fmt::bulk_ok(a.K) ? launch_scalar_dispatch<W4Fmt, true>(a, s)
                             : launch_scalar_dispatch<W4Fmt, false>(a, s);
}

}  // namespace wqp
