// W4A16 scalar-FMA GEMV: E2M1 codes with one E4M3 scale per 16 K and one FP32
// per-tensor scale ("spark_model/layers/w4a16_gemv_tiers.rs", module docs: the
// NVFP4 batched GEMV family with one specialisation per M).
#include "decode.cuh"
#include "gemv_scalar.cuh"

namespace wqp {

struct W4Fmt {
  static constexpr int kTK = 512;                  // 4 groups per stage
  static constexpr int kWRow = 256 + 32;           // codes + E4M3 scales of 512 K
  // Scale rows start at n * K/16: 16-byte aligned for every n iff K % 256 == 0
  // (which also makes every tile's 8 * tg scale bytes a multiple of 16).
  static bool bulk_ok(int K) { return K % 256 == 0; }
  __device__ static uint32_t row_tile_bytes(int tg) { return 64u * tg + 8u * tg; }
  __device__ static void issue_row_bulk(const ScalarParams& p, int n, int t, int tg, uint32_t dst,
                                        uint32_t bar, uint64_t pol) {
    const size_t K = static_cast<size_t>(p.K);
    bulk_g2s_stream(dst, p.W + n * (K / 2) + 256 * t, 64u * tg, bar, pol);
    bulk_g2s_stream(dst + 256, static_cast<const uint8_t*>(p.scales) + n * (K / 16) + 32 * t,
                    8u * tg, bar, pol);
  }
  __device__ static void copy_row_plain(const ScalarParams& p, int n, int t, int tg, uint8_t* dst,
                                        int lane) {
    const size_t K = static_cast<size_t>(p.K);
    const uint32_t* c = reinterpret_cast<const uint32_t*>(p.W + n * (K / 2) + 256 * t);
    for (int i = lane; i < 16 * tg; i += 32) reinterpret_cast<uint32_t*>(dst)[i] = __ldg(c + i);
    const uint32_t* sc =
        reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(p.scales) + n * (K / 16) + 32 * t);
    for (int i = lane; i < 2 * tg; i += 32) reinterpret_cast<uint32_t*>(dst + 256)[i] = __ldg(sc + i);
  }
  __device__ static constexpr float prescale(int) { return 1.0f; }
  // Segment sg = K elements [16 sg, 16 sg + 16) of the tile: 8 code bytes and
  // the one E4M3 scale of that 16-group.
  __device__ static void decode(const ScalarParams& p, int, int, int sg, const uint8_t* sW, Seg& g) {
    const uint2 c = *reinterpret_cast<const uint2*>(sW + 8 * sg);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      g.w[i] = f16x2_to_float2(e2m1x2_to_f16x2((c.x >> (8 * i)) & 0xFFu));
      g.w[4 + i] = f16x2_to_float2(e2m1x2_to_f16x2((c.y >> (8 * i)) & 0xFFu));
    }
    g.s = e4m3_to_f32(sW[256 + sg]) * p.gscale;
  }
};

cudaError_t launch_w4a16_gemv(const GemvArgs& a, cudaStream_t s) {
  return W4Fmt::bulk_ok(a.K) ? launch_scalar_dispatch<W4Fmt, true>(a, s)
                             : launch_scalar_dispatch<W4Fmt, false>(a, s);
}

}  // namespace wqp
