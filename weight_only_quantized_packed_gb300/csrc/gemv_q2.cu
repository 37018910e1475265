// Ternary Q2_0 scalar-FMA GEMV ("spark_model/layers/ops/gemv_q2_vec.rs":
// docs of `q2_0_gemv_vec` / `q2_0_gemv_vec_batchm`, test helper `gemv_row`).
#include "decode.cuh"
#include "gemv_scalar.cuh"

namespace wqp {

struct Q2Fmt {
  static constexpr int kTK = 1024;                 // 8 groups per stage
  static constexpr int kWRow = 8 * 34;             // 8 blocks x 34 bytes
  static constexpr int kW2Row = 0;
  // A row is 34 * K/128 bytes: a multiple of 16 (as tensor maps need) iff
  // K/128 is a multiple of 8.
  static bool bulk_ok(int K) { return (K / 128) % 8 == 0; }
  static cudaError_t make_maps(const GemvArgs& a, CUtensorMap* mw, CUtensorMap*) {
    const uint64_t row = 34ull * (a.K / 128);
    return make_rows_map(mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.W, row / 4, a.N, row, kWRow / 4, kRows);
  }
  __device__ static void issue_tile(const CUtensorMap* mw, const CUtensorMap*, uint32_t dst, uint32_t,
                                    int t, int n0, uint32_t bar, uint64_t pol) {
    tc::tma_load_2d_hint(dst, mw, t * (kWRow / 4), n0, bar, pol);
  }
  __device__ static void copy_row_plain(const ScalarParams& p, int n, int t, int tg, uint8_t* dst, uint8_t*,
                                        int lane) {
    const size_t G = static_cast<size_t>(p.K >> 7);
    const uint16_t* src = reinterpret_cast<const uint16_t*>(p.W + (n * G + 8 * t) * 34);
    uint16_t* d = reinterpret_cast<uint16_t*>(dst);
    for (int i = lane; i < 17 * tg; i += 32) d[i] = __ldg(src + i);
  }
  // The activation at position p of a 16-K segment is pre-scaled by
  // 2^80 over the decoded weight's position factor (see q2_decode_sub), so
  // each product is c * a * 2^-69; each segment's sum starts from its
  // offset -2^-69 * sum a (the -1 of every code), and the output is scaled
  // back by 2^69. The pre-scaled activations stay finite for |a| < 2^48, and
  // the products stay normal for |a| >= 2^-57.
  static constexpr bool kOffset = true;
  static constexpr float kOutScale = 590295810358705651712.0f;   // 2^69
  __device__ static constexpr float prescale(int pos) {
    return 1208925819614629174706176.0f / q2_pos_weight(pos);   // 2^80 / factor
  }
  // 2^-69 * (sum of the 16 activations in v0, v1), added in a fixed tree.
  __device__ static float seg_offset(uint4 v0, uint4 v1) {
    const float2 p0 = __fadd2_rn(make_float2(bf16lo(v0.x), bf16hi(v0.x)), make_float2(bf16lo(v0.y), bf16hi(v0.y)));
    const float2 p1 = __fadd2_rn(make_float2(bf16lo(v0.z), bf16hi(v0.z)), make_float2(bf16lo(v0.w), bf16hi(v0.w)));
    const float2 p2 = __fadd2_rn(make_float2(bf16lo(v1.x), bf16hi(v1.x)), make_float2(bf16lo(v1.y), bf16hi(v1.y)));
    const float2 p3 = __fadd2_rn(make_float2(bf16lo(v1.z), bf16hi(v1.z)), make_float2(bf16lo(v1.w), bf16hi(v1.w)));
    const float2 q = __fadd2_rn(__fadd2_rn(p0, p1), __fadd2_rn(p2, p3));
    return (q.x + q.y) * 1.6940658945086007e-21f;                  // 2^-69
  }
  // Segment sg of a tile = word (sg % 8) of block (sg / 8): K offset 16 * sg.
  __device__ static void decode(const ScalarParams&, int, int, int sg, const uint8_t* sW, const uint8_t*,
                                Seg& g) {
    const uint8_t* blk = sW + (sg >> 3) * 34;
    q2_decode_sub(q2_code_word(blk, sg & 7), g.w);
    g.s = q2_scale(blk);
  }
};

cudaError_t launch_q2_gemv(const GemvArgs& a, cudaStream_t s) {
  return Q2Fmt::bulk_ok(a.K) ? launch_scalar_dispatch<Q2Fmt, true>(a, s)
                             : launch_scalar_dispatch<Q2Fmt, false>(a, s);
}

}  // namespace wqp
