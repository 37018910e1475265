// Scalar-FMA packed GEMV: C[M, N] = A[M, K] @ dequant(W)^T for one weight
// format, with exact-M specialisation (M = 1..16, one template instance per M).
//
// Thread map (after "spark_model/layers/ops/gemv_q2_vec.rs", doc of
// `q2_0_gemv_vec`: one warp per output row, eight rows per CTA):
//   warps 0..7  consumers: warp w owns output row n0 + w and keeps M FP32
//               accumulators, so every weight word is read once for all M rows
//               (doc of `q2_0_gemv_vec_batchm`);
//   warp 8      producer: one lane streams the CTA's 8-row weight slab and
//               the M activation rows through a STAGES-deep shared-memory ring
//               of K tiles with non-multicast bulk copies (cp.async.bulk) and
//               mbarriers. Odd shapes whose rows are not 16-byte aligned use
//               plain loads by the whole producer warp instead.
//
// Per-row arithmetic (identical for every M, so a batched row equals the M = 1
// row bit for bit): for each 16-weight segment a lane owns, two FP32 chains
// (k = 0..7 and k = 8..15 of the segment) of fma(a_bf16, w_bf16) are added,
// the segment's scale is folded with one FP32 fma onto the lane accumulator,
// and the 32 lanes are summed by a fixed xor-butterfly. The order of the
// segments, of the K tiles and of the butterfly depends only on N and K.
// Weights are converted exactly to BF16 (every Q2_0/E2M1/E4M3 value is a BF16
// value), activations stay BF16, and fma.rn.f32.bf16 forms the exact product
// with a single FP32 rounding of the sum.
#pragma once
#include "common.cuh"

namespace wqp {

constexpr int kRows = 8;             // output rows per CTA (one consumer warp each)
constexpr int kConsumers = kRows * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kTileK = 1024;         // K elements per ring stage
constexpr int kSegsPerTile = kTileK / 16;

// fma.rn.f32.bf16 with explicit operand halves: fma_XY(a2, b2, c) =
// a2.X * b2.Y + c, X/Y in {l, h} (low / high BF16 of the 32-bit register).
__device__ __forceinline__ float fma_ll(uint32_t a2, uint32_t b2, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_hh(uint32_t a2, uint32_t b2, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_lh(uint32_t a2, uint32_t b2, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bh, %3;\n\t}"
      : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_hl(uint32_t a2, uint32_t b2, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bl, %3;\n\t}"
      : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
  return d;
}

// A segment of 16 consecutive weights w[0..15] decoded to BF16 pairs, plus
// the segment's scale. Natural layout: p[i] = (lo: w[2i], hi: w[2i+1]).
// J8 layout (Q2_0 decode): p[j] = (lo: w[j], hi: w[j+8]).
struct Seg {
  uint32_t p[8];
  float s;
};

// Dot products of one decoded segment with the M activation rows' matching
// 16 BF16 values (a[m][0..15] at sA + m * lda_s), folded onto acc[m]. Chain
// c0 runs over k = 0..7 and c1 over k = 8..15, both in ascending k.
template <int M, bool J8>
__device__ __forceinline__ void seg_fma(const Seg& g, const uint16_t* sA, int lda_s, float* acc) {
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(sA + m * lda_s);
    const uint4 a1 = *reinterpret_cast<const uint4*>(sA + m * lda_s + 8);
    float c0 = 0.0f, c1 = 0.0f;
    if (!J8) {
      c0 = fma_ll(a0.x, g.p[0], c0);
      c0 = fma_hh(a0.x, g.p[0], c0);
      c0 = fma_ll(a0.y, g.p[1], c0);
      c0 = fma_hh(a0.y, g.p[1], c0);
      c0 = fma_ll(a0.z, g.p[2], c0);
      c0 = fma_hh(a0.z, g.p[2], c0);
      c0 = fma_ll(a0.w, g.p[3], c0);
      c0 = fma_hh(a0.w, g.p[3], c0);
      c1 = fma_ll(a1.x, g.p[4], c1);
      c1 = fma_hh(a1.x, g.p[4], c1);
      c1 = fma_ll(a1.y, g.p[5], c1);
      c1 = fma_hh(a1.y, g.p[5], c1);
      c1 = fma_ll(a1.z, g.p[6], c1);
      c1 = fma_hh(a1.z, g.p[6], c1);
      c1 = fma_ll(a1.w, g.p[7], c1);
      c1 = fma_hh(a1.w, g.p[7], c1);
    } else {
      c0 = fma_ll(a0.x, g.p[0], c0);
      c0 = fma_hl(a0.x, g.p[1], c0);
      c0 = fma_ll(a0.y, g.p[2], c0);
      c0 = fma_hl(a0.y, g.p[3], c0);
      c0 = fma_ll(a0.z, g.p[4], c0);
      c0 = fma_hl(a0.z, g.p[5], c0);
      c0 = fma_ll(a0.w, g.p[6], c0);
      c0 = fma_hl(a0.w, g.p[7], c0);
      c1 = fma_lh(a1.x, g.p[0], c1);
      c1 = fma_hh(a1.x, g.p[1], c1);
      c1 = fma_lh(a1.y, g.p[2], c1);
      c1 = fma_hh(a1.y, g.p[3], c1);
      c1 = fma_lh(a1.z, g.p[4], c1);
      c1 = fma_hh(a1.z, g.p[5], c1);
      c1 = fma_lh(a1.w, g.p[6], c1);
      c1 = fma_hh(a1.w, g.p[7], c1);
    }
    acc[m] = fmaf(c0 + c1, g.s, acc[m]);
  }
}

// Kernel parameters (passed by value).
struct ScalarParams {
  const uint16_t* A;
  const uint8_t* W;
  const void* scales;
  uint16_t* C;
  int N, K, lda, ldc;
  float gscale;
  unsigned* err;
};

// Format traits interface (see gemv_q2.cu, gemv_w4.cu, gemv_w8.cu):
//   static constexpr int kWBytesPerRow;          // bytes of one row's full K tile in smem
//   static bool bulk_ok(int K);                  // host: bulk-copy fast path allowed
//   __device__ static uint32_t row_tile_bytes(int K, int tile, int segs);   // bytes copied per row
//   __device__ static void issue_row_bulk(...)   // producer lane: bulk copy one row's tile
//   __device__ static void copy_row_plain(...)   // producer warp: plain-load copy
//   __device__ static void decode(...)           // consumer: one segment -> Seg

template <class F, int M, bool BULK>
__global__ void __launch_bounds__(kThreads) gemv_scalar_kernel(ScalarParams p) {
  constexpr int kStages = (M <= 4) ? 6 : (M <= 8 ? 4 : 3);
  constexpr int kWStage = kRows * F::kWBytesPerRow;                  // weight bytes per stage
  constexpr int kAStage = M * kTileK * 2;                           // activation bytes per stage
  constexpr int kStageBytes = ((kWStage + kAStage) + 127) / 128 * 128;

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kRows;
  const int rows = min(kRows, p.N - n0);
  const int K = p.K;
  const int G = K >> 7;                                   // 128-wide groups per row
  const int tiles = (K + kTileK - 1) / kTileK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kRows);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kRows) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < tiles && ok; ++t) {
      const int s = t % kStages;
      if (t >= kStages) {
        uint32_t done = 0;
        if (lane == 0) done = mbar_wait(smem_u32(&empty_bar[s]), ((t / kStages) - 1) & 1, p.err);
        done = __shfl_sync(0xFFFFFFFFu, done, 0);
        if (!done) { ok = false; break; }
      }
      const int tg = min(8, G - t * 8);                    // groups in this tile
      uint8_t* sW = smem + s * kStageBytes;
      uint8_t* sAs = sW + kWStage;
      const uint32_t wrow = F::row_tile_bytes(K, t, tg);
      const uint32_t abytes = static_cast<uint32_t>(tg) * 128 * 2;
      const uint32_t fb = smem_u32(&full_bar[s]);
      if (!BULK) {
        for (int r = 0; r < rows; ++r) F::copy_row_plain(p, n0 + r, t, tg, sW + r * F::kWBytesPerRow, lane);
        __threadfence_block();
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t tx = (BULK ? wrow * rows : 0u) + abytes * M;
        mbar_arrive_expect_tx(fb, tx);
        if (BULK)
          for (int r = 0; r < rows; ++r) F::issue_row_bulk(p, n0 + r, t, tg, smem_u32(sW + r * F::kWBytesPerRow), fb, pol);
        if (t == 0) pdl_wait();            // activations may come from the previous kernel
        for (int m = 0; m < M; ++m)
          bulk_g2s(smem_u32(sAs + m * kTileK * 2), p.A + static_cast<size_t>(m) * p.lda + t * kTileK, abytes, fb);
      }
      issued = t + 1;
    }
    // Drain: never leave the CTA with bulk copies still writing its smem.
    if (lane == 0)
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(smem_u32(&full_bar[t % kStages]), (t / kStages) & 1, p.err);
    return;
  }

  // -------------------------------------------------------------- consumers
  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.0f;
  const bool live = warp < rows;
  const int n = n0 + warp;
  bool ok = true;
  for (int t = 0; t < tiles; ++t) {
    const int s = t % kStages;
    // Every lane waits (acquire), and the warp agrees on the outcome, so a
    // timeout never splits the warp before the __syncwarp below.
    const bool got = mbar_wait(smem_u32(&full_bar[s]), (t / kStages) & 1, p.err);
    if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }
    const int tg = min(8, G - t * 8);
    const int segs = tg * 8;
    const uint8_t* sW = smem + s * kStageBytes + warp * F::kWBytesPerRow;
    const uint16_t* sAs = reinterpret_cast<const uint16_t*>(smem + s * kStageBytes + kWStage);
    if (live) {
      for (int sg = lane; sg < segs; sg += 32) {
        Seg g;
        F::decode(p, n, t, sg, sW, g);
        seg_fma<M, F::kJ8>(g, sAs + sg * 16, kTileK, acc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
  }
  if (!ok || !live) return;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float v = warp_sum(acc[m]);
    if (lane == m) p.C[static_cast<size_t>(m) * p.ldc + n] = f32_to_bf16_rn(v);
  }
}

template <class F, int M, bool BULK>
constexpr int scalar_smem_bytes() {
  constexpr int kStages = (M <= 4) ? 6 : (M <= 8 ? 4 : 3);
  constexpr int kWStage = kRows * F::kWBytesPerRow;
  constexpr int kAStage = M * kTileK * 2;
  return kStages * (((kWStage + kAStage) + 127) / 128 * 128);
}

template <class F, int M, bool BULK>
cudaError_t launch_scalar_m(const GemvArgs& a, cudaStream_t s) {
  auto kern = gemv_scalar_kernel<F, M, BULK>;
  constexpr int smem = scalar_smem_bytes<F, M, BULK>();
  static bool attr_set = false;  // idempotent; racing writers set the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ScalarParams p;
  p.A = static_cast<const uint16_t*>(a.A);
  p.W = static_cast<const uint8_t*>(a.W);
  p.scales = a.scales;
  p.C = static_cast<uint16_t*>(a.C);
  p.N = a.N;
  p.K = a.K;
  p.lda = a.lda;
  p.ldc = a.ldc;
  p.gscale = a.gscale;
  p.err = a.err;
  dim3 grid((a.N + kRows - 1) / kRows);
  return launch(kern, grid, dim3(kThreads), smem, s, a.pdl, p);
}

template <class F, bool BULK>
cudaError_t launch_scalar_dispatch(const GemvArgs& a, cudaStream_t s) {
  switch (a.M) {
    case 1: return launch_scalar_m<F, 1, BULK>(a, s);
    case 2: return launch_scalar_m<F, 2, BULK>(a, s);
    case 3: return launch_scalar_m<F, 3, BULK>(a, s);
    case 4: return launch_scalar_m<F, 4, BULK>(a, s);
    case 5: return launch_scalar_m<F, 5, BULK>(a, s);
    case 6: return launch_scalar_m<F, 6, BULK>(a, s);
    case 7: return launch_scalar_m<F, 7, BULK>(a, s);
    case 8: return launch_scalar_m<F, 8, BULK>(a, s);
    case 9: return launch_scalar_m<F, 9, BULK>(a, s);
    case 10: return launch_scalar_m<F, 10, BULK>(a, s);
    case 11: return launch_scalar_m<F, 11, BULK>(a, s);
    case 12: return launch_scalar_m<F, 12, BULK>(a, s);
    case 13: return launch_scalar_m<F, 13, BULK>(a, s);
    case 14: return launch_scalar_m<F, 14, BULK>(a, s);
    case 15: return launch_scalar_m<F, 15, BULK>(a, s);
    case 16: return launch_scalar_m<F, 16, BULK>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wqp
