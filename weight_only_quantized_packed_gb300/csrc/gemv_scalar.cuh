// Scalar-FMA packed GEMV: C[M, N] = A[M, K] @ dequant(W)^T for one weight
// format, with exact-M specialisation (M = 1..16, one template instance per M).
//
// Thread map (after "spark_model/layers/ops/gemv_q2_vec.rs", doc of
// `q2_0_gemv_vec`, and the register-tiled T=2 tier of
// "spark_model/layers/w4a16_gemv_tiers.rs", doc of `resolve`):
//   warps 0..8  consumers: warp w owns output rows n0 + 2w and n0 + 2w + 1
//               and keeps M FP32 accumulator pairs per row, so every weight
//               word is read once for all M rows (doc of
//               `q2_0_gemv_vec_batchm`) and every activation load serves two
//               weight rows;
//   warp 9      producer: streams the CTA's 18-row weight slab through a
//               STAGES-deep ring of K tiles, one 2-D tensor-map copy
//               (cp.async.bulk.tensor) per tile (rows past N and K past the
//               end are zero-filled). If the weight rows are not 16-byte
//               aligned, the producer warp copies them with plain loads.
// Activations are widened to FP32 in shared memory (XOR-swizzled, with the
// format's per-position pre-scale). When M * K * 4 bytes fit (ARES), the
// consumers widen all of A once, straight from global memory, while the first
// weight tiles are in flight; afterwards each warp waits only on weight
// tiles. Otherwise the producer also copies each tile's M BF16 activation
// rows, and the consumers widen them tile by tile behind a named barrier.
//
// Per-row arithmetic (identical for every M, so a batched row equals the M = 1
// row bit for bit): weights are decoded to exact FP32 values (Q2_0: the code
// times a power of two, and the chain of each segment starts from the
// segment's -2^-69 * sum a, computed once when the activations are widened).
// For each 16-weight segment a lane owns, two chains of packed FFMA2
// (k = 0..7 and k = 8..15, even and odd k in the two halves) are added, the segment's scale
// is folded with one FFMA2 onto the lane's accumulator pair, and at the end
// the pair is summed and the 32 lanes reduced by a fixed xor-butterfly. The
// order depends only on N and K, never on M or on the staging path.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace wqp {

constexpr int kWarpsC = 9;                     // consumer warps
constexpr int kRowsPerWarp = 2;
constexpr int kRows = kWarpsC * kRowsPerWarp;  // output rows per CTA
constexpr int kThreads = (kWarpsC + 1) * 32;
constexpr int kAResMaxBytes = 96 * 1024;       // resident FP32 activations, at most

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

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

// A decoded 16-weight segment: w[i] = (w_{2i}, w_{2i+1}) as FP32, plus scale.
struct Seg {
  float2 w[8];
  float s;
};

// Position of the 16-byte chunk j (0..3) of segment sg in an FP32 activation
// row: XOR-swizzled so that the 8 lanes of a shared-memory phase, which read
// 8 consecutive segments, hit 8 distinct bank groups.
__device__ __forceinline__ int fa_chunk(int sg, int j) { return sg * 4 + (j ^ ((sg >> 1) & 3)); }

// Widens 16 BF16 activations (two 16-byte words) to FP32 with the format's
// pre-scale and stores them as segment sg of the FP32 row.
template <class F>
__device__ __forceinline__ void widen_segment(uint4 v0, uint4 v1, float* row, int sg) {
  float4* r4 = reinterpret_cast<float4*>(row);
  r4[fa_chunk(sg, 0)] = make_float4(bf16lo(v0.x) * F::prescale(0), bf16hi(v0.x) * F::prescale(1),
                                    bf16lo(v0.y) * F::prescale(2), bf16hi(v0.y) * F::prescale(3));
  r4[fa_chunk(sg, 1)] = make_float4(bf16lo(v0.z) * F::prescale(4), bf16hi(v0.z) * F::prescale(5),
                                    bf16lo(v0.w) * F::prescale(6), bf16hi(v0.w) * F::prescale(7));
  r4[fa_chunk(sg, 2)] = make_float4(bf16lo(v1.x) * F::prescale(8), bf16hi(v1.x) * F::prescale(9),
                                    bf16lo(v1.y) * F::prescale(10), bf16hi(v1.y) * F::prescale(11));
  r4[fa_chunk(sg, 3)] = make_float4(bf16lo(v1.z) * F::prescale(12), bf16hi(v1.z) * F::prescale(13),
                                    bf16lo(v1.w) * F::prescale(14), bf16hi(v1.w) * F::prescale(15));
}

// Format traits interface (gemv_q2.cu, gemv_w4.cu, gemv_w8.cu):
//   kTK                 K elements per ring stage (multiple of 128)
//   kWRow, kW2Row       weight bytes of one row per stage in the first and
//                       (W4 scales) second block of the stage
//   bulk_ok(K)          host: tensor-map path allowed for this K
//   make_maps(...)      host: tensor maps of the weight block(s)
//   issue_tile(...)     producer lane: tensor-map copies of one K tile
//   copy_row_plain(...) producer warp: plain-load copy of one row's tile
//   prescale(p)         factor applied to a[k] when widened (p = k % 16)
//   kOffset             each 16-K segment's sum starts from -seg_offset(a)
//                       (Q2_0: the -1 of every code), stored when widened
//   kOutScale           factor applied to the FP32 result before the store
//   decode(...)         consumer: one segment of one row -> Seg
template <class F, int M, bool ARES>
struct ScalarCfg {
  static constexpr int kW2Off = kRows * F::kWRow;
  static constexpr int kWStage = (kRows * (F::kWRow + F::kW2Row) + 127) / 128 * 128;
  // Ring depth. With resident activations and M >= 3 the ring is kept near
  // 24 KB, so that two CTAs still fit on an SM beside up to 80 KB of FP32
  // activations each.
  static constexpr int kStages = ARES ? (M <= 2 ? 6 : (kWStage > 8192 ? 2 : 4))
                                      : ((M <= 4) ? 4 : (M <= 8 ? 3 : 2));
  static constexpr bool kFADouble = !ARES && (M <= 4);    // double-buffered per-tile FP32 A
  static constexpr int kAW = F::kTK < 512 ? F::kTK : 512;   // K per activation box
  static constexpr int kAStage = ARES ? 0 : M * F::kTK * 2;
  static constexpr int kStageBytes = ((kWStage + kAStage) + 127) / 128 * 128;
  static constexpr int kFABytes = ARES ? 0 : M * F::kTK * 4;  // one per-tile FP32 buffer
  static constexpr int kOffBytes = (ARES || !F::kOffset) ? 0 : M * (F::kTK / 16) * 4;   // its segment offsets
  static constexpr int kSmemFixed = kStages * kStageBytes + (kFADouble ? 2 : 1) * (kFABytes + kOffBytes);
  // Resident activations: M * K FP32 values, then M * K / 16 segment offsets.
  static constexpr int kSmemMax = kSmemFixed + (ARES ? kAResMaxBytes + (F::kOffset ? kAResMaxBytes / 16 : 0) : 0);
  static constexpr int kMinBlocks = (M <= 8) ? 2 : 1;
  static_assert(kSmemMax <= 227 * 1024, "shared memory budget");
  static_assert(F::kW2Row == 0 || (kRows * F::kWRow) % 128 == 0, "second weight block alignment");
};

template <class F, int M, bool BULK, bool ARES>
__global__ void __launch_bounds__(kThreads, (ScalarCfg<F, M, ARES>::kMinBlocks))
    gemv_scalar_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                       const __grid_constant__ CUtensorMap tmA, ScalarParams p) {
  using Cfg = ScalarCfg<F, M, ARES>;
  constexpr int kStages = Cfg::kStages;
  constexpr int TK = F::kTK;
  constexpr int kSegT = TK / 16;                 // segments per row per full tile

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kRows;
  const int rows = min(kRows, p.N - n0);
  const int K = p.K;
  const int G = K >> 7;                          // 128-wide groups per row
  constexpr int kGT = TK / 128;                  // groups per full tile
  const int tiles = (G + kGT - 1) / kGT;
  float* fA = reinterpret_cast<float*>(smem + kStages * Cfg::kStageBytes);
  const int ldfa = ARES ? K : TK;                // FP32 activation row pitch (floats)
  // Segment offsets (formats with kOffset): after the FP32 activations.
  float* fOff = fA + (ARES ? M * K : (Cfg::kFADouble ? 2 : 1) * M * TK);
  const int ldoff = ldfa / 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kWarpsC);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kWarpsC) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      if (BULK) { tc::prefetch_tmap(&tmW); if (F::kW2Row) tc::prefetch_tmap(&tmW2); }
      if (!ARES) tc::prefetch_tmap(&tmA);
    }
    int issued = 0;
    for (int t = 0; t < tiles; ++t) {
      const int s = t % kStages;
      if (t >= kStages) {
        uint32_t done = 0;
        if (lane == 0) done = mbar_wait(smem_u32(&empty_bar[s]), ((t / kStages) - 1) & 1, p.err);
        done = __shfl_sync(0xFFFFFFFFu, done, 0);
        if (!done) break;
      }
      const int tg = min(kGT, G - t * kGT);      // groups in this tile
      uint8_t* sW = smem + s * Cfg::kStageBytes;
      uint8_t* sAs = sW + Cfg::kWStage;
      const uint32_t fb = smem_u32(&full_bar[s]);
      if (!BULK) {
        for (int r = 0; r < rows; ++r)
          F::copy_row_plain(p, n0 + r, t, tg, sW + r * F::kWRow, sW + Cfg::kW2Off + r * F::kW2Row, lane);
        __threadfence_block();
        __syncwarp();
      }
      if (lane == 0) {
        // Full boxes always land (out-of-range rows and K read as zero).
        const uint32_t tx = (BULK ? kRows * (F::kWRow + F::kW2Row) : 0u) + Cfg::kAStage;
        mbar_arrive_expect_tx(fb, tx);
        if (BULK) F::issue_tile(&tmW, &tmW2, smem_u32(sW), smem_u32(sW + Cfg::kW2Off), t, n0, fb, pol);
        if (!ARES) {
          if (t == 0) pdl_wait();          // activations may come from the previous kernel
#pragma unroll
          for (int bx = 0; bx < TK / Cfg::kAW; ++bx)
            tc::tma_load_2d(smem_u32(sAs + bx * M * Cfg::kAW * 2), &tmA, (t * TK + bx * Cfg::kAW) / 2, 0, fb);
        }
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
  constexpr int kCT = kWarpsC * 32;              // consumer threads
  if (ARES) {
    // Widen all of A once, straight from global memory (it may come from the
    // previous kernel, hence the dependency wait first).
    pdl_wait();
    const int segK = K / 16;
    for (int u = threadIdx.x; u < M * segK; u += kCT) {
      const int m = u / segK;
      const int sg = u - m * segK;
      const uint4* src = reinterpret_cast<const uint4*>(p.A + static_cast<size_t>(m) * p.lda + sg * 16);
      const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
      widen_segment<F>(v0, v1, fA + m * ldfa, sg);
      if constexpr (F::kOffset) fOff[m * ldoff + sg] = F::seg_offset(v0, v1);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory");
  }

  float2 acc[kRowsPerWarp][M];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = make_float2(0.0f, 0.0f);
  const int r0 = warp * kRowsPerWarp;             // first local row of this warp
  bool ok = true;
  for (int t = 0; t < tiles; ++t) {
    const int s = t % kStages;
    // Every lane waits (acquire) and the warp agrees on the outcome, so a
    // timeout never splits the warp. After a timeout the loop keeps running
    // the named barriers (no compute) so other warps never wait for ever.
    if (ok) {
      const bool got = mbar_wait(smem_u32(&full_bar[s]), (t / kStages) & 1, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) ok = false;
    }
    const int tg = min(kGT, G - t * kGT);
    const int segs = tg * 8;
    const uint8_t* sW = smem + s * Cfg::kStageBytes;
    const float* fAt;
    const float* fOt;
    int sg0;                                      // segment offset of this tile in fAt
    if (ARES) {
      fAt = fA;
      fOt = fOff;
      sg0 = t * kSegT;
    } else {
      const uint16_t* sAs = reinterpret_cast<const uint16_t*>(sW + Cfg::kWStage);
      float* fAw = fA + (Cfg::kFADouble ? (t & 1) * (M * TK) : 0);
      float* fOw = fOff + (Cfg::kFADouble ? (t & 1) * (M * kSegT) : 0);
      fAt = fAw;
      fOt = fOw;
      sg0 = 0;
      // With a single FP32 buffer, wait until every warp is done with the
      // previous tile before overwriting it.
      if (!Cfg::kFADouble && t > 0) asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory");
      if (ok) {
        for (int u = threadIdx.x; u < M * segs; u += kCT) {
          const int m = u / segs;
          const int sg = u - m * segs;
          // Activation tile layout: boxes of kAW K, each [M rows x kAW].
          const int k0 = sg * 16;
          const uint4* src = reinterpret_cast<const uint4*>(
              sAs + (k0 / Cfg::kAW) * (M * Cfg::kAW) + m * Cfg::kAW + (k0 % Cfg::kAW));
          const uint4 v0 = src[0], v1 = src[1];
          widen_segment<F>(v0, v1, fAw + m * ldfa, sg);
          if constexpr (F::kOffset) fOw[m * ldoff + sg] = F::seg_offset(v0, v1);
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory");
    }
    if (ok) {
      for (int sg = lane; sg < segs; sg += 32) {
        Seg g[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          // A row past N decodes the last valid row instead (no branch; its
          // sums are never stored).
          const int rr = min(r0 + r, rows - 1);
          F::decode(p, n0 + rr, t, sg, sW + rr * F::kWRow, sW + Cfg::kW2Off + rr * F::kW2Row, g[r]);
        }
        const int sa = sg0 + sg;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const float4* row = reinterpret_cast<const float4*>(fAt + m * ldfa);
          const float4 q0 = row[fa_chunk(sa, 0)], q1 = row[fa_chunk(sa, 1)];
          const float4 q2 = row[fa_chunk(sa, 2)], q3 = row[fa_chunk(sa, 3)];
          const float2 a[8] = {make_float2(q0.x, q0.y), make_float2(q0.z, q0.w),
                               make_float2(q1.x, q1.y), make_float2(q1.z, q1.w),
                               make_float2(q2.x, q2.y), make_float2(q2.z, q2.w),
                               make_float2(q3.x, q3.y), make_float2(q3.z, q3.w)};
          float2 c00 = make_float2(0.f, 0.f);     // where each row's chain starts
          if constexpr (F::kOffset) c00.x = -fOt[m * ldoff + sa];
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            float2 c0 = F::kOffset ? __ffma2_rn(a[0], g[r].w[0], c00) : __fmul2_rn(a[0], g[r].w[0]);
            float2 c1 = __fmul2_rn(a[4], g[r].w[4]);
            c0 = __ffma2_rn(a[1], g[r].w[1], c0);
            c1 = __ffma2_rn(a[5], g[r].w[5], c1);
            c0 = __ffma2_rn(a[2], g[r].w[2], c0);
            c1 = __ffma2_rn(a[6], g[r].w[6], c1);
            c0 = __ffma2_rn(a[3], g[r].w[3], c0);
            c1 = __ffma2_rn(a[7], g[r].w[7], c1);
            acc[r][m] = __ffma2_rn(__fadd2_rn(c0, c1), f2(g[r].s), acc[r][m]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
  }
  if (!ok) return;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int n = n0 + r0 + r;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float v = warp_sum(acc[r][m].x + acc[r][m].y);
      if (lane == m && r0 + r < rows) p.C[static_cast<size_t>(m) * p.ldc + n] = f32_to_bf16_rn(v * F::kOutScale);
    }
  }
}

// Host: tensor map of the activation rows, viewed as u32 pairs of BF16.
cudaError_t make_act_map(CUtensorMap* m, const GemvArgs& a, int box_k);
// Host: 2-D tensor map (rows x bytes) of a weight or scale block, shared by
// the format traits; cached per process like the tensor-core engines' maps.
cudaError_t make_rows_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);

template <class F, int M, bool BULK, bool ARES>
cudaError_t launch_scalar_m(const GemvArgs& a, cudaStream_t s) {
  using Cfg = ScalarCfg<F, M, ARES>;
  auto kern = gemv_scalar_kernel<F, M, BULK, ARES>;
  static AttrLatch latch;
  if (cudaError_t e0 = set_smem_attrs(kern, latch, Cfg::kSmemMax, false); e0 != cudaSuccess) return e0;
  const int smem = Cfg::kSmemFixed + (ARES ? M * a.K * 4 + (F::kOffset ? M * (a.K / 16) * 4 : 0) : 0);
  CUtensorMap mw = {}, mw2 = {}, ma = {};
  cudaError_t e = cudaSuccess;
  if (!ARES && (e = make_act_map(&ma, a, Cfg::kAW)) != cudaSuccess) return e;
  if (BULK && (e = F::make_maps(a, &mw, &mw2)) != cudaSuccess) return e;
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
  return launch(kern, grid, dim3(kThreads), smem, s, a.pdl, mw, mw2, ma, p);
}

template <class F, int M, bool BULK>
cudaError_t launch_scalar_m2(const GemvArgs& a, cudaStream_t s) {
  // Keep A resident when it fits; the per-tile path otherwise.
  if (static_cast<long long>(M) * a.K * 4 <= kAResMaxBytes) return launch_scalar_m<F, M, BULK, true>(a, s);
  return launch_scalar_m<F, M, BULK, false>(a, s);
}

template <class F, bool BULK>
cudaError_t launch_scalar_dispatch(const GemvArgs& a, cudaStream_t s) {
  switch (a.M) {
    case 1: return launch_scalar_m2<F, 1, BULK>(a, s);
    case 2: return launch_scalar_m2<F, 2, BULK>(a, s);
    case 3: return launch_scalar_m2<F, 3, BULK>(a, s);
    case 4: return launch_scalar_m2<F, 4, BULK>(a, s);
    case 5: return launch_scalar_m2<F, 5, BULK>(a, s);
    case 6: return launch_scalar_m2<F, 6, BULK>(a, s);
    case 7: return launch_scalar_m2<F, 7, BULK>(a, s);
    case 8: return launch_scalar_m2<F, 8, BULK>(a, s);
    case 9: return launch_scalar_m2<F, 9, BULK>(a, s);
    case 10: return launch_scalar_m2<F, 10, BULK>(a, s);
    case 11: return launch_scalar_m2<F, 11, BULK>(a, s);
    case 12: return launch_scalar_m2<F, 12, BULK>(a, s);
    case 13: return launch_scalar_m2<F, 13, BULK>(a, s);
    case 14: return launch_scalar_m2<F, 14, BULK>(a, s);
    case 15: return launch_scalar_m2<F, 15, BULK>(a, s);
    case 16: return launch_scalar_m2<F, 16, BULK>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wqp
