// W4A16 GEMM on the warp-level tensor cores for shapes of fewer than two
// 64-row tiles per SM and at most 8 stages of 1024 K: one short CTA per
// (64-row tile, 1024-K stage), three CTAs per SM, 8 activation rows per
// launch. The larger shapes run on the persistent kernel of gemm_mma_f16.cu.
//
// What it computes is the batched W4A16 GEMV of
// "spark_model/layers/w4a16_gemv_tiers.rs" (module docs) with the reading
// w = e2m1(nibble) * e4m3(scale[n, k/16]) and one FP32 per-tensor scale g on
// each FP32 result, with the exact FP16 operands of gemm_mma_f16.cu: the
// weight e2m1 * e4m3 is an FP16 value, the activations are scaled per
// (activation row, 128-K block) by a power of two and rounded to FP16, and
// each block's FP32 sum is multiplied back by 2^-e once.
//
// CTA: 64 weight rows x one stage (8 blocks of 128 K: one 3-D copy of 8
// blocks x 64 rows x 64 bytes of codes and one box of 64 rows x 64 bytes of
// E4M3 scales, by TMA); 8 compute warps (warp w owns block w for all four 16-row tiles) and
// one TMA warp. A cluster of one CTA per stage splits K; ranks >= 1 send their
// sums to rank 0 with st.async and leave at once (their SM slots go to the
// next call's CTAs), rank 0 adds them in rank order and stores. With 8
// activation rows the TMA warp copies the stage's activation rows in bulk
// after the grid-dependency wait; with fewer each compute warp loads its
// block's activations itself (faster up to 7 rows: 5.57 -> 5.23 us at M = 5).
#include <atomic>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "mma_f16.cuh"
#include "tc.cuh"

namespace wqp {
namespace mmaw4s {

using namespace f16op;

constexpr int BM = 64;
constexpr int kTiles = 4;
constexpr int kCompute = 8;
constexpr int kThreads = (kCompute + 1) * 32;
constexpr int kBlocks = 8;
constexpr int kMaxSplits = 8;
constexpr int kBoxBytes = BM * 64;                       // codes of one block
constexpr int kScaleOff = kBlocks * kBoxBytes;           // 32768
constexpr int kStageBytes = kScaleOff + BM * 64;         // 36864
constexpr int kSlot = kTiles * 32 * 16;                  // one warp's (and one rank's) sums: 2 KB
constexpr int kActOff = kStageBytes;
constexpr int kActPitch = kBlocks * 128 * 2 + 16;        // 16-byte pad spreads the rows over the banks
constexpr int kRecvOff = kActOff + 8 * kActPitch;

constexpr int smem_bytes(int splits) { return kRecvOff + (splits - 1) * kSlot; }
static_assert(kCompute * kSlot <= kStageBytes, "the warps' sums overlay the consumed stage");
static_assert(kRecvOff % 16 == 0 && 3 * (smem_bytes(kMaxSplits) + 1024) <= 228 * 1024, "shared memory");

struct Params {
  const uint16_t* A;   // bf16 [M, lda]
  uint16_t* C;         // bf16 [M, ldc]
  int lda, ldc;
  int M, N;
  float gscale;
  int splits;          // = stages (one stage per CTA)
  unsigned* err;
};

__global__ void __launch_bounds__(kThreads, 3)
    w4_short_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[3];   // stage landed, partial sums received, activation rows landed
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits;
  const int tile = blockIdx.x / S;
  const int rank = blockIdx.x - tile * S;       // == %cluster_ctarank == the CTA's stage
  const int n0 = tile * BM;
  const uint32_t full = smem_u32(&bars[0]), recv_bar = full + 8, act_bar = full + 16;
  const bool bulk_act = p.M > 7;

  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    mbar_init(recv_bar, 1);
    mbar_init(act_bar, 1);
    mbar_fence_init();
    if (rank == 0 && S > 1) mbar_arrive_expect_tx(recv_bar, (S - 1) * kSlot);
    abort_sh = 0;
  }
  if (S > 1) tc::cluster_arrive_relaxed();
  __syncthreads();
  pdl_launch_dependents();

  const int g = lane >> 2, t4 = lane & 3;
  if (warp == kCompute) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tmW);
      tc::prefetch_tmap(&tmS);
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(full, kStageBytes);
      tc::tma_load_3d_hint(smem_u32(smem), &tmW, 0, n0, rank * kBlocks, full, pol);   // the stage's 8 blocks
      tc::tma_load_2d_hint(smem_u32(smem + kScaleOff), &tmS, rank * 64, n0, full, pol);
      if (bulk_act) {
        pdl_wait();                               // activations may belong to the previous grid
        const int rows = min(p.M, 8);
        mbar_arrive_expect_tx(act_bar, rows * (kBlocks * 128 * 2));
        for (int m = 0; m < rows; ++m)
          bulk_g2s(smem_u32(smem + kActOff + m * kActPitch),
                   p.A + static_cast<size_t>(m) * p.lda + static_cast<size_t>(rank) * kBlocks * 128,
                   kBlocks * 128 * 2, act_bar);
      }
      // No copy into this CTA's shared memory may be in flight at exit.
      mbar_wait(full, 0, p.err);
      if (bulk_act) mbar_wait(act_bar, 0, p.err);
    }
    __syncwarp();
    if (S > 1) tc::cluster_wait();
    return;
  }

  // -------------------------------------------------------------- compute
  const int b = warp;
  if (S > 1) tc::cluster_wait();
  pdl_wait();                                     // activations (and C) may belong to the previous grid
  bool live = true;
  uint32_t bf[16];
  float inv;
  const int kb = (rank * kBlocks + b) * 128;
  if (bulk_act) {
    live = tc::wait_or_abort(act_bar, 0, p.err, abort_flag);
    live = __all_sync(0xFFFFFFFFu, live);
    const int m = min(g, p.M - 1);
    const uint8_t* src = smem + kActOff + m * kActPitch + (b * 128 + 32 * t4) * 2;
    uint32_t r[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * q);
      r[4 * q] = v.x;
      r[4 * q + 1] = v.y;
      r[4 * q + 2] = v.z;
      r[4 * q + 3] = v.w;
    }
    build_bfrag_regs(r, bf, inv);
  } else {
    build_bfrag(p.A, p.lda, p.M, kb, 0, g, t4, bf, inv);
  }
  // This thread's sums are activation rows 2t and 2t + 1: their 2^-e.
  const float f0 = __shfl_sync(0xFFFFFFFFu, inv, 8 * t4);
  const float f1 = __shfl_sync(0xFFFFFFFFu, inv, 8 * t4 + 4);
  float tot[kTiles][4];
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt)
#pragma unroll
    for (int i = 0; i < 4; ++i) tot[rt][i] = 0.f;
  if (live) live = tc::wait_or_abort(full, 0, p.err, abort_flag);
  live = __all_sync(0xFFFFFFFFu, live);
  if (live) {
    const uint8_t* box = smem + b * kBoxBytes;
#pragma unroll
    for (int r0 = 0; r0 < kTiles; r0 += 2) {      // two row tiles' chains interleaved
      uint32_t wg[2][4], wh[2][4], sg[2][2], sh[2][2];
      float c[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int rg = 16 * (r0 + i) + g, rh = rg + 8;
        const uint4 u = lds128(box + rg * 64 + 16 * t4);
        const uint4 v = lds128(box + rh * 64 + 16 * t4);
        wg[i][0] = u.x;
        wg[i][1] = u.y;
        wg[i][2] = u.z;
        wg[i][3] = u.w;
        wh[i][0] = v.x;
        wh[i][1] = v.y;
        wh[i][2] = v.z;
        wh[i][3] = v.w;
        // E4M3 scales of groups 2t and 2t + 1 of block b, as (s, s) f16x2.
        const uint32_t qg = *reinterpret_cast<const unsigned short*>(smem + kScaleOff + rg * 64 + 8 * b + 2 * t4);
        const uint32_t qh = *reinterpret_cast<const unsigned short*>(smem + kScaleOff + rh * 64 + 8 * b + 2 * t4);
        const uint32_t hg = e4m3x2_half<0>(qg), hh = e4m3x2_half<0>(qh);
        sg[i][0] = __byte_perm(hg, 0, 0x1010);
        sg[i][1] = __byte_perm(hg, 0, 0x3232);
        sh[i][0] = __byte_perm(hh, 0, 0x1010);
        sh[i][1] = __byte_perm(hh, 0, 0x3232);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {            // MMA jj: k = 32 t + 4 jj .. + 3 of every thread
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t xg = wg[i][jj >> 1], xh = wh[i][jj >> 1];
          const uint32_t s_g = sg[i][jj >> 2], s_h = sh[i][jj >> 2];
          uint32_t a0, a1, a2, a3;
          if (jj & 1) {
            a0 = mul_f16x2(e2m1x2_byte<2>(xg), s_g);
            a2 = mul_f16x2(e2m1x2_byte<3>(xg), s_g);
            a1 = mul_f16x2(e2m1x2_byte<2>(xh), s_h);
            a3 = mul_f16x2(e2m1x2_byte<3>(xh), s_h);
          } else {
            a0 = mul_f16x2(e2m1x2_byte<0>(xg), s_g);
            a2 = mul_f16x2(e2m1x2_byte<1>(xg), s_g);
            a1 = mul_f16x2(e2m1x2_byte<0>(xh), s_h);
            a3 = mul_f16x2(e2m1x2_byte<1>(xh), s_h);
          }
          if (jj == 0)
            mma_f16_16816_z(c[i], a0, a1, a2, a3, bf[0], bf[1]);
          else
            mma_f16_16816(c[i], a0, a1, a2, a3, bf[2 * jj], bf[2 * jj + 1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        tot[r0 + i][0] = f0 * c[i][0];
        tot[r0 + i][1] = f1 * c[i][1];
        tot[r0 + i][2] = f0 * c[i][2];
        tot[r0 + i][3] = f1 * c[i][3];
      }
    }
  }

  // ------------------------------------------------------------ reduce + store
  // The 8 warps' sums (one block each) in warp order, through shared memory
  // laid over the consumed stage; ranks 1.. send theirs to rank 0 and leave;
  // rank 0 adds them in rank order and stores.
  constexpr int kItems = kTiles * 32;
  float4* red = reinterpret_cast<float4*>(smem);
  asm volatile("bar.sync 1, %0;" ::"r"(kCompute * 32) : "memory");   // stage consumed by every warp
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt)
    red[warp * kItems + rt * 32 + lane] = make_float4(tot[rt][0], tot[rt][1], tot[rt][2], tot[rt][3]);
  asm volatile("bar.sync 1, %0;" ::"r"(kCompute * 32) : "memory");
  const int item = threadIdx.x;                   // (row tile, lane) of a warp's sums
  if (item >= kItems) return;
  float4 v = red[item];
#pragma unroll
  for (int w = 1; w < kCompute; ++w) {
    const float4 u = red[w * kItems + item];
    v.x += u.x;
    v.y += u.y;
    v.z += u.z;
    v.w += u.w;
  }
  if (rank != 0) {
    tc::st_async_f4(tc::mapa_shared(smem_u32(smem + kRecvOff + (rank - 1) * kSlot + item * 16), 0), v,
                    tc::mapa_shared(recv_bar, 0));
    return;
  }
  // Every peer sends, even one whose own waits gave up (each bounded by
  // kWaitLimitNs), so rank 0 waits three times as long: it never leaves while
  // a peer may still write into its shared memory.
  bool ok = S == 1 || mbar_wait_ns(recv_bar, 0, p.err, 3 * kWaitLimitNs);
  ok = ok && *abort_flag == 0;
  if (!ok) return;
  const float4* recv = reinterpret_cast<const float4*>(smem + kRecvOff) + item;
  for (int q = 1; q < S; ++q) {                   // rank order
    const float4 u = recv[(q - 1) * kItems];
    v.x += u.x;
    v.y += u.y;
    v.z += u.z;
    v.w += u.w;
  }
  const int rt = item / 32, ln = item % 32;
  const int r = n0 + 16 * rt + (ln >> 2), m = 2 * (ln & 3);
  const float acc[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int rr = r + 8 * (e >> 1), mm = m + (e & 1);
    if (mm < p.M && rr < p.N) p.C[static_cast<size_t>(mm) * p.ldc + rr] = f32_to_bf16_rn(acc[e] * p.gscale);
  }
}

cudaError_t set_attrs() {
  static AttrLatch latch;
  return set_smem_attrs(w4_short_kernel, latch, smem_bytes(kMaxSplits), true);
}

}  // namespace mmaw4s

bool w4a16_short_fits(const GemvArgs& a) {
  const int tiles = (a.N + mmaw4s::BM - 1) / mmaw4s::BM, stages = a.K / 1024;
  // Measured (5120-K shapes): short CTAs win up to 192 tiles (N = 12288:
  // 10.8 / 12.3 us at M = 1 / 8 against 13.8 / 14.5 persistent), the
  // persistent kernel from 272 (N = 17408: 13.6 / 15.2 against 14.1 / 15.7).
  return 4 * tiles < 7 * a.num_sms && stages <= mmaw4s::kMaxSplits;
}

// Requires K % 1024 == 0, K / 1024 <= 8 and M <= 8 (checked by the caller).
cudaError_t launch_w4a16_gemm_short(const GemvArgs& a, cudaStream_t s) {
  using namespace mmaw4s;
  const uint64_t K = static_cast<uint64_t>(a.K);
  CUtensorMap mw, ms;
  // Codes as [K/128 blocks][N rows][64 bytes]: row pitch K/2, block pitch 64.
  cudaError_t e = cached_map_3d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, {64, static_cast<uint64_t>(a.N), K / 128},
                                {K / 2, 64}, {64, BM, kBlocks}, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = cached_map_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scales, K / 16, static_cast<uint64_t>(a.N), K / 16, 64, BM,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if ((e = set_attrs()) != cudaSuccess) return e;
  Params p;
  p.A = static_cast<const uint16_t*>(a.A);
  p.C = static_cast<uint16_t*>(a.C);
  p.lda = a.lda;
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.gscale = a.gscale;
  p.splits = a.K / 1024;
  p.err = a.err;
  const int tiles = (a.N + BM - 1) / BM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * p.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes(p.splits);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = p.splits;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (a.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, w4_short_kernel, mw, ms, p);
}

}  // namespace wqp
