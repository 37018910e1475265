// FP8 (W8A16) and W4A16 GEMM on the warp-level tensor-core path
// (mma.sync m16n8k16, FP16 operands, FP32 accumulation), swap-AB: the MMA's
// 16 "rows" are weight rows n, its 8 "columns" are activation rows m (two
// column tiles when M > 8, so every weight is read once for all M <= 16 rows).
//
// What it computes:
//  * FP8: "metrale_model_layers/layers/ops/w8a16_gemm_m16.rs" (doc of
//    `w8a16_gemm_m16`: weight [N, K] E4M3, block_scale [N/128, K/128] FP32;
//    module docs: the 128-K block scale is folded once per block onto an
//    FP32 accumulator, never per element and never into BF16):
//      C[m, n] = bf16( sum_b s[n/128, b] * sum_{k in b} a[m, k] * e4m3(W[n, k]) ).
//  * W4: the batched W4A16 GEMV of "spark_model/layers/w4a16_gemv_tiers.rs"
//    (module docs) with the reading w = e2m1(nibble) * e4m3(scale[n, k/16]),
//    times one FP32 per-tensor scale g applied to each FP32 result.
//
// Exact products. Every E4M3 value, and every product of an E2M1 value with
// an E4M3 scale (at most 6 significant bits, within [2^-10, 2688]), is an
// FP16 value, so the weight operand is exact. The activations are scaled per
// (activation row, 128-K block) by a power of two 2^e that puts the block
// row's largest magnitude in [2^14, 2^15), then rounded to FP16: every BF16
// value of at least 2^-31 times that maximum is exact, and a smaller one is
// off by at most 2^-25 in the scaled units (2^-39 of the block's largest
// activation). The MMA multiplies FP16 by FP16 exactly into FP32; the block's
// FP32 sum is multiplied by 2^-e (and, for FP8, by the block scale) once and
// added to the FP32 accumulator. Only the order of the FP32 additions differs
// from the per-row sum.
//
// Work split: tiles of BM weight rows (64 for W4, 32 for FP8), stages of 8
// blocks of 128 K. A cluster of S CTAs splits K (rank r owns
// stages [r*stages/S, (r+1)*stages/S)); clusters are persistent over the
// tiles c, c + C, ...; each CTA streams its (tile, stage) items through a
// ring of raw stages filled by TMA.
// Warps: 0..7 compute (warp w owns block w of every stage, every 16-row tile
// of the tile), 8 the TMA producer, 9 the epilogue (sum of the 8 warps' partials in
// warp order; ranks >= 1 send theirs to rank 0 with st.async, rank 0 adds them
// in rank order and stores).
// Per 128-K block and thread (g = lane / 4, t = lane % 4): the thread's
// weights are the 32 consecutive k = 128 b + 32 t .. + 31 of rows g and g + 8
// of a 16-row tile, and its activations the same 32 k of activation row g
// (+ 8 for the second column tile). MMA j (j = 0..7) takes k + 4j .. + 3 of
// every thread: the MMA's k positions (2t, 2t + 1) and (2t + 8, 2t + 9) are
// k + 4j + (0, 1) and k + 4j + (2, 3). A and B use the same map, so the sum
// over the MMA's 16 k positions is the sum over those k.
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda_fp16.h>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"
#include "mma_f16.cuh"
#include "tc.cuh"

namespace wqp {
namespace mmaf {

using namespace f16op;

constexpr int kCompute = 8;                  // compute warps: one per 128-K block of a stage
constexpr int kProducer = kCompute;
constexpr int kEpilogue = kCompute + 1;
constexpr int kThreads = (kCompute + 2) * 32;
constexpr int kBlocks = 8;                   // 128-K blocks per stage (1024 K)
constexpr int kMaxSplits = 8;
constexpr int kMaxRing = 8;

// FP8 stage: 8 blocks of 32 rows x 128 bytes (128-byte swizzle; one 3-D
// copy), then the 8 FP32 block scales of the tile's 128-row group. Tiles of 32 rows keep a
// stage at 33 KB, so six stages stay in flight per SM.
struct Fp8F {
  static constexpr bool kW4 = false;
  static constexpr int BM = 32;                                         // weight rows per tile
  static constexpr int kTiles = BM / 16;                                // 16-row MMA tiles per tile
  static constexpr int kBoxBytes = BM * 128;
  static constexpr int kScaleOff = kBlocks * kBoxBytes;                 // 32768
  static constexpr int kTxBytes = kScaleOff + kBlocks * 4;
  static constexpr int kStageBytes = kScaleOff + 1024;                  // keeps slots 1024-aligned
};
// W4 stage: 8 blocks of 64 rows x 64 bytes of codes (one 3-D copy), then
// 64 rows x 64 bytes of E4M3 group scales (8 blocks x 8 groups of 16 K).
struct W4F {
  static constexpr bool kW4 = true;
  static constexpr int BM = 64;
  static constexpr int kTiles = BM / 16;
  static constexpr int kBoxBytes = BM * 64;
  static constexpr int kScaleOff = kBlocks * kBoxBytes;                 // 32768
  static constexpr int kTxBytes = kScaleOff + BM * 64;
  static constexpr int kStageBytes = kTxBytes;                          // 36864
};

template <class F, int MT>
struct Sizes {
  static constexpr int kItems = F::kTiles * MT * 32;   // float4 sums of one warp for one tile
  static constexpr int kSlot = kItems * 16;
  static constexpr int kRed = kCompute * kSlot;
};

struct Params {
  const uint16_t* A;   // bf16 [M, lda]
  uint16_t* C;         // bf16 [M, ldc]
  int lda, ldc;
  int M, N, K;
  float gscale;        // W4 per-tensor scale (1 for FP8)
  int tiles, stages, splits, clusters, ring;
  int red_off, recv_off, bf_off, fo_off;   // shared-memory offsets (ring at 0)
  unsigned* err;
};

// MT: column tiles of 8 activation rows (1: M <= 8, 2: M <= 16).
// kRegB: every rank owns one stage, so the B fragments stay in registers.
// kRebuild: the B fragments of every stage would not fit shared memory beside
//           the ring (16 rows with no K split, or a long K), so each item
//           rebuilds its block's fragments from the activations in L2 instead
//           of keeping them.
// kNS: a rank owns at most kNS stages and each warp keeps its block's B
//      fragments of all of them in registers (8 rows, one CTA per SM), which
//      leaves the shared memory to the ring.
template <class F, int MT, bool kRegB, int kOcc, bool kRebuild = false, int kNS = 0>
__global__ void __launch_bounds__(kThreads, kOcc)
    f16_stream_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                      const Params p) {
  using Z = Sizes<F, MT>;
  static_assert(kNS == 0 || (MT == 1 && !kRegB && !kRebuild), "register-held fragment sets: 8 rows");
  constexpr int BM = F::BM, kTiles = F::kTiles;
  extern __shared__ __align__(1024) uint8_t smem[];
  // full[R], empty[R], red_full, red_empty, recv_full[2], recv_free[2]
  __shared__ __align__(8) uint64_t bars[2 * kMaxRing + 6];
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits, C = p.clusters, R = p.ring;
  const int cl = blockIdx.x / S;
  const int rank = blockIdx.x - cl * S;           // == %cluster_ctarank
  const int st0 = (rank * p.stages) / S;
  const int nst = ((rank + 1) * p.stages) / S - st0;   // >= 1: S <= stages
  const int ntile = (p.tiles - cl + C - 1) / C;   // tiles cl, cl + C, ... (cl < tiles)
  const int items = ntile * nst;
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[kMaxRing]);
  const uint32_t red_full = smem_u32(&bars[2 * kMaxRing]), red_empty = red_full + 8;
  const uint32_t recv_full = red_full + 16, recv_free = red_full + 32;   // two slots each

  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kCompute);
    }
    mbar_init(red_full, kCompute);
    mbar_init(red_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(recv_full + 8 * i, 1);
      mbar_init(recv_free + 8 * i, 1);
    }
    mbar_fence_init();
    abort_sh = 0;
  }
  if (S > 1) tc::cluster_arrive_relaxed();
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tmW);
      tc::prefetch_tmap(&tmS);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int it = 0; it < items; ++it) {
        const int s = it % R;
        if (it >= R && !tc::wait_or_abort(empty0 + 8 * s, ((it / R) - 1) & 1, p.err, abort_flag)) break;
        const int tile = cl + (it / nst) * C, st = st0 + it % nst;
        const uint32_t dst = smem_u32(smem + s * F::kStageBytes), bar = full0 + 8 * s;
        mbar_arrive_expect_tx(bar, F::kTxBytes);
        // One copy of the stage's 8 blocks (a 3-D view: bytes of a block's
        // row, rows, blocks), landing block after block.
        tc::tma_load_3d_hint(dst, &tmW, 0, tile * BM, st * kBlocks, bar, pol);
        if constexpr (F::kW4)
          tc::tma_load_2d_hint(dst + F::kScaleOff, &tmS, st * 64, tile * BM, bar, pol);
        else
          tc::tma_load_2d(dst + F::kScaleOff, &tmS, st * kBlocks, (tile * BM) / 128, bar);
        issued = it + 1;
      }
      // No copy into this CTA's shared memory may be in flight at exit.
      for (int it = max(0, issued - R); it < issued; ++it) mbar_wait(full0 + 8 * (it % R), (it / R) & 1, p.err);
    }
    __syncwarp();
    if (S > 1) tc::cluster_wait();
  } else if (warp == kEpilogue) {
    // ------------------------------------------------------------ epilogue
    if (S > 1) tc::cluster_wait();
    pdl_wait();                                    // C may be read by the previous grid
    const float4* red = reinterpret_cast<const float4*>(smem + p.red_off);
    const float4* recv = reinterpret_cast<const float4*>(smem + p.recv_off);
    for (int tl = 0; tl < ntile; ++tl) {
      const int n0 = (cl + tl * C) * BM;
      bool ok = tc::wait_or_abort(red_full, tl & 1, p.err, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok);
      float4 v[kTiles * MT];
#pragma unroll
      for (int i = 0; i < kTiles * MT; ++i) {
        const int item = i * 32 + lane;
        v[i] = red[item];
#pragma unroll
        for (int w = 1; w < kCompute; ++w) {      // warp (block) order
          const float4 u = red[w * Z::kItems + item];
          v[i].x += u.x;
          v[i].y += u.y;
          v[i].z += u.z;
          v[i].w += u.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_empty);
      const int slot = tl & 1, use = tl >> 1;
      if (rank != 0) {
        if (use > 0 && ok) ok = tc::wait_cluster_or_abort(recv_free + 8 * slot, (use - 1) & 1, p.err, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
          const uint32_t dst0 =
              tc::mapa_shared(smem_u32(smem + p.recv_off + (slot * (S - 1) + rank - 1) * Z::kSlot), 0);
          const uint32_t bar0 = tc::mapa_shared(recv_full + 8 * slot, 0);
#pragma unroll
          for (int i = 0; i < kTiles * MT; ++i) tc::st_async_f4(dst0 + (i * 32 + lane) * 16, v[i], bar0);
        }
        continue;
      }
      if (S > 1) {
        if (lane == 0) mbar_arrive_expect_tx(recv_full + 8 * slot, (S - 1) * Z::kSlot);
        if (ok) ok = tc::wait_or_abort(recv_full + 8 * slot, use & 1, p.err, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
          const float4* rs = recv + slot * (S - 1) * Z::kItems;
          for (int q = 1; q < S; ++q) {           // rank order
#pragma unroll
            for (int i = 0; i < kTiles * MT; ++i) {
              const float4 u = rs[(q - 1) * Z::kItems + i * 32 + lane];
              v[i].x += u.x;
              v[i].y += u.y;
              v[i].z += u.z;
              v[i].w += u.w;
            }
          }
        }
        __syncwarp();
        if (ok && tl + 2 < ntile && lane < S - 1) tc::mbar_arrive_remote(tc::mapa_shared(recv_free + 8 * slot, lane + 1));
      }
      if (!ok || *abort_flag) continue;
#pragma unroll
      for (int i = 0; i < kTiles * MT; ++i) {
        const int rt = i / MT, mt = i % MT;
        const int r = n0 + 16 * rt + (lane >> 2), m = 8 * mt + 2 * (lane & 3);
        const float acc[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = r + 8 * (e >> 1), mm = m + (e & 1);
          if (mm < p.M && rr < p.N) p.C[static_cast<size_t>(mm) * p.ldc + rr] = f32_to_bf16_rn(acc[e] * p.gscale);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int b = warp;                           // block b of every stage
    const int g = lane >> 2, t4 = lane & 3;
    if (S > 1) tc::cluster_wait();
    pdl_wait();                                   // activations may belong to the previous grid
    uint32_t bf[MT][16];
    float fo[MT][2];                              // 2^-e of the two activation rows of this thread's sums
    uint4* bfs = reinterpret_cast<uint4*>(smem + p.bf_off);
    float2* fos = reinterpret_cast<float2*>(smem + p.fo_off);
    auto build = [&](int kb, int mt, uint32_t (&frag)[16], float (&f)[2]) {
      float inv;
      build_bfrag(p.A, p.lda, p.M, kb, mt, g, t4, frag, inv);
      // This thread's sums are activation rows 2t and 2t + 1 (+ 8 mt): take
      // their 2^-e from lanes 8t and 8t + 4.
      f[0] = __shfl_sync(0xFFFFFFFFu, inv, 8 * t4);
      f[1] = __shfl_sync(0xFFFFFFFFu, inv, 8 * t4 + 4);
    };
    uint32_t bfa[kNS > 0 ? kNS : 1][MT][16];      // kNS: every stage's fragments
    float foa[kNS > 0 ? kNS : 1][MT][2];
    if constexpr (kNS > 0) {
#pragma unroll
      for (int js = 0; js < kNS; ++js)
        if (js < nst) build(((st0 + js) * kBlocks + b) * 128, 0, bfa[js][0], foa[js][0]);
    } else if constexpr (kRegB) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) build((st0 * kBlocks + b) * 128, mt, bf[mt], fo[mt]);
    } else if constexpr (!kRebuild) {
      for (int j = 0; j < nst; ++j) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          build(((st0 + j) * kBlocks + b) * 128, mt, bf[mt], fo[mt]);
          const int set = (j * kCompute + b) * MT + mt;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            bfs[(set * 4 + q) * 32 + lane] = make_uint4(bf[mt][4 * q], bf[mt][4 * q + 1], bf[mt][4 * q + 2], bf[mt][4 * q + 3]);
          fos[set * 32 + lane] = make_float2(fo[mt][0], fo[mt][1]);
        }
      }
      __syncwarp();
    }
    float tot[kTiles][MT][4];
#pragma unroll
    for (int rt = 0; rt < kTiles; ++rt)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[rt][mt][i] = 0.f;
    float4* red = reinterpret_cast<float4*>(smem + p.red_off) + warp * Z::kItems;
    bool live = true;
    int s = 0, ph = 0, j = 0, tl = 0;
    // One (tile, stage) item against the stage's fragments bfx / fox.
    auto item = [&](const uint32_t (&bfx)[MT][16], const float (&fox)[MT][2]) {
      if (live) live = tc::wait_or_abort(full0 + 8 * s, ph, p.err, abort_flag);
      live = __all_sync(0xFFFFFFFFu, live);
      if (live) {
        const uint8_t* stage = smem + s * F::kStageBytes;
        const uint8_t* box = stage + b * F::kBoxBytes;
        // Fold factors of this block: 2^-e per activation row (and the FP8
        // block scale of the tile's 128-row group).
        float f[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if constexpr (F::kW4) {
            f[mt][0] = fox[mt][0];
            f[mt][1] = fox[mt][1];
          } else {
            const float sb = reinterpret_cast<const float*>(stage + F::kScaleOff)[b];
            f[mt][0] = sb * fox[mt][0];
            f[mt][1] = sb * fox[mt][1];
          }
        }
#pragma unroll
        for (int r0 = 0; r0 < kTiles; r0 += 2) {  // two row tiles' chains interleaved
          float c[2][MT][4];
          uint32_t wg[2][8], wh[2][8];            // this thread's weights of rows g, g + 8 (FP8: 8 words, W4: 4)
          uint32_t sg[2][2], sh[2][2];            // W4: (s, s) f16x2 of groups 2t and 2t + 1, rows g and g + 8
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int rg = 16 * (r0 + i) + g, rh = rg + 8;
            if constexpr (F::kW4) {
              const uint4 u = lds128(box + rg * 64 + 16 * t4);
              const uint4 v = lds128(box + rh * 64 + 16 * t4);
              wg[i][0] = u.x; wg[i][1] = u.y; wg[i][2] = u.z; wg[i][3] = u.w;
              wh[i][0] = v.x; wh[i][1] = v.y; wh[i][2] = v.z; wh[i][3] = v.w;
              const uint32_t qg = *reinterpret_cast<const unsigned short*>(stage + F::kScaleOff + rg * 64 + 8 * b + 2 * t4);
              const uint32_t qh = *reinterpret_cast<const unsigned short*>(stage + F::kScaleOff + rh * 64 + 8 * b + 2 * t4);
              const uint32_t hg = e4m3x2_half<0>(qg), hh = e4m3x2_half<0>(qh);
              sg[i][0] = __byte_perm(hg, 0, 0x1010);
              sg[i][1] = __byte_perm(hg, 0, 0x3232);
              sh[i][0] = __byte_perm(hh, 0, 0x1010);
              sh[i][1] = __byte_perm(hh, 0, 0x3232);
            } else {
              // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7).
              const uint4 u0 = lds128(box + rg * 128 + (((2 * t4) ^ (rg & 7)) << 4));
              const uint4 u1 = lds128(box + rg * 128 + (((2 * t4 + 1) ^ (rg & 7)) << 4));
              const uint4 v0 = lds128(box + rh * 128 + (((2 * t4) ^ (rh & 7)) << 4));
              const uint4 v1 = lds128(box + rh * 128 + (((2 * t4 + 1) ^ (rh & 7)) << 4));
              wg[i][0] = u0.x; wg[i][1] = u0.y; wg[i][2] = u0.z; wg[i][3] = u0.w;
              wg[i][4] = u1.x; wg[i][5] = u1.y; wg[i][6] = u1.z; wg[i][7] = u1.w;
              wh[i][0] = v0.x; wh[i][1] = v0.y; wh[i][2] = v0.z; wh[i][3] = v0.w;
              wh[i][4] = v1.x; wh[i][5] = v1.y; wh[i][6] = v1.z; wh[i][7] = v1.w;
            }
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {        // MMA jj: k + 4 jj .. + 3 of every thread
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              uint32_t a0, a1, a2, a3;
              if constexpr (F::kW4) {
                // Bytes 2 jj, 2 jj + 1 of the row's 16: elements 4 jj .. 4 jj + 3.
                const uint32_t xg = wg[i][jj >> 1], xh = wh[i][jj >> 1];
                const uint32_t s_g = sg[i][jj >> 2], s_h = sh[i][jj >> 2];
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
              } else {
                a0 = e4m3x2_half<0>(wg[i][jj]);
                a2 = e4m3x2_half<1>(wg[i][jj]);
                a1 = e4m3x2_half<0>(wh[i][jj]);
                a3 = e4m3x2_half<1>(wh[i][jj]);
              }
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                if (jj == 0)
                  mma_f16_16816_z(c[i][mt], a0, a1, a2, a3, bfx[mt][0], bfx[mt][1]);
                else
                  mma_f16_16816(c[i][mt], a0, a1, a2, a3, bfx[mt][2 * jj], bfx[mt][2 * jj + 1]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              float* t = tot[r0 + i][mt];
              t[0] = fmaf(f[mt][0], c[i][mt][0], t[0]);
              t[1] = fmaf(f[mt][1], c[i][mt][1], t[1]);
              t[2] = fmaf(f[mt][0], c[i][mt][2], t[2]);
              t[3] = fmaf(f[mt][1], c[i][mt][3], t[3]);
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
      if (++s == R) {
        s = 0;
        ph ^= 1;
      }
      if (++j == nst) {
        // Tile done: hand the sums to the epilogue (its buffer is free once it
        // has read the previous tile's).
        j = 0;
        if (tl > 0 && live) live = tc::wait_or_abort(red_empty, (tl - 1) & 1, p.err, abort_flag);
        live = __all_sync(0xFFFFFFFFu, live);
#pragma unroll
        for (int rt = 0; rt < kTiles; ++rt)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            red[(rt * MT + mt) * 32 + lane] = make_float4(tot[rt][mt][0], tot[rt][mt][1], tot[rt][mt][2], tot[rt][mt][3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) tot[rt][mt][i] = 0.f;
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full);
        ++tl;
      }
    };
    if constexpr (kNS > 0) {
      for (int ti = 0; ti < ntile; ++ti) {
#pragma unroll
        for (int js = 0; js < kNS; ++js)
          if (js < nst) item(bfa[js], foa[js]);
      }
    } else {
      for (int it = 0; it < items; ++it) {
        if constexpr (kRebuild) {
          if (nst > 1 || it == 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) build(((st0 + j) * kBlocks + b) * 128, mt, bf[mt], fo[mt]);
          }
        } else if constexpr (!kRegB) {
          if (nst > 1 || it == 0) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const int set = (j * kCompute + b) * MT + mt;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 u = bfs[(set * 4 + q) * 32 + lane];
                bf[mt][4 * q] = u.x;
                bf[mt][4 * q + 1] = u.y;
                bf[mt][4 * q + 2] = u.z;
                bf[mt][4 * q + 3] = u.w;
              }
              const float2 f2 = fos[set * 32 + lane];
              fo[mt][0] = f2.x;
              fo[mt][1] = f2.y;
            }
          }
        }
        item(bf, fo);
      }
    }
  }
  // Every CTA of the cluster stays until all are done: peers' st.async into
  // rank 0's shared memory and rank 0's arrives on the peers' barriers have
  // landed before any CTA exits.
  if (S > 1) tc::cluster_sync();
}

// ---------------------------------------------------------------- host side
constexpr int kMaxRegSets = 5;        // stages per rank whose fragment sets fit in registers
constexpr int kBudget2 = 110 * 1024;   // dynamic shared memory of a 2-CTA-per-SM variant
constexpr int kBudget1 = 220 * 1024;   // of a 1-CTA-per-SM variant

template <class F, int MT, bool kRegB, int kOcc, bool kRebuild = false, int kNS = 0>
struct Variant {
  static constexpr auto kernel = f16_stream_kernel<F, MT, kRegB, kOcc, kRebuild, kNS>;
  static constexpr int kBudget = kOcc == 2 ? kBudget2 : kBudget1;
};

template <class F, int MT, bool kRegB, int kOcc, bool kRebuild = false, int kNS = 0>
cudaError_t set_attrs() {
  static AttrLatch latch;
  using V = Variant<F, MT, kRegB, kOcc, kRebuild, kNS>;
  return set_smem_attrs(V::kernel, latch, V::kBudget, true);
}

// Clusters of s CTAs of a variant resident at once (0 if the query failed).
// Cached per device.
template <class F, int MT, bool kRegB, int kOcc, bool kRebuild = false>
int cluster_capacity(int s) {
  static std::atomic<int> cache[kMaxDevices][kMaxSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::atomic<int>& slot = cache[dev][s];
  int v = slot.load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  using V = Variant<F, MT, kRegB, kOcc, kRebuild>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = V::kBudget;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = s;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (set_attrs<F, MT, kRegB, kOcc, kRebuild>() != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, V::kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();            // the query's failure is not the caller's error
    n = 0;
  }
  slot.store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n > 0 ? n : 0;
}

struct Plan {
  bool regb = false;
  bool rebuild = false;
  int ns = 0;          // > 0: each warp keeps the fragments of its ns stages in registers
  int occ = 1;
  int splits = 1, clusters = 1, ring = 2;
  int red_off = 0, recv_off = 0, bf_off = 0, fo_off = 0, smem = 0;
  double cost = -1.0;
};

template <class F, int MT>
void layout(Plan& pl, int stages, int budget) {
  using Z = Sizes<F, MT>;
  const int nsmax = (stages + pl.splits - 1) / pl.splits;
  const int sets = (pl.regb || pl.rebuild || pl.ns > 0) ? 0 : nsmax * kCompute * MT;
  const int fixed = Z::kRed + 2 * (pl.splits - 1) * Z::kSlot + sets * (32 * 64 + 32 * 8);
  pl.ring = std::min(kMaxRing, (budget - fixed) / F::kStageBytes);
  pl.red_off = pl.ring * F::kStageBytes;
  pl.recv_off = pl.red_off + Z::kRed;
  pl.bf_off = pl.recv_off + 2 * (pl.splits - 1) * Z::kSlot;
  pl.fo_off = pl.bf_off + sets * 32 * 64;
  pl.smem = pl.fo_off + sets * 32 * 8;
}

// The busiest SM's (tile, stage) items over the relative rate of an SM with
// that many CTAs, plus the cross-CTA reduction of each tile when K is split
// (measured on GB300 at about a third of an item per tile).
constexpr double kSmRate[3] = {0.0, 1.0, 1.1};
constexpr double kSplitTileCost = 0.35;

template <class F, int MT, bool kRegB, int kOcc, bool kRebuild = false>
void consider(Plan& best, int splits, int tiles, int stages, int num_sms) {
  Plan pl;
  pl.regb = kRegB;
  pl.rebuild = kRebuild;
  pl.occ = kOcc;
  pl.splits = splits;
  layout<F, MT>(pl, stages, Variant<F, MT, kRegB, kOcc, kRebuild>::kBudget);
  if (pl.ring < 2) return;
  const int nsmax = (stages + splits - 1) / splits;
  const int cap = cluster_capacity<F, MT, kRegB, kOcc, kRebuild>(splits);
  const int clusters = std::min(tiles, cap > 0 ? cap : (kOcc * num_sms) / splits);
  if (clusters < 1) return;
  pl.clusters = clusters;
  const int per_sm = std::min(2, (clusters * splits + num_sms - 1) / num_sms);
  const int tpc = (tiles + clusters - 1) / clusters;   // tiles of the busiest cluster
  pl.cost = (static_cast<double>(tpc) * nsmax + (splits > 1 ? kSplitTileCost * tpc : 0.0)) * per_sm / kSmRate[per_sm];
  if (best.cost < 0 || pl.cost < best.cost - 1e-9) best = pl;
}

// Launch plan for (format, N, K, M tile) on the current device: cluster size
// (K split), variant and persistent clusters (one wave) minimising the
// busiest SM's work. It depends on N, K and the device, never on the
// activation rows, so a row's result does not depend on the other rows.
template <class F, int MT>
Plan choose_plan(int tiles, int stages, int num_sms, int only_splits = 0) {
  Plan best;
  for (int s = 1; s <= kMaxSplits && s <= stages; ++s) {
    if (only_splits > 0 && s != only_splits) continue;
    if (s == stages) {
      // Two column tiles need more registers than two CTAs per SM leave.
      if constexpr (MT == 1) consider<F, 1, true, 2>(best, s, tiles, stages, num_sms);
      consider<F, MT, true, 1>(best, s, tiles, stages, num_sms);
    } else {
      consider<F, MT, false, 1>(best, s, tiles, stages, num_sms);
    }
  }
  // Fragment sets that do not fit beside a ring of two stages (two column
  // tiles with no K split; any M tile past K = 57344 for FP8 and K = 43008
  // for W4 at 8 splits): each item rebuilds its block's fragments instead.
  if (best.cost < 0) {
    for (int s = 1; s <= kMaxSplits && s < stages; ++s)
      if (only_splits <= 0 || s == only_splits) consider<F, MT, false, 1, true>(best, s, tiles, stages, num_sms);
  }
  return best;
}

template <class F, int MT, bool kRegB, int kOcc, bool kRebuild = false, int kNS = 0>
cudaError_t launch_variant(const CUtensorMap& mw, const CUtensorMap& ms, const Params& p, bool pdl, int smem,
                           cudaStream_t s) {
  cudaError_t e = set_attrs<F, MT, kRegB, kOcc, kRebuild, kNS>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.clusters * p.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = p.splits;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, Variant<F, MT, kRegB, kOcc, kRebuild, kNS>::kernel, mw, ms, p);
}

// Plans cached per (device, format, N, K, M tile).
struct PlanKey {
  int dev, fmt, N, K, mt;
  bool operator==(const PlanKey& o) const {
    return dev == o.dev && fmt == o.fmt && N == o.N && K == o.K && mt == o.mt;
  }
};
constexpr int kPlanCache = 64;
struct PlanCache {
  std::mutex mu;
  PlanKey key[kPlanCache];
  Plan plan[kPlanCache];
  int n = 0, next = 0;
};
PlanCache& plan_cache() {
  static PlanCache c;
  return c;
}

template <class F>
cudaError_t launch_fmt(const GemvArgs& a, const CUtensorMap& mw, const CUtensorMap& ms, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int mt = a.M > 8 ? 2 : 1;
  const int tiles = (a.N + F::BM - 1) / F::BM, stages = a.K / (kBlocks * 128);
  const PlanKey key{dev, F::kW4 ? 1 : 0, a.N, a.K, mt};
  Plan pl;
  bool have = false;
  PlanCache& pc = plan_cache();
  {
    std::lock_guard<std::mutex> lk(pc.mu);
    for (int i = 0; i < pc.n && !have; ++i)
      if (pc.key[i] == key) {
        pl = pc.plan[i];
        have = true;
      }
  }
  if (!have) {
    // The K split (and so every row's summation order) is the one of the
    // 8-row plan for every M, so a row's result does not depend on how many
    // rows the call has.
    pl = choose_plan<F, 1>(tiles, stages, a.num_sms);
    if (pl.cost >= 0 && mt == 2) pl = choose_plan<F, 2>(tiles, stages, a.num_sms, pl.splits);
    std::lock_guard<std::mutex> lk(pc.mu);
    const int i = pc.n < kPlanCache ? pc.n++ : (pc.next++ % kPlanCache);
    pc.key[i] = key;
    pc.plan[i] = pl;
  }
  if (pl.cost < 0) {
    if (mt == 1) return cudaErrorInvalidConfiguration;
    // No two-column-tile plan fits this shape's shared memory: two launches
    // of 8 rows (each row's result is the one a call with M <= 8 gives).
    GemvArgs lo = a, hi = a;
    lo.M = 8;
    hi.M = a.M - 8;
    hi.A = static_cast<const uint16_t*>(a.A) + static_cast<size_t>(8) * a.lda;
    hi.C = static_cast<uint16_t*>(a.C) + static_cast<size_t>(8) * a.ldc;
    cudaError_t e1 = launch_fmt<F>(lo, mw, ms, s);
    return e1 != cudaSuccess ? e1 : launch_fmt<F>(hi, mw, ms, s);
  }
  Params p;
  p.A = static_cast<const uint16_t*>(a.A);
  p.C = static_cast<uint16_t*>(a.C);
  p.lda = a.lda;
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.gscale = a.gscale;
  p.tiles = tiles;
  p.stages = stages;
  p.splits = pl.splits;
  p.clusters = pl.clusters;
  p.ring = pl.ring;
  p.red_off = pl.red_off;
  p.recv_off = pl.recv_off;
  p.bf_off = pl.bf_off;
  p.fo_off = pl.fo_off;
  p.err = a.err;
  if (mt == 1) {
    if (pl.regb) return pl.occ == 2 ? launch_variant<F, 1, true, 2>(mw, ms, p, a.pdl, pl.smem, s)
                                    : launch_variant<F, 1, true, 1>(mw, ms, p, a.pdl, pl.smem, s);
    if (pl.rebuild) return launch_variant<F, 1, false, 1, true>(mw, ms, p, a.pdl, pl.smem, s);
    // FP8, a rank of at most kMaxRegSets stages: its fragment sets in
    // registers, the shared memory they would take to the ring (17408 x 5120:
    // 3 -> 6 raw stages in flight, 17.8 -> 15.8 us at M = 1). W4 measured
    // slower this way (13.6 -> 14.0 us at 17408 x 5120).
    if constexpr (!F::kW4) {
      const int nsmax = (stages + pl.splits - 1) / pl.splits;
      if (nsmax >= 2 && nsmax <= kMaxRegSets) {
        Plan pr = pl;
        pr.ns = nsmax;
        layout<F, 1>(pr, stages, kBudget1);
        p.ring = pr.ring;
        p.red_off = pr.red_off;
        p.recv_off = pr.recv_off;
        p.bf_off = pr.bf_off;
        p.fo_off = pr.fo_off;
        switch (nsmax) {
          case 2: return launch_variant<F, 1, false, 1, false, 2>(mw, ms, p, a.pdl, pr.smem, s);
          case 3: return launch_variant<F, 1, false, 1, false, 3>(mw, ms, p, a.pdl, pr.smem, s);
          case 4: return launch_variant<F, 1, false, 1, false, 4>(mw, ms, p, a.pdl, pr.smem, s);
          default: return launch_variant<F, 1, false, 1, false, 5>(mw, ms, p, a.pdl, pr.smem, s);
        }
      }
    }
    return launch_variant<F, 1, false, 1>(mw, ms, p, a.pdl, pl.smem, s);
  }
  if (pl.regb) return launch_variant<F, 2, true, 1>(mw, ms, p, a.pdl, pl.smem, s);
  if (pl.rebuild) return launch_variant<F, 2, false, 1, true>(mw, ms, p, a.pdl, pl.smem, s);
  return launch_variant<F, 2, false, 1>(mw, ms, p, a.pdl, pl.smem, s);
}

}  // namespace mmaf

// Requires K % 1024 == 0 (checked by the caller): stages of 8 whole blocks.
cudaError_t launch_w8a16_gemm_mma(const GemvArgs& a, cudaStream_t s) {
  using namespace mmaf;
  const uint64_t K = static_cast<uint64_t>(a.K);
  CUtensorMap mw, ms;
  // Codes as [K/128 blocks][N rows][128 bytes]: row pitch K, block pitch 128.
  cudaError_t e = cached_map_3d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, {128, static_cast<uint64_t>(a.N), K / 128},
                                {K, 128}, {128, Fp8F::BM, kBlocks}, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  // Block scales [ceil(N/128), K/128] FP32: one box of the stage's 8 scales.
  e = cached_map_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.scales, K / 128, static_cast<uint64_t>((a.N + 127) / 128),
                    (K / 128) * 4, kBlocks, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return launch_fmt<Fp8F>(a, mw, ms, s);
}

// Requires K % 1024 == 0 (checked by the caller).
cudaError_t launch_w4a16_gemm_mma(const GemvArgs& a, cudaStream_t s) {
  using namespace mmaf;
  // Fewer than 1.75 64-row tiles per SM (and at most 8 stages): short CTAs,
  // three per SM, 8 rows per launch. The choice depends on the shape only,
  // so a row's result does not depend on M.
  if (w4a16_short_fits(a)) {
    if (a.M <= 8) return launch_w4a16_gemm_short(a, s);
    GemvArgs lo = a, hi = a;
    lo.M = 8;
    hi.M = a.M - 8;
    hi.A = static_cast<const uint16_t*>(a.A) + static_cast<size_t>(8) * a.lda;
    hi.C = static_cast<uint16_t*>(a.C) + static_cast<size_t>(8) * a.ldc;
    const cudaError_t e1 = launch_w4a16_gemm_short(lo, s);
    return e1 != cudaSuccess ? e1 : launch_w4a16_gemm_short(hi, s);
  }
  const uint64_t K = static_cast<uint64_t>(a.K);
  CUtensorMap mw, ms;
  // Codes as [K/128 blocks][N rows][64 bytes]: row pitch K/2, block pitch 64.
  cudaError_t e = cached_map_3d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, {64, static_cast<uint64_t>(a.N), K / 128},
                                {K / 2, 64}, {64, W4F::BM, kBlocks}, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = cached_map_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scales, K / 16, static_cast<uint64_t>(a.N), K / 16, 64,
                    W4F::BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return launch_fmt<W4F>(a, mw, ms, s);
}

}  // namespace wqp
