// Persistent Q2_0 GEMM for 1 <= M <= 16 per launch on the warp-level tensor-core path
// (mma.sync m16n8k16, BF16 operands, FP32 accumulation), swap-AB: the MMA's
// 16 "rows" are weight rows n, its 8 "columns" are activation rows m (two
// column tiles when M > 8, so every weight is read once for all M rows).
//
// What it computes is the ternary Q2_0 product of
// "spark_model/layers/ops/gemv_q2_vec.rs" (module docs; the formula of the
// test helper `gemv_row`):
//   C[m, n] = bf16( sum_k A[m, k] * (c[n, k] - 1) * d[n, k / 128] ),
// with every product exact, so only the order of the FP32 additions differs
// from the per-row sum.
//
// Why registers instead of tensor memory: the GEMV is a weight stream, and
// every weight must pass through the converter exactly once. Here each warp
// turns its own code words into MMA operands in registers and issues the MMAs
// itself; nothing waits on another warp except the ring of raw stages and the
// hand-off of each tile's sums.
//
// Work split. The weight matrix is cut into tiles of BM = 64 rows and stages
// of 1024 K (8 blocks of 128 K, 272 bytes per row: the TMA box). A cluster of
// S CTAs splits K: rank r owns stages [r*stages/S, (r+1)*stages/S) of every
// tile. Clusters are persistent: cluster c handles tiles c, c + C, c + 2C, ...
// and each CTA streams its (tile, stage) items through a ring of raw stages.
//
// Warps of a CTA (W = 16 compute warps when one CTA has the SM and the
// launch has one 8-row column tile, else 8):
//   0..W-1 compute: warp w owns block w % 8 of every stage, for all four
//         16-row tiles (W = 8) or two of them (W = 16); after the
//         grid-dependency wait the MMA B fragments of its blocks are built
//         once per call (in registers when the rank owns one stage, else in
//         shared memory, the block's warps taking turns over its stages) and
//         then it only decodes codes and issues MMAs. At the end of a tile it hands its sums to
//         the epilogue;
//   W     producer: TMA of the raw stages (64 rows x 272 bytes) into the ring;
//   W+1   epilogue: adds the 8 blocks' sums of a tile (block order); ranks >= 1
//         send the result to rank 0 with st.async (completing on rank 0's
//         mbarrier), rank 0 adds them in rank order and stores C. A two-slot
//         receive buffer paces the peers: each peer has a "free" barrier per
//         slot, on which rank 0 arrives once it has read the slot.
// Per 128-K block b and thread (g = lane / 4, t = lane % 4):
//   * A fragment: code words 2t and 2t + 1 of the block, rows g and g + 8 of
//     a tile. Word bits 2q..2q+1 hold code q (q < 16). The pair of 16-bit
//     lanes (code x, code 8 + x), masked in place by
//     (word & 0x00030003 << 2x), is the BF16 pair (c_x 4^x, c_{8+x} 4^x) *
//     2^-133 (a subnormal or the smallest normal, exact); (word >> 8) gives
//     codes (4 + x, 12 + x).
//   * B fragment: activation row m = g (+ 8 for the second column tile; rows
//     past M repeat row M - 1): the 32 activations of k = 128 b + 32 t .. + 31,
//     paired the same way and multiplied by 2^(64 - 2x), so every product is
//     c * a * 2^-69 exactly.
//   * Each tile's chain starts from -2^-69 * sum_k a (four MMAs per block
//     with the raw activations as the A operand and -2^-69 as B, run once per
//     block and call), so it ends at 2^-69 * sum_k (c - 1) a.
//   * acc += d * chain, and C = bf16(acc * 2^69).
// Every wait is bounded (2 s of wall time); on expiry the CTA records the
// device error, skips the rest of its work, and still reaches the final
// cluster barrier, so no CTA exits while a peer may write into its shared
// memory or arrive on its barriers.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace wqp {
namespace mmas {

constexpr int BM = 64;                       // weight rows per tile
constexpr int kTiles = 4;                    // 16-row MMA tiles per tile
// Compute warps: one per 128-K block of a stage and all four row tiles when
// several CTAs share an SM or the launch has two column tiles (each warp's
// four row tiles against both keep enough MMA chains in flight: gate+up at
// M = 16 34.4 -> 31.6 us against 16 warps); with one CTA per SM and one
// column tile two per block, each with two of the row tiles (more warps to
// hide the mask -> MMA latencies).
constexpr int compute_warps(int occ, int mt) { return occ == 1 && mt == 1 ? 16 : 8; }
constexpr int threads_for(int occ, int mt) { return (compute_warps(occ, mt) + 2) * 32; }
constexpr int kBlocks = 8;                   // 128-K blocks per raw stage (1024 K)
constexpr int kRowBytes = kBlocks * 34;      // 272: 17 x 16 bytes
constexpr int kStageBytes = BM * kRowBytes;  // 17408
constexpr int kMaxSplits = 8;                // CTAs per cluster (K split) at most (portable size)
constexpr int kMaxRing = 12;                 // raw stage slots at most

// Shared-memory footprint per m tile count MT.
template <int MT>
struct Sizes {
  static constexpr int kItems = kTiles * MT * 32;   // float4 sums of one warp for one tile
  static constexpr int kSlot = kItems * 16;          // one rank's sums of a tile (bytes)
  static constexpr int kRed = kBlocks * kSlot;       // every block's sums of a tile
  static constexpr int kBf = MT * 32 * 64;           // B fragments of one block (16 words per lane per m tile)
  static constexpr int kNs = MT * 32 * 8;            // offset-chain pair of one block
};

struct StreamParams {
  const uint16_t* A;   // bf16 [M, lda]
  uint16_t* C;         // bf16 [M, ldc]
  int lda, ldc;
  int M, N;
  int tiles;           // ceil(N / 64)
  int stages;          // K / 1024
  int splits;          // S = cluster size
  int clusters;        // persistent clusters (<= tiles)
  int ring;            // raw stage slots (2..kMaxRing)
  int red_off, recv_off, bf_off, ns_off;   // shared-memory offsets (ring at 0)
  unsigned* err;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A * B + c with a separate accumulator input (the first MMA of a chain
// starts from c without copying it).
__device__ __forceinline__ void mma_bf16_16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1, float c0, float c1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%10,%11};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Code words 2t and 2t + 1 of the block at `blk` (34 b bytes into a raw row):
// 8 bytes at blk + 8 t. kA is the block's alignment class b % 4: 0 is
// 8-byte aligned, 2 is 4-byte aligned, 1 and 3 are 2 bytes off.
template <int kA>
__device__ __forceinline__ void load_codes(const uint8_t* blk, int t, uint32_t& w0, uint32_t& w1) {
  if constexpr (kA == 0) {
    const uint2 v = *reinterpret_cast<const uint2*>(blk + 8 * t);
    w0 = v.x;
    w1 = v.y;
  } else if constexpr (kA == 2) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(blk + 8 * t);
    w0 = p[0];
    w1 = p[1];
  } else {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(blk - 2 + 8 * t);
    const uint32_t x0 = p[0], x1 = p[1], x2 = p[2];
    w0 = __funnelshift_r(x0, x1, 16);
    w1 = __funnelshift_r(x1, x2, 16);
  }
}
__device__ __forceinline__ float load_d(const uint8_t* blk) {
  return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 32)));
}

// -2^-69 in both BF16 lanes.
constexpr uint32_t kNegUnit = 0x9D009D00u;
// 2^(64 - 2x) in both BF16 lanes.
__device__ __forceinline__ constexpr uint32_t prescale(int x) { return ((191u - 2u * x) << 7) * 0x00010001u; }

// The offset -2^-69 * sum_k a of a block for the activation rows of this
// thread's MMA columns 2t and 2t + 1. Four MMAs take the thread's 32 raw
// activations (row g) as the A operand, so rows g and g + 8 of the MMA each
// sum half of activation row g, against -2^-69 in every B element (every
// product exact); the two halves are added and each column's row sum is
// fetched from a lane of group 2t or 2t + 1.
__device__ __forceinline__ void offset_sums(const uint32_t (&r)[16], int t4, float (&ns)[2]) {
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 4; ++j) mma_bf16_16816(o, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3], kNegUnit, kNegUnit);
  const float s = o[0] + o[2];
  ns[0] = __shfl_sync(0xFFFFFFFFu, s, 8 * t4);
  ns[1] = __shfl_sync(0xFFFFFFFFu, s, 8 * t4 + 4);
}

// This thread's 32 activations of a block for one column tile: row
// min(g + 8 mt, M - 1), k = kb + 32 t .. + 31.
__device__ __forceinline__ void load_bact(const StreamParams& p, int kb, int mt, int g, int t4, uint32_t (&r)[16]) {
  const int m = min(g + 8 * mt, p.M - 1);         // rows past M: any valid row, results unused
  const uint16_t* src = p.A + static_cast<size_t>(m) * p.lda + kb + 32 * t4;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = ld_nc_v4(src + 8 * q);
    r[4 * q] = v.x;
    r[4 * q + 1] = v.y;
    r[4 * q + 2] = v.z;
    r[4 * q + 3] = v.w;
  }
}

// B fragments of one block for one column tile from this thread's 32
// activations r: permuted to the code-pair order and pre-scaled, and the
// offset -2^-69 * sum_k a of the activation rows of its MMA columns.
__device__ __forceinline__ void bfrag_from(const uint32_t (&r)[16], int t4, uint32_t (&bf)[16], float (&ns)[2]) {
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    const int x = st & 3, o = 8 * (st >> 2) + (x >> 1);
    const uint32_t sel = (x & 1) ? 0x7632u : 0x5410u;
    bf[2 * st] = mul_bf16x2(__byte_perm(r[o], r[o + 4], sel), prescale(x));
    bf[2 * st + 1] = mul_bf16x2(__byte_perm(r[o + 2], r[o + 6], sel), prescale(x));
  }
  offset_sums(r, t4, ns);
}

__device__ __forceinline__ void build_bfrag(const StreamParams& p, int kb, int mt, int g, int t4, uint32_t (&bf)[16],
                                            float (&ns)[2]) {
  uint32_t r[16];
  load_bact(p, kb, mt, g, t4, r);
  bfrag_from(r, t4, bf, ns);
}

// MT: column tiles of 8 activation rows (1: M <= 8, 2: M <= 16).
// kRegB: every rank owns exactly one stage, so each compute warp's B
//        fragments stay in registers for the whole call; otherwise they are
//        kept in shared memory, one set per stage of the rank.
// kOcc: CTAs per SM the registers are budgeted for.
// kPair: no K split, and the two CTAs of a cluster share the B-fragment
//        sets (each stores those of every other stage), for 16-row calls
//        whose sets would not fit one CTA.
template <int MT, bool kRegB, int kOcc, bool kPair = false>
__global__ void __launch_bounds__(threads_for(kOcc, MT), kOcc)
    q2_stream_kernel(const __grid_constant__ CUtensorMap tmW, const StreamParams p) {
  using Z = Sizes<MT>;
  constexpr int kCW = compute_warps(kOcc, MT);    // compute warps
  constexpr int kTPW = kTiles * kBlocks / kCW;    // row tiles per compute warp (4 or 2)
  constexpr int kProducer = kCW;                  // warp index of the TMA producer
  constexpr int kEpilogue = kCW + 1;              // warp index of the epilogue
  extern __shared__ __align__(1024) uint8_t smem[];
  // full[R], empty[R], red_full, red_empty, recv_full[2], recv_free[2]
  __shared__ __align__(8) uint64_t bars[2 * kMaxRing + 6];
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits, C = p.clusters, R = p.ring;
  // Paired CTAs (S = 1): each stores the B-fragment sets of every other stage
  // and reads the rest from its peer's shared memory.
  constexpr bool pair = kPair && !kRegB;
  const bool clustered = S > 1 || pair;
  const int prk = pair ? static_cast<int>(tc::cluster_rank()) : 0;
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
      mbar_init(empty0 + 8 * i, kCW);
    }
    mbar_init(red_full, kCW);
    mbar_init(red_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(recv_full + 8 * i, 1);
      mbar_init(recv_free + 8 * i, 1);
    }
    mbar_fence_init();
    abort_sh = 0;
  }
  if (clustered) tc::cluster_arrive_relaxed();
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kProducer) {
    // ------------------------------------------------------------ producer
    // Weights do not depend on the previous grid: the copies start at once.
    if (pair) {
      // The second cluster barrier (B-fragment sets written) must not wait
      // on this warp's copies: arrive now, wait at the end.
      tc::cluster_wait();
      tc::cluster_arrive();
    }
    if (lane == 0) {
      tc::prefetch_tmap(&tmW);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int it = 0; it < items; ++it) {
        const int s = it % R;
        if (it >= R && !tc::wait_or_abort(empty0 + 8 * s, ((it / R) - 1) & 1, p.err, abort_flag)) break;
        const int tile = cl + (it / nst) * C, st = st0 + it % nst;
        mbar_arrive_expect_tx(full0 + 8 * s, kStageBytes);
        tc::tma_load_2d_hint(smem_u32(smem + s * kStageBytes), &tmW, st * (kBlocks * 17), tile * BM,
                             full0 + 8 * s, pol);
        issued = it + 1;
      }
      // The CTA may not exit with a copy into its shared memory in flight:
      // wait until the last copies issued have landed.
      for (int it = max(0, issued - R); it < issued; ++it) mbar_wait(full0 + 8 * (it % R), (it / R) & 1, p.err);
    }
    __syncwarp();
    if (clustered) tc::cluster_wait();
  } else if (warp == kEpilogue) {
    // ------------------------------------------------------------ epilogue
    if (clustered) tc::cluster_wait();                 // every rank's barriers are initialised
    if (pair) tc::cluster_arrive();                    // second barrier: waited at the end
    pdl_wait();                                    // C may be read by the previous grid
    const float4* red = reinterpret_cast<const float4*>(smem + p.red_off);
    const float4* recv = reinterpret_cast<const float4*>(smem + p.recv_off);
    const float kUnscale = __uint_as_float((127u + 69u) << 23);   // 2^69
    for (int tl = 0; tl < ntile; ++tl) {
      const int n0 = (cl + tl * C) * BM;
      bool ok = tc::wait_or_abort(red_full, tl & 1, p.err, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok);
      float4 v[4 * MT];
#pragma unroll
      for (int i = 0; i < 4 * MT; ++i) {
        const int item = i * 32 + lane;            // (row tile, column tile, lane) of a warp's sums
        v[i] = red[item];
#pragma unroll
        for (int w = 1; w < kBlocks; ++w) {      // block order
          const float4 u = red[w * Z::kItems + item];
          v[i].x += u.x;
          v[i].y += u.y;
          v[i].z += u.z;
          v[i].w += u.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_empty);
      // Rank 0 receives tile tl's sums in slot tl % 2; a peer may send into a
      // slot once rank 0 has read what it held two tiles before.
      const int slot = tl & 1;
      const int use = tl >> 1;                     // earlier uses of this slot
      if (rank != 0) {
        if (use > 0 && ok) ok = tc::wait_cluster_or_abort(recv_free + 8 * slot, (use - 1) & 1, p.err, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {
          const uint32_t dst0 =
              tc::mapa_shared(smem_u32(smem + p.recv_off + (slot * (S - 1) + rank - 1) * Z::kSlot), 0);
          const uint32_t bar0 = tc::mapa_shared(recv_full + 8 * slot, 0);
#pragma unroll
          for (int i = 0; i < 4 * MT; ++i) tc::st_async_f4(dst0 + (i * 32 + lane) * 16, v[i], bar0);
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
            for (int i = 0; i < 4 * MT; ++i) {
              const float4 u = rs[(q - 1) * Z::kItems + i * 32 + lane];
              v[i].x += u.x;
              v[i].y += u.y;
              v[i].z += u.z;
              v[i].w += u.w;
            }
          }
        }
        __syncwarp();
        // Every lane has read the slot: the peers may send tile tl + 2 into it.
        if (ok && tl + 2 < ntile && lane < S - 1) tc::mbar_arrive_remote(tc::mapa_shared(recv_free + 8 * slot, lane + 1));
      }
      if (!ok || *abort_flag) continue;
#pragma unroll
      for (int i = 0; i < 4 * MT; ++i) {
        const int rt = i / MT, mt = i % MT;
        const int r = n0 + 16 * rt + (lane >> 2), m = 8 * mt + 2 * (lane & 3);
        const float acc[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = r + 8 * (e >> 1), mm = m + (e & 1);
          if (mm < p.M && rr < p.N) p.C[static_cast<size_t>(mm) * p.ldc + rr] = f32_to_bf16_rn(acc[e] * kUnscale);
        }
      }
    }
    if (pair) tc::cluster_wait();
  } else {
    // ------------------------------------------------------------ compute
    const int b = warp % kBlocks;                 // block b of every stage
    const int rq = warp / kBlocks;                // row tiles rq * kTPW .. + kTPW - 1
    const int g = lane >> 2, t4 = lane & 3;
    if (clustered) tc::cluster_wait();
    pdl_wait();                                   // activations may belong to the previous grid
    uint32_t bf[MT][16];
    float ns[MT][2];
    uint4* bfs = reinterpret_cast<uint4*>(smem + p.bf_off);
    float2* nss = reinterpret_cast<float2*>(smem + p.ns_off);
    if constexpr (kRegB) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) build_bfrag(p, (st0 * kBlocks + b) * 128, mt, g, t4, bf[mt], ns[mt]);
    } else {
      // One set per stage of the rank and block, read by the block's warps
      // (paired CTAs: stage j's set lives in CTA j % 2 of the pair, at index
      // j / 2). The block's warps take turns over its stages; each loads the
      // activations of its next set while it converts the current one.
      constexpr int kWPB = kCW / kBlocks;         // warps per block
      const int jstep = pair ? 2 * kWPB : kWPB;
      const int jfirst = (pair ? prk : 0) + (pair ? 2 : 1) * rq;
      uint32_t rn[16];
      if (jfirst < nst) load_bact(p, ((st0 + jfirst) * kBlocks + b) * 128, 0, g, t4, rn);
      for (int j = jfirst; j < nst; j += jstep) {
        const int jl = pair ? (j >> 1) : j;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t rc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) rc[i] = rn[i];
          if (mt + 1 < MT)
            load_bact(p, ((st0 + j) * kBlocks + b) * 128, mt + 1, g, t4, rn);
          else if (j + jstep < nst)
            load_bact(p, ((st0 + j + jstep) * kBlocks + b) * 128, 0, g, t4, rn);
          bfrag_from(rc, t4, bf[mt], ns[mt]);
          const int set = (jl * kBlocks + b) * MT + mt;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            bfs[(set * 4 + q) * 32 + lane] = make_uint4(bf[mt][4 * q], bf[mt][4 * q + 1], bf[mt][4 * q + 2], bf[mt][4 * q + 3]);
          nss[set * 32 + lane] = make_float2(ns[mt][0], ns[mt][1]);
        }
      }
      if constexpr (kCW > kBlocks)
        asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");   // every set written
      else
        __syncwarp();
      if (pair) {                                 // and the peer's
        tc::cluster_arrive();
        tc::cluster_wait();
      }
    }
    // Row tiles whose MMA chains run interleaved: all four when registers
    // allow, else two at a time.
    constexpr int kG = (kOcc >= 3 || MT == 2) ? 2 : kTPW;
    // Sums across the rank's stages of a tile (a rank with one stage writes
    // each item's sums straight to the epilogue's buffer instead).
    float tot[kRegB ? 1 : kTPW][MT][4];
    if constexpr (!kRegB) {
#pragma unroll
      for (int rt = 0; rt < kTPW; ++rt)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) tot[rt][mt][i] = 0.f;
    }
    float4* red = reinterpret_cast<float4*>(smem + p.red_off) + b * Z::kItems;
    bool live = true;
    auto run = [&](auto ac) {
      constexpr int kA = decltype(ac)::value;
      int s = 0, ph = 0;                           // ring slot and its phase
      int j = 0, tl = 0;                           // stage of the rank, tile of the cluster
      for (int it = 0; it < items; ++it) {
        if constexpr (!kRegB) {
          if (nst > 1 || it == 0) {
            const int jl = pair ? (j >> 1) : j;
            const bool remote = pair && (j & 1) != prk;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const int set = (jl * kBlocks + b) * MT + mt;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 u = remote ? tc::ld_dsmem_v4(tc::mapa_shared(smem_u32(&bfs[(set * 4 + q) * 32 + lane]), j & 1))
                                       : bfs[(set * 4 + q) * 32 + lane];
                bf[mt][4 * q] = u.x;
                bf[mt][4 * q + 1] = u.y;
                bf[mt][4 * q + 2] = u.z;
                bf[mt][4 * q + 3] = u.w;
              }
              const float2 n2 = remote ? tc::ld_dsmem_f2(tc::mapa_shared(smem_u32(&nss[set * 32 + lane]), j & 1))
                                       : nss[set * 32 + lane];
              ns[mt][0] = n2.x;
              ns[mt][1] = n2.y;
            }
          }
        }
        if (live) live = tc::wait_or_abort(full0 + 8 * s, ph, p.err, abort_flag);
        if constexpr (kRegB) {
          // The epilogue's buffer is free once it has read the previous tile.
          if (tl > 0 && live) live = tc::wait_or_abort(red_empty, (tl - 1) & 1, p.err, abort_flag);
        }
        live = __all_sync(0xFFFFFFFFu, live);
        if (live) {
          const uint8_t* blk = smem + s * kStageBytes + (16 * kTPW * rq + g) * kRowBytes + 34 * b;
#pragma unroll
          for (int r0 = 0; r0 < kTPW; r0 += kG) {
            uint32_t wg[kG][2], wh[kG][2];        // code words 2t, 2t + 1 of rows g, g + 8
            float dg[kG], dh[kG];
            float c[kG][MT][4];
#pragma unroll
            for (int i = 0; i < kG; ++i) {
              const uint8_t* rg = blk + 16 * (r0 + i) * kRowBytes;
              const uint8_t* rh = rg + 8 * kRowBytes;
              load_codes<kA>(rg, t4, wg[i][0], wg[i][1]);
              load_codes<kA>(rh, t4, wh[i][0], wh[i][1]);
              dg[i] = load_d(rg);
              dh[i] = load_d(rh);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {          // code word 2t + h: codes 16h .. 16h + 15 of the block
              uint32_t sg[kG], sh[kG];
#pragma unroll
              for (int i = 0; i < kG; ++i) {
                sg[i] = wg[i][h] >> 8;
                sh[i] = wh[i][h] >> 8;
              }
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const int st = 4 * h + x;
                const uint32_t m = 0x00030003u << (2 * x);
#pragma unroll
                for (int i = 0; i < kG; ++i) {
                  const uint32_t a0 = wg[i][h] & m, a1 = wh[i][h] & m, a2 = sg[i] & m, a3 = sh[i] & m;
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt) {
                    if (st == 0)                   // rows g and g + 8 start alike, from the offset
                      mma_bf16_16816_c(c[i][mt], a0, a1, a2, a3, bf[mt][0], bf[mt][1], ns[mt][0], ns[mt][1]);
                    else
                      mma_bf16_16816(c[i][mt], a0, a1, a2, a3, bf[mt][2 * st], bf[mt][2 * st + 1]);
                  }
                }
              }
            }
#pragma unroll
            for (int i = 0; i < kG; ++i)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                if constexpr (kRegB) {
                  red[((kTPW * rq + r0 + i) * MT + mt) * 32 + lane] =
                      make_float4(dg[i] * c[i][mt][0], dg[i] * c[i][mt][1], dh[i] * c[i][mt][2], dh[i] * c[i][mt][3]);
                } else {
                  float* t = tot[r0 + i][mt];
                  t[0] = fmaf(dg[i], c[i][mt][0], t[0]);
                  t[1] = fmaf(dg[i], c[i][mt][1], t[1]);
                  t[2] = fmaf(dh[i], c[i][mt][2], t[2]);
                  t[3] = fmaf(dh[i], c[i][mt][3], t[3]);
                }
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
          // Tile done: hand the sums to the epilogue.
          j = 0;
          if constexpr (!kRegB) {
            if (tl > 0 && live) live = tc::wait_or_abort(red_empty, (tl - 1) & 1, p.err, abort_flag);
            live = __all_sync(0xFFFFFFFFu, live);
#pragma unroll
            for (int rt = 0; rt < kTPW; ++rt)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                red[((kTPW * rq + rt) * MT + mt) * 32 + lane] =
                    make_float4(tot[rt][mt][0], tot[rt][mt][1], tot[rt][mt][2], tot[rt][mt][3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) tot[rt][mt][i] = 0.f;
              }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(red_full);
          ++tl;
        }
      }
    };
    if (b & 1)
      run(std::integral_constant<int, 1>{});
    else if (b & 2)
      run(std::integral_constant<int, 2>{});
    else
      run(std::integral_constant<int, 0>{});
  }
  // Every CTA of the cluster stays until all are done: peers' st.async into
  // rank 0's shared memory and rank 0's arrives on the peers' barriers have
  // all landed before any CTA exits.
  if (clustered) tc::cluster_sync();
}

// ---------------------------------------------------------------- host side
constexpr int kBudget3 = 74 * 1024;    // dynamic shared memory of a 3-CTA-per-SM variant
constexpr int kBudget2 = 110 * 1024;   // of a 2-CTA-per-SM variant
constexpr int kBudget1 = 220 * 1024;   // of a 1-CTA-per-SM variant

template <int MT, bool kRegB, int kOcc, bool kPair = false>
struct Variant {
  static constexpr auto kernel = q2_stream_kernel<MT, kRegB, kOcc, kPair>;
  static constexpr int kBudget = kOcc == 3 ? kBudget3 : (kOcc == 2 ? kBudget2 : kBudget1);
};

// Dynamic shared memory opt-in and the whole carveout, once per device.
template <int MT, bool kRegB, int kOcc, bool kPair = false>
cudaError_t set_attrs() {
  static AttrLatch latch;
  using V = Variant<MT, kRegB, kOcc, kPair>;
  return set_smem_attrs(V::kernel, latch, V::kBudget, true);
}

// Clusters of s CTAs of a variant resident at once (0 if the query failed),
// with the variant's shared-memory budget. Cached per device.
template <int MT, bool kRegB, int kOcc, bool kPair = false>
int cluster_capacity(int s) {
  static std::atomic<int> cache[kMaxDevices][kMaxSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::atomic<int>& slot = cache[dev][s];
  int v = slot.load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  using V = Variant<MT, kRegB, kOcc, kPair>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s);
  cfg.blockDim = dim3(threads_for(kOcc, MT));
  cfg.dynamicSmemBytes = V::kBudget;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = s;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (set_attrs<MT, kRegB, kOcc, kPair>() != cudaSuccess || cudaOccupancyMaxActiveClusters(&n, V::kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();            // the query's failure is not the caller's error
    n = 0;
  }
  slot.store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n > 0 ? n : 0;
}

// One launch configuration: variant, cluster size, clusters and ring depth.
struct Plan {
  int mt = 1;
  bool regb = false;
  int occ = 2;
  int splits = 1, clusters = 1, ring = 2;
  bool pair = false;   // no K split; the two CTAs of a cluster share the B-fragment sets
  int red_off = 0, recv_off = 0, bf_off = 0, ns_off = 0, smem = 0;
  double cost = -1.0;
};

template <int MT>
void layout(Plan& pl, int stages, int budget) {
  using Z = Sizes<MT>;
  const int nsmax = (stages + pl.splits - 1) / pl.splits;
  const int bfsets = pl.regb ? 0 : (pl.pair ? (nsmax + 1) / 2 : nsmax) * kBlocks * MT;
  const int fixed = Z::kRed + 2 * (pl.splits - 1) * Z::kSlot + bfsets * (32 * 64 + 32 * 8);
  pl.ring = std::min(kMaxRing, (budget - fixed) / kStageBytes);
  pl.red_off = pl.ring * kStageBytes;
  pl.recv_off = pl.red_off + Z::kRed;
  pl.bf_off = pl.recv_off + 2 * (pl.splits - 1) * Z::kSlot;
  pl.ns_off = pl.bf_off + bfsets * 32 * 64;
  pl.smem = pl.ns_off + bfsets * 32 * 8;
}

// Relative throughput of an SM running 1, 2 or 3 CTAs of a call: the decode
// (ALU pipe) and the MMAs (tensor pipe) of a warp do not overlap on this GPU,
// and more warps keep both pipes fed (measured: about 1.45x from one CTA to
// three).
constexpr double kSmRate[4] = {0.0, 1.0, 1.15, 1.45};
// Cross-CTA reduction of a tile when K is split, in items (measured on GB300
// at about a third of an item per tile).
constexpr double kSplitTileCost = 0.35;

template <int MT, bool kRegB, int kOcc>
void consider(Plan& best, int splits, int tiles, int stages, int num_sms, bool pair = false) {
  if (pair && (kRegB || splits != 1)) return;
  Plan pl;
  pl.mt = MT;
  pl.regb = kRegB;
  pl.occ = kOcc;
  pl.splits = splits;
  pl.pair = pair;
  layout<MT>(pl, stages, Variant<MT, kRegB, kOcc>::kBudget);
  if (pl.ring < 2) return;
  const int nsmax = (stages + splits - 1) / splits;
  // Paired plans: clusters of two CTAs; pl.clusters counts CTAs (even).
  const int csize = pair ? 2 : splits;
  int cap = 0;
  if constexpr (MT == 2 && !kRegB && kOcc == 1) {   // the only paired variant
    cap = pair ? cluster_capacity<MT, false, kOcc, true>(2) : cluster_capacity<MT, kRegB, kOcc>(csize);
  } else {
    if (pair) return;
    cap = cluster_capacity<MT, kRegB, kOcc>(csize);
  }
  // At most two CTAs of the call per SM: the next call's CTAs find a free
  // slot on every SM and load their weights while this call finishes.
  int clusters = pair ? std::min({tiles, cap > 0 ? 2 * cap : kOcc * num_sms, 2 * num_sms}) & ~1
                      : std::min({tiles, cap > 0 ? cap : (kOcc * num_sms) / splits, (2 * num_sms) / splits});
  if (clusters < (pair ? 2 : 1)) return;
  pl.clusters = clusters;
  // Work of the busiest SM, in (tile, stage) items of 64 x 1024 weights,
  // over the rate of an SM holding that many CTAs.
  const int per_sm = std::min(3, (clusters * splits + num_sms - 1) / num_sms);
  const int tpc = (tiles + clusters - 1) / clusters;   // tiles of the busiest cluster
  pl.cost = (static_cast<double>(tpc) * nsmax + (splits > 1 ? kSplitTileCost * tpc : 0.0)) * per_sm / kSmRate[per_sm];
  if (best.cost < 0 || pl.cost < best.cost - 1e-9) best = pl;
}

// The launch plan for (N, K, M tile) on the current device: the cluster size
// (K split), the variant and the number of persistent clusters (one wave)
// that minimise the busiest SM's work. It depends on N, K and the device,
// never on the activation rows, so a row's result does not depend on the
// other rows of the call.
template <int MT>
Plan choose_plan(int tiles, int stages, int num_sms, int only_splits = 0) {
  Plan best;
  for (int s = 1; s <= kMaxSplits && s <= stages; ++s) {
    if (only_splits > 0 && s != only_splits) continue;
    if (s == stages) {
      if constexpr (MT == 1) consider<1, true, 3>(best, s, tiles, stages, num_sms);
      consider<MT, true, 2>(best, s, tiles, stages, num_sms);
    } else {
      if constexpr (MT == 1) consider<1, false, 2>(best, s, tiles, stages, num_sms);
      consider<MT, false, 1>(best, s, tiles, stages, num_sms);
    }
  }
  // Two column tiles with no K split need the B fragments of both for every
  // stage; when they do not fit, a pair of CTAs shares them.
  if (MT == 2 && best.cost < 0 && only_splits <= 1 && stages > 1)
    consider<MT, false, 1>(best, 1, tiles, stages, num_sms, true);
  return best;
}

// Plans cached per (device, N, K, M tile).
struct PlanKey {
  int dev, N, K, mt;
  bool operator==(const PlanKey& o) const { return dev == o.dev && N == o.N && K == o.K && mt == o.mt; }
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

template <int MT, bool kRegB, int kOcc, bool kPair = false>
cudaError_t launch_variant(const CUtensorMap& mw, const StreamParams& p, bool pdl, int smem, cudaStream_t s) {
  cudaError_t e = set_attrs<MT, kRegB, kOcc, kPair>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.clusters * p.splits);
  cfg.blockDim = dim3(threads_for(kOcc, MT));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = kPair ? 2 : p.splits;
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
  return cudaLaunchKernelEx(&cfg, Variant<MT, kRegB, kOcc, kPair>::kernel, mw, p);
}

}  // namespace mmas

namespace mmas {
// The plan of a shape and M tile on the current device, cached. The K split
// (and so every row's summation order) is the one of the 8-row plan for
// every M, so a row's result does not depend on how many rows the call has.
cudaError_t plan_for(const GemvArgs& a, int mt, Plan& pl) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int tiles = (a.N + BM - 1) / BM, stages = a.K / (kBlocks * 128);
  const PlanKey key{dev, a.N, a.K, mt};
  PlanCache& pc = plan_cache();
  {
    std::lock_guard<std::mutex> lk(pc.mu);
    for (int i = 0; i < pc.n; ++i)
      if (pc.key[i] == key) {
        pl = pc.plan[i];
        return cudaSuccess;
      }
  }
  pl = choose_plan<1>(tiles, stages, a.num_sms);
  if (pl.cost >= 0 && mt == 2) pl = choose_plan<2>(tiles, stages, a.num_sms, pl.splits);
  std::lock_guard<std::mutex> lk(pc.mu);
  const int i = pc.n < kPlanCache ? pc.n++ : (pc.next++ % kPlanCache);
  pc.key[i] = key;
  pc.plan[i] = pl;
  return cudaSuccess;
}
}  // namespace mmas

// An 8-row plan needs a rank's B-fragment sets (18 KB per stage) and a ring
// of two stages in one CTA's shared memory: with 8 K splits, up to 7 stages
// per rank (K <= 57344). Longer K runs on the short-CTA kernel. The answer
// depends on N, K and the device only.
bool q2_gemm_stream_fits(const GemvArgs& a) {
  mmas::Plan pl;
  return mmas::plan_for(a, 1, pl) == cudaSuccess && pl.cost >= 0;
}

// Requires K % 1024 == 0 (checked by the caller): a row is then 34 * K / 128
// bytes, a multiple of 16, and each raw stage of 8 blocks starts on a 16-byte
// boundary (the TMA box's x = 136 * stage elements of 2 bytes).
cudaError_t launch_q2_gemm_stream(const GemvArgs& a, cudaStream_t s) {
  using namespace mmas;
  const int mt = a.M > 8 ? 2 : 1;
  const int tiles = (a.N + BM - 1) / BM, stages = a.K / (kBlocks * 128);
  Plan pl;
  cudaError_t e = plan_for(a, mt, pl);
  if (e != cudaSuccess) return e;
  if (pl.cost < 0) {
    if (mt == 1) return cudaErrorInvalidConfiguration;
    // No two-column-tile plan with that split fits: two launches of 8 rows.
    GemvArgs lo = a, hi = a;
    lo.M = 8;
    hi.M = a.M - 8;
    hi.A = static_cast<const uint16_t*>(a.A) + static_cast<size_t>(8) * a.lda;
    hi.C = static_cast<uint16_t*>(a.C) + static_cast<size_t>(8) * a.ldc;
    const cudaError_t e1 = launch_q2_gemm_stream(lo, s);
    return e1 != cudaSuccess ? e1 : launch_q2_gemm_stream(hi, s);
  }
  const uint64_t G = static_cast<uint64_t>(a.K / 128);
  CUtensorMap mw;
  e = cached_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.W, 17 * G, static_cast<uint64_t>(a.N), 34 * G,
                    kBlocks * 17, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  StreamParams p;
  p.A = static_cast<const uint16_t*>(a.A);
  p.C = static_cast<uint16_t*>(a.C);
  p.lda = a.lda;
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.tiles = tiles;
  p.stages = stages;
  p.splits = pl.splits;
  p.clusters = pl.clusters;
  p.ring = pl.ring;
  p.red_off = pl.red_off;
  p.recv_off = pl.recv_off;
  p.bf_off = pl.bf_off;
  p.ns_off = pl.ns_off;
  p.err = a.err;
  if (pl.mt == 1) {
    if (pl.regb) return pl.occ == 3 ? launch_variant<1, true, 3>(mw, p, a.pdl, pl.smem, s)
                                    : launch_variant<1, true, 2>(mw, p, a.pdl, pl.smem, s);
    if (pl.occ == 2) return launch_variant<1, false, 2>(mw, p, a.pdl, pl.smem, s);
    return launch_variant<1, false, 1>(mw, p, a.pdl, pl.smem, s);
  }
  if (pl.regb) return launch_variant<2, true, 2>(mw, p, a.pdl, pl.smem, s);
  if (pl.pair) return launch_variant<2, false, 1, true>(mw, p, a.pdl, pl.smem, s);
  return launch_variant<2, false, 1>(mw, p, a.pdl, pl.smem, s);
}

}  // namespace wqp
