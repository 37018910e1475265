// Q2_0 GEMM for 1 <= M <= 8 per launch (the C ABI splits M <= 16 into 8-row
// launches) on the warp-level tensor-core path
// (mma.sync m16n8k16, BF16 operands, FP32 accumulation), swap-AB: the MMA's
// 16 "rows" are weight rows n, its 8 "columns" are activation rows m.
//
// What it computes is the ternary Q2_0 product of
// "spark_model/layers/ops/gemv_q2_vec.rs" (module docs; the formula of the
// test helper `gemv_row`):
//   C[m, n] = bf16( sum_k A[m, k] * (c[n, k] - 1) * d[n, k / 128] ),
// the same result as q2_gemm_tc, within the tensor-core tolerance of
// "metrale_model_layers/layers/ops/w8a16_gemm_m16.rs" (module docs: the
// tensor core reduces 16 K-products in its own order).
//
// Why registers instead of tensor memory: the GEMV is a weight stream, and
// every weight must pass through the converter exactly once. Feeding tcgen05
// through tensor memory puts a store -> commit -> barrier -> MMA -> commit ->
// barrier round trip on every 128-K group; here each warp turns its own code
// words into MMA operands in registers and issues the MMAs itself, so nothing
// waits on another warp until the stage's sums are added.
//
// Layout of one CTA (BM = 64 or 96 weight rows x the CTA's K range):
//   warps 0..7  compute: warp w owns block w (128 K) of every stage, for all
//               BM / 16 row tiles of the CTA;
//   warp 8      producer: TMA of raw stages (BM rows x 8 blocks x 34 bytes).
// Per 128-K block b and thread (g = lane / 4, t = lane % 4):
//   * A fragment: code words 2t and 2t + 1 of the block, rows g and g + 8 of
//     a tile. Word bits 2q..2q+1 hold code q (q < 16). The pair of 16-bit
//     lanes (code x, code 8 + x), masked in place by
//     (word & 0x00030003 << 2x), is the BF16 pair (c_x 4^x, c_{8+x} 4^x) *
//     2^-133 (a subnormal or the smallest normal, exact); (word >> 8) gives
//     codes (4 + x, 12 + x).
//   * B fragment: activation row m = g (rows past M repeat row M - 1): the 32
//     activations of k = 128 b + 32 t .. + 31, paired the same way and
//     multiplied by 2^(64 - 2x), so every product is c * a * 2^-69 exactly.
//     Built once per block, in registers, and used for all row tiles.
//   * Each tile's chain starts from -2^-69 * sum_k a (four MMAs per block
//     with the raw activations as the A operand and -2^-69 as B, run once
//     per block), so it ends at 2^-69 * sum_k (c - 1) a.
//   * acc += d * chain, and C = bf16(acc * 2^69).
// Reduction: the 8 warps' sums are added in warp order in shared memory.
// Split-K: the CTAs of a cluster split the K stages. Rank 0 owns the tile:
// every other rank sends its sums into rank 0's shared memory with st.async
// (completing on an mbarrier of rank 0) and exits at once, freeing its SM
// for the next grid; rank 0 adds them in rank order and stores.
#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace wqp {
namespace mma {

constexpr int kBlocks = 8;                   // 128-K blocks per raw stage (1024 K)
constexpr int kCompute = kBlocks;            // compute warps: one per 128-K block of a stage
constexpr int kThreads = (kCompute + 1) * 32;
constexpr int kRowBytes = kBlocks * 34;      // 272: 17 x 16 bytes
constexpr int kMaxSplits = 8;                // CTAs per cluster (K split) at most (portable size)

// MT: m tiles of 8 activation rows per launch (1 is the one launched: a
// 16-row form measured slower than two 8-row launches).
// kMulti: a CTA runs more than one raw stage (two raw buffers, one refilled
// while the other is consumed); otherwise exactly one.
// kBM: weight rows per CTA (64, or 96 for grids that would need a fourth
// CTA slot per SM with 64).
template <int MT, bool kMulti, int kBM>
struct Cfg {
  static constexpr int kTiles = kBM / 16;                        // 16-row MMA tiles
  static constexpr int kStageBytes = kBM * kRowBytes;            // raw stage (17408 or 26112)
  static constexpr int SW = kMulti ? 2 : 1;                      // raw stage buffers
  static constexpr int kRawOff = 0;
  // Every compute warp's partial sums (tiles x MT x 32 lanes x 4 floats),
  // written over the raw buffers once all of them are consumed.
  static constexpr int kSlot = kTiles * MT * 32 * 16;
  static constexpr int kRedOff = 0;
  static constexpr int kBody = SW * kStageBytes > kCompute * kSlot ? SW * kStageBytes : kCompute * kSlot;
  // Multi-stage CTAs: the next stage's activations of each warp's block,
  // copied ahead with cp.async ([warp][MT][4 chunks][32 lanes][16 bytes]).
  // Single-stage CTAs: the stage's activation rows (1024 K each), copied in
  // bulk by the TMA warp when M > 4, one row per 2064 bytes (the 16-byte pad
  // spreads the rows over the shared-memory banks).
  static constexpr int kActOff = kBody;
  static constexpr int kActWarp = MT * 4 * 32 * 16;
  static constexpr int kActPitch = kBlocks * 128 * 2 + 16;
  static constexpr int kActBytes = kMulti ? kCompute * kActWarp : 8 * MT * kActPitch;
  static constexpr int kRecvOff = kActOff + kActBytes;            // ranks 1.. of the cluster, at rank 0
  // Dynamic shared memory for a cluster of `splits` CTAs.
  static constexpr int bytes(int splits) { return kRecvOff + (splits - 1) * kSlot; }
  static_assert(kBM % 16 == 0 && kStageBytes % 128 == 0 && kRecvOff % 16 == 0, "align");
  static_assert(kTiles % 2 == 0, "row tiles run in pairs");
  static_assert(2 * (bytes(kMaxSplits) + 1024) <= 227 * 1024, "shared memory per SM");
};

struct MmaParams {
  const uint16_t* A;   // bf16 [M, lda]
  uint16_t* C;         // bf16 [M, ldc]
  int lda, ldc;
  int M, N, K;
  int stages;          // K / 1024
  int splits;          // CTAs per tile = cluster size
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

// 16-byte asynchronous global -> shared copy (L2 only), and its completion.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Cluster barrier halves: the early arrive lets every rank know its peers
// have started before anyone stores into their shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Four floats into a peer CTA's shared memory (shared::cluster address),
// completing as 16 bytes on the peer's mbarrier.
__device__ __forceinline__ void st_async_f4(uint32_t addr, float x, float y, float z, float w, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "f"(x), "f"(y), "f"(z), "f"(w), "r"(bar)
               : "memory");
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

// kOcc: CTAs per SM the registers are budgeted for.
template <int MT, bool kMulti, int kOcc, int kBM>
__global__ void __launch_bounds__(kThreads, kOcc)
    q2_mma_kernel(const __grid_constant__ CUtensorMap tmW, const MmaParams p) {
  using L = Cfg<MT, kMulti, kBM>;
  constexpr int kTiles = L::kTiles;
  constexpr int kStageBytes = L::kStageBytes;
  constexpr int SW = L::SW;
  extern __shared__ __align__(1024) uint8_t smem[];
  // full[SW], empty[SW], partial sums received, activation rows landed
  __shared__ __align__(8) uint64_t bars[2 * SW + 2];
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = p.splits;
  const int tile = blockIdx.x / splits;
  const int rank = blockIdx.x - tile * splits;   // == %cluster_ctarank
  const int n0 = tile * kBM;
  const int st0 = (rank * p.stages) / splits;
  const int T = kMulti ? ((rank + 1) * p.stages) / splits - st0 : 1;   // >= 1: splits <= stages
  const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[SW]), recv_bar = smem_u32(&bars[2 * SW]);
  const uint32_t act_bar = recv_bar + 8;
  // Single-stage CTA with more than 4 rows: the TMA warp copies the stage's
  // activation rows in bulk (fewer, larger L2 requests than 32 lanes each
  // loading their 64 bytes).
  const bool bulk_act = !kMulti && p.M > 4;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SW; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kCompute);
    }
    mbar_init(recv_bar, 1);
    mbar_init(act_bar, 1);
    mbar_fence_init();
    if (rank == 0 && splits > 1) mbar_arrive_expect_tx(recv_bar, (splits - 1) * L::kSlot);
    abort_sh = 0;
  }
  if (splits > 1) cluster_arrive_relaxed();
  __syncthreads();
  pdl_launch_dependents();

  const int g = lane >> 2, t4 = lane & 3;

  if (warp == kCompute) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tmW);
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % SW;
        if (t >= SW && !tc::wait_or_abort(empty0 + 8 * s, ((t / SW) - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(full0 + 8 * s, kStageBytes);
        tc::tma_load_2d_hint(smem_u32(smem + L::kRawOff + s * kStageBytes), &tmW, (st0 + t) * (kBlocks * 17),
                             n0, full0 + 8 * s, pol);
        issued = t + 1;
      }
      if (bulk_act) {
        pdl_wait();                               // activations may belong to the previous grid
        const int rows = min(p.M, 8 * MT);
        mbar_arrive_expect_tx(act_bar, rows * (kBlocks * 128 * 2));
        for (int m = 0; m < rows; ++m)
          bulk_g2s(smem_u32(smem + L::kActOff + m * L::kActPitch),
                   p.A + static_cast<size_t>(m) * p.lda + static_cast<size_t>(st0) * kBlocks * 128,
                   kBlocks * 128 * 2, act_bar);
      }
      // The CTA may not exit with a copy into its shared memory in flight:
      // stay until the last copies issued have landed.
      for (int t = max(0, issued - SW); t < issued; ++t) mbar_wait(full0 + 8 * (t % SW), (t / SW) & 1, p.err);
      if (bulk_act) mbar_wait(act_bar, 0, p.err);
    }
    __syncwarp();
    if (splits > 1) cluster_wait();
    return;
  }

  // -------------------------------------------------------------- compute
  // Warp w owns block w of every stage, for all 64 rows of the tile.
  const int b = warp;
  // Every rank has started (its barriers are initialised) before anyone
  // sends to rank 0; waited here, where a CTA launched early waits anyway.
  if (splits > 1) cluster_wait();
  pdl_wait();                                     // activations (and C) may belong to the previous grid
  const uint16_t* arow[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = min(g + 8 * mt, p.M - 1);       // rows past M: any valid row, results unused
    arow[mt] = p.A + static_cast<size_t>(m) * p.lda + 32 * t4;
  }
  // This thread's 32 activations of the block, per m tile: straight into
  // registers for a single stage; for several, copied one stage ahead into
  // this warp's shared buffer.
  // Rows past M are never copied (no duplicate requests to the same lines):
  // their lanes read the slot of row M - 1, which some lane copies.
  uint4 act[MT][4];
  uint4* abuf = reinterpret_cast<uint4*>(smem + L::kActOff + warp * L::kActWarp);
  auto act_src = [&](int t, int mt, int q) {
    return arow[mt] + static_cast<size_t>(kBlocks * (st0 + t) + b) * 128 + 8 * q;
  };
  auto load_act = [&](int t) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (kMulti) {
          if (g + 8 * mt < p.M) cp_async16(abuf + (mt * 4 + q) * 32 + lane, act_src(t, mt, q));
        } else {
          if (!bulk_act) act[mt][q] = ld_nc_v4(act_src(t, mt, q));
        }
      }
    if constexpr (kMulti) cp_async_commit();
  };
  float tot[kTiles][MT][4];
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) tot[rt][mt][i] = 0.f;

  load_act(0);
  bool live = true;
  // One m tile at a time: its B fragments and offset, then every row tile
  // against them (for M > 8 the codes are decoded once per m tile, which
  // keeps a single set of fragments live).
  auto run = [&](auto ac) {
    constexpr int kA = decltype(ac)::value;
    for (int t = 0; t < T; ++t) {
      if constexpr (kMulti) {
        cp_async_wait_all();                        // this thread's copies of stage t
        __syncwarp();                               // and the other lanes' (rows past M)
      }
      const int s = t % SW;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t r[16];
        if constexpr (kMulti) {
          const int src = ((min(g + 8 * mt, p.M - 1) - 8 * mt) << 2) | t4;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = abuf[(mt * 4 + q) * 32 + src];
            r[4 * q] = v.x;
            r[4 * q + 1] = v.y;
            r[4 * q + 2] = v.z;
            r[4 * q + 3] = v.w;
          }
        } else {
          if (bulk_act) {
            if (mt == 0) {
              if (live) live = tc::wait_or_abort(act_bar, 0, p.err, abort_flag);
              live = __all_sync(0xFFFFFFFFu, live);
            }
            const int m = min(g + 8 * mt, p.M - 1);
            const uint8_t* src = smem + L::kActOff + m * L::kActPitch + (b * 128 + 32 * t4) * 2;
#pragma unroll
            for (int q = 0; q < 4; ++q) act[mt][q] = *reinterpret_cast<const uint4*>(src + 16 * q);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            r[4 * q] = act[mt][q].x;
            r[4 * q + 1] = act[mt][q].y;
            r[4 * q + 2] = act[mt][q].z;
            r[4 * q + 3] = act[mt][q].w;
          }
        }
        // B fragments of the block (permuted, pre-scaled) and the offset.
        uint32_t bf[16];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const int x = st & 3, o = 8 * (st >> 2) + (x >> 1);
          const uint32_t sel = (x & 1) ? 0x7632u : 0x5410u;
          bf[2 * st] = mul_bf16x2(__byte_perm(r[o], r[o + 4], sel), prescale(x));
          bf[2 * st + 1] = mul_bf16x2(__byte_perm(r[o + 2], r[o + 6], sel), prescale(x));
        }
        float ns[2];
        offset_sums(r, t4, ns);
        if (kMulti && mt == MT - 1 && t + 1 < T) {
          __syncwarp();                             // every lane has read the buffer
          load_act(t + 1);
        }
        if (mt == 0) {
          if (live) live = tc::wait_or_abort(full0 + 8 * s, (t / SW) & 1, p.err, abort_flag);
          live = __all_sync(0xFFFFFFFFu, live);
        }
        if (live) {
          // Two row tiles at a time: their MMA chains are independent, so one
          // waits while the other issues.
          const uint8_t* blk = smem + L::kRawOff + s * kStageBytes + g * kRowBytes + 34 * b;
#pragma unroll
          for (int r0 = 0; r0 < kTiles; r0 += 2) {
            uint32_t wg[2][2], wh[2][2];           // code words 2t, 2t + 1 of rows g, g + 8
            float dg[2], dh[2], c[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint8_t* rg = blk + 16 * (r0 + i) * kRowBytes;
              const uint8_t* rh = rg + 8 * kRowBytes;
              load_codes<kA>(rg, t4, wg[i][0], wg[i][1]);
              load_codes<kA>(rh, t4, wh[i][0], wh[i][1]);
              dg[i] = load_d(rg);
              dh[i] = load_d(rh);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {          // code word 2t + h: codes 16h .. 16h + 15 of the block
              const uint32_t sg[2] = {wg[0][h] >> 8, wg[1][h] >> 8};
              const uint32_t sh[2] = {wh[0][h] >> 8, wh[1][h] >> 8};
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const int st = 4 * h + x;
                const uint32_t m = 0x00030003u << (2 * x);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  const uint32_t a0 = wg[i][h] & m, a1 = wh[i][h] & m, a2 = sg[i] & m, a3 = sh[i] & m;
                  if (st == 0)                     // rows g and g + 8 start alike, from the offset
                    mma_bf16_16816_c(c[i], a0, a1, a2, a3, bf[0], bf[1], ns[0], ns[1]);
                  else
                    mma_bf16_16816(c[i], a0, a1, a2, a3, bf[2 * st], bf[2 * st + 1]);
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              tot[r0 + i][mt][0] = fmaf(dg[i], c[i][0], tot[r0 + i][mt][0]);
              tot[r0 + i][mt][1] = fmaf(dg[i], c[i][1], tot[r0 + i][mt][1]);
              tot[r0 + i][mt][2] = fmaf(dh[i], c[i][2], tot[r0 + i][mt][2]);
              tot[r0 + i][mt][3] = fmaf(dh[i], c[i][3], tot[r0 + i][mt][3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
  };
  if (b & 1)
    run(std::integral_constant<int, 1>{});
  else if (b & 2)
    run(std::integral_constant<int, 2>{});
  else
    run(std::integral_constant<int, 0>{});

  // ------------------------------------------------------------ reduce + store
  // The 8 warps' sums (one block each) are added in warp order through
  // shared memory laid over the consumed raw buffers. Ranks 1.. send the
  // result to rank 0 (slot rank - 1) with st.async and leave; rank 0 adds the
  // slots in rank order and stores.
  constexpr int kItems = kTiles * MT * 32;        // float4 items of one warp's sums
  float4* red = reinterpret_cast<float4*>(smem + L::kRedOff);
  asm volatile("bar.sync 1, %0;" ::"r"(kCompute * 32) : "memory");   // raw buffers consumed
#pragma unroll
  for (int rt = 0; rt < kTiles; ++rt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
      red[warp * kItems + (rt * MT + mt) * 32 + lane] =
          make_float4(tot[rt][mt][0], tot[rt][mt][1], tot[rt][mt][2], tot[rt][mt][3]);
  asm volatile("bar.sync 1, %0;" ::"r"(kCompute * 32) : "memory");
  const int item = threadIdx.x;                   // (tile, m tile, lane) of a warp's fragment
  if (item >= kItems) return;
  float4 v = red[item];
#pragma unroll
  for (int w = 1; w < kCompute; ++w) {            // warp (block) order
    const float4 u = red[w * kItems + item];
    v.x += u.x;
    v.y += u.y;
    v.z += u.z;
    v.w += u.w;
  }
  if (rank != 0) {
    const uint32_t dst = tc::mapa_shared(smem_u32(smem + L::kRecvOff + (rank - 1) * L::kSlot + item * 16), 0);
    st_async_f4(dst, v.x, v.y, v.z, v.w, tc::mapa_shared(recv_bar, 0));
    return;
  }
  // Every peer sends, even one whose own waits gave up (each of those is
  // bounded by kWaitLimitNs), so rank 0 waits three times as long: it never
  // leaves while a peer may still write into its shared memory.
  bool ok = splits == 1 || mbar_wait_ns(recv_bar, 0, p.err, 3 * kWaitLimitNs);
  ok = ok && *abort_flag == 0;
  if (!ok) return;
  const float4* recv = reinterpret_cast<const float4*>(smem + L::kRecvOff) + item;
  for (int q = 1; q < splits; ++q) {              // rank order
    const float4 u = recv[(q - 1) * kItems];
    v.x += u.x;
    v.y += u.y;
    v.z += u.z;
    v.w += u.w;
  }
  const float kUnscale = __uint_as_float((127u + 69u) << 23);   // 2^69
  const int rt = item / (MT * 32), mt = (item / 32) % MT, ln = item % 32;
  const int r = 16 * rt + (ln >> 2), m = 8 * mt + 2 * (ln & 3);
  const float acc[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rr = r + 8 * (i >> 1), mm = m + (i & 1);
    if (mm < p.M && n0 + rr < p.N) p.C[static_cast<size_t>(mm) * p.ldc + n0 + rr] = f32_to_bf16_rn(acc[i] * kUnscale);
  }
}

// ---------------------------------------------------------------- host side
// The compiled variants: (m tiles, several stages per CTA, CTAs per SM, rows
// per CTA). Single-stage calls run 64-row CTAs three to an SM; a grid that
// does not fit that runs 96-row CTAs three to an SM when those fit, else
// 64-row CTAs four to an SM (56 registers).
template <int MT, bool kMulti, int kOcc, int kBM>
struct Variant {
  static constexpr auto kernel = q2_mma_kernel<MT, kMulti, kOcc, kBM>;
};

// Opt-in shared memory above 48 KB (up to the largest cluster's size) and the
// whole carveout (several CTAs per SM). Set once, before the first launch or
// occupancy query.
template <int MT, bool kMulti, int kOcc, int kBM>
cudaError_t set_attrs() {
  static AttrLatch latch;
  return set_smem_attrs(Variant<MT, kMulti, kOcc, kBM>::kernel, latch, Cfg<MT, kMulti, kBM>::bytes(kMaxSplits), true);
}

// CTAs of a variant resident at once in clusters of s (0 if the query
// failed). Cached per device.
template <int MT, bool kMulti, int kOcc, int kBM>
int resident_ctas(int s) {
  static std::atomic<int> cache[kMaxDevices][kMaxSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = cache[dev][s].load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<MT, kMulti, kBM>::bytes(s);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = s;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (set_attrs<MT, kMulti, kOcc, kBM>() != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, Variant<MT, kMulti, kOcc, kBM>::kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();            // the query's failure is not the caller's error
    n = 0;
  }
  cache[dev][s].store(n > 0 ? n * s : -1, std::memory_order_relaxed);
  return n > 0 ? n * s : 0;
}

// K split per tile: minimise (waves of resident CTAs) x (stages per CTA);
// ties go to the larger split (more copies in flight). Depends on N, K and
// the device only, never on M, so a row's summation order does not depend on
// the other rows of the call.
int choose_splits(int tiles, int stages, int num_sms) {
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= kMaxSplits && s <= stages; ++s) {
    const int per_cta = (stages + s - 1) / s;
    int slots = per_cta > 1 ? resident_ctas<1, true, 3, 64>(s) : resident_ctas<1, false, 4, 64>(s);
    if (slots <= 0) slots = 3 * num_sms;
    const long long ctas = static_cast<long long>(tiles) * s;
    const long long waves = (ctas + slots - 1) / slots;
    const long long cost = waves * per_cta;
    if (best_cost < 0 || cost <= best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  return best;
}

template <int MT, bool kMulti, int kOcc, int kBM>
cudaError_t launch_variant(const CUtensorMap& mw, const MmaParams& p, int tiles, bool pdl, cudaStream_t s) {
  cudaError_t e = set_attrs<MT, kMulti, kOcc, kBM>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * p.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<MT, kMulti, kBM>::bytes(p.splits);
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
  return cudaLaunchKernelEx(&cfg, Variant<MT, kMulti, kOcc, kBM>::kernel, mw, p);
}

}  // namespace mma

// Requires K % 1024 == 0 (checked by the caller): a row is then 34 * K / 128
// bytes, a multiple of 16, and each raw stage of 8 blocks starts on a 16-byte
// boundary (the TMA box's x = 136 * stage elements of 2 bytes).
cudaError_t launch_q2_gemm_mma(const GemvArgs& a, cudaStream_t s) {
  using namespace mma;
  // At least two 64-row tiles per SM: the persistent kernel (weights read once
  // for up to 16 rows; B fragments built once per CTA), where its plan fits
  // (K <= 57344). Otherwise one short CTA per (tile, stage range) and 8
  // activation rows per launch. The choice depends on the shape only, so a
  // row's result does not depend on M.
  if ((a.N + 63) / 64 >= 2 * a.num_sms && q2_gemm_stream_fits(a)) return launch_q2_gemm_stream(a, s);
  if (a.M > 8) {
    GemvArgs lo = a, hi = a;
    lo.M = 8;
    hi.M = a.M - 8;
    hi.A = static_cast<const uint16_t*>(a.A) + static_cast<size_t>(8) * a.lda;
    hi.C = static_cast<uint16_t*>(a.C) + static_cast<size_t>(8) * a.ldc;
    const cudaError_t e1 = launch_q2_gemm_mma(lo, s);
    return e1 != cudaSuccess ? e1 : launch_q2_gemm_mma(hi, s);
  }
  const uint64_t G = static_cast<uint64_t>(a.K / 128);
  // Raw stages of `bm` rows: boxes of 8 blocks x bm rows.
  CUtensorMap mw;
  auto map = [&](int bm) {
    return cached_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.W, 17 * G, static_cast<uint64_t>(a.N), 34 * G,
                         kBlocks * 17, static_cast<uint32_t>(bm), CU_TENSOR_MAP_SWIZZLE_NONE);
  };
  MmaParams p;
  p.A = static_cast<const uint16_t*>(a.A);
  p.C = static_cast<uint16_t*>(a.C);
  p.lda = a.lda;
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.stages = a.K / (kBlocks * 128);
  p.splits = 1;
  p.err = a.err;
  const int tiles = (a.N + 63) / 64;
  p.splits = choose_splits(tiles, p.stages, a.num_sms);
  const bool multi = (p.stages + p.splits - 1) / p.splits > 1;
  cudaError_t e;
  // One 8-row activation tile (MT = 1): the C ABI calls this on 8-row chunks.
  if (multi) return (e = map(64)) != cudaSuccess ? e : launch_variant<1, true, 3, 64>(mw, p, tiles, a.pdl, s);
  // Three CTAs per SM spread a grid that fits them over more SMs (the cluster
  // scheduler fills an SM's free slots before the next SM's). A grid of
  // 64-row CTAs that does not fit runs as 96-row CTAs, three to an SM, when
  // those fit in one wave (7168 x 5120: 5.4 -> 4.8 us at M = 1); else as
  // 64-row CTAs four to an SM. The K split is the same in every case, so a
  // row's summation order depends on K only.
  auto fits = [&](int ctas, int slots) { return ctas <= (slots > 0 ? slots : 3 * a.num_sms); };
  if (fits(tiles * p.splits, resident_ctas<1, false, 3, 64>(p.splits)))
    return (e = map(64)) != cudaSuccess ? e : launch_variant<1, false, 3, 64>(mw, p, tiles, a.pdl, s);
  const int tiles96 = (a.N + 95) / 96;
  if (fits(tiles96 * p.splits, resident_ctas<1, false, 3, 96>(p.splits)))
    return (e = map(96)) != cudaSuccess ? e : launch_variant<1, false, 3, 96>(mw, p, tiles96, a.pdl, s);
  return (e = map(64)) != cudaSuccess ? e : launch_variant<1, false, 4, 64>(mw, p, tiles, a.pdl, s);
}

}  // namespace wqp
