// Tensor-core (tcgen05) swap-AB decode GEMM for packed weights, 1 <= M <= 16.
//
// FP8 E4M3 with FP32 128x128 block scales
// ("metrale_model_layers/layers/ops/w8a16_gemm_m16.rs": doc of
// `w8a16_gemm_m16` for the operands and the 16-row M tile; module docs for
// the block scale being folded once per 128-K block onto an FP32 outer
// accumulator, never per element and never into BF16), and ternary Q2_0 with
// its inline fp16 scale per 128-K group ("spark_model/layers/ops/gemv_q2_vec.rs",
// module docs), whose scale is folded the same way.
//
// Swap-AB: the 128 weight rows of a tile are the MMA's M side, and the M <= 16
// activation rows, zero-padded to 16, are its N side:
//   D[n, m] = sum_k W[n, k] * A[m, k]   (tcgen05.mma kind::f16, M=128 N=16 K=16)
// Every E4M3 value and every Q2_0 code - 1 is exactly representable in BF16,
// so the products are exact. The tensor core reduces each 16-K step in its
// own order, so the result is not bit-identical to the scalar kernels. Each
// output row still depends only on its own activation row.
//
// One CTA = one 128-row tile x a contiguous range of 128-K groups. Roles:
//   warp 20     TMA: raw weight tiles (FP8: [128 rows x 128 B] with 128-byte
//               swizzle; Q2_0: [128 rows x 272 B] = 8 groups) and activation
//               tiles [16 rows x 64 K] x 2 (128-byte swizzle, rows past M
//               zero-filled), through mbarrier rings;
//   warps 0..15 decode one row and a quarter group (32 K) per thread into the
//               K-major BF16 operand tile (128-byte swizzle, like the
//               activations);
//   warp 21     allocates TMEM and issues the 8 MMAs of each group into its
//               own 16-column accumulator slot, then commits;
//   warps 16..19 fold each group: tcgen05.ld of the slot (lane = weight row,
//               column = activation row), acc[m] += s * D[m] in FP32.
// When N is small, K is split over a thread-block cluster of up to 8 CTAs.
// The partial sums are added in rank order through distributed shared memory
// (deterministic, no global scratch).
#include "decode.cuh"
#include "tc.cuh"

namespace wqp {
namespace tc {

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BN = 16;             // activation rows (MMA N)
constexpr int GK = 128;            // K per group = scale granularity
constexpr int kConvWarps = 16;     // converters: row quarter = warp % 4, K quarter = warp / 4
constexpr int kEpiWarp0 = 16;      // epilogue warps 16..19 (TMEM lane quarter = warp % 4)
constexpr int kTmaWarp = 20;
constexpr int kMmaWarp = 21;
constexpr int kThreads = 22 * 32;
constexpr int SA = 8;              // activation stages (prefetched independently)
constexpr int NACC = 4;            // TMEM accumulator slots
constexpr int NSCL = 8;            // row-scale ring (Q2_0 d), deeper than SO + NACC
constexpr uint32_t kTmemCols = 64; // NACC * 16, rounded to a power of two >= 32
constexpr int kOpBytes = BM * GK * 2;      // 32 KB
constexpr int kActBytes = BN * GK * 2;     // 4 KB

struct TcParams {
  const float* scales;     // FP8: [ceil(N/128), K/128]; Q2_0: unused
  uint16_t* C;
  int M, N, K, ldc;
  int splits;              // CTAs per tile (cluster size)
  int stages;              // raw stages per tile (K / (128 * GPR))
  unsigned* err;
};

// Operand layout: a group's 128 rows x 128 K BF16 tile is two K-major blocks
// of 64 K, each [128 rows x 128 B] with the 128-byte swizzle (16-byte chunk c
// of row r stored at chunk c ^ (r % 8); 8-row atoms of 1024 B). cc is the
// 8-K chunk index within the group (0..15).
__device__ __forceinline__ uint8_t* op_chunk(uint8_t* op, int r, int cc) {
  return op + (cc >> 3) * (BM * 128) + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
}

// ------------------------------------------------------------------ formats
// FP8 E4M3: one group per raw stage, [128 rows x 128 B], 128-byte swizzle.
struct Fp8Tc {
  static constexpr int kGPR = 1;
  static constexpr int kSR = 4;
  static constexpr int kSO = 3;
  static constexpr int kRawBytes = BM * GK;
  static constexpr bool kRowScale = false;
  __device__ static void issue_raw(const CUtensorMap* m, uint32_t dst, int g0, int n0, uint32_t bar,
                                   uint64_t pol) {
    tma_load_2d_hint(dst, m, g0 * GK, n0, bar, pol);
  }
  // Row r, K quarter kq (32 K) of group gi of the raw stage -> operand stage op.
  __device__ static void convert(const uint8_t* raw, int, int r, int kq, uint8_t* op, float&) {
    const uint8_t* row = raw + r * 128;
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const int c = kq * 2 + c2;                                   // 16-byte chunk = 16 K
      const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
      uint4 lo, hi;
      e4m3x4_to_bf16(v.x, lo.x, lo.y);
      e4m3x4_to_bf16(v.y, lo.z, lo.w);
      e4m3x4_to_bf16(v.z, hi.x, hi.y);
      e4m3x4_to_bf16(v.w, hi.z, hi.w);
      *reinterpret_cast<uint4*>(op_chunk(op, r, 2 * c)) = lo;
      *reinterpret_cast<uint4*>(op_chunk(op, r, 2 * c + 1)) = hi;
    }
  }
};

// Q2_0: eight groups per raw stage, [128 rows x 8 blocks x 34 B], no swizzle.
struct Q2Tc {
  static constexpr int kGPR = 8;
  static constexpr int kSR = 2;
  static constexpr int kSO = 3;
  static constexpr int kRawBytes = BM * 8 * 34;
  static constexpr bool kRowScale = true;
  __device__ static void issue_raw(const CUtensorMap* m, uint32_t dst, int g0, int n0, uint32_t bar,
                                   uint64_t pol) {
    tma_load_2d_hint(dst, m, g0 * 17, n0, bar, pol);              // 17 u16 per block
  }
  __device__ static void convert(const uint8_t* raw, int gi, int r, int kq, uint8_t* op, float& d) {
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(raw + r * 272 + gi * 34);
    if (kq == 0) d = __half2float(__ushort_as_half(blk[16]));
#pragma unroll
    for (int w2 = 0; w2 < 2; ++w2) {
      const int w = kq * 2 + w2;                                   // 16-code word of the block
      const uint32_t q = static_cast<uint32_t>(blk[2 * w]) | (static_cast<uint32_t>(blk[2 * w + 1]) << 16);
      uint32_t p[8];
      q2_decode_word(q, p);                                        // p[j] = (c_j - 1, c_{j+8} - 1)
      uint4 lo, hi;                                                // natural pairs (c_2i, c_2i+1)
      lo.x = __byte_perm(p[0], p[1], 0x5410);
      lo.y = __byte_perm(p[2], p[3], 0x5410);
      lo.z = __byte_perm(p[4], p[5], 0x5410);
      lo.w = __byte_perm(p[6], p[7], 0x5410);
      hi.x = __byte_perm(p[0], p[1], 0x7632);
      hi.y = __byte_perm(p[2], p[3], 0x7632);
      hi.z = __byte_perm(p[4], p[5], 0x7632);
      hi.w = __byte_perm(p[6], p[7], 0x7632);
      *reinterpret_cast<uint4*>(op_chunk(op, r, 2 * w)) = lo;      // k = 16 w .. 16 w + 7
      *reinterpret_cast<uint4*>(op_chunk(op, r, 2 * w + 1)) = hi;  // k = 16 w + 8 .. + 15
    }
  }
};

template <class F>
struct Layout {
  static constexpr int kOpOff = 0;
  static constexpr int kRawOff = kOpOff + F::kSO * kOpBytes;
  static constexpr int kActOff = (kRawOff + F::kSR * F::kRawBytes + 1023) / 1024 * 1024;
  static constexpr int kSclOff = kActOff + SA * kActBytes;
  static constexpr int kBytes = kSclOff + NSCL * BM * 4;
  static_assert(NSCL > F::kSO + NACC, "row-scale ring must outlive the pipeline");
  static constexpr int kAlloc = kBytes + 1024;                     // slack for 1024-byte alignment
  static_assert(BM * BN * 4 <= F::kSR * F::kRawBytes, "split-K partials alias the raw ring");
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

template <class F>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
              TcParams p) {
  using L = Layout<F>;
  constexpr int SR = F::kSR;
  constexpr int SO = F::kSO;
  constexpr int GPR = F::kGPR;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[SR], raw_empty[SR];
  __shared__ __align__(8) uint64_t act_full[SA], act_empty[SA];
  __shared__ __align__(8) uint64_t op_full[SO], op_empty[SO];
  __shared__ __align__(8) uint64_t acc_full[NACC], acc_empty[NACC];
  __shared__ __align__(8) uint64_t scl_full[NSCL];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int splits = p.splits;
  const int tile = blockIdx.x / splits;
  const int rank = blockIdx.x - tile * splits;      // == %cluster_ctarank
  const int n0 = tile * BM;
  const int st_begin = (rank * p.stages) / splits;
  const int st_end = ((rank + 1) * p.stages) / splits;
  const int g_begin = st_begin * GPR;
  const int ng = (st_end - st_begin) * GPR;          // groups of this CTA
  const int nst = st_end - st_begin;                 // raw stages of this CTA
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SR; ++i) { mbar_init(smem_u32(&raw_full[i]), 1); mbar_init(smem_u32(&raw_empty[i]), kConvWarps); }
    for (int i = 0; i < SA; ++i) { mbar_init(smem_u32(&act_full[i]), 1); mbar_init(smem_u32(&act_empty[i]), 1); }
    for (int i = 0; i < SO; ++i) { mbar_init(smem_u32(&op_full[i]), kConvWarps); mbar_init(smem_u32(&op_empty[i]), 1); }
    for (int i = 0; i < NACC; ++i) { mbar_init(smem_u32(&acc_full[i]), 1); mbar_init(smem_u32(&acc_empty[i]), 4); }
    for (int i = 0; i < NSCL; ++i) mbar_init(smem_u32(&scl_full[i]), 4);
    abort_sh = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem = tmem_base_sh;

  float acc[BN];
#pragma unroll
  for (int m = 0; m < BN; ++m) acc[m] = 0.0f;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA
    // Lane 0 streams raw weight stages, lane 1 streams activation tiles, so
    // neither ring waits on the other.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int raw_issued = 0;
      for (int t = 0; t < nst; ++t) {
        const int sr = t % SR;
        if (t >= SR && !wait_or_abort(smem_u32(&raw_empty[sr]), ((t / SR) - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(smem_u32(&raw_full[sr]), F::kRawBytes);
        F::issue_raw(&tmW, sbase + L::kRawOff + sr * F::kRawBytes, g_begin + t * GPR, n0,
                     smem_u32(&raw_full[sr]), pol);
        raw_issued = t + 1;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      for (int t = max(0, raw_issued - SR); t < raw_issued; ++t)
        mbar_wait(smem_u32(&raw_full[t % SR]), (t / SR) & 1, p.err);
    } else if (lane == 1) {
      pdl_wait();                          // activations may come from the previous kernel
      int act_issued = 0;
      for (int j = 0; j < ng; ++j) {
        const int sa = j % SA;
        if (j >= SA && !wait_or_abort(smem_u32(&act_empty[sa]), ((j / SA) - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(smem_u32(&act_full[sa]), kActBytes);
        const uint32_t dst = sbase + L::kActOff + sa * kActBytes;
        tma_load_2d(dst, &tmA, (g_begin + j) * GK, 0, smem_u32(&act_full[sa]));
        tma_load_2d(dst + kActBytes / 2, &tmA, (g_begin + j) * GK + 64, 0, smem_u32(&act_full[sa]));
        act_issued = j + 1;
      }
      for (int j = max(0, act_issued - SA); j < act_issued; ++j)
        mbar_wait(smem_u32(&act_full[j % SA]), (j / SA) & 1, p.err);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      int issued = 0;
      for (int j = 0; j < ng; ++j) {
        const int so = j % SO, sa = j % SA, sc = j % NACC;
        if (!wait_or_abort(smem_u32(&op_full[so]), (j / SO) & 1, p.err, abort_flag)) break;
        if (!wait_or_abort(smem_u32(&act_full[sa]), (j / SA) & 1, p.err, abort_flag)) break;
        if (j >= NACC && !wait_or_abort(smem_u32(&acc_empty[sc]), ((j / NACC) - 1) & 1, p.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t opb = sbase + L::kOpOff + so * kOpBytes;
        const uint32_t actb = sbase + L::kActOff + sa * kActBytes;
#pragma unroll
        for (int i = 0; i < GK / 16; ++i) {
          // Weights: 128-byte swizzled K-major blocks of 64 K (see op_chunk);
          // 32 B per 16-K step; SBO = 1024 B (8-row atoms).
          const uint64_t ad = sdesc(opb + (i >> 2) * (BM * 128) + (i & 3) * 32, 16, 1024, 2);
          // Activations: 128-byte swizzled rows of 64 K; 32 B per 16-K step,
          // the second 64 K in the second box; SBO = 1024 B (8-row atoms).
          const uint64_t bd = sdesc(actb + (i >> 2) * (kActBytes / 2) + (i & 3) * 32, 16, 1024, 2);
          mma_bf16(tmem + sc * 16, ad, bd, idesc, i > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&op_empty[so]));
        mma_commit(smem_u32(&act_empty[sa]));
        mma_commit(smem_u32(&acc_full[sc]));
        issued = j + 1;
      }
      // Drain: all MMAs done before TMEM is freed.
      if (issued > 0) {
        const int j = issued - 1;
        mbar_wait(smem_u32(&acc_full[j % NACC]), (j / NACC) & 1, p.err);
      }
    }
  } else if (warp < kConvWarps) {
    // ------------------------------------------------------------ convert
    const int q = warp & 3;                 // row block
    const int kq = warp >> 2;               // which 32-K quarter of a group
    const int r = q * 32 + lane;            // row within the tile
    float* scl = reinterpret_cast<float*>(smem + L::kSclOff);     // [NSCL][BM] row scales
    for (int j = 0; j < ng; ++j) {
      const int t = j / GPR, gi = j % GPR;
      const int sr = t % SR, so = j % SO;
      const bool g1 = (gi != 0) || wait_or_abort(smem_u32(&raw_full[sr]), (t / SR) & 1, p.err, abort_flag);
      const bool g2 = g1 && (j < SO || wait_or_abort(smem_u32(&op_empty[so]), ((j / SO) - 1) & 1, p.err, abort_flag));
      if (!__all_sync(0xFFFFFFFFu, g1 && g2)) break;
      float d = 0.0f;
      F::convert(smem + L::kRawOff + sr * F::kRawBytes, gi, r, kq, smem + L::kOpOff + so * kOpBytes, d);
      // Slot j % NSCL is free: its previous group was folded before this
      // group's operand stage could be released (pipeline depth SO + NACC).
      if (F::kRowScale && kq == 0) scl[(j % NSCL) * BM + r] = d;
      fence_proxy_async_smem();
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&op_full[so]));
        if (gi == GPR - 1) mbar_arrive(smem_u32(&raw_empty[sr]));
        if (F::kRowScale && kq == 0) mbar_arrive(smem_u32(&scl_full[j % NSCL]));
      }
    }
  } else if (warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------------ fold
    const int q = warp & 3;                 // TMEM lane quarter
    const int r = q * 32 + lane;
    const float* scl = reinterpret_cast<const float*>(smem + L::kSclOff);
    const float* srow = F::kRowScale ? nullptr : p.scales + static_cast<size_t>(tile) * (p.K / GK);
    for (int j = 0; j < ng; ++j) {
      const int sc = j % NACC;
      // Warp-uniform outcome: tcgen05.ld below is .sync.aligned.
      const bool got = wait_or_abort(smem_u32(&acc_full[sc]), (j / NACC) & 1, p.err, abort_flag);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      float v[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + sc * 16, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[sc]));
      float s;
      if (F::kRowScale) {
        const bool gs = wait_or_abort(smem_u32(&scl_full[j % NSCL]), (j / NSCL) & 1, p.err, abort_flag);
        if (!__all_sync(0xFFFFFFFFu, gs)) break;
        s = scl[(j % NSCL) * BM + r];
      } else {
        s = __ldg(srow + g_begin + j);
      }
#pragma unroll
      for (int m = 0; m < BN; ++m) acc[m] = fmaf(v[m], s, acc[m]);
    }
  }

  // ---------------------------------------------------------- reduce + store
  __syncthreads();
  const bool failed = *abort_flag != 0;
  float* red = reinterpret_cast<float*>(smem + L::kRawOff);   // raw ring is idle now
  if (splits > 1) {
    const bool epi = warp >= kEpiWarp0 && warp < kEpiWarp0 + 4;
    const int er = (warp - kEpiWarp0) * 32 + lane;
    if (epi && rank != 0) {
      float4* dst = reinterpret_cast<float4*>(red + er * BN);
#pragma unroll
      for (int i = 0; i < BN / 4; ++i) dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
    }
    cluster_sync();
    if (epi && rank == 0) {
      const uint32_t mine = smem_u32(red + er * BN);
      for (int qq = 1; qq < splits; ++qq) {
        const uint32_t rem = mapa_shared(mine, qq);
#pragma unroll
        for (int i = 0; i < BN / 4; ++i) {
          const float4 v = ld_dsmem_f4(rem + 16 * i);
          acc[4 * i] += v.x;
          acc[4 * i + 1] += v.y;
          acc[4 * i + 2] += v.z;
          acc[4 * i + 3] += v.w;
        }
      }
    }
    cluster_sync();                       // remote partials stay alive until read
  }
  if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4 && rank == 0 && !failed) {
    const int n = n0 + (warp - kEpiWarp0) * 32 + lane;
    if (n < p.N) {
#pragma unroll
      for (int m = 0; m < BN; ++m)
        if (m < p.M) p.C[static_cast<size_t>(m) * p.ldc + n] = f32_to_bf16_rn(acc[m]);
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
int choose_splits(int tiles, int stages, int num_sms) {
  int s = num_sms / tiles;                   // one CTA per SM, a single wave
  if (s < 1) s = 1;
  if (s > 8) s = 8;                          // portable cluster size
  if (s > stages) s = stages;
  return s;
}

template <class F>
cudaError_t launch_tc(const GemvArgs& a, const CUtensorMap& mw, cudaStream_t s) {
  using L = Layout<F>;
  CUtensorMap ma;
  cudaError_t e = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.A, static_cast<uint64_t>(a.K),
                              static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.lda) * 2, 64, BN,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(tc_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int tiles = (a.N + BM - 1) / BM;
  TcParams p;
  p.scales = static_cast<const float*>(a.scales);
  p.C = static_cast<uint16_t*>(a.C);
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.ldc = a.ldc;
  p.stages = a.K / (GK * F::kGPR);
  p.splits = choose_splits(tiles, p.stages, a.num_sms);
  p.err = a.err;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * p.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
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
  return cudaLaunchKernelEx(&cfg, tc_kernel<F>, mw, ma, p);
}

}  // namespace tc

cudaError_t launch_w8a16_gemm_tc(const GemvArgs& a, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mw;
  cudaError_t e = make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, static_cast<uint64_t>(a.K),
                              static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K), GK, BM,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return launch_tc<Fp8Tc>(a, mw, s);
}

// Requires K % 1024 == 0 (checked by the caller): a row is then 34 * K / 128
// bytes, a multiple of 16, and each raw stage of 8 groups starts on a
// 16-byte boundary.
cudaError_t launch_q2_gemm_tc(const GemvArgs& a, cudaStream_t s) {
  using namespace tc;
  const uint64_t G = static_cast<uint64_t>(a.K / GK);
  CUtensorMap mw;
  cudaError_t e = make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.W, 17 * G, static_cast<uint64_t>(a.N),
                              34 * G, 8 * 17, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return launch_tc<Q2Tc>(a, mw, s);
}

}  // namespace wqp
