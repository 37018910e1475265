// Tensor-core (tcgen05) swap-AB decode GEMM for packed weights, 1 <= M <= 16.
//
// W4 (E2M1 codes, E4M3 scale per 16 K, FP32 per-tensor scale;
// "spark_model/layers/w4a16_gemv_tiers.rs", module docs),
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
//   D[n, m] = sum_k W[n, k] * A[m, k]   (tcgen05.mma kind::f16, BF16 in, FP32
//                                        accumulate, M=128 N=16 K=16)
// The weight operand lives in tensor memory: converter warps decode the packed
// bytes in registers and write BF16 pairs with tcgen05.st (one weight row per
// TMEM lane, two K elements per 32-bit column); the MMA reads A from TMEM and
// the activation operand B from shared memory. No operand round-trips through
// shared memory.
//
// Encodings (every product is exact in FP32):
//  * FP8: each E4M3 value is a BF16 value; B is the activation tile as loaded.
//  * W4: e2m1 * e4m3 scale has at most 6 significant bits and lies in
//    [2^-10, 2688], so it is exact in FP16 and in BF16; the per-tensor scale
//    multiplies the FP32 result once, at the store. B is the activation tile
//    as loaded.
//  * Q2_0: the two codes (c_j, c_{j+8}) of a 16-code word sit at bits (2j,
//    2j+16). Masking them in place (one LOP3 per pair) gives two BF16
//    subnormals c * 4^(j mod 4) * 2^-133 (exact: the field stays below the
//    first normal binade, where the BF16 encoding is linear). The matching
//    activations are pre-scaled by 2^(64 - 2 (j mod 4)) (exact), so each
//    product is c * a * 2^-69. Per 128-K group g and activation row m,
//    sum_k (c_k - 1) a_k = 2^69 * D[n, m] - S[m, g] with S = sum_k a_k, and the
//    fp16 scale d folds in FP32: acc += d * (2^69 D - S).
//    The MMA's K order inside a 16-K step is the code-pair order
//    (16i + c', 16i + c' + 8) for column c' = 0..7; the activation operand is
//    written in that same order.
// The tensor core reduces each 16-K step in its own order, so results are not
// bit-identical to the scalar kernels; each output element still depends only
// on its own weight row and activation row.
//
// One CTA = one tile of weight rows x a contiguous range of 128-K groups (a
// multiple of the raw stage). Two CTAs share an SM (16 warps, 256 TMEM
// columns and under half the shared memory each). Warps:
//   0..7   converters, in two sets (set h takes the groups h mod 2 of a raw
//          stage, or every other stage when a stage holds one group); TMEM
//          lane quarter = warp % 4; each thread converts one weight row of
//          one group (64 columns) into one of SO operand slots;
//   8..11  epilogue: per group, tcgen05.ld of the group's accumulator slot
//          (lane = weight row, column = activation row) and the FP32 fold;
//   12     TMA of the raw weight stages (lane 0);
//   13     MMA (allocates TMEM): per group one wait, then the elected lane
//          issues the 8 MMAs into the group's accumulator slot and commits
//          once ("MMA of group j done");
//   14..15 Q2_0: activation operand, read from global memory and written
//          permuted and pre-scaled into the MMA's activation slot;
//   15     FP8, W4: TMA of the activation tiles (lane 0), used as loaded.
// The MMA warp waits on one barrier per group, "group j may start", which
// completes after the four converter warps of the set, the four epilogue
// warps releasing the accumulator slot (pre-armed for the first NACC groups)
// and, for Q2_0, the operand warp; for FP8 and W4 it then waits for the
// activation tile's copy itself.
// Q2_0 tiles are 124 weight rows: the last lane of each 32-lane quarter of
// TMEM (lanes 31, 63, 95, 127) holds a row of all-ones codes, whose
// accumulator is 2^-69 * sum_k a_k, the group sum the fold needs, computed by
// the same MMAs and read by each epilogue warp from its own lane 31.
// When N is small, K is split over a thread-block cluster of up to 8 CTAs;
// each rank owns a slice of the tile's rows, the others push their partial
// sums into its shared memory, and it adds them in rank order
// (deterministic, no global scratch).
#include <atomic>

#include "decode.cuh"
#include "tc.cuh"

namespace wqp {
namespace tc {

constexpr int BM = 128;            // TMEM lanes = MMA M
constexpr int BN = 16;             // activation rows (MMA N)
constexpr int GK = 128;            // K per group = scale granularity
// Two CTAs share an SM (each 16 warps x 64 registers, 256 TMEM columns and
// under half the shared memory), so one CTA's latency chain overlaps
// another's: the split-K ranks of a small call, or the next call's CTAs,
// which start loading and converting their weights under programmatic
// dependent launch while this call finishes.
constexpr int kCtasPerSm = 2;
constexpr int kConvSets = 2;       // converter warps 0..7
constexpr int kEpiWarp0 = 8;       // epilogue warps 8..11
constexpr int kEpiSets = 1;
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;       // MMA warp; allocates TMEM
constexpr int kMmaWarps = 1;
constexpr int kMmaBatch = 1;       // groups issued per wait of the MMA warp
constexpr int kPrepWarp0 = 14;     // Q2_0: activation operand warps 14..15
constexpr int kPrepWarps = 2;
constexpr int kActWarp = 15;       // FP8, W4: activation TMA (its own warp: divergent lanes of
                                   // one warp that wait on different barriers delay each other)
constexpr int kThreads = 16 * 32;
constexpr int SO = 3;              // TMEM operand stages, one group (64 columns) each
constexpr int NACC = 4;            // TMEM accumulator slots, 16 columns each
constexpr uint32_t kAccCol = SO * 64;
constexpr uint32_t kTmemCols = 256;
static_assert(kAccCol + NACC * 16 <= kTmemCols, "TMEM budget");
static_assert(kCtasPerSm * kTmemCols <= 512, "TMEM columns of the co-resident CTAs");
static_assert(kCtasPerSm * kThreads * 64 <= 65536, "registers of the co-resident CTAs at 64 per thread");
constexpr int SB = 6;              // activation operand stages
constexpr int ND = 16;             // "MMA of group j done" and "group j may start" rings
// "Group j may start": the converter warps, the epilogue warps releasing the
// accumulator slot and, for Q2_0, the operand hand-off warp. FP8 and W4 tiles
// are used as loaded: the MMA warp waits for the tile's copy itself.
template <class F>
__host__ __device__ constexpr int go_count() { return 4 + 4 + (F::kQ2 ? 1 : 0); }
constexpr int NSC = 8;             // per-group row-scale ring (converters -> epilogue)

// Ring depth: a scale slot of group j is rewritten after the MMA of group
// j - SO completed; that MMA was issued after the epilogue released group
// j - SO - NACC and had read its scale. A waiter on "MMA of
// group g done" never lags the MMA by ND groups (the MMA cannot pass the
// epilogue by more than NACC; every other waiter runs ahead of it), so the
// parities never alias.
static_assert(NSC >= SO + NACC, "scale ring must outlive the pipeline");
static_assert(ND >= SB && ND >= SO && ND > NACC, "done ring depth");
static_assert(kMmaBatch <= NACC && kMmaBatch <= SO, "the MMA warp waits for a batch of groups at once");
// "Group j may start" slot j % ND receives arrivals for group j only after the
// MMA of group j - ND was issued: converters wait for MMA j - SO, the operand
// producer for MMA j - SB, the epilogue arrives after MMA j - NACC completed.
// Activation slot: two [16 rows x 64 K] boxes (2 KB apart), 128-byte swizzle.
// The TMA fills rows 0 .. NB-1 of each box (NB = M rounded up to a power of
// two, rows >= M zero-filled); rows NB..15 are never loaded and only reach
// accumulator columns >= NB, which nothing reads.
constexpr int kBBytes = BN * GK * 2;
// Split-K partial sums pushed to the owning rank: [splits][NB][rows per rank],
// at most 16 x (8 x 16 + 8) floats.
constexpr int kRecvBytes = BN * (BM + 8) * 4;

struct TcParams {
  const uint16_t* A;       // bf16 [M, lda] (Q2_0 operand warps read it directly)
  int lda;
  const float* scales;     // FP8: [ceil(N/128), K/128]; Q2_0, W4: unused here
  float gscale;            // W4 per-tensor scale (1 otherwise)
  uint16_t* C;
  int M, N, K, ldc;
  int splits;              // CTAs per tile (cluster size)
  int stages;              // raw stages per tile
  unsigned* err;
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------ formats
// FP8 E4M3: one group per raw stage, [128 rows x 128 B], 128-byte swizzle
// (16-byte chunk c of row r at chunk c ^ (r % 8)).
struct Fp8Tc {
  static constexpr int kRows = 128;              // weight rows per tile
  static constexpr int kGPR = 1;
  static constexpr int kSR = 4;
  static constexpr int kRawBytes = BM * GK;      // stage stride
  static constexpr int kBoxBytes = kRows * GK;   // bytes one stage load delivers
  static constexpr bool kQ2 = false;
  static constexpr bool kBlockScale = true;      // fold s[n/128, g] per group
  __device__ static void issue_raw(const CUtensorMap* m, const CUtensorMap*, uint32_t dst, int g0, int n0,
                                   uint32_t bar, uint64_t pol) {
    tma_load_2d_hint(dst, m, g0 * GK, n0, bar, pol);
  }
  // TMEM lane r = weight row r of the tile.
  __device__ static int raw_row(int r) { return r; }
  // Row r of the stage's group -> 64 TMEM columns from tcol: chunk c (K 16c..16c+15)
  // is MMA step c, natural pairs (16c + 2i, 16c + 2i + 1) in columns 8c + i.
  __device__ static void convert(const uint8_t* raw, int r, int /*gi*/, uint32_t tcol, float& d) {
    const uint8_t* row = raw + r * 128;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t v[16];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c = 2 * h + c2;
        const uint4 x = lds128(row + ((c ^ (r & 7)) << 4));
        e4m3x4_to_bf16(x.x, v[8 * c2 + 0], v[8 * c2 + 1]);
        e4m3x4_to_bf16(x.y, v[8 * c2 + 2], v[8 * c2 + 3]);
        e4m3x4_to_bf16(x.z, v[8 * c2 + 4], v[8 * c2 + 5]);
        e4m3x4_to_bf16(x.w, v[8 * c2 + 6], v[8 * c2 + 7]);
      }
      tmem_st16(tcol + 16 * h, v);
    }
    d = 1.0f;
  }
};

// Q2_0: eight groups per raw stage, [124 rows x 8 blocks x 34 B], no swizzle.
// A row is 272 B = 68 words (68 = 4 mod 32), so 16-byte loads of 31
// consecutive rows at the same offset are free of bank conflicts.
struct Q2Tc {
  static constexpr int kRows = 124;              // + an all-ones row per lane quarter
  static constexpr int kGPR = 8;
  static constexpr int kSR = 2;
  static constexpr int kRawBytes = BM * 8 * 34;  // stage stride
  // TMEM lane r = 32 q + l holds weight row 31 q + l for l < 31; lane 31 of
  // each quarter is the all-ones row.
  __device__ static int raw_row(int r) { return (r >> 5) * 31 + (r & 31); }
  static constexpr int kBoxBytes = kRows * 8 * 34;
  static constexpr bool kQ2 = true;
  static constexpr bool kBlockScale = false;
  __device__ static void issue_raw(const CUtensorMap* m, const CUtensorMap*, uint32_t dst, int g0, int n0,
                                   uint32_t bar, uint64_t pol) {
    tma_load_2d_hint(dst, m, g0 * 17, n0, bar, pol);              // 17 u16 per block
  }
  // Block gi of row r: its 34 bytes start off = 34 gi mod 16 bytes into a
  // 48-byte window of three aligned 16-byte chunks (one code path for every
  // gi: the window's words are realigned with selects and a funnel shift).
  // Word i of the block (codes 16i..16i+15) is MMA step i: columns 8i + j
  // (j < 4) hold the pair (c_j, c_{j+8}) of the word, columns 8i + 4 + j the
  // pair (c_{j+4}, c_{j+12}), both scaled by 4^j. The last lane of each
  // quarter writes codes 1 everywhere (it reads the quarter's first row and
  // discards it).
  __device__ static void convert(const uint8_t* raw, int r, int gi, uint32_t tcol, float& d) {
    const int b0 = 34 * gi;
    const int base = b0 & ~15;
    const int off = b0 - base;                     // 0, 2, ..., 14
    const int k0 = off >> 2;                       // first window word of the block
    const uint32_t sh = static_cast<uint32_t>(off & 3) * 8;   // 0 or 16
    const bool ones = (r & 31) == 31;
    const uint8_t* row = raw + raw_row(ones ? (r & ~31) : r) * 272 + base;
    const uint4 c0 = lds128(row), c1 = lds128(row + 16), c2 = lds128(row + 32);
    const uint32_t wv[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
    uint32_t a[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint32_t lo = (k0 & 1) ? wv[i + 1] : wv[i];
      const uint32_t hi = (k0 & 1) ? wv[i + 3] : wv[i + 2];
      a[i] = (k0 & 2) ? hi : lo;
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t v[16];
#pragma unroll
      for (int w2 = 0; w2 < 2; ++w2) {
        const int idx = 2 * h + w2;
        uint32_t q = __funnelshift_r(a[idx], a[idx + 1], sh);
        q = ones ? 0x55555555u : q;
        const uint32_t q8 = q >> 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * w2 + j] = q & (0x00030003u << (2 * j));
          v[8 * w2 + 4 + j] = q8 & (0x00030003u << (2 * j));
        }
      }
      tmem_st16(tcol + 16 * h, v);
    }
    const uint32_t dbits = (a[8] >> sh) & 0xFFFFu;
    d = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
  }
};

// W4: two groups per raw stage: codes [128 rows x 128 B] with the 128-byte
// swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)), then the E4M3
// scales [128 rows x 16 B]. Group gi of the stage is code chunks 4 gi .. 4 gi + 3
// and scale bytes 8 gi .. 8 gi + 7 of the row.
struct W4Tc {
  static constexpr int kRows = 128;
  static constexpr int kGPR = 2;
  static constexpr int kSR = 4;
  static constexpr int kCodeBytes = BM * 128;
  static constexpr int kRawBytes = kCodeBytes + BM * 16;   // stage stride (1024-multiple)
  static constexpr int kBoxBytes = kRawBytes;
  static constexpr bool kQ2 = false;
  static constexpr bool kBlockScale = false;
  static_assert(kRawBytes % 1024 == 0, "raw stages keep the swizzle atoms aligned");
  __device__ static void issue_raw(const CUtensorMap* m, const CUtensorMap* m2, uint32_t dst, int g0,
                                   int n0, uint32_t bar, uint64_t pol) {
    tma_load_2d_hint(dst, m, g0 * (GK / 2), n0, bar, pol);                // code bytes
    tma_load_2d_hint(dst + kCodeBytes, m2, g0 * (GK / 16), n0, bar, pol); // scale bytes
  }
  __device__ static int raw_row(int r) { return r; }
  // Row r, group gi of the stage -> 64 TMEM columns from tcol: 16-K step i is
  // code bytes 8i..8i+7 of the group and scale byte i; natural pairs
  // (16i + 2b, 16i + 2b + 1) = byte b in column 8i + b.
  __device__ static void convert(const uint8_t* raw, int r, int gi, uint32_t tcol, float& d) {
    const uint8_t* row = raw + r * 128;
    const uint2 sc = *reinterpret_cast<const uint2*>(raw + kCodeBytes + r * 16 + gi * 8);
#pragma unroll
    for (int h = 0; h < 4; ++h) {                              // one code chunk = steps 2h, 2h+1
      const int c = 4 * gi + h;
      const uint4 x = lds128(row + ((c ^ (r & 7)) << 4));
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
      uint32_t v[16];
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const int step = 2 * h + st;
        const uint32_t sbyte = ((step < 4 ? sc.x : sc.y) >> (8 * (step & 3))) & 0xFFu;
        const uint32_t s16 = e4m3x2_to_f16x2(sbyte) & 0xFFFFu;
        const uint32_t s2 = s16 | (s16 << 16);                 // {s, s} as f16x2
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t word = xs[2 * st + w];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t hp = e2m1x2_to_f16x2((word >> (8 * b)) & 0xFFu);
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hp) : "r"(hp), "r"(s2));
            v[8 * st + 4 * w + b] = f16x2_to_bf16x2_exact(hp);
          }
        }
      }
      tmem_st16(tcol + 16 * h, v);
    }
    d = 1.0f;
  }
};

template <class F>
struct Layout {
  static constexpr int kRawOff = 0;
  static constexpr int kBOff = (kRawOff + F::kSR * F::kRawBytes + 1023) / 1024 * 1024;
  static constexpr int kSclOff = kBOff + SB * kBBytes;
  static constexpr int kRecvOff = kSclOff + (F::kQ2 ? NSC * BM * 4 : 0);
  static constexpr int kBytes = kRecvOff + kRecvBytes;
  static constexpr int kAlloc = kBytes + 1024;                     // slack for 1024-byte alignment
  static_assert(kEpiSets * BM * BN * 4 <= F::kSR * F::kRawBytes, "split-K partials alias the raw ring");
  // Per SM: 228 KB of shared memory, 1 KB of it reserved per CTA, plus the
  // kernel's static shared memory (< 1 KB).
  static_assert(kCtasPerSm * (kAlloc + 2048) <= 228 * 1024, "shared memory budget of the co-resident CTAs");
};

// All mbarriers of a CTA live in one shared array; Bar<F>::X is the index of
// the first barrier of ring X, and bar(base, i) its shared-memory address.
template <class F>
struct Bar {
  static constexpr int kRawFull = 0;                  // [SR]  raw stage landed
  static constexpr int kRawEmpty = kRawFull + F::kSR; // [SR]  raw stage converted
  static constexpr int kBLoad = kRawEmpty + F::kSR;   // [SB]  activation tile landed (Q2_0)
  static constexpr int kGo = kBLoad + SB;             // [ND]  group j may start (go_count)
  static constexpr int kDone = kGo + ND;              // [ND]  MMA of group j complete
  static constexpr int kSclFull = kDone + ND;         // [NSC] row scales written
  static constexpr int kCount = kSclFull + NSC;
};
__device__ __forceinline__ uint32_t bar(uint32_t base, int i) { return base + 8u * static_cast<uint32_t>(i); }

// Convert group gi of raw stage t for this thread's row. False on abort.
template <class F>
__device__ __forceinline__ bool convert_group(const uint8_t* raw, int t, int gi, int q, int r, int lane,
                                              uint32_t tmem, uint32_t bars, float* scl, unsigned* err,
                                              volatile int* abort_flag) {
  using B = Bar<F>;
  const int j = t * F::kGPR + gi;
  const int so = j % SO;
  if (j >= SO) {
    const int g = j - SO;                            // previous user of the stage
    const bool ok = wait_or_abort(bar(bars, B::kDone + g % ND), (g / ND) & 1, err, abort_flag);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
  }
  tc_fence_after();
  float d;
  F::convert(raw, r, gi, tmem + (static_cast<uint32_t>(q * 32) << 16) + so * 64, d);
  tmem_wait_st();
  if (F::kQ2) scl[(j % NSC) * BM + r] = d;
  tc_fence_before();
  __syncwarp();                                      // the arrive below releases the whole warp's work
  if (lane == 0) {
    mbar_arrive(bar(bars, B::kGo + j % ND));
    if (F::kQ2) mbar_arrive(bar(bars, B::kSclFull + j % NSC));
  }
  return true;
}

template <class F, int NB>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
              const __grid_constant__ CUtensorMap tmA, TcParams p) {
  using L = Layout<F>;
  constexpr int SR = F::kSR;
  constexpr int GPR = F::kGPR;
  extern __shared__ uint8_t smem_raw[];
  using B = Bar<F>;
  __shared__ __align__(8) uint64_t bar_sh[B::kCount];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int splits = p.splits;
  const int tile = blockIdx.x / splits;
  const int rank = blockIdx.x - tile * splits;      // == %cluster_ctarank
  const int n0 = tile * F::kRows;
  const int st_begin = (rank * p.stages) / splits;
  const int st_end = ((rank + 1) * p.stages) / splits;
  const int g_begin = st_begin * GPR;
  const int nst = st_end - st_begin;                 // raw stages of this CTA
  const int ng = nst * GPR;                          // groups of this CTA
  volatile int* abort_flag = &abort_sh;
  const uint32_t bars = smem_u32(bar_sh);

  if (threadIdx.x == 0) {
    for (int i = 0; i < B::kCount; ++i) {
      uint32_t count = 1;
      // Converter warps that release a raw stage: the sets owning its groups.
      if (i >= B::kRawEmpty && i < B::kBLoad) count = 4 * (GPR < kConvSets ? GPR : kConvSets);
      if (i >= B::kGo && i < B::kDone) count = go_count<F>();
      if (i >= B::kSclFull) count = 4;
      mbar_init(bar(bars, i), count);
    }
    // The accumulator slots start free: the epilogue's four releases for
    // groups 0 .. NACC-1.
    for (int i = 0; i < NACC; ++i)
      for (int k = 0; k < 4; ++k) mbar_arrive(bar(bars, B::kGo + i));
    abort_sh = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  int raw_issued = 0, act_issued = 0;     // copies issued by lane 0 of the TMA / activation warp
  // Producer warps: the raw-weight TMA and, for FP8 and W4, the activation TMA.
  constexpr int kProducers = F::kQ2 ? 1 : 2;
  const bool producer = warp == kTmaWarp || (!F::kQ2 && warp == kActWarp);
  if (producer) {
    // ------------------------------------------------------------ TMA
    // Lane 0 of the TMA warp streams raw weight stages (independent of the
    // previous grid, so they start before griddepcontrol.wait); lane 0 of the
    // activation warp streams activation tiles.
    if (warp == kTmaWarp && lane == 0) {
      prefetch_tmap(&tmW);
      if (F::kGPR == 2) prefetch_tmap(&tmW2);
      const uint64_t pol = policy_evict_first();
      for (int t = 0; t < nst; ++t) {
        const int sr = t % SR;
        if (t >= SR && !wait_or_abort(bar(bars, B::kRawEmpty + sr), ((t / SR) - 1) & 1, p.err, abort_flag)) break;
        mbar_arrive_expect_tx(bar(bars, B::kRawFull + sr), F::kBoxBytes);
        F::issue_raw(&tmW, &tmW2, sbase + L::kRawOff + sr * F::kRawBytes, g_begin + t * GPR, n0,
                     bar(bars, B::kRawFull + sr), pol);
        raw_issued = t + 1;
      }
    } else if (!F::kQ2 && warp == kActWarp && lane == 0) {
      // Activation tiles [NB rows x 128 K] (rows >= M zero-filled) into the
      // operand ring; Q2_0 tiles are rewritten in place by the preparation
      // warps before the MMA reads them.
      prefetch_tmap(&tmA);
      pdl_wait();                          // activations may come from the previous grid
      for (int j = 0; j < ng; ++j) {
        const int s = j % SB;
        const int full = B::kBLoad + s;
        if (j >= SB) {
          const int g = j - SB;            // previous user of the stage
          if (!wait_or_abort(bar(bars, B::kDone + g % ND), (g / ND) & 1, p.err, abort_flag)) break;
        }
        mbar_arrive_expect_tx(bar(bars, full), NB * GK * 2);
        const uint32_t dst = sbase + L::kBOff + s * kBBytes;
        tma_load_2d(dst, &tmA, (g_begin + j) * GK, 0, bar(bars, full));
        tma_load_2d(dst + kBBytes / 2, &tmA, (g_begin + j) * GK + 64, 0, bar(bars, full));
        act_issued = j + 1;
      }
    }
    __syncwarp();                          // the CTA barriers below need a converged warp
  } else {
    // Everyone else needs the TMEM base address.
    if (warp == kMmaWarp) {
      tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
      tmem_relinquish();
      tc_fence_before();
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 32 * kProducers) : "memory");
    tc_fence_after();
  }
  const uint32_t tmem = producer ? 0u : tmem_base_sh;
  // Partial sums [kEpiSets][NB][BM] for the final reduction alias the raw
  // ring: an epilogue set writes them only after the MMAs of the last two
  // groups (one per MMA warp) completed, so every raw stage has been consumed
  // by then.
  float* red = reinterpret_cast<float*>(smem + L::kRawOff);

  if (warp >= kMmaWarp && warp < kMmaWarp + kMmaWarps) {
    // ------------------------------------------------------------ MMA
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    const uint32_t b_base = sbase + L::kBOff;
    int issued = -1;
    // A wait costs the MMA warp a fixed stall (it resumes only once the
    // tensor core has taken its earlier MMAs), so it waits for kMmaBatch
    // groups at a time. Nothing a later group needs depends on an earlier
    // group's MMA, so waiting ahead cannot deadlock.
    for (int j0 = (warp - kMmaWarp) * kMmaBatch; j0 < ng; j0 += kMmaWarps * kMmaBatch) {
      const int j1 = min(j0 + kMmaBatch, ng);
      bool ok = true;
      for (int j = j0; j < j1 && ok; ++j) {
        ok = wait_or_abort(bar(bars, B::kGo + j % ND), (j / ND) & 1, p.err, abort_flag);
        if (!F::kQ2 && ok) ok = wait_or_abort(bar(bars, B::kBLoad + j % SB), (j / SB) & 1, p.err, abort_flag);
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      if (elect_one()) {
        for (int j = j0; j < j1; ++j) {
          // B: two 128-byte-swizzled boxes of 64 K (2 KB apart), 32 B per
          // 16-K step, SBO = 1024 B (8-row atoms). The start-address field
          // is address >> 4, so a step adds 2 and a box adds 128 (no carry:
          // shared addresses stay below 2^18).
          const uint64_t bd0 = sdesc(b_base + (j % SB) * kBBytes, 16, 1024, 2);
          const uint32_t a0 = tmem + (j % SO) * 64;
          const uint32_t dcol = tmem + kAccCol + (j % NACC) * 16;
#pragma unroll
          for (int i = 0; i < GK / 16; ++i)
            mma_ts(dcol, a0 + 8 * i, bd0 + static_cast<uint64_t>((i >> 2) * 128 + (i & 3) * 2), idesc,
                   i > 0 ? 1u : 0u);
          mma_commit(bar(bars, B::kDone + j % ND));
        }
      }
      __syncwarp();
      issued = j1 - 1;
    }
    // Drain: this warp's MMAs are done before TMEM is freed.
    if (issued >= 0) mbar_wait(bar(bars, B::kDone + issued % ND), (issued / ND) & 1, p.err);
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ convert
    const int q = warp & 3;                 // TMEM lane quarter = 32-row block
    const int h = warp >> 2;                // converter set
    const int r = q * 32 + lane;
    float* scl = reinterpret_cast<float*>(smem + L::kSclOff);
    // Set h converts, in every raw stage it takes, the groups gi = h mod
    // kConvSets when a stage holds at least kConvSets groups; otherwise the
    // group h mod GPR of every (kConvSets / GPR)-th stage.
    constexpr int kGPS = GPR >= kConvSets ? GPR / kConvSets : 1;   // groups per set and stage
    static_assert(GPR % kConvSets == 0 || kConvSets % GPR == 0, "groups of a raw stage per converter set");
    const int t0 = GPR >= kConvSets ? 0 : h / GPR;
    const int dt = GPR >= kConvSets ? 1 : kConvSets / GPR;
    const int g0 = GPR >= kConvSets ? h : h % GPR;
    for (int t = t0; t < nst; t += dt) {
      const int sr = t % SR;
      const bool got = wait_or_abort(bar(bars, B::kRawFull + sr), (t / SR) & 1, p.err, abort_flag);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      const uint8_t* raw = smem + L::kRawOff + sr * F::kRawBytes;
      bool live = true;
      for (int k = 0; k < kGPS && live; ++k)
        live = convert_group<F>(raw, t, g0 + k * kConvSets, q, r, lane, tmem, bars, scl, p.err, abort_flag);
      if (!live) break;
      if (lane == 0) mbar_arrive(bar(bars, B::kRawEmpty + sr));
    }
  } else if (warp < kEpiWarp0 + 4 * kEpiSets) {
    // ------------------------------------------------------------ fold
    const int q = warp & 3;
    const int es = (warp - kEpiWarp0) >> 2;      // this set folds groups j = es mod 2
    const int r = q * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16) + kAccCol;
    const float* scl = reinterpret_cast<const float*>(smem + L::kSclOff);
    const float* srow = F::kBlockScale ? p.scales + static_cast<size_t>(tile) * (p.K / GK) : nullptr;
    float acc[NB];
#pragma unroll
    for (int m = 0; m < NB; ++m) acc[m] = 0.0f;
    bool live = true;
    for (int j = es; j < ng && live; j += kEpiSets) {
      const int sc = j % NACC, nsc = j % NSC;
      bool got = wait_or_abort(bar(bars, B::kDone + j % ND), (j / ND) & 1, p.err, abort_flag);
      if (F::kQ2) got = got && wait_or_abort(bar(bars, B::kSclFull + nsc), (j / NSC) & 1, p.err, abort_flag);
      // Warp-uniform outcome: tcgen05.ld below is .sync.aligned.
      if (!__all_sync(0xFFFFFFFFu, got)) { live = false; break; }
      tc_fence_after();
      float v[NB];
      tmem_ld<NB>(tl + sc * 16, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bars, B::kGo + (j + NACC) % ND));   // slot free for j + NACC
      if (F::kQ2) {
        // Lane 31 of the warp (the all-ones row) holds 2^-69 * sum_k a[m, k].
        const float d69 = scl[nsc * BM + r] * 0x1p69f;
#pragma unroll
        for (int m = 0; m < NB; ++m) acc[m] = fmaf(d69, v[m] - __shfl_sync(0xFFFFFFFFu, v[m], 31), acc[m]);
      } else if (F::kBlockScale) {
        const float s = __ldg(srow + g_begin + j);
#pragma unroll
        for (int m = 0; m < NB; ++m) acc[m] = fmaf(v[m], s, acc[m]);
      } else {
#pragma unroll
        for (int m = 0; m < NB; ++m) acc[m] += v[m];
      }
    }
    for (int g = ng - 2; live && g < ng; ++g) {
      if (g < 0) continue;
      live = __all_sync(0xFFFFFFFFu, wait_or_abort(bar(bars, B::kDone + g % ND), (g / ND) & 1, p.err, abort_flag));
    }
    if (live) {
#pragma unroll
      for (int m = 0; m < NB; ++m) red[(es * NB + m) * BM + r] = acc[m];
    }
  } else if (F::kQ2 && warp >= kPrepWarp0 && warp < kPrepWarp0 + kPrepWarps) {
    // ------------------------------------------------------------ Q2_0 activation operand
    // The operand is written straight from global memory into the MMA's
    // activation slot: in row m, the natural chunks k = 16i..16i+7 and
    // 16i+8..16i+15 become the pairs (16i + c', 16i + c' + 8), c' = 0..7,
    // times 2^(64 - 2 (c' mod 4)). One item = (row m, box half, step pair st)
    // = 32 contiguous bytes of A; a warp spreads the items of kTPB tiles over
    // its lanes (rows m >= M are skipped: they only reach accumulator columns
    // nothing reads), loads the next unit while it transforms this one, makes
    // a pass's writes visible to the tensor core once and releases its tiles.
    // Warp w takes the passes w mod 2.
    constexpr int kItems = NB * 8;                        // items per tile
    constexpr int kTPB = kItems >= 32 ? 1 : 32 / kItems;  // tiles per pass
    constexpr int kSub = kItems > 32 ? kItems / 32 : 1;   // units (32 items) per pass
    const int pw = warp - kPrepWarp0;
    const int tb = kItems >= 32 ? 0 : lane / kItems;      // this lane's tile in the pass
    constexpr uint32_t kS0 = 0x5F805F80u, kS1 = 0x5E805E80u, kS2 = 0x5D805D80u, kS3 = 0x5C805C80u;
    pdl_wait();                                           // activations may come from the previous grid
    // Unit u = (pass n, sub-pass sp); loads its 32 bytes into x, y.
    auto load_unit = [&](int n, int sp, uint4& x, uint4& y) {
      const int j = (pw + n * kPrepWarps) * kTPB + tb;
      const int it = kItems >= 32 ? sp * 32 + lane : lane % kItems;
      const int m = it >> 3;
      if (j < ng && m < p.M) {
        const uint16_t* src = p.A + static_cast<size_t>(m) * p.lda + static_cast<size_t>(g_begin + j) * GK +
                              ((it >> 2) & 1) * 64 + (it & 3) * 16;
        x = ld_nc_v4(src);
        y = ld_nc_v4(src + 8);
      }
    };
    uint4 cx = make_uint4(0, 0, 0, 0), cy = cx;
    load_unit(0, 0, cx, cy);
    bool live = true;
    for (int n = 0; live; ++n) {
      const int jb = (pw + n * kPrepWarps) * kTPB;
      if (jb >= ng) break;
      // The pass's slots are free once the MMAs of the tiles SB earlier completed.
      bool ok = true;
      if (lane < kTPB) {
        const int g = jb + lane - SB;
        if (g >= 0 && jb + lane < ng) ok = wait_or_abort(bar(bars, B::kDone + g % ND), (g / ND) & 1, p.err, abort_flag);
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
#pragma unroll
      for (int sp = 0; sp < kSub; ++sp) {
        uint4 nx = make_uint4(0, 0, 0, 0), ny = nx;
        if (sp + 1 < kSub) load_unit(n, sp + 1, nx, ny);
        else load_unit(n + 1, 0, nx, ny);
        const int j = jb + tb;
        const int it = kItems >= 32 ? sp * 32 + lane : lane % kItems;
        const int m = it >> 3, half = (it >> 2) & 1, st = it & 3;
        if (j < ng && m < p.M) {
          uint8_t* rowp = smem + L::kBOff + (j % SB) * kBBytes + half * (kBBytes / 2) + m * 128;
          uint4 o0, o1;
          o0.x = mul_bf16x2(__byte_perm(cx.x, cy.x, 0x5410), kS0);
          o0.y = mul_bf16x2(__byte_perm(cx.x, cy.x, 0x7632), kS1);
          o0.z = mul_bf16x2(__byte_perm(cx.y, cy.y, 0x5410), kS2);
          o0.w = mul_bf16x2(__byte_perm(cx.y, cy.y, 0x7632), kS3);
          o1.x = mul_bf16x2(__byte_perm(cx.z, cy.z, 0x5410), kS0);
          o1.y = mul_bf16x2(__byte_perm(cx.z, cy.z, 0x7632), kS1);
          o1.z = mul_bf16x2(__byte_perm(cx.w, cy.w, 0x5410), kS2);
          o1.w = mul_bf16x2(__byte_perm(cx.w, cy.w, 0x7632), kS3);
          *reinterpret_cast<uint4*>(rowp + (((2 * st) ^ (m & 7)) << 4)) = o0;
          *reinterpret_cast<uint4*>(rowp + (((2 * st + 1) ^ (m & 7)) << 4)) = o1;
        }
        cx = nx;
        cy = ny;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane < kTPB && jb + lane < ng) mbar_arrive(bar(bars, B::kGo + (jb + lane) % ND));
    }
  }

  // ---------------------------------------------------------- reduce + store
  // Rank q of the cluster owns tile rows [q R, q R + R), R = ceil(BM / splits).
  // Every rank adds its two epilogue sets' partials and pushes them into the
  // owner's receive area (slot = source rank); after one cluster barrier each
  // owner adds the slots in rank order and stores its rows. The order of the
  // additions depends only on N and K, never on M.
  __syncthreads();
  if (warp == kMmaWarp) {                 // every tcgen05 access of the CTA has completed
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  const bool failed = *abort_flag != 0;
  if (failed) {
    // Every copy has landed before the CTA may exit. Without an abort the
    // consumers waited for each one already.
    if (warp == kTmaWarp && lane == 0)
      for (int t = max(0, raw_issued - SR); t < raw_issued; ++t)
        mbar_wait(bar(bars, B::kRawFull + t % SR), (t / SR) & 1, p.err);
    if (warp == kActWarp && lane == 0)
      for (int j = max(0, act_issued - SB); j < act_issued; ++j)
        mbar_wait(bar(bars, B::kBLoad + j % SB), (j / SB) & 1, p.err);
  }
  const int rpr = (BM + splits - 1) / splits;
  float* recv = reinterpret_cast<float*>(smem + L::kRecvOff);
  const int et = threadIdx.x - kEpiWarp0 * 32;   // epilogue thread 0..255
  constexpr int kEpiThreads = 4 * kEpiSets * 32;
  if (et >= 0 && et < kEpiThreads) {
    for (int i = et; i < NB * BM; i += kEpiThreads) {
      const int m = i / BM, r = i - m * BM;
      float s = red[m * BM + r];
#pragma unroll
      for (int e = 1; e < kEpiSets; ++e) s += red[(e * NB + m) * BM + r];
      const int owner = r / rpr;
      const uint32_t dst = smem_u32(recv + (rank * NB + m) * rpr + (r - owner * rpr));
      st_dsmem_f32(splits > 1 ? mapa_shared(dst, owner) : dst, s);
    }
  }
  if (splits > 1) cluster_sync();         // pushes visible to their owners
  else __syncthreads();
  if (et >= 0 && et < kEpiThreads && !failed) {
    for (int i = et; i < NB * rpr; i += kEpiThreads) {
      const int m = i / rpr, lr = i - m * rpr;
      const int r = rank * rpr + lr;
      if (m >= p.M || r >= BM || F::raw_row(r) >= F::kRows || (F::kQ2 && (r & 31) == 31)) continue;
      const int n = n0 + F::raw_row(r);
      if (n >= p.N) continue;
      float acc = recv[m * rpr + lr];
      for (int q = 1; q < splits; ++q) acc += recv[(q * NB + m) * rpr + lr];
      p.C[static_cast<size_t>(m) * p.ldc + n] = f32_to_bf16_rn(acc * p.gscale);
    }
  }
}

// ---------------------------------------------------------------- host side
// Same block size, registers and shared memory as tc_kernel<F, *>, without
// tensor-memory instructions: the occupancy calculator reports one CTA per SM
// for any kernel that allocates tensor memory, while two such CTAs of 256
// columns do run side by side, so cluster capacities are taken from this twin.
__global__ void __launch_bounds__(kThreads, kCtasPerSm) tc_capacity_twin() {}

// Clusters of s CTAs (1 <= s <= 8) of format F that are resident at once on
// the current device (0 if the query failed). Cached per device.
template <class F>
int cluster_capacity(int s) {
  static std::atomic<int> cache[kMaxDevices][9];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = cache[dev][s].load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  using L = Layout<F>;
  int n = 0;
  cudaError_t e = cudaFuncSetAttribute(tc_capacity_twin, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_capacity_twin, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = s;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, tc_capacity_twin, &cfg);
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();              // the query's failure is not the caller's error
    n = 0;
  }
  cache[dev][s].store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n;
}

// CTAs per tile (the cluster's K split): the largest s <= 8 (portable
// cluster size), at most one raw stage per CTA, for which all tiles' clusters
// are resident at once; clusters live inside one GPC, so the capacity is
// queried, not derived from the SM count (which only serves when the query
// fails).
template <class F>
int choose_splits(int tiles, int stages, int num_sms) {
  int best = 1;
  for (int sp = 2; sp <= 8 && sp <= stages; ++sp) {
    const int cap = cluster_capacity<F>(sp);
    const bool fits = cap > 0 ? tiles <= cap : sp * tiles <= kCtasPerSm * num_sms;
    if (fits) best = sp;
  }
  return best;
}

template <class F, int NB>
cudaError_t launch_tc_nb(const CUtensorMap& mw, const CUtensorMap& mw2, const CUtensorMap& ma, const TcParams& p,
                         int tiles, bool pdl,
                         cudaStream_t s) {
  using L = Layout<F>;
  // Two CTAs per SM need the whole shared-memory carveout.
  static AttrLatch latch;
  if (cudaError_t e0 = set_smem_attrs(tc_kernel<F, NB>, latch, L::kAlloc, true); e0 != cudaSuccess) return e0;
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
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, tc_kernel<F, NB>, mw, mw2, ma, p);
}

template <class F>
cudaError_t launch_tc(const GemvArgs& a, const CUtensorMap& mw, const CUtensorMap& mw2, cudaStream_t s) {
  CUtensorMap ma;
  const int nb = a.M <= 1 ? 1 : (a.M <= 2 ? 2 : (a.M <= 4 ? 4 : (a.M <= 8 ? 8 : 16)));   // box rows = NB
  cudaError_t e = make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.A, static_cast<uint64_t>(a.K),
                              static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.lda) * 2, 64, nb,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const int tiles = (a.N + F::kRows - 1) / F::kRows;
  TcParams p;
  p.A = static_cast<const uint16_t*>(a.A);
  p.lda = a.lda;
  p.scales = static_cast<const float*>(a.scales);
  p.gscale = a.gscale;
  p.C = static_cast<uint16_t*>(a.C);
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.ldc = a.ldc;
  p.stages = a.K / (GK * F::kGPR);
  p.splits = choose_splits<F>(tiles, p.stages, a.num_sms);
  p.err = a.err;
  if (a.M <= 1) return launch_tc_nb<F, 1>(mw, mw2, ma, p, tiles, a.pdl, s);
  if (a.M <= 2) return launch_tc_nb<F, 2>(mw, mw2, ma, p, tiles, a.pdl, s);
  if (a.M <= 4) return launch_tc_nb<F, 4>(mw, mw2, ma, p, tiles, a.pdl, s);
  if (a.M <= 8) return launch_tc_nb<F, 8>(mw, mw2, ma, p, tiles, a.pdl, s);
  return launch_tc_nb<F, 16>(mw, mw2, ma, p, tiles, a.pdl, s);
}

}  // namespace tc

cudaError_t launch_w8a16_gemm_tc(const GemvArgs& a, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mw;
  cudaError_t e = cached_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, static_cast<uint64_t>(a.K),
                              static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K), GK, BM,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return launch_tc<Fp8Tc>(a, mw, mw, s);
}

// Requires K % 1024 == 0 (checked by the caller): a row is then 34 * K / 128
// bytes, a multiple of 16, and each raw stage of 8 groups starts on a
// 16-byte boundary.
cudaError_t launch_q2_gemm_tc(const GemvArgs& a, cudaStream_t s) {
  using namespace tc;
  const uint64_t G = static_cast<uint64_t>(a.K / GK);
  CUtensorMap mw;
  cudaError_t e = cached_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.W, 17 * G, static_cast<uint64_t>(a.N),
                              34 * G, 8 * 17, Q2Tc::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return launch_tc<Q2Tc>(a, mw, mw, s);
}

// Requires K % 256 == 0 (checked by the caller): the scale rows (K/16 bytes)
// are then a multiple of 16 bytes, as tensor maps need, and every raw stage
// holds two whole groups.
cudaError_t launch_w4a16_gemm_tc(const GemvArgs& a, cudaStream_t s) {
  using namespace tc;
  const uint64_t K = static_cast<uint64_t>(a.K);
  CUtensorMap mw, ms;
  cudaError_t e = cached_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, K / 2, static_cast<uint64_t>(a.N), K / 2,
                              128, W4Tc::kRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = cached_map_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.scales, K / 16, static_cast<uint64_t>(a.N), K / 16, 16,
                  W4Tc::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return launch_tc<W4Tc>(a, mw, ms, s);
}

}  // namespace wqp
