// Internal launch interface between the C-ABI layer (abi.cu) and the kernel
// translation units. Not installed; the public surface is include/wqp.h.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace wqp {

// Devices a process may use with the per-device caches below.
constexpr int kMaxDevices = 64;

// Per-device latch for kernel attributes. cudaFuncSetAttribute acts on the
// current device's context, so the opt-in above 48 KB of dynamic shared
// memory (and the carveout) is set once per device, not once per process.
struct AttrLatch {
  std::atomic<int> done[kMaxDevices];
};

// Sets the dynamic shared-memory limit of `kernel` to `bytes` (and, when
// asked, the largest shared-memory carveout) on the current device, once.
// Racing callers may both set it; the values are the same.
template <typename Kern>
cudaError_t set_smem_attrs(Kern kernel, AttrLatch& latch, int bytes, bool max_carveout) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (latch.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && max_carveout)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (e == cudaSuccess) latch.done[dev].store(1, std::memory_order_release);
  return e;
}

// Bits of the device error word.
constexpr unsigned WQP_DEV_ERR_TIMEOUT = 1u;

// One launch computes rows [0, M) of C with 1 <= M <= 16.
struct GemvArgs {
  const void* A;        // bf16 [M, lda]
  const void* W;        // packed weights
  const void* scales;   // format-specific (NULL for Q2_0)
  void* C;              // bf16 [M, ldc]
  int M, N, K;
  int lda, ldc;         // row pitches in elements
  float gscale;         // W4 per-tensor scale (1.0 otherwise)
  unsigned* err;        // device error word
  int num_sms;
  bool pdl;             // launch with programmatic stream serialization
};

struct DequantArgs {
  const void* W;
  const void* scales;
  float* out;           // f32 [N, K]
  int N, K;
  float gscale;
  bool pdl;
};

cudaError_t launch_q2_gemv(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_w4a16_gemv(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_w8a16_gemm(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_w8a16_gemm_tc(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_q2_gemm_tc(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_q2_gemm_mma(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_q2_gemm_stream(const GemvArgs& a, cudaStream_t s);
// Whether the persistent Q2_0 kernel has a plan for the shape (N, K, device).
bool q2_gemm_stream_fits(const GemvArgs& a);
cudaError_t launch_w4a16_gemm_tc(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_w8a16_gemm_mma(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_w4a16_gemm_mma(const GemvArgs& a, cudaStream_t s);
// W4 short-CTA kernel (gemm_mma_w4s.cu): shapes it serves, and its launch
// (M <= 8 per launch).
bool w4a16_short_fits(const GemvArgs& a);
cudaError_t launch_w4a16_gemm_short(const GemvArgs& a, cudaStream_t s);

cudaError_t launch_q2_dequant(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_w4a16_dequant(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_w8a16_dequant(const DequantArgs& a, cudaStream_t s);

// 2-D tensor map (tmap.cu): inner extent in elements, row pitch in bytes,
// box of box_inner x box_outer elements, no interleave, zero out-of-range fill.
cudaError_t make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle sw);

// Same, through a per-process cache keyed by every argument and the device
// (weight maps: encoding one costs about as much host time as a launch).
cudaError_t cached_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle sw);

// 3-D tensor map (tmap.cu): dims innermost first, byte strides of dims 1 and
// 2 (any order in memory: a block-of-rows view uses a row pitch for dim 1
// and a smaller block pitch for dim 2), box per dim; and its cached form.
cudaError_t make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle sw);
cudaError_t cached_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                          const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle sw);

// Launch helper: programmatic stream serialization when pdl is set.
template <typename Kern, typename... Args>
cudaError_t launch(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                   Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace wqp
