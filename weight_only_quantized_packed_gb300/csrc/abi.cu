// C-ABI layer of libwqp.so: argument validation, per-device set-up, row
// chunking and dispatch to the kernel translation units. Declarations and the
// contract of every entry point are in include/wqp.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/wqp.h"
#include "common.cuh"
#include "internal.h"

using namespace wqp;

namespace {

// Device error word (one per device image of this module).
__device__ unsigned g_device_error = 0;

thread_local char t_last_error[256] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(WQP_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

std::atomic<int> g_pdl{0};

struct DeviceInfo {
  std::once_flag once;
  int status = WQP_OK;
  int num_sms = 0;
  unsigned* err = nullptr;
  char msg[160] = "";
};
DeviceInfo g_dev[kMaxDevices];

// Per-device set-up, run once with that device current: checks for sm_103
// and resolves the device error word's address.
int device_setup(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(WQP_ERR_UNSUPPORTED, "device %d", dev);
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&] {
    int major = 0, minor = 0;
    cudaError_t e1 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaError_t e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaError_t e3 = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
      d.status = WQP_ERR_CUDA;
      snprintf(d.msg, sizeof(d.msg), "device attribute query failed");
      return;
    }
    if (major != 10 || minor != 3) {
      d.status = WQP_ERR_UNSUPPORTED;
      snprintf(d.msg, sizeof(d.msg), "device %d is sm_%d%d; libwqp is built for sm_103a", dev,
               major, minor);
      return;
    }
    cudaError_t e4 = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_device_error);
    if (e4 != cudaSuccess) {
      d.status = WQP_ERR_CUDA;
      snprintf(d.msg, sizeof(d.msg), "cudaGetSymbolAddress: %s", cudaGetErrorString(e4));
    }
  });
  if (d.status != WQP_OK) return fail(d.status, "%s", d.msg);
  *out = &d;
  return WQP_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

enum class Fmt { Q2, W4, W8, W8TC, Q2TC, W4TC, Q2MMA, W8MMA, W4MMA };

const char* fmt_name(Fmt f) {
  switch (f) {
    case Fmt::Q2: return "q2_gemv";
    case Fmt::W4: return "w4a16_gemv";
    case Fmt::W8: return "w8a16_gemm";
    case Fmt::W8TC: return "w8a16_gemm_tc";
    case Fmt::Q2TC: return "q2_gemm_tc";
    case Fmt::W4TC: return "w4a16_gemm_tc";
    case Fmt::Q2MMA: return "q2_gemm_mma";
    case Fmt::W8MMA: return "w8a16_gemm_mma";
    case Fmt::W4MMA: return "w4a16_gemm_mma";
  }
  return "?";
}

int validate(Fmt f, const void* A, int lda, const void* W, const void* scales, void* C, int ldc,
             int M, int N, int K) {
  const char* nm = fmt_name(f);
  if (M < 0) return fail(WQP_ERR_INVALID_ARG, "%s: M=%d < 0", nm, M);
  const bool w4 = (f == Fmt::W4 || f == Fmt::W4TC || f == Fmt::W4MMA);
  const bool q2 = (f == Fmt::Q2 || f == Fmt::Q2TC || f == Fmt::Q2MMA);
  if (N < 1 || N > (1 << 24)) return fail(WQP_ERR_INVALID_ARG, "%s: N=%d outside 1..2^24", nm, N);
  if (K < 128 || K > (1 << 20) || K % 128 != 0)
    return fail(WQP_ERR_INVALID_ARG, "%s: K=%d must be a multiple of 128 in [128, 2^20]", nm, K);
  if (!A || !W || !C) return fail(WQP_ERR_INVALID_ARG, "%s: NULL A, W or C", nm);
  if ((f == Fmt::Q2TC || f == Fmt::Q2MMA || f == Fmt::W8MMA || f == Fmt::W4MMA) && K % 1024 != 0)
    return fail(WQP_ERR_INVALID_ARG, "%s: K=%d must be a multiple of 1024", nm, K);
  if (f == Fmt::W4TC && K % 256 != 0)
    return fail(WQP_ERR_INVALID_ARG, "%s: K=%d must be a multiple of 256", nm, K);
  if (q2 && scales)
    return fail(WQP_ERR_INVALID_ARG, "%s: Q2_0 scales are inline; scales must be NULL", nm);
  if (!q2 && !scales) return fail(WQP_ERR_INVALID_ARG, "%s: NULL scales", nm);
  if (!aligned(A, 16) || !aligned(W, 16))
    return fail(WQP_ERR_INVALID_ARG, "%s: A and W must be 16-byte aligned", nm);
  if (w4 && !aligned(scales, 16))
    return fail(WQP_ERR_INVALID_ARG, "%s: scales must be 16-byte aligned", nm);
  if ((f == Fmt::W8 || f == Fmt::W8TC) && !aligned(scales, 4))
    return fail(WQP_ERR_INVALID_ARG, "%s: scales must be 4-byte aligned", nm);
  if (f == Fmt::W8MMA && !aligned(scales, 16))
    return fail(WQP_ERR_INVALID_ARG, "%s: scales must be 16-byte aligned", nm);
  if (!aligned(C, 2)) return fail(WQP_ERR_INVALID_ARG, "%s: C must be 2-byte aligned", nm);
  if (lda < K || lda % 8 != 0)
    return fail(WQP_ERR_INVALID_ARG, "%s: lda=%d must be >= K=%d and a multiple of 8", nm, lda, K);
  if (ldc < N) return fail(WQP_ERR_INVALID_ARG, "%s: ldc=%d must be >= N=%d", nm, ldc, N);
  return WQP_OK;
}

int run_gemm(Fmt f, const void* A, int lda, const void* W, const void* scales, float gscale,
             void* C, int ldc, int M, int N, int K, void* stream) {
  int st = validate(f, A, lda, W, scales, C, ldc, M, N, K);
  if (st != WQP_OK) return st;
  if ((f == Fmt::W4 || f == Fmt::W4TC || f == Fmt::W4MMA) && !(gscale == gscale))
    return fail(WQP_ERR_INVALID_ARG, "%s: global_scale is NaN", fmt_name(f));
  if (M == 0) return WQP_OK;
  DeviceInfo* dev = nullptr;
  if ((st = device_setup(&dev)) != WQP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemvArgs a = {};
  a.W = W;
  a.scales = scales;
  a.N = N;
  a.K = K;
  a.lda = lda;
  a.ldc = ldc;
  a.gscale = gscale;
  a.err = dev->err;
  a.num_sms = dev->num_sms;
  a.pdl = g_pdl.load(std::memory_order_relaxed) != 0;
  const int step = WQP_MAX_M_PER_LAUNCH;
  for (int r0 = 0; r0 < M; r0 += step) {
    a.M = (M - r0) < step ? (M - r0) : step;
    a.A = static_cast<const char*>(A) + static_cast<size_t>(r0) * lda * 2;
    a.C = static_cast<char*>(C) + static_cast<size_t>(r0) * ldc * 2;
    cudaError_t e = cudaSuccess;
    switch (f) {
      case Fmt::Q2: e = launch_q2_gemv(a, s); break;
      case Fmt::W4: e = launch_w4a16_gemv(a, s); break;
      case Fmt::W8: e = launch_w8a16_gemm(a, s); break;
      case Fmt::W8TC: e = launch_w8a16_gemm_tc(a, s); break;
      case Fmt::Q2TC: e = launch_q2_gemm_tc(a, s); break;
      case Fmt::W4TC: e = launch_w4a16_gemm_tc(a, s); break;
      case Fmt::Q2MMA: e = launch_q2_gemm_mma(a, s); break;
      case Fmt::W8MMA: e = launch_w8a16_gemm_mma(a, s); break;
      case Fmt::W4MMA: e = launch_w4a16_gemm_mma(a, s); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, fmt_name(f));
  }
  return WQP_OK;
}

int run_dequant(int fmt, const void* W, const void* scales, float gscale, float* out, int N, int K,
                void* stream) {
  static const char* names[] = {"q2_dequant", "w4a16_dequant", "w8a16_dequant"};
  const char* nm = names[fmt];
  if (N < 1 || N > (1 << 24)) return fail(WQP_ERR_INVALID_ARG, "%s: N=%d outside 1..2^24", nm, N);
  if (K < 128 || K > (1 << 20) || K % 128 != 0)
    return fail(WQP_ERR_INVALID_ARG, "%s: K=%d must be a multiple of 128 in [128, 2^20]", nm, K);
  if (!W || !out) return fail(WQP_ERR_INVALID_ARG, "%s: NULL W or out", nm);
  if (fmt == 0 && scales) return fail(WQP_ERR_INVALID_ARG, "%s: scales must be NULL", nm);
  if (fmt != 0 && !scales) return fail(WQP_ERR_INVALID_ARG, "%s: NULL scales", nm);
  if (!aligned(W, 16) || !aligned(out, 4))
    return fail(WQP_ERR_INVALID_ARG, "%s: W must be 16-byte and out 4-byte aligned", nm);
  if (fmt == 1 && !aligned(scales, 16))
    return fail(WQP_ERR_INVALID_ARG, "%s: scales must be 16-byte aligned", nm);
  if (fmt == 2 && !aligned(scales, 4))
    return fail(WQP_ERR_INVALID_ARG, "%s: scales must be 4-byte aligned", nm);
  DeviceInfo* dev = nullptr;
  int st = device_setup(&dev);
  if (st != WQP_OK) return st;
  DequantArgs a = {W, scales, out, N, K, gscale, g_pdl.load(std::memory_order_relaxed) != 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fmt == 0   ? launch_q2_dequant(a, s)
                  : fmt == 1 ? launch_w4a16_dequant(a, s)
                             : launch_w8a16_dequant(a, s);
  if (e != cudaSuccess) return cuda_fail(e, nm);
  return WQP_OK;
}

}  // namespace

namespace wqp {
// A bounded wait that nothing completes: one CTA waits, through the same
// helper the GEMM kernels use, on an mbarrier no thread arrives on. The wait
// gives up after limit_ns of wall time, records the timeout in the device
// error word and the kernel returns (no trap, no fault, no hang).
__global__ void wait_timeout_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t never;
  const uint32_t bar = smem_u32(&never);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_ns(bar, 0, err, limit_ns);
}
}  // namespace wqp

extern "C" {

int q2_gemv(const void* A, const void* W, const void* scales, void* C, int M, int N, int K,
            void* stream) {
  if (scales) return fail(WQP_ERR_INVALID_ARG, "q2_gemv: Q2_0 scales are inline; must be NULL");
  return run_gemm(Fmt::Q2, A, K, W, nullptr, 1.0f, C, N, M, N, K, stream);
}

int q2_gemv_strided(const void* A, int lda, const void* W, void* C, int ldc, int M, int N, int K,
                    void* stream) {
  return run_gemm(Fmt::Q2, A, lda, W, nullptr, 1.0f, C, ldc, M, N, K, stream);
}

int q2_gemm_tc(const void* A, const void* W, void* C, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::Q2TC, A, K, W, nullptr, 1.0f, C, N, M, N, K, stream);
}

int q2_gemm_tc_strided(const void* A, int lda, const void* W, void* C, int ldc, int M, int N, int K,
                       void* stream) {
  return run_gemm(Fmt::Q2TC, A, lda, W, nullptr, 1.0f, C, ldc, M, N, K, stream);
}

int q2_gemm_mma(const void* A, const void* W, void* C, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::Q2MMA, A, K, W, nullptr, 1.0f, C, N, M, N, K, stream);
}

int q2_gemm_mma_strided(const void* A, int lda, const void* W, void* C, int ldc, int M, int N, int K,
                        void* stream) {
  return run_gemm(Fmt::Q2MMA, A, lda, W, nullptr, 1.0f, C, ldc, M, N, K, stream);
}

int w4a16_gemv(const void* A, const void* W, const void* scales, void* C, int M, int N, int K,
               void* stream) {
  return run_gemm(Fmt::W4, A, K, W, scales, 1.0f, C, N, M, N, K, stream);
}

int w4a16_gemv_ex(const void* A, int lda, const void* W, const void* scales, float global_scale,
                  void* C, int ldc, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::W4, A, lda, W, scales, global_scale, C, ldc, M, N, K, stream);
}

int w4a16_gemm_tc(const void* A, const void* W, const void* scales, void* C, int M, int N, int K,
                  void* stream) {
  return run_gemm(Fmt::W4TC, A, K, W, scales, 1.0f, C, N, M, N, K, stream);
}

int w4a16_gemm_tc_ex(const void* A, int lda, const void* W, const void* scales, float global_scale,
                     void* C, int ldc, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::W4TC, A, lda, W, scales, global_scale, C, ldc, M, N, K, stream);
}

int w4a16_gemm_mma(const void* A, const void* W, const void* scales, void* C, int M, int N, int K,
                   void* stream) {
  return run_gemm(Fmt::W4MMA, A, K, W, scales, 1.0f, C, N, M, N, K, stream);
}

int w4a16_gemm_mma_ex(const void* A, int lda, const void* W, const void* scales, float global_scale,
                      void* C, int ldc, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::W4MMA, A, lda, W, scales, global_scale, C, ldc, M, N, K, stream);
}

int w8a16_gemm_mma(const void* A, const void* W, const float* scales, void* C, int M, int N, int K,
                   void* stream) {
  return run_gemm(Fmt::W8MMA, A, K, W, scales, 1.0f, C, N, M, N, K, stream);
}

int w8a16_gemm_mma_strided(const void* A, int lda, const void* W, const float* scales, void* C,
                           int ldc, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::W8MMA, A, lda, W, scales, 1.0f, C, ldc, M, N, K, stream);
}

int w8a16_gemm(const void* A, const void* W, const float* scales, void* C, int M, int N, int K,
               void* stream) {
  return run_gemm(Fmt::W8, A, K, W, scales, 1.0f, C, N, M, N, K, stream);
}

int w8a16_gemm_strided(const void* A, int lda, const void* W, const float* scales, void* C,
                       int ldc, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::W8, A, lda, W, scales, 1.0f, C, ldc, M, N, K, stream);
}

int w8a16_gemm_tc(const void* A, const void* W, const float* scales, void* C, int M, int N, int K,
                  void* stream) {
  return run_gemm(Fmt::W8TC, A, K, W, scales, 1.0f, C, N, M, N, K, stream);
}

int w8a16_gemm_tc_strided(const void* A, int lda, const void* W, const float* scales, void* C,
                          int ldc, int M, int N, int K, void* stream) {
  return run_gemm(Fmt::W8TC, A, lda, W, scales, 1.0f, C, ldc, M, N, K, stream);
}

int q2_dequant(const void* W, float* out, int N, int K, void* stream) {
  return run_dequant(0, W, nullptr, 1.0f, out, N, K, stream);
}

int w4a16_dequant(const void* W, const void* scales, float global_scale, float* out, int N, int K,
                  void* stream) {
  return run_dequant(1, W, scales, global_scale, out, N, K, stream);
}

int w8a16_dequant(const void* W, const float* scales, float* out, int N, int K, void* stream) {
  return run_dequant(2, W, scales, 1.0f, out, N, K, stream);
}

int wqp_row_chunks(int M, int K, int N, int max_rows, long long* out, int cap) {
  if (M < 0 || K < 0 || N < 0 || max_rows < 1 || cap < 0) return -1;
  int n = 0;
  for (int r0 = 0; r0 < M; r0 += max_rows) {
    if (n >= cap || !out) return -1;
    int rows = (M - r0) < max_rows ? (M - r0) : max_rows;
    out[3 * n + 0] = static_cast<long long>(r0) * K * 2;
    out[3 * n + 1] = static_cast<long long>(r0) * N * 2;
    out[3 * n + 2] = rows;
    ++n;
  }
  return n;
}

int wqp_set_pdl(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

int wqp_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(WQP_ERR_INVALID_ARG, "wqp_selftest_wait_timeout: limit_us=%d outside 1..10^6", limit_us);
  DeviceInfo* dev = nullptr;
  int st = device_setup(&dev);
  if (st != WQP_OK) return st;
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev->err, static_cast<uint64_t>(limit_us) * 1000u);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wqp_selftest_wait_timeout");
  return WQP_OK;
}

int wqp_get_device_error(void) {
  DeviceInfo* dev = nullptr;
  int st = device_setup(&dev);
  if (st != WQP_OK) return st;
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "wqp_get_device_error");
  if (v) {
    unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "wqp_get_device_error");
    return fail(WQP_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait expired (word 0x%x)", v);
  }
  return WQP_OK;
}

const char* wqp_status_string(int status) {
  switch (status) {
    case WQP_OK: return "WQP_OK";
    case WQP_ERR_INVALID_ARG: return "WQP_ERR_INVALID_ARG";
    case WQP_ERR_UNSUPPORTED: return "WQP_ERR_UNSUPPORTED";
    case WQP_ERR_CUDA: return "WQP_ERR_CUDA";
    case WQP_ERR_DEVICE_TIMEOUT: return "WQP_ERR_DEVICE_TIMEOUT";
  }
  return "WQP_ERR_UNKNOWN";
}

const char* wqp_last_error(void) { return t_last_error; }

int wqp_abi_version(void) { return WQP_ABI_VERSION; }

}  // extern "C"
