// Dequant entry points: unpack every weight to FP32 with the GEMV kernels'
// own decoders. A verification aid, not part of the hot path.
#include "decode.cuh"

namespace wqp {

// One thread per 16-code word: out[n, 128 g + 16 w + j] = ((c_j & 3) - 1) * d.
__global__ void q2_dequant_kernel(const uint8_t* W, float* out, int N, int K) {
  const int G = K >> 7;
  const long long words = static_cast<long long>(N) * G * 8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < words;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long blk = i >> 3;
    const int w = static_cast<int>(i & 7);
    const uint8_t* b = W + blk * 34;
    float2 v[8];
    const uint16_t* b16 = reinterpret_cast<const uint16_t*>(b);
    q2_decode_sub(static_cast<uint32_t>(__ldg(b16 + 2 * w)) | (static_cast<uint32_t>(__ldg(b16 + 2 * w + 1)) << 16), v);
    const float d = __half2float(__ushort_as_half(__ldg(b16 + 16)));
    float* o = out + (blk / G) * static_cast<long long>(K) + (blk % G) * 128 + 16 * w;
    // c * 4^j * 2^-149 times 2^75 and 2^74 / 4^j is the code c, exactly;
    // then (c - 1) times d, one rounding as in the oracle.
    constexpr float kTwo75 = 37778931862957161709568.0f, kTwo74 = 18889465931478580854784.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[2 * i] = ((v[i].x * kTwo75) * (kTwo74 / q2_pos_weight(2 * i)) - 1.0f) * d;
      o[2 * i + 1] = ((v[i].y * kTwo75) * (kTwo74 / q2_pos_weight(2 * i + 1)) - 1.0f) * d;
    }
  }
}

// One thread per code byte (two elements): (e2m1 * e4m3(scale)) * g.
__global__ void w4_dequant_kernel(const uint8_t* W, const uint8_t* S, float g, float* out, int N,
                                  int K) {
  const long long bytes = static_cast<long long>(N) * (K / 2);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < bytes;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long n = i / (K / 2);
    const long long j = i % (K / 2);
    const uint32_t h = e2m1x2_to_f16x2(__ldg(W + i));
    const float s = e4m3_to_f32(__ldg(S + n * (K / 16) + (2 * j) / 16));
    const float w0 = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
    const float w1 = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
    out[n * K + 2 * j] = (w0 * s) * g;
    out[n * K + 2 * j + 1] = (w1 * s) * g;
  }
}

// One thread per weight: e4m3(w) * s[n/128, k/128].
__global__ void w8_dequant_kernel(const uint8_t* W, const float* S, float* out, int N, int K) {
  const long long total = static_cast<long long>(N) * K;
  const int kb = K >> 7;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long n = i / K;
    const long long k = i % K;
    out[i] = e4m3_to_f32(__ldg(W + i)) * __ldg(S + (n >> 7) * kb + (k >> 7));
  }
}

namespace {
dim3 grid_for(long long items) {
  long long b = (items + 255) / 256;
  if (b > 65535LL * 16) b = 65535LL * 16;
  return dim3(static_cast<unsigned>(b < 1 ? 1 : b));
}
}  // namespace

cudaError_t launch_q2_dequant(const DequantArgs& a, cudaStream_t s) {
  return launch(q2_dequant_kernel, grid_for(static_cast<long long>(a.N) * (a.K / 128) * 8), dim3(256), 0, s,
                a.pdl, static_cast<const uint8_t*>(a.W), a.out, a.N, a.K);
}
cudaError_t launch_w4a16_dequant(const DequantArgs& a, cudaStream_t s) {
  return launch(w4_dequant_kernel, grid_for(static_cast<long long>(a.N) * (a.K / 2)), dim3(256), 0, s, a.pdl,
                static_cast<const uint8_t*>(a.W), static_cast<const uint8_t*>(a.scales), a.gscale,
                a.out, a.N, a.K);
}
cudaError_t launch_w8a16_dequant(const DequantArgs& a, cudaStream_t s) {
  return launch(w8_dequant_kernel, grid_for(static_cast<long long>(a.N) * a.K), dim3(256), 0, s, a.pdl,
                static_cast<const uint8_t*>(a.W), static_cast<const float*>(a.scales), a.out, a.N,
                a.K);
}

}  // namespace wqp
