// Host-side tensor-map encoding (cuTensorMapEncodeTiled, reached through the
// runtime's driver entry point so no driver library is linked).
#include <cudaTypedefs.h>

#include <mutex>

#include "gemv_scalar.cuh"
#include "internal.h"

namespace wqp {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

cudaError_t make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
// Encoded maps keyed by everything they encode (and the device). A map holds
// only the address, shape, pitch and box, so a cached one stays valid for
// any buffer later placed at the same address.
struct MapKey {
  int dev;
  CUtensorMapDataType dt;
  const void* base;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  CUtensorMapSwizzle sw;
  bool operator==(const MapKey& o) const {
    return dev == o.dev && dt == o.dt && base == o.base && inner == o.inner && outer == o.outer &&
           row_bytes == o.row_bytes && box_inner == o.box_inner && box_outer == o.box_outer && sw == o.sw;
  }
};
constexpr int kMapCache = 128;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int n = 0, next = 0;
};
MapCache& map_cache() {
  static MapCache c;
  return c;
}
}  // namespace

cudaError_t cached_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const MapKey k{dev, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw};
  MapCache& c = map_cache();
  {
    std::lock_guard<std::mutex> lk(c.mu);
    for (int i = 0; i < c.n; ++i)
      if (c.key[i] == k) {
        *m = c.map[i];
        return cudaSuccess;
      }
  }
  e = make_map_2d(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(c.mu);
  const int i = c.n < kMapCache ? c.n++ : (c.next++ % kMapCache);
  c.key[i] = k;
  c.map[i] = *m;
  return cudaSuccess;
}

cudaError_t make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t b[3] = {box[0], box[1], box[2]};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
struct Map3Key {
  int dev;
  CUtensorMapDataType dt;
  const void* base;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  CUtensorMapSwizzle sw;
  bool operator==(const Map3Key& o) const {
    return dev == o.dev && dt == o.dt && base == o.base && sw == o.sw && dims[0] == o.dims[0] &&
           dims[1] == o.dims[1] && dims[2] == o.dims[2] && strides[0] == o.strides[0] &&
           strides[1] == o.strides[1] && box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2];
  }
};
struct Map3Cache {
  std::mutex mu;
  Map3Key key[kMapCache];
  CUtensorMap map[kMapCache];
  int n = 0, next = 0;
};
Map3Cache& map3_cache() {
  static Map3Cache c;
  return c;
}
}  // namespace

cudaError_t cached_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                          const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle sw) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const Map3Key k{dev, dt, base, {dims[0], dims[1], dims[2]}, {strides_bytes[0], strides_bytes[1]},
                  {box[0], box[1], box[2]}, sw};
  Map3Cache& c = map3_cache();
  {
    std::lock_guard<std::mutex> lk(c.mu);
    for (int i = 0; i < c.n; ++i)
      if (c.key[i] == k) {
        *m = c.map[i];
        return cudaSuccess;
      }
  }
  e = make_map_3d(m, dt, base, dims, strides_bytes, box, sw);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(c.mu);
  const int i = c.n < kMapCache ? c.n++ : (c.next++ % kMapCache);
  c.key[i] = k;
  c.map[i] = *m;
  return cudaSuccess;
}

cudaError_t make_act_map(CUtensorMap* m, const GemvArgs& a, int box_k) {
  // BF16 pairs as u32: K/2 columns, M rows, pitch lda * 2 bytes.
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.A, static_cast<uint64_t>(a.K / 2),
                     static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.lda) * 2,
                     static_cast<uint32_t>(box_k / 2), static_cast<uint32_t>(a.M), CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t make_rows_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  return make_map_2d(m, dt, base, inner, rows, row_bytes, box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace wqp
