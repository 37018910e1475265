// Host-side tensor-map encoding (cuTensorMapEncodeTiled, reached through the
// runtime's driver entry point so no driver library is linked).
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

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
// any buffer later placed at the same address. Hashed: a model's weights
// make hundreds of maps, and each call looks its own up.
struct MapKey {
  uint64_t w[10];   // device, type, rank, swizzle | base | dims[3] | strides[2] | box[3]
  bool operator==(const MapKey& o) const { return std::memcmp(w, o.w, sizeof w) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = 0;
    for (uint64_t x : k.w) h = (h ^ x) * 0x100000001B3ull + (h >> 29);
    return static_cast<size_t>(h);
  }
};
struct MapBits {
  uint64_t b[16];   // a CUtensorMap's 128 bytes
};
static_assert(sizeof(CUtensorMap) == sizeof(MapBits), "tensor map size");
constexpr size_t kMapCacheMax = 4096;   // maps kept (128 bytes each); all dropped once full
struct MapCache {
  std::mutex mu;
  std::unordered_map<MapKey, MapBits, MapKeyHash> maps;
};
MapCache& map_cache() {
  static MapCache c;
  return c;
}

MapKey map_key(int dev, CUtensorMapDataType dt, int rank, CUtensorMapSwizzle sw, const void* base,
               const uint64_t (&dims)[3], const uint64_t (&strides)[2], const uint32_t (&box)[3]) {
  MapKey k;
  k.w[0] = static_cast<uint64_t>(static_cast<uint32_t>(dev)) | (static_cast<uint64_t>(dt) << 32) |
           (static_cast<uint64_t>(rank) << 48) | (static_cast<uint64_t>(sw) << 56);
  k.w[1] = reinterpret_cast<uintptr_t>(base);
  for (int i = 0; i < 3; ++i) k.w[2 + i] = dims[i];
  for (int i = 0; i < 2; ++i) k.w[5 + i] = strides[i];
  for (int i = 0; i < 3; ++i) k.w[7 + i] = box[i];
  return k;
}

// The cached map of key k, or one encoded by make() and stored.
template <class Make>
cudaError_t lookup_or_make(const MapKey& k, CUtensorMap* m, Make make) {
  MapCache& c = map_cache();
  {
    std::lock_guard<std::mutex> lk(c.mu);
    const auto it = c.maps.find(k);
    if (it != c.maps.end()) {
      std::memcpy(m, &it->second, sizeof(MapBits));
      return cudaSuccess;
    }
  }
  const cudaError_t e = make();
  if (e != cudaSuccess) return e;
  MapBits bits;
  std::memcpy(&bits, m, sizeof(MapBits));
  std::lock_guard<std::mutex> lk(c.mu);
  if (c.maps.size() >= kMapCacheMax) c.maps.clear();
  c.maps[k] = bits;
  return cudaSuccess;
}
}  // namespace

cudaError_t cached_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const MapKey k = map_key(dev, dt, 2, sw, base, {inner, outer, 0}, {row_bytes, 0}, {box_inner, box_outer, 0});
  return lookup_or_make(k, m,
                        [&] { return make_map_2d(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw); });
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

cudaError_t cached_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                          const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle sw) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const MapKey k = map_key(dev, dt, 3, sw, base, dims, strides_bytes, box);
  return lookup_or_make(k, m, [&] { return make_map_3d(m, dt, base, dims, strides_bytes, box, sw); });
}

cudaError_t make_act_map(CUtensorMap* m, const GemvArgs& a, int box_k) {
  // BF16 pairs as u32: K/2 columns, M rows, pitch lda * 2 bytes.
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.A, static_cast<uint64_t>(a.K / 2),
                     static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.lda) * 2,
                     static_cast<uint32_t>(box_k / 2), static_cast<uint32_t>(a.M), CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t make_rows_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  return cached_map_2d(m, dt, base, inner, rows, row_bytes, box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace wqp
