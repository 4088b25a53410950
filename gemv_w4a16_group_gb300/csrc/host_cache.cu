// Host-side launch setup shared by the kernels: TMA descriptors (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so the library needs no -lcuda) and the
// dynamic shared-memory limit of each kernel. Both are cached: a decode step calls the same
// matmul on the same buffers over and over, and on the host these calls cost more than the
// launch itself. A descriptor depends only on its encode arguments, so an entry can never
// go stale: a buffer freed and reallocated at the same address with the same shape gets a
// descriptor that is still exact.
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "launch.h"

namespace w4k {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct MapKey {
  const void* base;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  int dtype, swizzle;
};

struct MapKeyEq {
  bool operator()(const MapKey& a, const MapKey& b) const {
    return std::memcmp(&a, &b, sizeof(MapKey)) == 0;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {  // FNV-1a over the key's bytes
    const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};

// A model's worth of layers (a few hundred buffers, three descriptors each) fits; past the
// bound the cache starts over rather than grow without limit.
constexpr size_t kMaxMaps = 8192;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash, MapKeyEq> g_maps;
std::mutex g_map_mu;

struct SmemEntry {
  const void* func;
  int dev, bytes;
};
constexpr int kSmemSlots = 256;
SmemEntry g_smem[kSmemSlots];
int g_smem_count = 0;
std::mutex g_smem_mu;

}  // namespace

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in the comparison
  key.base = base;
  key.inner = inner;
  key.outer = outer;
  key.row_bytes = row_bytes;
  key.box_inner = box_inner;
  key.box_outer = box_outer;
  key.dtype = static_cast<int>(dt);
  key.swizzle = static_cast<int>(swizzle);
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    const auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *map = it->second;
      return cudaSuccess;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_maps.size() >= kMaxMaps) g_maps.clear();
  g_maps[key] = *map;
  return cudaSuccess;
}

cudaError_t set_max_dynamic_smem(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_smem_mu);
  for (int i = 0; i < g_smem_count; ++i)
    if (g_smem[i].func == func && g_smem[i].dev == dev) {
      if (g_smem[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) g_smem[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_smem_count < kSmemSlots) g_smem[g_smem_count++] = {func, dev, bytes};
  return e;
}

}  // namespace w4k
