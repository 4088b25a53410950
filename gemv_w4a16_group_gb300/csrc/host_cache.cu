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
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  int rank, dtype, swizzle;
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

namespace {

// Tiled descriptor of a rank-2 or rank-3 tensor (dims innermost first, byte strides of the
// outer dims), unit element strides, out-of-bounds elements read as zero; cached by its
// arguments.
cudaError_t encode_cached(CUtensorMap* map, CUtensorMapDataType dt, const void* base, int rank,
                          const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                          CUtensorMapSwizzle swizzle) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in the comparison
  key.base = base;
  key.rank = rank;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
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
  cuuint64_t d[3], s[2];
  cuuint32_t b[3];
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_maps.size() >= kMaxMaps) g_maps.clear();
  g_maps[key] = *map;
  return cudaSuccess;
}

}  // namespace

cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {row_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, dt, base, 2, dims, strides, box, swizzle);
}

cudaError_t encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                                 const uint64_t dims[3], const uint64_t strides[2],
                                 const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  return encode_cached(map, dt, base, 3, dims, strides, box, swizzle);
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
