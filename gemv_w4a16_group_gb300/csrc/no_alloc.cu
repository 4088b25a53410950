// w4a16_matmul_noalloc: the W4A16 matmul for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc, or to hand the library a buffer of
// their own: a plugin running inside another runtime that owns every byte of device
// memory, or a latency-critical loop where an allocation (and the device-wide
// synchronization cudaMalloc/cudaFree may cause) is not acceptable. The regular
// w4a16_matmul needs a caller-owned workspace to split K across thread blocks for small
// batches. This entry point runs the same tensor-core kernel with the same split plan,
// but its scratch (per-tile arrival counters and fp32 partial tiles) is a fixed array
// compiled into the library, so the call allocates nothing.
//
// Consequences a caller must know:
//   * Every GPU that loads the library reserves kScratchBytes (16 MiB) of device memory
//     for the array until the process exits.
//   * A shape whose split plan needs more than kScratchBytes is rejected with
//     W4A16_ERR_WORKSPACE before anything is launched.
//   * All calls on a device share the one array, and it keeps whatever the last call
//     left in it. Each call clears the counters it needs (cudaMemsetAsync on its
//     stream) before its launch. Two calls whose kernels overlap on the GPU (different
//     streams without ordering between them) race on the array; order them on one
//     stream, or with events.
//   * The first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (the array's name in host code is only a host-side stand-in,
//     not a device address). Make that first call before any stream capture.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "launch.h"
#include "w4a16.h"

namespace {
constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;
constexpr int kMaxDevices = 64;
}  // namespace

// Split-K scratch of w4a16_matmul_noalloc: counters first, partial tiles after them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Device address of g_noalloc_scratch on the current device, looked up once per device
// with that device current; nullptr if the lookup fails.
void* scratch_device_address() {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return nullptr;
    ptrs[dev] = ptr;
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" w4a16_status w4a16_matmul_noalloc(const uint16_t* x, const int32_t* qw,
                                             const uint16_t* scales, const uint16_t* mins,
                                             uint16_t* y, int M, int N, int K, int group,
                                             w4a16_stream_t stream) {
  if (!x || !qw || !scales || !mins || !y) return W4A16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (group != 128 || N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(scales) || !aligned16(mins) || !aligned16(y))
    return W4A16_ERR_MISALIGNED;
  size_t need = 0;
  w4k::TcSplit split = w4k::tc_split_plan(M, N, K, &need);
  if (need > kScratchBytes) return W4A16_ERR_WORKSPACE;
  uint32_t* status = w4k::status_word();
  if (status == nullptr) return W4A16_ERR_CUDA;
  void* base = scratch_device_address();
  if (base == nullptr) return W4A16_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int bm = w4k::tc_block_m(M);
  w4k::TcMaps maps;
  if (w4k::make_tc_maps(x, reinterpret_cast<const uint32_t*>(qw), scales, mins, M, N, K, bm,
                        &maps) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (split.splits > 1) {
    const size_t tiles = static_cast<size_t>((N + 127) / 128) * ((M + bm - 1) / bm);
    const size_t counters = ((tiles * 4 + 255) / 256) * 256;
    // The arrival counters must start at zero whatever an earlier call left behind.
    if (cudaMemsetAsync(base, 0, counters, s) != cudaSuccess) return W4A16_ERR_CUDA;
    split.counter = static_cast<uint32_t*>(base);
    split.partial = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + counters);
  } else {
    split = w4k::TcSplit();
  }
  const cudaError_t e = w4k::launch_w4a16_tc(maps, y, M, N, K, bm, status,
                                             w4k::kDefaultWaitLimitNs, split, s);
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}
