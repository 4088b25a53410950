// C ABI of the library: host-side argument validation, kernel choice by batch size and
// the per-device status word. No entry point allocates memory.
#include <cstdint>
#include <mutex>

#include "launch.h"
#include "w4a16.h"
#include "w4a16_testing.h"

namespace {

// Status word written by kernels that detect a failure themselves (an expired bounded
// wait). One per device; read and cleared by w4a16_device_status.
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;

// Device address of g_status_word for the current device (looked up once per device).
uint32_t* status_word_ptr_impl() {
  static uint32_t* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

uint32_t* status_word_ptr() { return status_word_ptr_impl(); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

w4a16_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

// Kernel choice for w4a16_matmul: 0 = by M (default), 1 = small-M GEMV kernel,
// 2 = TMA + tcgen05 tensor-core kernel.
int g_force_kernel = 0;
// M at or below which the GEMV kernel (mma.sync inner products) runs when the choice is by M.
int g_gemv_max_m = 8;
int g_skinny_min_m = 5;  // M = 5..8 measured faster on the skinny kernel than on the GEMV
int g_skinny_max_m = 32;
// Range of M for which w4a16_matmul_prepared runs the prepared-layout tensor-core kernel
// (measured on the 14336 x 4096 layer: 1.6-1.7x the canonical path at M = 48..128, even at
// 32, the skinny kernel ahead at 16 and below, a tie from 192).
int g_prep_min_m = 32;
int g_prep_max_m = 128;
bool prep_by_m(int M) { return M >= g_prep_min_m && M <= g_prep_max_m; }

// The skinny kernel keeps its converted activations in the workspace past a reserve it
// never writes: the split-K kernels keep their arrival counters (which must stay zero
// between calls) at the start of the workspace, and any split plan that fits a workspace of
// W bytes has at most W / 128 + 256 bytes of counters (its fp32 partials take at least 128
// times the counters' bytes). So a workspace may be shared by skinny and split-K shapes.
size_t skinny_reserve(size_t workspace_bytes) {
  return ((workspace_bytes / 128 + 256 + 255) / 256) * 256;
}

// Smallest workspace (a multiple of 256 bytes) whose part past the reserve holds `bytes`.
size_t skinny_workspace_total(size_t bytes) {
  size_t w = ((bytes + 512 + 255) / 256) * 256;
  while (w - skinny_reserve(w) < bytes) w += 256;
  return w;
}

bool skinny_by_m(int M) { return M >= g_skinny_min_m && M <= g_skinny_max_m; }

uint64_t g_wait_limit_ns = w4k::kDefaultWaitLimitNs;

}  // namespace

namespace w4k {
uint32_t* status_word() { return status_word_ptr_impl(); }
}  // namespace w4k

// Split-K plan of the tensor-core kernel for this shape on the current device.
w4k::TcSplit w4k::tc_split_plan(int M, int N, int K, size_t* bytes_needed) {
  w4k::TcSplit plan;
  *bytes_needed = 0;
  static int sms_cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return plan;
  if (sms_cache[dev] == 0)
    cudaDeviceGetAttribute(&sms_cache[dev], cudaDevAttrMultiProcessorCount, dev);
  const int sms = sms_cache[dev];
  const int bm = w4k::tc_block_m(M);
  const long long tiles = static_cast<long long>((N + 127) / 128) * ((M + bm - 1) / bm);
  const long long slots = static_cast<long long>(sms) * w4k::tc_ctas_per_sm(bm);
  const int kb = K / 64;
  int splits = static_cast<int>(slots / (tiles > 0 ? tiles : 1));
  if (splits > kb / 2) splits = kb / 2;  // at least two k-blocks per CTA
  if (splits > 16) splits = 16;
  if (splits < 2) return plan;
  plan.splits = splits;
  const size_t counters = ((static_cast<size_t>(tiles) * 4 + 255) / 256) * 256;
  const size_t mp = static_cast<size_t>((M + bm - 1) / bm) * bm;
  *bytes_needed = counters + static_cast<size_t>(splits) * mp * N * 4;
  return plan;
}


extern "C" {

const char* w4a16_status_string(w4a16_status status) {
  switch (status) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG";
    case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED";
    case W4A16_ERR_MISALIGNED: return "W4A16_ERR_MISALIGNED";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
    case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT";
    case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE";
    case W4A16_ERR_LAYOUT: return "W4A16_ERR_LAYOUT";
  }
  return "W4A16_ERR_UNKNOWN";
}

w4a16_status w4a16_quantize(const float* w, int N, int K, int group, uint8_t* codes,
                            uint16_t* scales, uint16_t* mins, w4a16_stream_t stream) {
  if (!w || !codes || !scales || !mins) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || group <= 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (group != 128) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(mins))
    return W4A16_ERR_MISALIGNED;
  uint32_t* status = status_word_ptr();
  if (status == nullptr) return W4A16_ERR_CUDA;
  return from_cuda(w4k::launch_w4a16_quantize(w, N, K, codes, scales, mins, status,
                                              g_wait_limit_ns,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_pack(const uint8_t* codes, int N, int K, int32_t* qw, w4a16_stream_t stream) {
  if (!codes || !qw) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 8 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(qw)) return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_w4a16_pack(codes, N, K, reinterpret_cast<uint32_t*>(qw),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

size_t w4a16_matmul_workspace_bytes(int M, int N, int K, int group) {
  if (M <= 0 || N <= 0 || K <= 0 || group != 128 || K % group != 0) return 0;
  size_t bytes = 0;
  w4k::SkinnyPlan sk;
  if (skinny_by_m(M) && w4k::skinny_plan(M, N, K, &sk)) return skinny_workspace_total(sk.ws_bytes);
  if (M <= g_gemv_max_m && w4k::gemv_supports(M, K))
    w4k::gemv_split_plan(M, N, K, &bytes);
  else
    w4k::tc_split_plan(M, N, K, &bytes);
  return bytes;
}

}  // extern "C"

namespace {

// Both weight formats: zp selects FP16 scales and zero points over BF16 scales and minimums.
w4a16_status matmul_impl(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                         const uint16_t* mins, uint16_t* y, int M, int N, int K, int group,
                         void* workspace, size_t workspace_bytes, w4a16_stream_t stream,
                         bool zp) {
  if (!x || !qw || !scales || !mins || !y) return W4A16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (group != 128 || N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(scales) || !aligned16(mins) || !aligned16(y))
    return W4A16_ERR_MISALIGNED;
  if ((workspace == nullptr) != (workspace_bytes == 0)) return W4A16_ERR_WORKSPACE;
  if (workspace != nullptr && !aligned16(workspace)) return W4A16_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t* q = reinterpret_cast<const uint32_t*>(qw);
  uint32_t* status = status_word_ptr();
  if (status == nullptr) return W4A16_ERR_CUDA;
  int kernel = g_force_kernel;
  w4k::SkinnyPlan sk;
  const bool sk_plan = w4k::skinny_plan(M, N, K, &sk);
  const size_t sk_reserve = skinny_reserve(workspace_bytes);
  const bool sk_room = workspace != nullptr && workspace_bytes >= sk_reserve &&
                       workspace_bytes - sk_reserve >= sk.ws_bytes;
  if (kernel == 0) {
    if (skinny_by_m(M) && sk_plan && sk_room)
      kernel = 3;
    else
      kernel = (M <= g_gemv_max_m && w4k::gemv_supports(M, K)) ? 1 : 2;
  }
  if (kernel == 3) {
    if (!sk_plan) return W4A16_ERR_UNSUPPORTED;
    if (!sk_room) return W4A16_ERR_WORKSPACE;
    return from_cuda(w4k::launch_w4a16_skinny(x, q, scales, mins, y, M, N, K,
                                              static_cast<char*>(workspace) + sk_reserve, sk,
                                              status, g_wait_limit_ns, s, zp));
  }
  if (kernel == 1) {
    // The GEMV takes up to gemv_max_rows() rows per launch; larger M (forced) loops.
    const int step = w4k::gemv_max_rows();
    if (!w4k::gemv_supports(M < step ? M : step, K)) return W4A16_ERR_UNSUPPORTED;
    for (int m0 = 0; m0 < M; m0 += step) {
      const int mb = (M - m0) < step ? (M - m0) : step;
      // Split K over thread blocks when the caller's workspace holds the plan.
      size_t need = 0;
      w4k::GemvSplit split = w4k::gemv_split_plan(mb, N, K, &need);
      if (split.splits > 1 && workspace != nullptr && workspace_bytes >= need) {
        split.counter = static_cast<uint32_t*>(workspace);
        split.partial =
            reinterpret_cast<float*>(static_cast<char*>(workspace) + split.partial_offset);
      } else {
        split = w4k::GemvSplit();
      }
      cudaError_t e = w4k::launch_w4a16_gemv(x + static_cast<size_t>(m0) * K, q, scales, mins,
                                             y + static_cast<size_t>(m0) * N, mb, N, K, split,
                                             status, g_wait_limit_ns, s, zp);
      if (e != cudaSuccess) return W4A16_ERR_CUDA;
    }
    return W4A16_OK;
  }
  const int bm = w4k::tc_block_m(M);
  w4k::TcMaps maps;
  cudaError_t e = w4k::make_tc_maps(x, q, scales, mins, M, N, K, bm, &maps, zp);
  if (e != cudaSuccess) return W4A16_ERR_CUDA;
  // Split K across CTAs when the caller's workspace holds the plan's partial tiles.
  size_t need = 0;
  w4k::TcSplit split = w4k::tc_split_plan(M, N, K, &need);
  if (split.splits > 1 && workspace != nullptr && workspace_bytes >= need) {
    const size_t tiles = static_cast<size_t>((N + 127) / 128) * ((M + bm - 1) / bm);
    const size_t counters = ((tiles * 4 + 255) / 256) * 256;
    split.counter = static_cast<uint32_t*>(workspace);
    split.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + counters);
  } else {
    split = w4k::TcSplit();
  }
  return from_cuda(
      w4k::launch_w4a16_tc(maps, y, M, N, K, bm, status, g_wait_limit_ns, split, s, zp));
}

}  // namespace

extern "C" {

w4a16_status w4a16_matmul(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                          const uint16_t* mins, uint16_t* y, int M, int N, int K, int group,
                          void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  return matmul_impl(x, qw, scales, mins, y, M, N, K, group, workspace, workspace_bytes, stream,
                     false);
}

w4a16_status w4a16_matmul_host(const uint16_t* x_host, const int32_t* qw, const uint16_t* scales,
                               const uint16_t* mins, uint16_t* y_host, int M, int N, int K,
                               int group, uint16_t* x_dev, uint16_t* y_dev, void* workspace,
                               size_t workspace_bytes, w4a16_stream_t stream) {
  if (!x_host || !y_host || !x_dev || !y_dev) return W4A16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // argument checks of the product first, so that an invalid call copies nothing
  if (!qw || !scales || !mins) return W4A16_ERR_INVALID_ARG;
  if (group <= 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (group != 128 || N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(x_dev) || !aligned16(y_dev) || !aligned16(qw) || !aligned16(scales) ||
      !aligned16(mins))
    return W4A16_ERR_MISALIGNED;
  if ((workspace == nullptr) != (workspace_bytes == 0)) return W4A16_ERR_WORKSPACE;
  const size_t xb = static_cast<size_t>(M) * K * 2, yb = static_cast<size_t>(M) * N * 2;
  if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return W4A16_ERR_CUDA;
  const w4a16_status st = matmul_impl(x_dev, qw, scales, mins, y_dev, M, N, K, group, workspace,
                                      workspace_bytes, stream, false);
  if (st != W4A16_OK) return st;
  return from_cuda(cudaMemcpyAsync(y_host, y_dev, yb, cudaMemcpyDeviceToHost, s));
}

size_t w4a16_prepared_bytes(int N, int K, int group) {
  if (group != 128 || N <= 0 || K <= 0 || K % group != 0) return 0;
  return w4k::w4a16_prepared_bytes(N, K);
}

w4a16_status w4a16_prepare(const int32_t* qw, const uint16_t* scales, const uint16_t* mins,
                           int N, int K, int group, void* prepared, size_t prepared_bytes,
                           w4a16_stream_t stream) {
  if (!qw || !scales || !mins || !prepared) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || group <= 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (group != 128) return W4A16_ERR_UNSUPPORTED;
  if (prepared_bytes < w4k::w4a16_prepared_bytes(N, K)) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(qw) || !aligned16(scales) || !aligned16(mins) || !aligned16(prepared))
    return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_w4a16_prepare(reinterpret_cast<const uint32_t*>(qw), scales, mins,
                                             N, K, static_cast<uint32_t*>(prepared),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

size_t w4a16_matmul_prepared_workspace_bytes(int M, int N, int K, int group) {
  if (M <= 0 || N <= 0 || K <= 0 || group != 128 || K % group != 0) return 0;
  if (!prep_by_m(M)) return w4a16_matmul_workspace_bytes(M, N, K, group);
  w4k::TcpPlan plan;
  if (!w4k::tcp_plan(M, N, K, w4k::device_sm_count(), true, &plan)) return 0;
  return plan.ws_bytes;
}

w4a16_status w4a16_matmul_prepared(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                                   const uint16_t* mins, const void* prepared, uint16_t* y, int M,
                                   int N, int K, int group, void* workspace,
                                   size_t workspace_bytes, w4a16_stream_t stream) {
  if (prepared == nullptr || !prep_by_m(M))
    return matmul_impl(x, qw, scales, mins, y, M, N, K, group, workspace, workspace_bytes, stream,
                       false);
  if (!x || !qw || !scales || !mins || !y) return W4A16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || group <= 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
  if (group != 128 || N % 8 != 0) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(qw) || !aligned16(scales) || !aligned16(mins) ||
      !aligned16(y) || !aligned16(prepared))
    return W4A16_ERR_MISALIGNED;
  if ((workspace == nullptr) != (workspace_bytes == 0)) return W4A16_ERR_WORKSPACE;
  if (workspace != nullptr && !aligned16(workspace)) return W4A16_ERR_MISALIGNED;
  uint32_t* status = status_word_ptr();
  if (status == nullptr) return W4A16_ERR_CUDA;
  const int sms = w4k::device_sm_count();
  w4k::TcpPlan plan;
  if (!w4k::tcp_plan(M, N, K, sms, workspace != nullptr, &plan)) return W4A16_ERR_UNSUPPORTED;
  if (plan.stream_k && workspace_bytes < plan.ws_bytes &&
      !w4k::tcp_plan(M, N, K, sms, false, &plan))
    return W4A16_ERR_UNSUPPORTED;
  return from_cuda(w4k::launch_w4a16_tcp(x, static_cast<const uint32_t*>(prepared), y, M, N, K,
                                         plan, workspace, status, g_wait_limit_ns,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16zp_quantize(const float* w, int N, int K, int group, uint32_t* qw_rows,
                              uint16_t* scales, uint16_t* zeros, w4a16_stream_t stream) {
  if (!w || !qw_rows || !scales || !zeros) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || group <= 0 || K % group != 0 || group % 8 != 0)
    return W4A16_ERR_INVALID_ARG;
  if (group != 128) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(qw_rows) || !aligned16(scales) || !aligned16(zeros))
    return W4A16_ERR_MISALIGNED;
  uint32_t* status = status_word_ptr();
  if (status == nullptr) return W4A16_ERR_CUDA;
  return from_cuda(w4k::launch_w4a16zp_quantize(w, N, K, qw_rows, scales, zeros, status,
                                                g_wait_limit_ns,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16zp_prepare(const uint32_t* qw_rows, const uint16_t* scales,
                             const uint16_t* zeros, int N, int K, int group, int32_t* qw,
                             uint16_t* scales_t, uint16_t* zeros_t, w4a16_stream_t stream) {
  if (!qw_rows || !scales || !zeros || !qw || !scales_t || !zeros_t) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || group <= 0 || K % group != 0 || group % 8 != 0)
    return W4A16_ERR_INVALID_ARG;
  if (group != 128) return W4A16_ERR_UNSUPPORTED;
  if (!aligned16(qw_rows) || !aligned16(scales) || !aligned16(zeros) || !aligned16(qw) ||
      !aligned16(scales_t) || !aligned16(zeros_t))
    return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_w4a16zp_prepare(qw_rows, scales, zeros, N, K,
                                               reinterpret_cast<uint32_t*>(qw), scales_t,
                                               zeros_t, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16zp_matmul(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                            const uint16_t* zeros, uint16_t* y, int M, int N, int K, int group,
                            void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  return matmul_impl(x, qw, scales, zeros, y, M, N, K, group, workspace, workspace_bytes, stream,
                     true);
}

w4a16_status w8a16_quantize(const float* w, int N, int K, int8_t* q, float* scales,
                            w4a16_stream_t stream) {
  if (!w || !q || !scales) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 64 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q) || !aligned16(scales)) return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_w8a16_quantize(w, N, K, q, scales,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

static int g_w8_variant = 1;

w4a16_status w8a16_gemv(const uint16_t* x, const int8_t* q, const float* scales, uint16_t* y,
                        int N, int K, w4a16_stream_t stream) {
  if (!x || !q || !scales || !y) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 64 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || !aligned16(y))
    return W4A16_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (g_w8_variant == 1 && w4k::w8a16_tc_supports(N, K)) {
    uint32_t* status = status_word_ptr();
    if (status == nullptr) return W4A16_ERR_CUDA;
    return from_cuda(w4k::launch_w8a16_gemv_tc(x, q, scales, y, N, K, status, g_wait_limit_ns, s));
  }
  // K % 512 != 0 or x too long for the ring: the plain-load kernel.
  if (w4k::w8a16_smem_bytes(K) > 227u * 1024u) return W4A16_ERR_UNSUPPORTED;
  return from_cuda(w4k::launch_w8a16_gemv(x, q, scales, y, N, K, s));
}

w4a16_status nvfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                            float* tensor_scale, w4a16_stream_t stream) {
  if (!w || !codes || !scales || !tensor_scale) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 128 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(tensor_scale))
    return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_nvfp4_quantize(w, N, K, codes, scales, tensor_scale,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

static int g_fp4_variant = 1;

w4a16_status nvfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                        const float* tensor_scale, uint16_t* y, int N, int K,
                        w4a16_stream_t stream) {
  if (!x || !codes || !scales || !tensor_scale || !y) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 128 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(tensor_scale) ||
      !aligned16(y))
    return W4A16_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (g_fp4_variant == 1 && w4k::fp4_tc_supports(N, K, false)) {
    uint32_t* status = status_word_ptr();
    if (status == nullptr) return W4A16_ERR_CUDA;
    return from_cuda(w4k::launch_fp4_gemv_tc(x, codes, scales, tensor_scale, y, N, K, false,
                                             status, g_wait_limit_ns, s));
  }
  // K % 512 != 0 or x too long for the ring beside it: the plain-load kernel.
  if (w4k::nvfp4_smem_bytes(K) > 227u * 1024u) return W4A16_ERR_UNSUPPORTED;
  return from_cuda(w4k::launch_nvfp4_gemv(x, codes, scales, tensor_scale, y, N, K, s));
}

w4a16_status mxfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                            w4a16_stream_t stream) {
  if (!w || !codes || !scales) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales)) return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_mxfp4_quantize(w, N, K, codes, scales,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status mxfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                        uint16_t* y, int N, int K, w4a16_stream_t stream) {
  if (!x || !codes || !scales || !y) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 128 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y))
    return W4A16_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (g_fp4_variant == 1 && w4k::fp4_tc_supports(N, K, true)) {
    uint32_t* status = status_word_ptr();
    if (status == nullptr) return W4A16_ERR_CUDA;
    return from_cuda(w4k::launch_fp4_gemv_tc(x, codes, scales, nullptr, y, N, K, true, status,
                                             g_wait_limit_ns, s));
  }
  if (w4k::nvfp4_smem_bytes(K) > 227u * 1024u) return W4A16_ERR_UNSUPPORTED;
  return from_cuda(w4k::launch_mxfp4_gemv(x, codes, scales, y, N, K, s));
}

size_t fp4_matmul_workspace_bytes(int M, int K) {
  if (M <= 1 || K <= 0 || K % 512 != 0) return 0;
  return w4k::fp4_matmul_workspace_bytes(M, K);
}

static w4a16_status fp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                               const float* tensor_scale, uint16_t* y, int M, int N, int K,
                               bool mx, void* workspace, size_t workspace_bytes,
                               w4a16_stream_t stream) {
  if (M == 1)
    return mx ? mxfp4_gemv(x, codes, scales, y, N, K, stream)
              : nvfp4_gemv(x, codes, scales, tensor_scale, y, N, K, stream);
  if (!x || !codes || !scales || !y || (!mx && !tensor_scale)) return W4A16_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || K % 512 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y) ||
      (!mx && !aligned16(tensor_scale)))
    return W4A16_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < w4k::fp4_matmul_workspace_bytes(M, K))
    return W4A16_ERR_WORKSPACE;
  if (!aligned16(workspace)) return W4A16_ERR_MISALIGNED;
  if (!w4k::fp4_matmul_supports(N, K, mx)) return W4A16_ERR_UNSUPPORTED;
  uint32_t* status = status_word_ptr();
  if (status == nullptr) return W4A16_ERR_CUDA;
  return from_cuda(w4k::launch_fp4_matmul(x, codes, scales, tensor_scale, y, M, N, K, mx,
                                          workspace, status, g_wait_limit_ns,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status nvfp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                          const float* tensor_scale, uint16_t* y, int M, int N, int K,
                          void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  return fp4_matmul(x, codes, scales, tensor_scale, y, M, N, K, false, workspace,
                    workspace_bytes, stream);
}

w4a16_status mxfp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                          uint16_t* y, int M, int N, int K, void* workspace,
                          size_t workspace_bytes, w4a16_stream_t stream) {
  return fp4_matmul(x, codes, scales, nullptr, y, M, N, K, true, workspace, workspace_bytes,
                    stream);
}

w4a16_status q4b32_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales,
                            w4a16_stream_t stream) {
  if (!w || !codes || !scales) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales)) return W4A16_ERR_MISALIGNED;
  return from_cuda(w4k::launch_q4b32_quantize(w, N, K, codes, scales,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

static int g_q4_variant = 2;

w4a16_status q4b32_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                        uint16_t* y, int N, int K, w4a16_stream_t stream) {
  if (!x || !codes || !scales || !y) return W4A16_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y))
    return W4A16_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (g_q4_variant == 2 && w4k::q4b32_tc_supports(N, K)) {
    uint32_t* status = status_word_ptr();
    if (status == nullptr) return W4A16_ERR_CUDA;
    return from_cuda(
        w4k::launch_q4b32_gemv_tc(x, codes, scales, y, N, K, status, g_wait_limit_ns, s));
  }
  // Shapes the tensor-pipe kernel does not take (K % 256 != 0, very long K) use the
  // CUDA-core kernel.
  return from_cuda(w4k::launch_q4b32_gemv(x, codes, scales, y, N, K,
                                          g_q4_variant == 0 ? 0 : 1, s));
}

w4a16_status w4a16_device_status(w4a16_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return W4A16_ERR_CUDA;
  uint32_t* p = status_word_ptr();
  if (p == nullptr) return W4A16_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return W4A16_ERR_CUDA;
  }
  if (word & w4k::kStatusTimeout) return W4A16_ERR_TIMEOUT;
  return (word & w4k::kStatusLayout) ? W4A16_ERR_LAYOUT : W4A16_OK;
}

w4a16_status w4a16_selftest_bounded_wait(uint32_t limit_us, w4a16_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return W4A16_ERR_INVALID_ARG;
  uint32_t* p = status_word_ptr();
  if (p == nullptr) return W4A16_ERR_CUDA;
  return from_cuda(w4k::launch_bounded_wait_selftest(
      p, static_cast<uint64_t>(limit_us) * 1000ull, reinterpret_cast<cudaStream_t>(stream)));
}

// Test and benchmark hooks (declared in w4a16_testing.h, not part of the public header).
int w4a16_testing_force_kernel(int kernel) {
  if (kernel < 0 || kernel > 3) return -1;
  const int prev = g_force_kernel;
  g_force_kernel = kernel;
  return prev;
}

int w4a16_testing_set_gemv_max_m(int m) {
  const int prev = g_gemv_max_m;
  if (m >= 0) g_gemv_max_m = m;
  return prev;
}

int w4a16_testing_set_skinny_range(int lo, int hi) {
  const int prev = (g_skinny_min_m << 8) | g_skinny_max_m;
  if (lo >= 0 && hi >= 0 && lo <= 255 && hi <= w4k::kSkinnyMaxRows) {
    g_skinny_min_m = lo;
    g_skinny_max_m = hi;
  }
  return prev;
}

int w4a16_testing_set_prepared_min_m(int m) {
  const int prev = g_prep_min_m;
  if (m >= 1) g_prep_min_m = m;
  return prev;
}

int w4a16_testing_set_prepared_max_m(int m) {
  const int prev = g_prep_max_m;
  if (m >= 1) g_prep_max_m = m;
  return prev;
}

int w4a16_testing_set_q4_variant(int v) {
  const int prev = g_q4_variant;
  if (v >= 0 && v <= 2) g_q4_variant = v;
  return prev;
}

int w4a16_testing_set_w8_variant(int v) {
  const int prev = g_w8_variant;
  if (v >= 0 && v <= 1) g_w8_variant = v;
  return prev;
}

int w4a16_testing_set_fp4_variant(int v) {
  const int prev = g_fp4_variant;
  if (v >= 0 && v <= 1) g_fp4_variant = v;
  return prev;
}

}  // extern "C"
