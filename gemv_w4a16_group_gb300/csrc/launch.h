// Internal interface between the C ABI layer (api.cu) and the kernel files. Each
// launcher assumes its arguments were validated by the caller and returns the launch
// error (cudaGetLastError) without synchronizing.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace w4k {

// TMA descriptor of a 2-D tensor (inner dimension contiguous, rows `row_bytes` apart),
// box {box_inner, box_outer}, out-of-bounds elements read as zero. Cached by arguments.
cudaError_t encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                              uint64_t inner, uint64_t outer, uint64_t row_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
// The same for a rank-3 tensor: dims innermost first, byte strides of dims 1 and 2 (any
// order), box per dim.
cudaError_t encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                                 const uint64_t dims[3], const uint64_t strides[2],
                                 const uint32_t box[3], CUtensorMapSwizzle swizzle);
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device, size).
cudaError_t set_max_dynamic_smem(const void* func, int bytes);

// Bits of the per-device status word (read and cleared by w4a16_device_status).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusLayout = 2u;  // a kernel found its shared memory misaligned, skipped

// Default limit of a bounded wait (nanoseconds of %globaltimer).
constexpr uint64_t kDefaultWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Group-128 quantizers: a CTA per piece of up to 8192 floats of a row, staged by one bulk
// copy (bounded wait; an expiry is latched in `status`).
cudaError_t launch_w4a16_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales,
                                  uint16_t* mins, uint32_t* status, uint64_t wait_limit_ns,
                                  cudaStream_t stream);
cudaError_t launch_w4a16_pack(const uint8_t* codes, int N, int K, uint32_t* qw,
                              cudaStream_t stream);
cudaError_t launch_q4b32_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales,
                                  cudaStream_t stream);
// Zero-point format: quantize into [N, K/8] words and [N, K/128] FP16 scales and zeros, and
// transpose those into the matmul's [K/8, N] and [K/128, N].
cudaError_t launch_w4a16zp_quantize(const float* w, int N, int K, uint32_t* qw_rows,
                                    uint16_t* scales, uint16_t* zeros, uint32_t* status,
                                    uint64_t wait_limit_ns, cudaStream_t stream);
cudaError_t launch_w4a16zp_prepare(const uint32_t* qw_rows, const uint16_t* scales,
                                   const uint16_t* zeros, int N, int K, uint32_t* qw,
                                   uint16_t* scales_t, uint16_t* zeros_t, cudaStream_t stream);

// GEMV for M <= 8 (weights staged by TMA, codes widened to FP16 pairs in registers, inner
// products on mma.sync, per-group fold in fp32). With a split plan (splits > 1) the K range
// of each slab is divided over thread blocks: fp32 partials [splits][mr][N] and one arrival
// counter per slab (zero before the launch; the kernel leaves it zero). gemv_supports()
// tells whether M and K fit its limits. zero_point: `scales` and `mins` hold FP16 scales
// and zero points (w_hat = (q - z) s) instead of BF16 scales and minimums; the same holds
// for the skinny and tensor-core launchers below.
struct GemvSplit {
  int splits = 1;
  float* partial = nullptr;
  uint32_t* counter = nullptr;
  size_t partial_offset = 0;  // bytes of the workspace before the partials (the counters)
};
int gemv_max_rows();
bool gemv_supports(int M, int K);
GemvSplit gemv_split_plan(int M, int N, int K, size_t* bytes_needed);
cudaError_t launch_w4a16_gemv(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                              const uint16_t* mins, uint16_t* y, int M, int N, int K,
                              const GemvSplit& split, uint32_t* status, uint64_t wait_limit_ns,
                              cudaStream_t stream, bool zero_point = false);

// TMA + tcgen05 kernel: y^T tile = W_hat tile (tensor memory) x x^T tile (shared memory).
struct TcMaps {
  CUtensorMap x;       // bf16 [M, K], box {64, BM}, 128-byte swizzle
  CUtensorMap qw;      // int32 [K/8, N], box {128, 8}
  CUtensorMap scales;  // bf16 (fp16 with a zero point) [K/128, N], box {128, 1}
  CUtensorMap mins;    // bf16 minimums (fp16 zero points) [K/128, N], box {128, 1}
};
// Split-K over gridDim.z CTAs: fp32 partial tiles [splits][ceil(M/bm)*bm][N] and one
// arrival counter per output tile (zero before the launch; the kernel leaves it zero).
struct TcSplit {
  int splits = 1;
  float* partial = nullptr;
  uint32_t* counter = nullptr;
};
int tc_block_m(int M);
int tc_ctas_per_sm(int bm);  // resident CTAs per SM that tensor memory allows
// Split plan for this shape on the current device; *bytes_needed = workspace bytes
// (counters rounded to 256 B, then the partial tiles), 0 when the plan does not split.
TcSplit tc_split_plan(int M, int N, int K, size_t* bytes_needed);
// Device address of the library's status word on the current device (nullptr on error).
uint32_t* status_word();
cudaError_t make_tc_maps(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                         const uint16_t* mins, int M, int N, int K, int bm, TcMaps* maps,
                         bool zero_point = false);
cudaError_t launch_w4a16_tc(const TcMaps& maps, uint16_t* y, int M, int N, int K, int bm,
                            uint32_t* status, uint64_t wait_limit_ns, const TcSplit& split,
                            cudaStream_t stream, bool zero_point = false);

// Skinny W4A16 matmul for 1 <= M <= kSkinnyMaxRows (one to four n8 tiles of batch rows on
// mma.sync): a prep kernel converts x into the caller's workspace (FP16 fragments and
// per-group constants), then one CTA per SM streams its columns' weights and that x. Needs at
// least 32 columns per SM and at most 192; skinny_plan() tells and sizes the workspace.
constexpr int kSkinnyMaxRows = 32;
struct SkinnyPlan {
  int nt = 0;       // n8 tiles of batch rows
  int qw = 0;       // 32-column quarters per CTA
  int col_q = 0;    // columns per CTA: 8 col_q, the first col_r CTAs 8 (col_q + 1)
  int col_r = 0;
  int ctas = 0;
  int stages = 0;
  int rows_pad = 0;       // packed rows of x fragments (K/8 rounded up to whole chunks)
  size_t xs_bytes = 0;    // fragments, then the per-group constants
  size_t ws_bytes = 0;
};
bool skinny_plan(int M, int N, int K, SkinnyPlan* plan);
cudaError_t launch_w4a16_skinny(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                                const uint16_t* mins, uint16_t* y, int M, int N, int K,
                                void* workspace, const SkinnyPlan& plan, uint32_t* status,
                                uint64_t wait_limit_ns, cudaStream_t stream,
                                bool zero_point = false);

// Prepared (reordered) W4A16 layout: 128-column x 128-k records of 8704 bytes (codes with
// the even weights in the low half of each word, then one scale|minimum word per column),
// and the persistent tensor-core matmul that reads it (prepared.cu). The plan fixes the
// batch tile (BN rows, the MMA's N), the unit grid and, with a workspace, the stream-K
// split: arrival counters (zero before the launch; the kernel leaves them zero) and two
// fp32 partial tiles per CTA.
struct TcpPlan {
  int bn = 0;        // batch rows per tile
  int P = 0;         // row tiles
  int T = 0;         // 128-column tiles
  int ctas = 0;
  bool stream_k = false;
  size_t counter_bytes = 0;
  size_t ws_bytes = 0;  // 0 without stream-K
};
size_t w4a16_prepared_bytes(int N, int K);
int tcp_block_n(int M);
bool tcp_plan(int M, int N, int K, int sms, bool want_stream, TcpPlan* plan);
cudaError_t launch_w4a16_prepare(const uint32_t* qw, const uint16_t* scales, const uint16_t* mins,
                                 int N, int K, uint32_t* prep, cudaStream_t stream);
cudaError_t launch_w4a16_tcp(const uint16_t* x, const uint32_t* prep, uint16_t* y, int M, int N,
                             int K, const TcpPlan& plan, void* workspace, uint32_t* status,
                             uint64_t wait_limit_ns, cudaStream_t stream);

// Q4 block-32 GEMV.
cudaError_t launch_q4b32_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                              uint16_t* y, int N, int K, int variant, cudaStream_t stream);
// Q4 block-32 GEMV on the tensor pipe (TMA-staged, mma.sync FP16 -> fp32). Needs K % 256 == 0
// (TMA row strides of the scales) and x, its per-block constants and a two-stage ring in
// shared memory; q4b32_tc_supports() tells. Bounded waits report through `status`.
bool q4b32_tc_supports(int N, int K);
cudaError_t launch_q4b32_gemv_tc(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                                 uint16_t* y, int N, int K, uint32_t* status,
                                 uint64_t wait_limit_ns, cudaStream_t stream);

// W8A16 (symmetric per-row INT8): quantize, one CTA per row; GEMV, 16 rows per CTA with x
// (2 K bytes) in shared memory. K % 64 == 0.
uint32_t w8a16_smem_bytes(int K);
int device_sm_count();  // SMs of the current device (cached per device)
cudaError_t launch_w8a16_quantize(const float* w, int N, int K, int8_t* q, float* s,
                                  cudaStream_t stream);
cudaError_t launch_w8a16_gemv(const uint16_t* x, const int8_t* q, const float* s, uint16_t* y,
                              int N, int K, cudaStream_t stream);

// NVFP4 weights (E2M1 codes [N, K/2], E4M3 block scales [N, K/16], one fp32 tensor scale):
// quantize (amax, per-block codes, finalize; four stream-ordered steps) and the M = 1 GEMV.
// K % 128 == 0.
uint32_t nvfp4_smem_bytes(int K);
cudaError_t launch_nvfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                                  float* tensor_scale, cudaStream_t stream);
cudaError_t launch_nvfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                              const float* tensor_scale, uint16_t* y, int N, int K,
                              cudaStream_t stream);

// MXFP4 weights (E2M1 codes [N, K/2], E8M0 block scales [N, K/32]): quantize (K % 32 == 0)
// and the M = 1 GEMV (K % 128 == 0, shared memory as the NVFP4 GEMV).
cudaError_t launch_mxfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream);
cudaError_t launch_mxfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                              uint16_t* y, int N, int K, cudaStream_t stream);

// NVFP4 (mx = false) / MXFP4 (mx = true) GEMV on the tensor pipe (TMA-staged, mma.sync
// FP16 -> fp32), M = 1. Needs K % 512 == 0 and x, its per-block constants and a two-stage
// ring in shared memory; fp4_tc_supports() tells. `tensor_scale` is read for NVFP4 only.
// Bounded waits report through `status`.
bool fp4_tc_supports(int N, int K, bool mx);
cudaError_t launch_fp4_gemv_tc(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                               const float* tensor_scale, uint16_t* y, int N, int K, bool mx,
                               uint32_t* status, uint64_t wait_limit_ns, cudaStream_t stream);

// NVFP4 / MXFP4 matmul for M > 1: x prepared into the workspace (fp4_matmul_workspace_bytes),
// then one tensor-pipe pass per 32 rows of x. Needs K % 512 == 0; fp4_matmul_supports() tells
// whether every pass size fits in shared memory.
size_t fp4_matmul_workspace_bytes(int M, int K);
bool fp4_matmul_supports(int N, int K, bool mx);
cudaError_t launch_fp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                              const float* tensor_scale, uint16_t* y, int M, int N, int K,
                              bool mx, void* workspace, uint32_t* status, uint64_t wait_limit_ns,
                              cudaStream_t stream);

// W8A16 GEMV on the tensor pipe (TMA-staged, mma.sync FP16 -> fp32): K % 512 == 0 and x and
// a two-stage ring in shared memory; w8a16_tc_supports() tells. Bounded waits report through
// `status`.
bool w8a16_tc_supports(int N, int K);
cudaError_t launch_w8a16_gemv_tc(const uint16_t* x, const int8_t* q, const float* scales,
                                 uint16_t* y, int N, int K, uint32_t* status,
                                 uint64_t wait_limit_ns, cudaStream_t stream);

// Bounded-wait self test: waits on a barrier nothing arrives at.
cudaError_t launch_bounded_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace w4k
