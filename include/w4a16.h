/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 group-quantized matmul library.
 *
 * What it computes
 *   y = x . W_hat^T with x BF16 [M, K] activations and W_hat [N, K] rebuilt from
 *   4-bit codes as w_hat = q * s + min, one BF16 scale s = (max - min) / 15 and one
 *   BF16 minimum per group of 128 weights along K (4.25 bits per weight); eight codes
 *   are packed per int32 along K into a K/8 x N matrix ("Low-Precision Kernels: INT4,
 *   INT8 and FP8 Matmuls, Measured", Step 2). A second format is the 18-byte Q4 block
 *   of 32 codes plus an FP16 scale, w_hat = (q - 8) * s ("Why My 4-Bit CUDA Kernel
 *   Wasn't Faster", "Why fewer bytes should have helped"). A third is the zero-point
 *   form w_hat = (q - z) * s with FP16 scale and zero point per group of 128
 *   ("Quantization and GEMV", "The quantization formulas"), and the page's W8A16
 *   exercise adds symmetric per-row INT8 weights, w_hat = q * s; NVFP4 weights (E2M1
 *   codes with E4M3 block scales and an fp32 tensor scale) and MXFP4 weights (E2M1 codes
 *   with power-of-two E8M0 block scales) run weight-only as well.
 *
 * Conventions shared by every entry point
 *   - Every array pointer is DEVICE memory owned by the caller. The library keeps no
 *     pointer after a call returns and allocates nothing per call.
 *   - BF16 and FP16 arrays are passed as uint16_t bit patterns.
 *   - Every array is dense row-major (C order) with the shape given below; base
 *     pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Arguments are validated on the host before anything is launched; a
 *     call that returns an error status launched nothing.
 *   - W4A16_ERR_CUDA means a CUDA runtime call failed (the sticky or launch error is
 *     not cleared). Device-side faults the kernels detect themselves (a bounded wait
 *     that expired) are latched in a per-device status word that
 *     w4a16_device_status() reads and clears.
 *   - Weights must be finite.
 *   - The library caches per-device addresses of its own device variables (the status word
 *     and the scratch array of w4a16_matmul_noalloc) on first use. Resetting a device
 *     (cudaDeviceReset) after the library has been used on it is not supported: the
 *     cached addresses would no longer be valid.
 */
#ifndef W4A16_GB300_H
#define W4A16_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* w4a16_stream_t; /* identical to cudaStream_t */

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_INVALID_ARG = 1, /* null pointer, non-positive or inconsistent size */
  W4A16_ERR_UNSUPPORTED = 2, /* valid for the format but not by these kernels    */
  W4A16_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned                */
  W4A16_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed            */
  W4A16_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired (device status) */
  W4A16_ERR_WORKSPACE = 6,   /* workspace pointer/size does not meet the query  */
  W4A16_ERR_LAYOUT = 7       /* a kernel found its shared memory misaligned and
                                skipped its work (device status)                  */
} w4a16_status;

/* Human-readable name of a status (static string, never NULL). */
const char* w4a16_status_string(w4a16_status status);

/*
 * w4a16_quantize -- fp32 weights to 4-bit codes with a BF16 scale and minimum per
 * group ("Low-Precision Kernels ...", Step 2: a group is 128 neighbouring weights
 * along K, its scale is (max - min) / 15 and a weight's code is the integer
 * round((w - min) / scale), 0..15).
 *   w      fp32 [N, K]        (one output feature per row, K contiguous)
 *   codes  uint8 [N, K]       (one code 0..15 per byte)
 *   scales bf16 [K/group, N]  s = bf16_rne(fp32(max - min) / 15)
 *   mins   bf16 [K/group, N]  min = bf16_rne(min)
 * Per weight: q = clamp(rint((w - min_bf16) / s_bf16), 0, 15) in fp32 with
 * round-half-to-even; a group whose BF16 scale is 0 stores q = 0.
 * Requires N > 0, K > 0, group == 128, K % group == 0.
 */
w4a16_status w4a16_quantize(const float* w, int N, int K, int group, uint8_t* codes,
                            uint16_t* scales, uint16_t* mins, w4a16_stream_t stream);

/*
 * w4a16_pack -- eight codes per int32 along K ("Low-Precision Kernels ...", Step 2:
 * the N x K weights turn into a K/8 x N matrix of words, its listing takes k = 8r + j
 * from nibble j of word r; "Quantization and GEMV": the lowest nibble is the first
 * weight).
 *   codes uint8 [N, K] (values 0..15; higher bits are ignored)
 *   qw    int32 [K/8, N]: word (r, n) = sum_j codes[n, 8r + j] << 4j
 * Requires N > 0, K > 0, K % 8 == 0.
 */
w4a16_status w4a16_pack(const uint8_t* codes, int N, int K, int32_t* qw,
                        w4a16_stream_t stream);

/*
 * w4a16_matmul -- y = x . W_hat^T with w_hat[n, k] = q * s + min rebuilt in registers
 * ("Low-Precision Kernels ...", Step 2 and "Where the time goes at M = 1").
 *   x      bf16 [M, K]
 *   qw     int32 [K/8, N]  (as written by w4a16_pack)
 *   scales bf16 [K/group, N], mins bf16 [K/group, N]
 *   y      bf16 [M, N]     (fp32 accumulation, rounded to nearest even)
 * Kernel choice is by M: for 5 <= M <= 32 a skinny kernel (FP16 mma.sync with the batch in
 * n8 tiles) when the caller's workspace holds its converted activations; otherwise a GEMV for
 * M <= 8 and a TMA + tcgen05 tensor-core kernel above. Accuracy:
 * |y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k| per output, y_ref the exact
 * product on the same 4-bit weights. Results are deterministic (no floating-point
 * atomics).
 *   workspace / workspace_bytes: optional caller-owned device scratch that lets small-N
 *   shapes split K across thread blocks and lets 5 <= M <= 32 use the skinny kernel; size
 *   it with w4a16_matmul_workspace_bytes(). NULL (with 0 bytes) is always accepted. The
 *   workspace must be zero-filled before its first use and not shared by calls that may
 *   run concurrently. The split-K counters live in its first workspace_bytes / 128 + 256
 *   bytes (rounded up to 256), which the kernels leave zeroed; the skinny kernel writes
 *   its converted activations only past that reserve. Pass the same workspace_bytes for
 *   every call that shares a buffer.
 * Requires M > 0, N > 0, K > 0, group == 128, K % group == 0, N % 8 == 0.
 */
w4a16_status w4a16_matmul(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                          const uint16_t* mins, uint16_t* y, int M, int N, int K, int group,
                          void* workspace, size_t workspace_bytes, w4a16_stream_t stream);

/*
 * w4a16_matmul_host -- the same product with x and y in HOST memory: enqueues on `stream` the
 * copy of x_host (bf16 [M, K]) into x_dev, w4a16_matmul into y_dev, and the copy of y_dev
 * (bf16 [M, N]) back into y_host, then returns; synchronize the stream before reading
 * y_host. x_dev and y_dev are caller-owned device buffers of M*K and M*N bf16 (16-byte
 * aligned); host buffers should be page-locked for the copies to be asynchronous. Weights,
 * workspace, kernel choice, tolerance and errors as for w4a16_matmul; an argument error is
 * returned before anything is enqueued.
 */
w4a16_status w4a16_matmul_host(const uint16_t* x_host, const int32_t* qw, const uint16_t* scales,
                               const uint16_t* mins, uint16_t* y_host, int M, int N, int K,
                               int group, uint16_t* x_dev, uint16_t* y_dev, void* workspace,
                               size_t workspace_bytes, w4a16_stream_t stream);

/* Bytes of workspace that let w4a16_matmul split K for this shape, or run the skinny
 * kernel for 5 <= M <= 32 (0 = no benefit). */
size_t w4a16_matmul_workspace_bytes(int M, int N, int K, int group);

/*
 * Prepared (reordered) weights ("Quantization and GEMV", "What production kernels do": the
 * weights are rearranged once, offline, so that the kernel's wide reads feed the tensor-core
 * operand; "Low-Precision Kernels ...", "In the real world": reordered tiles whose nibbles
 * convert with one mask-and-or; "Hardware-invariant NVFP4 progress report 1", "Is it
 * faster?": a handle that owns prepared weights). The same codes, scales and minimums as
 * (qw, scales, mins), 4.25 bits per weight, in records of 128 columns x 128 k:
 *   record (t, g), at byte (t * K/128 + g) * 8704, is 2176 uint32 words:
 *     word b*1024 + h*512 + n*4 + j (b, h < 2, n < 128, j < 4) holds the 8 codes of column
 *       128 t + n at k = 128 g + 64 b + 8 (4 h + j) + 0..7: the code of k0 + 2i in bits
 *       4i..4i+3, the code of k0 + 2i + 1 in bits 16 + 4i..16 + 4i + 3;
 *     word 2048 + n: the BF16 scale of (g, column 128 t + n) in bits 0..15 and its BF16
 *       minimum in bits 16..31.
 *   Columns past N (in the last tile) hold code 0, scale 0 and minimum 0.
 *
 * w4a16_prepared_bytes -- bytes of the prepared copy: ceil(N / 128) * (K / 128) * 8704
 *   (0 for unsupported arguments: group != 128, K % 128 != 0).
 */
size_t w4a16_prepared_bytes(int N, int K, int group);

/*
 * w4a16_prepare -- writes the prepared copy of packed weights (one kernel, asynchronous).
 *   qw int32 [K/8, N], scales / mins bf16 [K/group, N] (as for w4a16_matmul)
 *   prepared: caller-owned device buffer of at least w4a16_prepared_bytes(N, K, group)
 *   bytes, 16-byte aligned, not overlapping the inputs.
 * Returns W4A16_ERR_INVALID_ARG if prepared_bytes is too small. Requires N > 0, K > 0,
 * group == 128, K % group == 0.
 */
w4a16_status w4a16_prepare(const int32_t* qw, const uint16_t* scales, const uint16_t* mins,
                           int N, int K, int group, void* prepared, size_t prepared_bytes,
                           w4a16_stream_t stream);

/*
 * w4a16_matmul_prepared -- y = x . W_hat^T as w4a16_matmul, with the prepared copy of the
 * same weights at hand. For 32 <= M <= 128 (by default) it runs the persistent tensor-core
 * kernel that reads `prepared` (TMA + tcgen05, rebuilt weights in tensor memory, fp32
 * sums); for other M, or with prepared == NULL, it is exactly w4a16_matmul on (qw, scales,
 * mins). Same tolerance and determinism as w4a16_matmul.
 *   x bf16 [M, K]; qw, scales, mins as for w4a16_matmul; prepared from w4a16_prepare on the
 *   same weights; y bf16 [M, N].
 *   workspace / workspace_bytes: optional caller-owned device scratch sized with
 *   w4a16_matmul_prepared_workspace_bytes(); for shapes with fewer 128-column tiles than half
 *   the SMs it lets the kernel split K evenly over the SMs (per-tile arrival counters and fp32
 *   partial tiles). Zero-fill it before its first use and do not share it with calls that may
 *   run concurrently or with other entry points. NULL (with 0 bytes) is accepted: the kernel
 *   then gives each CTA whole tiles.
 * Requires M > 0, N > 0, K > 0, group == 128, K % group == 0, N % 8 == 0.
 */
w4a16_status w4a16_matmul_prepared(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                                   const uint16_t* mins, const void* prepared, uint16_t* y,
                                   int M, int N, int K, int group, void* workspace,
                                   size_t workspace_bytes, w4a16_stream_t stream);

/* Bytes of workspace that let w4a16_matmul_prepared balance this shape (0 = none needed). */
size_t w4a16_matmul_prepared_workspace_bytes(int M, int N, int K, int group);

/*
 * Zero-point format ("Quantization and GEMV", "The quantization formulas" and "W4A16:
 * dequantizing in registers"): w_hat = (q - z) * s with one FP16 scale s and one FP16
 * zero point z per group of 128 weights along K (4.25 bits per weight).
 *
 * w4a16zp_quantize -- fp32 weights to codes, scales and zero points in the layout that
 * page stores them in.
 *   w       fp32 [N, K]
 *   qw_rows uint32 [N, K/8]    word (n, r) holds k = 8r + j in bits 4j..4j+3
 *   scales  fp16 [N, K/group]  s = fp16_rne(fp32(max - min) / 15); 1 if that is 0
 *   zeros   fp16 [N, K/group]  z = fp16_rne(round(fp32(-min / s)))
 * Per weight: q = clamp(round(fp32(w / s)) + z, 0, 15), round() half away from zero (the
 * page's host code uses std::round), s and z as stored. A group whose zero point is beyond
 * FP16's range (all weights far from zero next to their spread) is outside the format.
 * Requires N > 0, K > 0, group == 128, K % group == 0.
 */
w4a16_status w4a16zp_quantize(const float* w, int N, int K, int group, uint32_t* qw_rows,
                              uint16_t* scales, uint16_t* zeros, w4a16_stream_t stream);

/*
 * w4a16zp_prepare -- the same numbers in the matmul's layout (a transpose of each array):
 *   qw_rows [N, K/8], scales [N, K/group], zeros [N, K/group]  (as above)
 *   -> qw int32 [K/8, N], scales_t fp16 [K/group, N], zeros_t fp16 [K/group, N]
 * Inputs and outputs must not overlap. Requires N > 0, K > 0, group == 128,
 * K % group == 0.
 */
w4a16_status w4a16zp_prepare(const uint32_t* qw_rows, const uint16_t* scales,
                             const uint16_t* zeros, int N, int K, int group, int32_t* qw,
                             uint16_t* scales_t, uint16_t* zeros_t, w4a16_stream_t stream);

/*
 * w4a16zp_matmul -- y = x . W_hat^T with w_hat[n, k] = (q - z) * s: the same kernels,
 * kernel choice, workspace rules (w4a16_matmul_workspace_bytes), tolerance and
 * determinism as w4a16_matmul. In the fold -s z stands for the minimum; it is exact in
 * fp32 (two 11-bit significands).
 *   x bf16 [M, K]; qw int32 [K/8, N]; scales, zeros fp16 [K/group, N] (w4a16zp_prepare);
 *   y bf16 [M, N]
 * Requires M > 0, N > 0, K > 0, group == 128, K % group == 0, N % 8 == 0.
 */
w4a16_status w4a16zp_matmul(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                            const uint16_t* zeros, uint16_t* y, int M, int N, int K, int group,
                            void* workspace, size_t workspace_bytes, w4a16_stream_t stream);

/*
 * w4a16_matmul_noalloc -- the same product as w4a16_matmul for callers that cannot
 * allocate device memory or lend the library a buffer (for example a plugin inside a
 * runtime that owns all device memory, or a loop that must not pay for an allocation).
 * The pages have no counterpart: it exists only for such callers.
 *   Arguments as for w4a16_matmul, without a workspace. It always runs the tensor-core
 *   kernel; when that kernel splits K, its scratch is a 16 MiB array compiled into the
 *   library (held on every device that loads the library until the process exits).
 *   Returns W4A16_ERR_WORKSPACE, launching nothing, for a shape whose split needs more
 *   than 16 MiB of scratch.
 *   All calls on a device share that array: calls whose kernels may overlap on the GPU
 *   race, so order them (one stream, or events). Each call clears the counters it uses
 *   first. The first call on a device looks up the array's device address and caches it
 *   for the life of the process; make it before any stream capture, and do not reset the
 *   device afterwards.
 */
w4a16_status w4a16_matmul_noalloc(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                                  const uint16_t* mins, uint16_t* y, int M, int N, int K,
                                  int group, w4a16_stream_t stream);

/*
 * q4b32_quantize -- fp32 weights to Q4 blocks of 32 ("Why My 4-Bit CUDA Kernel Wasn't
 * Faster": an 18-byte block, 32 codes in 16 bytes and one 2-byte scale for all 32).
 *   w      fp32 [N, K]
 *   codes  uint8 [N, K/2]  byte j of block b holds weight 32b+2j in its low nibble
 *                          and weight 32b+2j+1 in its high nibble
 *   scales fp16 [N, K/32]  s = fp16_rne(fp32(max|w| / 8))
 * Per weight: q = clamp(rint(w / s) + 8, 0, 15) (round-half-to-even); a block whose
 * FP16 scale is 0 stores q = 8. Requires N > 0, K > 0, K % 32 == 0.
 */
w4a16_status q4b32_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales,
                            w4a16_stream_t stream);

/*
 * q4b32_gemv -- y[n] = sum_b s[n, b] * sum_j (q[n, b, j] - 8) * x[32 b + j]
 * ("Why My 4-Bit CUDA Kernel Wasn't Faster": a weight is rebuilt as its code minus
 * the bias, times the block's scale; codes and scales in separate arrays).
 *   x fp16 [K]; codes uint8 [N, K/2]; scales fp16 [N, K/32]; y fp16 [N]
 * fp32 accumulation, y rounded to nearest even; the same tolerance as w4a16_matmul.
 * Requires N > 0, K > 0, K % 32 == 0.
 */
w4a16_status q4b32_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                        uint16_t* y, int N, int K, w4a16_stream_t stream);

/*
 * W8A16 ("Quantization and GEMV", exercise 1): symmetric per-row INT8 weights,
 * w_hat = q * s, one fp32 scale per row (8 bits per weight plus 4 bytes per row).
 *
 * w8a16_quantize -- w fp32 [N, K] -> q int8 [N, K], scales fp32 [N]:
 *   s = fl(max_k |w[n, k]| / 127); q = clamp(round(fl(w / s)), -127, 127) with round()
 *   half away from zero (the page's host code uses std::round); a row of zeros stores
 *   s = 0 and q = 0. Requires N > 0, K > 0, K % 64 == 0.
 */
w4a16_status w8a16_quantize(const float* w, int N, int K, int8_t* q, float* scales,
                            w4a16_stream_t stream);

/*
 * w8a16_gemv -- y[n] = s[n] * sum_k q[n, k] x[k] (the scale once per row, after the sum).
 *   x bf16 [K]; q int8 [N, K]; scales fp32 [N]; y bf16 [N] (fp32 accumulation, rounded to
 *   nearest even). The tolerance of w4a16_matmul applies. x is held in shared memory in
 *   FP16: for K % 512 == 0 (the tensor-pipe kernel) under one power of two for the vector,
 *   K up to about 100,000; for other K under a power of two per 64 k, K up to about
 *   110,000 (W4A16_ERR_UNSUPPORTED beyond). Requires N > 0, K > 0, K % 64 == 0.
 */
w4a16_status w8a16_gemv(const uint16_t* x, const int8_t* q, const float* scales, uint16_t* y,
                        int N, int K, w4a16_stream_t stream);

/*
 * NVFP4 weights with 16-bit activations ("Hardware-invariant NVFP4 progress report 1", "The
 * NVFP4 layout"; "Low-Precision Kernels ...", Step 6): E2M1 codes (values 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6 and their negatives), one E4M3 scale per 16 weights along K and one fp32 scale
 * per tensor; w_hat = e2m1(q) * e4m3(s_b) * S (4.5 bits per weight).
 *
 * nvfp4_quantize -- w fp32 [N, K] -> codes uint8 [N, K/2] (byte j of a row: k = 2j in the
 *   low nibble, 2j + 1 in the high one), scales E4M3 bytes [N, K/16], tensor_scale one fp32:
 *   S = fl(amax / 2688) (1 for an all-zero tensor); a block's scale is the smallest E4M3
 *   value >= fl(amax_b / fl(6 S)) (at most 448), so that the block's largest weight is not
 *   clipped; codes are fl(w / fl(s_b S)) rounded to the nearest E2M1 value, ties to the even
 *   code, saturating at 6; a block of zeros stores scale 0 and codes 0. Four launches on
 *   `stream` (the tensor_scale word holds amax in between). Requires N > 0, K > 0,
 *   K % 128 == 0.
 */
w4a16_status nvfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                            float* tensor_scale, w4a16_stream_t stream);

/*
 * nvfp4_gemv -- y[n] = S * sum_b e4m3(s[n, b]) * sum_j e2m1(q[n, 16 b + j]) x[16 b + j]:
 *   x bf16 [K]; codes, scales, tensor_scale as above (device memory); y bf16 [N] (fp32
 *   accumulation, rounded to nearest even). The tolerance of w4a16_matmul applies. For
 *   K % 512 == 0 up to 92,160 the tensor-pipe kernel runs: x is held in shared memory in
 *   FP16 under a power of two per 32-k block (its largest magnitude in [2^14, 2^15)), so
 *   elements more than 29 binades below their block's largest lose bits (their terms lie
 *   far below the tolerance). Other K take a kernel with x in FP16 per 128-k chunk: K up to
 *   about 110,000 (W4A16_ERR_UNSUPPORTED beyond). Requires N > 0, K > 0, K % 128 == 0.
 */
w4a16_status nvfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                        const float* tensor_scale, uint16_t* y, int N, int K,
                        w4a16_stream_t stream);

/*
 * MXFP4 weights with 16-bit activations ("Low-Precision Kernels ...", Step 6, the OCP MX
 * blocks): E2M1 codes, one E8M0 scale (2^(code - 127)) per 32 weights along K; w_hat =
 * e2m1(q) * 2^(s_b - 127) (4.25 bits per weight).
 *
 * mxfp4_quantize -- w fp32 [N, K] -> codes uint8 [N, K/2] (as NVFP4), scales E8M0 bytes
 *   [N, K/32]: the scale is the largest power of two <= max|w| of the block, divided by 4
 *   (the largest power of two E2M1 holds), exponent in [-127, 127]; codes are w / scale
 *   rounded to the nearest E2M1 value, ties to the even code, values past 6 clamped to 6; a
 *   block of zeros stores scale code 0 and codes 0. Requires N > 0, K > 0, K % 32 == 0.
 */
w4a16_status mxfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                            w4a16_stream_t stream);

/*
 * mxfp4_gemv -- y[n] = sum_b 2^(s[n, b] - 127) * sum_j e2m1(q[n, 32 b + j]) x[32 b + j]:
 *   x bf16 [K]; codes, scales as above; y bf16 [N] (fp32 accumulation, rounded to nearest
 *   even). The tolerance of w4a16_matmul applies. For K % 512 == 0 up to 102,912 the
 *   tensor-pipe kernel runs (x in FP16 under a power of two per 32-k block, each block's sum
 *   times its scale in fp32); other K take a kernel in which, within a 128-k chunk of a row,
 *   a block more than 2^24 below the chunk's largest block scale adds nothing (its terms are
 *   below the tolerance): K up to about 110,000 (W4A16_ERR_UNSUPPORTED beyond). Requires
 *   N > 0, K > 0, K % 128 == 0.
 */
w4a16_status mxfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                        uint16_t* y, int N, int K, w4a16_stream_t stream);

/*
 * nvfp4_matmul / mxfp4_matmul -- Y[m, n] = sum_k x[m, k] w_hat[n, k] for a batch of M rows
 *   (the formats above; "Low-Precision Kernels ...", Step 6, and "Step 3: measured from 1
 *   row to 4,096" for the batch). x bf16 [M, K] row-major; codes, scales (and tensor_scale
 *   for NVFP4) as for the GEMVs; y bf16 [M, N] row-major. M = 1 runs the GEMV and needs no
 *   workspace. For M > 1, a first kernel writes each row of x into `workspace` in FP16
 *   under the row's power of two (largest magnitude in [2^14, 2^15)) in the order the MMAs
 *   read it, and a second kernel streams the weights once per 32 rows of x, decoding each
 *   weight fragment once for those rows (for M > 32 the weights stream again for every
 *   further 32 rows). The tolerance of w4a16_matmul applies per output. Workspace: at least
 *   fp4_matmul_workspace_bytes(M, K) bytes of device memory, 16-byte aligned, owned by the
 *   caller and not touched by other work while the call runs on `stream`; too small or
 *   NULL for M > 1 gives W4A16_ERR_WORKSPACE, launching nothing. Requires M > 0, N > 0,
 *   K > 0, K % 512 == 0 for M > 1 (K % 128 == 0 for M = 1); W4A16_ERR_UNSUPPORTED when the
 *   shape's ring does not fit in shared memory (K beyond about 100,000 at the widest tiles).
 */
size_t fp4_matmul_workspace_bytes(int M, int K);
w4a16_status nvfp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                          const float* tensor_scale, uint16_t* y, int M, int N, int K,
                          void* workspace, size_t workspace_bytes, w4a16_stream_t stream);
w4a16_status mxfp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                          uint16_t* y, int M, int N, int K, void* workspace,
                          size_t workspace_bytes, w4a16_stream_t stream);

/*
 * w4a16_device_status -- synchronizes `stream`, then reads and clears the current
 * device's status word. Returns W4A16_ERR_TIMEOUT if any kernel of this library gave
 * up a bounded wait since the last query, W4A16_ERR_LAYOUT if a kernel found its
 * dynamic shared memory less than 128-byte aligned and skipped its work (its output is
 * then not written), W4A16_ERR_CUDA if the synchronization failed, W4A16_OK otherwise.
 * (The pages have no counterpart; this is the library's failure-detection hook.)
 */
w4a16_status w4a16_device_status(w4a16_stream_t stream);

/*
 * w4a16_selftest_bounded_wait -- launches one tiny kernel that waits on a shared-memory
 * barrier nothing ever arrives at, with the same bounded-wait helper the tensor-core
 * kernel uses, limited to `limit_us` microseconds (1..1000000). The kernel then
 * records the expiry in the status word and returns, so a correct build makes the
 * following w4a16_device_status() return W4A16_ERR_TIMEOUT. It holds no tensor
 * memory and issues no copies. (No counterpart on the pages: a failure-detection
 * test hook.)
 */
w4a16_status w4a16_selftest_bounded_wait(uint32_t limit_us, w4a16_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_GB300_H */
