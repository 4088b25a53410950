// Offline weight preparation on the GPU: group-128 asymmetric 4-bit quantization, packing
// eight codes per int32 along K, the zero-point variant and its move into the matmul's
// layout, and Q4 block-32 quantization.
//
// W4A16 format ("Low-Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", Step 2):
// a group is 128 neighbouring weights along K with scale (max - min) / 15 and its
// minimum, both kept in BF16; a weight's code is round((w - min) / scale), 0..15; words of
// eight codes along K form a K/8 x N matrix.
// Q4 format ("Why My 4-Bit CUDA Kernel Wasn't Faster"): 32 weights share one FP16
// scale; the 32 codes fill 16 bytes, low nibble = even weight, decode (q - 8) * s.
//
// Every step is an IEEE fp32 operation rounded to nearest even (__fsub_rn, __fdiv_rn,
// rintf, __float2bfloat16_rn, __float2half_rn), so the GPU result is bit-identical to a
// scalar fp32 reference taking the same steps. All three kernels are bound by HBM.
#include "common.cuh"
#include "launch.h"

namespace w4k {

// rint(fl(d / s)), the code rule of both quantizers (fp32 quotient, rounded to nearest
// even), with one multiply instead of a correctly rounded division per weight. rs = fl(1/s).
// t = fl(d rs) has relative error at most 2^-23, and fl(d / s) is within half an ulp of d / s,
// so for |d / s| <= 16 the two lie within 2^-19 + 2^-20 < 2^-17 of each other: rounding t to
// an integer gives the same result unless t is within 2^-17 of a half-integer (|t - rint(t)|
// above 1/2 - 2^-17), and there the quotient is computed exactly (this also catches every
// exact tie). Past 16 both clamp to the same end code; the exact fallback is always right.
__device__ __forceinline__ float rint_quotient(float d, float s, float rs) {
  const float t = __fmul_rn(d, rs);
  const float r = rintf(t);
  if (fabsf(__fsub_rn(t, r)) > 0.5f - 0x1p-17f) return rintf(__fdiv_rn(d, s));
  return r;
}

// Both group-128 quantizers stage a piece of a weight row (up to kQPiece floats, whole
// groups) in shared memory with one bulk copy, so that every resident CTA has its whole piece
// in flight at once (with the weights staged in registers, 80 KB per SM were in flight and the
// quantizer ran at 0.58 of HBM; a 4096-float row per 128-thread CTA puts 13 rows, 208 KB, in
// flight per SM). Warp w then takes groups w, w + 4, ... of the piece, 4 consecutive weights
// per lane.
constexpr int kQPiece = 8192;
constexpr int kQThreads = 128;
constexpr int kQWarps = kQThreads / 32;

// Copies `bytes` (a multiple of 16) from `src` into `dst` and waits for them (bounded). After
// an expired wait the CTA has waited once more (bounded) for its copy and must return.
__device__ __forceinline__ bool stage_piece(float* dst, const float* src, uint32_t bytes,
                                            uint64_t* bar, volatile uint32_t* abort_flag,
                                            uint32_t* status, uint64_t limit_ns) {
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(dst, src, bytes, bar);
  }
  if (mbar_wait_bounded(bar, 0u, abort_flag, status, limit_ns)) return true;
  if (threadIdx.x == 0) {
    volatile uint32_t no_abort = 0u;
    mbar_wait_bounded(bar, 0u, &no_abort, status, limit_ns);
  }
  return false;
}

__device__ __forceinline__ float4 lds128f(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

// Dynamic shared memory of a quantizer CTA: one piece.
inline size_t piece_bytes(int K) { return static_cast<size_t>(K < kQPiece ? K : kQPiece) * 4u; }

// CTA b: row b / pieces, piece b % pieces of kQPiece floats.
__global__ void __launch_bounds__(kQThreads)
w4a16_quantize_kernel(const float* __restrict__ w, int N, int K, uint8_t* __restrict__ codes,
                      uint16_t* __restrict__ scales, uint16_t* __restrict__ mins,
                      uint32_t* __restrict__ status, uint64_t limit_ns) {
  extern __shared__ __align__(128) float piece[];  // min(K, kQPiece) floats
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  const int pieces = (K + kQPiece - 1) / kQPiece;
  const int n = static_cast<int>(blockIdx.x / pieces), p = static_cast<int>(blockIdx.x % pieces);
  const int k0 = p * kQPiece, cnt = min(kQPiece, K - k0);
  if (!stage_piece(piece, w + static_cast<size_t>(n) * K + k0, static_cast<uint32_t>(cnt) * 4u,
                   &bar, &abort_flag, status, limit_ns))
    return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int gl = warp; gl < (cnt >> 7); gl += kQWarps) {  // warp-uniform
    const float4 v = lds128f(piece + gl * 128 + lane * 4);
    const int g = (k0 >> 7) + gl;
    float lo = fminf(fminf(v.x, v.y), fminf(v.z, v.w));
    float hi = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    const __nv_bfloat16 s_b = __float2bfloat16_rn(s32);
    const __nv_bfloat16 m_b = __float2bfloat16_rn(lo);
    const float s = __bfloat162float(s_b);
    const float m = __bfloat162float(m_b);
    const float rs = s != 0.0f ? __frcp_rn(s) : 0.0f;
    auto code = [&](float x) -> uint32_t {
      if (s == 0.0f) return 0u;
      const float d = __fsub_rn(x, m);
      return static_cast<uint32_t>(fminf(fmaxf(rint_quotient(d, s, rs), 0.0f), 15.0f));
    };
    const uint32_t packed = code(v.x) | (code(v.y) << 8) | (code(v.z) << 16) | (code(v.w) << 24);
    *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(n) * K +
                                 static_cast<size_t>(g) * 128 + lane * 4) = packed;
    if (lane == 0) {
      scales[static_cast<size_t>(g) * N + n] = __bfloat16_as_ushort(s_b);
      mins[static_cast<size_t>(g) * N + n] = __bfloat16_as_ushort(m_b);
    }
  }
}

// round(fl(d / s)) with ties away from zero (std::round, the rounding of the zero-point
// format's host code), by the same argument as rint_quotient: for |t| < 32, t = fl(d rs) lies
// within 3 * 33 * 2^-24 < 2^-17 of fl(d / s), so both round to the same integer unless t is
// within 2^-17 of a half-integer; there, and for larger quotients, the quotient is exact.
__device__ __forceinline__ float round_quotient_away(float d, float s, float rs) {
  const float t = __fmul_rn(d, rs);
  const float r = rintf(t);
  if (fabsf(t) < 32.0f && fabsf(__fsub_rn(t, r)) <= 0.5f - 0x1p-17f) return r;
  return roundf(__fdiv_rn(d, s));
}

// Zero-point W4A16 ("Quantization and GEMV", "The quantization formulas"): per group of 128
// weights of a row, s = fp16((max - min) / 15) (1 when that is 0), z = fp16(round(-min / s)),
// q = clamp(round(w / s) + z, 0, 15), in the layout the page stores: words [N, K/8] (first
// weight in the lowest nibble), scales and zeros [N, K/128]. Same staging and split as the
// minimum-form quantizer; lanes 2i and 2i + 1 hold the 8 weights of word i of a group.
__global__ void __launch_bounds__(kQThreads)
w4a16zp_quantize_kernel(const float* __restrict__ w, int N, int K, uint32_t* __restrict__ qw_rows,
                        uint16_t* __restrict__ scales, uint16_t* __restrict__ zeros,
                        uint32_t* __restrict__ status, uint64_t limit_ns) {
  extern __shared__ __align__(128) float piece[];  // min(K, kQPiece) floats
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  const int groups = K >> 7;
  const int pieces = (K + kQPiece - 1) / kQPiece;
  const int n = static_cast<int>(blockIdx.x / pieces), p = static_cast<int>(blockIdx.x % pieces);
  const int k0 = p * kQPiece, cnt = min(kQPiece, K - k0);
  if (!stage_piece(piece, w + static_cast<size_t>(n) * K + k0, static_cast<uint32_t>(cnt) * 4u,
                   &bar, &abort_flag, status, limit_ns))
    return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int gl = warp; gl < (cnt >> 7); gl += kQWarps) {  // warp-uniform
    const float4 v = lds128f(piece + gl * 128 + lane * 4);
    const int g = (k0 >> 7) + gl;
    float lo = fminf(fminf(v.x, v.y), fminf(v.z, v.w));
    float hi = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    __half s_h = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
    if (__half2float(s_h) == 0.0f) s_h = __float2half_rn(1.0f);
    const float s = __half2float(s_h);
    const __half z_h = __float2half_rn(roundf(__fdiv_rn(-lo, s)));
    const float z = __half2float(z_h);
    const float rs = __frcp_rn(s);
    auto code = [&](float x) -> uint32_t {
      const float q = round_quotient_away(x, s, rs) + z;  // integers: exact
      return static_cast<uint32_t>(fminf(fmaxf(q, 0.0f), 15.0f));
    };
    const uint32_t nib = code(v.x) | (code(v.y) << 4) | (code(v.z) << 8) | (code(v.w) << 12);
    const uint32_t upper = __shfl_down_sync(0xffffffffu, nib, 1);
    if ((lane & 1) == 0)
      qw_rows[static_cast<size_t>(n) * (K >> 3) + static_cast<size_t>(g) * 16 + (lane >> 1)] =
          nib | (upper << 16);
    if (lane == 0) {
      scales[static_cast<size_t>(n) * groups + g] = __half_as_ushort(s_h);
      zeros[static_cast<size_t>(n) * groups + g] = __half_as_ushort(z_h);
    }
  }
}

// Transpose of a rows x cols matrix of T (4 or 2 bytes) into cols x rows, 64 x 64 tiles
// through shared memory so that reads and writes are both coalesced. Prepares the
// zero-point format's [N, K/8] words and [N, K/128] scales and zeros for the matmul,
// which reads [K/8, N] and [K/128, N].
template <typename T>
__global__ void __launch_bounds__(256)
transpose_kernel(const T* __restrict__ in, int rows, int cols, T* __restrict__ out) {
  __shared__ T tile[64][65];
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int rl = (tid >> 6) + 4 * i, cl = tid & 63;
    if (r0 + rl < rows && c0 + cl < cols)
      tile[rl][cl] = in[static_cast<size_t>(r0 + rl) * cols + c0 + cl];
  }
  __syncthreads();
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int cl = (tid >> 6) + 4 * i, rl = tid & 63;
    if (r0 + rl < rows && c0 + cl < cols)
      out[static_cast<size_t>(c0 + cl) * rows + r0 + rl] = tile[rl][cl];
  }
}

// Pack: tile of 64 rows (n) x 64 words (r) through shared memory so that both the
// byte reads along K and the word writes along N are coalesced.
__global__ void __launch_bounds__(256)
w4a16_pack_kernel(const uint8_t* __restrict__ codes, int N, int K, uint32_t* __restrict__ qw) {
  __shared__ uint32_t tile[64][65];
  const int R = K >> 3;
  const int n0 = blockIdx.y * 64, r0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
  {
    const int rl = tid & 63;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int nl = (tid >> 6) + 4 * i;
      const int n = n0 + nl, r = r0 + rl;
      uint32_t word = 0;
      if (n < N && r < R) {
        const uint2 b = *reinterpret_cast<const uint2*>(codes + static_cast<size_t>(n) * K + 8 * r);
        // byte j of the 8 holds code k = 8r + j; nibble j of the word
        const uint32_t lo = b.x & 0x0F0F0F0Fu, hi = b.y & 0x0F0F0F0Fu;
        // spread: codes 0..3 from lo bytes, 4..7 from hi bytes
        word = (lo & 0xFu) | ((lo >> 4) & 0xF0u) | ((lo >> 8) & 0xF00u) | ((lo >> 12) & 0xF000u) |
               ((hi & 0xFu) << 16) | ((hi << 12) & 0xF00000u) | ((hi << 8) & 0xF000000u) |
               ((hi << 4) & 0xF0000000u);
      }
      tile[rl][nl] = word;
    }
  }
  __syncthreads();
  {
    const int nl = tid & 63;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int rl = (tid >> 6) + 4 * i;
      const int n = n0 + nl, r = r0 + rl;
      if (n < N && r < R) qw[static_cast<size_t>(r) * N + n] = tile[rl][nl];
    }
  }
}

// Q4: a warp takes 512 consecutive weights as four slots of 128 (8 lanes per block of 32,
// 4 weights per lane in each slot); the four loads of a lane are issued before any is used.
__global__ void __launch_bounds__(256)
q4b32_quantize_kernel(const float* __restrict__ w, int N, int K, uint8_t* __restrict__ codes,
                      uint16_t* __restrict__ scales) {
  const long long total = static_cast<long long>(N) * K;  // weights
  const long long base = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * 512;
  const int lane = threadIdx.x & 31;
  float4 v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const long long e = base + j * 128 + lane * 4;  // blocks of 32 never straddle rows
    v[j] = e < total ? __ldcs(reinterpret_cast<const float4*>(w + e)) : make_float4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const long long e = base + j * 128 + lane * 4;
    float a = fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const __half s_h = __float2half_rn(__fdiv_rn(a, 8.0f));
    const float s = __half2float(s_h);
    const float rs = s != 0.0f ? __frcp_rn(s) : 0.0f;
    auto code = [&](float x) -> uint32_t {
      if (s == 0.0f) return 8u;
      const float r = rint_quotient(x, s, rs) + 8.0f;
      return static_cast<uint32_t>(fminf(fmaxf(r, 0.0f), 15.0f));
    };
    if (e >= total) continue;
    const uint32_t b0 = code(v[j].x) | (code(v[j].y) << 4);
    const uint32_t b1 = code(v[j].z) | (code(v[j].w) << 4);
    *reinterpret_cast<uint16_t*>(codes + e / 2) = static_cast<uint16_t>(b0 | (b1 << 8));
    if ((lane & 7) == 0) scales[e / 32] = __half_as_ushort(s_h);
  }
}

cudaError_t launch_w4a16_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales,
                                  uint16_t* mins, uint32_t* status, uint64_t limit_ns,
                                  cudaStream_t stream) {
  const long long blocks = static_cast<long long>(N) * ((K + kQPiece - 1) / kQPiece);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  w4a16_quantize_kernel<<<static_cast<unsigned>(blocks), kQThreads, piece_bytes(K), stream>>>(
      w, N, K, codes, scales, mins, status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_w4a16_pack(const uint8_t* codes, int N, int K, uint32_t* qw,
                              cudaStream_t stream) {
  const int R = K >> 3;
  dim3 grid((R + 63) / 64, (N + 63) / 64);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  w4a16_pack_kernel<<<grid, 256, 0, stream>>>(codes, N, K, qw);
  return cudaGetLastError();
}

cudaError_t launch_w4a16zp_quantize(const float* w, int N, int K, uint32_t* qw_rows,
                                    uint16_t* scales, uint16_t* zeros, uint32_t* status,
                                    uint64_t limit_ns, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(N) * ((K + kQPiece - 1) / kQPiece);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  w4a16zp_quantize_kernel<<<static_cast<unsigned>(blocks), kQThreads, piece_bytes(K), stream>>>(
      w, N, K, qw_rows, scales, zeros, status, limit_ns);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_transpose(const T* in, int rows, int cols, T* out, cudaStream_t stream) {
  const dim3 grid((cols + 63) / 64, (rows + 63) / 64);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  transpose_kernel<T><<<grid, 256, 0, stream>>>(in, rows, cols, out);
  return cudaGetLastError();
}

cudaError_t launch_w4a16zp_prepare(const uint32_t* qw_rows, const uint16_t* scales,
                                   const uint16_t* zeros, int N, int K, uint32_t* qw,
                                   uint16_t* scales_t, uint16_t* zeros_t, cudaStream_t stream) {
  cudaError_t e = launch_transpose<uint32_t>(qw_rows, N, K >> 3, qw, stream);
  if (e != cudaSuccess) return e;
  e = launch_transpose<uint16_t>(scales, N, K >> 7, scales_t, stream);
  if (e != cudaSuccess) return e;
  return launch_transpose<uint16_t>(zeros, N, K >> 7, zeros_t, stream);
}

cudaError_t launch_q4b32_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales,
                                  cudaStream_t stream) {
  const long long total = static_cast<long long>(N) * K;  // weights, 512 per warp
  const long long blocks = (total + 8 * 512 - 1) / (8 * 512);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  q4b32_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, N, K, codes, scales);
  return cudaGetLastError();
}

}  // namespace w4k
