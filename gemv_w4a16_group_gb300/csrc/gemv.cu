// CUDA-core W4A16 GEMV for small M: y[m, n] = sum_g ( s[g,n] * sum_{k in g} x[m,k] q[n,k]
//                                                     + min[g,n] * sum_{k in g} x[m,k] ).
//
// The factorised per-group form is the one the pages give for their M = 1 kernel ("Low-
// Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", "How the measurements were
// taken": a GEMV that "sums s x sum x.q + min x sum x per group in FP32 without tensor
// cores"). The launch shape follows "Quantization and GEMV", "Writing a GEMV kernel"
// (128-bit coalesced loads, K split across the block, warp-shuffle reduction), adapted
// to the K/8 x N packed layout in which N is contiguous:
//
//   * a CTA owns 32 output columns and the whole of K; 8 lanes x 4 columns read one
//     128-byte line of a packed row, so a warp instruction reads 4 full lines;
//   * warp w owns a contiguous range of groups; lane (rs, cq) reads rows
//     16g + 4rs + t (t = 0..3) of each group, i.e. a contiguous quarter of the group;
//   * codes become exact floats with an offset (mantissa trick, see common.cuh); the
//     offsets and the min term are removed per quarter-group with sums of x that the
//     CTA computes once in its prologue, while the first weight loads are in flight;
//   * partial sums are reduced over the 4 row-phases with shuffles and over the 8 warps
//     through shared memory in a fixed order (deterministic, no atomics).
//
// HBM-bound in principle; at 4 bits the dequantisation is a real share of the issue
// slots ("Where the time goes at M = 1"), hence the two inner-product variants:
//   VARIANT 0: codes -> fp32 (one LOP3 each) and packed fp32x2 FMA;
//   VARIANT 1: codes -> BF16 pairs (one LOP3 per pair) and mixed BF16xBF16->fp32 FMA.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kColsPerCta = 32;
constexpr int kMaxRows = 8;

__device__ __forceinline__ uint4 ld_weights(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc += sum_j (offset_j + q_j) * x_j for the 8 codes of `w` (VARIANT 1).
// p_i = (128 + q_i, 128 + q_{i+4}) as BF16; x01 = (x0, x1), ..., x67 = (x6, x7).
__device__ __forceinline__ float dot8_mixed_bf16(uint32_t w, uint32_t x01, uint32_t x23,
                                                 uint32_t x45, uint32_t x67, float acc) {
  const uint32_t p0 = (w & 0x000F000Fu) | 0x43004300u;
  const uint32_t p1 = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
  const uint32_t p2 = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
  const uint32_t p3 = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
  asm("{\n\t"
      ".reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b32 {a2, a3}, %2;\n\t"
      "mov.b32 {a4, a5}, %3;\n\tmov.b32 {a6, a7}, %4;\n\t"
      "mov.b32 {b0, b1}, %5;\n\tmov.b32 {b2, b3}, %6;\n\t"
      "mov.b32 {b4, b5}, %7;\n\tmov.b32 {b6, b7}, %8;\n\t"
      "fma.rn.f32.bf16 %0, a0, b0, %0;\n\t"  // q0 x0
      "fma.rn.f32.bf16 %0, a2, b1, %0;\n\t"  // q1 x1
      "fma.rn.f32.bf16 %0, a4, b2, %0;\n\t"  // q2 x2
      "fma.rn.f32.bf16 %0, a6, b3, %0;\n\t"  // q3 x3
      "fma.rn.f32.bf16 %0, a1, b4, %0;\n\t"  // q4 x4
      "fma.rn.f32.bf16 %0, a3, b5, %0;\n\t"  // q5 x5
      "fma.rn.f32.bf16 %0, a5, b6, %0;\n\t"  // q6 x6
      "fma.rn.f32.bf16 %0, a7, b7, %0;\n\t"  // q7 x7
      "}"
      : "+f"(acc)
      : "r"(p0), "r"(p1), "r"(p2), "r"(p3), "r"(x01), "r"(x23), "r"(x45), "r"(x67));
  return acc;
}

template <int MR, int VARIANT>
__global__ void __launch_bounds__(kThreads)
    gemv_w4a16_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ qw,
                      const uint16_t* __restrict__ scales, const uint16_t* __restrict__ mins,
                      uint16_t* __restrict__ y, int M, int N, int K) {
  extern __shared__ float smem[];
  const int Q = K >> 5;  // quarter-groups of 32 k
  float* sX = smem;                // [MR][Q] sum of x over the quarter
  float* sC = smem + MR * Q;       // [MR][Q] sum of offset_k * x_k over the quarter
  float* sRed = smem + 2 * MR * Q; // [kWarps][MR][32]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cq = lane & 7, rs = lane >> 3;
  const int n = blockIdx.x * kColsPerCta + cq * 4;  // first of this lane's 4 columns
  const bool col_ok = n < N;                         // N % 4 == 0: a quad is in or out
  const int m0 = blockIdx.y * MR;
  const int G = K >> 7;
  const int gpw = (G + kWarps - 1) / kWarps;
  const int g_begin = min(G, warp * gpw);
  const int g_end = min(G, g_begin + gpw);

  uint4 wa[4], wb[4];
  uint2 sa = make_uint2(0, 0), ma = make_uint2(0, 0), sb = make_uint2(0, 0), mb = make_uint2(0, 0);
  auto fetch = [&](int g, uint4(&wr)[4], uint2& s2, uint2& m2) {
    if (col_ok) {
      const uint32_t* p = qw + static_cast<size_t>(g * 16 + rs * 4) * N + n;
#pragma unroll
      for (int t = 0; t < 4; ++t) wr[t] = ld_weights(p + static_cast<size_t>(t) * N);
      s2 = __ldg(reinterpret_cast<const uint2*>(scales + static_cast<size_t>(g) * N + n));
      m2 = __ldg(reinterpret_cast<const uint2*>(mins + static_cast<size_t>(g) * N + n));
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t) wr[t] = make_uint4(0, 0, 0, 0);
    }
  };
  if (g_begin < g_end) fetch(g_begin, wa, sa, ma);

  // Prologue: per quarter-group sums of x and of offset-weighted x.
  for (int i = tid; i < MR * Q; i += kThreads) {
    const int mm = i / Q, q = i - mm * Q;
    float X = 0.f, C = 0.f;
    if (m0 + mm < M) {
      const uint4* xp = reinterpret_cast<const uint4*>(x + static_cast<size_t>(m0 + mm) * K + q * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 u = __ldg(xp + v);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float lo = bf16_bits_to_f32(wd[h] & 0xFFFFu);  // even k
          const float hi = __uint_as_float(wd[h] & 0xFFFF0000u);  // odd k
          X += lo + hi;
          if (VARIANT == 0) {
            C += code_offset_f32(0) * lo + code_offset_f32(1) * hi;
          } else {
            C += 128.0f * lo + 128.0f * hi;
          }
        }
      }
    }
    sX[i] = X;
    sC[i] = C;
  }
  __syncthreads();

  float yacc[4][MR];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int mm = 0; mm < MR; ++mm) yacc[c][mm] = 0.f;

  auto process = [&](int g, const uint4(&wr)[4], uint2 s2, uint2 m2) {
    float acc[4][MR];
    float acc_odd[4][MR];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int mm = 0; mm < MR; ++mm) acc[c][mm] = acc_odd[c][mm] = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int r = g * 16 + rs * 4 + t;
      const uint32_t wd[4] = {wr[t].x, wr[t].y, wr[t].z, wr[t].w};
      if (VARIANT == 0) {
        float f[4][8];
#pragma unroll
        for (int c = 0; c < 4; ++c) codes_to_f32_offset(wd[c], f[c]);
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) {
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (m0 + mm < M)
            xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m0 + mm) * K + 8 * r));
          const float2 x01 = make_float2(bf16_bits_to_f32(xv.x & 0xFFFFu), __uint_as_float(xv.x & 0xFFFF0000u));
          const float2 x23 = make_float2(bf16_bits_to_f32(xv.y & 0xFFFFu), __uint_as_float(xv.y & 0xFFFF0000u));
          const float2 x45 = make_float2(bf16_bits_to_f32(xv.z & 0xFFFFu), __uint_as_float(xv.z & 0xFFFF0000u));
          const float2 x67 = make_float2(bf16_bits_to_f32(xv.w & 0xFFFFu), __uint_as_float(xv.w & 0xFFFF0000u));
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float2 a = make_float2(acc[c][mm], acc_odd[c][mm]);
            a = __ffma2_rn(make_float2(f[c][0], f[c][1]), x01, a);
            a = __ffma2_rn(make_float2(f[c][2], f[c][3]), x23, a);
            a = __ffma2_rn(make_float2(f[c][4], f[c][5]), x45, a);
            a = __ffma2_rn(make_float2(f[c][6], f[c][7]), x67, a);
            acc[c][mm] = a.x;
            acc_odd[c][mm] = a.y;
          }
        }
      } else {
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) {
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (m0 + mm < M)
            xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m0 + mm) * K + 8 * r));
#pragma unroll
          for (int c = 0; c < 4; ++c)
            acc[c][mm] = dot8_mixed_bf16(wd[c], xv.x, xv.y, xv.z, xv.w, acc[c][mm]);
        }
      }
    }
    const int q = g * 4 + rs;
    const uint32_t sw[2] = {s2.x, s2.y}, mw[2] = {m2.x, m2.y};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t sbits = (c & 1) ? (sw[c >> 1] >> 16) : (sw[c >> 1] & 0xFFFFu);
      const uint32_t mbits = (c & 1) ? (mw[c >> 1] >> 16) : (mw[c >> 1] & 0xFFFFu);
      const float s = bf16_bits_to_f32(sbits), mn = bf16_bits_to_f32(mbits);
#pragma unroll
      for (int mm = 0; mm < MR; ++mm) {
        const float a = acc[c][mm] + acc_odd[c][mm];
        yacc[c][mm] = fmaf(s, a - sC[mm * Q + q], fmaf(mn, sX[mm * Q + q], yacc[c][mm]));
      }
    }
  };

  int g = g_begin;
  for (; g + 1 < g_end; g += 2) {
    fetch(g + 1, wb, sb, mb);
    process(g, wa, sa, ma);
    if (g + 2 < g_end) fetch(g + 2, wa, sa, ma);
    process(g + 1, wb, sb, mb);
  }
  if (g < g_end) process(g, wa, sa, ma);

  // Reduce over the 4 row phases (lanes cq, cq+8, cq+16, cq+24), then over warps.
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int mm = 0; mm < MR; ++mm) {
      float v = yacc[c][mm];
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      yacc[c][mm] = v;
    }
  if (rs == 0) {
#pragma unroll
    for (int mm = 0; mm < MR; ++mm)
#pragma unroll
      for (int c = 0; c < 4; ++c) sRed[(warp * MR + mm) * 32 + cq * 4 + c] = yacc[c][mm];
  }
  __syncthreads();
  for (int i = tid; i < MR * 32; i += kThreads) {
    const int mm = i >> 5, col = i & 31;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += sRed[(w * MR + mm) * 32 + col];
    const int nn = blockIdx.x * kColsPerCta + col;
    if (m0 + mm < M && nn < N)
      y[static_cast<size_t>(m0 + mm) * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

template <int MR, int VARIANT>
cudaError_t launch_mr(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                      const uint16_t* mins, uint16_t* y, int M, int N, int K, cudaStream_t stream) {
  const size_t smem = (2 * static_cast<size_t>(MR) * (K >> 5) + kWarps * MR * 32) * sizeof(float);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = gemv_w4a16_kernel<MR, VARIANT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid((N + kColsPerCta - 1) / kColsPerCta, (M + MR - 1) / MR);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  kern<<<grid, kThreads, smem, stream>>>(x, qw, scales, mins, y, M, N, K);
  return cudaGetLastError();
}

template <int VARIANT>
cudaError_t launch_variant(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                           const uint16_t* mins, uint16_t* y, int M, int N, int K,
                           cudaStream_t stream) {
  if (M <= 1) return launch_mr<1, VARIANT>(x, qw, scales, mins, y, M, N, K, stream);
  if (M <= 2) return launch_mr<2, VARIANT>(x, qw, scales, mins, y, M, N, K, stream);
  if (M <= 4) return launch_mr<4, VARIANT>(x, qw, scales, mins, y, M, N, K, stream);
  return launch_mr<8, VARIANT>(x, qw, scales, mins, y, M, N, K, stream);
}

}  // namespace

int gemv_max_rows() { return kMaxRows; }

cudaError_t launch_w4a16_gemv(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                              const uint16_t* mins, uint16_t* y, int M, int N, int K, int variant,
                              cudaStream_t stream) {
  if (variant == 1) return launch_variant<1>(x, qw, scales, mins, y, M, N, K, stream);
  return launch_variant<0>(x, qw, scales, mins, y, M, N, K, stream);
}

}  // namespace w4k
