// Q4 block-32 GEMV: y[n] = sum_b s[n,b] * sum_{j<32} (q[n,b,j] - 8) * x[32b + j].
//
// Format from "Why My 4-Bit CUDA Kernel Wasn't Faster" ("Why fewer bytes should have
// helped": 16 code bytes + a 2-byte FP16 scale per 32 weights; decode = code minus the
// bias, times the scale), with codes and scales in separate arrays ("Loading the same
// bytes differently": row_scales[...] and row_codes + block * 16). That page's lesson is
// that load count and width decide the speed (49 -> 18 -> 6 loads per block); here
// every lane reads a whole block's codes with one 16-byte load, a warp instruction
// reads 512 contiguous bytes of a row, and each x fetch is shared by 8 rows. The page's
// "what I'd try next" (split rows across warps, keep x close) is the launch shape:
//
//   * a CTA owns 8 rows and the whole of K; warp w owns a contiguous range of blocks;
//   * lane l takes blocks b = b_begin + l + 32 i of all 8 rows: 8 x 16-byte code loads
//     and one 64-byte x fetch (4 x 16 B) per block;
//   * the bias and the code offsets are removed per block with sum_j (B_j + 8) x_j,
//     computed once per block and shared by the 8 rows;
//   * warp-shuffle reduction, then a fixed-order sum over warps (deterministic).
//
// VARIANT 0: codes -> fp32 with offset (one LOP3 each) + packed fp32x2 FMA on fp32 x.
// VARIANT 1: codes -> FP16 pairs 1024 + q (one LOP3 per pair) + mixed FP16xFP16->fp32 FMA.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 8;

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc += sum_j (1024 + q_j) * x_j for the 8 codes of word w (FP16 halves).
__device__ __forceinline__ float dot8_mixed_f16(uint32_t w, uint32_t x01, uint32_t x23,
                                                uint32_t x45, uint32_t x67, float acc) {
  const uint32_t magic = 0x64006400u;
  const uint32_t p0 = and_or<0x000F000Fu>(w, magic);
  const uint32_t p1 = and_or<0x000F000Fu>(w >> 4, magic);
  const uint32_t p2 = and_or<0x000F000Fu>(w >> 8, magic);
  const uint32_t p3 = and_or<0x000F000Fu>(w >> 12, magic);
  asm("{\n\t"
      ".reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b32 {a2, a3}, %2;\n\t"
      "mov.b32 {a4, a5}, %3;\n\tmov.b32 {a6, a7}, %4;\n\t"
      "mov.b32 {b0, b1}, %5;\n\tmov.b32 {b2, b3}, %6;\n\t"
      "mov.b32 {b4, b5}, %7;\n\tmov.b32 {b6, b7}, %8;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
      "fma.rn.f32.f16 %0, a2, b1, %0;\n\t"
      "fma.rn.f32.f16 %0, a4, b2, %0;\n\t"
      "fma.rn.f32.f16 %0, a6, b3, %0;\n\t"
      "fma.rn.f32.f16 %0, a1, b4, %0;\n\t"
      "fma.rn.f32.f16 %0, a3, b5, %0;\n\t"
      "fma.rn.f32.f16 %0, a5, b6, %0;\n\t"
      "fma.rn.f32.f16 %0, a7, b7, %0;\n\t"
      "}"
      : "+f"(acc)
      : "r"(p0), "r"(p1), "r"(p2), "r"(p3), "r"(x01), "r"(x23), "r"(x45), "r"(x67));
  return acc;
}

__device__ __forceinline__ float2 h2f(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

template <int VARIANT>
__global__ void __launch_bounds__(kThreads)
    q4b32_gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
                      const uint16_t* __restrict__ scales, uint16_t* __restrict__ y, int N,
                      int K) {
  __shared__ float sRed[kWarps][kRows];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = K >> 5;  // blocks per row
  const int n0 = blockIdx.x * kRows;
  const int bpw = (nb + kWarps - 1) / kWarps;
  const int b_begin = min(nb, warp * bpw);
  const int b_end = min(nb, b_begin + bpw);
  const size_t row_bytes = static_cast<size_t>(K) >> 1;

  if (tid == 0) pdl_launch_dependents();
  pdl_wait();  // x may be written by the previous kernel on the stream

  float yacc[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) yacc[r] = 0.f;

  for (int b = b_begin + lane; b < b_end; b += 32) {
    uint4 cw[kRows];
    float sc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int n = n0 + r;
      if (n < N) {
        cw[r] = ld_stream16(codes + static_cast<size_t>(n) * row_bytes + static_cast<size_t>(b) * 16);
        sc[r] = __half2float(__ushort_as_half(__ldg(scales + static_cast<size_t>(n) * nb + b)));
      } else {
        cw[r] = make_uint4(0, 0, 0, 0);
        sc[r] = 0.f;
      }
    }
    const uint4* xp = reinterpret_cast<const uint4*>(x + static_cast<size_t>(b) * 32);
    uint4 xv[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) xv[v] = __ldg(xp + v);

    if (VARIANT == 0) {
      float2 xf[4][4];  // [word v][pair h] = (x_{8v+2h}, x_{8v+2h+1})
      float corr = 0.f;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t xw[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          xf[v][h] = h2f(xw[h]);
          corr += (code_offset_f32(0) + 8.0f) * xf[v][h].x + (code_offset_f32(1) + 8.0f) * xf[v][h].y;
        }
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const uint32_t cwv[4] = {cw[r].x, cw[r].y, cw[r].z, cw[r].w};
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[8];
          codes_to_f32_offset(cwv[v], f);
          a = __ffma2_rn(make_float2(f[0], f[1]), xf[v][0], a);
          a = __ffma2_rn(make_float2(f[2], f[3]), xf[v][1], a);
          a = __ffma2_rn(make_float2(f[4], f[5]), xf[v][2], a);
          a = __ffma2_rn(make_float2(f[6], f[7]), xf[v][3], a);
        }
        yacc[r] = fmaf(sc[r], (a.x + a.y) - corr, yacc[r]);
      }
    } else {
      float corr = 0.f;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t xw[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = h2f(xw[h]);
          corr += 1032.0f * f.x + 1032.0f * f.y;
        }
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const uint32_t cwv[4] = {cw[r].x, cw[r].y, cw[r].z, cw[r].w};
        float a = 0.f;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          a = dot8_mixed_f16(cwv[v], xv[v].x, xv[v].y, xv[v].z, xv[v].w, a);
        yacc[r] = fmaf(sc[r], a - corr, yacc[r]);
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    float v = yacc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sRed[warp][r] = v;
  }
  __syncthreads();
  if (tid < kRows) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += sRed[w][tid];
    const int n = n0 + tid;
    if (n < N) y[n] = __half_as_ushort(__float2half_rn(v));
  }
}

}  // namespace

cudaError_t launch_q4b32_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                              uint16_t* y, int N, int K, int variant, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((N + kRows - 1) / kRows);
  auto kern = variant == 1 ? q4b32_gemv_kernel<1> : q4b32_gemv_kernel<0>;
  return launch_with_pdl(kern, dim3(blocks), dim3(kThreads), 0, stream, x, codes, scales, y, N, K);
}

}  // namespace w4k
