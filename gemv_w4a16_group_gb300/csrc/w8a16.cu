// W8A16 GEMV: symmetric per-row INT8 weights, BF16 activations ("Quantization and GEMV",
// exercise 1: s = max|w| / 127 per row, q = round(w / s) in -127..127, one 16-byte load of
// 16 codes per lane, the row's scale applied once after the sum).
//
//   y[n] = s[n] * sum_k q[n, k] x[k]
//
// Where the time goes. At one byte per weight the GEMV reads N K bytes; at the measured
// HBM bandwidth a 14336 x 4096 layer takes 8.7 us. Converting a code costs the integer pipe
// 3/4 of an operation (one LOP3 flips the sign bits of four codes, u = q + 128; two PRMTs
// place two bytes each under the FP16 exponent of 1024, giving 1152 + q exactly), and the
// products run on the tensor pipe (mma.sync m16n8k16, FP16 x FP16 -> fp32).
//
// Work split. A CTA works on 16 rows at a time (the MMA's 16 rows), its 8 warps taking the
// 64-k chunks of K in turn (warp w: chunks w, w + 8, ...), four chunks' loads in flight per
// warp; the grid is at most three CTAs per SM, each looping over row tiles, so that x is
// converted once per CTA and the SMs' tile counts differ by at most one. Lane (g, c) =
// (lane / 4, lane % 4) loads the 16 codes k = 64 ch + 16 c .. + 15 of rows g and g + 8 (16
// bytes each, a warp reads 64 contiguous bytes of 16 rows). The MMA adds over k in any order as long as A and B agree:
// in MMA i of a chunk, k-slots (2c, 2c + 1, 2c + 8, 2c + 9) of lane c's fragments hold
// k = 64 ch + 16 c + 4 i + (0, 1, 2, 3), so the B fragment of lane (g, c) is the same 16
// consecutive x values, read from shared memory in natural order.
//
// x is converted to FP16 exactly once per CTA: per 64-k chunk a power of two 2^e puts the
// largest |x| in [2^14, 2^15) (a BF16 value has 8 significant bits, a normal FP16 11). Per
// chunk the MMAs return D = 2^e sum (1152 + q) x, and
//   acc += 2^-e (D - 1152 X),  X = 2^e sum x over the chunk,
// with X and 2^-e computed once per CTA. The 8 warps' partial sums are added in a fixed
// order; y = s acc, rounded to BF16.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kW8Threads = 256;
constexpr int kW8Warps = kW8Threads / 32;
constexpr int kW8Unroll = 4;  // chunks whose loads a warp has in flight together
constexpr int kW8MinBlocks = 3;  // resident CTAs per SM (72 registers a thread)

__device__ __forceinline__ uint4 ldg_stream128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// FP16 pairs (1152 + q0, 1152 + q1) and (1152 + q2, 1152 + q3) of the four signed codes in
// `w` (byte j = code j).
__device__ __forceinline__ void int8_pairs_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;  // two's complement byte q -> q + 128
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// Shared memory: x as FP16 [K] (2^e per chunk), per chunk {1152 X, 2^-e}, warp partials.
struct W8Layout {
  uint32_t cst_off, red_off, total;
  __host__ __device__ explicit W8Layout(int K) {
    cst_off = static_cast<uint32_t>(K) * 2u;
    red_off = cst_off + static_cast<uint32_t>(K / 64) * 8u;
    total = red_off + kW8Warps * 16u * 4u;
  }
};

__global__ void __launch_bounds__(kW8Threads, kW8MinBlocks)
    w8a16_gemv_kernel(const uint16_t* __restrict__ x, const int8_t* __restrict__ q,
                      const float* __restrict__ s, uint16_t* __restrict__ y, int N, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  const W8Layout L(K);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float2* cst = reinterpret_cast<float2*>(smem + L.cst_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunks = K >> 6;

  // x -> FP16, 16 values per thread, the 4 threads of a chunk on adjacent lanes.
  for (int base = 0; base < 4 * chunks; base += kW8Threads) {  // uniform per CTA
    const int i = base + tid;
    const bool valid = i < 4 * chunks;
    uint4 in[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    if (valid) {
      const uint4* src = reinterpret_cast<const uint4*>(x + 16 * i);
      in[0] = __ldg(src);
      in[1] = __ldg(src + 1);
    }
    float v[16];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t xw[4] = {in[r].x, in[r].y, in[r].z, in[r].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v[8 * r + 2 * h] = bf16_bits_to_f32(xw[h] & 0xFFFFu);
        v[8 * r + 2 * h + 1] = __uint_as_float(xw[h] & 0xFFFF0000u);
      }
    }
    float amax = 0.f, sum = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      amax = fmaxf(amax, fabsf(v[j]));
      sum += v[j];
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    // amax 2^e in [2^14, 2^15): e = 141 - biased exponent, kept where 2^e is a normal float.
    int e = 0;
    if (amax > 0.f) e = max(-100, min(100, 141 - static_cast<int>(__float_as_uint(amax) >> 23)));
    const float sc = pow2f(e);
    if (valid) {
      uint4 out[2];
      out[0] = make_uint4(f16x2_bits(v[0] * sc, v[1] * sc), f16x2_bits(v[2] * sc, v[3] * sc),
                          f16x2_bits(v[4] * sc, v[5] * sc), f16x2_bits(v[6] * sc, v[7] * sc));
      out[1] = make_uint4(f16x2_bits(v[8] * sc, v[9] * sc), f16x2_bits(v[10] * sc, v[11] * sc),
                          f16x2_bits(v[12] * sc, v[13] * sc), f16x2_bits(v[14] * sc, v[15] * sc));
      reinterpret_cast<uint4*>(xs + 16 * i)[0] = out[0];
      reinterpret_cast<uint4*>(xs + 16 * i)[1] = out[1];
      if ((i & 3) == 0) cst[i >> 2] = make_float2(1152.0f * (sum * sc), pow2f(-e));
    }
  }
  __syncthreads();

  const int g = lane >> 2, c = lane & 3;
  const int ntiles = (N + 15) / 16;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {  // uniform per CTA
    const int n0 = tile * 16;
    const int8_t* pa = q + static_cast<size_t>(min(n0 + g, N - 1)) * K + 16 * c;
    const int8_t* pb = q + static_cast<size_t>(min(n0 + g + 8, N - 1)) * K + 16 * c;
    const uint32_t xlane = smem_addr(xs) + static_cast<uint32_t>(32 * c);
    float acc_a = 0.f, acc_b = 0.f;  // rows g and g + 8
    for (int ch0 = warp; ch0 < chunks; ch0 += kW8Warps * kW8Unroll) {
      uint4 wa[kW8Unroll], wb[kW8Unroll];
  #pragma unroll
      for (int u = 0; u < kW8Unroll; ++u) {
        const int ch = ch0 + u * kW8Warps;
        if (ch < chunks) {
          wa[u] = ldg_stream128(pa + 64 * static_cast<size_t>(ch));
          wb[u] = ldg_stream128(pb + 64 * static_cast<size_t>(ch));
        }
      }
  #pragma unroll
      for (int u = 0; u < kW8Unroll; ++u) {
        const int ch = ch0 + u * kW8Warps;
        if (ch >= chunks) break;  // warp-uniform
        const uint4 x0 = lds128(xlane + 128u * ch), x1 = lds128(xlane + 128u * ch + 16u);
        const uint32_t xa[4][2] = {{x0.x, x0.y}, {x0.z, x0.w}, {x1.x, x1.y}, {x1.z, x1.w}};
        const uint32_t ra[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
        const uint32_t rb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
        float d[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t a0, a2, a1, a3;
          int8_pairs_f16(ra[i], a0, a2);  // row g: k-slots (2c, 2c + 1), (2c + 8, 2c + 9)
          int8_pairs_f16(rb[i], a1, a3);  // row g + 8
          mma_f16_16816(d, a0, a1, a2, a3, xa[i][0], xa[i][1]);
        }
        // every B column holds x, so d[0] (row g) and d[2] (row g + 8) are the chunk's sums
        const float2 cc = cst[ch];
        acc_a = fmaf(cc.y, d[0] - cc.x, acc_a);
        acc_b = fmaf(cc.y, d[2] - cc.x, acc_b);
      }
    }
    if (c == 0) {
      red[warp * 16 + g] = acc_a;
      red[warp * 16 + g + 8] = acc_b;
    }
    __syncthreads();
    if (tid < 16 && n0 + tid < N) {
      float v = 0.f;
  #pragma unroll
      for (int w = 0; w < kW8Warps; ++w) v += red[w * 16 + tid];
      y[n0 + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(v * s[n0 + tid]));
    }
    __syncthreads();  // red is rewritten by the next tile
  }
}

// round(fl(d / s)) half away from zero for |d / s| <= 127 (1 + 2^-23): t = fl(d rs) lies
// within 3 * 128 * 2^-24 < 2^-14 of fl(d / s), so both round to the same integer unless t
// is within 2^-14 of a half-integer, where the quotient is computed exactly.
__device__ __forceinline__ float round_quotient_w8(float d, float s, float rs) {
  const float t = __fmul_rn(d, rs);
  const float r = rintf(t);
  if (fabsf(__fsub_rn(t, r)) <= 0.5f - 0x1p-14f) return r;
  return roundf(__fdiv_rn(d, s));
}

// One CTA per row: max |w| over the row, s = fl(max / 127), then the codes (second read of
// the row, from L2).
__global__ void __launch_bounds__(kW8Threads)
    w8a16_quantize_kernel(const float* __restrict__ w, int K, int8_t* __restrict__ q,
                          float* __restrict__ s) {
  __shared__ float warp_max[kW8Warps];
  const int n = blockIdx.x, tid = threadIdx.x;
  const float* row = w + static_cast<size_t>(n) * K;
  float amax = 0.f;
  for (int k = 4 * tid; k < K; k += 4 * kW8Threads) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(row + k));
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) warp_max[tid >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int i = 1; i < kW8Warps; ++i) amax = fmaxf(amax, warp_max[i]);
  const float s32 = __fdiv_rn(amax, 127.0f);
  if (tid == 0) s[n] = s32;
  const float rs = s32 != 0.f ? __frcp_rn(s32) : 0.f;
  auto code = [&](float v) -> uint32_t {
    if (s32 == 0.f) return 0u;
    const float r = fminf(fmaxf(round_quotient_w8(v, s32, rs), -127.f), 127.f);
    return static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu;
  };
  for (int k = 4 * tid; k < K; k += 4 * kW8Threads) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(row + k));
    *reinterpret_cast<uint32_t*>(q + static_cast<size_t>(n) * K + k) =
        code(v.x) | (code(v.y) << 8) | (code(v.z) << 16) | (code(v.w) << 24);
  }
}

}  // namespace

int device_sm_count() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

uint32_t w8a16_smem_bytes(int K) { return W8Layout(K).total; }

cudaError_t launch_w8a16_quantize(const float* w, int N, int K, int8_t* q, float* s,
                                  cudaStream_t stream) {
  w8a16_quantize_kernel<<<static_cast<unsigned>(N), kW8Threads, 0, stream>>>(w, K, q, s);
  return cudaGetLastError();
}

cudaError_t launch_w8a16_gemv(const uint16_t* x, const int8_t* q, const float* s, uint16_t* y,
                              int N, int K, cudaStream_t stream) {
  const uint32_t smem = W8Layout(K).total;
  if (smem > 48u * 1024u) {
    const cudaError_t e =
        set_max_dynamic_smem(reinterpret_cast<const void*>(w8a16_gemv_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int tiles = (N + 15) / 16;
  const int grid = tiles < sms * kW8MinBlocks ? tiles : sms * kW8MinBlocks;
  w8a16_gemv_kernel<<<static_cast<unsigned>(grid), kW8Threads, smem, stream>>>(x, q, s, y, N, K);
  return cudaGetLastError();
}

}  // namespace w4k
