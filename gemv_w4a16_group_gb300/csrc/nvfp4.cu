// 4-bit float weights with 16-bit activations: NVFP4A16 (E2M1 codes, one E4M3 scale per 16
// weights along K and one fp32 scale per tensor: "Hardware-invariant NVFP4 progress report
// 1", "The NVFP4 layout") and MXFP4A16 (E2M1 codes, one E8M0 power-of-two scale per 32:
// "Low-Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", Step 6). The weight-only
// path decodes the codes to 16-bit floats and multiplies on the half-precision tensor path
// (NVFP4 shown; MXFP4 has 2^(s - 127) per 32 and no S):
//
//   y[n] = S * sum_b e4m3(s[n, b]) * sum_{j < 16} e2m1(q[n, 16 b + j]) x[16 b + j]
//
// Codes: uint8 [N, K/2], byte j of a row holding k = 2j (low nibble) and 2j + 1; scales:
// E4M3 bytes [N, K/16]; S: one fp32 in device memory.
//
// GEMV (M = 1). Same split as the W8A16 GEMV: a CTA works on 16 rows at a time (at most three
// CTAs per SM, looping over row tiles), its 8 warps take the 128-k chunks in turn with four
// chunks' loads in flight; lane (g, c) loads the 32 codes k = 128 ch + 32 c .. + 31 of rows g and
// g + 8 with one 16-byte load each. sm_103a converts a byte of two E2M1 codes to an FP16 pair
// in one instruction (cvt.rn.f16x2.e2m1x2), and the block scale multiplies the pair in FP16
// exactly (an E2M1 value has 2 significant bits and an E4M3 scale 4, and their product lies
// between 2^-10 and 2688, inside FP16's normal range). An MMA's 16 k-slots span four lanes and
// so four blocks, which is why the scale goes in before the MMA and not after. In MMA i of a
// chunk, lane c's k-slots hold k = 128 ch + 32 c + 4 i + (0, 1, 2, 3), so the B fragment is x in
// natural order; x is FP16 under a power of two per chunk (exact), undone per chunk in fp32,
// and S multiplies once at the end.
//
// Quantizer: the tensor's amax (one atomicMax of the float bits per warp into the tensor-scale
// word, zeroed first), then per block of 16: S = amax / 2688, the block scale the smallest
// E4M3 value not below amax_b / (6 S) (rounded up when the nearest one is below: the report's
// rule against clipping the block's largest weight), codes rounded to nearest even E2M1 with
// saturation at 6; a last one-thread kernel replaces amax by S.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kNvThreads = 256;
constexpr int kNvWarps = kNvThreads / 32;
constexpr int kNvUnroll = 4;     // chunks whose loads a warp has in flight together
constexpr int kNvMinBlocks = 3;  // resident CTAs per SM (79 registers a thread)

__device__ __forceinline__ uint4 ldg_stream128_nv(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// FP16 pairs of the four bytes of `w` (byte j -> (code 2j, code 2j + 1)).
__device__ __forceinline__ void e2m1_pairs_f16(uint32_t w, uint32_t (&p)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3])
      : "r"(w));
}

// FP16 pair of the two E4M3 bytes in the low 16 bits of `v`.
__device__ __forceinline__ uint32_t e4m3x2_f16(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(v));
  return r;
}

// Byte of two E2M1 codes: `hi` rounded into the high nibble, `lo` into the low one (nearest,
// ties to even, saturating at 6).
__device__ __forceinline__ uint32_t e2m1x2_rn(float hi, float lo) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

struct NvLayout {
  uint32_t cst_off, red_off, total;
  __host__ __device__ explicit NvLayout(int K) {
    cst_off = static_cast<uint32_t>(K) * 2u;  // x as FP16 [K]
    red_off = cst_off + static_cast<uint32_t>(K / 128) * 4u;  // 2^-e per chunk
    total = red_off + kNvWarps * 16u * 4u;
  }
};

// FP16 pair (2^d, 2^d) for -254 <= d <= 0; 0 below 2^-24 (FP16's smallest subnormal).
__device__ __forceinline__ uint32_t f16x2_pow2(int d) {
  const uint32_t h = d >= -14 ? static_cast<uint32_t>(d + 15) << 10
                              : (d >= -24 ? 1u << (d + 24) : 0u);
  return h | (h << 16);
}

// MX: MXFP4 (E8M0 scale per 32 codes, no tensor scale) instead of NVFP4 (E4M3 scale per 16
// codes and a tensor scale). A lane's 32 codes of a row are one MX block; its scale 2^X
// enters the FP16 codes as 2^(X - R), R the largest X of the row's four blocks in the chunk
// (exact down to FP16's smallest subnormal: a block 2^24 below its neighbours adds nothing
// the tolerance sees), and 2^R multiplies the chunk's fp32 sum.
template <bool MX>
__global__ void __launch_bounds__(kNvThreads, kNvMinBlocks)
    nvfp4_gemv_kernel(const uint16_t* __restrict__ x, const uint8_t* __restrict__ codes,
                      const uint8_t* __restrict__ scales, const float* __restrict__ tensor_scale,
                      uint16_t* __restrict__ y, int N, int K) {
  extern __shared__ __align__(16) uint8_t smem[];
  const NvLayout L(K);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* cst = reinterpret_cast<float*>(smem + L.cst_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunks = K >> 7;

  // x -> FP16: 16 values per thread, the 8 threads of a chunk on adjacent lanes.
  for (int base = 0; base < 8 * chunks; base += kNvThreads) {  // uniform per CTA
    const int i = base + tid;
    const bool valid = i < 8 * chunks;
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
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // amax 2^e in [2^14, 2^15): products with the rebuilt weights (at most 2688) stay far
    // inside fp32; e kept where 2^e is a normal float.
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
      if ((i & 7) == 0) cst[i >> 3] = pow2f(-e);
    }
  }
  __syncthreads();

  const int g = lane >> 2, c = lane & 3;
  const int ntiles = (N + 15) / 16;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {  // uniform per CTA
    const int n0 = tile * 16;
    const size_t ra = static_cast<size_t>(min(n0 + g, N - 1));
    const size_t rb = static_cast<size_t>(min(n0 + g + 8, N - 1));
    const uint8_t* pa = codes + ra * (K / 2) + 16 * c;
    const uint8_t* pb = codes + rb * (K / 2) + 16 * c;
    const uint8_t* qa = MX ? scales + ra * (K / 32) + c : scales + ra * (K / 16) + 2 * c;
    const uint8_t* qb = MX ? scales + rb * (K / 32) + c : scales + rb * (K / 16) + 2 * c;
    const uint32_t xlane = smem_addr(xs) + static_cast<uint32_t>(64 * c);
    float acc_a = 0.f, acc_b = 0.f;
    for (int ch0 = warp; ch0 < chunks; ch0 += kNvWarps * kNvUnroll) {
      uint4 wa[kNvUnroll], wb[kNvUnroll];
      uint32_t sa[kNvUnroll], sb[kNvUnroll];
  #pragma unroll
      for (int u = 0; u < kNvUnroll; ++u) {
        const int ch = ch0 + u * kNvWarps;
        if (ch < chunks) {
          wa[u] = ldg_stream128_nv(pa + 64 * static_cast<size_t>(ch));
          wb[u] = ldg_stream128_nv(pb + 64 * static_cast<size_t>(ch));
          if constexpr (MX) {
            sa[u] = __ldg(qa + 4 * static_cast<size_t>(ch));
            sb[u] = __ldg(qb + 4 * static_cast<size_t>(ch));
          } else {
            sa[u] = __ldg(reinterpret_cast<const unsigned short*>(qa + 8 * static_cast<size_t>(ch)));
            sb[u] = __ldg(reinterpret_cast<const unsigned short*>(qb + 8 * static_cast<size_t>(ch)));
          }
        }
      }
  #pragma unroll
      for (int u = 0; u < kNvUnroll; ++u) {
        const int ch = ch0 + u * kNvWarps;
        if (ch >= chunks) break;  // warp-uniform
        uint32_t sa_lo, sa_hi, sb_lo, sb_hi;
        int Ra = 0, Rb = 0;
        if constexpr (MX) {
          // largest exponent of the row's four blocks (lanes c = 0..3) in this chunk
          Ra = static_cast<int>(sa[u]);
          Rb = static_cast<int>(sb[u]);
          Ra = max(Ra, __shfl_xor_sync(0xffffffffu, Ra, 1));
          Rb = max(Rb, __shfl_xor_sync(0xffffffffu, Rb, 1));
          Ra = max(Ra, __shfl_xor_sync(0xffffffffu, Ra, 2));
          Rb = max(Rb, __shfl_xor_sync(0xffffffffu, Rb, 2));
          sa_lo = sa_hi = f16x2_pow2(static_cast<int>(sa[u]) - Ra);
          sb_lo = sb_hi = f16x2_pow2(static_cast<int>(sb[u]) - Rb);
        } else {
          // block scales 2c, 2c + 1 of this lane's 32 k, each duplicated into an FP16 pair
          const uint32_t s2a = e4m3x2_f16(sa[u]), s2b = e4m3x2_f16(sb[u]);
          sa_lo = __byte_perm(s2a, 0u, 0x1010);
          sa_hi = __byte_perm(s2a, 0u, 0x3232);
          sb_lo = __byte_perm(s2b, 0u, 0x1010);
          sb_hi = __byte_perm(s2b, 0u, 0x3232);
        }
        const uint32_t ra4[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
        const uint32_t rb4[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
        float d[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
        for (int wi = 0; wi < 4; ++wi) {  // word wi: MMAs 2 wi and 2 wi + 1
          uint32_t pa4[4], pb4[4];
          e2m1_pairs_f16(ra4[wi], pa4);
          e2m1_pairs_f16(rb4[wi], pb4);
          const uint32_t ska = wi < 2 ? sa_lo : sa_hi, skb = wi < 2 ? sb_lo : sb_hi;
          const uint4 xb = lds128(xlane + 256u * ch + 16u * wi);  // k = 32 c + 8 wi .. + 7
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a0 = hmul2_bits(pa4[2 * h], ska), a2 = hmul2_bits(pa4[2 * h + 1], ska);
            const uint32_t a1 = hmul2_bits(pb4[2 * h], skb), a3 = hmul2_bits(pb4[2 * h + 1], skb);
            mma_f16_16816(d, a0, a1, a2, a3, h ? xb.z : xb.x, h ? xb.w : xb.y);
          }
        }
        const float u2 = cst[ch];
        if constexpr (MX) {
          acc_a = fmaf(ldexpf(u2, Ra - 127), d[0], acc_a);
          acc_b = fmaf(ldexpf(u2, Rb - 127), d[2], acc_b);
        } else {
          acc_a = fmaf(u2, d[0], acc_a);
          acc_b = fmaf(u2, d[2], acc_b);
        }
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
      for (int w = 0; w < kNvWarps; ++w) v += red[w * 16 + tid];
      if constexpr (!MX) v *= __ldg(tensor_scale);
      y[n0 + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
    __syncthreads();  // red is rewritten by the next tile
  }
}

// ---------------------------------------------------------------------------------------
// Quantizer
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(kNvThreads)
    nvfp4_amax_kernel(const float* __restrict__ w, long long n4, uint32_t* __restrict__ amax_bits) {
  float m = 0.f;
  for (long long i = static_cast<long long>(blockIdx.x) * kNvThreads + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * kNvThreads) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(w) + i);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));  // m >= 0
}

// Value of a non-negative E4M3 code (exact in FP16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(e4m3x2_f16(code) & 0xFFFFu)));
}

__device__ __forceinline__ float tensor_scale_of(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// Smallest E4M3 code whose value is >= v (v >= 0), at most 0x7E (448).
__device__ __forceinline__ uint32_t e4m3_ceil(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
  uint32_t code = r & 0xFFu;
  const float back = e4m3_to_f32(code);
  if (back < v && code < 0x7Eu) ++code;
  return code;
}

// A warp takes 8 blocks of 16 (128 consecutive weights of a row), 4 weights per lane.
__global__ void __launch_bounds__(kNvThreads)
    nvfp4_quantize_kernel(const float* __restrict__ w, long long nblocks8,
                          const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                          uint8_t* __restrict__ scales) {
  const long long wi = static_cast<long long>(blockIdx.x) * kNvWarps + (threadIdx.x >> 5);
  if (wi >= nblocks8) return;
  const int lane = threadIdx.x & 31;
  const float S = tensor_scale_of(__uint_as_float(__ldg(amax_bits)));
  const float d6 = __fmul_rn(6.0f, S);
  const long long e0 = wi * 128 + lane * 4;  // first of this lane's 4 weights
  const float4 v = __ldcs(reinterpret_cast<const float4*>(w + e0));
  float bmax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 2));
  uint32_t sc = 0u, packed = 0u;
  if (bmax > 0.f) {
    sc = e4m3_ceil(__fdiv_rn(bmax, d6));
    const float sval = e4m3_to_f32(sc);
    const float den = __fmul_rn(sval, S);
    const uint32_t b0 = e2m1x2_rn(__fdiv_rn(v.y, den), __fdiv_rn(v.x, den));
    const uint32_t b1 = e2m1x2_rn(__fdiv_rn(v.w, den), __fdiv_rn(v.z, den));
    packed = (b0 & 0xFFu) | ((b1 & 0xFFu) << 8);
  }
  *reinterpret_cast<uint16_t*>(codes + e0 / 2) = static_cast<uint16_t>(packed);
  if ((lane & 3) == 0) scales[e0 / 16] = static_cast<uint8_t>(sc);
}

// MXFP4 ("Low-Precision Kernels ...", Step 6): per block of 32, scale 2^X with
// X = floor(log2 max|w|) - 2 (the largest power of two not above max|w|, over 4, the largest
// power of two E2M1 holds), kept in [-127, 127]; codes round w 2^-X (exact) to nearest even
// E2M1, clamped at 6; a block of zeros stores scale code 0 and codes 0. A warp takes 128
// consecutive weights (K % 32 == 0: blocks never straddle rows), 8 lanes per block.
__global__ void __launch_bounds__(kNvThreads)
    mxfp4_quantize_kernel(const float* __restrict__ w, long long total, uint8_t* __restrict__ codes,
                          uint8_t* __restrict__ scales) {
  const long long wi = static_cast<long long>(blockIdx.x) * kNvWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long e0 = wi * 128 + lane * 4;
  if (wi * 128 >= total) return;  // warp-uniform
  const bool valid = e0 < total;  // total is a multiple of 32: a block is valid or not
  const float4 v = valid ? __ldcs(reinterpret_cast<const float4*>(w + e0)) : make_float4(0, 0, 0, 0);
  float bmax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
  uint32_t sc = 0u, packed = 0u;
  if (bmax > 0.f) {
    int e;
    frexpf(bmax, &e);  // bmax = m 2^e, m in [0.5, 1)
    const int X = min(127, max(-127, e - 3));
    sc = static_cast<uint32_t>(X + 127);
    const float inv = pow2f(-X);  // -125 <= -X <= 127: a normal float
    const uint32_t b0 = e2m1x2_rn(__fmul_rn(v.y, inv), __fmul_rn(v.x, inv));
    const uint32_t b1 = e2m1x2_rn(__fmul_rn(v.w, inv), __fmul_rn(v.z, inv));
    packed = (b0 & 0xFFu) | ((b1 & 0xFFu) << 8);
  }
  if (!valid) return;
  *reinterpret_cast<uint16_t*>(codes + e0 / 2) = static_cast<uint16_t>(packed);
  if ((lane & 7) == 0) scales[e0 / 32] = static_cast<uint8_t>(sc);
}

__global__ void nvfp4_finalize_kernel(float* tensor_scale) {
  *tensor_scale = tensor_scale_of(*tensor_scale);  // the word holds amax until now
}

}  // namespace

uint32_t nvfp4_smem_bytes(int K) { return NvLayout(K).total; }

cudaError_t launch_nvfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                                  float* tensor_scale, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(tensor_scale, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const long long n4 = static_cast<long long>(N) * K / 4;
  long long blocks = (n4 + kNvThreads - 1) / kNvThreads;
  if (blocks > 4096) blocks = 4096;
  nvfp4_amax_kernel<<<static_cast<unsigned>(blocks), kNvThreads, 0, stream>>>(
      w, n4, reinterpret_cast<uint32_t*>(tensor_scale));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long nb8 = static_cast<long long>(N) * K / 128;
  const long long qblocks = (nb8 + kNvWarps - 1) / kNvWarps;
  if (qblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  nvfp4_quantize_kernel<<<static_cast<unsigned>(qblocks), kNvThreads, 0, stream>>>(
      w, nb8, reinterpret_cast<const uint32_t*>(tensor_scale), codes, scales);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  nvfp4_finalize_kernel<<<1, 1, 0, stream>>>(tensor_scale);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                              const float* tensor_scale, uint16_t* y, int N, int K,
                              cudaStream_t stream) {
  const uint32_t smem = NvLayout(K).total;
  if (smem > 48u * 1024u) {
    const cudaError_t e = set_max_dynamic_smem(
        reinterpret_cast<const void*>(nvfp4_gemv_kernel<false>), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int tiles = (N + 15) / 16;
  const int grid = tiles < sms * kNvMinBlocks ? tiles : sms * kNvMinBlocks;
  nvfp4_gemv_kernel<false><<<static_cast<unsigned>(grid), kNvThreads, smem, stream>>>(
      x, codes, scales, tensor_scale, y, N, K);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream) {
  const long long total = static_cast<long long>(N) * K;
  const long long blocks = (total + 128LL * kNvWarps - 1) / (128LL * kNvWarps);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  mxfp4_quantize_kernel<<<static_cast<unsigned>(blocks), kNvThreads, 0, stream>>>(w, total, codes,
                                                                                  scales);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                              uint16_t* y, int N, int K, cudaStream_t stream) {
  const uint32_t smem = NvLayout(K).total;
  if (smem > 48u * 1024u) {
    const cudaError_t e = set_max_dynamic_smem(
        reinterpret_cast<const void*>(nvfp4_gemv_kernel<true>), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int tiles = (N + 15) / 16;
  const int grid = tiles < sms * kNvMinBlocks ? tiles : sms * kNvMinBlocks;
  nvfp4_gemv_kernel<true><<<static_cast<unsigned>(grid), kNvThreads, smem, stream>>>(
      x, codes, scales, nullptr, y, N, K);
  return cudaGetLastError();
}

}  // namespace w4k
