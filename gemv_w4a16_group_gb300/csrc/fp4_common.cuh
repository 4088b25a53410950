// Device helpers shared by the NVFP4 / MXFP4 kernels: E2M1 and E4M3 conversions on sm_103a,
// FP16 pair arithmetic, the m16n8k16 MMA and shared-memory loads by address.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace w4k {
namespace {

__device__ __forceinline__ void f_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f_lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 f_lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t f_lds_u8(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t f_lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// FP16 pairs of the four bytes of `w` (byte j -> (code 2j, code 2j + 1)).
__device__ __forceinline__ void f_e2m1_pairs(uint32_t w, uint32_t (&p)[4]) {
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
__device__ __forceinline__ uint32_t f_e4m3_pair(uint32_t v) {
  uint32_t r;
  asm("{\n\t.reg .b16 t, u;\n\tmov.b32 {t, u}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(v));
  return r;
}

__device__ __forceinline__ uint32_t f_hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t f_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f_pow2(int e) {  // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// e with amax 2^e in [2^14, 2^15) (0 for amax = 0), kept where 2^e and 2^-e are normal.
__device__ __forceinline__ int f_x_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  return max(-100, min(100, 141 - static_cast<int>(__float_as_uint(amax) >> 23)));
}

// The 8 BF16 values of a 16-byte segment as floats.
__device__ __forceinline__ void f_bf16x8(uint4 in, float (&v)[8]) {
  const uint32_t xw[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    v[2 * h] = __uint_as_float(xw[h] << 16);
    v[2 * h + 1] = __uint_as_float(xw[h] & 0xFFFF0000u);
  }
}

// 8 floats times sc, as FP16 (exact for BF16 inputs scaled into FP16's normal range).
__device__ __forceinline__ uint4 f_f16x8(const float (&v)[8], float sc) {
  return make_uint4(f_f16x2(v[0] * sc, v[1] * sc), f_f16x2(v[2] * sc, v[3] * sc),
                    f_f16x2(v[4] * sc, v[5] * sc), f_f16x2(v[6] * sc, v[7] * sc));
}

// 2^(code - 127) for an E8M0 code (0..254; code 0 is 2^-127, a subnormal float).
__device__ __forceinline__ float f_e8m0(uint32_t code) {
  return __uint_as_float(code == 0u ? 0x00400000u : (code << 23));
}

}  // namespace
}  // namespace w4k
