// Device-side helpers shared by the sm_103a kernels: shared-memory barriers with
// bounded waits, TMA tile loads, tcgen05 (tensor memory + 5th-gen MMA) wrappers and
// the nibble -> number conversions used by every kernel.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace w4k {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the previous kernel on its stream has finished.
// pdl_wait() blocks until that previous grid has completed and its memory is visible;
// everything that reads data a previous kernel may produce (activations) or writes
// data it may read (outputs, workspace) must come after it. Weights are never written
// by kernels of a decode step, so they may be streamed before it. Without the launch
// attribute both instructions are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launch `kern` with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_with_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// One bounded test of the phase. A thread whose phase is not complete is suspended by the
// hardware until the phase completes or ~20 us pass, so waiting warps do not spin on the
// issue slots the working warps need.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return done != 0;
}

// Waits until the barrier phase with the given parity completes. Gives up when the
// CTA-wide abort flag is raised, or after `limit_ns` of global time, in which case it
// raises the abort flag and latches kStatusTimeout in the device status word.
// Returns true only if the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile uint32_t* abort_flag,
                                                  uint32_t* status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) tile loads into this CTA's shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Contiguous copy of `bytes` from global memory into this CTA's shared memory, completing
// on `bar`. Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// x (innermost) must be a multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

// Rank-3 tile load; x (innermost) must be a multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA (single-CTA forms)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_in_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_in_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives (once) on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], kind::f16 (BF16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_a_tmem(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Store 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Store 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Load 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the 128-byte
// swizzle: rows of 128 bytes (64 BF16), 8-row atoms of 1024 bytes (stride byte
// offset), descriptor version 1 (sm_100 family), swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;    // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1u) << 46;          // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;          // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, BF16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Nibble conversions
// ---------------------------------------------------------------------------
// The fp32 pattern 0x43000000 | (v << 16) is 128 + v for 0 <= v < 16, and
// 0x45000000 | (v << 12) is 2048 + v: a 4-bit code placed in the mantissa under a
// fixed exponent is an exact float with a known offset ("Low-Precision Kernels ...",
// "Where the time goes at M = 1": the code goes into the low mantissa bits of a float
// whose exponent is fixed; "Quantization and GEMV", "What production kernels do").
//
// codes_to_f32_offset: word w holds codes q0..q7 (q_j in bits 4j..4j+3). Returns
// f[j] = B_j + q_j with B_j = 2048 for even j and 128 for odd j, using four shifts and
// eight AND/OR (LOP3) operations.
__device__ __forceinline__ void codes_to_f32_offset(uint32_t w, float (&f)[8]) {
  const uint32_t u0 = w << 12, u1 = w << 4, u2 = w >> 4, u3 = w >> 12;
  f[0] = __uint_as_float((u0 & 0x0000F000u) | 0x45000000u);
  f[1] = __uint_as_float((u0 & 0x000F0000u) | 0x43000000u);
  f[2] = __uint_as_float((u1 & 0x0000F000u) | 0x45000000u);
  f[3] = __uint_as_float((u1 & 0x000F0000u) | 0x43000000u);
  f[4] = __uint_as_float((u2 & 0x0000F000u) | 0x45000000u);
  f[5] = __uint_as_float((u2 & 0x000F0000u) | 0x43000000u);
  f[6] = __uint_as_float((u3 & 0x0000F000u) | 0x45000000u);
  f[7] = __uint_as_float((u3 & 0x000F0000u) | 0x43000000u);
}
// (a & MASK) | c as one LOP3. Written out in PTX because the same expression in C++, four
// times per packed word in an unrolled loop, compiled to code that issued more ALU
// instructions: the M = 1 GEMV on a 14336 x 4096 layer took 8.02 us per launch with the C++
// form and 7.09 us with this one (the Q4 block-32 GEMV on 16384 x 16384: 33.1 vs 27.2 us).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "n"(MASK), "r"(c));
  return r;
}

// ---------------------------------------------------------------------------
// FP16 code pairs and the legacy tensor-core MMA (GEMV and skinny kernels)
// ---------------------------------------------------------------------------
// (1024 + q) / (1024 + 16 q) FP16 pairs for the 8 codes of `w` (q_j in bits 4j..4j+3):
// p0 = (q0, q4), p1 = (16 q1, 16 q5), p2 = (q2, q6), p3 = (16 q3, 16 q7).
__device__ __forceinline__ void code_pairs_f16(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t magic = 0x64006400u;
  p[0] = and_or<0x000F000Fu>(w, magic);
  p[1] = and_or<0x00F000F0u>(w, magic);
  p[2] = and_or<0x000F000Fu>(w8, magic);
  p[3] = and_or<0x00F000F0u>(w8, magic);
}

// D += A (16x16, FP16) * B (16x8, FP16), fp32 accumulators; fragment layout of mma.sync
// m16n8k16 (row-major A, column-major B).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// Offsets used by codes_to_f32_offset for code j of a word.
__host__ __device__ constexpr float code_offset_f32(int j) { return (j & 1) ? 128.0f : 2048.0f; }

// codes_to_bf16x2_consecutive: word w holds codes q0..q7. Returns four BF16 pairs
// p[i] = (128 + q_{2i}, 128 + q_{2i+1}) (low half = even code), each exact.
__device__ __forceinline__ void codes_to_bf16x2_consecutive(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t v = w >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // byte 0 <- byte i of w (q_{2i} low), byte 2 <- byte i of v (q_{2i+1} low)
    const uint32_t t = __byte_perm(w, v, (i) | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12));
    p[i] = and_or<0x000F000Fu>(t, 0x43004300u);
  }
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// Scale s and offset of one group in fp32, so that w_hat = q s + offset. Minimum form: BF16
// s and minimum. Zero-point form ("Quantization and GEMV", "The quantization formulas":
// w_hat = (q - z) s): FP16 s and z, offset -s z, exact in fp32 (two 11-bit significands).
template <bool ZP>
__device__ __forceinline__ void group_scale_offset(uint32_t sbits, uint32_t obits, float& sc,
                                                   float& off) {
  if constexpr (ZP) {
    sc = f16_bits_to_f32(sbits);
    off = -sc * f16_bits_to_f32(obits);
  } else {
    sc = bf16_bits_to_f32(sbits);
    off = bf16_bits_to_f32(obits);
  }
}

}  // namespace w4k
