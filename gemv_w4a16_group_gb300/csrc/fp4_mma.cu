// NVFP4A16 / MXFP4A16 GEMV on a TMA ring: y[n] = S sum_b e4m3(s[n,b]) sum_{j<16} e2m1(q) x
// (NVFP4, "Hardware-invariant NVFP4 progress report 1", "The NVFP4 layout") or
// y[n] = sum_b 2^(s[n,b] - 127) sum_{j<32} e2m1(q) x (MXFP4, "Low-Precision Kernels: INT4,
// INT8 and FP8 Matmuls, Measured", Step 6).
//
// The codes are laid out like the Q4 block-32 format ([N, K/2], byte j of a row holding k = 2j
// in its low nibble), so this kernel streams them the way the Q4 tensor-pipe GEMV does: work
// units of T tiles of 16 rows and all of K, a producer warp copying 512-k chunks by TMA (two
// 128-byte-wide code boxes with the 128-byte swizzle, one box of block scales) into a ring,
// consumer lanes (gq, c) reading word c of a 32-k block of rows gq and gq + 8 of a tile, two
// m16n8k16 MMAs per block (FP16 x FP16 -> fp32; x fills the n8 columns).
//
//   * Warps: T x P consumer warps, warp (t, p) taking tile t and the 32-k blocks p, p + P, ...
//     of every chunk, with (T, P) picked per shape from (1, 16), (2, 8), (3, 8), (4, 4),
//     (6, 4), (8, 2), (12, 2) so that the units spread over the SMs and 16 or 24 warps
//     compute (the loop is latency-bound: more warps, not fewer instructions, is what moved
//     it). Per unit the P partial sums of a row are added in a fixed order; no atomics.
//   * A byte of two codes becomes an FP16 pair in one cvt.rn.f16x2.e2m1x2 (natural k order,
//     so x waits in shared memory in natural order, 8 k per 16 bytes).
//   * x is FP16 under a power of two per 32-k block (its largest |x| in [2^14, 2^15)).
//   * NVFP4: the n8 columns of the MMAs keep the 16-k blocks apart: over a group of
//     up to four 32-k blocks of a warp, column 2g + h of B is x on the h-th 16-k half of the
//     group's g-th block and zero elsewhere (a lane whose column is not the block's reads a
//     zero segment instead of x; the choice is made once, in its per-block x offset). After
//     the group, column n of D holds the rows' sums over 16-k block n alone, and lane c,
//     which holds columns 2c and 2c + 1, multiplies the two sums of block c by their E4M3
//     scales and the block's x scale in fp32. The tensor scale multiplies each output once.
//   * MXFP4: each 32-k block's MMAs start from zero, and the block's power-of-two scale times
//     the x scale multiplies its fp32 sum (lane c folds the c-th block of each group of four,
//     like the Q4 scale).
//   * The codes carry no offset, so there is no correction term.
#include "common.cuh"
#include "fp4_common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kFMaxWarps = 24;  // consumer warps of the widest configuration
constexpr int kFBoxK = 256;     // 128 code bytes per row: one 128-byte swizzle row
constexpr int kFChunkK = 512;   // two code boxes per chunk
constexpr int kFBlocks = kFChunkK / 32;  // 32-k blocks per chunk
constexpr int kFMaxStages = 12;
constexpr uint32_t kFSmem = 227u * 1024u - 1024u;  // the base is aligned up to 1024 B

// Shared-memory layout for T tiles per unit and K; sb = scale bytes per row and chunk (32 for
// NVFP4's 32 E4M3 scales of 512 k, 16 for MXFP4's E8M0 ones).
// x in shared memory, per 512-k chunk: MXFP4 its 64 16-byte segments (8 k each); NVFP4 the
// same 64 segments, then zero segments at 64 and 68 (72 segments = 1152 bytes per chunk), one
// on each half of the banks.
constexpr uint32_t kFXChunkMX = 64u * 16u;
constexpr uint32_t kFXChunkNV = 72u * 16u;

struct FLayout {
  uint32_t code_bytes, scale_bytes, stage_bytes, red_off, cst_off, xperm_off, bar_off, total;
  __host__ __device__ FLayout(int T, int K, int stages, int sb) {
    code_bytes = 4096u * static_cast<uint32_t>(T);  // two boxes of 16 T rows x 128 B
    scale_bytes = static_cast<uint32_t>(sb) * 16u * static_cast<uint32_t>(T);
    stage_bytes = (code_bytes + scale_bytes + 1023u) & ~1023u;
    red_off = static_cast<uint32_t>(stages) * stage_bytes;          // [P][16 T] fp32
    cst_off = red_off + 16u * kFMaxWarps * 4u;                      // [K/32] 2^-e
    xperm_off = (cst_off + (static_cast<uint32_t>(K) / 32u) * 4u + 127u) & ~127u;
    const uint32_t xchunk = sb == 32 ? kFXChunkNV : kFXChunkMX;
    bar_off = (xperm_off + (static_cast<uint32_t>(K) / 512u) * xchunk + 7u) & ~7u;
    total = bar_off + 2u * kFMaxStages * 8u + 16u;
  }
};

template <int NT>
__device__ __forceinline__ void f_consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

struct FMaps {
  CUtensorMap codes;   // uint8 [N, K/2], box {128, 16 T}, 128-byte swizzle
  // uint8 [N, K/16] (NVFP4, box {32, 16 T}, 32-byte swizzle) or [N, K/32] (MXFP4, box
  // {16, 16 T}, no swizzle)
  CUtensorMap scales;
};

template <bool MX, int T, int P>
__global__ void __launch_bounds__(T * P * 32 + 32, 1)
    fp4_gemv_tc_kernel(const __grid_constant__ FMaps maps, const uint16_t* __restrict__ x,
                       const float* __restrict__ tensor_scale, uint16_t* __restrict__ y, int N,
                       int K, int nunits, int stages, uint32_t* __restrict__ status,
                       uint64_t limit_ns) {
  constexpr int W = T * P;            // consumer warps
  constexpr int NC = W * 32;          // consumer threads
  constexpr int NB = kFBlocks / P;    // 32-k blocks of a chunk per warp
  constexpr int SB = MX ? 16 : 32;    // scale bytes per row and chunk
  constexpr int ROWS = 16 * T;        // rows per unit
  static_assert(kFBlocks % P == 0 && W <= kFMaxWarps, "bad warp split");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const FLayout L(T, K, stages, SB);
  float* sRed = reinterpret_cast<float*>(smem + L.red_off);  // [P][ROWS]
  float* sCst = reinterpret_cast<float*>(smem + L.cst_off);  // [K/32] 2^-e per 32-k block
  uint4* sX = reinterpret_cast<uint4*>(smem + L.xperm_off);  // FP16, natural order per chunk
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kFMaxStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kFMaxStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kchunks = K / kFChunkK;
  const uint32_t tx_bytes = L.code_bytes + L.scale_bytes;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    *abort_flag = 0u;
    fence_barrier_init();
    pdl_launch_dependents();
  }
  __syncthreads();

  if (warp == W) {
    // ---------------- producer: weights only, no wait on the previous kernel -----------
    if (lane == 0) {
      tma_prefetch_desc(&maps.codes);
      tma_prefetch_desc(&maps.scales);
      int j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int row0 = u * ROWS;
        for (int kc = 0; kc < kchunks; ++kc, ++j) {
          const int s = j % stages;
          const uint32_t use = static_cast<uint32_t>(j / stages);
          if (use > 0 &&
              !mbar_wait_bounded(&empty[s], (use - 1) & 1u, abort_flag, status, limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* buf = smem + s * L.stage_bytes;
          mbar_arrive_expect_tx(&full[s], tx_bytes);
          tma_load_2d(buf, &maps.codes, &full[s], kc * (kFChunkK / 2), row0);
          tma_load_2d(buf + L.code_bytes / 2, &maps.codes, &full[s],
                      kc * (kFChunkK / 2) + kFBoxK / 2, row0);
          tma_load_2d(buf + L.code_bytes, &maps.scales, &full[s], kc * SB, row0);
        }
      }
      // Stay until this CTA's last copies have landed (bounded).
      const int issued = j;
      for (int s = 0; s < stages && s < issued; ++s) {
        const int last = (issued - 1 - s) / stages;
        volatile uint32_t no_abort = 0u;
        mbar_wait_bounded(&full[s], static_cast<uint32_t>(last) & 1u, &no_abort, status,
                          limit_ns);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  pdl_wait();  // x and y may belong to the previous kernel on the stream
  const int segs = K / 8;  // segment R = 8 k
  // x (BF16) -> FP16 in natural order with a power-of-two scale per 32-k block (its largest
  // |x| in [2^14, 2^15)), the 4 segments of a block on 4 adjacent lanes (segs and the thread
  // count are multiples of 32, so a warp is either wholly inside x or wholly past it).
  // NVFP4 puts segment R at slot 72 (R / 64) + R % 64, beside each chunk's zero segments.
  for (int base = 0; base < segs; base += NC) {
    const int R = base + tid;
    if (R >= segs) break;  // warp-uniform
    float v[8];
    f_bf16x8(__ldg(reinterpret_cast<const uint4*>(x) + R), v);
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(v[q]));
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = f_x_exponent(amax);
    sX[MX ? R : (R >> 6) * 72 + (R & 63)] = f_f16x8(v, f_pow2(e));
    if ((R & 3) == 0) sCst[R >> 2] = f_pow2(-e);
  }
  if constexpr (!MX) {
    for (int z = tid; z < 2 * kchunks; z += NC)
      sX[(z >> 1) * 72 + 64 + 4 * (z & 1)] = make_uint4(0u, 0u, 0u, 0u);
  }
  f_consumer_bar<NC>();

  const int gq = lane >> 2, c = lane & 3;
  const int t = warp % T, p = warp / T;  // tile in the unit, first 32-k block in a chunk
  const uint32_t rowA = static_cast<uint32_t>(16 * t + gq);  // rowB = rowA + 8
  // Blocks per fold group: MXFP4 folds each block's sum, NVFP4 each 16-k block's (both by
  // lane c for the group's c-th block).
  constexpr int G = NB < 4 ? NB : 4;
  // Per block r of this warp (block p + P r of a chunk): the offset of row rowA's word c in
  // a stage (rows gq and gq + 8 share the 128-byte swizzle phase gq = row mod 8) and of this
  // lane's 16 bytes of x in a chunk. NVFP4: words c = 0, 1 of a 32-k block hold its first
  // 16-k block and c = 2, 3 its second, so lane (gq, c) carries x for column gq exactly when
  // gq = 2 (r mod G) + c / 2, and otherwise the zero segment on the other half of the banks.
  uint32_t code_off[NB], x_off[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    const uint32_t j = static_cast<uint32_t>(p + P * r);
    code_off[r] = (j >> 3) * (L.code_bytes / 2) + rowA * 128u +
                  (((j & 7u) ^ static_cast<uint32_t>(gq)) << 4) + 4u * static_cast<uint32_t>(c);
    x_off[r] = (j * 4u + static_cast<uint32_t>(c)) * 16u;
    if (!MX && gq != 2 * (r % G) + (c >> 1)) x_off[r] = (j & 1u) ? 64u * 16u : 68u * 16u;
  }
  // NVFP4: the offset of row rowA's two scale bytes of the block this lane folds in each
  // group (the scale box comes with the 32-byte swizzle: the 16-byte halves of a row swap
  // where bit 2 of the row is set).
  constexpr int NG = NB / G;
  uint32_t s_off[NG];
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    const uint32_t j = static_cast<uint32_t>(p + P * (G * i + (c < G ? c : 0)));
    s_off[i] = rowA * SB + ((2u * j) ^ ((static_cast<uint32_t>(gq) & 4u) << 2));
  }
  const uint32_t ring_base = smem_addr(smem);
  const uint32_t xbase = smem_addr(sX);
  const float S = MX ? 1.0f : __ldg(tensor_scale);
  int s = 0;
  uint32_t phase = 0u;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const int row0 = u * ROWS;
    float accA = 0.f, accB = 0.f;  // rows rowA, rowB: this lane's blocks
    for (int kc = 0; kc < kchunks; ++kc) {
      // On an expired wait every warp keeps walking without computing, so all consumer
      // warps still meet at the per-unit barriers below.
      const bool landed = mbar_wait_bounded(&full[s], phase, abort_flag, status, limit_ns);
      const uint32_t buf = ring_base + static_cast<uint32_t>(s) * L.stage_bytes;
      const uint32_t sbox = buf + L.code_bytes;  // [16 T rows][SB bytes]
      const uint32_t xk = xbase + static_cast<uint32_t>(kc) * (MX ? kFXChunkMX : kFXChunkNV);
      if (landed) {
        if constexpr (!MX) {
#pragma unroll
          for (int i = 0; i < NG; ++i) {
            // two chains: the first and the second MMA of each block
            float d0[4] = {}, d1[4] = {};
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const int r = G * i + g;
              const uint32_t w0 = f_lds32(buf + code_off[r]);
              const uint32_t w1 = f_lds32(buf + code_off[r] + 1024u);
              const uint4 e = f_lds128(xk + x_off[r]);
              uint32_t p0[4], p1[4];
              f_e2m1_pairs(w0, p0);
              f_e2m1_pairs(w1, p1);
              // k-slots (2c, 2c + 1) and (2c + 8, 2c + 9) of an MMA hold k = 8c + 0, 1 and
              // 8c + 2, 3 (first MMA) or 8c + 4, 5 and 8c + 6, 7 (second): x in natural order.
              f_mma(d0, p0[0], p1[0], p0[1], p1[1], e.x, e.y);
              f_mma(d1, p0[2], p1[2], p0[3], p1[3], e.z, e.w);
            }
            // Lane c: columns 2c, 2c + 1 = the two 16-k halves of the group's block c (the
            // lanes past the group's blocks hold zero columns and fold nothing), times their
            // E4M3 scales and the block's x scale 2^-e.
            if (c < G) {
              const uint32_t j = static_cast<uint32_t>(p + P * (G * i + c));
              const float u2 = sCst[kc * kFBlocks + static_cast<int>(j)];
              const uint32_t qa = f_e4m3_pair(f_lds_u16(sbox + s_off[i]));
              const uint32_t qb = f_e4m3_pair(f_lds_u16(sbox + s_off[i] + 8u * SB));
              const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&qa));
              const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&qb));
              accA = fmaf(u2, fmaf(fa.x, d0[0] + d1[0], fa.y * (d0[1] + d1[1])), accA);
              accB = fmaf(u2, fmaf(fb.x, d0[2] + d1[2], fb.y * (d0[3] + d1[3])), accB);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < NB / G; ++i) {
            float d[G][4];
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const int r = G * i + g;
              const uint32_t w0 = f_lds32(buf + code_off[r]);
              const uint32_t w1 = f_lds32(buf + code_off[r] + 1024u);
              const uint4 e = f_lds128(xk + x_off[r]);
              uint32_t p0[4], p1[4];
              f_e2m1_pairs(w0, p0);
              f_e2m1_pairs(w1, p1);
#pragma unroll
              for (int f = 0; f < 4; ++f) d[g][f] = 0.f;
              f_mma(d[g], p0[0], p1[0], p0[1], p1[1], e.x, e.y);
              f_mma(d[g], p0[2], p1[2], p0[3], p1[3], e.z, e.w);
            }
            // Lane c folds block G i + c of the group for both rows (its D equals the other
            // lanes'); with fewer than four blocks in a group the other lanes add nothing.
            if (c < G) {
              float dA = d[0][0], dB = d[0][2];
#pragma unroll
              for (int g = 1; g < G; ++g) {
                if (c == g) {
                  dA = d[g][0];
                  dB = d[g][2];
                }
              }
              const uint32_t j = static_cast<uint32_t>(p + P * (G * i + c));
              const float u2 = sCst[kc * kFBlocks + static_cast<int>(j)];
              const float sA = f_e8m0(f_lds_u8(sbox + rowA * SB + j));
              const float sB = f_e8m0(f_lds_u8(sbox + (rowA + 8u) * SB + j));
              accA = fmaf(sA * u2, dA, accA);
              accB = fmaf(sB * u2, dB, accB);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == stages) {
        s = 0;
        phase ^= 1u;
      }
    }
    // Row sums: the 4 lanes of a row group (fixed order).
    accA += __shfl_xor_sync(0xffffffffu, accA, 1);
    accA += __shfl_xor_sync(0xffffffffu, accA, 2);
    accB += __shfl_xor_sync(0xffffffffu, accB, 1);
    accB += __shfl_xor_sync(0xffffffffu, accB, 2);
    if (c == 0) {
      sRed[p * ROWS + static_cast<int>(rowA)] = accA;
      sRed[p * ROWS + static_cast<int>(rowA) + 8] = accB;
    }
    f_consumer_bar<NC>();
    // then the P parts of each row (fixed order)
    for (int i = tid; i < ROWS; i += NC) {
      const int n = row0 + i;
      if (n < N) {
        float v = sRed[i];
#pragma unroll
        for (int q = 1; q < P; ++q) v += sRed[q * ROWS + i];
        y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(S * v));
      }
    }
    f_consumer_bar<NC>();
  }
}

struct FCfg {
  int T, P;
};
// (tiles per unit, k-parts per chunk), by growing T; 16 or 24 consumer warps each.
constexpr FCfg kFCfgs[] = {{1, 16}, {2, 8}, {3, 8}, {4, 4}, {6, 4}, {8, 2}, {12, 2}};
constexpr int kFNumCfgs = static_cast<int>(sizeof(kFCfgs) / sizeof(kFCfgs[0]));

struct FPlan {
  int cfg = -1, nunits = 0, stages = 0;
};

// The smallest unit (T tiles of 16 rows) that spreads the rows over the SMs in one wave,
// else the largest; then the largest unit no larger than that whose ring of at least two
// stages fits beside x; the deepest such ring.
FPlan f_plan(int N, int K, int sms, int sb) {
  FPlan p;
  if (K % kFChunkK != 0 || N <= 0 || sms <= 0) return p;
  const int tiles = (N + 15) / 16;
  const int need = (tiles + sms - 1) / sms;
  int ci = 0;
  while (ci + 1 < kFNumCfgs && kFCfgs[ci].T < need) ++ci;
  for (; ci >= 0; --ci) {
    const int T = kFCfgs[ci].T;
    const uint32_t fixed = FLayout(T, K, 0, sb).total;
    const uint32_t stage = FLayout(T, K, 0, sb).stage_bytes;
    int stages = fixed < kFSmem ? static_cast<int>((kFSmem - fixed) / stage) : 0;
    if (stages > kFMaxStages) stages = kFMaxStages;
    if (stages >= 2) {
      p.cfg = ci;
      p.nunits = (tiles + T - 1) / T;
      p.stages = stages;
      return p;
    }
  }
  return p;
}

template <bool MX, int T, int P>
cudaError_t launch_fp4(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                       const float* tensor_scale, uint16_t* y, int N, int K, const FPlan& plan,
                       int sms, uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  constexpr int SB = MX ? 16 : 32;
  FMaps maps;
  cudaError_t e = encode_tensor_map(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                                    static_cast<uint64_t>(K) / 2, static_cast<uint64_t>(N),
                                    static_cast<uint64_t>(K) / 2, kFBoxK / 2,
                                    static_cast<uint32_t>(16 * T), CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const uint64_t srow = MX ? static_cast<uint64_t>(K) / 32 : static_cast<uint64_t>(K) / 16;
  e = encode_tensor_map(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, srow,
                        static_cast<uint64_t>(N), srow, static_cast<uint32_t>(SB),
                        static_cast<uint32_t>(16 * T),
                        MX ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  const uint32_t smem = FLayout(T, K, plan.stages, SB).total + 1024u;
  auto kern = fp4_gemv_tc_kernel<MX, T, P>;
  e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = plan.nunits < sms ? plan.nunits : sms;
  return launch_with_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(T * P * 32 + 32), smem,
                         stream, maps, x, tensor_scale, y, N, K, plan.nunits, plan.stages,
                         status, limit_ns);
}

template <bool MX>
cudaError_t launch_fp4_cfg(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                           const float* tensor_scale, uint16_t* y, int N, int K,
                           const FPlan& plan, int sms, uint32_t* status, uint64_t limit_ns,
                           cudaStream_t stream) {
#define W4K_FP4_CASE(I, T_, P_)                                                       \
  case I:                                                                             \
    return launch_fp4<MX, T_, P_>(x, codes, scales, tensor_scale, y, N, K, plan, sms, \
                                  status, limit_ns, stream);
  switch (plan.cfg) {
    W4K_FP4_CASE(0, 1, 16)
    W4K_FP4_CASE(1, 2, 8)
    W4K_FP4_CASE(2, 3, 8)
    W4K_FP4_CASE(3, 4, 4)
    W4K_FP4_CASE(4, 6, 4)
    W4K_FP4_CASE(5, 8, 2)
    W4K_FP4_CASE(6, 12, 2)
    default:
      return cudaErrorNotSupported;
  }
#undef W4K_FP4_CASE
}

}  // namespace

bool fp4_tc_supports(int N, int K, bool mx) {
  return f_plan(N, K, device_sm_count(), mx ? 16 : 32).cfg >= 0;
}

cudaError_t launch_fp4_gemv_tc(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                               const float* tensor_scale, uint16_t* y, int N, int K, bool mx,
                               uint32_t* status, uint64_t wait_limit_ns, cudaStream_t stream) {
  const int sms = device_sm_count();
  const FPlan plan = f_plan(N, K, sms, mx ? 16 : 32);
  if (plan.cfg < 0) return cudaErrorNotSupported;
  if (mx)
    return launch_fp4_cfg<true>(x, codes, scales, nullptr, y, N, K, plan, sms, status,
                                wait_limit_ns, stream);
  return launch_fp4_cfg<false>(x, codes, scales, tensor_scale, y, N, K, plan, sms, status,
                               wait_limit_ns, stream);
}

}  // namespace w4k
