// Q4 block-32 GEMV on the tensor pipe: y[n] = sum_b s[n,b] * sum_{j<32} (q[n,b,j] - 8) x[32b+j].
//
// Format from "Why My 4-Bit CUDA Kernel Wasn't Faster" ("Why fewer bytes should have helped":
// 16 code bytes + one FP16 scale per 32 weights, decode = (code - 8) * scale), codes and
// scales in separate arrays ("Loading the same bytes differently"). That page's lesson is
// that the load width and count decide the speed; on GB300 the next limit is the integer
// pipe that turns nibbles into numbers, so this kernel spends 4 masks + 1 shift per 8 codes
// and hands the products to mma.sync:
//
//   * a packed word's nibbles become FP16 pairs in place: 0x6400 | q = 1024 + q (bits 0..3
//     of a half) and 0x6400 | 16 q = 1024 + 16 q (bits 4..7), one LOP3 per pair, one shift
//     per word for the upper bytes; x is converted to FP16 exactly with a power-of-two scale
//     2^e per block of 32 (largest |x| in [2^14, 2^15)), the slots holding 16 q get
//     x 2^(e-4). Per block the tensor core returns D = 2^e (sum q x + 1024 sum_even x +
//     64 sum_odd x), so sum (q - 8) x = 2^-e D - T with T = 1032 sum_even x + 72 sum_odd x
//     (even / odd: position of k in its 4-byte word), computed once per CTA;
//   * work units are 16 T consecutive rows (T <= 8 tiles of 16, chosen so that the units
//     spread over the SMs) and all of K; a producer warp streams chunks of 512 k with TMA:
//     the codes as two 128-byte-wide boxes with the 128-byte swizzle (the 16-byte groups of
//     a row are XORed with the row index mod 8, so the lanes' 4-byte loads of 8 rows hit
//     distinct banks) and the scales as a 32-byte-wide box;
//   * 16 consumer warps: warp (t, h) takes tile t and k-half h (one box, 8 blocks) of
//     every chunk, so a barrier wait covers 8 blocks of work. Lane
//     (gq, c) = (lane / 4, lane % 4) reads word c of each 32-k block of rows gq and gq + 8
//     of the tile: those two words fill the A fragments of the block's two m16n8k16 MMAs
//     (k order permuted to match the code pairs; x waits in shared memory in B-fragment
//     order). The four lanes of a row group hold the same D (one batch row), so lane c
//     folds blocks c and c + 4: y += (s 2^-e) D - s T;
//   * per unit the lane sums are reduced over the row group and the two k-halves in a
//     fixed order; no atomics.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kQConsumerWarps = 16;  // (tile t < 8) x (k-half h < 2)
constexpr int kQConsumers = kQConsumerWarps * 32;
constexpr int kQThreads = kQConsumers + 32;
constexpr int kQMaxTiles = 8;
constexpr int kQBoxK = 256;    // 128 code bytes per row: one 128-byte swizzle row
constexpr int kQChunkK = 512;  // two boxes per chunk, one per k-half
constexpr int kQMaxStages = 12;
constexpr uint32_t kQSmem = 227u * 1024u - 1024u;  // the base is aligned up to 1024 B

// Shared-memory layout for T tiles per unit and K.
struct Q4Layout {
  uint32_t code_bytes, stage_bytes, red_off, cst_off, xperm_off, bar_off, total;
  __host__ __device__ Q4Layout(int T, int K, int stages) {
    code_bytes = 4096u * static_cast<uint32_t>(T);  // two boxes of 16 T rows x 128 B
    stage_bytes = (code_bytes + 512u * static_cast<uint32_t>(T) + 1023u) & ~1023u;
    red_off = static_cast<uint32_t>(stages) * stage_bytes;    // [2][128] fp32
    cst_off = red_off + 2u * 128u * 4u;                       // [K/32] x {2^-e, T}
    xperm_off = (cst_off + (static_cast<uint32_t>(K) / 32u) * 8u + 15u) & ~15u;
    bar_off = (xperm_off + (static_cast<uint32_t>(K) / 8u) * 16u + 7u) & ~7u;
    total = bar_off + 2u * kQMaxStages * 8u + 16u;
  }
};

// (1024 + q) / (1024 + 16 q) FP16 pairs for the 8 codes of `w` (q_j in bits 4j..4j+3).
__device__ __forceinline__ void q4_pairs(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t magic = 0x64006400u;
  p[0] = and_or<0x000F000Fu>(w, magic);
  p[1] = and_or<0x00F000F0u>(w, magic);
  p[2] = and_or<0x000F000Fu>(w8, magic);
  p[3] = and_or<0x00F000F0u>(w8, magic);
}

__device__ __forceinline__ void q4_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128q(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_f16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float pow2(int e) {  // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}
__device__ __forceinline__ void q4_consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kQConsumers) : "memory");
}

struct Q4Maps {
  CUtensorMap codes;   // uint8 [N, K/2], box {128, 16 T}, 128-byte swizzle
  CUtensorMap scales;  // fp16 [N, K/32], box {16, 16 T}
};

__global__ void __launch_bounds__(kQThreads, 1)
    q4b32_gemv_tc_kernel(const __grid_constant__ Q4Maps maps, const uint16_t* __restrict__ x,
                         uint16_t* __restrict__ y, int N, int K, int T, int nunits, int stages,
                         uint32_t* __restrict__ status, uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const Q4Layout L(T, K, stages);
  float* sRed = reinterpret_cast<float*>(smem + L.red_off);  // [2][128]
  float2* sCst = reinterpret_cast<float2*>(smem + L.cst_off);  // [K/32] {2^-e, T}
  uint4* sXperm = reinterpret_cast<uint4*>(smem + L.xperm_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kQMaxStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kQMaxStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kchunks = K / kQChunkK;
  const int rows_per_unit = 16 * T;
  const uint32_t tx_bytes = L.code_bytes + 512u * static_cast<uint32_t>(T);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQConsumerWarps);
    }
    *abort_flag = 0u;
    fence_barrier_init();
    pdl_launch_dependents();
  }
  __syncthreads();

  if (warp == kQConsumerWarps) {
    // ---------------- producer: weights only, no wait on the previous kernel -----------
    if (lane == 0) {
      tma_prefetch_desc(&maps.codes);
      tma_prefetch_desc(&maps.scales);
      int j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int row0 = u * rows_per_unit;
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
          tma_load_2d(buf, &maps.codes, &full[s], kc * (kQChunkK / 2), row0);
          tma_load_2d(buf + L.code_bytes / 2, &maps.codes, &full[s], kc * (kQChunkK / 2) + kQBoxK / 2,
                      row0);
          tma_load_2d(buf + L.code_bytes, &maps.scales, &full[s], kc * (kQChunkK / 32), row0);
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
  {
    // x -> FP16 in B-fragment order with a power-of-two scale per block of 32; per block
    // 2^-e and T = 1032 sum_even x + 72 sum_odd x. Segment R = 8 k; the 4 segments of a
    // block are 4 adjacent lanes. Loads of up to 4 segments per thread go out first.
    const int segs = K / 8;
    for (int base = 0; base < segs; base += 4 * kQConsumers) {
      uint4 xin[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int R = base + t * kQConsumers + tid;
        xin[t] = R < segs ? __ldg(reinterpret_cast<const uint4*>(x) + R) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int R = base + t * kQConsumers + tid;
        if (base + t * kQConsumers >= segs) break;  // warp-uniform: segs is a multiple of 4
        const uint32_t xw[4] = {xin[t].x, xin[t].y, xin[t].z, xin[t].w};
        float v[8];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          v[2 * h] = __half2float(__ushort_as_half(static_cast<unsigned short>(xw[h] & 0xFFFFu)));
          v[2 * h + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(xw[h] >> 16)));
        }
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(v[q]));
        float se = (v[0] + v[2]) + (v[4] + v[6]);
        float so = (v[1] + v[3]) + (v[5] + v[7]);
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          se += __shfl_xor_sync(0xffffffffu, se, o);
          so += __shfl_xor_sync(0xffffffffu, so, o);
        }
        int e = 0;
        if (amax > 0.f)
          e = max(-100, min(100, 141 - static_cast<int>(__float_as_uint(amax) >> 23)));
        const float lo = pow2(e), hi = pow2(e - 4);
        if (R < segs) {
          uint4 out;
          out.x = f16x2_of(v[0] * lo, v[4] * lo);  // (x0, x4) 2^e
          out.y = f16x2_of(v[1] * hi, v[5] * hi);  // (x1, x5) 2^(e-4)
          out.z = f16x2_of(v[2] * lo, v[6] * lo);  // (x2, x6) 2^e
          out.w = f16x2_of(v[3] * hi, v[7] * hi);  // (x3, x7) 2^(e-4)
          sXperm[R] = out;
          if ((R & 3) == 0) sCst[R >> 2] = make_float2(pow2(-e), fmaf(1032.0f, se, 72.0f * so));
        }
      }
    }
  }
  q4_consumer_bar();

  const int gq = lane >> 2, c = lane & 3;
  const int t = warp & 7, h = warp >> 3;  // tile in the unit, k-half of each chunk
  const bool active = t < T;
  const uint32_t ring_base = smem_addr(smem);
  const uint32_t xbase = smem_addr(sXperm);
  // Rows gq and gq + 8 of the tile share the 128-byte swizzle phase gq (row mod 8).
  const uint32_t rowA = static_cast<uint32_t>(16 * t + gq), rowB = rowA + 8u;
  int s = 0;
  uint32_t phase = 0u;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const int row0 = u * rows_per_unit;
    float accA = 0.f, accB = 0.f;  // rows rowA, rowB: this lane's blocks
    for (int kc = 0; kc < kchunks; ++kc) {
      // On an expired wait every warp keeps walking without computing, so all consumer
      // warps still meet at the per-unit barriers below.
      const bool landed = mbar_wait_bounded(&full[s], phase, abort_flag, status, limit_ns);
      const uint32_t buf = ring_base + static_cast<uint32_t>(s) * L.stage_bytes;
      if (landed && active) {
        const uint32_t box = buf + static_cast<uint32_t>(h) * (L.code_bytes / 2);
        float d[8][4];  // one accumulator per 32-k block of this k-half
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t b = static_cast<uint32_t>(8 * h + j);  // block within the chunk
          const uint32_t chunk16 = ((static_cast<uint32_t>(j) ^ static_cast<uint32_t>(gq)) << 4) + 4u * c;
          const uint32_t w0 = lds32(box + rowA * 128u + chunk16);
          const uint32_t w1 = lds32(box + rowB * 128u + chunk16);
          const uint4 e = lds128q(xbase + ((kc * 16 + b) * 4 + c) * 16u);
          uint32_t p0[4], p1[4];
          q4_pairs(w0, p0);
          q4_pairs(w1, p1);
#pragma unroll
          for (int f = 0; f < 4; ++f) d[j][f] = 0.f;
          q4_mma(d[j], p0[0], p1[0], p0[1], p1[1], e.x, e.y);
          q4_mma(d[j], p0[2], p1[2], p0[3], p1[3], e.z, e.w);
        }
        // Lane c folds blocks c and c + 4 of this k-half for both rows (its D equals the
        // other lanes').
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float dA = (c & 2) ? ((c & 1) ? d[4 * i + 3][0] : d[4 * i + 2][0])
                                   : ((c & 1) ? d[4 * i + 1][0] : d[4 * i][0]);
          const float dB = (c & 2) ? ((c & 1) ? d[4 * i + 3][2] : d[4 * i + 2][2])
                                   : ((c & 1) ? d[4 * i + 1][2] : d[4 * i][2]);
          const uint32_t b = static_cast<uint32_t>(8 * h + 4 * i + c);
          const float2 cst = sCst[kc * 16 + b];
          const uint32_t sa = buf + L.code_bytes + rowA * 32u + 2u * b;
          const float sA = lds_f16(sa), sB = lds_f16(sa + 8u * 32u);
          accA = fmaf(sA * cst.x, dA, fmaf(-sA, cst.y, accA));
          accB = fmaf(sB * cst.x, dB, fmaf(-sB, cst.y, accB));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == stages) {
        s = 0;
        phase ^= 1u;
      }
    }
    // Row sums: the 4 lanes of a row group, then the two k-halves (fixed order).
    accA += __shfl_xor_sync(0xffffffffu, accA, 1);
    accA += __shfl_xor_sync(0xffffffffu, accA, 2);
    accB += __shfl_xor_sync(0xffffffffu, accB, 1);
    accB += __shfl_xor_sync(0xffffffffu, accB, 2);
    if (active && c == 0) {
      sRed[h * 128 + rowA] = accA;
      sRed[h * 128 + rowB] = accB;
    }
    q4_consumer_bar();
    for (int i = tid; i < rows_per_unit; i += kQConsumers) {
      const int n = row0 + i;
      if (n < N) y[n] = __half_as_ushort(__float2half_rn(sRed[i] + sRed[128 + i]));
    }
    q4_consumer_bar();
  }
}

}  // namespace

namespace {

int q4_sm_count() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

struct Q4Plan {
  int T = 0, nunits = 0, stages = 0;
};

// Units of T tiles (16 rows each) so that the units spread over the SMs; the deepest ring
// that fits beside x.
Q4Plan q4_plan(int N, int K, int sms) {
  Q4Plan p;
  if (K % kQChunkK != 0 || N <= 0 || sms <= 0) return p;
  const int tiles = (N + 15) / 16;
  int T = (tiles + sms - 1) / sms;
  if (T > kQMaxTiles) T = kQMaxTiles;
  const uint32_t fixed = Q4Layout(T, K, 0).total;
  if (fixed >= kQSmem) return p;
  int stages = static_cast<int>((kQSmem - fixed) / Q4Layout(T, K, 0).stage_bytes);
  if (stages > kQMaxStages) stages = kQMaxStages;
  if (stages < 2) return p;
  p.T = T;
  p.nunits = (tiles + T - 1) / T;
  p.stages = stages;
  return p;
}

}  // namespace

bool q4b32_tc_supports(int N, int K) { return q4_plan(N, K, q4_sm_count()).T > 0; }

cudaError_t launch_q4b32_gemv_tc(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                                 uint16_t* y, int N, int K, uint32_t* status, uint64_t limit_ns,
                                 cudaStream_t stream) {
  const int sms = q4_sm_count();
  const Q4Plan plan = q4_plan(N, K, sms);
  if (plan.T == 0) return cudaErrorNotSupported;
  Q4Maps maps;
  cudaError_t e = encode_tensor_map(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                            static_cast<uint64_t>(K) / 2, static_cast<uint64_t>(N),
                            static_cast<uint64_t>(K) / 2, kQBoxK / 2,
                            static_cast<uint32_t>(16 * plan.T), CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_tensor_map(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales,
                static_cast<uint64_t>(K) / 32, static_cast<uint64_t>(N),
                static_cast<uint64_t>(K) / 16, kQChunkK / 32, static_cast<uint32_t>(16 * plan.T),
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  const uint32_t smem = Q4Layout(plan.T, K, plan.stages).total + 1024u;
  e = set_max_dynamic_smem(reinterpret_cast<const void*>(q4b32_gemv_tc_kernel),
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = plan.nunits < sms ? plan.nunits : sms;
  return launch_with_pdl(q4b32_gemv_tc_kernel, dim3(static_cast<unsigned>(grid)),
                         dim3(kQThreads), smem, stream, maps, x, y, N, K, plan.T, plan.nunits,
                         plan.stages, status, limit_ns);
}

}  // namespace w4k
