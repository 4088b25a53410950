// W8A16 GEMV on a TMA ring: y[n] = s[n] * sum_k q[n, k] x[k] ("Quantization and GEMV",
// exercise 1: symmetric per-row INT8 codes, the row's fp32 scale once after the sum).
//
// The structure of the 4-bit-float ring kernel (fp4_gemv_tc_kernel), for one byte per weight:
//   * a producer warp streams 512-k chunks of a unit of 16 T rows by TMA: four 128-byte-wide
//     boxes of codes with the 128-byte swizzle; no scales travel with the codes;
//   * T x P consumer warps, warp (t, p) taking tile t and the 32-k blocks p, p + P, ... of
//     every chunk; lane (gq, c) reads the 8 codes k = 32 b + 8 c .. + 7 of rows gq and gq + 8
//     (one 8-byte load each: the rows' 16-byte units sit at unit ^ (row mod 8), so a warp's
//     loads hit every bank twice, the minimum for 256 bytes);
//   * a word of four codes becomes two FP16 pairs (1152 + q) with one LOP3 (q + 128, the
//     sign bit flipped) and two PRMTs placing each byte under the FP16 exponent of 1024, exact;
//   * x is FP16 under one power of two for the whole vector (largest |x| in [2^14, 2^15)), so
//     the MMAs (m16n8k16, x in the n8 columns) accumulate D = 2^e sum (1152 + q) x over all of
//     K in four independent chains, and y = s 2^-e (D - 1152 X) with X = 2^e sum_k x once
//     per CTA; the P parts of a row are added in a fixed order.
#include "common.cuh"
#include "fp4_common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kEMaxWarps = 24;
constexpr int kEBoxK = 128;             // 128 code bytes per row: one 128-byte swizzle row
constexpr int kEChunkK = 512;           // four code boxes per chunk
constexpr int kEBlocks = kEChunkK / 32; // 32-k blocks per chunk
constexpr int kEMaxStages = 8;
constexpr uint32_t kESmem = 227u * 1024u - 1024u;  // the base is aligned up to 1024 B

struct ELayout {
  uint32_t box_bytes, stage_bytes, red_off, cst_off, x_off, bar_off, total;
  __host__ __device__ ELayout(int T, int K, int stages) {
    box_bytes = 2048u * static_cast<uint32_t>(T);  // 16 T rows x 128 B
    stage_bytes = 4u * box_bytes;
    red_off = static_cast<uint32_t>(stages) * stage_bytes;  // [P][16 T] fp32
    cst_off = red_off + 16u * kEMaxWarps * 4u;               // {1152 X, 2^-e}
    x_off = (cst_off + 16u + 15u) & ~15u;                    // [K] FP16
    bar_off = (x_off + static_cast<uint32_t>(K) * 2u + 7u) & ~7u;
    total = bar_off + 2u * kEMaxStages * 8u + 16u;
  }
};

template <int NT>
__device__ __forceinline__ void e_consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

__device__ __forceinline__ uint2 e_lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// FP16 pairs (1152 + q0, 1152 + q1) and (1152 + q2, 1152 + q3) of the four signed codes of w.
__device__ __forceinline__ void e_int8_pairs(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;  // two's complement byte q -> q + 128
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}

template <int T, int P>
__global__ void __launch_bounds__(T * P * 32 + 32, 1)
    w8a16_gemv_tc_kernel(const __grid_constant__ CUtensorMap codes_map,
                         const uint16_t* __restrict__ x, const float* __restrict__ scales,
                         uint16_t* __restrict__ y, int N, int K, int nunits, int stages,
                         uint32_t* __restrict__ status, uint64_t limit_ns) {
  constexpr int W = T * P;
  constexpr int NC = W * 32;
  constexpr int NB = kEBlocks / P;
  constexpr int ROWS = 16 * T;
  static_assert(kEBlocks % P == 0 && W <= kEMaxWarps, "bad warp split");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const ELayout L(T, K, stages);
  float* sRed = reinterpret_cast<float*>(smem + L.red_off);  // [P][ROWS]
  float* sCst = reinterpret_cast<float*>(smem + L.cst_off);  // {1152 X, 2^-e}
  uint4* sX = reinterpret_cast<uint4*>(smem + L.x_off);      // [K/8] FP16, natural order
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kEMaxStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kEMaxStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kchunks = K / kEChunkK;

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
      tma_prefetch_desc(&codes_map);
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
          mbar_arrive_expect_tx(&full[s], L.stage_bytes);
#pragma unroll
          for (int bx = 0; bx < 4; ++bx)
            tma_load_2d(buf + bx * L.box_bytes, &codes_map, &full[s], kc * kEChunkK + bx * kEBoxK,
                        row0);
        }
      }
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
    // x (BF16) -> FP16 in natural order under one power of two; X = sum of the scaled x.
    // With one segment per thread (K <= 8 NC) the segment stays in registers.
    const int segs = K / 8;
    const bool one = segs <= NC;
    float v1[8] = {};
    float amax = 0.f;
    if (one) {
      if (tid < segs) f_bf16x8(__ldg(reinterpret_cast<const uint4*>(x) + tid), v1);
#pragma unroll
      for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(v1[q]));
    } else {
      for (int R = tid; R < segs; R += NC) {
        float v[8];
        f_bf16x8(__ldg(reinterpret_cast<const uint4*>(x) + R), v);
#pragma unroll
        for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(v[q]));
      }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) sRed[warp] = amax;
    e_consumer_bar<NC>();
    amax = sRed[0];
#pragma unroll
    for (int w = 1; w < W; ++w) amax = fmaxf(amax, sRed[w]);
    const int e = f_x_exponent(amax);
    const float sc = f_pow2(e);
    float xs = 0.f;  // this thread's sum of the FP16 x it stores (exact values)
    auto store = [&](int R, const float (&v)[8]) {
      const uint4 h = f_f16x8(v, sc);
      sX[R] = h;
      const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[i]));
        xs += f.x + f.y;
      }
    };
    if (one) {
      if (tid < segs) store(tid, v1);
    } else {
      for (int R = tid; R < segs; R += NC) {
        float v[8];
        f_bf16x8(__ldg(reinterpret_cast<const uint4*>(x) + R), v);
        store(R, v);
      }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) xs += __shfl_xor_sync(0xffffffffu, xs, o);
    e_consumer_bar<NC>();  // every warp has read sRed[0 .. W)
    if (lane == 0) sRed[warp] = xs;
    e_consumer_bar<NC>();
    if (tid == 0) {
      float X = 0.f;
      for (int w = 0; w < W; ++w) X += sRed[w];  // fixed order
      sCst[0] = 1152.0f * X;
      sCst[1] = f_pow2(-e);
    }
    e_consumer_bar<NC>();
  }

  const int gq = lane >> 2, c = lane & 3;
  const int t = warp % T, p = warp / T;
  const uint32_t rowA = static_cast<uint32_t>(16 * t + gq);  // rowB = rowA + 8
  // Per block r of this warp (block j = p + P r of a chunk, box j / 4): the offset of row
  // rowA's 8 codes in a stage and of this lane's 16 bytes of x in a chunk.
  uint32_t code_off[NB], x_off[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    const uint32_t j = static_cast<uint32_t>(p + P * r);
    const uint32_t unit = 2u * (j & 3u) + static_cast<uint32_t>(c >> 1);  // 16-byte unit
    code_off[r] = (j >> 2) * L.box_bytes + rowA * 128u +
                  ((unit ^ static_cast<uint32_t>(gq)) << 4) + 8u * static_cast<uint32_t>(c & 1);
    x_off[r] = (j * 4u + static_cast<uint32_t>(c)) * 16u;
  }
  const uint32_t ring_base = smem_addr(smem);
  const uint32_t xbase = smem_addr(sX);
  const float corr = sCst[0], u2 = sCst[1];
  int s = 0;
  uint32_t phase = 0u;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const int row0 = u * ROWS;
    float dacc[4][4] = {};
    for (int kc = 0; kc < kchunks; ++kc) {
      const bool landed = mbar_wait_bounded(&full[s], phase, abort_flag, status, limit_ns);
      const uint32_t buf = ring_base + static_cast<uint32_t>(s) * L.stage_bytes;
      const uint32_t xk = xbase + static_cast<uint32_t>(kc) * (kEBlocks * 64u);
      if (landed) {
#pragma unroll
        for (int r = 0; r < NB; ++r) {
          const uint2 wa = e_lds64(buf + code_off[r]);
          const uint2 wb = e_lds64(buf + code_off[r] + 1024u);  // row + 8
          const uint4 ex = f_lds128(xk + x_off[r]);
          uint32_t a0, a2, a4, a6, b0, b2, b4, b6;
          e_int8_pairs(wa.x, a0, a2);  // k 8c + 0, 1 | 8c + 2, 3
          e_int8_pairs(wa.y, a4, a6);  // k 8c + 4, 5 | 8c + 6, 7
          e_int8_pairs(wb.x, b0, b2);
          e_int8_pairs(wb.y, b4, b6);
          f_mma(dacc[2 * (r & 1)], a0, b0, a2, b2, ex.x, ex.y);
          f_mma(dacc[2 * (r & 1) + 1], a4, b4, a6, b6, ex.z, ex.w);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == stages) {
        s = 0;
        phase ^= 1u;
      }
    }
    const float accA = (dacc[0][0] + dacc[1][0]) + (dacc[2][0] + dacc[3][0]);
    const float accB = (dacc[0][2] + dacc[1][2]) + (dacc[2][2] + dacc[3][2]);
    if (c == 0) {
      sRed[p * ROWS + static_cast<int>(rowA)] = accA;
      sRed[p * ROWS + static_cast<int>(rowA) + 8] = accB;
    }
    e_consumer_bar<NC>();
    for (int i = tid; i < ROWS; i += NC) {
      const int n = row0 + i;
      if (n < N) {
        float v = sRed[i];
#pragma unroll
        for (int q = 1; q < P; ++q) v += sRed[q * ROWS + i];
        // the P parts' sums together hold 1152 X once
        y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(__ldg(scales + n) * u2 * (v - corr)));
      }
    }
    e_consumer_bar<NC>();
  }
}

struct ECfg {
  int T, P;
};
constexpr ECfg kECfgs[] = {{1, 16}, {2, 8}, {3, 8}, {4, 4}, {6, 4}, {8, 2}, {12, 2}};
constexpr int kENumCfgs = static_cast<int>(sizeof(kECfgs) / sizeof(kECfgs[0]));

struct EPlan {
  int cfg = -1, nunits = 0, stages = 0;
};

// The smallest unit (T tiles of 16 rows) that covers N in one wave of SMs, else the largest;
// a smaller unit (several per CTA) when that one leaves fewer than four stages beside x.
EPlan e_plan(int N, int K, int sms) {
  EPlan p;
  if (K % kEChunkK != 0 || N <= 0 || sms <= 0) return p;
  const int tiles = (N + 15) / 16;
  const int need = (tiles + sms - 1) / sms;
  int ci = 0;
  while (ci + 1 < kENumCfgs && kECfgs[ci].T < need) ++ci;
  auto stages_of = [&](int c) {
    const uint32_t fixed = ELayout(kECfgs[c].T, K, 0).total;
    const uint32_t stage = ELayout(kECfgs[c].T, K, 0).stage_bytes;
    const int st = fixed < kESmem ? static_cast<int>((kESmem - fixed) / stage) : 0;
    return st > kEMaxStages ? kEMaxStages : st;
  };
  int best = -1;
  for (int c = ci; c >= 0; --c) {
    const int st = stages_of(c);
    if (st >= 2 && best < 0) best = c;
    if (st >= 4) {
      best = c;
      break;
    }
  }
  if (best < 0) return p;
  p.cfg = best;
  p.nunits = (tiles + kECfgs[best].T - 1) / kECfgs[best].T;
  p.stages = stages_of(best);
  return p;
}

template <int T, int P>
cudaError_t launch_e(const uint16_t* x, const int8_t* q, const float* scales, uint16_t* y, int N,
                     int K, const EPlan& plan, int sms, uint32_t* status, uint64_t limit_ns,
                     cudaStream_t stream) {
  CUtensorMap map;
  cudaError_t e = encode_tensor_map(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, q,
                                    static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                                    static_cast<uint64_t>(K), kEBoxK,
                                    static_cast<uint32_t>(16 * T), CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const uint32_t smem = ELayout(T, K, plan.stages).total + 1024u;
  auto kern = w8a16_gemv_tc_kernel<T, P>;
  e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = plan.nunits < sms ? plan.nunits : sms;
  return launch_with_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(T * P * 32 + 32), smem,
                         stream, map, x, scales, y, N, K, plan.nunits, plan.stages, status,
                         limit_ns);
}

}  // namespace

bool w8a16_tc_supports(int N, int K) { return e_plan(N, K, device_sm_count()).cfg >= 0; }

cudaError_t launch_w8a16_gemv_tc(const uint16_t* x, const int8_t* q, const float* scales,
                                 uint16_t* y, int N, int K, uint32_t* status,
                                 uint64_t wait_limit_ns, cudaStream_t stream) {
  const int sms = device_sm_count();
  const EPlan plan = e_plan(N, K, sms);
  switch (plan.cfg) {
    case 0: return launch_e<1, 16>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    case 1: return launch_e<2, 8>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    case 2: return launch_e<3, 8>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    case 3: return launch_e<4, 4>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    case 4: return launch_e<6, 4>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    case 5: return launch_e<8, 2>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    case 6: return launch_e<12, 2>(x, q, scales, y, N, K, plan, sms, status, wait_limit_ns, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace w4k
