// W4A16 GEMV / skinny kernel for small M (M <= 8): weights staged by TMA, dequantised in
// registers, the multiply-adds done by BF16 mma.sync fragments built straight from the
// packed words.
//
//   y[m, n] = sum_g ( s[g,n] * sum_{k in g} x[m,k] q[n,k] + min[g,n] * sum_{k in g} x[m,k] )
//
// The factorised per-group form is the one the pages give for their M = 1 kernel ("Low-
// Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", "How the measurements were
// taken": it "sums s x sum x.q + min x sum x per group in FP32"). The work split follows
// "Quantization and GEMV", "Writing a GEMV kernel": 128-bit reads, K split across warps
// (and, for balance, across thread blocks), a shuffle/shared-memory reduction, adapted to
// the K/8 x N packed layout (N contiguous).
//
// Why the tensor core in a GEMV: at 4 bits the unpacking is a real share of the issue
// slots ("Where the time goes at M = 1"). A CUDA-core inner product costs one FMA per code
// plus the unpacking; here one m16n8k16 instruction takes 256 codes, so a packed word
// costs 3 shifts + 4 LOP3 (code pairs ORed into BF16 mantissas: 0x4300 | q = 128 + q)
// plus a quarter of an MMA, and M up to 8 costs the same as M = 1. The kernel stays bound
// by HBM.
//
// Launch shape (measured on GB300: the TMA engine is limited by box rows, so boxes must be
// wide; and a launch must overlap the previous one to stream at full bandwidth):
//   * work units = (slab of 128 columns, k-range); with a workspace the K range of a slab
//     is split so that the units balance over the SMs; persistent grid (<= one CTA per
//     SM), CTA c takes units c, c + G, ...;
//   * a producer warp streams each unit in chunks of 128 columns x 512 k (64 rows of 512 B:
//     32 KB of packed words + 2 KB of scales and minimums) into a shared-memory ring with
//     TMA (~200 KB in flight per SM at M = 1). It issues its weight loads before it waits
//     for the previous kernel on the stream (programmatic dependent launch);
//   * 16 consumer warps: warp w takes column quarter w % 4 (32 columns) of group w / 4 of
//     each chunk. Lane (gq, c) = (lane / 4, lane % 4) reads packed row 4b + c of block b
//     (b = 0..3) and columns 4gq..4gq+3 with one 16-byte shared load; its four words fill
//     the A fragments of two 16-row MMA tiles (tile t: rows gq <- column 4gq + 2t,
//     gq + 8 <- column 4gq + 2t + 1);
//   * the k order inside an MMA is permuted so that code pairs (q_j, q_{j+4}) -- one LOP3
//     each -- are fragment pairs; x is stored once per CTA in shared memory in the matching
//     order (B fragments);
//   * per group the fp32 accumulator D = sum (128 + q) x is folded into y with
//     y += s * D + (min - 128 s) * sum_g x, the group sums of x computed once per CTA;
//   * per unit the 4 warps of a column quarter are summed in a fixed order; a split slab
//     writes fp32 partials and the last CTA to arrive (arrival counter) sums them in split
//     order (deterministic, no float atomics) and resets the counter.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kSlabCols = 128;
constexpr int kChunkRows = 64;                                     // packed rows (512 k)
constexpr int kChunkGroups = kChunkRows / 16;                      // 4 groups of 128
constexpr uint32_t kChunkWordBytes = kChunkRows * kSlabCols * 4;   // 32 KB
constexpr uint32_t kChunkRowBytes = kChunkGroups * kSlabCols * 2;  // 1 KB (scales or mins)
constexpr uint32_t kChunkBytes = kChunkWordBytes + 2 * kChunkRowBytes;
constexpr int kMaxRows = 8;

static_assert(kChunkGroups * (kSlabCols / 32) == kConsumerWarps, "one (group, quarter) per warp");

template <int MR>
struct GemvSmem {
  // Weights in flight per SM: 6 x 34 KB at M = 1, fewer stages as x grows with M.
  static constexpr int kStages = MR <= 1 ? 6 : MR <= 2 ? 5 : MR <= 4 ? 4 : 3;
  static constexpr uint32_t ring = kStages * kChunkBytes;
  static constexpr uint32_t red_off = ring;  // [kConsumerWarps][MR][32] floats
  static constexpr uint32_t xsum_off = red_off + kConsumerWarps * MR * 32 * 4;
  // x in B-fragment order: per packed row R and batch row m, 16 bytes
  // {(x0, x4), (x1, x5), (x2, x6), (x3, x7)} of x[m, 8R .. 8R + 8).
  __host__ __device__ static uint32_t xperm_off(int K) {
    return (xsum_off + MR * (K >> 7) * 4u + 15u) & ~15u;
  }
  // mbarriers need 8-byte alignment.
  __host__ __device__ static uint32_t bar_off(int K) { return xperm_off(K) + 2u * MR * K; }
  __host__ __device__ static uint32_t total(int K) { return bar_off(K) + (2 * kStages) * 8 + 16; }
};

// D += A (16x16, BF16) * B (16x8, BF16), fp32 accumulators; fragment layout of mma.sync
// m16n8k16 (row-major A, column-major B).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (128 + q_i, 128 + q_{i+4}) as a BF16 pair, for the 8 codes of `w`.
__device__ __forceinline__ void code_pairs(uint32_t w, uint32_t (&p)[4]) {
  p[0] = (w & 0x000F000Fu) | 0x43004300u;
  p[1] = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
  p[2] = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
  p[3] = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
}

struct GemvMaps {
  CUtensorMap qw;      // int32 [K/8, N], box {128, 64}
  CUtensorMap scales;  // bf16 [K/128, N], box {128, 4}
  CUtensorMap mins;    // bf16 [K/128, N], box {128, 4}
};

template <int MR>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_w4a16_kernel(const __grid_constant__ GemvMaps maps, const uint16_t* __restrict__ x,
                      uint16_t* __restrict__ y, int M, int N, int K, int splits,
                      float* __restrict__ ws_partial, uint32_t* __restrict__ ws_counter,
                      uint32_t* __restrict__ status, uint64_t limit_ns) {
  static_assert(MR <= 8, "one n8 tile of batch rows");
  using L = GemvSmem<MR>;
  constexpr int kStages = L::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  float* sRed = reinterpret_cast<float*>(smem + L::red_off);
  float* sXsum = reinterpret_cast<float*>(smem + L::xsum_off);       // [MR][G]
  uint4* sXperm = reinterpret_cast<uint4*>(smem + L::xperm_off(K));  // [K/8][MR]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bar_off(K));
  uint64_t* empty = full + kStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kStages);
  volatile uint32_t* last_flag = abort_flag + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = K >> 7;
  const int kchunks = (K / 8 + kChunkRows - 1) / kChunkRows;
  const int per_unit = (kchunks + splits - 1) / splits;  // chunks per k-range
  const int nslab = (N + kSlabCols - 1) / kSlabCols;
  const int nunits = nslab * splits;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0u;
    fence_barrier_init();
    pdl_launch_dependents();  // the next kernel may start streaming its own weights
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: weights only, no wait on the previous kernel -------
    if (lane == 0) {
      tma_prefetch_desc(&maps.qw);
      int j = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < nunits && !stop; u += gridDim.x) {
        const int slab = u / splits, kr = u - (u / splits) * splits;
        const int kc_end = min(kchunks, (kr + 1) * per_unit);
        for (int kc = kr * per_unit; kc < kc_end; ++kc, ++j) {
          const int s = j % kStages;
          if (j >= kStages && !mbar_wait_bounded(&empty[s], ((j / kStages) - 1) & 1u, abort_flag,
                                                 status, limit_ns)) {
            stop = true;
            break;
          }
          uint8_t* buf = smem + s * kChunkBytes;
          mbar_arrive_expect_tx(&full[s], kChunkBytes);
          tma_load_2d(buf, &maps.qw, &full[s], slab * kSlabCols, kc * kChunkRows);
          tma_load_2d(buf + kChunkWordBytes, &maps.scales, &full[s], slab * kSlabCols,
                      kc * kChunkGroups);
          tma_load_2d(buf + kChunkWordBytes + kChunkRowBytes, &maps.mins, &full[s],
                      slab * kSlabCols, kc * kChunkGroups);
        }
      }
      // Stay until this CTA's last copies have landed (bounded), so none is in flight
      // when the CTA exits, whatever the consumers did.
      const int issued = j;
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % kStages);
        volatile uint32_t no_abort = 0u;
        mbar_wait_bounded(&full[s], (last / kStages) & 1u, &no_abort, status, limit_ns);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  pdl_wait();  // x, y and the workspace may belong to the previous kernel on the stream
  // Group sums of x, one warp per (row, group), fixed reduction order.
  for (int it = warp; it < MR * G; it += kConsumerWarps) {
    const int mm = it / G, g = it - mm * G;
    float v = 0.f;
    if (mm < M) {
      const uint2 u2 = __ldg(reinterpret_cast<const uint2*>(
          x + static_cast<size_t>(mm) * K + g * 128 + lane * 4));
      v = (bf16_bits_to_f32(u2.x & 0xFFFFu) + __uint_as_float(u2.x & 0xFFFF0000u)) +
          (bf16_bits_to_f32(u2.y & 0xFFFFu) + __uint_as_float(u2.y & 0xFFFF0000u));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sXsum[it] = v;
  }
  // x in B-fragment order.
  for (int i = tid; i < (K >> 3) * MR; i += kConsumers) {
    const int R = i / MR, mm = i - R * MR;
    uint4 e = make_uint4(0u, 0u, 0u, 0u);
    if (mm < M) {
      const uint4 xv =
          __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(mm) * K + 8 * R));
      e.x = __byte_perm(xv.x, xv.z, 0x5410);  // (x0, x4)
      e.y = __byte_perm(xv.x, xv.z, 0x7632);  // (x1, x5)
      e.z = __byte_perm(xv.y, xv.w, 0x5410);  // (x2, x6)
      e.w = __byte_perm(xv.y, xv.w, 0x7632);  // (x3, x7)
    }
    sXperm[i] = e;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");

  const int gq = lane >> 2, c = lane & 3;
  const int q4 = warp & 3, gl = warp >> 2;  // column quarter, group within a chunk
  int j = 0;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const int slab = u / splits, kr = u - (u / splits) * splits;
    const int kc_end = min(kchunks, (kr + 1) * per_unit);
    // yacc[col jj][bb]: column slab*128 + 32*q4 + 4*gq + jj, batch row 2c + bb
    float yacc[4][2];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) yacc[jj][0] = yacc[jj][1] = 0.f;

    for (int kc = kr * per_unit; kc < kc_end; ++kc, ++j) {
      const int s = j % kStages;
      const int g = kc * kChunkGroups + gl;  // this warp's group
      // On an expired wait every warp keeps walking the chunk list without computing, so
      // all consumer warps still meet at the per-unit barriers below.
      const bool landed =
          mbar_wait_bounded(&full[s], (j / kStages) & 1u, abort_flag, status, limit_ns);
      const uint8_t* buf = smem + s * kChunkBytes;
      if (landed && g < G) {
        // Two independent accumulator chains (even / odd blocks).
        float d[2][2][4];  // [chain][tile t][fragment]
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int f = 0; f < 4; ++f) d[ch][t][f] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int rl = gl * 16 + b * 4 + c;  // packed row in the chunk
          const int R = kc * kChunkRows + rl;  // global packed row
          const uint4 wv = *reinterpret_cast<const uint4*>(buf + rl * 512 + q4 * 128 + gq * 16);
          // B fragment: batch row gq (zero where that row does not exist)
          const uint4 e =
              gq < MR ? sXperm[R * MR + (gq < MR ? gq : 0)] : make_uint4(0u, 0u, 0u, 0u);
          uint32_t p[4][4];
          code_pairs(wv.x, p[0]);
          code_pairs(wv.y, p[1]);
          code_pairs(wv.z, p[2]);
          code_pairs(wv.w, p[3]);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            // rows gq <- column 4gq + 2t, rows gq + 8 <- column 4gq + 2t + 1
            mma_bf16_16816(d[b & 1][t], p[2 * t][0], p[2 * t + 1][0], p[2 * t][1],
                           p[2 * t + 1][1], e.x, e.y);
            mma_bf16_16816(d[b & 1][t], p[2 * t][2], p[2 * t + 1][2], p[2 * t][3],
                           p[2 * t + 1][3], e.z, e.w);
          }
        }
        // Fold this group into y: y += s * D + (min - 128 s) * sum_g x, for batch rows that
        // exist (row 2c + bb; lanes whose rows do not exist add zeros).
        const uint32_t soff = kChunkWordBytes + gl * 256 + (q4 * 32 + gq * 4) * 2;
        const uint2 s2 = *reinterpret_cast<const uint2*>(buf + soff);
        const uint2 m2 = *reinterpret_cast<const uint2*>(buf + soff + kChunkRowBytes);
        const uint32_t sw[2] = {s2.x, s2.y}, mw[2] = {m2.x, m2.y};
        float xs[2];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int mrow = 2 * c + bb;
          xs[bb] = (bb < MR && mrow < MR) ? sXsum[(mrow < MR ? mrow : 0) * G + g] : 0.f;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float sc =
              bf16_bits_to_f32((jj & 1) ? (sw[jj >> 1] >> 16) : (sw[jj >> 1] & 0xFFFFu));
          const float mn =
              bf16_bits_to_f32((jj & 1) ? (mw[jj >> 1] >> 16) : (mw[jj >> 1] & 0xFFFFu));
          const float off = fmaf(-128.0f, sc, mn);
          const int t = jj >> 1, h = jj & 1;  // column 4gq + jj is tile t, fragment half h
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            if (bb >= MR) continue;  // no lane holds an existing row here
            const float dv = d[0][t][2 * h + bb] + d[1][t][2 * h + bb];
            yacc[jj][bb] = fmaf(sc, dv, fmaf(off, xs[bb], yacc[jj][bb]));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // Unit done: warp partials to shared memory, fixed-order sum over the 4 groups of
    // each column quarter.
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int mrow = 2 * c + bb;
        if (mrow < MR) sRed[(warp * MR + mrow) * 32 + gq * 4 + jj] = yacc[jj][bb];
      }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    for (int i = tid; i < MR * kSlabCols; i += kConsumers) {
      const int mm = i / kSlabCols, col = i - mm * kSlabCols, qq = col >> 5, c32 = col & 31;
      float v = 0.f;
#pragma unroll
      for (int gg = 0; gg < kChunkGroups; ++gg) v += sRed[((gg * 4 + qq) * MR + mm) * 32 + c32];
      const int nn = slab * kSlabCols + col;
      if (mm < M && nn < N) {
        if (splits == 1)
          y[static_cast<size_t>(mm) * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        else
          __stcg(ws_partial + (static_cast<size_t>(kr) * MR + mm) * N + nn, v);
      }
    }
    if (splits > 1) {
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
      if (tid == 0)
        *last_flag = (atomicAdd(ws_counter + slab, 1u) + 1u == static_cast<uint32_t>(splits));
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
      if (*last_flag) {
        __threadfence();
        for (int i = tid; i < MR * kSlabCols; i += kConsumers) {
          const int mm = i / kSlabCols, col = i - mm * kSlabCols;
          const int nn = slab * kSlabCols + col;
          if (mm < M && nn < N) {
            float v = 0.f;
            for (int z = 0; z < splits; ++z)
              v += __ldcg(ws_partial + (static_cast<size_t>(z) * MR + mm) * N + nn);
            y[static_cast<size_t>(mm) * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
          }
        }
        if (tid == 0) ws_counter[slab] = 0u;  // ready for the next call
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

cudaError_t encode(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

int mr_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

template <int MR>
cudaError_t launch_mr(const GemvMaps& maps, const uint16_t* x, uint16_t* y, int M, int N, int K,
                      const GemvSplit& split, uint32_t* status, uint64_t limit_ns,
                      cudaStream_t stream) {
  using L = GemvSmem<MR>;
  const uint32_t smem = L::total(K);
  auto kern = gemv_w4a16_kernel<MR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int nunits = ((N + kSlabCols - 1) / kSlabCols) * split.splits;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  dim3 grid(static_cast<unsigned>(nunits < sms ? nunits : sms));
  return launch_with_pdl(kern, grid, dim3(kThreads), smem, stream, maps, x, y, M, N, K,
                         split.splits, split.partial, split.counter, status, limit_ns);
}

}  // namespace

int gemv_max_rows() { return kMaxRows; }

// x in fragment order and its group sums must fit in shared memory next to the ring.
bool gemv_supports(int M, int K) {
  if (M < 1 || M > kMaxRows) return false;
  const uint32_t total = M <= 1 ? GemvSmem<1>::total(K)
                         : M <= 2 ? GemvSmem<2>::total(K)
                         : M <= 4 ? GemvSmem<4>::total(K)
                                  : GemvSmem<8>::total(K);
  return total <= 227u * 1024u;
}

GemvSplit gemv_split_plan(int M, int N, int K, size_t* bytes_needed) {
  GemvSplit plan;
  *bytes_needed = 0;
  const int sms = sm_count();
  const int nslab = (N + kSlabCols - 1) / kSlabCols;
  const int kchunks = (K / 8 + kChunkRows - 1) / kChunkRows;
  if (sms <= 0 || nslab >= sms) return plan;
  // About three units per SM; each k-range at least one chunk.
  int splits = (3 * sms + nslab - 1) / nslab;
  if (splits > kchunks) splits = kchunks;
  if (splits > 64) splits = 64;
  const int per_unit = (kchunks + splits - 1) / splits;
  splits = (kchunks + per_unit - 1) / per_unit;  // no empty k-range
  if (splits < 2) return plan;
  plan.splits = splits;
  const size_t counters = ((static_cast<size_t>(nslab) * 4 + 255) / 256) * 256;
  *bytes_needed = counters + static_cast<size_t>(splits) * mr_of(M) * N * 4;
  return plan;
}

cudaError_t launch_w4a16_gemv(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                              const uint16_t* mins, uint16_t* y, int M, int N, int K,
                              const GemvSplit& split, uint32_t* status, uint64_t limit_ns,
                              cudaStream_t stream) {
  GemvMaps maps;
  cudaError_t e;
  e = encode(&maps.qw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, static_cast<uint64_t>(N),
             static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N) * 4, kSlabCols, kChunkRows);
  if (e != cudaSuccess) return e;
  e = encode(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, scales, static_cast<uint64_t>(N),
             static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N) * 2, kSlabCols, kChunkGroups);
  if (e != cudaSuccess) return e;
  e = encode(&maps.mins, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, mins, static_cast<uint64_t>(N),
             static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N) * 2, kSlabCols, kChunkGroups);
  if (e != cudaSuccess) return e;
  switch (mr_of(M)) {
    case 1: return launch_mr<1>(maps, x, y, M, N, K, split, status, limit_ns, stream);
    case 2: return launch_mr<2>(maps, x, y, M, N, K, split, status, limit_ns, stream);
    case 4: return launch_mr<4>(maps, x, y, M, N, K, split, status, limit_ns, stream);
    default: return launch_mr<8>(maps, x, y, M, N, K, split, status, limit_ns, stream);
  }
}

}  // namespace w4k
