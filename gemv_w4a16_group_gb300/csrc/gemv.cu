// CUDA-core W4A16 GEMV for small M: y[m, n] = sum_g ( s[g,n] * sum_{k in g} x[m,k] q[n,k]
//                                                     + min[g,n] * sum_{k in g} x[m,k] ).
//
// The factorised per-group form is the one the pages give for their M = 1 kernel ("Low-
// Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", "How the measurements were
// taken": a GEMV that "sums s x sum x.q + min x sum x per group in FP32 without tensor
// cores"). The work split follows "Quantization and GEMV", "Writing a GEMV kernel"
// (128-bit reads, K split across the block, warp-shuffle reduction), adapted to the K/8 x N
// packed layout in which N is contiguous.
//
// At M = 1 the whole matrix is only a few times the bytes that must be in flight to cover
// DRAM latency, so the kernel is built to have almost all of it requested at once:
//
//   * persistent grid, one CTA per SM; CTA c owns the 32-column slabs c, c + G, c + 2G, ...
//     (G = grid size) over the whole of K;
//   * a producer warp streams the CTA's slabs in chunks of 32 columns x 2048 k (32 KB of
//     packed words + 2 KB of scales and minimums) into a 6-deep shared-memory ring with
//     TMA, so up to 204 KB per SM are in flight from the first microsecond;
//   * 16 consumer warps take one group (16 packed rows) of a chunk each; lane (rs, cq)
//     reads 4 columns x 4 rows with 16-byte shared loads (a warp reads 4 full 128-byte
//     rows: no bank conflicts);
//   * codes become exact numbers with a fixed offset (mantissa trick, see common.cuh); the
//     offsets and the min term are removed per quarter-group with sums of x computed once
//     per CTA while the first chunks are in flight;
//   * per slab, partial sums are reduced over row phases with shuffles and over warps
//     through shared memory in a fixed order (deterministic, no atomics).
//
// Inner product variants (`VARIANT`): 0 = codes -> fp32 + packed fp32x2 FMA; 1 = codes ->
// BF16 pairs + mixed BF16 x BF16 -> fp32 FMA (fewer instructions per code).
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kSlabCols = 32;
constexpr int kChunkRows = 256;                          // packed rows (2048 k) per chunk
constexpr int kChunkGroups = kChunkRows / 16;            // 16 groups of 128
constexpr uint32_t kChunkWordBytes = kChunkRows * kSlabCols * 4;   // 32 KB
constexpr uint32_t kChunkRowBytes = kChunkGroups * kSlabCols * 2;  // 1 KB (scales or mins)
constexpr uint32_t kChunkBytes = kChunkWordBytes + 2 * kChunkRowBytes;
constexpr int kStages = 6;
constexpr int kMaxRows = 2;

template <int MR>
struct GemvSmem {
  static constexpr uint32_t ring = kStages * kChunkBytes;
  static constexpr uint32_t red_off = ring;                         // [kConsumerWarps][MR][32]
  static constexpr uint32_t xc_off = red_off + kConsumerWarps * MR * 32 * 4;
  __host__ __device__ static uint32_t bar_off(int K) { return xc_off + 2u * MR * (K >> 5) * 4u; }
  __host__ __device__ static uint32_t total(int K) { return bar_off(K) + (2 * kStages) * 8 + 16; }
};

// acc += sum_j (128 + q_j) * x_j for the 8 codes of `w` (mixed BF16 x BF16 -> fp32).
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

struct GemvMaps {
  CUtensorMap qw;      // int32 [K/8, N], box {32, 256}
  CUtensorMap scales;  // bf16 [K/128, N], box {32, 16}
  CUtensorMap mins;    // bf16 [K/128, N], box {32, 16}
};

template <int MR, int VARIANT>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_w4a16_kernel(const __grid_constant__ GemvMaps maps, const uint16_t* __restrict__ x,
                      uint16_t* __restrict__ y, int M, int N, int K, uint32_t* __restrict__ status,
                      uint64_t limit_ns) {
  using L = GemvSmem<MR>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* sRed = reinterpret_cast<float*>(smem + L::red_off);
  const int Q = K >> 5;  // quarter-groups of 32 k
  float* sX = reinterpret_cast<float*>(smem + L::xc_off);  // [MR][Q]
  float* sC = sX + MR * Q;                                  // [MR][Q]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bar_off(K));
  uint64_t* empty = full + kStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = K >> 7;
  const int kchunks = (K / 8 + kChunkRows - 1) / kChunkRows;
  const int nslab = (N + kSlabCols - 1) / kSlabCols;
  const int my_slabs = (nslab - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x;
  const int total = my_slabs * kchunks;
  const int m0 = blockIdx.y * MR;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      tma_prefetch_desc(&maps.qw);
      int issued = 0;
      for (int j = 0; j < total; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait_bounded(&empty[s], ((j / kStages) - 1) & 1u, abort_flag, status, limit_ns))
          break;
        const int slab = blockIdx.x + (j / kchunks) * gridDim.x;
        const int kc = j % kchunks;
        uint8_t* buf = smem + s * kChunkBytes;
        mbar_arrive_expect_tx(&full[s], kChunkBytes);
        tma_load_2d(buf, &maps.qw, &full[s], slab * kSlabCols, kc * kChunkRows);
        tma_load_2d(buf + kChunkWordBytes, &maps.scales, &full[s], slab * kSlabCols,
                    kc * kChunkGroups);
        tma_load_2d(buf + kChunkWordBytes + kChunkRowBytes, &maps.mins, &full[s],
                    slab * kSlabCols, kc * kChunkGroups);
        ++issued;
      }
      // Stay until this CTA's last copies have landed (bounded), so none is in flight
      // when the CTA exits, whatever the consumers did.
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % kStages);
        volatile uint32_t no_abort = 0u;
        mbar_wait_bounded(&full[s], (last / kStages) & 1u, &no_abort, status, limit_ns);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  // Per quarter-group sums of x (X) and of offset-weighted x (C), while chunks land.
  for (int i = tid; i < MR * Q; i += kConsumers) {
    const int mm = i / Q, q = i - mm * Q;
    float X = 0.f, C = 0.f;
    if (m0 + mm < M) {
      const uint4* xp =
          reinterpret_cast<const uint4*>(x + static_cast<size_t>(m0 + mm) * K + q * 32);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 u = __ldg(xp + v);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float lo = bf16_bits_to_f32(wd[h] & 0xFFFFu);      // even k
          const float hi = __uint_as_float(wd[h] & 0xFFFF0000u);  // odd k
          X += lo + hi;
          if (VARIANT == 0)
            C += code_offset_f32(0) * lo + code_offset_f32(1) * hi;
          else
            C += 128.0f * (lo + hi);
        }
      }
    }
    sX[i] = X;
    sC[i] = C;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");

  const int cq = lane & 7, rs = lane >> 3;
  float yacc[4][MR];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int mm = 0; mm < MR; ++mm) yacc[c][mm] = 0.f;

  for (int j = 0; j < total; ++j) {
    const int s = j % kStages;
    const int kc = j % kchunks;
    const int g = kc * kChunkGroups + warp;  // this warp's group in the chunk
    // On an expired wait every warp keeps walking the chunk list without computing, so
    // all consumer warps still meet at the per-slab barriers below.
    const bool landed = mbar_wait_bounded(&full[s], (j / kStages) & 1u, abort_flag, status, limit_ns);
    const uint8_t* buf = smem + s * kChunkBytes;
    if (landed && g < G) {
      const uint4* wrow = reinterpret_cast<const uint4*>(buf) + (warp * 16 + rs * 4) * 8 + cq;
      uint4 wr[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) wr[t] = wrow[t * 8];
      const uint2 s2 = *reinterpret_cast<const uint2*>(buf + kChunkWordBytes + warp * 64 + cq * 8);
      const uint2 m2 = *reinterpret_cast<const uint2*>(buf + kChunkWordBytes + kChunkRowBytes +
                                                       warp * 64 + cq * 8);
      float acc[4][MR], acc_odd[4][MR];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) acc[c][mm] = acc_odd[c][mm] = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int r = g * 16 + rs * 4 + t;  // global packed row
        const uint32_t wd[4] = {wr[t].x, wr[t].y, wr[t].z, wr[t].w};
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) {
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (m0 + mm < M)
            xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m0 + mm) * K + 8 * r));
          if (VARIANT == 0) {
            const float2 x01 = make_float2(bf16_bits_to_f32(xv.x & 0xFFFFu), __uint_as_float(xv.x & 0xFFFF0000u));
            const float2 x23 = make_float2(bf16_bits_to_f32(xv.y & 0xFFFFu), __uint_as_float(xv.y & 0xFFFF0000u));
            const float2 x45 = make_float2(bf16_bits_to_f32(xv.z & 0xFFFFu), __uint_as_float(xv.z & 0xFFFF0000u));
            const float2 x67 = make_float2(bf16_bits_to_f32(xv.w & 0xFFFFu), __uint_as_float(xv.w & 0xFFFF0000u));
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float f[8];
              codes_to_f32_offset(wd[c], f);
              float2 a = make_float2(acc[c][mm], acc_odd[c][mm]);
              a = __ffma2_rn(make_float2(f[0], f[1]), x01, a);
              a = __ffma2_rn(make_float2(f[2], f[3]), x23, a);
              a = __ffma2_rn(make_float2(f[4], f[5]), x45, a);
              a = __ffma2_rn(make_float2(f[6], f[7]), x67, a);
              acc[c][mm] = a.x;
              acc_odd[c][mm] = a.y;
            }
          } else {
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
        const float sc = bf16_bits_to_f32(sbits), mn = bf16_bits_to_f32(mbits);
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) {
          const float a = acc[c][mm] + acc_odd[c][mm];
          yacc[c][mm] = fmaf(sc, a - sC[mm * Q + q], fmaf(mn, sX[mm * Q + q], yacc[c][mm]));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (kc == kchunks - 1) {
      // This slab is done: reduce over row phases, then over warps, store.
      const int slab = blockIdx.x + (j / kchunks) * gridDim.x;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int mm = 0; mm < MR; ++mm) {
          float v = yacc[c][mm];
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          yacc[c][mm] = 0.f;
          if (rs == 0) sRed[(warp * MR + mm) * 32 + cq * 4 + c] = v;
        }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
      if (tid < MR * 32) {
        const int mm = tid >> 5, col = tid & 31;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) v += sRed[(w * MR + mm) * 32 + col];
        const int nn = slab * kSlabCols + col;
        if (m0 + mm < M && nn < N)
          y[static_cast<size_t>(m0 + mm) * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    }
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

template <int MR, int VARIANT>
cudaError_t launch_mr(const GemvMaps& maps, const uint16_t* x, uint16_t* y, int M, int N, int K,
                      uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  using L = GemvSmem<MR>;
  const uint32_t smem = L::total(K);
  auto kern = gemv_w4a16_kernel<MR, VARIANT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int nslab = (N + kSlabCols - 1) / kSlabCols;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  dim3 grid(static_cast<unsigned>(nslab < sms ? nslab : sms), (M + MR - 1) / MR);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  kern<<<grid, kThreads, smem, stream>>>(maps, x, y, M, N, K, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace

int gemv_max_rows() { return kMaxRows; }

// The per-CTA sums of x must fit in shared memory next to the ring.
bool gemv_supports(int M, int K) {
  return M <= kMaxRows && GemvSmem<kMaxRows>::total(K) <= 227u * 1024u;
}

cudaError_t launch_w4a16_gemv(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                              const uint16_t* mins, uint16_t* y, int M, int N, int K, int variant,
                              uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
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
  if (M <= 1) {
    return variant == 1 ? launch_mr<1, 1>(maps, x, y, M, N, K, status, limit_ns, stream)
                        : launch_mr<1, 0>(maps, x, y, M, N, K, status, limit_ns, stream);
  }
  return variant == 1 ? launch_mr<2, 1>(maps, x, y, M, N, K, status, limit_ns, stream)
                      : launch_mr<2, 0>(maps, x, y, M, N, K, status, limit_ns, stream);
}

}  // namespace w4k
