// W4A16 skinny matmul for a few batch rows (M <= 32): the GEMV's weight stream and FP16
// code pairs, with the batch rows in one to four n8 tiles of mma.sync m16n8k16.
//
//   y[m, n] = sum_g ( s[g,n] * sum_{k in g} x[m,k] q[n,k] + min[g,n] * sum_{k in g} x[m,k] )
//
// Same per-group factorised form as the M = 1 kernel ("Low-Precision Kernels: INT4, INT8 and
// FP8 Matmuls, Measured", "How the measurements were taken"). Between one row and the
// tensor-core tile GEMM the pages measure the weight-only kernel's gain holding to about 16
// rows and shrinking past that ("Batch size: where the 4-bit advantage ends"). With so few
// rows as tcgen05's N, every 128 x 16 weight tile would be rebuilt into tensor memory for
// only those rows (the tcgen05 kernel measured about twice this kernel's time at 16 rows).
// mma.sync keeps n8 granularity and the weights in registers: 4 MMAs per 256 codes and n8
// tile.
//
// Two kernels per call, chained by programmatic dependent launch:
//   * skinny_xprep_kernel converts x once per call into the caller's workspace: FP16 B
//     fragments xs [rows_pad][MRP] (16 bytes = the 8 x values of one packed row) with a
//     power-of-two scale 2^e per (row, group of 128) that puts the group's largest magnitude
//     in [2^14, 2^15) (exact: BF16 has 8 significant bits, FP16 11), the k slots of 16 q
//     getting x 2^(e-4); and per (group, row) the constants {X, T, U} = {sum x, 1024 sum_even
//     x + 64 sum_odd x, 2^-e} as float4 (even / odd: position of k in its packed word). Batch
//     row n of packed row R is stored at n ^ (2 ((R >> 1) & 3)): the lanes of one shared-
//     memory phase then read 8 distinct 16-byte chunks.
//   * w4a16_skinny_kernel: one CTA per SM, each owning 8 q or 8 (q + 1) consecutive columns
//     and all of K. A producer warp streams per 128 GPC k: the packed words (32-column
//     boxes, 128-byte swizzle), the scale and minimum rows, and that k range's x fragments and
//     constants (contiguous bulk copies), all on one stage barrier; weights are requested
//     before the wait on the prep kernel. 12 consumer warps: warp w takes column quarter
//     w % QW of group w / QW, lane (gq, c) rows 2c + (b & 1) + 8 (b >> 1) as in the GEMV; per
//     block 4 NT MMAs, per group the fold y += (s U) D + (min X - s T) for its 4 columns and
//     2 NT batch rows. Group partials meet in shared memory in a fixed order.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kSkConsumerWarps = 12;
constexpr int kSkThreads = kSkConsumerWarps * 32 + 32;
constexpr int kSkMaxStages = 4;
constexpr uint32_t kSkAlignPad = 1024u - 128u;  // the base is rounded up to 1024 B
constexpr uint32_t kSkSmemOneCta = 227u * 1024u;
constexpr uint32_t kSkSmemTwoCtas = 113u * 1024u;
constexpr int kSkPrepThreads = 256;

template <int NT, int QW>
struct SkShape {
  static constexpr int MRP = 8 * NT;                 // batch rows padded to whole n8 tiles
  static constexpr int W = 32 * QW;                  // slab width (columns)
  static constexpr int GPC = kSkConsumerWarps / QW;  // groups of 128 k per chunk
  static constexpr int ROWS = 16 * GPC;              // packed rows per chunk
  static constexpr uint32_t box_bytes = static_cast<uint32_t>(ROWS) * 128u;  // one quarter
  static constexpr uint32_t word_bytes = box_bytes * QW;
  static constexpr uint32_t row_bytes = static_cast<uint32_t>(GPC) * W * 2u;  // scale box
  static constexpr uint32_t row_stride = (row_bytes + 127u) & ~127u;
  static constexpr uint32_t x_bytes = static_cast<uint32_t>(ROWS) * MRP * 16u;
  static constexpr uint32_t c_bytes = static_cast<uint32_t>(GPC) * MRP * 16u;
  static constexpr uint32_t x_off = word_bytes + 2u * row_stride;
  static constexpr uint32_t tx_bytes = word_bytes + 2u * row_bytes + x_bytes + c_bytes;
  static constexpr uint32_t stage_bytes =
      (word_bytes + 2u * row_stride + x_bytes + c_bytes + 1023u) & ~1023u;
  // Group partials [MRP][W + 1] fp32: the extra column puts the rows 2c of a warp's lanes in
  // different banks.
  static constexpr int RED_LD = W + 1;
  static constexpr uint32_t red_bytes = (static_cast<uint32_t>(RED_LD) * MRP * 4u + 15u) & ~15u;
  static constexpr int kMinBlocks = NT == 1 ? 2 : 1;
  static_assert(GPC * QW == kSkConsumerWarps, "one (group, quarter) per consumer warp");
  static_assert(box_bytes % 1024u == 0u, "swizzled word boxes start on 1024-byte boundaries");
};

// Shared memory from the 1024-byte aligned base: the ring (stages x stage_bytes), the
// reduction buffer, the barriers; `total` includes the alignment pad.
template <int NT, int QW>
__host__ __device__ constexpr uint32_t sk_smem_total(int stages) {
  return static_cast<uint32_t>(stages) * SkShape<NT, QW>::stage_bytes +
         SkShape<NT, QW>::red_bytes + 2u * kSkMaxStages * 8u + 16u + kSkAlignPad;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// x [M][K] BF16 -> xs [rows_pad][MRP] FP16 fragments and cst [rows_pad / 16][MRP] constants.
// Thread i converts 16 consecutive x values (packed rows 2p and 2p + 1) of batch row
// n = i / half, p = i % half (half = rows_pad / 2); the 8 items of a group are adjacent
// lanes. Rows past K/8 and batch rows past M are written as zeros (constants {0, 0, 1, 0}).
template <int MRP>
__global__ void __launch_bounds__(kSkPrepThreads)
    skinny_xprep_kernel(const uint16_t* __restrict__ x, uint4* __restrict__ xs,
                        float4* __restrict__ cst, int M, int K, int rows_pad) {
  pdl_launch_dependents();  // the matmul may start streaming its weights
  pdl_wait();  // x may come from the previous kernel, which may also still read xs / cst
  const int half = rows_pad >> 1;
  const int items = MRP * half;
  const int i = static_cast<int>(blockIdx.x) * kSkPrepThreads + static_cast<int>(threadIdx.x);
  const int n = i / half, p = i - n * half, R = 2 * p;
  const int rows = K >> 3;
  uint4 xin[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
  if (i < items && n < M && R < rows) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(n) * K + 8 * R);
    xin[0] = __ldg(src);
    xin[1] = __ldg(src + 1);
  }
  float v[16];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t xw[4] = {xin[r].x, xin[r].y, xin[r].z, xin[r].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * r + 2 * h] = bf16_bits_to_f32(xw[h] & 0xFFFFu);
      v[8 * r + 2 * h + 1] = __uint_as_float(xw[h] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
  float sum_even = ((v[0] + v[2]) + (v[4] + v[6])) + ((v[8] + v[10]) + (v[12] + v[14]));
  float sum_odd = ((v[1] + v[3]) + (v[5] + v[7])) + ((v[9] + v[11]) + (v[13] + v[15]));
  // Every lane of the warp takes part (items past the end carry zeros): the grid is a
  // multiple of 32 threads and a group's 8 items never straddle a batch row (half % 8 == 0).
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    sum_even += __shfl_xor_sync(0xffffffffu, sum_even, o);
    sum_odd += __shfl_xor_sync(0xffffffffu, sum_odd, o);
  }
  if (i >= items) return;
  int e = 0;  // amax 2^e in [2^14, 2^15); an all-zero group keeps e = 0
  if (amax > 0.f) e = max(-100, min(100, 141 - static_cast<int>(__float_as_uint(amax) >> 23)));
  const float lo = pow2f(e), hi = pow2f(e - 4);
  const int slot = n ^ (2 * (p & 3));  // (R >> 1) & 3 = p & 3 for both rows of the item
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float* w = v + 8 * r;
    uint4 out;
    out.x = f16x2_bits(w[0] * lo, w[4] * lo);  // (x0, x4) 2^e
    out.y = f16x2_bits(w[1] * hi, w[5] * hi);  // (x1, x5) 2^(e-4)
    out.z = f16x2_bits(w[2] * lo, w[6] * lo);  // (x2, x6) 2^e
    out.w = f16x2_bits(w[3] * hi, w[7] * hi);  // (x3, x7) 2^(e-4)
    xs[static_cast<size_t>(R + r) * MRP + slot] = out;
  }
  if ((p & 7) == 0)
    cst[static_cast<size_t>(p >> 3) * MRP + n] =
        make_float4(sum_even + sum_odd, fmaf(1024.0f, sum_even, 64.0f * sum_odd), pow2f(-e), 0.f);
}

struct SkMaps {
  CUtensorMap qw;      // int32 [K/8, N], box {32, ROWS}, 128-byte swizzle
  CUtensorMap scales;  // bf16 (fp16 with a zero point) [K/128, N], box {W, GPC}
  CUtensorMap mins;    // bf16 minimums (fp16 zero points) [K/128, N], box {W, GPC}
};

// ZP: FP16 scales and zero points (w_hat = (q - z) s) instead of BF16 scales and minimums.
template <int NT, int QW, bool ZP>
__global__ void __launch_bounds__(kSkThreads, SkShape<NT, QW>::kMinBlocks)
    w4a16_skinny_kernel(const __grid_constant__ SkMaps maps, const uint4* __restrict__ xs,
                        const float4* __restrict__ cst, uint16_t* __restrict__ y, int M, int N,
                        int K, int stages, int col_q, int col_r, uint32_t* __restrict__ status,
                        uint64_t limit_ns) {
  using S = SkShape<NT, QW>;
  constexpr int GPC = S::GPC, ROWS = S::ROWS, MRP = S::MRP, NC = kSkConsumerWarps * 32;
  const int G = K >> 7;
  const int kchunks = (G + GPC - 1) / GPC;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  if (pad > kSkAlignPad) {  // base less than 128-byte aligned: report, touch nothing
    if (threadIdx.x == 0) atomicOr(status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t ring_bytes = static_cast<uint32_t>(stages) * S::stage_bytes;
  float* sRed = reinterpret_cast<float*>(smem + ring_bytes);  // [MRP][W + 1]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_bytes + S::red_bytes);
  uint64_t* empty = full + kSkMaxStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kSkMaxStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = static_cast<int>(blockIdx.x);
  const int col0 = 8 * (cta * col_q + min(cta, col_r));
  const int col_end = min(N, col0 + 8 * (col_q + (cta < col_r ? 1 : 0)));

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSkConsumerWarps);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  if (warp == kSkConsumerWarps) {
    // ---------------- producer warp ----------------
    if (lane == 0) {
      tma_prefetch_desc(&maps.qw);
      tma_prefetch_desc(&maps.scales);
      tma_prefetch_desc(&maps.mins);
      auto issue_weights = [&](int j) {
        const int s = j % stages;
        uint8_t* buf = smem + s * S::stage_bytes;
        mbar_arrive_expect_tx(&full[s], S::tx_bytes);
#pragma unroll
        for (int q = 0; q < QW; ++q)
          tma_load_2d(buf + q * S::box_bytes, &maps.qw, &full[s], col0 + 32 * q, j * ROWS);
        tma_load_2d(buf + S::word_bytes, &maps.scales, &full[s], col0, j * GPC);
        tma_load_2d(buf + S::word_bytes + S::row_stride, &maps.mins, &full[s], col0, j * GPC);
      };
      auto issue_x = [&](int j) {
        const int s = j % stages;
        uint8_t* buf = smem + s * S::stage_bytes + S::x_off;
        bulk_load(buf, xs + static_cast<size_t>(j) * ROWS * MRP, S::x_bytes, &full[s]);
        bulk_load(buf + S::x_bytes, cst + static_cast<size_t>(j) * GPC * MRP, S::c_bytes,
                  &full[s]);
      };
      // Weights of the first round before the wait on the prep kernel, x after it.
      const int first = stages < kchunks ? stages : kchunks;
      for (int j = 0; j < first; ++j) issue_weights(j);
      pdl_wait();
      for (int j = 0; j < first; ++j) issue_x(j);
      int issued = first;
      for (int j = first; j < kchunks; ++j) {
        const int s = j % stages;
        const uint32_t use = static_cast<uint32_t>(j / stages);
        if (!mbar_wait_bounded(&empty[s], (use - 1u) & 1u, abort_flag, status, limit_ns)) break;
        issue_weights(j);
        issue_x(j);
        issued = j + 1;
      }
      // Stay until this CTA's last copies have landed (bounded), so none is in flight when
      // the CTA exits, whatever the consumers did.
      for (int s = 0; s < stages && s < issued; ++s) {
        const int last = (issued - 1 - s) / stages;  // last use of stage s
        volatile uint32_t no_abort = 0u;
        mbar_wait_bounded(&full[s], static_cast<uint32_t>(last) & 1u, &no_abort, status,
                          limit_ns);
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  pdl_wait();  // y may still be read by a kernel before the prep kernel
  const int gq = lane >> 2, c = lane & 3;
  const int qq = warp % QW, gl = warp / QW;
  // Lane (gq, c) of block b reads packed row r_even + (b & 1) + 8 (b >> 1) of its group: words
  // from the swizzled quarter box (16-byte chunk gq of row r at gq ^ (r mod 8)), x of batch
  // row 8 j + gq from slot (8 j + gq) ^ 2c of that row (the prep kernel's layout).
  const uint32_t ring_base = smem_addr(smem);
  const int r_even = gl * 16 + 2 * c;
  const uint32_t w_even = static_cast<uint32_t>(qq) * S::box_bytes +
                          static_cast<uint32_t>(r_even * 128 + ((gq ^ (2 * c)) << 4));
  const uint32_t w_odd = static_cast<uint32_t>(qq) * S::box_bytes +
                         static_cast<uint32_t>((r_even + 1) * 128 + ((gq ^ (2 * c + 1)) << 4));
  const uint32_t x_lane =
      S::x_off + static_cast<uint32_t>((r_even * MRP + (gq ^ (2 * c))) * 16);
  // Scales / minimums of columns 4gq..4gq+3 of the quarter, row gl of the chunk's boxes.
  const uint32_t s_off =
      S::word_bytes + static_cast<uint32_t>((gl * S::W + qq * 32 + gq * 4) * 2);
  // Constants {X, T, U} of batch rows 8j + 2c and 8j + 2c + 1, group gl of the chunk.
  const uint32_t c_lane =
      S::x_off + S::x_bytes + static_cast<uint32_t>((gl * MRP + 2 * c) * 16);

  // yacc[j][col][r]: column 4gq + col of the quarter, batch row 8j + 2c + r.
  float yacc[NT][4][2];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int col = 0; col < 4; ++col) yacc[j][col][0] = yacc[j][col][1] = 0.f;

  int s = 0;
  uint32_t phase = 0u;
  for (int kc = 0; kc < kchunks; ++kc) {
    const int g = kc * GPC + gl;  // this warp's group
    // On an expired wait every warp keeps walking the chunks without computing, so all
    // consumer warps still meet at the barriers below.
    const bool landed = mbar_wait_bounded(&full[s], phase, abort_flag, status, limit_ns);
    const uint32_t buf = ring_base + static_cast<uint32_t>(s) * S::stage_bytes;
    if (landed && g < G) {
      float d[NT][2][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int f = 0; f < 4; ++f) d[j][t][f] = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4 wv = lds128(buf + ((b & 1) ? w_odd : w_even) + (b >> 1) * 1024);
        uint32_t p[4][4];
        code_pairs_f16(wv.x, p[0]);
        code_pairs_f16(wv.y, p[1]);
        code_pairs_f16(wv.z, p[2]);
        code_pairs_f16(wv.w, p[3]);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint4 e = lds128(buf + x_lane + ((b & 1) + 8 * (b >> 1)) * (MRP * 16) + j * 128);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            // rows gq <- column 4gq + 2t, rows gq + 8 <- column 4gq + 2t + 1
            mma_f16_16816(d[j][t], p[2 * t][0], p[2 * t + 1][0], p[2 * t][1], p[2 * t + 1][1],
                          e.x, e.y);
            mma_f16_16816(d[j][t], p[2 * t][2], p[2 * t + 1][2], p[2 * t][3], p[2 * t + 1][3],
                          e.z, e.w);
          }
        }
      }
      // Fold the group: y += (s U) D + (min X - s T). d[j][t][2h + r] is column 4gq + 2t + h,
      // batch row 8j + 2c + r.
      const uint2 sv = lds64(buf + s_off), mv = lds64(buf + s_off + S::row_stride);
      float sc[4], mn[4];
      group_scale_offset<ZP>(sv.x & 0xFFFFu, mv.x & 0xFFFFu, sc[0], mn[0]);
      group_scale_offset<ZP>(sv.x >> 16, mv.x >> 16, sc[1], mn[1]);
      group_scale_offset<ZP>(sv.y & 0xFFFFu, mv.y & 0xFFFFu, sc[2], mn[2]);
      group_scale_offset<ZP>(sv.y >> 16, mv.y >> 16, sc[3], mn[3]);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float4 cr[2] = {lds128f(buf + c_lane + j * 128),
                              lds128f(buf + c_lane + j * 128 + 16)};
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int col = 2 * t + h;
              yacc[j][col][r] =
                  fmaf(sc[col] * cr[r].z, d[j][t][2 * h + r],
                       fmaf(mn[col], cr[r].x, fmaf(-sc[col], cr[r].y, yacc[j][col][r])));
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

  // The GPC warps of a quarter add their partials in group order.
  for (int gg = 0; gg < GPC; ++gg) {
    if (gl == gg) {
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int col = 0; col < 4; ++col)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float* dst = sRed + (8 * j + 2 * c + r) * S::RED_LD + qq * 32 + gq * 4 + col;
            *dst = gg == 0 ? yacc[j][col][r] : *dst + yacc[j][col][r];
          }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
  }
  for (int i = tid; i < MRP * S::W; i += NC) {
    const int m = i / S::W, col = i - m * S::W;
    const int nn = col0 + col;
    if (m < M && nn < col_end)
      y[static_cast<size_t>(m) * N + nn] =
          __bfloat16_as_ushort(__float2bfloat16_rn(sRed[m * S::RED_LD + col]));
  }
}

int sk_sm_count() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

// Ring depth for a shape: two CTAs per SM when the small shapes can still hold two stages
// (so the next call's CTA can stream its weights during this one), else the whole SM.
template <int NT, int QW>
int sk_stages() {
  using S = SkShape<NT, QW>;
  auto fit = [](uint32_t budget) {
    const uint32_t fixed = sk_smem_total<NT, QW>(0);
    if (fixed >= budget) return 0;
    const int s = static_cast<int>((budget - fixed) / S::stage_bytes);
    return s > kSkMaxStages ? kSkMaxStages : s;
  };
  const int two = S::kMinBlocks == 2 ? fit(kSkSmemTwoCtas) : 0;
  return two >= 2 ? two : fit(kSkSmemOneCta);
}

int sk_stages_of(int nt, int qw) {
#define W4K_SK_STAGES(NT, QW) \
  if (nt == NT && qw == QW) return sk_stages<NT, QW>();
  W4K_SK_STAGES(1, 2) W4K_SK_STAGES(1, 3) W4K_SK_STAGES(1, 4) W4K_SK_STAGES(1, 6)
  W4K_SK_STAGES(2, 2) W4K_SK_STAGES(2, 3) W4K_SK_STAGES(2, 4) W4K_SK_STAGES(2, 6)
  W4K_SK_STAGES(4, 2) W4K_SK_STAGES(4, 3) W4K_SK_STAGES(4, 4) W4K_SK_STAGES(4, 6)
#undef W4K_SK_STAGES
  return 0;
}

template <int NT, int QW, bool ZP>
cudaError_t sk_launch_shape(const SkMaps& maps, const uint4* xs, const float4* cst, uint16_t* y,
                            int M, int N, int K, const SkinnyPlan& plan, uint32_t* status,
                            uint64_t limit_ns, cudaStream_t stream) {
  auto kern = w4a16_skinny_kernel<NT, QW, ZP>;
  const uint32_t smem = sk_smem_total<NT, QW>(plan.stages);
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_with_pdl(kern, dim3(static_cast<unsigned>(plan.ctas)), dim3(kSkThreads), smem,
                         stream, maps, xs, cst, y, M, N, K, plan.stages, plan.col_q, plan.col_r,
                         status, limit_ns);
}

}  // namespace

bool skinny_plan(int M, int N, int K, SkinnyPlan* plan) {
  if (M < 1 || M > kSkinnyMaxRows || N <= 0 || K <= 0 || K % 128 != 0 || N % 8 != 0)
    return false;
  const int sms = sk_sm_count();
  if (sms <= 0) return false;
  const int n8 = N / 8, q = n8 / sms, r = n8 % sms;
  const int maxw = 8 * (q + (r > 0 ? 1 : 0));
  if (q < 4 || maxw > 192) return false;  // at least 32 columns per SM, at most 6 quarters
  SkinnyPlan p;
  // Two n8 tiles for every M <= 16: with one, the launch measured slower (11.8 against
  // 10.9 us at M = 5..8 on 14336 x 4096).
  p.nt = M <= 16 ? 2 : 4;
  p.qw = maxw <= 64 ? 2 : maxw <= 96 ? 3 : maxw <= 128 ? 4 : 6;
  p.col_q = q;
  p.col_r = r;
  p.ctas = sms;
  p.stages = sk_stages_of(p.nt, p.qw);
  if (p.stages < 2) return false;
  const int gpc = kSkConsumerWarps / p.qw;
  const int kchunks = ((K >> 7) + gpc - 1) / gpc;
  p.rows_pad = kchunks * 16 * gpc;
  const size_t mrp = static_cast<size_t>(8 * p.nt);
  p.xs_bytes = ((static_cast<size_t>(p.rows_pad) * mrp * 16 + 255) / 256) * 256;
  p.ws_bytes = p.xs_bytes + static_cast<size_t>(kchunks) * gpc * mrp * 16;
  *plan = p;
  return true;
}

cudaError_t launch_w4a16_skinny(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                                const uint16_t* mins, uint16_t* y, int M, int N, int K,
                                void* workspace, const SkinnyPlan& plan, uint32_t* status,
                                uint64_t wait_limit_ns, cudaStream_t stream, bool zero_point) {
  const uint32_t w = 32u * plan.qw, gpc = static_cast<uint32_t>(kSkConsumerWarps / plan.qw);
  const CUtensorMapDataType st =
      zero_point ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  SkMaps maps;
  cudaError_t e;
  e = encode_tensor_map(&maps.qw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N) * 4, 32u, 16u * gpc,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_tensor_map(&maps.scales, st, scales,
                        static_cast<uint64_t>(N), static_cast<uint64_t>(K / 128),
                        static_cast<uint64_t>(N) * 2, w, gpc, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = encode_tensor_map(&maps.mins, st, mins,
                        static_cast<uint64_t>(N), static_cast<uint64_t>(K / 128),
                        static_cast<uint64_t>(N) * 2, w, gpc, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  uint4* xs = static_cast<uint4*>(workspace);
  float4* cst = reinterpret_cast<float4*>(static_cast<char*>(workspace) + plan.xs_bytes);
  const int mrp = 8 * plan.nt;
  const int items = mrp * (plan.rows_pad / 2);
  const dim3 pgrid(static_cast<unsigned>((items + kSkPrepThreads - 1) / kSkPrepThreads));
  switch (plan.nt) {
    case 1: e = launch_with_pdl(skinny_xprep_kernel<8>, pgrid, dim3(kSkPrepThreads), 0, stream, x, xs, cst, M, K, plan.rows_pad); break;
    case 2: e = launch_with_pdl(skinny_xprep_kernel<16>, pgrid, dim3(kSkPrepThreads), 0, stream, x, xs, cst, M, K, plan.rows_pad); break;
    default: e = launch_with_pdl(skinny_xprep_kernel<32>, pgrid, dim3(kSkPrepThreads), 0, stream, x, xs, cst, M, K, plan.rows_pad); break;
  }
  if (e != cudaSuccess) return e;
#define W4K_SK_CASE(NT, QW)                                                                  \
  if (plan.nt == NT && plan.qw == QW)                                                        \
    return zero_point ? sk_launch_shape<NT, QW, true>(maps, xs, cst, y, M, N, K, plan, status, \
                                                      wait_limit_ns, stream)                 \
                      : sk_launch_shape<NT, QW, false>(maps, xs, cst, y, M, N, K, plan,      \
                                                       status, wait_limit_ns, stream);
  W4K_SK_CASE(1, 2) W4K_SK_CASE(1, 3) W4K_SK_CASE(1, 4) W4K_SK_CASE(1, 6)
  W4K_SK_CASE(2, 2) W4K_SK_CASE(2, 3) W4K_SK_CASE(2, 4) W4K_SK_CASE(2, 6)
  W4K_SK_CASE(4, 2) W4K_SK_CASE(4, 3) W4K_SK_CASE(4, 4) W4K_SK_CASE(4, 6)
#undef W4K_SK_CASE
  return cudaErrorInvalidValue;
}

}  // namespace w4k
