// W4A16 GEMV / skinny kernel for small M (M <= 8): packed words staged by TMA, codes widened
// to FP16 in registers with one mask per pair of codes, inner products on the tensor
// pipe (mma.sync m16n8k16, FP16 x FP16 -> FP32), scale and minimum folded per group.
//
//   y[m, n] = sum_g ( s[g,n] * sum_{k in g} x[m,k] q[n,k] + min[g,n] * sum_{k in g} x[m,k] )
//
// The factorised per-group form is the one the pages give for their M = 1 kernel ("Low-
// Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", "How the measurements were
// taken": FP32 sums of s x sum x.q plus min x sum x, group by group). The work split
// follows "Quantization and GEMV", "Writing a GEMV kernel" (wide reads, K split over
// warps, fixed-order reductions), adapted to the K/8 x N packed layout (N contiguous).
//
// What bounds it on GB300. At 4 bits an SM must turn ~6 packed words per clock into
// products to keep up with its share of HBM ("Where the time goes at M = 1": the unpacking
// decides). Masks and shifts run on the integer pipe at half the FMA rate, so the kernel
// spends as few of them as it can: in an FP16 the mantissa holds bits 0..9, so a 16-bit
// half of a word yields two codes in place (0x6400 | q = 1024 + q from bits 0..3, and
// 0x6400 | 16 q = 1024 + 16 q from bits 4..7). A word costs 4 masks + 1 shift for its 8
// codes (BF16, with 7 mantissa bits, would need 3 shifts). The products go to the tensor
// pipe (one m16n8k16 per 256 codes, batch rows in the n8 dimension), which runs beside the
// integer pipe.
//
// x is converted to FP16 exactly, scaled per group of 128 by a power of two 2^e so that its
// largest magnitude lands in [2^14, 2^15) (a BF16 value has 8 significant bits, a normal
// FP16 11), and the k slots holding 16 q get x 2^(e-4). Per group the tensor core then
// returns D = 2^e (sum q x + 1024 sum_even x + 64 sum_odd x) (even / odd: position of k in
// its packed word), so
//   y += (s 2^-e) D + (min X - s T),  X = sum_g x,  T = 1024 sum_even x + 64 sum_odd x,
// with X, T and 2^-e computed once per CTA in fp32.
//
// Launch shape:
//   * even mode (N >= 48 columns per SM): exactly one CTA per SM, CTA c owns 8 q or
//     8 (q + 1) consecutive columns (N = 14336: 120 CTAs of 96, 32 of 88) and all of K. Its
//     shared-memory ring leaves room for a second CTA on the SM, which is the next launch's:
//     with one CTA per SM in every launch the block scheduler has exactly one free slot per
//     SM for the next launch, so no SM runs two CTAs of one launch (with more CTAs than SMs
//     and room for two per SM, a launch's CTAs doubled up on a few SMs and set its tail);
//   * slab mode (narrow N, or N too wide for 128 columns per SM): slabs of W = 64, 96 or 128
//     columns, persistent grid (<= one CTA per SM, CTA c takes units c, c + G, ...), one
//     CTA per SM; with a workspace a slab's K range may be split across CTAs;
//   * a producer warp streams each unit in chunks of W columns x (consumer warps) / (W / 32)
//     groups (1 KB of packed words per consumer warp, plus scales and minimums) into the
//     ring with TMA, starting before it waits for the previous kernel on the stream
//     (programmatic dependent launch; weights are not written by the kernels it overlaps),
//     so in even mode the next launch's weights stream while this launch computes;
//   * 12 (even mode) or 24 (slab mode) consumer warps: warp w takes column quarter
//     w % (W / 32) (32 columns) of group w / (W / 32) of each chunk. Lane (gq, c) =
//     (lane / 4, lane % 4) reads packed row 4b + c of block b (b = 0..3) and columns
//     4gq..4gq+3 with one 16-byte shared load; its four words fill the A fragments of two
//     16-row MMA tiles (tile t: rows gq <- column 4gq + 2t, gq + 8 <- column 4gq + 2t + 1);
//     x waits in shared memory in B-fragment order (the lanes' offsets are fixed per warp;
//     blocks and stages add constants);
//   * per unit the group partials of each column are summed in a fixed order; a split slab
//     writes fp32 partials and the last CTA to arrive (arrival counter) sums them in split
//     order (deterministic, no float atomics) and resets the counter.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kMaxRows = 8;
constexpr int kMaxStages = 8;
constexpr uint32_t kSmemOneCta = 227u * 1024u;
constexpr uint32_t kSmemTwoCtas = 113u * 1024u;  // two CTAs (and their reserves) per SM
// The packed words land 128-byte swizzled, which wants 1024-byte aligned destinations; the
// dynamic shared-memory base is 128-byte aligned, so the kernel rounds it up (at most 896 B).
constexpr uint32_t kAlignPad = 1024u - 128u;

// Slab of W = 32 QW columns; a chunk holds GPC groups of 128 k (16 packed rows each) so that
// every consumer warp owns one (group, column quarter).
// CW consumer warps + one producer warp. 12 consumer warps leave room (registers, shared
// memory) for a second CTA on the SM, 24 do not.
template <int QW, int CW>
struct Shape {
  static constexpr int kConsumers = CW * 32;
  static constexpr int kThreads = kConsumers + 32;
  static constexpr int kMinBlocks = CW <= 12 ? 2 : 1;
  static constexpr int W = 32 * QW;
  static constexpr int GPC = CW / QW;
  static constexpr int ROWS = 16 * GPC;
  static constexpr uint32_t word_bytes = static_cast<uint32_t>(W) * ROWS * 4u;  // 1 KB x CW
  static constexpr uint32_t row_bytes = static_cast<uint32_t>(GPC) * W * 2u;    // scales
  // TMA destinations must be 128-byte aligned: the scale and minimum boxes each start on
  // their own 128-byte boundary (a box of 5 groups x 96 columns is 960 bytes).
  static constexpr uint32_t row_stride = (row_bytes + 127u) & ~127u;
  static constexpr uint32_t tx_bytes = word_bytes + 2u * row_bytes;  // bytes one stage receives
  static constexpr uint32_t sc_bytes = 2u * row_stride;  // scales + minimums of one stage
  static constexpr uint32_t stage_bytes = word_bytes + sc_bytes;
  static constexpr uint32_t box_bytes = static_cast<uint32_t>(ROWS) * 128u;  // one quarter
  static_assert(GPC * QW == CW, "one (group, quarter) per consumer warp");
  static_assert(box_bytes % 1024u == 0u && word_bytes == box_bytes * QW,
                "swizzled word boxes start on 1024-byte boundaries");
  static_assert(row_stride % 128u == 0u, "TMA destinations stay 128-byte aligned");
};

// Shared-memory layout (from the 1024-byte aligned base): the word ring (stages x
// word_bytes), the scale/minimum ring (stages x sc_bytes), per-warp partials, per-(row,
// group) constants of x, x in B-fragment order, barriers; `total` includes the alignment pad.
struct GemvLayout {
  uint32_t red_off, cst_off, xperm_off, bar_off, total;
  __host__ __device__ GemvLayout(uint32_t stage_bytes, int rows_pad, int MR, int G, int stages,
                                 int CW) {
    red_off = static_cast<uint32_t>(stages) * stage_bytes;               // [CW][MR][32] fp32
    cst_off = red_off + static_cast<uint32_t>(CW) * MR * 32u * 4u;       // X, T, U: [3][MR][G]
    xperm_off = (cst_off + 3u * MR * G * 4u + 15u) & ~15u;               // [rows_pad][MR] 16 B
    bar_off = (xperm_off + static_cast<uint32_t>(rows_pad) * MR * 16u + 7u) & ~7u;
    total = bar_off + 2u * kMaxStages * 8u + 16u + kAlignPad;
  }
};

template <int NC>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
}

struct GemvMaps {
  CUtensorMap qw;      // int32 [K/8, N], box {32, ROWS}, 128-byte swizzle
  CUtensorMap scales;  // bf16 (fp16 with a zero point) [K/128, N], box {W, GPC}
  CUtensorMap mins;    // bf16 minimums (fp16 zero points) [K/128, N], box {W, GPC}
};

// ZP: the zero-point format (FP16 scale and zero point, w_hat = (q - z) s); otherwise the
// minimum format (BF16 scale and minimum). Only the fold's reading of the two differs.
template <int MR, int QW, int CW, bool ZP>
__global__ void __launch_bounds__(Shape<QW, CW>::kThreads, Shape<QW, CW>::kMinBlocks)
    gemv_w4a16_kernel(const __grid_constant__ GemvMaps maps, const uint16_t* __restrict__ x,
                      uint16_t* __restrict__ y, int M, int N, int K, int stages, int splits,
                      int col_q, int col_r, float* __restrict__ ws_partial,
                      uint32_t* __restrict__ ws_counter, uint32_t* __restrict__ status,
                      uint64_t limit_ns) {
  static_assert(MR <= 8, "one n8 tile of batch rows");
  using S = Shape<QW, CW>;
  constexpr int W = S::W, GPC = S::GPC, ROWS = S::ROWS, NC = S::kConsumers;
  const int G = K >> 7;
  const int kchunks = (G + GPC - 1) / GPC;
  const int rows_pad = kchunks * ROWS;
  const GemvLayout L(S::stage_bytes, rows_pad, MR, G, stages, CW);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  if (pad > kAlignPad) {  // base less than 128-byte aligned: report, touch nothing
    if (threadIdx.x == 0) atomicOr(status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  float* sRed = reinterpret_cast<float*>(smem + L.red_off);
  float* sX = reinterpret_cast<float*>(smem + L.cst_off);  // [MR][G] sum x
  float* sT = sX + MR * G;                                  // [MR][G] 1024 sum_even + 64 sum_odd
  float* sU = sT + MR * G;                                  // [MR][G] 2^-e
  uint4* sXperm = reinterpret_cast<uint4*>(smem + L.xperm_off);  // [rows_pad][MR]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kMaxStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kMaxStages);
  volatile uint32_t* last_flag = abort_flag + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_unit = (kchunks + splits - 1) / splits;  // chunks per k-range
  // Slabs: W columns each, or (col_q > 0) one per CTA with 8 col_q or 8 (col_q + 1)
  // columns, the first col_r slabs wider, so that every SM gets the same share of N.
  const int nslab = col_q > 0 ? static_cast<int>(gridDim.x) : (N + W - 1) / W;
  const int nunits = nslab * splits;
  auto slab_col0 = [&](int slab) {
    return col_q > 0 ? 8 * (slab * col_q + min(slab, col_r)) : slab * W;
  };
  auto slab_cols = [&](int slab) {
    return col_q > 0 ? 8 * (col_q + (slab < col_r ? 1 : 0)) : W;
  };

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CW);
    }
    *abort_flag = 0u;
    fence_barrier_init();
    pdl_launch_dependents();  // the next kernel may start streaming its own weights
  }
  __syncthreads();

  if (warp == CW) {
    // ---------------- producer warp: weights only, no wait on the previous kernel -------
    if (lane == 0) {
      tma_prefetch_desc(&maps.qw);
      tma_prefetch_desc(&maps.scales);
      tma_prefetch_desc(&maps.mins);
      int j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int slab = u / splits, kr = u - slab * splits;
        const int kc_end = min(kchunks, (kr + 1) * per_unit);
        for (int kc = kr * per_unit; kc < kc_end; ++kc, ++j) {
          const int s = j % stages;
          const uint32_t use = static_cast<uint32_t>(j / stages);
          if (use > 0 &&
              !mbar_wait_bounded(&empty[s], (use - 1) & 1u, abort_flag, status, limit_ns)) {
            ok = false;
            break;
          }
          uint8_t* wbuf = smem + s * S::word_bytes;
          uint8_t* sbuf = smem + stages * S::word_bytes + s * S::sc_bytes;
          mbar_arrive_expect_tx(&full[s], S::tx_bytes);
          const int col0 = slab_col0(slab);
#pragma unroll
          for (int q = 0; q < QW; ++q)
            tma_load_2d(wbuf + q * S::box_bytes, &maps.qw, &full[s], col0 + 32 * q, kc * ROWS);
          tma_load_2d(sbuf, &maps.scales, &full[s], col0, kc * GPC);
          tma_load_2d(sbuf + S::row_stride, &maps.mins, &full[s], col0, kc * GPC);
        }
      }
      // Stay until this CTA's last copies have landed (bounded), so none is in flight
      // when the CTA exits, whatever the consumers did.
      const int issued = j;
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
  // x -> FP16 in B-fragment order, per (row m, group g) scale 2^e and the sums X, T. An
  // item is 16 consecutive x values (packed rows R = r_lo + 2p and R + 1); the 8 items of a
  // group sit on 8 adjacent lanes. Item i = m * half + p (p fastest), half = (r_hi - r_lo) / 2;
  // this thread's items are tid + t * NC. Their indices do not depend on the previous
  // kernel, so the first kBatch are worked out before waiting on it.
  // A CTA that owns a single unit of a split plan reads only its own k-range of x, so it
  // converts only those rows (whole chunks: the 8 items of a group stay together).
  int r_lo = 0, r_hi = rows_pad;
  if (splits > 1 && static_cast<int>(gridDim.x) >= nunits) {
    const int kr = static_cast<int>(blockIdx.x) % splits;
    r_lo = kr * per_unit * ROWS;
    r_hi = min(kchunks, (kr + 1) * per_unit) * ROWS;
  }
  const int half = (r_hi - r_lo) >> 1;
  const int items = MR * half;
  const int items_pad = (items + 31) & ~31;  // warp-uniform trip count for the shuffles
  // items per thread whose loads are issued together (with 12 consumer warps and K = 4096,
  // all of x in one round up to MR = 4; more would spill at MR = 8)
  constexpr int kBatch = MR >= 4 ? 3 : 2;
  int im0[kBatch], ip0[kBatch];
#pragma unroll
  for (int t = 0; t < kBatch; ++t) {
    const int i = t * NC + tid;
    im0[t] = i / half;
    ip0[t] = i - im0[t] * half;
  }
  pdl_wait();  // x, y and the workspace may belong to the previous kernel on the stream
  {
    const int rows = K >> 3;
    // Loads of up to kBatch items per thread are issued before any of them is used.
    for (int base = 0; base < items_pad; base += kBatch * NC) {
      uint4 xin[kBatch][2];
      int im[kBatch], ip[kBatch];
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        const int i = base + t * NC + tid;
        im[t] = base == 0 ? im0[t] : i / half;
        ip[t] = base == 0 ? ip0[t] : i - im[t] * half;
        const int R = r_lo + 2 * ip[t];
        xin[t][0] = xin[t][1] = make_uint4(0u, 0u, 0u, 0u);
        if (i < items && im[t] < M && R < rows) {
          const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(im[t]) * K + 8 * R);
          xin[t][0] = __ldg(src);
          xin[t][1] = __ldg(src + 1);
        }
      }
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        const int i = base + t * NC + tid;
        if (i >= items_pad) break;  // warp-uniform: items_pad and the strides are multiples of 32
        const int m = im[t], R = r_lo + 2 * ip[t];
        float v[16];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint32_t xw[4] = {xin[t][r].x, xin[t][r].y, xin[t][r].z, xin[t][r].w};
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
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          sum_even += __shfl_xor_sync(0xffffffffu, sum_even, o);
          sum_odd += __shfl_xor_sync(0xffffffffu, sum_odd, o);
        }
        // amax 2^e in [2^14, 2^15): e = 141 - biased exponent, kept where 2^e is a normal
        // float; an all-zero group keeps e = 0.
        int e = 0;
        if (amax > 0.f)
          e = max(-100, min(100, 141 - static_cast<int>(__float_as_uint(amax) >> 23)));
        const float lo = pow2f(e), hi = pow2f(e - 4);
        if (i < items) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float* w = v + 8 * r;
            uint4 out;
            out.x = f16x2_bits(w[0] * lo, w[4] * lo);  // (x0, x4) 2^e
            out.y = f16x2_bits(w[1] * hi, w[5] * hi);  // (x1, x5) 2^(e-4)
            out.z = f16x2_bits(w[2] * lo, w[6] * lo);  // (x2, x6) 2^e
            out.w = f16x2_bits(w[3] * hi, w[7] * hi);  // (x3, x7) 2^(e-4)
            sXperm[(R + r) * MR + m] = out;
          }
          if ((R & 15) == 0 && R < rows) {
            const int g = R >> 4;
            sX[m * G + g] = sum_even + sum_odd;
            sT[m * G + g] = fmaf(1024.0f, sum_even, 64.0f * sum_odd);
            sU[m * G + g] = pow2f(-e);
          }
        }
      }
    }
  }
  consumer_bar<NC>();

  const int gq = lane >> 2, c = lane & 3;
  const int qq = warp % QW, gl = warp / QW;  // column quarter, group within a chunk
  // Lane (gq, c) reads packed row 16 gl + 2c + (b & 1) + 8 (b >> 1) of its column quarter in
  // block b: the 16 rows of the group once each, in an order where the 8 lanes of a shared-
  // memory phase (gq in {2p, 2p + 1}, c = 0..3) hit 16-byte chunks gq ^ (2c + (b & 1)) of the
  // swizzled rows (chunk j of row r sits at j ^ (r mod 8)): 8 distinct chunks, all 32 banks,
  // no conflict. x follows the same row order, so each MMA still pairs matching k.
  // Per-lane constant addresses: odd blocks use the odd row, blocks 2 and 3 add 8 rows, a
  // stage adds word_bytes / sc_bytes.
  const uint32_t ring_base = smem_addr(smem);
  const int r_even = gl * 16 + 2 * c, r_odd = r_even + 1;
  const uint32_t w_even =
      static_cast<uint32_t>(qq) * S::box_bytes + static_cast<uint32_t>(r_even * 128 + ((gq ^ (2 * c)) << 4));
  const uint32_t w_odd =
      static_cast<uint32_t>(qq) * S::box_bytes + static_cast<uint32_t>(r_odd * 128 + ((gq ^ (2 * c + 1)) << 4));
  const uint32_t sc_ring = ring_base + static_cast<uint32_t>(stages) * S::word_bytes;
  const uint32_t s_off = static_cast<uint32_t>(gl * (W * 2) + (qq * 32 + gq * 4) * 2);
  // B fragment: lane (gq, c) supplies batch row gq & (MR - 1), so product column n holds
  // row n & (MR - 1), and lane c's fragment columns 2c, 2c + 1 hold rows (2c + bb) & (MR - 1).
  const uint32_t x_lane = smem_addr(sXperm) + static_cast<uint32_t>((r_even * MR + (gq & (MR - 1))) * 16);
  // Lanes whose fragments hold the same rows share the fold: with MR <= 2 all four c-lanes
  // hold every row and fold one column each, with MR = 4 lanes c and c ^ 2 split four
  // columns, with MR = 8 each lane folds its own two rows of all four columns.
  constexpr int CPL = MR <= 2 ? 1 : MR == 4 ? 2 : 4;  // columns folded per lane
  constexpr int NBB = MR == 1 ? 1 : 2;                // fragment columns (rows) per lane
  const int jj0 = MR <= 2 ? c : MR == 4 ? 2 * (c >> 1) : 0;
  int s = 0;
  uint32_t phase = 0u;  // ring position of the next chunk
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const int slab = u / splits, kr = u - slab * splits;
    const int kc_end = min(kchunks, (kr + 1) * per_unit);
    const int col0 = slab_col0(slab), col_end = min(N, col0 + slab_cols(slab));
    // yacc[i][bb]: column col0 + 32*qq + 4*gq + jj0 + i, batch row (2c + bb) & (MR - 1)
    float yacc[CPL][NBB];
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
      for (int bb = 0; bb < NBB; ++bb) yacc[i][bb] = 0.f;

    for (int kc = kr * per_unit; kc < kc_end; ++kc) {
      const int g = kc * GPC + gl;  // this warp's group
      // On an expired wait every warp keeps walking the chunk list without computing, so
      // all consumer warps still meet at the per-unit barriers below.
      const bool landed = mbar_wait_bounded(&full[s], phase, abort_flag, status, limit_ns);
      const uint32_t wbuf = ring_base + static_cast<uint32_t>(s) * S::word_bytes;
      const uint32_t sbuf = sc_ring + static_cast<uint32_t>(s) * S::sc_bytes;
      if (landed && g < G) {
        const uint32_t xa = x_lane + static_cast<uint32_t>(kc * (ROWS * MR * 16));
        float d[2][2][4];  // [chain][tile t][fragment]: even / odd blocks
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int f = 0; f < 4; ++f) d[ch][t][f] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint4 wv = lds128(wbuf + ((b & 1) ? w_odd : w_even) + (b >> 1) * 1024);
          const uint4 e = lds128(xa + ((b & 1) + 8 * (b >> 1)) * (MR * 16));
          uint32_t p[4][4];
          code_pairs_f16(wv.x, p[0]);
          code_pairs_f16(wv.y, p[1]);
          code_pairs_f16(wv.z, p[2]);
          code_pairs_f16(wv.w, p[3]);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            // rows gq <- column 4gq + 2t, rows gq + 8 <- column 4gq + 2t + 1
            mma_f16_16816(d[b & 1][t], p[2 * t][0], p[2 * t + 1][0], p[2 * t][1],
                          p[2 * t + 1][1], e.x, e.y);
            mma_f16_16816(d[b & 1][t], p[2 * t][2], p[2 * t + 1][2], p[2 * t][3],
                          p[2 * t + 1][3], e.z, e.w);
          }
        }
        // Fold this group: y += (s 2^-e) D + (min X - s T). Column 4gq + jj is tile jj / 2,
        // fragment half jj % 2.
        float dsum[4][NBB];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int bb = 0; bb < NBB; ++bb)
            dsum[jj][bb] = d[0][jj >> 1][2 * (jj & 1) + bb] + d[1][jj >> 1][2 * (jj & 1) + bb];
        float gx[NBB], gt[NBB], gu[NBB];
#pragma unroll
        for (int bb = 0; bb < NBB; ++bb) {
          const int ci = ((2 * c + bb) & (MR - 1)) * G + g;
          gx[bb] = sX[ci];
          gt[bb] = sT[ci];
          gu[bb] = sU[ci];
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const int jj = jj0 + i;
          float sc, mn;
          group_scale_offset<ZP>(lds_u16(sbuf + s_off + 2 * jj),
                                 lds_u16(sbuf + s_off + S::row_stride + 2 * jj), sc, mn);
#pragma unroll
          for (int bb = 0; bb < NBB; ++bb) {
            float dv;
            if constexpr (CPL == 4) {
              dv = dsum[i][bb];
            } else if constexpr (CPL == 2) {
              dv = (c >> 1) ? dsum[2 + i][bb] : dsum[i][bb];
            } else {
              dv = (c & 2) ? ((c & 1) ? dsum[3][bb] : dsum[2][bb])
                           : ((c & 1) ? dsum[1][bb] : dsum[0][bb]);
            }
            yacc[i][bb] =
                fmaf(sc * gu[bb], dv, fmaf(mn, gx[bb], fmaf(-sc, gt[bb], yacc[i][bb])));
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

    // Unit done: warp partials to shared memory, fixed-order sum over the GPC groups of
    // each column quarter.
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
      for (int bb = 0; bb < NBB; ++bb)
        sRed[(warp * MR + ((2 * c + bb) & (MR - 1))) * 32 + gq * 4 + jj0 + i] = yacc[i][bb];
    consumer_bar<NC>();
    for (int i = tid; i < MR * W; i += NC) {
      const int mm = i / W, col = i - mm * W, q = col >> 5, c32 = col & 31;
      float v = 0.f;
#pragma unroll
      for (int gg = 0; gg < GPC; ++gg) v += sRed[((gg * QW + q) * MR + mm) * 32 + c32];
      const int nn = col0 + col;
      if (mm < M && nn < col_end) {
        if (splits == 1)
          y[static_cast<size_t>(mm) * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        else
          __stcg(ws_partial + (static_cast<size_t>(kr) * MR + mm) * N + nn, v);
      }
    }
    if (splits > 1) {
      __threadfence();
      consumer_bar<NC>();
      if (tid == 0)
        *last_flag = (atomicAdd(ws_counter + slab, 1u) + 1u == static_cast<uint32_t>(splits));
      consumer_bar<NC>();
      if (*last_flag) {
        __threadfence();
        for (int i = tid; i < MR * W; i += NC) {
          const int mm = i / W, col = i - mm * W;
          const int nn = col0 + col;
          if (mm < M && nn < col_end) {
            float v = 0.f;
            for (int z = 0; z < splits; ++z)
              v += __ldcg(ws_partial + (static_cast<size_t>(z) * MR + mm) * N + nn);
            y[static_cast<size_t>(mm) * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
          }
        }
        if (tid == 0) ws_counter[slab] = 0u;  // ready for the next call
      }
    }
    consumer_bar<NC>();
  }
}

int sm_count() {
  static int count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count[dev] == 0) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

int mr_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

// Slab width 32 qw: the fewest columns per SM in the busiest round; ties go to wider slabs.
int choose_qw(int N, int sms) {
  int best = 4, best_cost = 0;
  for (int qw = 4; qw >= 2; --qw) {
    const int w = 32 * qw, nslab = (N + w - 1) / w;
    const int cost = ((nslab + sms - 1) / sms) * w;
    if (qw == 4 || cost < best_cost) {
      best = qw;
      best_cost = cost;
    }
  }
  return best;
}

// How a launch covers N. Even mode (col_q > 0): one CTA per SM, CTA c owns 8 col_q or
// 8 (col_q + 1) columns, and the ring leaves room for the next launch's CTA on the same SM
// (12 consumer warps); with exactly one CTA per SM in every launch, the block scheduler
// has one free slot per SM for the next launch, so no SM ever runs two CTAs of one launch.
// Slab mode: slabs of 32 qw columns, persistent grid, 24 consumer warps, one CTA per SM.
struct GemvPlan {
  int qw = 4, cw = 24, col_q = 0, col_r = 0, nslab = 0;
};

GemvPlan make_plan(int N, int sms) {
  GemvPlan p;
  const int n8 = N / 8, q = n8 / sms, r = n8 % sms;
  const int maxw = 8 * (q + (r > 0 ? 1 : 0));
  if (q >= 6 && maxw <= 128) {
    p.qw = maxw <= 64 ? 2 : maxw <= 96 ? 3 : 4;
    p.cw = 12;
    p.col_q = q;
    p.col_r = r;
    p.nslab = sms;
  } else {
    p.qw = choose_qw(N, sms);
    p.nslab = (N + 32 * p.qw - 1) / (32 * p.qw);
  }
  return p;
}

template <int QW, int CW>
uint32_t fixed_smem(int MR, int K) {
  using S = Shape<QW, CW>;
  const int G = K >> 7;
  const int rows_pad = ((G + S::GPC - 1) / S::GPC) * S::ROWS;
  return GemvLayout(S::stage_bytes, rows_pad, MR, G, 0, CW).total;
}

// Ring depth: as deep as the budget allows beside x and the partials (at most kMaxStages).
template <int QW, int CW>
int stages_for(int MR, int K, uint32_t budget) {
  const uint32_t fixed = fixed_smem<QW, CW>(MR, K);
  if (fixed >= budget) return 0;
  const int s = static_cast<int>((budget - fixed) / Shape<QW, CW>::stage_bytes);
  return s > kMaxStages ? kMaxStages : s;
}

template <int QW, int CW>
int stages_of(int MR, int K) {
  // Two CTAs per SM when the ring can still hold three stages, else the whole SM (with x
  // for four or eight rows in shared memory, two stages were slower than one CTA per SM).
  const int two = CW <= 12 ? stages_for<QW, CW>(MR, K, kSmemTwoCtas) : 0;
  return two >= 3 ? two : stages_for<QW, CW>(MR, K, kSmemOneCta);
}

template <int MR, int QW, int CW, bool ZP>
cudaError_t launch_shape(const GemvMaps& maps, const uint16_t* x, uint16_t* y, int M, int N,
                         int K, const GemvSplit& split, const GemvPlan& plan, uint32_t* status,
                         uint64_t limit_ns, int sms, cudaStream_t stream) {
  using S = Shape<QW, CW>;
  const int stages = stages_of<QW, CW>(MR, K);
  if (stages < 2) return cudaErrorInvalidValue;
  const int G = K >> 7;
  const int rows_pad = ((G + S::GPC - 1) / S::GPC) * S::ROWS;
  const GemvLayout L(S::stage_bytes, rows_pad, MR, G, stages, CW);
  auto kern = gemv_w4a16_kernel<MR, QW, CW, ZP>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                       static_cast<int>(L.total));
  if (e != cudaSuccess) return e;
  const int nunits = plan.nslab * split.splits;
  dim3 grid(static_cast<unsigned>(plan.col_q > 0 ? plan.nslab : (nunits < sms ? nunits : sms)));
  return launch_with_pdl(kern, grid, dim3(S::kThreads), L.total, stream, maps, x, y, M, N, K,
                         stages, split.splits, plan.col_q, plan.col_r, split.partial,
                         split.counter, status, limit_ns);
}

template <int MR, bool ZP>
cudaError_t launch_mr(const GemvMaps& maps, const uint16_t* x, uint16_t* y, int M, int N, int K,
                      const GemvSplit& split, const GemvPlan& plan, uint32_t* status,
                      uint64_t limit_ns, int sms, cudaStream_t stream) {
#define W4K_GEMV_CASE(QW, CW)                                                                  \
  if (plan.qw == QW && plan.cw == CW)                                                         \
    return launch_shape<MR, QW, CW, ZP>(maps, x, y, M, N, K, split, plan, status, limit_ns, sms, \
                                    stream);
  W4K_GEMV_CASE(4, 24)
  W4K_GEMV_CASE(3, 24)
  W4K_GEMV_CASE(2, 24)
  W4K_GEMV_CASE(4, 12)
  W4K_GEMV_CASE(3, 12)
  W4K_GEMV_CASE(2, 12)
#undef W4K_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

int gemv_max_rows() { return kMaxRows; }

// x in B-fragment order and its per-group constants must leave room for a 2-stage ring in
// every shape a launch may take.
bool gemv_supports(int M, int K) {
  if (M < 1 || M > kMaxRows || K < 128) return false;
  const int mr = mr_of(M);
  return stages_of<4, 24>(mr, K) >= 2 && stages_of<3, 24>(mr, K) >= 2 &&
         stages_of<2, 24>(mr, K) >= 2 && stages_of<4, 12>(mr, K) >= 2 &&
         stages_of<3, 12>(mr, K) >= 2 && stages_of<2, 12>(mr, K) >= 2;
}

GemvSplit gemv_split_plan(int M, int N, int K, size_t* bytes_needed) {
  GemvSplit split;
  *bytes_needed = 0;
  const int sms = sm_count();
  if (sms <= 0) return split;
  const GemvPlan plan = make_plan(N, sms);
  if (plan.col_q > 0) return split;  // every SM already has its share of N
  const int gpc = plan.cw / plan.qw;
  const int kchunks = ((K >> 7) + gpc - 1) / gpc;
  // One unit per CTA: split each slab's K range over the SMs the slabs leave idle.
  int splits = sms / plan.nslab;
  if (splits > kchunks) splits = kchunks;
  if (splits > 64) splits = 64;
  if (splits < 2) return split;
  const int per_unit = (kchunks + splits - 1) / splits;
  splits = (kchunks + per_unit - 1) / per_unit;  // no empty k-range
  if (splits < 2) return split;
  // The last CTA of a slab adds the partials after a fence and an atomic: about 1.5 us on
  // the critical path, worth it only when a CTA skips three chunks or more (4096 x 4096:
  // 6.3 us split in two vs 4.7 us whole; 1536 x 8960: 5.8 us split in six vs 7.6 us whole).
  if (kchunks - per_unit < 3) return split;
  split.splits = splits;
  split.partial_offset = ((static_cast<size_t>(plan.nslab) * 4 + 255) / 256) * 256;
  *bytes_needed = split.partial_offset + static_cast<size_t>(splits) * mr_of(M) * N * 4;
  return split;
}

cudaError_t launch_w4a16_gemv(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                              const uint16_t* mins, uint16_t* y, int M, int N, int K,
                              const GemvSplit& split, uint32_t* status, uint64_t limit_ns,
                              cudaStream_t stream, bool zero_point) {
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const GemvPlan plan = make_plan(N, sms);
  if (plan.col_q > 0 && split.splits != 1) return cudaErrorInvalidValue;
  const uint32_t w = 32u * plan.qw, gpc = static_cast<uint32_t>(plan.cw / plan.qw);
  const CUtensorMapDataType st =
      zero_point ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  GemvMaps maps;
  cudaError_t e;
  e = encode_tensor_map(&maps.qw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N) * 4, 32u, 16u * gpc,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_tensor_map(&maps.scales, st, scales, static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N) * 2, w, gpc,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = encode_tensor_map(&maps.mins, st, mins, static_cast<uint64_t>(N),
                        static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N) * 2, w, gpc,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
#define W4K_GEMV_MR(MR)                                                                      \
  return zero_point                                                                          \
             ? launch_mr<MR, true>(maps, x, y, M, N, K, split, plan, status, limit_ns, sms,  \
                                   stream)                                                   \
             : launch_mr<MR, false>(maps, x, y, M, N, K, split, plan, status, limit_ns, sms, \
                                    stream);
  switch (mr_of(M)) {
    case 1: W4K_GEMV_MR(1)
    case 2: W4K_GEMV_MR(2)
    case 4: W4K_GEMV_MR(4)
    default: W4K_GEMV_MR(8)
  }
#undef W4K_GEMV_MR
}

}  // namespace w4k
