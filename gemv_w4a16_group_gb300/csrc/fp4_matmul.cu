// NVFP4A16 / MXFP4A16 matmul for M > 1: Y[m, n] = sum_k x[m, k] w_hat[n, k], the weights as
// the GEMV kernel reads them (E2M1 codes [N, K/2], E4M3 scales per 16 and a tensor scale S for
// NVFP4, "Hardware-invariant NVFP4 progress report 1", "The NVFP4 layout"; E8M0 scales per 32
// for MXFP4, "Low-Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", Step 6).
//
// Two kernels per pass of up to 32 rows of x:
//   * fp4_xprep_kernel, one CTA per row of x (rows padded with zeros to whole passes):
//     the row in FP16 under one power of two (largest |x| in [2^14, 2^15); exact for BF16
//     values within 29 binades of the row's largest), written in the MMA's B-fragment order
//     (for 8 rows and a 32-k block: row-major 16-byte runs of 8 k, unit 4 row + quarter, so
//     lane 4 gq + c of a warp reads unit lane of one 512-byte run, without bank conflicts),
//     and 2^-e per row;
//   * fp4_matmul_tc_kernel: the GEMV kernel's structure (units of T tiles of 16 weight rows
//     and all of K, a producer warp streaming 512-k chunks by TMA into a ring, warp (t, p)
//     taking tile t and the 32-k blocks p, p + P, ... of every chunk) with each chunk's slice
//     of x (8 KB per 8 rows) copied beside the weights, so that a weight fragment is decoded
//     once and feeds the m16n8k16 MMAs of every 8 rows of x (the n8 columns). NVFP4 scales the
//     FP16 code pairs by their E4M3 block scale before the MMAs (exact: an E2M1 value times an
//     E4M3 scale lies inside FP16's normal range; the GEMV instead keeps the 16-k blocks apart
//     in the n8 columns, which here hold the rows of x) and accumulates over all of K; MXFP4
//     starts each 32-k block's MMAs from zero and adds the block's fp32 sums times its
//     power-of-two scale. The P k-parts of a unit are added in a
//     fixed order through shared memory; y = S 2^-e_m (sum) in BF16.
// Rows of x beyond 32 take further passes (the weights stream again; a larger M belongs on a
// tcgen05 tile kernel).
#include "common.cuh"
#include "fp4_common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kMBoxK = 256;               // 128 code bytes per row: one 128-byte swizzle row
constexpr int kMChunkK = 512;             // two code boxes per chunk
constexpr int kMBlocks = kMChunkK / 32;   // 32-k blocks per chunk
constexpr int kMXSlice = kMBlocks * 512;  // bytes of x per 8 rows and chunk
constexpr int kMMaxStages = 8;
constexpr uint32_t kMSmem = 227u * 1024u - 1024u;  // the base is aligned up to 1024 B
constexpr int kXprepThreads = 256;

struct MLayout {
  uint32_t code_bytes, scale_bytes, x_off, stage_bytes, red_off, bar_off, total;
  __host__ __device__ MLayout(int T, int MB, int stages, int sb) {
    code_bytes = 4096u * static_cast<uint32_t>(T);  // two boxes of 16 T rows x 128 B
    scale_bytes = static_cast<uint32_t>(sb) * 16u * static_cast<uint32_t>(T);
    x_off = (code_bytes + scale_bytes + 1023u) & ~1023u;
    stage_bytes = x_off + static_cast<uint32_t>(MB) * kMXSlice;
    red_off = static_cast<uint32_t>(stages) * stage_bytes;             // [8 MB][16 T + 1] fp32
    bar_off = red_off + (16u * static_cast<uint32_t>(T) + 1u) * 8u * static_cast<uint32_t>(MB) * 4u;
    total = bar_off + 2u * kMMaxStages * 8u + 16u;
  }
};

template <int NT>
__device__ __forceinline__ void m_consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// x [M, K] BF16 -> xf (FP16, B-fragment order, Mp rows: M rounded up to a whole number of
// passes, the rows past M zero) and u[m] = 2^-e_m (0 past M).
// Unit (16 bytes) ((mc * K/32 + b) * 8 + gq) * 4 + c of xf holds x[8 mc + gq, 32 b + 8 c ..
// 32 b + 8 c + 7] 2^e.
__global__ void __launch_bounds__(kXprepThreads)
    fp4_xprep_kernel(const uint16_t* __restrict__ x, int M, int K, uint4* __restrict__ xf,
                     float* __restrict__ u) {
  __shared__ float red[kXprepThreads / 32];
  pdl_launch_dependents();
  pdl_wait();  // x may come from the previous kernel; xf and u may still be read by it
  const int m = blockIdx.x, tid = threadIdx.x;
  const int segs = K / 8;
  const int mc = m >> 3, gq = m & 7;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K);
  float amax = 0.f;
  if (m < M) {
    for (int s = tid; s < segs; s += kXprepThreads) {
      float v[8];
      f_bf16x8(__ldg(src + s), v);
#pragma unroll
      for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(v[q]));
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kXprepThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const int e = f_x_exponent(amax);
  const float sc = f_pow2(e);
  const size_t base = static_cast<size_t>(mc) * (K / 32);
  for (int s = tid; s < segs; s += kXprepThreads) {
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (m < M) {
      float v[8];
      f_bf16x8(__ldg(src + s), v);
      out = f_f16x8(v, sc);
    }
    xf[((base + static_cast<size_t>(s >> 2)) * 8 + gq) * 4 + static_cast<size_t>(s & 3)] = out;
  }
  if (tid == 0) u[m] = m < M ? f_pow2(-e) : 0.f;
}

struct MMaps {
  CUtensorMap codes;   // uint8 [N, K/2], box {128, 16 T}, 128-byte swizzle
  // uint8 [N, K/16] (NVFP4, box {32, 16 T}, 32-byte swizzle) or [N, K/32] (MXFP4, box
  // {16, 16 T}, no swizzle)
  CUtensorMap scales;
};

// One pass over rows m0 .. m0 + 8 MB - 1 of x (those below M are written). xf points at the
// pass's first 8-row group.
template <bool MX, int T, int P, int MB>
__global__ void __launch_bounds__(T * P * 32 + 32, 1)
    fp4_matmul_tc_kernel(const __grid_constant__ MMaps maps, const uint8_t* __restrict__ xf,
                         const float* __restrict__ u, const float* __restrict__ tensor_scale,
                         uint16_t* __restrict__ y, int M, int N, int K, int m0, int nunits,
                         int stages, uint32_t* __restrict__ status, uint64_t limit_ns) {
  constexpr int W = T * P;          // consumer warps
  constexpr int NC = W * 32;        // consumer threads
  constexpr int NB = kMBlocks / P;  // 32-k blocks of a chunk per warp
  constexpr int SB = MX ? 16 : 32;  // scale bytes per row and chunk
  constexpr int ROWS = 16 * T;      // weight rows per unit
  constexpr int NCH = MB == 1 ? 2 : 1;  // NVFP4 accumulator chains per 8 rows of x
  static_assert(kMBlocks % P == 0, "bad warp split");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const MLayout L(T, MB, stages, SB);
  float* sRed = reinterpret_cast<float*>(smem + L.red_off);  // [8 MB][ROWS + 1]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kMMaxStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kMMaxStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kchunks = K / kMChunkK;
  const size_t xrow_bytes = static_cast<size_t>(K) * 16;  // one 8-row group of xf
  const uint32_t w_bytes = L.code_bytes + L.scale_bytes;
  const uint32_t tx_bytes = w_bytes + static_cast<uint32_t>(MB) * kMXSlice;

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
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&maps.codes);
      tma_prefetch_desc(&maps.scales);
      const int per_cta = kchunks * ((nunits - static_cast<int>(blockIdx.x) +
                                      static_cast<int>(gridDim.x) - 1) /
                                     static_cast<int>(gridDim.x));
      auto weights = [&](int j) {
        const int s = j % stages;
        const int unit = static_cast<int>(blockIdx.x) + (j / kchunks) * static_cast<int>(gridDim.x);
        const int kc = j % kchunks;
        uint8_t* buf = smem + s * L.stage_bytes;
        mbar_arrive_expect_tx(&full[s], tx_bytes);
        tma_load_2d(buf, &maps.codes, &full[s], kc * (kMChunkK / 2), unit * ROWS);
        tma_load_2d(buf + L.code_bytes / 2, &maps.codes, &full[s],
                    kc * (kMChunkK / 2) + kMBoxK / 2, unit * ROWS);
        tma_load_2d(buf + L.code_bytes, &maps.scales, &full[s], kc * SB, unit * ROWS);
      };
      auto xslices = [&](int j) {
        const int s = j % stages;
        const int kc = j % kchunks;
        uint8_t* buf = smem + s * L.stage_bytes + L.x_off;
#pragma unroll
        for (int i = 0; i < MB; ++i)
          bulk_load(buf + i * kMXSlice,
                    xf + static_cast<size_t>(i) * xrow_bytes + static_cast<size_t>(kc) * kMXSlice,
                    kMXSlice, &full[s]);
      };
      // The weights of the first stages go out before the wait for the previous kernel (which
      // writes xf); their x follows it.
      const int first = per_cta < stages ? per_cta : stages;
      for (int j = 0; j < first; ++j) weights(j);
      pdl_wait();
      for (int j = 0; j < first; ++j) xslices(j);
      int j = first;
      for (; j < per_cta; ++j) {
        const int s = j % stages;
        const uint32_t use = static_cast<uint32_t>(j / stages);
        if (!mbar_wait_bounded(&empty[s], (use - 1) & 1u, abort_flag, status, limit_ns)) break;
        weights(j);
        xslices(j);
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
  pdl_wait();  // u comes from the previous kernel; y may still be read by an earlier one
  const int gq = lane >> 2, c = lane & 3;
  const int t = warp % T, p = warp / T;  // tile in the unit, first 32-k block in a chunk
  const uint32_t rowA = static_cast<uint32_t>(16 * t + gq);  // rowB = rowA + 8
  // NVFP4 scale box: 32-byte swizzle (16-byte halves of a row swap where bit 2 of the row is
  // set), so rows gq and gq + 4 read different banks.
  uint32_t code_off[NB], x_off[NB], s_off[NB];
  const uint32_t sswz = MX ? 0u : (static_cast<uint32_t>(gq) & 4u) << 2;
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    const uint32_t j = static_cast<uint32_t>(p + P * r);
    code_off[r] = (j >> 3) * (L.code_bytes / 2) + rowA * 128u +
                  (((j & 7u) ^ static_cast<uint32_t>(gq)) << 4) + 4u * static_cast<uint32_t>(c);
    x_off[r] = L.x_off + (j * 32u + static_cast<uint32_t>(lane)) * 16u;  // unit 32 j + 4 gq + c
    s_off[r] = rowA * SB + (MX ? j : ((2u * j) ^ sswz));
  }
  const uint32_t ssel = static_cast<uint32_t>(c >> 1) * 0x11u;
  const uint32_t ring_base = smem_addr(smem);
  const float S = MX ? 1.0f : __ldg(tensor_scale);
  int s = 0;
  uint32_t phase = 0u;
  for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
    const int row0 = unit * ROWS;
    // acc[i][NCH][4]: D fragment of x rows 8 i + 2c, 8 i + 2c + 1 and weight rows rowA, rowB
    float acc[MB][NCH][4] = {};
    for (int kc = 0; kc < kchunks; ++kc) {
      const bool landed = mbar_wait_bounded(&full[s], phase, abort_flag, status, limit_ns);
      const uint32_t buf = ring_base + static_cast<uint32_t>(s) * L.stage_bytes;
      const uint32_t sbox = buf + L.code_bytes;
      if (landed) {
#pragma unroll
        for (int r = 0; r < NB; ++r) {
          const uint32_t w0 = f_lds32(buf + code_off[r]);
          const uint32_t w1 = f_lds32(buf + code_off[r] + 1024u);
          uint32_t p0[4], p1[4];
          f_e2m1_pairs(w0, p0);
          f_e2m1_pairs(w1, p1);
          if constexpr (!MX) {
            const uint32_t qa = f_lds_u16(sbox + s_off[r]);
            const uint32_t qb = f_lds_u16(sbox + s_off[r] + 8u * SB);
            const uint32_t sA = f_e4m3_pair(__byte_perm(qa, 0u, ssel));
            const uint32_t sB = f_e4m3_pair(__byte_perm(qb, 0u, ssel));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              p0[q] = f_hmul2(p0[q], sA);
              p1[q] = f_hmul2(p1[q], sB);
            }
#pragma unroll
            for (int i = 0; i < MB; ++i) {
              const uint4 e = f_lds128(buf + x_off[r] + static_cast<uint32_t>(i) * kMXSlice);
              float (&d)[4] = acc[i][NCH == 2 ? (r & 1) : 0];
              f_mma(d, p0[0], p1[0], p0[1], p1[1], e.x, e.y);
              f_mma(d, p0[2], p1[2], p0[3], p1[3], e.z, e.w);
            }
          } else {
            const float sA = f_e8m0(f_lds_u8(sbox + s_off[r]));
            const float sB = f_e8m0(f_lds_u8(sbox + s_off[r] + 8u * SB));
#pragma unroll
            for (int i = 0; i < MB; ++i) {
              const uint4 e = f_lds128(buf + x_off[r] + static_cast<uint32_t>(i) * kMXSlice);
              float d[4] = {0.f, 0.f, 0.f, 0.f};
              f_mma(d, p0[0], p1[0], p0[1], p1[1], e.x, e.y);
              f_mma(d, p0[2], p1[2], p0[3], p1[3], e.z, e.w);
              acc[i][0][0] = fmaf(sA, d[0], acc[i][0][0]);
              acc[i][0][1] = fmaf(sA, d[1], acc[i][0][1]);
              acc[i][0][2] = fmaf(sB, d[2], acc[i][0][2]);
              acc[i][0][3] = fmaf(sB, d[3], acc[i][0][3]);
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
    // The P k-parts of the unit, in order p = 0, 1, ...: red[row][m] (8 MB columns).
    for (int q = 0; q < P; ++q) {
      if (p == q) {
#pragma unroll
        for (int i = 0; i < MB; ++i) {
          float v[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) v[f] = NCH == 2 ? acc[i][0][f] + acc[i][NCH - 1][f] : acc[i][0][f];
          const int mA = 8 * i + 2 * c;
          float* ra = sRed + mA * (ROWS + 1) + rowA;  // column m of D, rows rowA, rowA + 8
          float* rb = ra + 8;
          if (q == 0) {
            ra[0] = v[0];
            ra[ROWS + 1] = v[1];
            rb[0] = v[2];
            rb[ROWS + 1] = v[3];
          } else {
            ra[0] += v[0];
            ra[ROWS + 1] += v[1];
            rb[0] += v[2];
            rb[ROWS + 1] += v[3];
          }
        }
      }
      m_consumer_bar<NC>();
    }
    for (int idx = tid; idx < ROWS * 8 * MB; idx += NC) {
      const int m = idx / ROWS, row = idx % ROWS;
      const int n = row0 + row, mg = m0 + m;
      if (n < N && mg < M)
        y[static_cast<size_t>(mg) * N + n] = __bfloat16_as_ushort(
            __float2bfloat16_rn(S * __ldg(u + mg) * sRed[m * (ROWS + 1) + row]));
    }
    m_consumer_bar<NC>();
  }
}

struct MCfg {
  int T, P;
};
constexpr MCfg kMCfgs[] = {{2, 8}, {6, 4}, {12, 2}};
constexpr int kMNumCfgs = static_cast<int>(sizeof(kMCfgs) / sizeof(kMCfgs[0]));

struct MPlan {
  int cfg = -1, nunits = 0, stages = 0;
};

MPlan m_plan(int N, int K, int MB, int sms, int sb) {
  MPlan p;
  if (K % kMChunkK != 0 || N <= 0 || sms <= 0) return p;
  const int tiles = (N + 15) / 16;
  const int need = (tiles + sms - 1) / sms;
  int ci = 0;
  while (ci + 1 < kMNumCfgs && kMCfgs[ci].T < need) ++ci;
  for (; ci >= 0; --ci) {
    const int T = kMCfgs[ci].T;
    const uint32_t fixed = MLayout(T, MB, 0, sb).total;
    const uint32_t stage = MLayout(T, MB, 0, sb).stage_bytes;
    int stages = fixed < kMSmem ? static_cast<int>((kMSmem - fixed) / stage) : 0;
    if (stages > kMMaxStages) stages = kMMaxStages;
    if (stages >= 2) {
      p.cfg = ci;
      p.nunits = (tiles + T - 1) / T;
      p.stages = stages;
      return p;
    }
  }
  return p;
}

template <bool MX, int T, int P, int MB>
cudaError_t launch_pass(const MMaps& maps, const uint8_t* xf, const float* u,
                        const float* tensor_scale, uint16_t* y, int M, int N, int K, int m0,
                        const MPlan& plan, int sms, uint32_t* status, uint64_t limit_ns,
                        cudaStream_t stream) {
  const uint32_t smem = MLayout(T, MB, plan.stages, MX ? 16 : 32).total + 1024u;
  auto kern = fp4_matmul_tc_kernel<MX, T, P, MB>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = plan.nunits < sms ? plan.nunits : sms;
  return launch_with_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(T * P * 32 + 32), smem,
                         stream, maps, xf, u, tensor_scale, y, M, N, K, m0, plan.nunits,
                         plan.stages, status, limit_ns);
}

template <bool MX, int MB>
cudaError_t launch_pass_mb(const MMaps& maps, const uint8_t* xf, const float* u,
                           const float* tensor_scale, uint16_t* y, int M, int N, int K, int m0,
                           const MPlan& plan, int sms, uint32_t* status, uint64_t limit_ns,
                           cudaStream_t stream) {
  switch (plan.cfg) {
    case 0:
      return launch_pass<MX, 2, 8, MB>(maps, xf, u, tensor_scale, y, M, N, K, m0, plan, sms,
                                       status, limit_ns, stream);
    case 1:
      return launch_pass<MX, 6, 4, MB>(maps, xf, u, tensor_scale, y, M, N, K, m0, plan, sms,
                                       status, limit_ns, stream);
    case 2:
      return launch_pass<MX, 12, 2, MB>(maps, xf, u, tensor_scale, y, M, N, K, m0, plan, sms,
                                        status, limit_ns, stream);
    default:
      return cudaErrorNotSupported;
  }
}

int pass_blocks(int rows) { return rows <= 8 ? 1 : rows <= 16 ? 2 : 4; }

// Rows of x that the prepared copy holds: M rounded up to the passes' 8, 16 or 32 rows.
int padded_rows(int M) { return M <= 8 ? 8 : M <= 16 ? 16 : (M + 31) / 32 * 32; }

}  // namespace

size_t fp4_matmul_workspace_bytes(int M, int K) {
  if (M <= 1 || K <= 0) return 0;
  const size_t mp = static_cast<size_t>(padded_rows(M));
  return mp * static_cast<size_t>(K) * 2 + mp * 4;
}

bool fp4_matmul_supports(int N, int K, bool mx) {
  const int sms = device_sm_count();
  for (int mb : {1, 2, 4})
    if (m_plan(N, K, mb, sms, mx ? 16 : 32).cfg < 0) return false;
  return true;
}

cudaError_t launch_fp4_matmul(const uint16_t* x, const uint8_t* codes, const uint8_t* scales,
                              const float* tensor_scale, uint16_t* y, int M, int N, int K,
                              bool mx, void* workspace, uint32_t* status, uint64_t wait_limit_ns,
                              cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int mp = padded_rows(M);
  uint8_t* xf = static_cast<uint8_t*>(workspace);
  float* u = reinterpret_cast<float*>(xf + static_cast<size_t>(mp) * K * 2);
  cudaError_t e = launch_with_pdl(fp4_xprep_kernel, dim3(static_cast<unsigned>(mp)),
                                  dim3(kXprepThreads), 0, stream, x, M, K,
                                  reinterpret_cast<uint4*>(xf), u);
  if (e != cudaSuccess) return e;
  for (int m0 = 0; m0 < M; m0 += 32) {
    const int mb = pass_blocks(M - m0);
    const MPlan plan = m_plan(N, K, mb, sms, mx ? 16 : 32);
    if (plan.cfg < 0) return cudaErrorNotSupported;
    const int T = kMCfgs[plan.cfg].T;
    MMaps maps;
    e = encode_tensor_map(&maps.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes,
                          static_cast<uint64_t>(K) / 2, static_cast<uint64_t>(N),
                          static_cast<uint64_t>(K) / 2, kMBoxK / 2,
                          static_cast<uint32_t>(16 * T), CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const uint64_t srow = mx ? static_cast<uint64_t>(K) / 32 : static_cast<uint64_t>(K) / 16;
    e = encode_tensor_map(&maps.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, scales, srow,
                          static_cast<uint64_t>(N), srow, mx ? 16u : 32u,
                          static_cast<uint32_t>(16 * T),
                          mx ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_32B);
    if (e != cudaSuccess) return e;
    const uint8_t* xp = xf + static_cast<size_t>(m0 / 8) * static_cast<size_t>(K) * 16;
    if (mx) {
      e = mb == 1 ? launch_pass_mb<true, 1>(maps, xp, u, nullptr, y, M, N, K, m0, plan, sms,
                                            status, wait_limit_ns, stream)
        : mb == 2 ? launch_pass_mb<true, 2>(maps, xp, u, nullptr, y, M, N, K, m0, plan, sms,
                                            status, wait_limit_ns, stream)
                  : launch_pass_mb<true, 4>(maps, xp, u, nullptr, y, M, N, K, m0, plan, sms,
                                            status, wait_limit_ns, stream);
    } else {
      e = mb == 1 ? launch_pass_mb<false, 1>(maps, xp, u, tensor_scale, y, M, N, K, m0, plan,
                                             sms, status, wait_limit_ns, stream)
        : mb == 2 ? launch_pass_mb<false, 2>(maps, xp, u, tensor_scale, y, M, N, K, m0, plan,
                                             sms, status, wait_limit_ns, stream)
                  : launch_pass_mb<false, 4>(maps, xp, u, tensor_scale, y, M, N, K, m0, plan,
                                             sms, status, wait_limit_ns, stream);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4k
