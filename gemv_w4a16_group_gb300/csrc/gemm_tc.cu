// W4A16 tensor-core kernel for sm_103a: TMA + tcgen05.mma with accumulators in tensor
// memory (TMEM).
//
// What it computes is the pages' tile GEMM ("Low-Precision Kernels: INT4, INT8 and FP8
// Matmuls, Measured", Step 2): per k-block, load packed words and this group's scale and
// minimum, rebuild w_hat = q * s + min as BF16 in registers, multiply on BF16 tensor
// cores with fp32 sums, store BF16. The BF16 weights never reach global memory.
//
// GB300 design (not the Triton kernel's):
//   * Roles: the dequantising warps (4, or 8 for BM = 256: two per TMEM lane quarter, each
//     taking half of every 64-k block) rebuild the weight tile and write it into TMEM with
//     tcgen05.st (a warp owns the 32 TMEM lanes of its quarter); the next warp issues TMA
//     loads (x tile, packed-word tile, scale and min rows) into a shared-memory ring of 4 to
//     12 stages (deeper for narrow tiles); the last issues tcgen05.mma from one thread; the
//     dequantising warps then drain the accumulator (with split K: fp32 partials, summed by
//     the last CTA of the tile to arrive, in split order).
//   * The weight tile is the MMA's A operand straight from TMEM (128 weight columns =
//     128 TMEM lanes, 16 k = 8 columns of BF16 pairs), so the dequantised tile costs no
//     shared-memory bandwidth; x is the B operand (K-major, 128-byte swizzle) from
//     shared memory. The accumulator is y^T: lane = weight column n, column = row m.
//   * One MMA is 128 (n) x BM (m) x 16 (k); BM = 16..256 follows M, so small batches
//     use a narrow tile rather than padding M to 128.
//   * Every mbarrier wait is bounded; an expired wait latches a status bit, stops the
//     pipeline, waits (bounded) for this CTA's copies and MMAs in flight, frees TMEM and
//     returns.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kBN = 128;  // weight columns per CTA (MMA M)
constexpr int kBK = 64;   // k per stage (one 128-byte swizzle row of BF16)
// Warp roles: dequantising warps 0..DQ-1 (TMEM lane quarter w % 4, k-part w / 4 of each
// 64-k block), then the TMA warp and the MMA warp. The widest tile (BM = 256) keeps the
// tensor pipe busiest and gets two dequantising warps per lane quarter; narrower tiles keep
// four so that two CTAs fit on an SM.
template <int BM>
struct Roles {
  static constexpr int kDequantWarps = BM >= 256 ? 8 : 4;
  static constexpr int kParts = kDequantWarps / 4;  // k-parts of a 64-k block
  static constexpr int kTmaWarp = kDequantWarps;
  static constexpr int kMmaWarp = kDequantWarps + 1;
  static constexpr int kThreads = (kDequantWarps + 2) * 32;
  static constexpr int kMinBlocks = BM >= 256 ? 1 : 2;
};
constexpr uint32_t kPkBytes = kBK / 8 * kBN * 4;  // 8 rows x 128 words = 4 KB
constexpr uint32_t kRowBytes = kBN * 2;           // one scale (or min) row = 256 B

template <int BM>
struct Smem {
  // Shared-memory ring (x tile + packed words + scale/min rows per stage): deep for narrow
  // tiles so that ~80-100 KB per SM are in flight against DRAM latency. The rebuilt
  // weight tiles live in a separate, shorter ring of TMEM stages.
  static constexpr int kStages = BM <= 16 ? 12 : BM <= 32 ? 10 : BM <= 64 ? 8 : BM <= 128 ? 6 : 4;
  static constexpr int kAStages = BM <= 32 ? 3 : 4;
  static constexpr uint32_t x_bytes = BM * 128;
  static constexpr uint32_t x_off = 0;
  static constexpr uint32_t pk_off = x_off + kStages * x_bytes;
  static constexpr uint32_t sc_off = pk_off + kStages * kPkBytes;
  static constexpr uint32_t mn_off = sc_off + kStages * kRowBytes;
  static constexpr uint32_t bar_off = mn_off + kStages * kRowBytes;
  // full[S], empty[S], afull[SA], aempty[SA], accfull, drain
  static constexpr uint32_t nbars = 2 * kStages + 2 * kAStages + 2;
  static constexpr uint32_t misc_off = bar_off + nbars * 8;
  static constexpr uint32_t total = misc_off + 16;  // tmem address, abort flag, split count
  static constexpr uint32_t alloc = total + 1024;  // slack to align the base to 1024 B
  static constexpr uint32_t tx_bytes = x_bytes + kPkBytes + 2 * kRowBytes;
  // TMEM: accumulator columns [0, BM), weight stages from a 32-column boundary after it;
  // the allocation is a power of two.
  static constexpr uint32_t a_col0 = BM < 32 ? 32u : static_cast<uint32_t>(BM);
  static constexpr uint32_t tmem_cols =
      (a_col0 + kAStages * 32 <= 128) ? 128u : (a_col0 + kAStages * 32 <= 256) ? 256u : 512u;
  static_assert(a_col0 + kAStages * 32 <= 512, "TMEM overflow");
  static_assert(alloc <= 227u * 1024u, "shared memory overflow");
  static_assert(x_bytes % 1024 == 0, "x stage must keep 1024-byte alignment");
};

// ZP: FP16 scales and zero points (w_hat = (q - z) s) instead of BF16 scales and minimums.
template <int BM, bool ZP>
__global__ void __launch_bounds__(Roles<BM>::kThreads, Roles<BM>::kMinBlocks)
    w4a16_tc_kernel(const __grid_constant__ TcMaps maps, uint16_t* __restrict__ y, int M, int N,
                    int K, uint32_t* __restrict__ status, uint64_t limit_ns,
                    float* __restrict__ ws_partial, uint32_t* __restrict__ ws_counter) {
  using L = Smem<BM>;
  using R = Roles<BM>;
  constexpr int kStages = L::kStages;
  constexpr int kAStages = L::kAStages;
  constexpr int kDequantWarps = R::kDequantWarps, kParts = R::kParts;
  constexpr int kTmaWarp = R::kTmaWarp, kMmaWarp = R::kMmaWarp;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sx = smem + L::x_off;
  uint32_t* spk = reinterpret_cast<uint32_t*>(smem + L::pk_off);
  uint16_t* ssc = reinterpret_cast<uint16_t*>(smem + L::sc_off);
  uint16_t* smn = reinterpret_cast<uint16_t*>(smem + L::mn_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint64_t* full = bars;                        // TMA bytes landed (count 1 + tx)
  uint64_t* empty = bars + kStages;             // MMAs reading the stage are done (commit)
  uint64_t* afull = bars + 2 * kStages;         // weight stage written to TMEM (4 warps)
  uint64_t* aempty = afull + kAStages;          // MMAs reading that TMEM stage are done
  uint64_t* accfull = aempty + kAStages;
  uint64_t* drain = accfull + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * BM;
  // Split K over gridDim.z CTAs: this CTA takes k-blocks [kb0, kb0 + KB).
  const int splits = gridDim.z;
  const int KB_all = K / kBK;
  const int per_split = (KB_all + splits - 1) / splits;
  const int kb0 = blockIdx.z * per_split;
  const int KB = min(KB_all, kb0 + per_split) - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&afull[s], kDequantWarps);
      mbar_init(&aempty[s], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, L::tmem_cols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.qw);
    tma_prefetch_desc(&maps.scales);
    tma_prefetch_desc(&maps.mins);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  // Dependent launches only after this CTA holds its tensor memory: a dependent CTA on the
  // same SM may then wait for this one's columns, but this one never waits for it.
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == kTmaWarp) {
    if (lane == 0) {
      pdl_wait();  // x (in every stage) may be written by the previous kernel
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = (kb / kStages) & 1u;
        if (kb >= kStages && !mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, status, limit_ns))
          break;
        mbar_arrive_expect_tx(&full[s], L::tx_bytes);
        const int gkb = kb0 + kb;
        tma_load_2d(sx + s * L::x_bytes, &maps.x, &full[s], gkb * kBK, m0);
        tma_load_2d(spk + s * (kPkBytes / 4), &maps.qw, &full[s], n0, gkb * (kBK / 8));
        tma_load_2d(ssc + s * kBN, &maps.scales, &full[s], n0, gkb / 2);
        tma_load_2d(smn + s * kBN, &maps.mins, &full[s], n0, gkb / 2);
        ++issued;
      }
      if (*abort_flag) {
        // Let this CTA's copies in flight land before the CTA can exit.
        for (int s = 0; s < kStages && s < issued; ++s) {
          const int last = issued - 1 - ((issued - 1 - s) % kStages);  // last fill of stage s
          volatile uint32_t no_abort = 0u;
          mbar_wait_bounded(&full[s], (last / kStages) & 1u, &no_abort, status, limit_ns);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBN, BM);
      bool ok = true;
      for (int kb = 0; kb < KB && ok; ++kb) {
        const int s = kb % kStages, sa = kb % kAStages;
        ok = mbar_wait_bounded(&afull[sa], (kb / kAStages) & 1u, abort_flag, status, limit_ns) &&
             mbar_wait_bounded(&full[s], (kb / kStages) & 1u, abort_flag, status, limit_ns);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t xs = smem_addr(sx + s * L::x_bytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          tc_mma_a_tmem(tmem, tmem + L::a_col0 + sa * 32 + kk * 8,
                        smem_desc_kmajor_sw128(xs + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
        tc_commit(&aempty[sa]);
      }
      if (ok) tc_commit(accfull);
      // Whatever happened, wait until every MMA issued here has completed.
      tc_commit(drain);
      volatile uint32_t no_abort = 0u;
      mbar_wait_bounded(drain, 0u, &no_abort, status, limit_ns);
    }
  } else if (warp < kDequantWarps) {
    pdl_wait();  // y and the workspace may still be in use by the previous kernel
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = weight column n0 + row
    const int part = warp >> 2;              // this warp's k-part of each 64-k block
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t b128 = 0x43004300u;  // BF16 (128, 128)
    bool ok = true;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % kStages, sa = kb % kAStages;
      bool got = mbar_wait_bounded(&full[s], (kb / kStages) & 1u, abort_flag, status, limit_ns) &&
                 (kb < kAStages || mbar_wait_bounded(&aempty[sa], ((kb / kAStages) - 1) & 1u,
                                                     abort_flag, status, limit_ns));
      // Lanes leave the waits at different times; the TMEM store below is .sync.aligned and
      // must be executed by the whole warp together.
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      const uint32_t sb = ssc[s * kBN + row], mb = smn[s * kBN + row];
      // Zero point: w_hat = (128 + q) s - (128 + z) s in one fp32 FMA per weight (exact for
      // |z| < 8064, where (128 + z) s has at most 24 significant bits), then one rounding to
      // BF16, the same single rounding the minimum form's BF16 FMA makes.
      float zs = 0.f, zc = 0.f;
      if constexpr (ZP) {
        zs = f16_bits_to_f32(sb);
        zc = -zs * (128.0f + f16_bits_to_f32(mb));
      }
      const uint32_t s2u = sb | (sb << 16), m2u = mb | (mb << 16);
      const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2u);
      const __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&m2u);
      const __nv_bfloat162 off = *reinterpret_cast<const __nv_bfloat162*>(&b128);
      constexpr int kWords = kBK / 8 / kParts;  // packed words of this warp's k-part
      uint32_t out[4 * kWords];
#pragma unroll
      for (int cc = 0; cc < kWords; ++cc) {
        const int c = part * kWords + cc;
        const uint32_t w = spk[s * (kPkBytes / 4) + c * kBN + row];
        uint32_t p[4];
        codes_to_bf16x2_consecutive(w, p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if constexpr (ZP) {
            const float lo = __uint_as_float(p[i] << 16), hi = __uint_as_float(p[i] & 0xFFFF0000u);
            const __nv_bfloat162 wv = __floats2bfloat162_rn(fmaf(lo, zs, zc), fmaf(hi, zs, zc));
            out[4 * cc + i] = *reinterpret_cast<const uint32_t*>(&wv);
          } else {
            const __nv_bfloat162 q2 =
                __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p[i]), off);
            const __nv_bfloat162 wv = __hfma2(q2, s2, m2);  // q*s + min, one rounding
            out[4 * cc + i] = *reinterpret_cast<const uint32_t*>(&wv);
          }
        }
      }
      __syncwarp();
      if constexpr (kParts == 1)
        tmem_st_32cols(lane_base + L::a_col0 + sa * 32, out);
      else
        tmem_st_16cols(lane_base + L::a_col0 + sa * 32 + part * 16, out);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[sa]);
    }
    // Epilogue: accumulator lane `row` holds y[m0 + j, n0 + row] in column j.
    const bool have_acc =
        __all_sync(0xffffffffu, ok && mbar_wait_bounded(accfull, 0u, abort_flag, status, limit_ns));
    const int n = n0 + row;
    constexpr int kChunks = BM >= 32 ? BM / 32 : 1;
    if (have_acc) tc_fence_after_sync();
    if (splits == 1) {
      if (have_acc) {
#pragma unroll 1
        for (int c = part; c < kChunks; c += kParts) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld_32cols(lane_base + c * 32, v);  // BM < 32: columns >= BM are never stored
          tmem_ld_wait();
          if (n < N) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + c * 32 + j;
              if (j < BM && m < M)
                y[static_cast<size_t>(m) * N + n] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
            }
          }
        }
      }
    } else {
      // Split K: write this CTA's fp32 partial tile, count arrivals per output tile; the
      // last CTA of the tile sums the partials in split order (deterministic) and stores.
      const size_t Mp = static_cast<size_t>(gridDim.y) * BM;
      if (have_acc) {
        float* mine = ws_partial + static_cast<size_t>(blockIdx.z) * Mp * N;
#pragma unroll 1
        for (int c = part; c < kChunks; c += kParts) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld_32cols(lane_base + c * 32, v);
          tmem_ld_wait();
          if (n < N) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = m0 + c * 32 + j;
              if (j < BM) __stcg(mine + static_cast<size_t>(m) * N + n, __uint_as_float(v[j]));
            }
          }
        }
      }
      __threadfence();
      __syncwarp();
      asm volatile("bar.sync 2, %0;" ::"n"(kDequantWarps * 32) : "memory");
      uint32_t* tile_count = ws_counter + blockIdx.y * gridDim.x + blockIdx.x;
      // Low 16 bits count arrivals; a CTA without a valid partial also sets bit 16.
      if (threadIdx.x == 0) {
        const uint32_t inc = have_acc ? 1u : 0x10001u;
        *reinterpret_cast<volatile uint32_t*>(tmem_holder + 2) = atomicAdd(tile_count, inc) + inc;
      }
      __syncwarp();
      asm volatile("bar.sync 2, %0;" ::"n"(kDequantWarps * 32) : "memory");
      const uint32_t after = *reinterpret_cast<volatile uint32_t*>(tmem_holder + 2);
      const bool last = (after & 0xFFFFu) == static_cast<uint32_t>(splits);
      if (last && after < 0x10000u) {
        __threadfence();
        if (n < N) {
          // 4 rows at a time, up to 4 splits per round: 16 independent loads in flight.
#pragma unroll 1
          for (int j0 = 4 * part; j0 < BM && m0 + j0 < M; j0 += 4 * kParts) {
            float acc[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[jj] = 0.f;
#pragma unroll 1
            for (int z0 = 0; z0 < splits; z0 += 4) {
              float v[4][4];
#pragma unroll
              for (int dz = 0; dz < 4; ++dz)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                  const int z = z0 + dz, m = m0 + j0 + jj;
                  v[dz][jj] = (z < splits && m < M)
                                  ? __ldcg(ws_partial + (static_cast<size_t>(z) * Mp + m) * N + n)
                                  : 0.f;
                }
#pragma unroll
              for (int dz = 0; dz < 4; ++dz)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[jj] += v[dz][jj];
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int m = m0 + j0 + jj;
              if (m < M)
                y[static_cast<size_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[jj]));
            }
          }
        }
      }
      if (threadIdx.x == 0 && last) *tile_count = 0u;  // ready for the next call

    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::tmem_cols);
  }
}

__global__ void bounded_wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the wait must give up after limit_ns.
    mbar_wait_bounded(&bar, 0u, &abort_flag, status, limit_ns);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
cudaError_t encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                      uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle swz) {
  return encode_tensor_map(map, dt, base, inner, outer, row_bytes, box_inner, box_outer, swz);
}

template <int BM, bool ZP>
cudaError_t launch_bm(const TcMaps& maps, uint16_t* y, int M, int N, int K, uint32_t* status,
                      uint64_t limit_ns, const TcSplit& split, cudaStream_t stream) {
  using L = Smem<BM>;
  auto kern = w4a16_tc_kernel<BM, ZP>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern),
                                       static_cast<int>(L::alloc));
  if (e != cudaSuccess) return e;
  dim3 grid((N + kBN - 1) / kBN, (M + BM - 1) / BM, split.splits);
  if (grid.y > 65535 || split.splits < 1) return cudaErrorInvalidConfiguration;
  return launch_with_pdl(kern, grid, dim3(Roles<BM>::kThreads), L::alloc, stream, maps, y, M, N, K, status,
                         limit_ns, split.partial, split.counter);
}

template <int BM>
int ctas_per_sm_by_tmem() {
  const int by_tmem = static_cast<int>(512u / Smem<BM>::tmem_cols);
  const int by_smem = static_cast<int>((228u * 1024u) / (Smem<BM>::alloc + 1024u));
  return by_tmem < by_smem ? by_tmem : by_smem;
}

}  // namespace

int tc_block_m(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

cudaError_t make_tc_maps(const uint16_t* x, const uint32_t* qw, const uint16_t* scales,
                         const uint16_t* mins, int M, int N, int K, int bm, TcMaps* maps,
                         bool zero_point) {
  const CUtensorMapDataType st =
      zero_point ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cudaError_t e;
  e = encode_2d(&maps->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(K),
                static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 2, kBK,
                static_cast<uint32_t>(bm), CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_2d(&maps->qw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, static_cast<uint64_t>(N),
                static_cast<uint64_t>(K / 8), static_cast<uint64_t>(N) * 4, kBN, kBK / 8,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = encode_2d(&maps->scales, st, scales, static_cast<uint64_t>(N),
                static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N) * 2, kBN, 1,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return encode_2d(&maps->mins, st, mins, static_cast<uint64_t>(N),
                   static_cast<uint64_t>(K / 128), static_cast<uint64_t>(N) * 2, kBN, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t launch_w4a16_tc(const TcMaps& maps, uint16_t* y, int M, int N, int K, int bm,
                            uint32_t* status, uint64_t limit_ns, const TcSplit& split,
                            cudaStream_t stream, bool zero_point) {
#define W4K_TC_BM(BM)                                                                        \
  return zero_point ? launch_bm<BM, true>(maps, y, M, N, K, status, limit_ns, split, stream) \
                    : launch_bm<BM, false>(maps, y, M, N, K, status, limit_ns, split, stream);
  switch (bm) {
    case 16: W4K_TC_BM(16)
    case 32: W4K_TC_BM(32)
    case 64: W4K_TC_BM(64)
    case 128: W4K_TC_BM(128)
    case 256: W4K_TC_BM(256)
    default: return cudaErrorInvalidValue;
  }
#undef W4K_TC_BM
}

int tc_ctas_per_sm(int bm) {
  switch (bm) {
    case 16: return ctas_per_sm_by_tmem<16>();
    case 32: return ctas_per_sm_by_tmem<32>();
    case 64: return ctas_per_sm_by_tmem<64>();
    case 128: return ctas_per_sm_by_tmem<128>();
    default: return ctas_per_sm_by_tmem<256>();
  }
}

cudaError_t launch_bounded_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace w4k
