// The prepared (reordered) W4A16 layout and the tensor-core matmul that reads it.
//
// The pages' production advice is to rearrange the weights once, offline, so that the
// kernel's wide reads feed the tensor-core operand directly ("Quantization and GEMV", "What
// production kernels do"; "Low-Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", "In
// the real world": reordered tiles whose nibbles convert with one mask-and-or; "Hardware-
// invariant NVFP4 progress report 1", "Is it faster?": a handle that owns prepared weights).
// The prepared layout holds the same codes, scales and minimums as the canonical one, cut into
// records of 128 weight columns x 128 k (one group), 8704 bytes each (4.25 bits per weight):
//
//   record (t, g) at byte (t * K/128 + g) * 8704:
//     uint32 word b*1024 + h*512 + n*4 + j (b, h < 2, n < 128, j < 4): the 8 codes of column
//       128 t + n at k = 128 g + 64 b + 8 (4 h + j) + 0..7, the code of k0 + 2i in bits 4i and
//       the code of k0 + 2i + 1 in bits 16 + 4i;
//     uint32 word 2048 + n: BF16 scale (bits 0..15) and BF16 minimum (bits 16..31).
//   Columns past N (the last tile) hold code 0, scale 0 and minimum 0.
//
// Why this order. Each 64-k half of a record is one contiguous 4 KB copy; the thread that
// rebuilds column n reads its 8 words with two 16-byte shared loads that are contiguous across
// the warp (no bank conflict, no swizzle); in each word the even weights sit in the low half
// and the odd ones in the high half, so ((w >> 4i) & 0x000F000F) | 0x43004300 is the BF16 pair
// (128 + q_2i, 128 + q_2i+1) for the MMA operand, one shift and one LOP3 per pair (the
// canonical order needs a byte permute instead of the shift); the scale and minimum of a
// column arrive as one 32-bit word.
//
// w4a16_tcp_kernel<BN>: y^T tile (128 weight columns x BN batch rows) = W_hat tile (tensor
// memory, the MMA's A operand) x x tile (shared memory, B operand), BF16 in, fp32 sums.
//   * Warp roles: warp 0 streams x tiles (TMA, 128-byte swizzle) and the prepared codes and
//     scale|minimum words (bulk copies) into a ring; warp 1 issues tcgen05.mma (one thread);
//     warps 2-5 drain the accumulator (one TMEM lane quarter each); warps 6-13 rebuild the
//     weights in two sets of four (one per lane quarter), each set taking every other
//     64-k block, so that two blocks are rebuilt at a time into a ring of TMEM stages.
//   * Persistent grid, at most one CTA per SM. The work is the list of (128-column tile,
//     BN-row tile) units, each K/64 blocks long. With a workspace the blocks of all units are
//     cut into equal contiguous ranges, one per CTA (stream-K): a unit split between CTAs is
//     summed by the last CTA to finish its part, which adds the fp32 partials in k order
//     (deterministic) and resets the unit's arrival counter. Without one, CTAs take whole
//     units in turn.
//   * Accumulators are double-buffered in tensor memory when 2 BN columns fit beside the
//     weight stages (BN <= 128), so that the drain of one unit overlaps the next unit's MMAs.
//   * Every mbarrier wait is bounded; an expired wait latches a status bit, the roles stop,
//     the CTA waits (bounded) for its copies and MMAs in flight, frees TMEM and returns.
#include "common.cuh"
#include "launch.h"

namespace w4k {
namespace {

constexpr int kTile = 128;                  // weight columns per tile (MMA M)
constexpr uint32_t kRecWords = 2176;        // one (tile, group) record
constexpr uint32_t kRecBytes = kRecWords * 4u;
constexpr int kDequantSets = 2;

// Per batch tile BN: SA slots of x (two 64-k slabs of BN rows) paired with SA TMEM stages of
// rebuilt weights (64 columns = 128 k each) and LS slots of prepared records (a deeper ring:
// the weights stream ahead of x). Copies are issued by four producer warps (records and x,
// each split by stage parity): one issuing thread sustains only ~7.5 B/cycle of 4 KB
// requests and ~15 of 8 KB ones, a quarter to two thirds of an SM's share of HBM. For BN <= 64
// two MMA issuers take alternate stages into accumulators of their own (one issuer spends
// ~56 cycles per small MMA, two reach the tensor pipe's ~40). Accumulators are
// double-buffered when they fit beside the weight stages.
template <int BN>
struct Tcp {
  static constexpr bool kDual = BN <= 64;
  static constexpr int kIssuers = kDual ? 2 : 1;
  static constexpr bool kDoubleAcc = BN <= 128;
  static constexpr int kAccBufs = kDoubleAcc ? 2 : 1;
  static constexpr int kAccCols = BN * kIssuers * kAccBufs;
  static constexpr uint32_t kACol0 = static_cast<uint32_t>(kAccCols < 32 ? 32 : kAccCols);
  static constexpr uint32_t kTmemCols = 512u;
  // Stage i uses slot i % depth, and its copies, rebuild and MMAs are done by the producer,
  // rebuild set and (with two) MMA issuer of parity i & 1. Even depths keep every slot with
  // one party of each kind, whose waits then step through the slot's barrier phases one by
  // one; with an odd depth consecutive uses of a slot alternate between parties, and a party
  // can fall two phases behind and read a completed phase of the same parity as its own.
  static constexpr int SA = BN <= 16 ? 6 : BN == 32 ? 6 : BN <= 128 ? 4 : 2;
  static constexpr int LS = BN <= 32 ? 12 : BN == 64 ? 10 : BN == 128 ? 8 : 10;
  // warps: 0 records (even stages), 1 MMA (even stages, or all), 2-5 epilogue, 6-13 rebuild,
  // 14 records (odd), 15 x (even), 16 x (odd), 17 MMA (odd; two issuers only)
  static constexpr int kWarps = kDual ? 18 : 17;
  static constexpr int kThreads = kWarps * 32;
  static constexpr uint32_t x_bytes = static_cast<uint32_t>(BN) * 256u;  // [2][BN][64] bf16
  static constexpr uint32_t x_off = 0;
  static constexpr uint32_t code_off = x_off + SA * x_bytes;
  static constexpr uint32_t bar_off = code_off + LS * kRecBytes;
  // cfull[LS], cempty[LS], xfull[SA], afull[SA], done[SA], accfull[2], accempty[2], drain[2]
  static constexpr uint32_t nbars = 2u * LS + 3u * SA + 6u;
  static constexpr uint32_t misc_off = bar_off + nbars * 8u;
  static constexpr uint32_t total = misc_off + 16u;  // tmem address, abort, fixup, drain-fail flags
  static constexpr uint32_t alloc = total + 1024u;    // slack to align the base to 1024 B
  static_assert(SA % 2 == 0 && LS % 2 == 0, "each ring slot must belong to one stage parity");
  static_assert(kACol0 % 32u == 0u && kACol0 + SA * 64u <= kTmemCols, "TMEM overflow");
  static_assert(x_bytes % 1024u == 0u, "x slabs keep 1024-byte alignment");
  static_assert(alloc <= 227u * 1024u, "shared memory overflow");
};

// The list of (unit, stage range) segments one CTA works on, identical in every role; a
// stage is 128 k (one group, one prepared record). Stream-K: CTA c covers linear stages
// [c total / G, (c + 1) total / G) of the units laid end to end (unit u = stages
// [u KS, (u + 1) KS)); G <= total, so no range is empty. Whole units: CTA c takes units c,
// c + G, ...
struct Segments {
  long long idx, hi;
  int KS, u_next, G, nunits;
  bool stream, first;
  __device__ Segments(bool stream_mode, int c, int G_, long long total, int KS_, int nunits_)
      : KS(KS_), u_next(c), G(G_), nunits(nunits_), stream(stream_mode), first(true) {
    idx = stream ? static_cast<long long>(c) * total / G : 0;
    hi = stream ? static_cast<long long>(c + 1) * total / G : 0;
  }
  // Next segment: unit u, stages [s0, s1); is_first = first segment of this CTA.
  __device__ bool next(int& u, int& s0, int& s1, bool& is_first) {
    is_first = first;
    first = false;
    if (stream) {
      if (idx >= hi) return false;
      u = static_cast<int>(idx / KS);
      s0 = static_cast<int>(idx - static_cast<long long>(u) * KS);
      const long long end = min(hi, static_cast<long long>(u + 1) * KS);
      s1 = s0 + static_cast<int>(end - idx);
      idx = end;
      return true;
    }
    if (u_next >= nunits) return false;
    u = u_next;
    s0 = 0;
    s1 = KS;
    u_next += G;
    return true;
  }
};

// The same list one stage at a time: unit u and group g of each stage.
struct Stages {
  Segments seg;
  int u = 0, g = 0, g1 = 0;
  __device__ explicit Stages(const Segments& s) : seg(s) {}
  __device__ bool next(int& uo, int& go) {
    if (g >= g1) {
      bool f;
      if (!seg.next(u, g, g1, f)) return false;
    }
    uo = u;
    go = g++;
    return true;
  }
};

// The CTA whose stream-K range holds linear stage `idx`: the c with
// floor(c T / G) <= idx < floor((c + 1) T / G), i.e. ceil((idx + 1) G / T) - 1.
__device__ __forceinline__ int sk_owner(long long idx, long long total, int G) {
  return static_cast<int>(((idx + 1) * G - 1) / total);
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Load 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Rebuild one packed word of the prepared layout (even codes in the low half, odd in the
// high half) into four BF16 pairs w_hat = q s + min, k = 2i and 2i + 1 in pair i.
__device__ __forceinline__ void rebuild_word(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 m2,
                                             uint32_t* out) {
  const uint32_t b128 = 0x43004300u;  // BF16 (128, 128)
  const __nv_bfloat162 off = *reinterpret_cast<const __nv_bfloat162*>(&b128);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p = and_or<0x000F000Fu>(i == 0 ? w : (w >> (4 * i)), b128);  // 128 + q, exact
    const __nv_bfloat162 q2 = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&p), off);
    const __nv_bfloat162 wv = __hfma2(q2, s2, m2);  // q s + min, one rounding
    out[i] = *reinterpret_cast<const uint32_t*>(&wv);
  }
}

template <int BN>
__global__ void __launch_bounds__(Tcp<BN>::kThreads, 1)
    w4a16_tcp_kernel(const __grid_constant__ CUtensorMap xmap, const uint8_t* __restrict__ prep,
                     uint16_t* __restrict__ y, int M, int N, int K, int P, int T, int stream_k,
                     float* __restrict__ ws_partial, uint32_t* __restrict__ ws_counter,
                     uint32_t* __restrict__ status, uint64_t limit_ns) {
  using L = Tcp<BN>;
  constexpr int SA = L::SA, LS = L::LS, NI = L::kIssuers;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint64_t* cfull = bars;             // a prepared record landed (bulk copy bytes)
  uint64_t* cempty = cfull + LS;      // its rebuild set has read it (4 warps)
  uint64_t* xfull = cempty + LS;      // an x slot landed (TMA bytes)
  uint64_t* afull = xfull + SA;       // a weight stage is in TMEM and its x landed (4 warps)
  uint64_t* done = afull + SA;        // the stage's MMAs are done: x slot and TMEM stage free
  uint64_t* accfull = done + SA;      // [2] (one commit per issuer)
  uint64_t* accempty = accfull + 2;   // [2] (4 epilogue warps)
  uint64_t* drain = accempty + 2;     // [2] (one per issuer)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile uint32_t* abort_flag = tmem_holder + 1;
  volatile uint32_t* fix_flag = tmem_holder + 2;
  volatile uint32_t* epi_fail = tmem_holder + 3;  // an epilogue warp's wait expired

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KS = K / 128;  // stages (groups) per unit
  const int nunits = P * T;
  const long long total = static_cast<long long>(nunits) * KS;
  const int G = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < LS; ++s) {
      mbar_init(&cfull[s], 1);
      mbar_init(&cempty[s], 4);
    }
    for (int a = 0; a < SA; ++a) {
      mbar_init(&xfull[a], 1);
      mbar_init(&afull[a], 4);
      mbar_init(&done[a], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], NI);
      mbar_init(&accempty[b], 4);
      mbar_init(&drain[b], 1);
    }
    *abort_flag = 0u;
    *epi_fail = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 15 && lane == 0) tma_prefetch_desc(&xmap);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  // Dependent launches only once this CTA holds its tensor memory.
  if (threadIdx.x == 0) pdl_launch_dependents();

  const Segments segs0(stream_k != 0, static_cast<int>(blockIdx.x), G, total, KS, nunits);
  Segments segs = segs0;
  int u = 0, g0 = 0, g1 = 0;
  bool first = false;

  if (warp == 0 || warp == 14) {
    // ---------------- prepared records, one producer per stage parity ----------------
    // Weights are never written by the kernels this one overlaps: no wait on the previous
    // kernel here.
    if (lane == 0) {
      const int par = warp == 0 ? 0 : 1;
      Stages st(segs0);
      int i = 0, uu = 0, gg = 0, issued = 0;
      while (st.next(uu, gg)) {
        if ((i & 1) == par) {
          const int s = i % LS;
          if (i >= LS &&
              !mbar_wait_bounded(&cempty[s], ((i / LS) - 1) & 1, abort_flag, status, limit_ns))
            break;
          mbar_arrive_expect_tx(&cfull[s], kRecBytes);
          bulk_load(smem + L::code_off + s * kRecBytes,
                    prep + (static_cast<size_t>(uu / P) * KS + gg) * kRecBytes, kRecBytes,
                    &cfull[s]);
          issued = i + 1;
        }
        ++i;
      }
      if (*abort_flag) {
        // Let this warp's copies in flight land before the CTA can exit.
        volatile uint32_t no_abort = 0u;
        for (int k = (issued - 2 * LS > 0 ? issued - 2 * LS : 0); k < issued; ++k)
          if ((k & 1) == par && k + LS >= issued)
            mbar_wait_bounded(&cfull[k % LS], (k / LS) & 1, &no_abort, status, limit_ns);
      }
    }
  } else if (warp == 15 || warp == 16) {
    // ---------------- x, one producer per stage parity ----------------
    if (lane == 0) {
      const int par = warp == 15 ? 0 : 1;
      pdl_wait();  // x may be written by the previous kernel
      Stages st(segs0);
      int i = 0, uu = 0, gg = 0, issued = 0;
      while (st.next(uu, gg)) {
        if ((i & 1) == par) {
          const int a = i % SA;
          if (i >= SA &&
              !mbar_wait_bounded(&done[a], ((i / SA) - 1) & 1, abort_flag, status, limit_ns))
            break;
          mbar_arrive_expect_tx(&xfull[a], L::x_bytes);
          const int p = uu - (uu / P) * P;
          tma_load_3d(smem + L::x_off + a * L::x_bytes, &xmap, &xfull[a], 0, p * BN, 2 * gg);
          issued = i + 1;
        }
        ++i;
      }
      if (*abort_flag) {
        volatile uint32_t no_abort = 0u;
        for (int k = (issued - 2 * SA > 0 ? issued - 2 * SA : 0); k < issued; ++k)
          if ((k & 1) == par && k + SA >= issued)
            mbar_wait_bounded(&xfull[k % SA], (k / SA) & 1, &no_abort, status, limit_ns);
      }
    }
  } else if (warp == 1 || warp == 17) {
    // ---------------- MMA issuers: one wait, eight MMAs, one commit per stage -----------
    if (lane == 0) {
      const int par = warp == 1 ? 0 : 1;
      constexpr uint32_t idesc = idesc_bf16_f32(kTile, BN);
      int i = 0, j = 0;
      bool ok = true;
      while (ok && segs.next(u, g0, g1, first)) {
        const int buf = L::kDoubleAcc ? (j & 1) : 0;
        if (j >= L::kAccBufs &&
            !mbar_wait_bounded(&accempty[buf], ((j / L::kAccBufs) - 1) & 1, abort_flag, status,
                               limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>((buf * NI + par) * BN);
        bool started = false;
        for (int g = g0; g < g1; ++g, ++i) {
          if (NI == 2 && (i & 1) != par) continue;
          const int a = i % SA;
          if (!mbar_wait_bounded(&afull[a], (i / SA) & 1, abort_flag, status, limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t xs = smem_addr(smem + L::x_off + a * L::x_bytes);
          const uint32_t ac = tmem + L::kACol0 + static_cast<uint32_t>(a * 64);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_a_tmem(d, ac + kk * 8,
                          smem_desc_kmajor_sw128(xs + (kk >> 2) * (BN * 128) + (kk & 3) * 32),
                          idesc, (started || kk > 0) ? 1u : 0u);
          started = true;
          tc_commit(&done[a]);
        }
        if (!ok) break;
        tc_commit(&accfull[buf]);  // also when this issuer had no stage in the segment
        ++j;
      }
      // Whatever happened, wait until every MMA issued here has completed.
      tc_commit(&drain[par]);
      volatile uint32_t no_abort = 0u;
      mbar_wait_bounded(&drain[par], 0u, &no_abort, status, limit_ns);
    }
  } else if (warp < 6) {
    // ---------------- epilogue: drain accumulators ----------------
    // After an expired wait the four warps keep walking the segment list without working,
    // so that all of them still meet at every named barrier of the split units.
    pdl_wait();  // y and the workspace may still be in use by the previous kernel
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int nl = q * 32 + lane;  // column within the tile
    int j = 0, i = 0;
    bool ok = true;
    while (segs.next(u, g0, g1, first)) {
      const int t = u / P, p = u - t * P;
      const int buf = L::kDoubleAcc ? (j & 1) : 0;
      const bool whole = g0 == 0 && g1 == KS;
      // With two issuers, parity r's accumulator holds this segment's stages of parity r;
      // a one-stage segment leaves the other parity's accumulator unwritten.
      const int len = g1 - g0;
      const bool use1 = NI == 2 && (len >= 2 || (i & 1) == 1);
      const bool use0 = NI == 1 || len >= 2 || (i & 1) == 0;
      i += len;
      ++j;
      if (ok && !mbar_wait_bounded(&accfull[buf], ((j - 1) / L::kAccBufs) & 1, abort_flag,
                                   status, limit_ns))
        ok = false;
      // Lanes leave the wait at different times: the tcgen05 loads below are .sync.aligned and
      // must be executed by the whole warp together.
      ok = __all_sync(0xffffffffu, ok);
      const int n = t * kTile + nl;
      if (ok) {
        tc_fence_after_sync();
        const uint32_t acc0 = tmem + lane_off + static_cast<uint32_t>(buf * NI * BN);
        float* part = nullptr;
        if (!whole)
          part = ws_partial + (static_cast<size_t>(2 * blockIdx.x + (first ? 0 : 1)) * BN) * kTile;
        constexpr int CH = BN < 32 ? BN : 32;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += CH) {
          // Both accumulators are loaded unconditionally (a .sync.aligned load must not sit in
          // a branch); an unwritten one is ignored below.
          uint32_t v[32], w[32];
          __syncwarp();
          if constexpr (CH == 32)
            tmem_ld_32cols(acc0 + c0, v);
          else
            tmem_ld_16cols(acc0 + c0, v);
          if constexpr (NI == 2) {
            if constexpr (CH == 32)
              tmem_ld_32cols(acc0 + BN + c0, w);
            else
              tmem_ld_16cols(acc0 + BN + c0, w);
          }
          tmem_ld_wait();
          float f[32];
#pragma unroll
          for (int jj = 0; jj < CH; ++jj)
            f[jj] = (use0 ? __uint_as_float(v[jj]) : 0.f) +
                    ((NI == 2 && use1) ? __uint_as_float(w[jj]) : 0.f);
          if (whole) {
            if (n < N) {
#pragma unroll
              for (int jj = 0; jj < CH; ++jj) {
                const int m = p * BN + c0 + jj;
                if (m < M)
                  y[static_cast<size_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(f[jj]));
              }
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < CH; ++jj) __stcg(part + (c0 + jj) * kTile + nl, f[jj]);
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[buf]);
      } else if (lane == 0) {
        *epi_fail = 1u;
      }
      if (whole) continue;
      // Split unit: count this CTA's part in; the last part to arrive adds all of them in
      // k order and stores y. A CTA whose drain failed does not count its part.
      __threadfence();
      __syncwarp();
      asm volatile("bar.sync 3, 128;" ::: "memory");
      const long long ub = static_cast<long long>(u) * KS;
      const int c_first = sk_owner(ub, total, G), c_last = sk_owner(ub + KS - 1, total, G);
      if (threadIdx.x == 64) {
        const uint32_t ncov = static_cast<uint32_t>(c_last - c_first + 1);
        *fix_flag = (*epi_fail == 0u && atomicAdd(ws_counter + u, 1u) + 1u == ncov) ? 1u : 0u;
      }
      __syncwarp();
      asm volatile("bar.sync 3, 128;" ::: "memory");
      if (*epi_fail) ok = false;
      if (*fix_flag) {
        __threadfence();
        const int rows = min(BN, M - p * BN);
        constexpr int RB = BN < 32 ? BN : 32;  // rows per batch: all their loads in flight
#pragma unroll 1
        for (int r0 = 0; r0 < rows; r0 += RB) {
          float sum[RB];
#pragma unroll
          for (int rr = 0; rr < RB; ++rr) sum[rr] = 0.f;
#pragma unroll 1
          for (int cc = c_first; cc <= c_last; ++cc) {
            const long long beg = static_cast<long long>(cc) * total / G;
            const int slot = 2 * cc + (beg / KS == u ? 0 : 1);
            const float* src = ws_partial + (static_cast<size_t>(slot) * BN + r0) * kTile + nl;
            float v[RB];
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) v[rr] = __ldcg(src + rr * kTile);
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) sum[rr] += v[rr];
          }
          if (n < N) {
#pragma unroll
            for (int rr = 0; rr < RB; ++rr)
              if (r0 + rr < rows)
                y[static_cast<size_t>(p * BN + r0 + rr) * N + n] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(sum[rr]));
          }
        }
      }
      __syncwarp();
      asm volatile("bar.sync 3, 128;" ::: "memory");
      if (threadIdx.x == 64 && *fix_flag) ws_counter[u] = 0u;  // ready for the next call
    }
  } else if (warp < 14) {
    // ---------------- weight rebuild: two sets of four warps, alternate stages ----------
    const int set = (warp - 6) >> 2;
    const int q = warp & 3;
    const int nl = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t code_base = smem_addr(smem + L::code_off) + static_cast<uint32_t>(nl * 16);
    const uint32_t const_base = smem_addr(smem + L::code_off) + 8192u + static_cast<uint32_t>(nl * 4);
    int i = 0;
    bool ok = true;
    while (ok && segs.next(u, g0, g1, first)) {
      for (int g = g0; g < g1; ++g, ++i) {
        if ((i & 1) != set) continue;
        const int s = i % LS, a = i % SA;
        bool got = mbar_wait_bounded(&cfull[s], (i / LS) & 1, abort_flag, status, limit_ns) &&
                   mbar_wait_bounded(&xfull[a], (i / SA) & 1, abort_flag, status, limit_ns) &&
                   (i < SA || mbar_wait_bounded(&done[a], ((i / SA) - 1) & 1, abort_flag, status,
                                                limit_ns));
        got = __all_sync(0xffffffffu, got);  // reconverge: the TMEM stores below are aligned
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t cb = code_base + static_cast<uint32_t>(s) * kRecBytes;
        const uint4 v0 = lds128(cb);          // (b 0, h 0): k 0..31 of the group
        const uint4 v1 = lds128(cb + 2048u);  // (b 0, h 1): k 32..63
        const uint4 v2 = lds128(cb + 4096u);  // (b 1, h 0): k 64..95
        const uint4 v3 = lds128(cb + 6144u);  // (b 1, h 1): k 96..127
        const uint32_t cs = lds32(const_base + static_cast<uint32_t>(s) * kRecBytes);
        __syncwarp();
        if (lane == 0) mbar_arrive(&cempty[s]);  // the record is in registers
        const uint32_t s2u = __byte_perm(cs, 0u, 0x1010), m2u = __byte_perm(cs, 0u, 0x3232);
        const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2u);
        const __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&m2u);
        const uint32_t dst = lane_base + L::kACol0 + static_cast<uint32_t>(a * 64);
        uint32_t out[32];
        rebuild_word(v0.x, s2, m2, out + 0);
        rebuild_word(v0.y, s2, m2, out + 4);
        rebuild_word(v0.z, s2, m2, out + 8);
        rebuild_word(v0.w, s2, m2, out + 12);
        rebuild_word(v1.x, s2, m2, out + 16);
        rebuild_word(v1.y, s2, m2, out + 20);
        rebuild_word(v1.z, s2, m2, out + 24);
        rebuild_word(v1.w, s2, m2, out + 28);
        __syncwarp();
        tmem_st_32cols(dst, out);
        rebuild_word(v2.x, s2, m2, out + 0);
        rebuild_word(v2.y, s2, m2, out + 4);
        rebuild_word(v2.z, s2, m2, out + 8);
        rebuild_word(v2.w, s2, m2, out + 12);
        rebuild_word(v3.x, s2, m2, out + 16);
        rebuild_word(v3.y, s2, m2, out + 20);
        rebuild_word(v3.z, s2, m2, out + 24);
        rebuild_word(v3.w, s2, m2, out + 28);
        __syncwarp();
        tmem_st_32cols(dst + 32u, out);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[a]);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// canonical -> prepared
// ---------------------------------------------------------------------------
// Even codes of a canonical word (nibbles 0, 2, 4, 6) to the low half, odd ones to the high.
__device__ __forceinline__ uint32_t interleave_word(uint32_t w) {
  const uint32_t e = (w & 0xFu) | ((w >> 4) & 0xF0u) | ((w >> 8) & 0xF00u) | ((w >> 12) & 0xF000u);
  const uint32_t o =
      ((w >> 4) & 0xFu) | ((w >> 8) & 0xF0u) | ((w >> 12) & 0xF00u) | ((w >> 16) & 0xF000u);
  return e | (o << 16);
}

// One thread per (tile t, group g, block b, half h, column n): four words (j = 0..3) written
// as one 16-byte store; the (b, h) = (0, 0) thread also writes the column's scale|minimum.
__global__ void w4a16_prepare_kernel(const uint32_t* __restrict__ qw,
                                     const uint16_t* __restrict__ scales,
                                     const uint16_t* __restrict__ mins, int N, int K,
                                     uint32_t* __restrict__ prep, long long items) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= items) return;
  const int groups = K / 128;
  const int n = static_cast<int>(idx % kTile);
  long long rest = idx / kTile;
  const int h = static_cast<int>(rest & 1);
  rest >>= 1;
  const int b = static_cast<int>(rest & 1);
  rest >>= 1;
  const int g = static_cast<int>(rest % groups);
  const int t = static_cast<int>(rest / groups);
  const int col = t * kTile + n;
  uint32_t* rec = prep + (static_cast<size_t>(t) * groups + g) * kRecWords;
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 16 * g + 8 * b + 4 * h + j;
    out[j] = col < N ? interleave_word(__ldg(qw + static_cast<size_t>(r) * N + col)) : 0u;
  }
  *reinterpret_cast<uint4*>(rec + b * 1024 + h * 512 + n * 4) = make_uint4(out[0], out[1], out[2], out[3]);
  if (b == 0 && h == 0) {
    uint32_t sm = 0u;
    if (col < N)
      sm = static_cast<uint32_t>(__ldg(scales + static_cast<size_t>(g) * N + col)) |
           (static_cast<uint32_t>(__ldg(mins + static_cast<size_t>(g) * N + col)) << 16);
    rec[2048 + n] = sm;
  }
}

template <int BN>
cudaError_t launch_bn(const uint16_t* x, const uint8_t* prep, uint16_t* y, int M, int N, int K,
                      const TcpPlan& plan, float* partial, uint32_t* counter, uint32_t* status,
                      uint64_t limit_ns, cudaStream_t stream) {
  using L = Tcp<BN>;
  auto kern = w4a16_tcp_kernel<BN>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(L::alloc));
  if (e != cudaSuccess) return e;
  // x [M, K] seen as [K/64][M][64]: one load brings both 64-k slabs of a 128-k stage.
  CUtensorMap xmap;
  const uint64_t dims[3] = {64u, static_cast<uint64_t>(M), static_cast<uint64_t>(K / 64)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K) * 2, 128u};
  const uint32_t box[3] = {64u, static_cast<uint32_t>(BN), 2u};
  e = encode_tensor_map_3d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  return launch_with_pdl(kern, dim3(static_cast<unsigned>(plan.ctas)), dim3(L::kThreads), L::alloc,
                         stream, xmap, prep, y, M, N, K, plan.P, plan.T, plan.stream_k ? 1 : 0,
                         partial, counter, status, limit_ns);
}

}  // namespace

size_t w4a16_prepared_bytes(int N, int K) {
  if (N <= 0 || K <= 0 || K % 128 != 0) return 0;
  return static_cast<size_t>((N + kTile - 1) / kTile) * (K / 128) * kRecBytes;
}

int tcp_block_n(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

bool tcp_plan(int M, int N, int K, int sms, bool want_stream, TcpPlan* plan) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 != 0 || sms <= 0) return false;
  TcpPlan p;
  p.bn = tcp_block_n(M);
  p.P = (M + p.bn - 1) / p.bn;
  p.T = (N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(p.P) * p.T;
  const long long total = units * (K / 128);
  if (units > 0x7FFFFFFFll / 2 || p.P > 0x7FFF) return false;
  // Whole units unless they would leave most SMs idle (or there is no workspace): measured on
  // the 14336 x 4096 layer (112 units), whole units beat the stream-K split at every M; on
  // narrow layers (a few units) the split is what puts the SMs to work.
  if (!want_stream || units * 2 >= sms) {
    p.stream_k = false;
    p.ctas = static_cast<int>(units < sms ? units : sms);
    p.counter_bytes = 0;
    p.ws_bytes = 0;
  } else {
    p.stream_k = true;
    long long g = total;  // at least one stage (128 k) per CTA
    if (g > sms) g = sms;
    if (g < 1) g = 1;
    p.ctas = static_cast<int>(g);
    p.counter_bytes = ((static_cast<size_t>(units) * 4 + 255) / 256) * 256;
    p.ws_bytes = p.counter_bytes + static_cast<size_t>(2 * p.ctas) * p.bn * kTile * 4;
  }
  *plan = p;
  return true;
}

cudaError_t launch_w4a16_prepare(const uint32_t* qw, const uint16_t* scales, const uint16_t* mins,
                                 int N, int K, uint32_t* prep, cudaStream_t stream) {
  const long long items = static_cast<long long>((N + kTile - 1) / kTile) * (K / 128) * 4 * kTile;
  const long long blocks = (items + 255) / 256;
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  w4a16_prepare_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(qw, scales, mins, N, K,
                                                                          prep, items);
  return cudaGetLastError();
}

cudaError_t launch_w4a16_tcp(const uint16_t* x, const uint32_t* prep, uint16_t* y, int M, int N,
                             int K, const TcpPlan& plan, void* workspace, uint32_t* status,
                             uint64_t limit_ns, cudaStream_t stream) {
  float* partial = nullptr;
  uint32_t* counter = nullptr;
  if (plan.stream_k) {
    if (workspace == nullptr) return cudaErrorInvalidValue;
    counter = static_cast<uint32_t*>(workspace);
    partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.counter_bytes);
  }
  const uint8_t* pb = reinterpret_cast<const uint8_t*>(prep);
  switch (plan.bn) {
    case 16: return launch_bn<16>(x, pb, y, M, N, K, plan, partial, counter, status, limit_ns, stream);
    case 32: return launch_bn<32>(x, pb, y, M, N, K, plan, partial, counter, status, limit_ns, stream);
    case 64: return launch_bn<64>(x, pb, y, M, N, K, plan, partial, counter, status, limit_ns, stream);
    case 128: return launch_bn<128>(x, pb, y, M, N, K, plan, partial, counter, status, limit_ns, stream);
    case 256: return launch_bn<256>(x, pb, y, M, N, K, plan, partial, counter, status, limit_ns, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4k
