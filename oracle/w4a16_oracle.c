/*
 * CPU oracle for the W4A16 group-quantized matmul and the Q4 block-32 GEMV.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, scalar, obviously-correct
 * restatement of what the pages define. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it. The CUDA library never calls it and
 * shares no code with it.
 *
 * Build: gcc -O1 -ffp-contract=off -fPIC -shared (no fast-math, no FMA
 * contraction), so that every fp32 step below is one IEEE-754 operation rounded
 * to nearest-even, exactly as written.
 *
 * Sources (page title, section):
 *   [P1] "Low-Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured",
 *        Step 2 (group-128 scale/min, q = round((w-min)/scale), 8 nibbles per
 *        int32 along K, K/8 x N packed matrix, K/128 x N scales and minimums;
 *        the Triton listing's unpacking, which takes k = 8r + j from nibble j
 *        of word r, and its dequantization q*s + m).
 *   [P2] "Why My 4-Bit CUDA Kernel Wasn't Faster", sections "Why fewer bytes
 *        should have helped" and "Loading the same bytes differently" (18-byte
 *        block of 32 codes + 2-byte FP16 scale; decode = code minus bias, times
 *        scale; low nibble is the even weight, high nibble the odd one).
 *   [P4] "Hardware-invariant NVFP4 progress report 1", "The NVFP4 layout"
 *        (E2M1 weights, largest value 6, an E4M3 scale per 16 weights and an
 *        FP32 scale per tensor; NVFP4A16 decodes to 16-bit floats) and [P1]
 *        Step 6 (4.5 bits per value; MX blocks of 32 with an E8M0 scale, the
 *        scale rule, 4.25 bits per value for MXFP4).
 *   [P3] "Quantization and GEMV", exercise 1 (W8A16 GEMV: symmetric per-row
 *        INT8, s = max|w| / 127, one 16-byte load of 16 codes per lane, the
 *        row's scale applied after the sum) and section "W4A16: dequantizing in registers"
 *        (k = 8r + j at bits 4j..4j+3: the lowest nibble holds the first
 *        weight) and "The quantization formulas".
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - round() is round-half-to-even (IEEE default; PyTorch's torch.round).
 *   - s and min are rounded to BF16 first; q is computed against the stored
 *     BF16 values, in fp32: t = (w - min_bf16) / s_bf16, then RNE, then clamp
 *     to [0, 15].
 *   - scale = bf16_rne(fp32((max - min) / 15)) (fp32 subtract, fp32 divide).
 *   - A group whose BF16 scale is zero stores q = 0 (so w_hat = min).
 *   - Q4: scale = fp16_rne(fp32(max|w| / 8)); q = clamp(rne(w / s) + 8, 0, 15);
 *     a zero scale stores q = 8 (w_hat = 0).
 *   - Weights are finite.
 *   - Zero-point format [P3]: s = fp16_rne(fp32((max - min) / 15)); a stored
 *     s of zero becomes 1 (the pages' host code sets s = 1 when it is zero);
 *     z = round(-min / s) against the stored s, stored as fp16;
 *     q = clamp(round(w / s) + z, 0, 15) (the section's formula: the integer
 *     z is added after rounding); round() here is half away from zero, the
 *     rounding of the pages' own host code for this format (std::round).
 *     Codes stay in the pages' layout: words [N, K/8], scales and zeros
 *     [N, K/G].
 *   - NVFP4 [P1 Step 6, P4 "The NVFP4 layout"]: E2M1 codes (2 exponent bits,
 *     bias 1, 1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per 16
 *     weights along K and one fp32 scale per tensor, w_hat = e2m1 * e4m3 * S.
 *     S = fl(amax / 2688) (2688 = 6 * 448 puts the largest block scale at
 *     E4M3's largest finite value; 1 for an all-zero tensor); a block's scale
 *     is the smallest E4M3 value >= fl(amax_b / fl(6 S)), at most 448 ([P4]
 *     "What's left to tune": a scale that E4M3 rounds down would clip the
 *     block's largest weight, so it is rounded up); codes round fl(w / fl(s_b S)) to
 *     the nearest E2M1 value, ties to the even code, saturating at 6; a block
 *     of zeros stores scale 0 and codes 0. Codes [N, K/2] (low nibble = even
 *     k), scales [N, K/16].
 *   - MXFP4 [P1 Step 6]: E2M1 codes, one E8M0 scale (2^(code - 127)) per 32
 *     weights along K. The block scale is the largest power of two <= max|w|
 *     divided by 4 (the largest power of two E2M1 holds): 2^(floor(log2 amax) - 2),
 *     exponent kept in [-127, 127]; codes round w / scale (exact) to the nearest
 *     E2M1 value, ties to the even code, values past 6 clamped to 6; a block of
 *     zeros stores scale code 0 and codes 0. Codes [N, K/2], scales [N, K/32].
 *   - W8A16 [P3 exercise 1]: per row s = fp32(max|w| / 127), kept in fp32 (no
 *     storage type is given); q = clamp(round(fl(w / s)), -127, 127) with the
 *     same half-away rounding; a row of zeros stores s = 0 and q = 0. x and y
 *     are BF16 as in the W4A16 path.
 *
 * Parity pins (tests/test_oracle_pins.py): rounding helpers against PyTorch's
 * own conversions; hand-worked groups in tests/golden/; 4.25 bits/weight and
 * the pages' byte counts; round trips for on-grid weights; one-hot x; constant
 * groups; brute force at N,K <= 64 against exact rational arithmetic; the
 * fp64 matmul against torch.matmul; the pages' ~10 % quantization error band.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE conversions, written from the format definitions.                    */
/* ------------------------------------------------------------------------ */

/* Round a finite double to an integer, ties to even, without relying on the
 * current floating-point environment. */
static double round_half_even(double v) {
  double f = floor(v);
  double frac = v - f; /* exact for |v| < 2^52 */
  if (frac > 0.5) return f + 1.0;
  if (frac < 0.5) return f;
  /* exact tie: pick the even neighbour */
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Convert an fp32 value to a binary format with `mbits` explicit mantissa bits,
 * exponent bias `bias` and largest exponent `emax` (of a finite value), rounding
 * to nearest, ties to even. Returns the bit pattern (sign at bit 15). */
static uint16_t to_small_float(float f, int mbits, int bias, int emax) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  int ebits = 15 - mbits;
  uint16_t exp_all_ones = (uint16_t)(((1u << ebits) - 1u) << mbits);
  if (isnan(f)) return (uint16_t)(sign | exp_all_ones | (1u << (mbits - 1)));
  double a = fabs((double)f);
  if (isinf(f)) return (uint16_t)(sign | exp_all_ones);
  if (a == 0.0) return sign;
  int emin = 1 - bias; /* exponent of the smallest normal */
  int e;
  frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  e -= 1;       /* a = 1.xxx * 2^e */
  if (e < emin) {
    /* subnormal range: units of 2^(emin - mbits) */
    double q = round_half_even(ldexp(a, mbits - emin));
    /* q == 2^mbits is the smallest normal; the encoding below is continuous */
    return (uint16_t)(sign | (uint16_t)q);
  }
  double sig = round_half_even(ldexp(a, mbits - e)); /* in [2^mbits, 2^(mbits+1)] */
  if (sig == ldexp(1.0, mbits + 1)) {
    sig = ldexp(1.0, mbits);
    e += 1;
  }
  if (e > emax) return (uint16_t)(sign | exp_all_ones); /* overflow -> inf */
  uint16_t biased = (uint16_t)(e + bias);
  return (uint16_t)(sign | (uint16_t)(biased << mbits) |
                    (uint16_t)((uint32_t)sig - (1u << mbits)));
}

uint16_t oracle_bf16_rne(float f) { return to_small_float(f, 7, 127, 127); }
uint16_t oracle_fp16_rne(float f) { return to_small_float(f, 10, 15, 15); }

float oracle_bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

float oracle_fp16_to_float(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0x1f) {
    v = m ? NAN : INFINITY;
  } else if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else {
    v = ldexp((double)(m + 1024), e - 15 - 10);
  }
  return (float)(sign ? -v : v);
}

/* Array forms of the conversions (same arithmetic, one call per array). */
void oracle_bf16_rne_array(const float* in, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = oracle_bf16_rne(in[i]);
}
void oracle_fp16_rne_array(const float* in, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = oracle_fp16_rne(in[i]);
}
void oracle_fp16_to_float_array(const uint16_t* in, float* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = oracle_fp16_to_float(in[i]);
}

/* Round an fp32 value to the nearest integer, ties to even (the reading of
 * "round" in [P1] Step 2). */
static float rne_int(float t) { return (float)round_half_even((double)t); }

/* Round an fp32 value to the nearest integer, ties away from zero, keeping the
 * sign of zero (-0.3 -> -0): the rounding of [P3]'s zero-point host code. */
static float round_half_away(float t) {
  double a = floor(fabs((double)t) + 0.5); /* exact: |t| < 2^53 */
  return (float)copysign(a, (double)t);
}

/* ------------------------------------------------------------------------ */
/* W4A16: quantize, pack, dequantize, matmul ([P1] Step 2).                  */
/* ------------------------------------------------------------------------ */

/* w: fp32 [N, K] row-major (one output feature per row, K contiguous).
 * codes: u8 [N, K] (one 4-bit code per byte).
 * scales, mins: bf16 bit patterns [K/G, N] (group-major, N contiguous).
 * Per group of G consecutive weights along K: scale = (max - min) / 15 and
 * q = round((w - min) / scale), 0..15. */
void oracle_w4a16_quantize(const float* w, int N, int K, int G, uint8_t* codes,
                           uint16_t* scales, uint16_t* mins) {
  int groups = K / G;
  for (int n = 0; n < N; ++n) {
    for (int g = 0; g < groups; ++g) {
      const float* wg = w + (size_t)n * K + (size_t)g * G;
      float lo = wg[0], hi = wg[0];
      for (int i = 1; i < G; ++i) {
        if (wg[i] < lo) lo = wg[i];
        if (wg[i] > hi) hi = wg[i];
      }
      volatile float range = hi - lo;        /* one fp32 subtraction */
      volatile float s32 = range / 15.0f;    /* one fp32 division */
      uint16_t s_b = oracle_bf16_rne(s32);
      uint16_t m_b = oracle_bf16_rne(lo);
      scales[(size_t)g * N + n] = s_b;
      mins[(size_t)g * N + n] = m_b;
      float s = oracle_bf16_to_float(s_b);
      float m = oracle_bf16_to_float(m_b);
      for (int i = 0; i < G; ++i) {
        int q;
        if (s == 0.0f) {
          q = 0;
        } else {
          volatile float diff = wg[i] - m; /* fp32 subtraction */
          volatile float t = diff / s;     /* fp32 division */
          float r = rne_int(t);
          q = r < 0.0f ? 0 : (r > 15.0f ? 15 : (int)r);
        }
        codes[(size_t)n * K + (size_t)g * G + i] = (uint8_t)q;
      }
    }
  }
}

/* Pack 8 codes per 32-bit word along K: word (r, n) holds k = 8r + j in bits
 * 4j..4j+3, first element in the low nibble ([P1] Step 2 listing comment
 * places k = 8r + j in nibble j of word r; [P3] puts the first weight in the lowest
 * nibble).
 * qw: int32 [K/8, N], N contiguous. */
void oracle_w4a16_pack(const uint8_t* codes, int N, int K, int32_t* qw) {
  for (int r = 0; r < K / 8; ++r) {
    for (int n = 0; n < N; ++n) {
      uint32_t word = 0;
      for (int j = 0; j < 8; ++j) {
        uint32_t q = codes[(size_t)n * K + (size_t)r * 8 + j] & 0xFu;
        word |= q << (4 * j);
      }
      qw[(size_t)r * N + n] = (int32_t)word;
    }
  }
}

/* Code of weight (n, k) read back from the packed matrix. */
static int unpack_code(const int32_t* qw, int N, int n, int k) {
  uint32_t word = (uint32_t)qw[(size_t)(k / 8) * N + n];
  return (int)((word >> (4 * (k % 8))) & 0xFu);
}

/* w_hat[n, k] = q * s + min in fp64 ([P1] Step 2: "q * s + m"). The product of
 * a 4-bit integer and a BF16 scale is exact in fp64, and so is the sum with a
 * BF16 minimum unless their exponents differ by more than ~40. */
void oracle_w4a16_dequant(const int32_t* qw, const uint16_t* scales, const uint16_t* mins,
                          int N, int K, int G, double* w_hat) {
  for (int n = 0; n < N; ++n) {
    for (int k = 0; k < K; ++k) {
      int g = k / G;
      double s = (double)oracle_bf16_to_float(scales[(size_t)g * N + n]);
      double m = (double)oracle_bf16_to_float(mins[(size_t)g * N + n]);
      w_hat[(size_t)n * K + k] = (double)unpack_code(qw, N, n, k) * s + m;
    }
  }
}

/* y_ref[m, n] = sum_k x[m, k] * w_hat[n, k] in fp64, and
 * abs_ref[m, n] = sum_k |x[m, k] * w_hat[n, k]| (the scale of the rounding
 * error allowed to a BF16/fp32 implementation).
 * x: bf16 bit patterns [M, K]; result arrays [M, N]. */
void oracle_w4a16_matmul(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                         const uint16_t* mins, int M, int N, int K, int G, double* y_ref,
                         double* abs_ref) {
  for (int m = 0; m < M; ++m) {
    for (int n = 0; n < N; ++n) {
      double acc = 0.0, acc_abs = 0.0;
      for (int k = 0; k < K; ++k) {
        int g = k / G;
        double s = (double)oracle_bf16_to_float(scales[(size_t)g * N + n]);
        double mn = (double)oracle_bf16_to_float(mins[(size_t)g * N + n]);
        double w_hat = (double)unpack_code(qw, N, n, k) * s + mn;
        double xv = (double)oracle_bf16_to_float(x[(size_t)m * K + k]);
        acc += xv * w_hat;
        acc_abs += fabs(xv * w_hat);
      }
      y_ref[(size_t)m * N + n] = acc;
      if (abs_ref) abs_ref[(size_t)m * N + n] = acc_abs;
    }
  }
}

/* Same as oracle_w4a16_matmul but only for the listed output columns
 * (cols[i] for i < ncols); results are [M, ncols]. Used to check full-size
 * launches on a sample of outputs. */
void oracle_w4a16_matmul_cols(const uint16_t* x, const int32_t* qw, const uint16_t* scales,
                              const uint16_t* mins, int M, int N, int K, int G,
                              const int32_t* cols, int ncols, double* y_ref,
                              double* abs_ref) {
  for (int m = 0; m < M; ++m) {
    for (int i = 0; i < ncols; ++i) {
      int n = cols[i];
      double acc = 0.0, acc_abs = 0.0;
      for (int k = 0; k < K; ++k) {
        int g = k / G;
        double s = (double)oracle_bf16_to_float(scales[(size_t)g * N + n]);
        double mn = (double)oracle_bf16_to_float(mins[(size_t)g * N + n]);
        double w_hat = (double)unpack_code(qw, N, n, k) * s + mn;
        double xv = (double)oracle_bf16_to_float(x[(size_t)m * K + k]);
        acc += xv * w_hat;
        acc_abs += fabs(xv * w_hat);
      }
      y_ref[(size_t)m * ncols + i] = acc;
      if (abs_ref) abs_ref[(size_t)m * ncols + i] = acc_abs;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Prepared (reordered) W4A16 layout ([P3] "What production kernels do": the  */
/* weights are rearranged offline so that one wide read feeds the tensor-core */
/* operand; [P1] "In the real world": reordered tiles whose nibbles convert   */
/* with one mask-and-or; [P4] "Is it faster?": a handle that owns prepared    */
/* weights). The same codes, scales and minimums, in another order:           */
/*                                                                            */
/*   Columns are cut into tiles of 128 (the last one padded with code 0,      */
/*   scale 0, minimum 0) and K into groups of 128. Tile t, group g is one      */
/*   record of 2176 uint32 words (8704 bytes, so 4.25 bits per weight), at    */
/*   word offset (t * K/128 + g) * 2176:                                       */
/*     word b*1024 + h*512 + n*4 + j   (b, h in {0,1}; n < 128; j < 4):        */
/*       the 8 codes of column 128t + n at k = 128g + 64b + 8(4h + j) + 0..7, */
/*       code of k0 + 2i in bits 4i..4i+3 and code of k0 + 2i + 1 in bits     */
/*       16 + 4i..16 + 4i + 3 (i < 4): the even weights in the low half, the   */
/*       odd ones in the high half;                                            */
/*     word 2048 + n: BF16 scale of (g, column 128t + n) in bits 0..15, BF16   */
/*       minimum in bits 16..31.                                               */
/* ------------------------------------------------------------------------ */

#define PREP_TILE 128
#define PREP_RECORD_WORDS 2176

long oracle_w4a16_prepared_words(int N, int K, int G) {
  long tiles = (N + PREP_TILE - 1) / PREP_TILE;
  return tiles * (long)(K / G) * PREP_RECORD_WORDS;
}

/* qw [K/8, N], scales / mins [K/G, N] (G = 128) -> prep (prepared_words words). */
void oracle_w4a16_prepare(const int32_t* qw, const uint16_t* scales, const uint16_t* mins,
                          int N, int K, int G, uint32_t* prep) {
  int tiles = (N + PREP_TILE - 1) / PREP_TILE;
  int groups = K / G;
  for (int t = 0; t < tiles; ++t) {
    for (int g = 0; g < groups; ++g) {
      uint32_t* rec = prep + ((size_t)t * groups + g) * PREP_RECORD_WORDS;
      for (int n = 0; n < PREP_TILE; ++n) {
        int col = t * PREP_TILE + n;
        for (int b = 0; b < 2; ++b) {
          for (int h = 0; h < 2; ++h) {
            for (int j = 0; j < 4; ++j) {
              int k0 = g * G + 64 * b + 8 * (4 * h + j);
              uint32_t word = 0;
              for (int i = 0; i < 4; ++i) {
                uint32_t even = 0, odd = 0;
                if (col < N) {
                  even = (uint32_t)unpack_code(qw, N, col, k0 + 2 * i);
                  odd = (uint32_t)unpack_code(qw, N, col, k0 + 2 * i + 1);
                }
                word |= even << (4 * i);
                word |= odd << (16 + 4 * i);
              }
              rec[b * 1024 + h * 512 + n * 4 + j] = word;
            }
          }
        }
        uint32_t s = 0, m = 0;
        if (col < N) {
          s = scales[(size_t)g * N + col];
          m = mins[(size_t)g * N + col];
        }
        rec[2048 + n] = s | (m << 16);
      }
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Q4 block-32 ([P2]): 32 codes + one FP16 scale, w_hat = (q - 8) * s.       */
/* ------------------------------------------------------------------------ */

/* w: fp32 [N, K]; codes: u8 [N, K/2] (= [N, K/32, 16]; byte j of a block holds
 * weight 2j in the low nibble and weight 2j+1 in the high nibble);
 * scales: fp16 bit patterns [N, K/32]. */
void oracle_q4b32_quantize(const float* w, int N, int K, uint8_t* codes, uint16_t* scales) {
  int blocks = K / 32;
  for (int n = 0; n < N; ++n) {
    for (int b = 0; b < blocks; ++b) {
      const float* wb = w + (size_t)n * K + (size_t)b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(wb[i]);
        if (a > amax) amax = a;
      }
      volatile float s32 = amax / 8.0f; /* one fp32 division */
      uint16_t s_h = oracle_fp16_rne(s32);
      scales[(size_t)n * blocks + b] = s_h;
      float s = oracle_fp16_to_float(s_h);
      int q[32];
      for (int i = 0; i < 32; ++i) {
        if (s == 0.0f) {
          q[i] = 8;
        } else {
          volatile float t = wb[i] / s; /* fp32 division */
          float r = rne_int(t) + 8.0f;
          q[i] = r < 0.0f ? 0 : (r > 15.0f ? 15 : (int)r);
        }
      }
      uint8_t* cb = codes + (size_t)n * (K / 2) + (size_t)b * 16;
      for (int j = 0; j < 16; ++j) cb[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    }
  }
}

static int q4_code(const uint8_t* codes, int K, int n, int k) {
  uint8_t byte = codes[(size_t)n * (K / 2) + (size_t)(k / 2)];
  return (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
}

/* w_hat[n, k] = (q - 8) * s in fp64 (exact). */
void oracle_q4b32_dequant(const uint8_t* codes, const uint16_t* scales, int N, int K,
                          double* w_hat) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) {
      double s = (double)oracle_fp16_to_float(scales[(size_t)n * (K / 32) + k / 32]);
      w_hat[(size_t)n * K + k] = (double)(q4_code(codes, K, n, k) - 8) * s;
    }
}

/* y_ref[n] = sum_b s[n, b] * sum_j (q[n, b, j] - 8) * x[32 b + j], in fp64;
 * abs_ref[n] = sum_k |x[k] * w_hat[n, k]|. x: fp16 bit patterns [K]. Only the
 * listed rows (rows[i], i < nrows) are computed; pass rows = NULL for all N. */
void oracle_q4b32_gemv(const uint16_t* x, const uint8_t* codes, const uint16_t* scales,
                       int N, int K, const int32_t* rows, int nrows, double* y_ref,
                       double* abs_ref) {
  int count = rows ? nrows : N;
  for (int i = 0; i < count; ++i) {
    int n = rows ? rows[i] : i;
    double acc = 0.0, acc_abs = 0.0;
    for (int b = 0; b < K / 32; ++b) {
      double s = (double)oracle_fp16_to_float(scales[(size_t)n * (K / 32) + b]);
      double block = 0.0;
      for (int j = 0; j < 32; ++j) {
        int k = 32 * b + j;
        double xv = (double)oracle_fp16_to_float(x[k]);
        double qv = (double)(q4_code(codes, K, n, k) - 8);
        block += qv * xv;
        acc_abs += fabs(qv * s * xv);
      }
      acc += s * block;
    }
    y_ref[i] = acc;
    if (abs_ref) abs_ref[i] = acc_abs;
  }
}

/* ------------------------------------------------------------------------ */
/* W4A16 with a zero point ([P3] "The quantization formulas", "W4A16:        */
/* dequantizing in registers"): w_hat = (q - z) * s, fp16 s and z.           */
/* ------------------------------------------------------------------------ */

/* w: fp32 [N, K]. qw_rows: uint32 [N, K/8], word (n, r) holds k = 8r + j in
 * bits 4j..4j+3 (the lowest nibble holds the first weight). scales, zeros: fp16 bit
 * patterns [N, K/G] (one per row and group, as [P3] stores them). */
void oracle_w4a16zp_quantize(const float* w, int N, int K, int G, uint32_t* qw_rows,
                             uint16_t* scales, uint16_t* zeros) {
  int groups = K / G;
  memset(qw_rows, 0, (size_t)N * (K / 8) * sizeof(uint32_t));
  for (int n = 0; n < N; ++n) {
    for (int g = 0; g < groups; ++g) {
      const float* wg = w + (size_t)n * K + (size_t)g * G;
      float lo = wg[0], hi = wg[0];
      for (int i = 1; i < G; ++i) {
        if (wg[i] < lo) lo = wg[i];
        if (wg[i] > hi) hi = wg[i];
      }
      volatile float range = hi - lo;     /* fp32 subtraction */
      volatile float s32 = range / 15.0f; /* fp32 division by 2^4 - 1 */
      uint16_t s_h = oracle_fp16_rne(s32);
      if (oracle_fp16_to_float(s_h) == 0.0f) s_h = oracle_fp16_rne(1.0f);
      float s = oracle_fp16_to_float(s_h);
      volatile float neg_lo = -lo;
      volatile float zq = neg_lo / s;     /* fp32 division */
      uint16_t z_h = oracle_fp16_rne(round_half_away(zq));
      float z = oracle_fp16_to_float(z_h);
      scales[(size_t)n * groups + g] = s_h;
      zeros[(size_t)n * groups + g] = z_h;
      for (int i = 0; i < G; ++i) {
        volatile float t = wg[i] / s;     /* fp32 division */
        double r = (double)round_half_away(t) + (double)z;
        int q = r < 0.0 ? 0 : (r > 15.0 ? 15 : (int)r);
        int k = g * G + i;
        qw_rows[(size_t)n * (K / 8) + k / 8] |= (uint32_t)q << (4 * (k % 8));
      }
    }
  }
}

/* Code of weight (n, k) in the [N, K/8] word layout. */
static int unpack_code_rows(const uint32_t* qw_rows, int K, int n, int k) {
  return (int)((qw_rows[(size_t)n * (K / 8) + k / 8] >> (4 * (k % 8))) & 0xFu);
}

/* w_hat[n, k] = (q - z) * s in fp64 ([P3]: subtract the zero point, multiply by
 * the scale). Exact: q - z is an integer below 2^17 and s has 11 significant
 * bits. */
void oracle_w4a16zp_dequant(const uint32_t* qw_rows, const uint16_t* scales,
                            const uint16_t* zeros, int N, int K, int G, double* w_hat) {
  int groups = K / G;
  for (int n = 0; n < N; ++n) {
    for (int k = 0; k < K; ++k) {
      double s = (double)oracle_fp16_to_float(scales[(size_t)n * groups + k / G]);
      double z = (double)oracle_fp16_to_float(zeros[(size_t)n * groups + k / G]);
      w_hat[(size_t)n * K + k] = ((double)unpack_code_rows(qw_rows, K, n, k) - z) * s;
    }
  }
}

/* y_ref[m, i] = sum_k x[m, k] * w_hat[cols[i], k] in fp64 and abs_ref the sum
 * of the magnitudes of the terms; cols == NULL means every column (ncols = N).
 * x: bf16 bit patterns [M, K]; results [M, ncols]. */
void oracle_w4a16zp_matmul(const uint16_t* x, const uint32_t* qw_rows, const uint16_t* scales,
                           const uint16_t* zeros, int M, int N, int K, int G,
                           const int32_t* cols, int ncols, double* y_ref, double* abs_ref) {
  int groups = K / G;
  if (!cols) ncols = N;
  for (int m = 0; m < M; ++m) {
    for (int i = 0; i < ncols; ++i) {
      int n = cols ? cols[i] : i;
      double acc = 0.0, acc_abs = 0.0;
      for (int k = 0; k < K; ++k) {
        double s = (double)oracle_fp16_to_float(scales[(size_t)n * groups + k / G]);
        double z = (double)oracle_fp16_to_float(zeros[(size_t)n * groups + k / G]);
        double w_hat = ((double)unpack_code_rows(qw_rows, K, n, k) - z) * s;
        double xv = (double)oracle_bf16_to_float(x[(size_t)m * K + k]);
        acc += xv * w_hat;
        acc_abs += fabs(xv * w_hat);
      }
      y_ref[(size_t)m * ncols + i] = acc;
      if (abs_ref) abs_ref[(size_t)m * ncols + i] = acc_abs;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* W8A16 ([P3] exercise 1): symmetric per-row INT8, w_hat = q * s.          */
/* ------------------------------------------------------------------------ */

/* w: fp32 [N, K]; q: int8 [N, K]; s: fp32 [N]. */
void oracle_w8a16_quantize(const float* w, int N, int K, int8_t* q, float* s) {
  for (int n = 0; n < N; ++n) {
    const float* row = w + (size_t)n * K;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k)
      if (fabsf(row[k]) > amax) amax = fabsf(row[k]);
    volatile float s32 = amax / 127.0f; /* fp32 division */
    s[n] = s32;
    for (int k = 0; k < K; ++k) {
      int v = 0;
      if (s32 != 0.0f) {
        volatile float t = row[k] / s32; /* fp32 division */
        double r = (double)round_half_away(t);
        v = r < -127.0 ? -127 : (r > 127.0 ? 127 : (int)r);
      }
      q[(size_t)n * K + k] = (int8_t)v;
    }
  }
}

/* y_ref[i] = sum_k x[k] * q[n, k] * s[n] for n = rows[i] (every row when rows
 * is NULL) in fp64, and abs_ref the sum of the magnitudes of the terms.
 * x: bf16 bit patterns [K]. */
void oracle_w8a16_gemv(const uint16_t* x, const int8_t* q, const float* s, int N, int K,
                       const int32_t* rows, int nrows, double* y_ref, double* abs_ref) {
  if (!rows) nrows = N;
  for (int i = 0; i < nrows; ++i) {
    int n = rows ? rows[i] : i;
    double acc = 0.0, acc_abs = 0.0;
    for (int k = 0; k < K; ++k) {
      double w_hat = (double)q[(size_t)n * K + k] * (double)s[n];
      double xv = (double)oracle_bf16_to_float(x[k]);
      acc += xv * w_hat;
      acc_abs += fabs(xv * w_hat);
    }
    y_ref[i] = acc;
    if (abs_ref) abs_ref[i] = acc_abs;
  }
}

/* ------------------------------------------------------------------------ */
/* NVFP4 weights, 16-bit activations ([P4], [P1] Step 6).                   */
/* ------------------------------------------------------------------------ */

/* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal (0 or 0.5). */
double oracle_e2m1_value(int code) {
  int e = (code >> 1) & 3, m = code & 1;
  double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (code & 8) ? -mag : mag;
}

/* E4M3 (the finite-only FN variant): sign, 4 exponent bits (bias 7), 3
 * mantissa bits; exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN, so
 * the largest finite value is 0x7E = 1.75 * 2^8 = 448. */
double oracle_e4m3_value(int code) {
  int e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return (code & 0x80) ? -mag : mag;
}

/* Nearest E2M1 code to t, ties to the code with mantissa bit 0, |t| >= 6
 * gives 6; the sign is kept, zeros included. */
int oracle_e2m1_rne(float t) {
  int sign = signbit(t) ? 8 : 0;
  double a = fabs((double)t);
  int best = 7;
  if (a < 6.0) {
    best = 0;
    for (int c = 0; c < 7; ++c) {
      double lo = oracle_e2m1_value(c), hi = oracle_e2m1_value(c + 1);
      double mid = 0.5 * (lo + hi);
      if (a < mid) { best = c; break; }
      if (a == mid) { best = (c & 1) ? c + 1 : c; break; }
      best = c + 1;
    }
  }
  return sign | best;
}

/* Smallest non-negative E4M3 code whose value is >= v (v >= 0), at most 0x7E. */
int oracle_e4m3_ceil(float v) {
  for (int c = 0; c <= 0x7E; ++c)
    if (oracle_e4m3_value(c) >= (double)v) return c;
  return 0x7E;
}

/* w: fp32 [N, K] (K % 16 == 0); codes: uint8 [N, K/2], byte j of a row holds
 * k = 2j in its low nibble and k = 2j + 1 in its high nibble; scales: E4M3
 * [N, K/16]; tensor_scale: one fp32. */
void oracle_nvfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales,
                           float* tensor_scale) {
  float amax = 0.0f;
  for (size_t i = 0; i < (size_t)N * K; ++i)
    if (fabsf(w[i]) > amax) amax = fabsf(w[i]);
  volatile float S = amax > 0.0f ? amax / 2688.0f : 1.0f; /* fp32 division */
  *tensor_scale = S;
  volatile float d6 = 6.0f * S;
  for (int n = 0; n < N; ++n) {
    for (int b = 0; b < K / 16; ++b) {
      const float* wb = w + (size_t)n * K + (size_t)b * 16;
      float bmax = 0.0f;
      for (int j = 0; j < 16; ++j)
        if (fabsf(wb[j]) > bmax) bmax = fabsf(wb[j]);
      int sc = 0;
      int q[16] = {0};
      if (bmax > 0.0f) {
        volatile float v = bmax / d6; /* fp32 division */
        sc = oracle_e4m3_ceil(v);
        volatile float den = (float)oracle_e4m3_value(sc) * S; /* fp32 product */
        for (int j = 0; j < 16; ++j) {
          volatile float t = wb[j] / den; /* fp32 division */
          q[j] = oracle_e2m1_rne(t);
        }
      }
      scales[(size_t)n * (K / 16) + b] = (uint8_t)sc;
      for (int j = 0; j < 8; ++j)
        codes[(size_t)n * (K / 2) + (size_t)b * 8 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    }
  }
}

/* w_hat[n, k] = e2m1(q) * e4m3(s_b) * S, exact in fp64. */
static double nvfp4_w_hat(const uint8_t* codes, const uint8_t* scales, float S, int K, int n,
                          int k) {
  uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
  int q = (k & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(q) * oracle_e4m3_value(scales[(size_t)n * (K / 16) + k / 16]) *
         (double)S;
}

void oracle_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float S, int N, int K,
                          double* w_hat) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) w_hat[(size_t)n * K + k] = nvfp4_w_hat(codes, scales, S, K, n, k);
}

/* y_ref[i] = sum_k x[k] * w_hat[n, k] for n = rows[i] (every row when rows is
 * NULL), fp64; abs_ref the sum of the magnitudes. x: bf16 bit patterns [K]. */
void oracle_nvfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales, float S,
                       int N, int K, const int32_t* rows, int nrows, double* y_ref,
                       double* abs_ref) {
  if (!rows) nrows = N;
  for (int i = 0; i < nrows; ++i) {
    int n = rows ? rows[i] : i;
    double acc = 0.0, acc_abs = 0.0;
    for (int k = 0; k < K; ++k) {
      double t = (double)oracle_bf16_to_float(x[k]) * nvfp4_w_hat(codes, scales, S, K, n, k);
      acc += t;
      acc_abs += fabs(t);
    }
    y_ref[i] = acc;
    if (abs_ref) abs_ref[i] = acc_abs;
  }
}

/* ------------------------------------------------------------------------ */
/* MXFP4 weights, 16-bit activations ([P1] Step 6, the OCP MX blocks).      */
/* ------------------------------------------------------------------------ */

/* E8M0: an unsigned biased exponent, 2^(code - 127); 255 is NaN. */
double oracle_e8m0_value(int code) { return code == 255 ? NAN : ldexp(1.0, code - 127); }

/* w: fp32 [N, K] (K % 32 == 0); codes: uint8 [N, K/2] (byte j: k = 2j low nibble,
 * 2j + 1 high nibble); scales: E8M0 [N, K/32]. */
void oracle_mxfp4_quantize(const float* w, int N, int K, uint8_t* codes, uint8_t* scales) {
  for (int n = 0; n < N; ++n) {
    for (int b = 0; b < K / 32; ++b) {
      const float* wb = w + (size_t)n * K + (size_t)b * 32;
      double amax = 0.0;
      for (int j = 0; j < 32; ++j)
        if (fabs((double)wb[j]) > amax) amax = fabs((double)wb[j]);
      int sc = 0;
      int q[32] = {0};
      if (amax > 0.0) {
        int e;
        frexp(amax, &e);   /* amax = m 2^e, m in [0.5, 1): floor(log2 amax) = e - 1 */
        int X = (e - 1) - 2;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
        sc = X + 127;
        for (int j = 0; j < 32; ++j) {
          double t = ldexp((double)wb[j], -X); /* exact */
          q[j] = oracle_e2m1_rne((float)t);     /* exact for |t| < 8 */
        }
      }
      scales[(size_t)n * (K / 32) + b] = (uint8_t)sc;
      for (int j = 0; j < 16; ++j)
        codes[(size_t)n * (K / 2) + (size_t)b * 16 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    }
  }
}

static double mxfp4_w_hat(const uint8_t* codes, const uint8_t* scales, int K, int n, int k) {
  uint8_t byte = codes[(size_t)n * (K / 2) + k / 2];
  int q = (k & 1) ? (byte >> 4) : (byte & 15);
  return oracle_e2m1_value(q) * oracle_e8m0_value(scales[(size_t)n * (K / 32) + k / 32]);
}

void oracle_mxfp4_dequant(const uint8_t* codes, const uint8_t* scales, int N, int K,
                          double* w_hat) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) w_hat[(size_t)n * K + k] = mxfp4_w_hat(codes, scales, K, n, k);
}

/* y_ref[i] = sum_k x[k] * w_hat[n, k] for n = rows[i] (every row when rows is
 * NULL), fp64; abs_ref the sum of the magnitudes. x: bf16 bit patterns [K]. */
void oracle_mxfp4_gemv(const uint16_t* x, const uint8_t* codes, const uint8_t* scales, int N,
                       int K, const int32_t* rows, int nrows, double* y_ref, double* abs_ref) {
  if (!rows) nrows = N;
  for (int i = 0; i < nrows; ++i) {
    int n = rows ? rows[i] : i;
    double acc = 0.0, acc_abs = 0.0;
    for (int k = 0; k < K; ++k) {
      double t = (double)oracle_bf16_to_float(x[k]) * mxfp4_w_hat(codes, scales, K, n, k);
      acc += t;
      acc_abs += fabs(t);
    }
    y_ref[i] = acc;
    if (abs_ref) abs_ref[i] = acc_abs;
  }
}
