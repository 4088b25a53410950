"""Each plausible mistake planted in (a temporary copy of) the oracle source must make
at least one pin fail. The mistakes are planted in the oracle, on the CPU; nothing
here touches the CUDA library."""
import os
import tempfile

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "w4a16_oracle.c")

# (id, text in the oracle source, replacement, occurrence index or None for all)
MUTANTS = [
    ("pack_nibble_order_reversed", "word |= q << (4 * j);", "word |= q << (4 * (7 - j));", None),
    ("unpack_nibble_order_reversed", "(word >> (4 * (k % 8)))", "(word >> (4 * (7 - k % 8)))", None),
    ("matmul_drops_min_term", "double w_hat = (double)unpack_code(qw, N, n, k) * s + mn;",
     "double w_hat = (double)unpack_code(qw, N, n, k) * s;", None),
    ("scale_divides_by_16", "range / 15.0f", "range / 16.0f", None),
    ("scale_from_max_not_range", "volatile float range = hi - lo;", "volatile float range = hi;", None),
    ("round_half_away", "static float rne_int(float t) { return (float)round_half_even((double)t); }",
     "static float rne_int(float t) { return roundf(t); }", None),
    ("q_against_fp32_min", "volatile float diff = wg[i] - m;", "volatile float diff = wg[i] - lo;", None),
    ("no_clamp_at_15", "q = r < 0.0f ? 0 : (r > 15.0f ? 15 : (int)r);", "q = r < 0.0f ? 0 : (int)r;", 0),
    ("degenerate_group_code_8", "if (s == 0.0f) {\n          q = 0;", "if (s == 0.0f) {\n          q = 8;", None),
    ("scale_layout_transposed_in_matmul",
     "double s = (double)oracle_bf16_to_float(scales[(size_t)g * N + n]);\n"
     "        double mn = (double)oracle_bf16_to_float(mins[(size_t)g * N + n]);\n"
     "        double w_hat = (double)unpack_code(qw, N, n, k) * s + mn;\n"
     "        double xv = (double)oracle_bf16_to_float(x[(size_t)m * K + k]);\n"
     "        acc += xv * w_hat;",
     "double s = (double)oracle_bf16_to_float(scales[(size_t)n * (K / G) + g]);\n"
     "        double mn = (double)oracle_bf16_to_float(mins[(size_t)n * (K / G) + g]);\n"
     "        double w_hat = (double)unpack_code(qw, N, n, k) * s + mn;\n"
     "        double xv = (double)oracle_bf16_to_float(x[(size_t)m * K + k]);\n"
     "        acc += xv * w_hat;", 0),
    ("matmul_sign_error", "acc += xv * w_hat;", "acc -= xv * w_hat;", None),
    ("x_index_transposed", "x[(size_t)m * K + k]", "x[(size_t)k * M + m]", None),
    ("bf16_truncates", "double sig = round_half_even(ldexp(a, mbits - e));",
     "double sig = floor(ldexp(a, mbits - e));", None),
    ("q4_bias_7", "float r = rne_int(t) + 8.0f;", "float r = rne_int(t) + 7.0f;", None),
    ("q4_nibble_pair_swapped", "cb[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));",
     "cb[j] = (uint8_t)(q[2 * j + 1] | (q[2 * j] << 4));", None),
    ("q4_decode_bias_7", "double qv = (double)(q4_code(codes, K, n, k) - 8);",
     "double qv = (double)(q4_code(codes, K, n, k) - 7);", None),
    ("q4_scale_divides_by_7", "volatile float s32 = amax / 8.0f;", "volatile float s32 = amax / 7.0f;", None),
    ("q4_zero_block_code_0", "if (s == 0.0f) {\n          q[i] = 8;", "if (s == 0.0f) {\n          q[i] = 0;", None),
    ("zp_round_half_even", "return (float)copysign(a, (double)t);",
     "return (float)round_half_even((double)t);", None),
    ("zp_zero_added_before_rounding", "double r = (double)round_half_away(t) + (double)z;",
     "double r = (double)round_half_away(t + z);", None),
    ("zp_zero_sign_flipped", "volatile float neg_lo = -lo;", "volatile float neg_lo = lo;", None),
    ("zp_dequant_adds_zero", "(double)unpack_code_rows(qw_rows, K, n, k) - z) * s;",
     "(double)unpack_code_rows(qw_rows, K, n, k) + z) * s;", None),
    ("zp_zero_scale_kept", "s_h = oracle_fp16_rne(1.0f);", "s_h = s_h;", None),
    ("zp_scale_in_bf16", "uint16_t s_h = oracle_fp16_rne(s32);",
     "uint16_t s_h = oracle_fp16_rne(oracle_bf16_to_float(oracle_bf16_rne(s32)));", None),
    ("zp_matmul_scale_layout_transposed",
     "double s = (double)oracle_fp16_to_float(scales[(size_t)n * groups + k / G]);\n"
     "        double z = (double)oracle_fp16_to_float(zeros[(size_t)n * groups + k / G]);\n"
     "        double w_hat = ((double)unpack_code_rows(qw_rows, K, n, k) - z) * s;\n"
     "        double xv",
     "double s = (double)oracle_fp16_to_float(scales[(size_t)(k / G) * N + n]);\n"
     "        double z = (double)oracle_fp16_to_float(zeros[(size_t)(k / G) * N + n]);\n"
     "        double w_hat = ((double)unpack_code_rows(qw_rows, K, n, k) - z) * s;\n"
     "        double xv", None),
    ("w8_scale_divides_by_128", "volatile float s32 = amax / 127.0f;",
     "volatile float s32 = amax / 128.0f;", None),
    ("w8_round_half_even", "double r = (double)round_half_away(t);\n        v = r < -127.0",
     "double r = round_half_even((double)t);\n        v = r < -127.0", None),
    ("w8_codes_truncated", "double r = (double)round_half_away(t);\n        v = r < -127.0",
     "double r = (double)truncf(t);\n        v = r < -127.0", None),
    ("w8_scale_of_next_row", "double w_hat = (double)q[(size_t)n * K + k] * (double)s[n];",
     "double w_hat = (double)q[(size_t)n * K + k] * (double)s[(n + 1) % N];", None),
    ("w8_amax_without_abs", "if (fabsf(row[k]) > amax) amax = fabsf(row[k]);",
     "if (row[k] > amax) amax = row[k];", None),
    ("nv_ties_away", "if (a == mid) { best = (c & 1) ? c + 1 : c; break; }",
     "if (a == mid) { best = c + 1; break; }", None),
    ("nv_block_scale_nearest", "if (oracle_e4m3_value(c) >= (double)v) return c;",
     "if (oracle_e4m3_value(c) >= (double)v) return (c > 0 && (double)v - oracle_e4m3_value(c - 1) < oracle_e4m3_value(c) - (double)v) ? c - 1 : c;",
     None),
    ("nv_tensor_scale_448", "amax / 2688.0f", "amax / 448.0f", None),
    ("nv_nibbles_swapped", "(uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));",
     "(uint8_t)(q[2 * j + 1] | (q[2 * j] << 4));", None),
    ("nv_e4m3_bias_8", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", None),
    ("nv_e2m1_subnormal_1", "double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
     "double mag = e == 0 ? 1.0 * m : ldexp(1.0 + 0.5 * m, e - 1);", None),
    ("nv_gemv_drops_tensor_scale",
     "return oracle_e2m1_value(q) * oracle_e4m3_value(scales[(size_t)n * (K / 16) + k / 16]) *\n         (double)S;",
     "return oracle_e2m1_value(q) * oracle_e4m3_value(scales[(size_t)n * (K / 16) + k / 16]);",
     None),
    ("mx_scale_exponent_minus_1", "int X = (e - 1) - 2;", "int X = (e - 1) - 1;", None),
    ("mx_scale_from_ceil", "int X = (e - 1) - 2;", "int X = e - 2;", None),
    ("mx_e8m0_bias_128", "ldexp(1.0, code - 127); }", "ldexp(1.0, code - 128); }", None),
    ("mx_codes_unscaled", "double t = ldexp((double)wb[j], -X); /* exact */",
     "double t = (double)wb[j];", None),
    ("mx_scale_code_off_by_one", "sc = X + 127;", "sc = X + 128;", None),
    ("zp_nibble_order_reversed", "(uint32_t)q << (4 * (k % 8));", "(uint32_t)q << (4 * (7 - k % 8));",
     None),
    ("prep_even_odd_halves_swapped",
     "word |= even << (4 * i);\n                word |= odd << (16 + 4 * i);",
     "word |= odd << (4 * i);\n                word |= even << (16 + 4 * i);", None),
    ("prep_words_reversed_in_quad", "int k0 = g * G + 64 * b + 8 * (4 * h + j);",
     "int k0 = g * G + 64 * b + 8 * (4 * h + (3 - j));", None),
    ("prep_halves_of_kblock_swapped", "int k0 = g * G + 64 * b + 8 * (4 * h + j);",
     "int k0 = g * G + 64 * b + 8 * (4 * (1 - h) + j);", None),
    ("prep_kblocks_swapped", "int k0 = g * G + 64 * b + 8 * (4 * h + j);",
     "int k0 = g * G + 64 * (1 - b) + 8 * (4 * h + j);", None),
    ("prep_scale_min_swapped", "rec[2048 + n] = s | (m << 16);", "rec[2048 + n] = m | (s << 16);",
     None),
    ("prep_pairs_adjacent_nibbles", "word |= even << (4 * i);\n                word |= odd << (16 + 4 * i);",
     "word |= even << (8 * i);\n                word |= odd << (8 * i + 4);", None),
]


def _mutate(text, old, new, occurrence):
    assert old in text, f"mutation anchor not found: {old!r}"
    if occurrence is None:
        return text.replace(old, new)
    parts = text.split(old)
    return old.join(parts[:occurrence + 1]) + new + old.join(parts[occurrence + 1:])


@pytest.mark.parametrize("mid,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(mid, old, new, occ, tmp_path):
    with open(SRC) as f:
        text = f.read()
    mutated = _mutate(text, old, new, occ)
    assert mutated != text
    src = tmp_path / f"{mid}.c"
    src.write_text(mutated)
    lib = oracle.compile_to(str(src), str(tmp_path / f"{mid}.so"))
    caught = []
    with oracle.use_library(lib):
        for pin in pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, IndexError, ValueError):
                caught.append(pin.__name__)
                break
    assert caught, f"mutant {mid} passed every pin"


def _matmul_first_row_only(x_bits, *args, **kw):
    import numpy as np
    x = np.asarray(x_bits)
    return _REAL_NV(np.repeat(x[:1], x.shape[0], axis=0), *args, **kw)


def _matmul_rows_reversed(x_bits, *args, **kw):
    import numpy as np
    y, a = _REAL_NV(x_bits, *args, **kw)
    return np.ascontiguousarray(y[::-1]), np.ascontiguousarray(a[::-1])


_REAL_NV = oracle.nvfp4_matmul


@pytest.mark.parametrize("mistake", [_matmul_first_row_only, _matmul_rows_reversed],
                         ids=["fp4_matmul_first_row_only", "fp4_matmul_rows_reversed"])
def test_planted_fp4_matmul_mistake_is_caught(mistake, monkeypatch):
    """The row loop of the FP4 matmul oracle, with a mistake planted in it, fails its pin."""
    monkeypatch.setattr(oracle, "nvfp4_matmul", mistake)
    with pytest.raises(AssertionError):
        pins.pin_fp4_matmul_exact_and_library()
