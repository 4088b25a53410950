"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, never against the oracle itself or the CUDA path.

Every pin is a function ``pin_xxx() -> None`` that raises AssertionError when the
oracle (whatever build ``oracle`` currently routes to) disagrees with the fact.
``tests/test_oracle_pins.py`` runs them against the real oracle and
``tests/test_oracle_mutants.py`` checks that each planted mistake in the oracle
source is caught by at least one of them.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- #
# fixture readers
# --------------------------------------------------------------------------- #

def _records(name):
    """Parse a golden file into a list of (tag, {key: [tokens]}) records."""
    recs, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key in ("group", "block"):
                cur = (vals[0], {})
                recs.append(cur)
            elif key == "codes":
                cur = ("pack", {"codes": vals})
                recs.append(cur)
            else:
                cur[1][key] = vals
    return recs


def _page_sizes():
    out = {}
    with open(os.path.join(GOLDEN, "page_sizes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


def _weights_from(rec):
    if "w_hex" in rec:
        bits = np.array([int(t, 16) for t in rec["w_hex"]], dtype=np.uint32)
        return bits.view(np.float32)
    return np.array([float(t) for t in rec["w_dec"]], dtype=np.float32)


def _bf16(bits):
    return float(torch.tensor([int(bits) & 0xFFFF], dtype=torch.int32).to(torch.int16)
                 .view(torch.bfloat16).float())


def _fp16(bits):
    return float(torch.tensor([int(bits) & 0xFFFF], dtype=torch.int32).to(torch.int16)
                 .view(torch.float16).float())


def _torch_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------- #
# pins
# --------------------------------------------------------------------------- #

def pin_rounding_helpers_match_pytorch():
    """bf16/fp16 round-to-nearest-even against PyTorch's own conversions (a library
    routine), on special values, exact ties and 2^20 random bit patterns."""
    g = np.random.default_rng(123)
    rnd = g.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    specials = np.array([0x00000000, 0x80000000, 0x3F800000, 0x7F7FFFFF, 0xFF7FFFFF,
                         0x7F800000, 0xFF800000, 0x00000001, 0x807FFFFF, 0x3F808000,
                         0x3F818000, 0x3F80C000, 0x477FE000, 0x477FF000, 0x477FEFFF,
                         0x33000000, 0x33000001, 0x33800000, 0x387FE000, 0x38800000],
                        dtype=np.uint32)
    bits = np.concatenate([rnd, specials])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    t = torch.from_numpy(f.copy())
    np.testing.assert_array_equal(oracle.bf16_rne(f), _torch_bits(t.to(torch.bfloat16)))
    np.testing.assert_array_equal(oracle.fp16_rne(f), _torch_bits(t.to(torch.float16)))
    all16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    fin = ((all16 >> 10) & 0x1F) != 0x1F
    got = oracle.fp16_to_float(all16[fin])
    ref = torch.from_numpy(all16[fin].view(np.int16).copy()).view(torch.float16).float().numpy()
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def pin_quantize_hand_worked_groups():
    """Hand-worked groups (tests/golden/w4a16_quantize_groups.txt)."""
    for tag, rec in _records("w4a16_quantize_groups.txt"):
        w = _weights_from(rec).reshape(1, -1)
        codes, scales, mins = oracle.w4a16_quantize(w, group=w.shape[1])
        assert int(scales[0, 0]) == int(rec["scale"][0], 16), (tag, hex(scales[0, 0]))
        assert int(mins[0, 0]) == int(rec["min"][0], 16), (tag, hex(mins[0, 0]))
        assert codes[0].tolist() == [int(v) for v in rec["q"]], (tag, codes[0].tolist())


def pin_pack_hand_worked_words():
    """Hand-worked packed words (tests/golden/w4a16_pack_words.txt)."""
    for _, rec in _records("w4a16_pack_words.txt"):
        codes = np.array([int(v) for v in rec["codes"]], dtype=np.uint8).reshape(1, -1)
        qw = oracle.w4a16_pack(codes)
        got = [int(v) & 0xFFFFFFFF for v in qw[:, 0]]
        assert got == [int(v, 16) for v in rec["words"]], [hex(v) for v in got]
    # layout: word (r, n) at qw[r, n] -- a 3-column matrix with distinct rows
    codes = np.array([[c] * 16 for c in (1, 2, 3)], dtype=np.uint8)
    qw = oracle.w4a16_pack(codes).view(np.uint32)
    assert qw.shape == (2, 3)
    assert qw[0].tolist() == [0x11111111, 0x22222222, 0x33333333]


def _prepared_golden():
    """(total words, [(record, index, word)]) from tests/golden/w4a16_prepared_words.txt."""
    total, words = None, []
    with open(os.path.join(GOLDEN, "w4a16_prepared_words.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "words_total":
                total = int(vals[0])
            elif key == "word":
                words.append((int(vals[0]), int(vals[1]), int(vals[2], 16)))
    return total, words


def pin_prepared_layout_golden_words():
    """The prepared layout against hand-worked words (tests/golden/w4a16_prepared_words.txt):
    nibble interleave, word order within a record, record order, the fused scale|minimum
    words and the zero padding of a partial tile."""
    N, K = 8, 256
    codes = np.empty((N, K), dtype=np.uint8)
    for n in range(N):
        for k in range(K):
            codes[n, k] = (n + k + k // 8) % 16
    qw = oracle.w4a16_pack(codes)
    g_idx = np.arange(K // 128).reshape(-1, 1)
    n_idx = np.arange(N).reshape(1, -1)
    s = (0x3C00 + n_idx + 16 * g_idx).astype(np.uint16)
    m = (0xBC00 + n_idx + 16 * g_idx).astype(np.uint16)
    prep = oracle.w4a16_prepare(qw, s, m)
    total, words = _prepared_golden()
    assert prep.size == total
    for rec, idx, want in words:
        got = int(prep[rec * 2176 + idx])
        assert got == want, (rec, idx, hex(got), hex(want))


def pin_prepared_layout_keeps_4_25_bits_and_every_weight():
    """The prepared copy is 4.25 bits per weight ("Low-Precision Kernels ...", Step 2) when N
    fills whole tiles, and it holds every code, scale and minimum exactly once: decoding
    each weight from it gives the canonical layout's w_hat bit for bit (ragged N too)."""
    for N, K in ((256, 256), (136, 384)):
        w = workloads.weights(N, K, seed=N + K).numpy()
        codes, s, m = oracle.w4a16_quantize(w)
        qw = oracle.w4a16_pack(codes)
        prep = oracle.w4a16_prepare(qw, s, m)
        if N % 128 == 0:
            assert prep.nbytes * 8 / (N * K) == 4.25
        rec = prep.reshape(-1, K // 128, 2176)            # [tile][group][word]
        cw = rec[:, :, :2048].reshape(-1, K // 128, 2, 2, 128, 4)  # [t][g][b][h][n][j]
        got = np.empty((N, K), dtype=np.int64)
        for t in range(rec.shape[0]):
            for n in range(128):
                col = 128 * t + n
                if col >= N:
                    assert not cw[t, :, :, :, n, :].any() and not rec[t, :, 2048 + n].any()
                    continue
                for g in range(K // 128):
                    for b in range(2):
                        for h in range(2):
                            for j in range(4):
                                word = int(cw[t, g, b, h, n, j])
                                k0 = 128 * g + 64 * b + 8 * (4 * h + j)
                                for i in range(4):
                                    got[col, k0 + 2 * i] = (word >> (4 * i)) & 15
                                    got[col, k0 + 2 * i + 1] = (word >> (16 + 4 * i)) & 15
        assert np.array_equal(got, codes.astype(np.int64))
        sm = rec[:, :, 2048:].transpose(1, 0, 2).reshape(K // 128, -1)[:, :N]
        assert np.array_equal((sm & 0xFFFF).astype(np.uint16), s)
        assert np.array_equal((sm >> 16).astype(np.uint16), m)


def pin_sizes_printed_on_pages():
    """4.25 bits/weight, 3.76x, 31.2 MB, the 4 KB vs 16 KB tile, 18-byte Q4 blocks,
    3.56x and 144 MiB, all computed from the array sizes the oracle produces."""
    p = _page_sizes()
    N, K, G = 64, 256, 128
    codes, s, m = oracle.w4a16_quantize(workloads.weights(N, K, seed=1).numpy(), group=G)
    qw = oracle.w4a16_pack(codes)
    bits = 8.0 * (qw.nbytes + s.nbytes + m.nbytes) / (N * K)
    assert bits == p["w4a16_bits_per_weight"]
    assert round(16.0 / bits, 2) == p["w4a16_speedup_cap"]
    # the Llama up-projection: bytes per weight from the small case, scaled
    n_w = int(p["w4a16_llama_up_N"] * p["w4a16_llama_up_K"])
    total = n_w * (qw.nbytes + s.nbytes + m.nbytes) // (N * K)
    assert total == 31_195_136 and round(total / 1e6, 1) == p["w4a16_llama_up_mb"]
    # a 128 (K) x 64 (N) tile of packed words vs BF16
    tk, tn = int(p["w4a16_tile_K"]), int(p["w4a16_tile_N"])
    tile_q = oracle.w4a16_pack(np.zeros((tn, tk), dtype=np.uint8))
    assert tile_q.nbytes == p["w4a16_tile_packed_bytes"]
    assert tk * tn * 2 == p["w4a16_tile_bf16_bytes"]
    # Q4: 16 code bytes + 2 scale bytes per 32 weights
    qc, qs = oracle.q4b32_quantize(workloads.weights(4, 64, seed=2).numpy())
    per_block = (qc.nbytes + qs.nbytes) / (4 * 64 / 32)
    assert per_block == p["q4_block_bytes"]
    assert round(p["q4_block_fp16_bytes"] / per_block, 2) == p["q4_ratio"]
    n2 = int(p["q4_square_N"]) ** 2
    assert n2 // 32 * per_block == p["q4_square_mib"] * 2**20


def pin_round_trip_on_grid():
    """Weights already on the 16-level grid (q*s + min exact, q = 0 and 15 present
    in every group) quantize back to exactly (q, s, min) and rebuild bit for bit."""
    rng = np.random.default_rng(7)
    N, K, G = 24, 256, 32
    groups = K // G
    s_b = oracle.bf16_rne(2.0 ** rng.uniform(-10, -5, size=(groups, N)))
    m_b = oracle.bf16_rne(rng.uniform(-0.5, 0.0, size=(groups, N)))
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::G] = 0
    q[:, 1::G] = 15
    w = np.empty((N, K), dtype=np.float64)
    for n in range(N):
        for k in range(K):
            w[n, k] = q[n, k] * _bf16(s_b[k // G, n]) + _bf16(m_b[k // G, n])
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w), "grid values must be exact in fp32"
    codes, s2, m2 = oracle.w4a16_quantize(w32, group=G)
    np.testing.assert_array_equal(s2, s_b)
    np.testing.assert_array_equal(m2, m_b)
    np.testing.assert_array_equal(codes, q.astype(np.uint8))
    w_hat = oracle.w4a16_dequant(oracle.w4a16_pack(codes), s2, m2, group=G)
    np.testing.assert_array_equal(w_hat, w)


def pin_quantize_nearest_grid_point():
    """For random groups, every code is a nearest grid point to w in exact arithmetic
    (ties to the even code), unless the clamp applies or the exact quotient lies within
    fp32 rounding of a tie; and the stored scale is the BF16 rounding of (max-min)/15."""
    w = workloads.weights(16, 256, seed=11).numpy()
    G = 64
    codes, s, m = oracle.w4a16_quantize(w, group=G)
    for n in range(w.shape[0]):
        for g in range(w.shape[1] // G):
            grp = w[n, g * G:(g + 1) * G]
            sf, mf = Fraction(_bf16(s[g, n])), Fraction(_bf16(m[g, n]))
            exact_s = (Fraction(float(grp.max())) - Fraction(float(grp.min()))) / 15
            assert abs(sf - exact_s) <= exact_s / 2**8, "scale must be bf16(range/15)"
            assert abs(mf - Fraction(float(grp.min()))) <= abs(Fraction(float(grp.min()))) / 2**8
            for i, wv in enumerate(grp):
                t = (Fraction(float(wv)) - mf) / sf
                q = int(codes[n, g * G + i])
                best = min(range(16), key=lambda c: (abs(t - c), c % 2))
                if q != best:
                    near_tie = abs(abs(t - math.floor(t)) - Fraction(1, 2)) < Fraction(1, 2**18)
                    assert near_tie, (n, g, i, float(t), q, best)


def pin_one_hot_activation():
    """x = e_k gives y[n] = w_hat[n, k] = q*s + min exactly: pins nibble order, the
    [K/8, N] layout and the group index of the scale/min."""
    N, K, G = 40, 384, 128
    codes, s, m = oracle.w4a16_quantize(workloads.weights(N, K, seed=3).numpy(), group=G)
    qw = oracle.w4a16_pack(codes)
    one = _torch_bits(torch.tensor([1.0], dtype=torch.bfloat16))[0]
    for k in (0, 1, 7, 8, 127, 128, 200, 383):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = one
        y, a = oracle.w4a16_matmul(x, qw, s, m, group=G)
        for n in range(N):
            want = int(codes[n, k]) * _bf16(s[k // G, n]) + _bf16(m[k // G, n])
            assert y[0, n] == want and a[0, n] == abs(want), (k, n)


def pin_constant_codes():
    """All codes equal c in a group: y = sum_g (c*s_g + min_g) * sum_{k in g} x_k, summed
    exactly with rationals."""
    N, K, G = 6, 256, 128
    rng = np.random.default_rng(5)
    for c in (0, 9, 15):
        codes = np.full((N, K), c, dtype=np.uint8)
        s = oracle.bf16_rne(rng.uniform(0.001, 0.01, size=(K // G, N)))
        mn = oracle.bf16_rne(rng.uniform(-0.05, 0.0, size=(K // G, N)))
        x = workloads.bits16(workloads.activations_bf16(2, K, seed=c))
        y, _ = oracle.w4a16_matmul(x, oracle.w4a16_pack(codes), s, mn, group=G)
        for r in range(2):
            for n in range(N):
                tot = Fraction(0)
                for g in range(K // G):
                    sx = sum(Fraction(_bf16(v)) for v in x[r, g * G:(g + 1) * G])
                    tot += (c * Fraction(_bf16(s[g, n])) + Fraction(_bf16(mn[g, n]))) * sx
                assert abs(Fraction(y[r, n]) - tot) <= Fraction(1, 2**40), (c, r, n)


def pin_brute_force_small():
    """N, K <= 64, groups 8..64: y from the packed path equals the exact rational triple
    loop over the unpacked codes to fp64 rounding."""
    rng = np.random.default_rng(9)
    for (M, N, K, G) in ((1, 8, 64, 8), (3, 17, 64, 16), (2, 64, 64, 32), (4, 33, 64, 64),
                         (1, 64, 32, 32)):
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        codes, s, mn = oracle.w4a16_quantize(w, group=G)
        x = workloads.bits16(workloads.activations_bf16(M, K, seed=N + K))
        y, a = oracle.w4a16_matmul(x, oracle.w4a16_pack(codes), s, mn, group=G)
        for r in range(M):
            for n in range(N):
                exact = sum(Fraction(_bf16(x[r, k])) *
                            (int(codes[n, k]) * Fraction(_bf16(s[k // G, n])) +
                             Fraction(_bf16(mn[k // G, n]))) for k in range(K))
                assert abs(Fraction(y[r, n]) - exact) <= Fraction(a[r, n]) * Fraction(1, 2**45), \
                    (M, N, K, G, r, n)


def pin_matches_library_matmul():
    """The fp64 sum equals torch.matmul (fp64) on the rebuilt weights to ~1e-12."""
    N, K, G, M = 96, 512, 128, 3
    codes, s, mn = oracle.w4a16_quantize(workloads.weights(N, K, seed=4).numpy(), group=G)
    qw = oracle.w4a16_pack(codes)
    x = workloads.bits16(workloads.activations_bf16(M, K, seed=4))
    y, a = oracle.w4a16_matmul(x, qw, s, mn, group=G)
    sv = torch.from_numpy(s.view(np.int16).copy()).view(torch.bfloat16).double()
    mv = torch.from_numpy(mn.view(np.int16).copy()).view(torch.bfloat16).double()
    w_hat = (torch.from_numpy(codes.astype(np.float64)) * sv.repeat_interleave(G, 0).T
             + mv.repeat_interleave(G, 0).T)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
    ref = (xv @ w_hat.T).numpy()
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    # sampled-column entry point agrees with the full one
    cols = np.array([0, 5, 95, 17], dtype=np.int32)
    y2, a2 = oracle.w4a16_matmul(x, qw, s, mn, group=G, cols=cols)
    np.testing.assert_array_equal(y2, y[:, cols])
    np.testing.assert_array_equal(a2, a[:, cols])


def pin_quantization_error_band():
    """Rounding N(0, 0.02^2) weights to 16 levels per group of 128 gives ~10 % output
    error against the original weights (the pages report 10 %); accept 6-14 %."""
    N, K, G = 256, 2048, 128
    w = workloads.weights(N, K, seed=0).numpy()
    codes, s, mn = oracle.w4a16_quantize(w, group=G)
    w_hat = oracle.w4a16_dequant(oracle.w4a16_pack(codes), s, mn, group=G)
    x = workloads.activations_bf16(4, K, seed=0).double().numpy()
    y_q = x @ w_hat.T
    y_o = x @ w.astype(np.float64).T
    rel = np.linalg.norm(y_q - y_o) / np.linalg.norm(y_o)
    assert 0.06 < rel < 0.14, rel
    # every rebuilt weight lies within half a step of the original (no clamp at this scale)
    step = np.repeat(torch.from_numpy(s.view(np.int16).copy()).view(torch.bfloat16).double()
                     .numpy(), G, axis=0).T
    assert np.all(np.abs(w_hat - w) <= 0.5 * step * (1 + 2**-7) + 2**-9 * np.abs(w))


def pin_q4_hand_worked_blocks():
    """Hand-worked Q4 blocks (tests/golden/q4b32_blocks.txt)."""
    recs = _records("q4b32_blocks.txt")
    w = np.stack([_weights_from(r) for _, r in recs])
    codes, scales = oracle.q4b32_quantize(w)
    for i, (tag, rec) in enumerate(recs):
        assert int(scales[i, 0]) == int(rec["scale"][0], 16), tag
        assert codes[i].tolist() == [int(v, 16) for v in rec["bytes"]], (tag, codes[i].tolist())


def pin_q4_round_trip_and_gemv():
    """On-grid Q4 blocks round-trip; the GEMV equals the exact rational sum, and a
    one-hot x picks (q - 8) * s."""
    rng = np.random.default_rng(21)
    N, K = 12, 128
    q = rng.integers(1, 16, size=(N, K))
    q[:, ::32] = 0              # -8 * s sets max|w| = 8 s
    s_h = oracle.fp16_rne(2.0 ** rng.uniform(-12, -6, size=(N, K // 32)))
    w = np.empty((N, K), dtype=np.float64)
    for n in range(N):
        for k in range(K):
            w[n, k] = (q[n, k] - 8) * _fp16(s_h[n, k // 32])
    codes, s2 = oracle.q4b32_quantize(w.astype(np.float32))
    np.testing.assert_array_equal(s2, s_h)
    np.testing.assert_array_equal(oracle.q4b32_dequant(codes, s2), w)
    x = workloads.bits16(workloads.activations_fp16(K, seed=3))
    y, a = oracle.q4b32_gemv(x, codes, s2)
    for n in range(N):
        exact = sum((q[n, k] - 8) * Fraction(_fp16(s_h[n, k // 32])) * Fraction(_fp16(x[k]))
                    for k in range(K))
        assert abs(Fraction(y[n]) - exact) <= Fraction(a[n]) * Fraction(1, 2**45)
    one = _torch_bits(torch.tensor([1.0], dtype=torch.float16))[0]
    for k in (0, 1, 31, 32, 127):
        xo = np.zeros(K, dtype=np.uint16)
        xo[k] = one
        y, _ = oracle.q4b32_gemv(xo, codes, s2)
        assert np.array_equal(y, w[:, k]), k
    rows = np.array([3, 0, 11], dtype=np.int32)
    y_full, _ = oracle.q4b32_gemv(x, codes, s2)
    y_rows, _ = oracle.q4b32_gemv(x, codes, s2, rows=rows)
    np.testing.assert_array_equal(y_rows, y_full[rows])


# --------------------------------------------------------------------------- #
# zero-point format: w_hat = (q - z) s, fp16 s and z, words [N, K/8]
# --------------------------------------------------------------------------- #

def _zp_codes(qw_rows):
    """Codes [N, K] from words [N, K/8] (k = 8r + j in bits 4j..4j+3), with numpy."""
    w = np.asarray(qw_rows, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    return ((w[:, :, None] >> shifts) & 0xF).reshape(w.shape[0], -1).astype(np.int64)


def _fp16_array(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy()) \
        .view(torch.float16).double().numpy()


def _zp_w_hat(qw_rows, s, z, G):
    """(q - z) s in fp64 from numpy unpacking and PyTorch's fp16 conversion."""
    q = _zp_codes(qw_rows)
    sv = np.repeat(_fp16_array(s), G, axis=1)
    zv = np.repeat(_fp16_array(z), G, axis=1)
    return (q - zv) * sv


def pin_zp_hand_worked_groups():
    """Hand-worked zero-point groups (tests/golden/w4a16zp_groups.txt): scale, zero,
    codes and the packed word."""
    for tag, rec in _records("w4a16zp_groups.txt"):
        w = _weights_from(rec).reshape(1, -1)
        qw_rows, scales, zeros = oracle.w4a16zp_quantize(w, group=w.shape[1])
        assert int(scales[0, 0]) == int(rec["scale"][0], 16), (tag, hex(scales[0, 0]))
        assert int(zeros[0, 0]) == int(rec["zero"][0], 16), (tag, hex(zeros[0, 0]))
        assert int(qw_rows[0, 0]) == int(rec["word"][0], 16), (tag, hex(qw_rows[0, 0]))
        assert _zp_codes(qw_rows)[0].tolist() == [int(v) for v in rec["q"]], tag


def pin_zp_round_trip_on_grid():
    """Weights (q - z) s with fp16 s, integer z in 0..15 and q = 0 and 15 in every group
    quantize back to exactly (q, s, z) and rebuild bit for bit."""
    rng = np.random.default_rng(17)
    N, K, G = 20, 256, 64
    groups = K // G
    s_h = oracle.fp16_rne(2.0 ** rng.uniform(-10, -4, size=(N, groups)))
    z = rng.integers(0, 16, size=(N, groups))
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::G] = 0
    q[:, 3::G] = 15
    sv = np.repeat(_fp16_array(s_h), G, axis=1)
    w = (q - np.repeat(z, G, axis=1)) * sv
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w), "grid values must be exact in fp32"
    qw_rows, s2, z2 = oracle.w4a16zp_quantize(w32, group=G)
    np.testing.assert_array_equal(s2, s_h)
    np.testing.assert_array_equal(_fp16_array(z2), z.astype(np.float64))
    np.testing.assert_array_equal(_zp_codes(qw_rows), q)
    np.testing.assert_array_equal(oracle.w4a16zp_dequant(qw_rows, s2, z2, group=G), w)


def pin_zp_codes_follow_the_formula():
    """On random groups, every scale, zero and code equals the formula evaluated with
    exact rationals (a rounding of the exact quotient: the fp32 quotient can only move a
    result that lies within 2^-20 of a half-integer, and such cases are skipped)."""
    w = workloads.weights(12, 512, seed=21).numpy()
    w[3, :128] += 0.5  # one group entirely positive: negative zero point
    G = 128
    qw_rows, s, z = oracle.w4a16zp_quantize(w, group=G)
    codes = _zp_codes(qw_rows)

    def rha(t):  # half away from zero
        a = math.floor(abs(t) + Fraction(1, 2))
        return a if t >= 0 else -a

    for n in range(w.shape[0]):
        for g in range(w.shape[1] // G):
            grp = w[n, g * G:(g + 1) * G]
            lo, hi = Fraction(float(grp.min())), Fraction(float(grp.max()))
            sf = Fraction(_fp16(s[n, g]))
            assert abs(sf - (hi - lo) / 15) <= (hi - lo) / 15 / 2**10 + Fraction(1, 2**30)
            zt = -lo / sf
            if abs(abs(zt - math.floor(zt)) - Fraction(1, 2)) > Fraction(1, 2**20):
                assert Fraction(_fp16(z[n, g])) == rha(zt), (n, g)
            zf = Fraction(_fp16(z[n, g]))
            for i, wv in enumerate(grp):
                t = Fraction(float(wv)) / sf
                if abs(abs(t - math.floor(t)) - Fraction(1, 2)) <= Fraction(1, 2**20):
                    continue
                want = min(15, max(0, rha(t) + zf))
                assert codes[n, g * G + i] == want, (n, g, i, float(t))


def pin_zp_one_hot_activation():
    """x = e_k gives y[n] = (q - z) s exactly: pins the [N, K/8] word layout, nibble
    order, the [N, K/G] scale/zero layout and the sign of the zero point."""
    N, K, G = 24, 384, 128
    w = workloads.weights(N, K, seed=5).numpy()
    qw_rows, s, z = oracle.w4a16zp_quantize(w, group=G)
    w_hat = _zp_w_hat(qw_rows, s, z, G)
    one = _torch_bits(torch.tensor([1.0], dtype=torch.bfloat16))[0]
    for k in (0, 1, 7, 8, 127, 128, 255, 383):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = one
        y, a = oracle.w4a16zp_matmul(x, qw_rows, s, z, group=G)
        np.testing.assert_array_equal(y[0], w_hat[:, k])
        np.testing.assert_array_equal(a[0], np.abs(w_hat[:, k]))


def pin_zp_matmul_exact_small():
    """Small cases: the fp64 sum equals the exact rational sum over (q - z) s to fp64
    rounding, and the sampled-column entry point matches the full one."""
    rng = np.random.default_rng(23)
    for (M, N, K, G) in ((1, 8, 64, 8), (3, 9, 64, 32), (2, 16, 128, 64)):
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        qw_rows, s, z = oracle.w4a16zp_quantize(w, group=G)
        q = _zp_codes(qw_rows)
        x = workloads.bits16(workloads.activations_bf16(M, K, seed=N + K))
        y, a = oracle.w4a16zp_matmul(x, qw_rows, s, z, group=G)
        for r in range(M):
            for n in range(N):
                exact = sum(Fraction(_bf16(x[r, k])) *
                            (int(q[n, k]) - Fraction(_fp16(z[n, k // G]))) *
                            Fraction(_fp16(s[n, k // G])) for k in range(K))
                assert abs(Fraction(y[r, n]) - exact) <= Fraction(a[r, n]) / 2**45, (M, N, r, n)
        cols = np.array([N - 1, 0, 3], dtype=np.int32)
        y2, a2 = oracle.w4a16zp_matmul(x, qw_rows, s, z, group=G, cols=cols)
        np.testing.assert_array_equal(y2, y[:, cols])
        np.testing.assert_array_equal(a2, a[:, cols])


def pin_zp_matches_library_matmul_and_error_band():
    """torch.matmul (fp64) on independently rebuilt weights agrees to ~1e-12, and the
    zero-point format's error on N(0, 0.02^2) weights is the same ~10 % band as the
    minimum form (16 levels over the group's range); the kernel layout is a transpose."""
    N, K, G, M = 128, 1024, 128, 4
    w = workloads.weights(N, K, seed=8).numpy()
    qw_rows, s, z = oracle.w4a16zp_quantize(w, group=G)
    w_hat = _zp_w_hat(qw_rows, s, z, G)
    np.testing.assert_array_equal(oracle.w4a16zp_dequant(qw_rows, s, z, group=G), w_hat)
    x = workloads.bits16(workloads.activations_bf16(M, K, seed=8))
    y, a = oracle.w4a16zp_matmul(x, qw_rows, s, z, group=G)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
    ref = (xv @ torch.from_numpy(w_hat).T).numpy()
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    y_o = xv.numpy() @ w.astype(np.float64).T
    rel = np.linalg.norm(y - y_o) / np.linalg.norm(y_o)
    assert 0.06 < rel < 0.14, rel
    qk, sk, zk = oracle.w4a16zp_kernel_layout(qw_rows, s, z)
    assert qk.shape == (K // 8, N) and sk.shape == (K // G, N) and zk.shape == (K // G, N)
    assert int(qk[5, 7]) & 0xFFFFFFFF == int(qw_rows[7, 5]) and sk[2, 9] == s[9, 2]
    assert zk[3, 1] == z[1, 3]


# --------------------------------------------------------------------------- #
# W8A16: symmetric per-row INT8, w_hat = q s
# --------------------------------------------------------------------------- #

def _half_away(t):
    a = math.floor(abs(t) + Fraction(1, 2))
    return a if t >= 0 else -a


def pin_w8_hand_worked_rows():
    """Hand-worked rows (tests/golden/w8a16_rows.txt): the fp32 scale and every code."""
    for tag, rec in _records("w8a16_rows.txt"):
        w = _weights_from(rec).reshape(1, -1)
        q, s = oracle.w8a16_quantize(w)
        assert int(s.view(np.uint32)[0]) == int(rec["scale"][0], 16), (tag, s[0])
        assert q[0].tolist() == [int(v) for v in rec["q"]], (tag, q[0].tolist())


def pin_w8_round_trip_on_grid():
    """Rows q s with s a power of two and |q| = 127 present quantize back to exactly
    (q, s) and rebuild bit for bit."""
    rng = np.random.default_rng(31)
    N, K = 16, 256
    e = rng.integers(-14, -4, size=N)
    q = rng.integers(-127, 128, size=(N, K))
    q[:, 0] = np.where(rng.random(N) < 0.5, 127, -127)
    w = q * np.exp2(e)[:, None]
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w)
    q2, s2 = oracle.w8a16_quantize(w32)
    np.testing.assert_array_equal(q2, q.astype(np.int8))
    np.testing.assert_array_equal(s2.astype(np.float64), np.exp2(e))
    one = _torch_bits(torch.tensor([1.0], dtype=torch.bfloat16))[0]
    for k in (0, 5, 255):
        x = np.zeros(K, dtype=np.uint16)
        x[k] = one
        y, a = oracle.w8a16_gemv(x, q2, s2)
        np.testing.assert_array_equal(y, w[:, k])
        np.testing.assert_array_equal(a, np.abs(w[:, k]))


def pin_w8_codes_follow_the_formula():
    """On random rows the scale is max|w| / 127 to fp32 rounding and each code is the
    exact quotient rounded half away from zero (quotients within 2^-16 of a half-integer,
    where the fp32 quotient may decide otherwise, are skipped)."""
    w = workloads.weights(6, 512, seed=33).numpy()
    q, s = oracle.w8a16_quantize(w)
    for n in range(w.shape[0]):
        amax = Fraction(float(np.abs(w[n]).max()))
        sf = Fraction(float(s[n]))
        assert abs(sf - amax / 127) <= amax / 127 / 2**23
        for k in range(w.shape[1]):
            t = Fraction(float(w[n, k])) / sf
            if abs(abs(t - math.floor(t)) - Fraction(1, 2)) <= Fraction(1, 2**16):
                continue
            assert int(q[n, k]) == max(-127, min(127, _half_away(t))), (n, k, float(t))


def pin_w8_gemv_exact_small_and_library():
    """Small cases equal the exact rational sum; a larger one equals torch.matmul (fp64)
    on the rebuilt weights; the row subset entry point matches; INT8 per-row quantization
    of N(0, 0.02^2) weights gives an output error near 1 % (0.3-2 % accepted)."""
    rng = np.random.default_rng(35)
    for (N, K) in ((3, 64), (9, 96)):
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        q, s = oracle.w8a16_quantize(w)
        x = workloads.bits16(workloads.activations_bf16(1, K, seed=N))[0]
        y, a = oracle.w8a16_gemv(x, q, s)
        for n in range(N):
            exact = sum(Fraction(_bf16(x[k])) * int(q[n, k]) * Fraction(float(s[n]))
                        for k in range(K))
            assert abs(Fraction(y[n]) - exact) <= Fraction(a[n]) / 2**45, (N, K, n)
    N, K = 128, 2048
    w = workloads.weights(N, K, seed=36).numpy()
    q, s = oracle.w8a16_quantize(w)
    x = workloads.bits16(workloads.activations_bf16(1, K, seed=36))[0]
    y, a = oracle.w8a16_gemv(x, q, s)
    w_hat = torch.from_numpy(q.astype(np.float64)) * torch.from_numpy(s.astype(np.float64))[:, None]
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
    ref = (w_hat @ xv).numpy()
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    rows = np.array([N - 1, 0, 17], dtype=np.int32)
    y2, a2 = oracle.w8a16_gemv(x, q, s, rows=rows)
    np.testing.assert_array_equal(y2, y[rows])
    np.testing.assert_array_equal(a2, a[rows])
    y_o = w.astype(np.float64) @ xv.numpy()
    rel = np.linalg.norm(y - y_o) / np.linalg.norm(y_o)
    assert 0.003 < rel < 0.02, rel


# --------------------------------------------------------------------------- #
# NVFP4 weights: E2M1 codes, E4M3 block scales of 16, one fp32 scale per tensor
# --------------------------------------------------------------------------- #

def _nv_codes(codes):
    """Codes [N, K] from bytes [N, K/2] (low nibble = even k), with numpy."""
    c = np.asarray(codes, dtype=np.uint8)
    return np.stack([c & 15, c >> 4], axis=-1).reshape(c.shape[0], -1).astype(np.int64)


def _e4m3_table():
    """Values of the 256 E4M3 codes from PyTorch's float8_e4m3fn (a library routine)."""
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    return t.float().double().numpy()


def _nv_w_hat(codes, scales, S):
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    e4 = _e4m3_table()
    return e2[_nv_codes(codes)] * np.repeat(e4[np.asarray(scales)], 16, axis=1) * S


def pin_nvfp4_element_formats():
    """E4M3 values of every code against PyTorch's float8_e4m3fn; E2M1 magnitudes are the
    page's doubled grid (0, 1, 2, 3, 4, 6, 8, 12) halved, the largest 6; rounding to E2M1
    picks a nearest value (ties: the even code) and saturates; the E4M3 ceiling is the
    smallest code not below its argument."""
    e4 = _e4m3_table()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if np.isnan(e4[c]):
            assert np.isnan(v), c
        else:
            assert v == e4[c], (c, v, e4[c])
    assert [2 * oracle.e2m1_value(c) for c in range(8)] == [0, 1, 2, 3, 4, 6, 8, 12]
    assert [oracle.e2m1_value(c + 8) for c in range(8)] == [-oracle.e2m1_value(c) for c in range(8)]
    grid = [Fraction(int(2 * oracle.e2m1_value(c)), 2) for c in range(8)]
    rng = np.random.default_rng(41)
    ts = list(rng.uniform(-7, 7, size=2000).astype(np.float32)) + \
        [np.float32(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, 6.0, 100.0, -0.1)]
    for t in ts:
        code = oracle.e2m1_rne(float(t))
        a = abs(Fraction(float(t)))
        if a >= 6:
            assert code & 7 == 7
        else:
            d = [abs(a - g) for g in grid]
            best = min(range(8), key=lambda i: (d[i], i & 1))
            assert code & 7 == best, (float(t), code)
        assert (code >> 3) == (1 if np.signbit(t) else 0)
    finite = sorted(set(float(v) for v in e4[:0x7F]))
    for v in list(rng.uniform(0, 500, size=500)) + list(2.0 ** rng.uniform(-12, 9, size=500)):
        v32 = float(np.float32(v))
        c = oracle.e4m3_ceil(v32)
        if v32 > 448:
            assert c == 0x7E
            continue
        assert e4[c] >= v32 and all(f < v32 for f in finite if f < e4[c]), (v32, c)


def pin_nvfp4_hand_worked_tensors():
    """Hand-worked tensors (tests/golden/nvfp4_blocks.txt): tensor scale, block scales,
    code bytes."""
    for tag, rec in _records("nvfp4_blocks.txt"):
        w = _weights_from(rec).reshape(1, -1)
        codes, scales, S = oracle.nvfp4_quantize(w)
        assert int(np.float32(S).view(np.uint32)) == int(rec["S"][0], 16), tag
        assert [int(v) for v in scales[0]] == [int(v, 16) for v in rec["scales"]], tag
        assert [int(v) for v in codes[0]] == [int(v, 16) for v in rec["bytes"]], tag


def pin_nvfp4_round_trip_and_bits():
    """Weights on the grid (tensor scale 1, each block's largest |w| six times an E4M3 scale,
    every weight an E2M1 value times it) quantize back to exactly those codes and scales
    and rebuild exactly; the format costs 4.5 bits per weight plus one fp32 per tensor."""
    rng = np.random.default_rng(43)
    N, K = 12, 256
    e4 = _e4m3_table()
    sc = rng.integers(0x08, 0x70, size=(N, K // 16))
    sc[0, 0] = 0x7E  # 6 * 448 = 2688 makes S = 1
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::16] = 7  # the block maximum, +6
    w = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])[q] * \
        np.repeat(e4[sc], 16, axis=1)
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w)
    codes, scales, S = oracle.nvfp4_quantize(w32)
    assert S == 1.0
    np.testing.assert_array_equal(scales, sc.astype(np.uint8))
    np.testing.assert_array_equal(_nv_codes(codes), q)  # -0 (code 8) included
    np.testing.assert_array_equal(oracle.nvfp4_dequant(codes, scales, S), w)
    bits = (codes.nbytes + scales.nbytes) * 8 / (N * K)
    assert bits == 4.5


def pin_nvfp4_gemv_exact_and_error():
    """Small GEMVs equal the exact rational sum; a larger one equals torch.matmul (fp64) on
    weights rebuilt with PyTorch's E4M3; the row subset entry point matches; on weights with
    0.1 % outliers NVFP4's weight error is below INT4's with groups of 128 (the pages: 9.4 %
    against 12.8 % on a real layer)."""
    rng = np.random.default_rng(45)
    for (N, K) in ((2, 32), (5, 64)):
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        codes, scales, S = oracle.nvfp4_quantize(w)
        x = workloads.bits16(workloads.activations_bf16(1, K, seed=N))[0]
        y, a = oracle.nvfp4_gemv(x, codes, scales, S)
        qn = _nv_codes(codes)
        for n in range(N):
            exact = sum(Fraction(_bf16(x[k])) * Fraction(oracle.e2m1_value(int(qn[n, k]))) *
                        Fraction(oracle.e4m3_value(int(scales[n, k // 16]))) * Fraction(S)
                        for k in range(K))
            assert abs(Fraction(y[n]) - exact) <= Fraction(a[n]) / 2**45, (N, K, n)
    N, K = 64, 1024
    w = workloads.weights(N, K, seed=46, outlier_frac=0.001).numpy()
    codes, scales, S = oracle.nvfp4_quantize(w)
    w_hat = _nv_w_hat(codes, scales, S)
    np.testing.assert_array_equal(oracle.nvfp4_dequant(codes, scales, S), w_hat)
    x = workloads.bits16(workloads.activations_bf16(1, K, seed=46))[0]
    y, a = oracle.nvfp4_gemv(x, codes, scales, S)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
    ref = (torch.from_numpy(w_hat) @ xv).numpy()
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    rows = np.array([N - 1, 3], dtype=np.int32)
    y2, _ = oracle.nvfp4_gemv(x, codes, scales, S, rows=rows)
    np.testing.assert_array_equal(y2, y[rows])
    w = workloads.weights(256, 2048, seed=0, outlier_frac=0.001).numpy()
    c, sc, S = oracle.nvfp4_quantize(w)
    e_nv = np.linalg.norm(oracle.nvfp4_dequant(c, sc, S) - w) / np.linalg.norm(w)
    cq, sq, mq = oracle.w4a16_quantize(w)
    e_i4 = np.linalg.norm(oracle.w4a16_dequant(oracle.w4a16_pack(cq), sq, mq) - w) / np.linalg.norm(w)
    assert 0.07 < e_nv < e_i4 < 0.15, (e_nv, e_i4)


# --------------------------------------------------------------------------- #
# MXFP4 weights: E2M1 codes, one E8M0 (power-of-two) scale per 32
# --------------------------------------------------------------------------- #

def pin_mxfp4_hand_worked_blocks_and_scale_format():
    """Hand-worked blocks (tests/golden/mxfp4_blocks.txt); E8M0 values against PyTorch's
    float8_e8m0fnu; 4.25 bits per value (the page's figure) from the array sizes."""
    for tag, rec in _records("mxfp4_blocks.txt"):
        w = _weights_from(rec).reshape(1, -1)
        codes, scales = oracle.mxfp4_quantize(w)
        assert int(scales[0, 0]) == int(rec["scale"][0], 16), (tag, hex(scales[0, 0]))
        assert [int(v) for v in codes[0]] == [int(v, 16) for v in rec["bytes"]], tag
    if hasattr(torch, "float8_e8m0fnu"):
        t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu)
        ref = t.float().double().numpy()
        for c in range(255):
            assert oracle.e8m0_value(c) == ref[c], c
    else:  # the format's definition: a biased exponent
        for c in range(255):
            assert oracle.e8m0_value(c) == 2.0 ** (c - 127), c
    assert np.isnan(oracle.e8m0_value(255))
    codes, scales = oracle.mxfp4_quantize(np.ones((3, 64), dtype=np.float32))
    assert (codes.nbytes + scales.nbytes) * 8 / (3 * 64) == 4.25


def pin_mxfp4_scale_rule_and_round_trip():
    """On random blocks the scale is 2^(floor(log2 max|w|) - 2) and every code is a nearest
    E2M1 value of w / scale (ties to the even code, clamped at 6); weights on the grid (a
    block maximum of 4 or 6 times a power of two) come back exactly."""
    rng = np.random.default_rng(51)
    w = (rng.standard_normal((8, 256)) * 10.0 ** rng.uniform(-4, 2, size=(8, 1))).astype(np.float32)
    codes, scales = oracle.mxfp4_quantize(w)
    grid = [Fraction(int(2 * oracle.e2m1_value(c)), 2) for c in range(8)]
    qn = _nv_codes(codes)
    for n in range(8):
        for b in range(8):
            blk = w[n, 32 * b:32 * (b + 1)]
            amax = Fraction(float(np.abs(blk).max()))
            X = int(scales[n, b]) - 127
            assert 2 ** (X + 2) <= amax < 2 ** (X + 3), (n, b, X, float(amax))
            for j, wv in enumerate(blk):
                t = abs(Fraction(float(wv)) / Fraction(2) ** X)
                c = int(qn[n, 32 * b + j]) & 7
                if t >= 6:
                    assert c == 7
                else:
                    d = [abs(t - g) for g in grid]
                    assert c == min(range(8), key=lambda i: (d[i], i & 1)), (n, b, j, float(t))
    X = rng.integers(-20, 10, size=(4, 4))
    q = rng.integers(0, 16, size=(4, 128))
    q[:, ::32] = 7  # +6: the block maximum
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    w = (e2[q] * np.repeat(np.exp2(X), 32, axis=1)).astype(np.float32)
    codes, scales = oracle.mxfp4_quantize(w)
    np.testing.assert_array_equal(scales.astype(int) - 127, X)
    np.testing.assert_array_equal(_nv_codes(codes), q)
    np.testing.assert_array_equal(oracle.mxfp4_dequant(codes, scales), w.astype(np.float64))


def pin_mxfp4_gemv_exact_and_error():
    """Small GEMVs equal the exact rational sum; torch.matmul (fp64) agrees on a larger one;
    the row subset matches; on weights with 0.1 % outliers MXFP4's weight error lies above
    NVFP4's (the pages: 11.8 % against 9.4 % on a real layer) and within 8-16 %."""
    rng = np.random.default_rng(53)
    for (N, K) in ((2, 32), (3, 96)):
        w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        codes, scales = oracle.mxfp4_quantize(w)
        x = workloads.bits16(workloads.activations_bf16(1, K, seed=N))[0]
        y, a = oracle.mxfp4_gemv(x, codes, scales)
        qn = _nv_codes(codes)
        for n in range(N):
            exact = sum(Fraction(_bf16(x[k])) * Fraction(oracle.e2m1_value(int(qn[n, k]))) *
                        Fraction(2) ** (int(scales[n, k // 32]) - 127) for k in range(K))
            assert abs(Fraction(y[n]) - exact) <= Fraction(a[n]) / 2**45, (N, K, n)
    N, K = 48, 1024
    w = workloads.weights(N, K, seed=54, outlier_frac=0.001).numpy()
    codes, scales = oracle.mxfp4_quantize(w)
    w_hat = oracle.mxfp4_dequant(codes, scales)
    x = workloads.bits16(workloads.activations_bf16(1, K, seed=54))[0]
    y, a = oracle.mxfp4_gemv(x, codes, scales)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
    ref = (torch.from_numpy(w_hat) @ xv).numpy()
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    rows = np.array([N - 1, 2], dtype=np.int32)
    y2, _ = oracle.mxfp4_gemv(x, codes, scales, rows=rows)
    np.testing.assert_array_equal(y2, y[rows])
    w = workloads.weights(256, 2048, seed=0, outlier_frac=0.001).numpy()
    c, s = oracle.mxfp4_quantize(w)
    e_mx = np.linalg.norm(oracle.mxfp4_dequant(c, s) - w) / np.linalg.norm(w)
    c4, s4, S4 = oracle.nvfp4_quantize(w)
    e_nv = np.linalg.norm(oracle.nvfp4_dequant(c4, s4, S4) - w) / np.linalg.norm(w)
    assert e_nv < e_mx and 0.08 < e_mx < 0.16, (e_nv, e_mx)


def pin_fp4_matmul_exact_and_library():
    """The NVFP4A16 / MXFP4A16 matmuls: every output of small batches equals the exact
    rational sum over the rebuilt weights (rows of x of different magnitudes, so a
    transposed or shared row fails); a larger batch equals torch.matmul (fp64) of x and the
    dequantized weights; the row subset matches."""
    rng = np.random.default_rng(61)
    M, N, K = 3, 4, 64
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = workloads.bits16(workloads.activations_bf16(M, K, seed=61)
                         * torch.tensor([[1.0], [-8.0], [0.25]]).to(torch.bfloat16))
    c4, s4, S4 = oracle.nvfp4_quantize(w)
    cm, sm = oracle.mxfp4_quantize(w)
    y4, a4 = oracle.nvfp4_matmul(x, c4, s4, S4)
    ym, am = oracle.mxfp4_matmul(x, cm, sm)
    assert y4.shape == (M, N) and ym.shape == (M, N)
    q4, qm = _nv_codes(c4), _nv_codes(cm)
    for m in range(M):
        for n in range(N):
            e4 = sum(Fraction(_bf16(x[m, k])) * Fraction(oracle.e2m1_value(int(q4[n, k]))) *
                     Fraction(oracle.e4m3_value(int(s4[n, k // 16]))) * Fraction(S4)
                     for k in range(K))
            em = sum(Fraction(_bf16(x[m, k])) * Fraction(oracle.e2m1_value(int(qm[n, k]))) *
                     Fraction(2) ** (int(sm[n, k // 32]) - 127) for k in range(K))
            assert abs(Fraction(y4[m, n]) - e4) <= Fraction(a4[m, n]) / 2**45, (m, n)
            assert abs(Fraction(ym[m, n]) - em) <= Fraction(am[m, n]) / 2**45, (m, n)
    M, N, K = 5, 40, 512
    w = workloads.weights(N, K, seed=62, outlier_frac=0.001).numpy()
    c4, s4, S4 = oracle.nvfp4_quantize(w)
    cm, sm = oracle.mxfp4_quantize(w)
    x = workloads.bits16(workloads.activations_bf16(M, K, seed=62))
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).double()
    for (y, a), w_hat in ((oracle.nvfp4_matmul(x, c4, s4, S4), oracle.nvfp4_dequant(c4, s4, S4)),
                          (oracle.mxfp4_matmul(x, cm, sm), oracle.mxfp4_dequant(cm, sm))):
        ref = (xv @ torch.from_numpy(w_hat).T).numpy()
        assert np.all(np.abs(y - ref) <= 1e-12 * a)
    rows = np.array([N - 1, 7], dtype=np.int32)
    y, _ = oracle.mxfp4_matmul(x, cm, sm)
    y2, _ = oracle.mxfp4_matmul(x, cm, sm, rows=rows)
    np.testing.assert_array_equal(y2, y[:, rows])

ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
