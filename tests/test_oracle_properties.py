"""Property checks of the oracle's element rules on generated inputs (no GPU): each code the
oracle stores is a nearest grid point of its quotient in exact arithmetic, with the tie rule
the format's page gives, and rebuilding from the codes never moves a weight by more than half
a step (plus the clamp at the ends). Cases near a tie, where the fp32 quotient may decide
otherwise, are skipped."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402
from hypothesis.extra import numpy as hnp  # noqa: E402

finite = st.floats(min_value=-1e4, max_value=1e4, allow_nan=False, allow_infinity=False,
                   width=32)
scale_exp = st.integers(min_value=-20, max_value=10)


def near_tie(t: Fraction, eps=Fraction(1, 2**16)) -> bool:
    return abs(abs(t - math.floor(t)) - Fraction(1, 2)) <= eps


def half_away(t: Fraction) -> int:
    a = math.floor(abs(t) + Fraction(1, 2))
    return a if t >= 0 else -a


@settings(max_examples=60, deadline=None)
@given(hnp.arrays(np.float32, (2, 64), elements=finite), scale_exp)
def test_w8a16_codes_are_nearest(w, e):
    w = (w * np.float32(2.0 ** e)).astype(np.float32)
    q, s = oracle.w8a16_quantize(w)
    for n in range(2):
        if s[n] == 0:
            assert not q[n].any()
            continue
        sf = Fraction(float(s[n]))
        for k in range(64):
            t = Fraction(float(w[n, k])) / sf
            if near_tie(t):
                continue
            assert int(q[n, k]) == max(-127, min(127, half_away(t)))


@settings(max_examples=60, deadline=None)
@given(hnp.arrays(np.float32, (1, 128), elements=finite), scale_exp)
def test_zero_point_codes_within_half_a_step(w, e):
    w = (w * np.float32(2.0 ** e)).astype(np.float32)
    qw_rows, s, z = oracle.w4a16zp_quantize(w)
    w_hat = oracle.w4a16zp_dequant(qw_rows, s, z)
    sf = float(oracle.fp16_to_float(s.ravel())[0])
    zf = float(oracle.fp16_to_float(z.ravel())[0])
    if not (math.isfinite(sf) and math.isfinite(zf)) or abs(zf) > 2048:
        return  # outside the format (a zero point beyond FP16's integers)
    lo, hi = (-zf) * sf, (15 - zf) * sf
    for k in range(128):
        wk = float(w[0, k])
        if lo - 0.5 * sf <= wk <= hi + 0.5 * sf:
            assert abs(w_hat[0, k] - wk) <= 0.5 * sf * (1 + 2**-10) + 2**-20 * abs(wk), (k, wk)


@settings(max_examples=60, deadline=None)
@given(hnp.arrays(np.float32, (1, 64), elements=finite), scale_exp)
def test_mxfp4_codes_are_nearest_and_scale_fits(w, e):
    w = (w * np.float32(2.0 ** e)).astype(np.float32)
    codes, scales = oracle.mxfp4_quantize(w)
    grid = [Fraction(int(2 * oracle.e2m1_value(c)), 2) for c in range(8)]
    c = np.stack([codes & 15, codes >> 4], axis=-1).reshape(1, -1)
    for b in range(2):
        blk = w[0, 32 * b:32 * (b + 1)]
        amax = float(np.abs(blk).max())
        if amax == 0:
            assert scales[0, b] == 0 and not c[0, 32 * b:32 * (b + 1)].any()
            continue
        X = int(scales[0, b]) - 127
        assert 2.0 ** (X + 2) <= amax < 2.0 ** (X + 3) or X == -127
        for j, wv in enumerate(blk):
            t = abs(Fraction(float(wv)) / Fraction(2) ** X)
            code = int(c[0, 32 * b + j]) & 7
            if t >= 6:
                assert code == 7
            else:
                d = [abs(t - g) for g in grid]
                assert code == min(range(8), key=lambda i: (d[i], i & 1))


@settings(max_examples=40, deadline=None)
@given(hnp.arrays(np.float32, (1, 32), elements=finite), scale_exp)
def test_nvfp4_block_scale_never_clips(w, e):
    """The round-up rule: a block's largest weight divided by its rebuilt scale is at most
    6 (up to the fp32 rounding of the quotient), so no weight saturates below its value."""
    w = (w * np.float32(2.0 ** e)).astype(np.float32)
    codes, scales, S = oracle.nvfp4_quantize(w)
    for b in range(2):
        blk = w[0, 16 * b:16 * (b + 1)]
        amax = float(np.abs(blk).max())
        if amax == 0 or scales[0, b] == 0x7E:
            continue
        sb = oracle.e4m3_value(int(scales[0, b]))
        assert amax / (sb * S) <= 6 * (1 + 2**-20), (amax, sb, S)
