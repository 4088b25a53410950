"""NVFP4 weights with BF16 activations (E2M1 codes, E4M3 block scales of 16, one fp32 tensor
scale) through the C ABI against the oracle.

Quantize must match the oracle bit for bit (codes, block scales, tensor scale); the GEMV must
meet |y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k| on every output, at sizes spanning
several 16-row tiles with a ragged last tile and at the full 14336 x 4096 layer.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemv_w4a16_group_gb300 as mod

    return mod


@pytest.fixture(params=[1, 0], ids=["ring", "plain"])
def fp4_variant(request, w4):
    """Run the GEMV test through the tensor-pipe ring kernel (shapes it does not take fall
    back to the plain-load kernel) and through the plain-load kernel."""
    prev = w4.testing_set_fp4_variant(request.param)
    yield request.param
    w4.testing_set_fp4_variant(prev)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def special_weights(N, K, seed):
    """Seeded N(0, 0.02^2) weights with 0.1 % outliers, plus a block of zeros, a block of
    negative zeros, blocks of exact ties (x.25, x.75 and 2.5, 5 on the E2M1 grid) and a block
    whose scale E4M3 would round down."""
    w = workloads.weights(N, K, seed=seed, outlier_frac=0.001).numpy().copy()
    if N >= 4 and K >= 64:
        amax = float(np.abs(w).max())
        S = np.float32(np.float32(amax) / np.float32(2688))
        w[0, :16] = 0.0
        w[0, 16:32] = -0.0
        # a block whose largest |w| is 6 s_b with s_b = 0.25 S: quotients on the E2M1 grid
        # and at its midpoints
        grid = np.array([6, 2.5, 5, 0.25, 0.75, 1.25, 1.75, 3.5, -2.5, -5, -0.25, -6, 0, 1, 4, -1.5])
        w[1, :16] = grid * 0.25 * S
        w[2, :16] = np.linspace(-0.87, 0.87, 16) * 64 * S
    return np.ascontiguousarray(w, dtype=np.float32)


@pytest.mark.parametrize("N,K", [(16, 128), (100, 512), (1000, 4096), (7, 8192)])
def test_nvfp4_quantize_bit_exact(w4, N, K):
    w = special_weights(N, K, seed=N + K)
    c_ref, s_ref, S_ref = oracle.nvfp4_quantize(w)
    c, s, S = w4.nvfp4_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert S.cpu().numpy().view(np.uint32)[0] == np.float32(S_ref).view(np.uint32)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(c.cpu().numpy(), c_ref)


def test_nvfp4_quantize_hand_worked_tensors(w4):
    """The tensors of tests/golden/nvfp4_blocks.txt, each row repeated four times (K = 128)."""
    import pins

    for tag, rec in pins._records("nvfp4_blocks.txt"):
        w = np.tile(pins._weights_from(rec), 4).reshape(1, -1).astype(np.float32)
        c, s, S = w4.nvfp4_quantize(torch.from_numpy(w).cuda())
        torch.cuda.synchronize()
        assert S.cpu().numpy().view(np.uint32)[0] == int(rec["S"][0], 16), tag
        assert [int(v) for v in s.cpu().numpy()[0, :2]] == [int(v, 16) for v in rec["scales"]], tag
        assert [int(v) for v in c.cpu().numpy()[0, :16]] == [int(v, 16) for v in rec["bytes"]], tag


# K % 512 == 0 takes the ring kernel, units of T tiles of 16 rows split over P k-parts (on
# 152 SMs): N = 13, 40, 333, 1000 (T = 1, P = 16), 4096 (2, 8), 6000 (3, 8), 9000 (4, 4),
# 14336 (6, 4), 12008 (6, 4; the last unit one ragged tile), 16384 (8, 2), 28672 (12, 2);
# x up to 64 k long, and the longest K the ring takes (NVFP4 92,160) beside the next multiple
# of 512, which falls back to the plain-load kernel. P = 16 and 8 fold groups of one and two
# 32-k blocks, P = 4 one group of four, P = 2 two groups of four per chunk.
@pytest.mark.parametrize("N,K", [(16, 128), (17, 256), (13, 512), (333, 1024), (1000, 4224),
                                 (1000, 4608), (4096, 4096), (6000, 2048), (9000, 1536),
                                 (14336, 4096), (12008, 1536), (16384, 1024), (28672, 1024),
                                 (40, 65536), (16, 92160), (16, 92672)])
def test_nvfp4_gemv_every_output(w4, fp4_variant, N, K):
    w = special_weights(N, K, seed=N * 5 + K)
    c_np, s_np, S = oracle.nvfp4_quantize(w)
    x = workloads.activations_bf16(1, K, seed=N)[0]
    c, s = torch.from_numpy(c_np).cuda(), torch.from_numpy(s_np).cuda()
    St = torch.tensor([S], dtype=torch.float32, device="cuda")
    y = w4.nvfp4_gemv(x.cuda(), c, s, St)
    y2 = w4.nvfp4_gemv(x.cuda(), c, s, St)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    y_ref, a_ref = oracle.nvfp4_gemv(bits(x), c_np, s_np, S)
    yv = y.float().cpu().numpy()
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.flatnonzero(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} out of tolerance: "
                             f"{[(int(n), float(yv[n]), float(y_ref[n])) for n in bad]}")


def test_nvfp4_gemv_special_activations(w4, fp4_variant):
    """x with a zero chunk, a 2^20 range of magnitudes inside a chunk and a large value."""
    N, K = 96, 1024
    w = special_weights(N, K, seed=9)
    c_np, s_np, S = oracle.nvfp4_quantize(w)
    x = workloads.activations_bf16(1, K, seed=9)[0].clone()
    x[:128] = 0
    x[128:256] = x[128:256] * torch.logspace(-10, 10, 128, base=2.0).to(torch.bfloat16)
    x[300] = 3.0e4
    St = torch.tensor([S], dtype=torch.float32, device="cuda")
    y = w4.nvfp4_gemv(x.cuda(), torch.from_numpy(c_np).cuda(), torch.from_numpy(s_np).cuda(), St)
    torch.cuda.synchronize()
    y_ref, a_ref = oracle.nvfp4_gemv(bits(x), c_np, s_np, S)
    assert oracle.within_tolerance(y.float().cpu().numpy(), y_ref, a_ref).all()


# --------------------------------------------------------------------------- #
# MXFP4 (E2M1 codes, E8M0 power-of-two scale per 32)
# --------------------------------------------------------------------------- #

def mx_special_weights(N, K, seed):
    """Seeded weights with 0.1 % outliers, a zero block, blocks on the grid with exact ties,
    a block needing the clamp at 6, and rows whose blocks differ by large powers of two."""
    w = workloads.weights(N, K, seed=seed, outlier_frac=0.001).numpy().copy()
    if N >= 4 and K >= 128:
        w[0, :32] = 0.0
        grid = np.array([6, 2.5, 5, 0.25, 0.75, 1.25, 1.75, 3.5, -2.5, -5, -0.25, -6, 0, 1, 4,
                         -1.5] * 2)
        w[1, :32] = grid * 2.0 ** -9
        w[2, :32] = np.linspace(-0.9, 0.9, 32) * 2.0 ** -5  # 0.9 scaled past 6: clamped
        w[3, :128] *= np.repeat(2.0 ** np.array([-30, 0, -12, 10]), 32)
    return np.ascontiguousarray(w, dtype=np.float32)


@pytest.mark.parametrize("N,K", [(16, 128), (100, 512), (1000, 4096), (7, 8224)])
def test_mxfp4_quantize_bit_exact(w4, N, K):
    w = mx_special_weights(N, K, seed=N + K)
    c_ref, s_ref = oracle.mxfp4_quantize(w)
    c, s = w4.mxfp4_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(c.cpu().numpy(), c_ref)


def test_mxfp4_quantize_hand_worked_blocks(w4):
    """The blocks of tests/golden/mxfp4_blocks.txt, one row each."""
    import pins

    recs = pins._records("mxfp4_blocks.txt")
    w = np.stack([pins._weights_from(rec) for _, rec in recs]).astype(np.float32)
    c, s = w4.mxfp4_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    for i, (tag, rec) in enumerate(recs):
        assert int(s.cpu().numpy()[i, 0]) == int(rec["scale"][0], 16), tag
        assert [int(v) for v in c.cpu().numpy()[i]] == [int(v, 16) for v in rec["bytes"]], tag


@pytest.mark.parametrize("N,K", [(16, 128), (17, 256), (13, 512), (333, 1024), (1000, 4224),
                                 (1000, 4608), (4096, 4096), (6000, 2048), (9000, 1536),
                                 (14336, 4096), (12008, 1536), (16384, 1024), (28672, 1024),
                                 (40, 65536), (16, 102912), (16, 103424)])
def test_mxfp4_gemv_every_output(w4, fp4_variant, N, K):
    w = mx_special_weights(N, K, seed=N * 7 + K)
    c_np, s_np = oracle.mxfp4_quantize(w)
    x = workloads.activations_bf16(1, K, seed=N)[0]
    c, s = torch.from_numpy(c_np).cuda(), torch.from_numpy(s_np).cuda()
    y = w4.mxfp4_gemv(x.cuda(), c, s)
    y2 = w4.mxfp4_gemv(x.cuda(), c, s)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    y_ref, a_ref = oracle.mxfp4_gemv(bits(x), c_np, s_np)
    yv = y.float().cpu().numpy()
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.flatnonzero(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} out of tolerance: "
                             f"{[(int(n), float(yv[n]), float(y_ref[n])) for n in bad]}")


# --------------------------------------------------------------------------- #
# M > 1: nvfp4_matmul / mxfp4_matmul (x prepared once, one pass per 32 rows)
# --------------------------------------------------------------------------- #

def _fp4_case(fmt, N, K, seed):
    if fmt == "nv":
        w = special_weights(N, K, seed=seed)
        c, s, S = oracle.nvfp4_quantize(w)
        return c, s, S
    w = mx_special_weights(N, K, seed=seed)
    c, s = oracle.mxfp4_quantize(w)
    return c, s, None


def _fp4_run(w4, fmt, x, c, s, S, y=None, workspace=None):
    cd, sd = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    if fmt == "nv":
        St = torch.tensor([S], dtype=torch.float32, device="cuda")
        return w4.nvfp4_matmul(x, cd, sd, St, y=y, workspace=workspace)
    return w4.mxfp4_matmul(x, cd, sd, y=y, workspace=workspace)


def _fp4_ref(fmt, x, c, s, S, rows=None):
    xb = bits(x).reshape(x.shape[0], -1)
    if fmt == "nv":
        return oracle.nvfp4_matmul(xb, c, s, S, rows=rows)
    return oracle.mxfp4_matmul(xb, c, s, rows=rows)


def _fp4_check(y, y_ref, a_ref, cols=None):
    yv = y.float().cpu().numpy()
    if cols is not None:
        yv = yv[:, cols]
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} out of tolerance: "
                             f"{[(int(i), int(j), float(yv[i, j]), float(y_ref[i, j])) for i, j in bad]}")


# Passes of 8, 16 and 32 rows (M = 2 .. 8, 9 .. 16, 17 .. 32) and several passes (33, 70);
# units of (2, 8), (6, 4) and (12, 2) tiles x k-parts; ragged N and the last unit.
@pytest.mark.parametrize("fmt", ["nv", "mx"])
@pytest.mark.parametrize("M,N,K", [(2, 16, 512), (3, 40, 1024), (8, 333, 512), (9, 1000, 1536),
                                   (16, 256, 512), (17, 136, 1024), (32, 5000, 1024),
                                   (33, 520, 512), (70, 264, 2048), (5, 28680, 512)])
def test_fp4_matmul_every_output(w4, fmt, M, N, K):
    c, s, S = _fp4_case(fmt, N, K, seed=M * 31 + N)
    x = workloads.activations_bf16(M, K, seed=M + K)
    x[M // 2] *= 64  # rows of different magnitudes: each row keeps its own power of two
    xd = x.cuda()
    y1 = _fp4_run(w4, fmt, xd, c, s, S)
    y2 = _fp4_run(w4, fmt, xd, c, s, S)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    y_ref, a_ref = _fp4_ref(fmt, x, c, s, S)
    _fp4_check(y1, y_ref, a_ref)
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("fmt", ["nv", "mx"])
@pytest.mark.parametrize("M", [2, 8, 16, 32, 64])
def test_fp4_matmul_full_size(w4, fmt, M):
    """The 14336 x 4096 up-projection at batch sizes up to 64: every batch row of one weight
    row in each 16-row tile (and both tile halves), with the library's own workspace."""
    N, K = 14336, 4096
    c, s, S = _fp4_case(fmt, N, K, seed=7)
    x = workloads.activations_bf16(M, K, seed=M)
    ws = torch.zeros(w4.fp4_matmul_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y = _fp4_run(w4, fmt, x.cuda(), c, s, S, workspace=ws)
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    cols = (np.arange(0, N, 16) + rng.integers(0, 16, size=N // 16)).astype(np.int32)
    y_ref, a_ref = _fp4_ref(fmt, x, c, s, S, rows=cols)
    _fp4_check(y, y_ref, a_ref, cols)
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("fmt", ["nv", "mx"])
def test_fp4_matmul_m1_is_the_gemv_and_guard_bands(w4, fmt):
    """M = 1 gives the GEMV's bits; for M > 1 exactly y[M, N] is written."""
    N, K = 200, 1024
    c, s, S = _fp4_case(fmt, N, K, seed=3)
    x = workloads.activations_bf16(1, K, seed=3).cuda()
    y = _fp4_run(w4, fmt, x, c, s, S)
    cd, sd = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    if fmt == "nv":
        g = w4.nvfp4_gemv(x[0], cd, sd, torch.tensor([S], dtype=torch.float32, device="cuda"))
    else:
        g = w4.mxfp4_gemv(x[0], cd, sd)
    torch.cuda.synchronize()
    assert torch.equal(y[0].view(torch.int16), g.view(torch.int16))
    M, pad = 11, 4096
    buf = torch.full((pad + M * N + pad,), 12345, dtype=torch.int16, device="cuda")
    yv = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    x = workloads.activations_bf16(M, K, seed=4)
    _fp4_run(w4, fmt, x.cuda(), c, s, S, y=yv)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + M * N:] == 12345)
    y_ref, a_ref = _fp4_ref(fmt, x, c, s, S)
    _fp4_check(yv, y_ref, a_ref)
