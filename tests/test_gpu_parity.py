"""Parity of the CUDA path (through the C ABI) with the CPU oracle on seeded inputs.

Quantize and pack must match bit for bit; matmul and Q4 outputs must satisfy
|y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k| per output. Full-size launches are
checked on every output where the oracle is fast enough, else on sampled columns.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

GEMV, TCGEN05 = 1, 2
KERNELS = {"gemv": GEMV, "tcgen05": TCGEN05}


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemv_w4a16_group_gb300 as mod

    return mod


@pytest.fixture
def force_kernel(w4):
    prev = []

    def set_kernel(k):
        prev.append(w4.testing_force_kernel(k))

    yield set_kernel
    w4.testing_force_kernel(0)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def quantized(N, K, seed=0, outliers=0.0):
    """CPU weights and their oracle quantization, packed."""
    w = workloads.weights(N, K, seed=seed, outlier_frac=outliers)
    codes, s, m = oracle.w4a16_quantize(w.numpy())
    return w, codes, s, m, oracle.w4a16_pack(codes)


def to_dev_params(codes, s, m, qw):
    dev = "cuda"
    return (torch.from_numpy(qw).to(dev),
            torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).to(dev),
            torch.from_numpy(m.view(np.int16)).view(torch.bfloat16).to(dev))


def check_matmul(w4, x, qw_np, s_np, m_np, qw, s, m, cols=None):
    y = w4.w4a16_matmul(x.cuda(), qw, s, m)
    torch.cuda.synchronize()
    yv = y.float().cpu().numpy()
    y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np, cols=cols)
    if cols is not None:
        yv = yv[:, cols]
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(int(i), int(j), float(yv[i, j]), float(y_ref[i, j])) for i, j in bad]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} outputs out of tolerance: {detail}")
    return y


# --------------------------------------------------------------------------- #
# quantize / pack: bit-exact
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("N,K,outliers", [(256, 512, 0.0), (72, 384, 0.0), (1000, 1280, 0.001),
                                          (14336, 4096, 0.0), (14336, 4096, 0.001)])
def test_quantize_pack_bit_exact(w4, N, K, outliers):
    w, codes, s, m, qw = quantized(N, K, seed=N + K, outliers=outliers)
    gc, gs, gm = w4.w4a16_quantize(w.cuda())
    gq = w4.w4a16_pack(gc)
    torch.cuda.synchronize()
    assert np.array_equal(gc.cpu().numpy(), codes)
    assert np.array_equal(bits(gs), s)
    assert np.array_equal(bits(gm), m)
    assert np.array_equal(gq.cpu().numpy(), qw)


def test_quantize_on_grid_and_degenerate_groups(w4):
    """Constant groups (scale 0), on-grid groups and exact ties, bit-exact."""
    N, K = 16, 512
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[0, :128] = 0.3                      # constant group -> scale 0, q = 0
    w[1, 128:256] = -1.5                  # constant negative
    q = rng.integers(0, 16, size=128)
    q[0], q[1] = 0, 15
    w[2, 256:384] = (-0.75 + 0.25 * q).astype(np.float32)           # on the grid
    w[3, 384:512] = (-0.75 + 0.25 * (q + 0.5)).astype(np.float32)   # exact ties
    w[3, 384], w[3, 385] = -0.75, 3.0
    codes, s, m = oracle.w4a16_quantize(w)
    gc, gs, gm = w4.w4a16_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(gc.cpu().numpy(), codes)
    assert np.array_equal(bits(gs), s) and np.array_equal(bits(gm), m)


@pytest.mark.parametrize("N,K", [(8, 8), (64, 512), (100, 520), (333, 1024), (4096, 4104)])
def test_pack_bit_exact_with_high_bits(w4, N, K):
    rng = np.random.default_rng(N)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)  # high nibble must be ignored
    ref = oracle.w4a16_pack(codes)
    got = w4.w4a16_pack(torch.from_numpy(codes).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)


# --------------------------------------------------------------------------- #
# matmul: tolerance, every kernel
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (1, 8, 128), (2, 264, 384), (3, 136, 1536),
                                   (4, 1536, 1536), (5, 256, 640), (8, 520, 256),
                                   (13, 256, 512), (16, 384, 1024), (17, 256, 512),
                                   (32, 640, 768), (64, 256, 1536), (100, 392, 512),
                                   (128, 256, 512), (200, 264, 640), (256, 384, 384),
                                   (300, 256, 256), (191, 256, 512), (192, 136, 384),
                                   (193, 264, 640), (385, 256, 256), (700, 520, 384)])
def test_matmul_small_shapes(w4, force_kernel, kernel, M, N, K):
    """Every output; batch tiles with a ragged last one (M = 191, 193, 385, 700)."""
    if kernel == "gemv" and M > 64:
        pytest.skip("the GEMV kernel is only meant for small M")
    force_kernel(KERNELS[kernel])
    w, codes, s_np, m_np, qw_np = quantized(N, K, seed=M * 7 + N)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x = workloads.activations_bf16(M, K, seed=M + K)
    check_matmul(w4, x, qw_np, s_np, m_np, qw, s, m)


def oracle_matmul_par(x_bits, qw_np, s_np, m_np, cols):
    """The unchanged oracle over disjoint slices of `cols`, one host thread per slice (the
    oracle is C behind ctypes, which releases the GIL)."""
    import concurrent.futures as cf
    import os

    cols = np.asarray(cols, dtype=np.int32)
    try:
        cores = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        cores = os.cpu_count() or 1
    parts = [p for p in np.array_split(cols, max(1, min(cores, 64))) if len(p)]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        res = list(ex.map(lambda p: oracle.w4a16_matmul(x_bits, qw_np, s_np, m_np, cols=p),
                          parts))
    return np.concatenate([r[0] for r in res], axis=1), np.concatenate([r[1] for r in res],
                                                                         axis=1)


def tile_quarter_columns(N, seed):
    """One seeded column in every 32-column quarter of every 128-column tile: each tile of
    the tensor-core kernels and each 32-lane quarter of its accumulator is compared."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, N, 32)
    return np.array([s + rng.integers(0, min(32, N - s)) for s in starts], dtype=np.int32)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64, 128, 256, 1024, 4096])
def test_batch_sweep_full_size(w4, M):
    """Llama-3-8B up-projection shape with 0.1 % outliers x10, automatic kernel choice (the
    launch the benchmark times): every output at M <= 256; at M = 1024 and 4096 every row
    of one column in each 32-column quarter of every 128-column tile (448 columns)."""
    cfg = workloads.BATCH_SWEEP
    N, K = cfg["N"], cfg["K"]
    w, codes, s_np, m_np, qw_np = _sweep_weights()
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x = workloads.activations_bf16(M, K, seed=M)
    cols = np.arange(N, dtype=np.int32) if M <= 256 else tile_quarter_columns(N, seed=M)
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda") if need else None
    y_ref, a_ref = oracle_matmul_par(bits(x), qw_np, s_np, m_np, cols)
    # with the workspace the library asks for (the benchmark's launch), and without one
    for workspace in ([ws, None] if need else [None]):
        y = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=workspace)
        torch.cuda.synchronize()
        yv = y.float().cpu().numpy()[:, cols]
        ok = oracle.within_tolerance(yv, y_ref, a_ref)
        if not ok.all():
            bad = np.argwhere(~ok)[:5]
            detail = [(int(i), int(cols[j]), float(yv[i, j]), float(y_ref[i, j]))
                      for i, j in bad]
            raise AssertionError(f"workspace={workspace is not None}: {int((~ok).sum())}/"
                                 f"{ok.size} outputs out of tolerance: {detail}")
    assert w4.w4a16_device_status() == 0


_SWEEP = {}


def _sweep_weights():
    if "w" not in _SWEEP:
        cfg = workloads.BATCH_SWEEP
        _SWEEP["w"] = quantized(cfg["N"], cfg["K"], seed=0, outliers=cfg["outlier_frac"])
    return _SWEEP["w"]


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_llama_up_proj_m1_every_output(w4, force_kernel, kernel):
    cfg = workloads.LLAMA_UP
    force_kernel(KERNELS[kernel])
    w, codes, s_np, m_np, qw_np = quantized(cfg["N"], cfg["K"], seed=0)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x = workloads.activations_bf16(1, cfg["K"], seed=0)
    check_matmul(w4, x, qw_np, s_np, m_np, qw, s, m)


@pytest.mark.parametrize("name,N,K", [(n, N, K) for n, N, K in workloads.QWEN_BLOCK])
def test_qwen_stack_shapes_m1(w4, name, N, K):
    w, codes, s_np, m_np, qw_np = quantized(N, K, seed=sum(map(ord, name)))
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x = workloads.activations_bf16(1, K, seed=K)
    check_matmul(w4, x, qw_np, s_np, m_np, qw, s, m)


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_matmul_special_inputs(w4, force_kernel, kernel):
    """x = 0 gives exactly 0; one-hot x gives w_hat[n, k] to BF16 rounding; constant
    groups; deterministic results (same bits twice)."""
    force_kernel(KERNELS[kernel])
    N, K = 256, 512
    w, codes, s_np, m_np, qw_np = quantized(N, K, seed=5)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x0 = torch.zeros(3, K, dtype=torch.bfloat16)
    y0 = w4.w4a16_matmul(x0.cuda(), qw, s, m)
    assert torch.count_nonzero(y0).item() == 0
    w_hat = oracle.w4a16_dequant(qw_np, s_np, m_np)
    scale = torch.from_numpy(s_np.view(np.int16)).view(torch.bfloat16).double().numpy()
    for k in (0, 127, 128, 511):
        x1 = torch.zeros(1, K, dtype=torch.bfloat16)
        x1[0, k] = 1.0
        y1 = w4.w4a16_matmul(x1.cuda(), qw, s, m).float().cpu().numpy()[0]
        ref = w_hat[:, k]
        # BF16 rounding of y, plus the fp32 rounding of the factorised form
        # s * (128 + q) + (min - 128 s), which is absolute and scales with s.
        assert np.all(np.abs(y1 - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -12 * scale[k // 128]), k
    x = workloads.activations_bf16(4, K, seed=9).cuda()
    a = w4.w4a16_matmul(x, qw, s, m)
    b = w4.w4a16_matmul(x, qw, s, m)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_matmul_guard_bands(w4, force_kernel, kernel):
    """The kernels write exactly y[M, N]: sentinels around it stay untouched."""
    force_kernel(KERNELS[kernel])
    M, N, K = 3, 264, 384
    w, codes, s_np, m_np, qw_np = quantized(N, K, seed=11)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    x = workloads.activations_bf16(M, K, seed=1)
    w4.w4a16_matmul(x.cuda(), qw, s, m, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + M * N:] == 12345)
    y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np)
    assert oracle.within_tolerance(y.float().cpu().numpy(), y_ref, a_ref).all()


def test_matmul_rejects_misaligned_views(w4):
    N, K = 256, 512
    w, codes, s_np, m_np, qw_np = quantized(N, K)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    xbuf = torch.zeros(K + 1, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4A16Error, match="MISALIGNED"):
        w4.w4a16_matmul(xbuf[1:].view(1, K), qw, s, m)


# --------------------------------------------------------------------------- #
# Q4 block-32
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("N,K", [(256, 512), (8, 32), (13, 96), (1000, 1056), (4096, 4096),
                                 (13, 1024), (2056, 2560), (300, 5120)])
def test_q4_quantize_and_gemv(w4, variant, N, K):
    """Variant 2 is the TMA / tensor-pipe kernel where it takes the shape (K % 512 == 0),
    else the CUDA-core kernel; 0 and 1 force the CUDA-core inner products."""
    prev = w4.testing_set_q4_variant(variant)
    try:
        w = workloads.weights(N, K, seed=N)
        codes, sc = oracle.q4b32_quantize(w.numpy())
        gc, gs = w4.q4b32_quantize(w.cuda())
        torch.cuda.synchronize()
        assert np.array_equal(gc.cpu().numpy(), codes)
        assert np.array_equal(bits(gs), sc)
        x = workloads.activations_fp16(K, seed=K)
        y = w4.q4b32_gemv(x.cuda(), gc, gs).float().cpu().numpy()
        y_ref, a_ref = oracle.q4b32_gemv(bits(x), codes, sc)
        ok = oracle.within_tolerance(y, y_ref, a_ref)
        assert ok.all(), int((~ok).sum())
    finally:
        w4.testing_set_q4_variant(prev)


def test_q4_square_full_size(w4):
    cfg = workloads.Q4_SQUARE
    N, K = cfg["N"], cfg["K"]
    w = workloads.weights(N, K, seed=0)
    codes, sc = oracle.q4b32_quantize(w.numpy())
    gc, gs = w4.q4b32_quantize(w.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(gc.cpu().numpy(), codes)
    assert np.array_equal(bits(gs), sc)
    del w
    x = workloads.activations_fp16(K, seed=0)
    y = w4.q4b32_gemv(x.cuda(), gc, gs).float().cpu().numpy()
    rows = workloads.sample_indices(N, 2048, seed=1).numpy()
    y_ref, a_ref = oracle.q4b32_gemv(bits(x), codes, sc, rows=rows)
    assert oracle.within_tolerance(y[rows], y_ref, a_ref).all()


# --------------------------------------------------------------------------- #
# failure detection without a fault
# --------------------------------------------------------------------------- #

def test_bounded_wait_expires_and_is_reported(w4):
    assert w4.w4a16_device_status() == 0
    assert w4.w4a16_selftest_bounded_wait(2000) == 0
    assert w4.w4a16_device_status() == 5  # W4A16_ERR_TIMEOUT, then cleared
    assert w4.w4a16_device_status() == 0
    # the context is still usable
    z = torch.ones(4, device="cuda") * 2
    assert z.sum().item() == 8.0


# --------------------------------------------------------------------------- #
# split K through a caller-owned workspace
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("M,N,K", [(1, 14336, 4096), (3, 1536, 1536), (8, 1536, 8960),
                                   (16, 14336, 4096), (32, 256, 1536), (64, 8960, 1536),
                                   (128, 1536, 1536), (200, 1024, 4096)])
def test_matmul_split_k_workspace(w4, M, N, K):
    """Small-M tensor-core launches split K over CTAs through the workspace: same
    tolerance, same bits twice, and the workspace's counters are left at zero."""
    prev = w4.testing_set_gemv_max_m(0)  # every M takes the tensor-core kernel
    try:
        need = w4.w4a16_matmul_workspace_bytes(M, N, K)
        w, codes, s_np, m_np, qw_np = quantized(N, K, seed=M + N)
        qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
        x = workloads.activations_bf16(M, K, seed=M)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
        y1 = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws if need else None)
        y2 = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws if need else None)
        torch.cuda.synchronize()
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
        cols = None if M * N * K <= 2**31 else workloads.sample_indices(N, 64, seed=M).numpy()
        y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np, cols=cols)
        yv = y1.float().cpu().numpy()
        if cols is not None:
            yv = yv[:, cols]
        assert oracle.within_tolerance(yv, y_ref, a_ref).all()
        if need:
            tiles = (N + 127) // 128  # one m-tile at every M used here
            assert torch.count_nonzero(ws[:256 * ((tiles * 4 + 255) // 256)]).item() == 0
        assert w4.w4a16_device_status() == 0
    finally:
        w4.testing_set_gemv_max_m(prev)


@pytest.mark.parametrize("M,N,K", [(1, 1536, 8960), (2, 4096, 14336), (4, 1536, 8960),
                                   (8, 512, 8192), (1, 4096, 4096), (3, 256, 8192)])
def test_gemv_split_k_workspace(w4, M, N, K):
    """GEMV launches (M <= 8) that split K over CTAs through the workspace (and one shape,
    4096 x 4096, whose plan no longer splits): the oracle's tolerance, the same bits twice,
    and the arrival counters (at most 64 slabs here: the first 256 bytes) left at zero."""
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    w, codes, s_np, m_np, qw_np = quantized(N, K, seed=3 * M + N)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x = workloads.activations_bf16(M, K, seed=K + M)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    y1 = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws if need else None)
    y2 = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws if need else None)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    cols = None if N * K <= 2**24 else workloads.sample_indices(N, 128, seed=M).numpy()
    y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np, cols=cols)
    yv = y1.float().cpu().numpy()
    if cols is not None:
        yv = yv[:, cols]
    assert oracle.within_tolerance(yv, y_ref, a_ref).all()
    assert torch.count_nonzero(ws[:256]).item() == 0
    assert w4.w4a16_device_status() == 0


def test_q4_quantize_exact_ties(w4):
    """Q4 blocks whose quotients w / s are exact half-integers (s = 0.125 exactly), plus the
    +-8 s ends that clamp: codes and scales bit-exact against the oracle (rounding to even)."""
    N, K = 4, 128
    ties = (np.arange(-8, 8) + 0.5) * 0.125                       # 16 exact ties
    w = np.zeros((N, K), dtype=np.float32)
    for n in range(N):
        for b in range(K // 32):
            blk = np.concatenate([ties, ties[::-1]]).astype(np.float32)
            blk[(n + b) % 32] = 1.0 if (n + b) % 2 == 0 else -1.0  # max |w| = 8 s
            w[n, 32 * b:32 * (b + 1)] = blk
    codes, sc = oracle.q4b32_quantize(w)
    gc, gs = w4.q4b32_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(gc.cpu().numpy(), codes)
    assert np.array_equal(bits(gs), sc)


@pytest.mark.parametrize("M,N,K", [(1, 14336, 4096), (3, 1536, 1536), (40, 4096, 1024)])
def test_matmul_host_buffers(w4, M, N, K):
    """w4a16_matmul_host (x and y in pinned host memory, one call) gives the device call's
    bits, with and without the caller's staging buffers."""
    _, codes, s_np, m_np, qw_np = quantized(N, K, seed=M)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    x = workloads.activations_bf16(M, K, seed=M)
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda") if need else None
    y_dev = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws)
    stream = torch.cuda.current_stream()
    xh = x.pin_memory()  # alive until the stream has copied it
    y_host = w4.w4a16_matmul_host(xh, qw, s, m, workspace=ws)
    stream.synchronize()
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    xd = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    yd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    w4.w4a16_matmul_host(xh, qw, s, m, y_host=y2, x_dev=xd, y_dev=yd, workspace=ws)
    stream.synchronize()
    assert torch.equal(y2.view(torch.int16), y_dev.cpu().view(torch.int16))
    with pytest.raises(ValueError, match="host"):
        w4.w4a16_matmul_host(x.cuda(), qw, s, m)
    assert w4.w4a16_device_status() == 0
