"""The prepared (reordered) W4A16 layout on the GPU, through the C ABI: w4a16_prepare bit for
bit against the oracle's permutation, and w4a16_matmul_prepared (the persistent tensor-core
kernel that reads it) within the parity tolerance of the oracle,
|y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k|, per output."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import bits, oracle_matmul_par, quantized, tile_quarter_columns, to_dev_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemv_w4a16_group_gb300 as mod

    return mod


@pytest.fixture
def prepared_from_m(w4):
    """Send every M >= m to the prepared-layout kernel for the duration of a test."""
    prev = []

    def set_min(m):
        prev.append((w4.testing_set_prepared_min_m(m), w4.testing_set_prepared_max_m(1 << 30)))

    yield set_min
    if prev:
        w4.testing_set_prepared_min_m(prev[0][0])
        w4.testing_set_prepared_max_m(prev[0][1])


def _counter_bytes(M, N):
    """Bytes of per-unit arrival counters at the start of the split workspace: one uint32 per
    (128-column tile, batch tile), batch tiles of 16, 32, 64, 128 or 256 rows by M."""
    bn = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
    return 4 * ((N + 127) // 128) * ((M + bn - 1) // bn)


def _check(w4, x, qw_np, s_np, m_np, y, cols=None):
    yv = y.float().cpu().numpy()
    if cols is None:
        cols = np.arange(qw_np.shape[1], dtype=np.int32)
    y_ref, a_ref = oracle_matmul_par(bits(x), qw_np, s_np, m_np, cols)
    yv = yv[:, cols]
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(int(i), int(cols[j]), float(yv[i, j]), float(y_ref[i, j])) for i, j in bad]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} outputs out of tolerance: {detail}")


@pytest.mark.parametrize("N,K", [(8, 128), (136, 256), (256, 512), (1000, 1280), (14336, 4096)])
def test_prepare_bit_exact(w4, N, K):
    """w4a16_prepare writes exactly the oracle's prepared words, padding included."""
    _, codes, s_np, m_np, qw_np = quantized(N, K, seed=N + 3 * K)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    prep = w4.w4a16_prepare(qw, s, m)
    torch.cuda.synchronize()
    ref = oracle.w4a16_prepare(qw_np, s_np, m_np)
    got = prep.cpu().numpy().view(np.uint32)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("with_ws", [True, False])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (3, 136, 384), (8, 520, 256), (16, 384, 1024),
                                   (17, 256, 512), (32, 640, 768), (40, 1536, 1536),
                                   (64, 256, 1536), (100, 392, 512), (128, 256, 512),
                                   (200, 264, 640), (256, 384, 384), (300, 256, 256),
                                   (700, 136, 256)])
def test_matmul_prepared_small_shapes_every_output(w4, prepared_from_m, with_ws, M, N, K):
    """Every batch tile (16..256 rows), ragged N and M, several row tiles, with the stream-K
    split (workspace) and with whole tiles per CTA (none)."""
    prepared_from_m(1)
    _, codes, s_np, m_np, qw_np = quantized(N, K, seed=M * 5 + N)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    prep = w4.w4a16_prepare(qw, s, m)
    x = workloads.activations_bf16(M, K, seed=M + 2 * K)
    ws = None
    if with_ws:
        need = w4.w4a16_matmul_prepared_workspace_bytes(M, N, K)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    y = w4.w4a16_matmul_prepared(x.cuda(), qw, s, m, prep, workspace=ws)
    y2 = w4.w4a16_matmul_prepared(x.cuda(), qw, s, m, prep, workspace=ws)
    torch.cuda.synchronize()
    _check(w4, x, qw_np, s_np, m_np, y)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))  # deterministic split
    if ws is not None:
        assert torch.count_nonzero(ws[:_counter_bytes(M, N)]).item() == 0  # left at zero
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(64, 1536, 8960), (128, 256, 1536), (48, 8960, 1536)])
def test_matmul_prepared_narrow_layers_split_k(w4, M, N, K):
    """Qwen2.5-1.5B-shaped layers at the default range: the narrow ones (few 128-column tiles)
    split K over the SMs through the workspace; sampled outputs within tolerance, same bits
    twice, counters left at zero."""
    _, codes, s_np, m_np, qw_np = quantized(N, K, seed=M + N + K)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    prep = w4.w4a16_prepare(qw, s, m)
    x = workloads.activations_bf16(M, K, seed=K)
    need = w4.w4a16_matmul_prepared_workspace_bytes(M, N, K)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    xd = x.cuda()
    y1 = w4.w4a16_matmul_prepared(xd, qw, s, m, prep, workspace=ws)
    y2 = w4.w4a16_matmul_prepared(xd, qw, s, m, prep, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    cols = workloads.sample_indices(N, 256, seed=N).numpy().astype(np.int32) if N > 256 else None
    _check(w4, x, qw_np, s_np, m_np, y1, cols)
    if ws is not None:
        assert torch.count_nonzero(ws[:_counter_bytes(M, N)]).item() == 0
    assert w4.w4a16_device_status() == 0


_SWEEP = {}


def _sweep():
    if "w" not in _SWEEP:
        cfg = workloads.BATCH_SWEEP
        _SWEEP["w"] = quantized(cfg["N"], cfg["K"], seed=0, outliers=cfg["outlier_frac"])
    return _SWEEP["w"]


@pytest.mark.parametrize("M", [1, 2, 8, 16, 32, 64, 128, 256, 1024, 4096])
def test_matmul_prepared_full_size(w4, prepared_from_m, M):
    """The Llama-3-8B up-projection with 0.1 % outliers x10 through the prepared kernel (forced
    for every M; 112 column tiles, so whole tiles per CTA and no workspace): every output at
    M <= 256, and at M = 1024, 4096 every row of one column in each 32-column quarter of
    every 128-column tile. Two calls give the same bits."""
    prepared_from_m(1)
    cfg = workloads.BATCH_SWEEP
    N, K = cfg["N"], cfg["K"]
    _, codes, s_np, m_np, qw_np = _sweep()
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    prep = w4.w4a16_prepare(qw, s, m)
    x = workloads.activations_bf16(M, K, seed=M)
    need = w4.w4a16_matmul_prepared_workspace_bytes(M, N, K)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    xd = x.cuda()
    y1 = w4.w4a16_matmul_prepared(xd, qw, s, m, prep, workspace=ws)
    y2 = w4.w4a16_matmul_prepared(xd, qw, s, m, prep, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    cols = None if M <= 256 else tile_quarter_columns(N, seed=M)
    _check(w4, x, qw_np, s_np, m_np, y1, cols)
    assert need == 0  # 112 column tiles: whole tiles per CTA, no workspace
    assert w4.w4a16_device_status() == 0


def test_matmul_prepared_guard_bands_and_default_choice(w4):
    """The kernel writes exactly y[M, N] (sentinels around it stay), and at the default
    threshold small M takes the canonical kernels (same bits as w4a16_matmul)."""
    M, N, K = 40, 264, 384
    _, codes, s_np, m_np, qw_np = quantized(N, K, seed=11)
    qw, s, m = to_dev_params(codes, s_np, m_np, qw_np)
    prep = w4.w4a16_prepare(qw, s, m)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    x = workloads.activations_bf16(M, K, seed=1)
    w4.w4a16_matmul_prepared(x.cuda(), qw, s, m, prep, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + M * N:] == 12345)
    _check(w4, x, qw_np, s_np, m_np, y)
    x1 = workloads.activations_bf16(2, K, seed=2).cuda()
    a = w4.w4a16_matmul_prepared(x1, qw, s, m, prep)
    b = w4.w4a16_matmul(x1, qw, s, m)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert w4.w4a16_device_status() == 0
