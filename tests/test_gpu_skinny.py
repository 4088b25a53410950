"""Skinny W4A16 kernel (9 <= M <= 32 by default; any M <= 32 when forced) against the oracle.

The kernel takes the batch rows in one to four n8 tiles of mma.sync and needs the caller's
workspace for the converted activations. Shapes cover every column split it plans (2, 3, 4
and 6 quarters of 32 columns per SM) and a ragged last chunk of k.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

SKINNY = 3


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemv_w4a16_group_gb300 as mod

    return mod


@pytest.fixture
def skinny_everywhere(w4):
    """Every M <= 32 may take the skinny kernel; restored afterwards."""
    prev = w4.testing_set_skinny_range(1, 32)
    yield
    w4.testing_set_skinny_range(*prev)
    w4.testing_force_kernel(0)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def quantized(N, K, seed):
    w = workloads.weights(N, K, seed=seed)
    codes, s, m = oracle.w4a16_quantize(w.numpy())
    qw = oracle.w4a16_pack(codes)
    dev = "cuda"
    return (qw, s, m, torch.from_numpy(qw).to(dev),
            torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).to(dev),
            torch.from_numpy(m.view(np.int16)).view(torch.bfloat16).to(dev))


def reserve_bytes(ws_bytes):
    """Leading bytes the skinny kernel never writes (split-K counters live there)."""
    return ((ws_bytes // 128 + 256 + 255) // 256) * 256


# (N, K): columns per SM 8q..8(q+1) -> quarters 2 (N=4872), 3 (14336), 4 (19456), 6 (29184);
# K = 640 (5 groups, one ragged chunk), 4224 (33 groups), 1024, 512.
SHAPES = [(4872, 640), (14336, 4224), (19456, 1024), (29184, 512)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 5, 8, 9, 13, 16, 17, 24, 32])
def test_skinny_matches_oracle(w4, skinny_everywhere, M, N, K):
    w4.testing_force_kernel(SKINNY)
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    assert need > 0
    qw_np, s_np, m_np, qw, s, m = quantized(N, K, seed=M * 31 + N)
    x = workloads.activations_bf16(M, K, seed=M + 3 * K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y1 = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws)
    y2 = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    cols = workloads.sample_indices(N, 96, seed=M).numpy()
    cols = np.unique(np.concatenate([cols, [0, 7, N - 8, N - 1]]))  # first and last columns
    y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np, cols=cols)
    yv = y1.float().cpu().numpy()[:, cols]
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(int(i), int(cols[j]), float(yv[i, j]), float(y_ref[i, j])) for i, j in bad]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} out of tolerance: {detail}")
    # the leading reserve (where split-K counters live) is never written
    assert torch.count_nonzero(ws[:reserve_bytes(need)]).item() == 0
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("M", [5, 8, 9, 16, 32])
def test_skinny_by_m_every_output(w4, M):
    """Default range: 5 <= M <= 32 on the Llama up-projection picks the skinny kernel when
    the workspace holds its plan (two n8 tiles up to M = 16); every output checked."""
    N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    assert need >= (K // 8) * 8 * ((M + 7) // 8) * 16  # at least the converted activations
    qw_np, s_np, m_np, qw, s, m = quantized(N, K, seed=M)
    x = workloads.activations_bf16(M, K, seed=M)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws)
    torch.cuda.synchronize()
    y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np)
    assert oracle.within_tolerance(y.float().cpu().numpy(), y_ref, a_ref).all()
    assert w4.w4a16_device_status() == 0


def test_skinny_without_room_is_rejected_when_forced(w4, skinny_everywhere):
    N, K, M = 14336, 4096, 16
    w4.testing_force_kernel(SKINNY)
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    _, _, _, qw, s, m = quantized(N, K, seed=1)
    x = workloads.activations_bf16(M, K, seed=1).cuda()
    ws = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="W4A16_ERR_WORKSPACE"):
        w4.w4a16_matmul(x, qw, s, m, workspace=ws)
    with pytest.raises(RuntimeError, match="W4A16_ERR_WORKSPACE"):
        w4.w4a16_matmul(x, qw, s, m)


def test_workspace_shared_by_skinny_and_split_k(w4):
    """One buffer, declared with one size, serves skinny calls and split-K calls in turn: a
    skinny call leaves the leading reserve exactly as it found it, and after every call the
    split-K arrival counters (the first 256 bytes for these shapes: at most 64 slabs) are
    zero."""
    shapes = [(16, 14336, 4096), (3, 1536, 1536), (8, 1536, 8960), (16, 14336, 4096),
              (3, 1536, 1536)]
    size = max(w4.w4a16_matmul_workspace_bytes(M, N, K) for M, N, K in shapes)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    reserve = reserve_bytes(size)
    for M, N, K in shapes:
        qw_np, s_np, m_np, qw, s, m = quantized(N, K, seed=M + N)
        x = workloads.activations_bf16(M, K, seed=N)
        before = ws[:reserve].clone()
        y = w4.w4a16_matmul(x.cuda(), qw, s, m, workspace=ws)
        torch.cuda.synchronize()
        cols = workloads.sample_indices(N, 64, seed=M).numpy()
        y_ref, a_ref = oracle.w4a16_matmul(bits(x), qw_np, s_np, m_np, cols=cols)
        assert oracle.within_tolerance(y.float().cpu().numpy()[:, cols], y_ref, a_ref).all()
        if M >= 9:  # the skinny kernel
            assert torch.equal(ws[:reserve], before)
        assert torch.count_nonzero(ws[:256]).item() == 0
    assert w4.w4a16_device_status() == 0
