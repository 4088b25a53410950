"""Zero-point W4A16 format (w_hat = (q - z) s, FP16 scale and zero point per group of 128)
through the C ABI against the oracle.

The quantizer and the layout move must match the oracle bit for bit; the matmul must meet
|y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k| per output on every kernel (GEMV,
skinny, tcgen05; split K with a workspace) at sizes spanning several tiles with a ragged
tail, and at full size on sampled columns.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

GEMV, TCGEN05, SKINNY = 1, 2, 3


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemv_w4a16_group_gb300 as mod

    return mod


@pytest.fixture
def restore(w4):
    prev = w4.testing_set_skinny_range(-1, -1)
    yield
    w4.testing_force_kernel(0)
    w4.testing_set_skinny_range(*prev)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def special_weights(N, K, seed):
    """Seeded N(0, 0.02^2) weights with rows of special groups: constant groups, groups
    entirely positive or negative (negative or large zero points), groups on the grid with
    exact half-step ties, and a group of exact zeros."""
    w = workloads.weights(N, K, seed=seed).numpy().copy()
    rng = np.random.default_rng(seed)
    G = 128
    if N >= 8 and K >= 2 * G:
        w[0, :G] = 0.3
        w[1, G:2 * G] = 2.6
        w[2, :G] = np.abs(w[2, :G]) + 0.05
        w[3, :G] = -np.abs(w[3, :G]) - 0.05
        w[4, :G] = 0.0
        # on a grid of step 2^-8 with z = 5, plus half steps: ties of w / s
        q = rng.integers(0, 16, size=G)
        q[0], q[1] = 0, 15
        w[5, :G] = (q - 5) * 2.0 ** -8
        w[5, 2:G:3] += 2.0 ** -9
        w[5, 2:G:3] = np.minimum(w[5, 2:G:3], 10 * 2.0 ** -8)
    return np.ascontiguousarray(w, dtype=np.float32)


def dev_page_layout(qw_rows, s, z):
    return (torch.from_numpy(qw_rows.view(np.int32)).cuda(),
            torch.from_numpy(s.view(np.int16)).view(torch.float16).cuda(),
            torch.from_numpy(z.view(np.int16)).view(torch.float16).cuda())


@pytest.mark.parametrize("N,K", [(64, 512), (72, 384), (1000, 1280), (4096, 4096)])
def test_zp_quantize_bit_exact(w4, N, K):
    w = special_weights(N, K, seed=N + K)
    q_ref, s_ref, z_ref = oracle.w4a16zp_quantize(w)
    q, s, z = w4.w4a16zp_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy().view(np.uint32), q_ref)
    np.testing.assert_array_equal(bits(s), s_ref)
    np.testing.assert_array_equal(bits(z), z_ref)


def test_zp_quantize_hand_worked_groups(w4):
    """The six hand-worked groups of tests/golden/w4a16zp_groups.txt, each repeated to a
    group of 128 (repeating values keeps min, max and every quotient)."""
    import pins

    recs = pins._records("w4a16zp_groups.txt")
    rows = [np.tile(pins._weights_from(rec), 16) for _, rec in recs]
    w = np.stack(rows).astype(np.float32)
    q, s, z = w4.w4a16zp_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    words = q.cpu().numpy().view(np.uint32)
    for i, (tag, rec) in enumerate(recs):
        assert int(bits(s)[i, 0]) == int(rec["scale"][0], 16), tag
        assert int(bits(z)[i, 0]) == int(rec["zero"][0], 16), tag
        assert int(words[i, 0]) == int(rec["word"][0], 16), tag
        assert np.all(words[i] == words[i, 0]), tag


@pytest.mark.parametrize("N,K", [(8, 128), (100, 512), (333, 1024), (4096, 4224)])
def test_zp_prepare_is_a_transpose(w4, N, K):
    rng = np.random.default_rng(N)
    qw_rows = rng.integers(0, 2**32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s = rng.integers(0, 2**16, size=(N, K // 128), dtype=np.uint64).astype(np.uint16)
    z = rng.integers(0, 2**16, size=(N, K // 128), dtype=np.uint64).astype(np.uint16)
    qk, sk, zk = oracle.w4a16zp_kernel_layout(qw_rows, s, z)
    q, st, zt = w4.w4a16zp_prepare(*dev_page_layout(qw_rows, s, z))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), qk)
    np.testing.assert_array_equal(bits(st), sk)
    np.testing.assert_array_equal(bits(zt), zk)


def run_and_check(w4, M, N, K, seed, cols=None, workspace=True):
    w = special_weights(N, K, seed)
    qw_rows, s, z = oracle.w4a16zp_quantize(w)
    qw, st, zt = w4.w4a16zp_prepare(*dev_page_layout(qw_rows, s, z))
    x = workloads.activations_bf16(M, K, seed=seed + 7)
    ws = None
    if workspace:
        need = w4.w4a16_matmul_workspace_bytes(M, N, K)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    y = w4.w4a16zp_matmul(x.cuda(), qw, st, zt, workspace=ws)
    y2 = w4.w4a16zp_matmul(x.cuda(), qw, st, zt, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    y_ref, a_ref = oracle.w4a16zp_matmul(bits(x), qw_rows, s, z, cols=cols)
    yv = y.float().cpu().numpy()
    if cols is not None:
        yv = yv[:, cols]
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} out of tolerance, first "
                             f"{[(int(i), int(j), float(yv[i, j]), float(y_ref[i, j])) for i, j in bad]}")
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("kernel", [GEMV, SKINNY, TCGEN05])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (3, 136, 1536), (8, 1000, 1280),
                                   (13, 4872, 640), (32, 4872, 1024), (37, 264, 384),
                                   (200, 1000, 512)])
def test_zp_matmul_every_output(w4, restore, kernel, M, N, K):
    if kernel == SKINNY and M > 32:
        pytest.skip("the skinny kernel takes M <= 32")
    if kernel == SKINNY and N < 32 * 152:
        pytest.skip("the skinny kernel needs at least 32 columns per SM")
    w4.testing_set_skinny_range(1, 32)
    w4.testing_force_kernel(kernel)
    run_and_check(w4, M, N, K, seed=M * 7 + N)


@pytest.mark.parametrize("M", [1, 4, 16, 32, 64, 256])
def test_zp_llama_up_proj_by_m(w4, M):
    """Default kernel choice on the 14336 x 4096 up-projection, sampled columns (first and
    last included)."""
    N, K = workloads.LLAMA_UP["N"], workloads.LLAMA_UP["K"]
    cols = np.unique(np.concatenate([workloads.sample_indices(N, 128, seed=M).numpy(),
                                     [0, 1, N - 2, N - 1]]))
    run_and_check(w4, M, N, K, seed=M, cols=cols)


@pytest.mark.parametrize("M,N,K", [(1, 1536, 8960), (8, 1536, 8960), (2, 4096, 14336),
                                   (64, 1536, 1536)])
def test_zp_split_k(w4, M, N, K):
    """Shapes whose plans split K with a workspace (GEMV and tcgen05 partial sums)."""
    assert w4.w4a16_matmul_workspace_bytes(M, N, K) > 0
    run_and_check(w4, M, N, K, seed=N + M)
