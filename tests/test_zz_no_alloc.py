"""The allocation-free matmul entry point, w4a16_matmul_noalloc.

It is meant for callers that may not allocate device memory (its scratch is a fixed
array inside the library). This file is named to be collected last, so that a run that
stops at the first failure has run every other test before it. It passes on its own in a
fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20
W4A16_ERR_WORKSPACE = 6


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemv_w4a16_group_gb300 as w4

    lib = ctypes.CDLL(w4.library_path())
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.w4a16_matmul_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, P]
    lib.w4a16_matmul_noalloc.restype = I
    return w4, lib


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _weights(N, K, seed):
    w = workloads.weights(N, K, seed=seed)
    codes, s, m = oracle.w4a16_quantize(w.numpy())
    qw = oracle.w4a16_pack(codes)
    dev = (torch.from_numpy(qw).cuda(),
           torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).cuda(),
           torch.from_numpy(m.view(np.int16)).view(torch.bfloat16).cuda())
    return (qw, s, m), dev


@pytest.mark.parametrize("M,N,K", [(16, 14336, 4096), (3, 1536, 1536), (40, 256, 1536),
                                   (128, 1536, 1536)])
def test_noalloc_matches_oracle_twice(libs, M, N, K):
    """Two calls in a row through the C ABI: every sampled output within the parity
    tolerance of the oracle, |y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k|, and
    (an extra check) of w4a16_matmul given a workspace."""
    w4, lib = libs
    (qw_np, s_np, m_np), (qw, s, m) = _weights(N, K, seed=M + N + K)
    x_cpu = workloads.activations_bf16(M, K, seed=M)
    x = x_cpu.cuda()
    need = w4.w4a16_matmul_workspace_bytes(M, N, K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda") if need else None
    y_lib = w4.w4a16_matmul(x, qw, s, m, workspace=ws).float().cpu().numpy()
    cols = workloads.sample_indices(N, 256, seed=N).numpy()
    y_ref, abs_ref = oracle.w4a16_matmul(_bits(x_cpu), qw_np, s_np, m_np, cols=cols)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = lib.w4a16_matmul_noalloc(x.data_ptr(), qw.data_ptr(), s.data_ptr(),
                                          m.data_ptr(), y.data_ptr(), M, N, K, 128, stream)
        assert status == 0, status
        torch.cuda.synchronize()
        got = y.float().cpu().numpy()
        assert np.isfinite(got).all()
        a = got[:, cols]
        assert oracle.within_tolerance(a, y_ref, abs_ref).all()
        b = y_lib[:, cols]
        assert np.all(np.abs(a - b) <= 8e-3 * np.abs(b) + 2e-3 * abs_ref)
    assert w4.w4a16_device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(libs):
    """A shape whose split plan needs more than the fixed scratch is refused up front, and
    nothing is launched (y keeps its sentinel)."""
    w4, lib = libs
    K = 4096
    shape = None
    for M in (256, 128, 64):
        for N in range(2048, 19456 + 1, 128):
            if w4.w4a16_matmul_workspace_bytes(M, N, K) > SCRATCH_BYTES:
                shape = (M, N)
                break
        if shape:
            break
    assert shape is not None, "no shape here needs more than the fixed scratch"
    M, N = shape
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros(K // 8, N, dtype=torch.int32, device="cuda")
    s = torch.zeros(K // 128, N, dtype=torch.bfloat16, device="cuda")
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    status = lib.w4a16_matmul_noalloc(x.data_ptr(), qw.data_ptr(), s.data_ptr(), s.data_ptr(),
                                      y.data_ptr(), M, N, K, 128,
                                      torch.cuda.current_stream().cuda_stream)
    assert status == W4A16_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    assert w4.w4a16_device_status() == 0
