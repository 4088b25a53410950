"""W8A16 (symmetric per-row INT8, w_hat = q s) through the C ABI against the oracle.

Quantize must match the oracle bit for bit (codes and fp32 scales); the GEMV must meet
|y - y_ref| <= 4e-3 |y_ref| + 1e-3 sum_k |x_k w_hat_k| on every output, at sizes spanning
several 16-row tiles with a ragged last tile, a K large enough to need the opt-in shared
memory, and the full 14336 x 4096 layer.
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
def w8_variant(request, w4):
    """Run the GEMV test through the tensor-pipe ring kernel (shapes it does not take fall
    back to the plain-load kernel) and through the plain-load kernel."""
    prev = w4.testing_set_w8_variant(request.param)
    yield request.param
    w4.testing_set_w8_variant(prev)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def special_rows(N, K, seed):
    """Seeded N(0, 0.02^2) rows, with a zero row, a row of exact half-integer quotients
    and a row with one outlier 100x the rest."""
    w = workloads.weights(N, K, seed=seed).numpy().copy()
    if N >= 4:
        w[0] = 0.0
        k = np.arange(K)
        w[1] = ((k % 255) - 127 + np.where(k % 3 == 0, 0.5, 0.0)) * 2.0 ** -9
        w[1] = np.clip(w[1], -127 * 2.0 ** -9, 127 * 2.0 ** -9)
        w[1, 0] = 127 * 2.0 ** -9
        w[2, K // 2] = 2.0
    return np.ascontiguousarray(w, dtype=np.float32)


@pytest.mark.parametrize("N,K", [(16, 64), (100, 512), (1000, 4096), (7, 8192)])
def test_w8_quantize_bit_exact(w4, N, K):
    w = special_rows(N, K, seed=N + K)
    q_ref, s_ref = oracle.w8a16_quantize(w)
    q, s = w4.w8a16_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_w8_quantize_hand_worked_rows(w4):
    """The rows of tests/golden/w8a16_rows.txt, each repeated to K = 64."""
    import pins

    recs = pins._records("w8a16_rows.txt")
    w = np.stack([np.tile(pins._weights_from(rec), 8) for _, rec in recs]).astype(np.float32)
    q, s = w4.w8a16_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    q, s = q.cpu().numpy(), s.cpu().numpy()
    for i, (tag, rec) in enumerate(recs):
        assert int(s.view(np.uint32)[i]) == int(rec["scale"][0], 16), tag
        assert q[i, :8].tolist() == [int(v) for v in rec["q"]], tag


# K % 512 == 0 takes the ring kernel: units of T tiles of 16 rows split over P k-parts
# (13, 333: T = 1; 4096: 2; 12008: 6 with a ragged last unit; 28672: 12) and x up to 64 k.
@pytest.mark.parametrize("N,K", [(16, 64), (17, 128), (13, 512), (333, 1024), (1000, 4160),
                                 (4096, 4096), (14336, 4096), (12008, 1536), (28672, 1024),
                                 (64, 65536)])
def test_w8_gemv_every_output(w4, w8_variant, N, K):
    w = special_rows(N, K, seed=N * 3 + K)
    q_np, s_np = oracle.w8a16_quantize(w)
    x = workloads.activations_bf16(1, K, seed=N)[0]
    q, s = torch.from_numpy(q_np).cuda(), torch.from_numpy(s_np).cuda()
    y = w4.w8a16_gemv(x.cuda(), q, s)
    y2 = w4.w8a16_gemv(x.cuda(), q, s)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    y_ref, a_ref = oracle.w8a16_gemv(bits(x), q_np, s_np)
    yv = y.float().cpu().numpy()
    ok = oracle.within_tolerance(yv, y_ref, a_ref)
    if not ok.all():
        bad = np.flatnonzero(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())}/{ok.size} out of tolerance: "
                             f"{[(int(n), float(yv[n]), float(y_ref[n])) for n in bad]}")
    assert yv[0] == 0.0  # the zero row


def test_w8_gemv_special_activations(w4, w8_variant):
    """x with zeros, a 2^20 range of magnitudes inside a chunk, and an all-zero chunk."""
    N, K = 96, 1024
    w = special_rows(N, K, seed=5)
    q_np, s_np = oracle.w8a16_quantize(w)
    x = workloads.activations_bf16(1, K, seed=5)[0].clone()
    x[:64] = 0
    x[64:128] = x[64:128] * torch.logspace(-10, 10, 64, base=2.0).to(torch.bfloat16)
    x[200] = 3.0e4
    y = w4.w8a16_gemv(x.cuda(), torch.from_numpy(q_np).cuda(), torch.from_numpy(s_np).cuda())
    torch.cuda.synchronize()
    y_ref, a_ref = oracle.w8a16_gemv(bits(x), q_np, s_np)
    assert oracle.within_tolerance(y.float().cpu().numpy(), y_ref, a_ref).all()
