"""The C-ABI library without a GPU: it loads, exports every function the public headers
declare, and rejects invalid arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("w4a16.h", "w4a16_testing.h")]

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, TIMEOUT, WORKSPACE = range(7)
A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)
B = 0x20000


def _declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\([^;]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib(cuda_lib):
    lib = ctypes.CDLL(cuda_lib)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.w4a16_matmul.argtypes = [P, P, P, P, P, I, I, I, I, P, S, P]
    lib.w4a16_quantize.argtypes = [P, I, I, I, P, P, P, P]
    lib.w4a16_pack.argtypes = [P, I, I, P, P]
    lib.q4b32_quantize.argtypes = [P, I, I, P, P, P]
    lib.q4b32_gemv.argtypes = [P, P, P, P, I, I, P]
    lib.w4a16_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P]
    lib.w4a16_status_string.argtypes = [I]
    lib.w4a16_status_string.restype = ctypes.c_char_p
    lib.w4a16_matmul_workspace_bytes.argtypes = [I, I, I, I]
    lib.w4a16_matmul_workspace_bytes.restype = S
    lib.w4a16zp_quantize.argtypes = [P, I, I, I, P, P, P, P]
    lib.w4a16zp_prepare.argtypes = [P, P, P, I, I, I, P, P, P, P]
    lib.w4a16zp_matmul.argtypes = [P, P, P, P, P, I, I, I, I, P, S, P]
    lib.w8a16_quantize.argtypes = [P, I, I, P, P, P]
    lib.w8a16_gemv.argtypes = [P, P, P, P, I, I, P]
    lib.nvfp4_quantize.argtypes = [P, I, I, P, P, P, P]
    lib.nvfp4_gemv.argtypes = [P, P, P, P, P, I, I, P]
    lib.w4a16_matmul_host.argtypes = [P, P, P, P, P, I, I, I, I, P, P, P, S, P]
    lib.mxfp4_quantize.argtypes = [P, I, I, P, P, P]
    lib.mxfp4_gemv.argtypes = [P, P, P, P, I, I, P]
    lib.w4a16_prepare.argtypes = [P, P, P, I, I, I, P, S, P]
    lib.w4a16_matmul_prepared.argtypes = [P, P, P, P, P, P, I, I, I, I, P, S, P]
    lib.w4a16_prepared_bytes.argtypes = [I, I, I]
    lib.w4a16_prepared_bytes.restype = S
    lib.w4a16_matmul_prepared_workspace_bytes.argtypes = [I, I, I, I]
    lib.w4a16_matmul_prepared_workspace_bytes.restype = S
    lib.nvfp4_matmul.argtypes = [P, P, P, P, P, I, I, I, P, S, P]
    lib.mxfp4_matmul.argtypes = [P, P, P, P, I, I, I, P, S, P]
    lib.fp4_matmul_workspace_bytes.argtypes = [I, I]
    lib.fp4_matmul_workspace_bytes.restype = S
    return lib


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("w4a16_quantize", "w4a16_pack", "w4a16_matmul", "q4b32_gemv",
                     "q4b32_quantize", "w4a16_matmul_workspace_bytes", "w4a16_device_status",
                     "w4a16_status_string", "w4a16zp_quantize", "w4a16zp_prepare",
                     "w4a16zp_matmul", "w8a16_quantize", "w8a16_gemv", "nvfp4_quantize",
                     "nvfp4_gemv", "w4a16_matmul_host", "mxfp4_quantize", "mxfp4_gemv",
                     "w4a16_prepared_bytes", "w4a16_prepare", "w4a16_matmul_prepared",
                     "w4a16_matmul_prepared_workspace_bytes"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    for code, name in enumerate(["W4A16_OK", "W4A16_ERR_INVALID_ARG", "W4A16_ERR_UNSUPPORTED",
                                 "W4A16_ERR_MISALIGNED", "W4A16_ERR_CUDA", "W4A16_ERR_TIMEOUT",
                                 "W4A16_ERR_WORKSPACE", "W4A16_ERR_LAYOUT"]):
        assert lib.w4a16_status_string(code).decode() == name
    assert lib.w4a16_status_string(99).decode() == "W4A16_ERR_UNKNOWN"


def test_matmul_rejects_bad_arguments_on_host(lib):
    m = lib.w4a16_matmul
    good = (A, A, A, A, B)
    assert m(None, A, A, A, B, 1, 256, 512, 128, None, 0, None) == INVALID
    assert m(*good, 0, 256, 512, 128, None, 0, None) == INVALID          # M = 0
    assert m(*good, 1, 0, 512, 128, None, 0, None) == INVALID            # N = 0
    assert m(*good, 1, 256, -128, 128, None, 0, None) == INVALID         # K < 0
    assert m(*good, 1, 256, 500, 128, None, 0, None) == INVALID          # K % group
    assert m(*good, 1, 256, 512, 64, None, 0, None) == UNSUPPORTED       # group 64
    assert m(*good, 1, 260, 512, 128, None, 0, None) == UNSUPPORTED      # N % 8
    assert m(A + 2, A, A, A, B, 1, 256, 512, 128, None, 0, None) == MISALIGNED
    assert m(A, A, A, A, B + 8, 1, 256, 512, 128, None, 0, None) == MISALIGNED
    assert m(*good, 1, 256, 512, 128, A, 0, None) == WORKSPACE           # ptr without size
    assert m(*good, 1, 256, 512, 128, None, 64, None) == WORKSPACE       # size without ptr
    assert m(*good, 1, 256, 512, 128, A + 4, 64, None) == MISALIGNED


def test_quantize_pack_q4_reject_bad_arguments_on_host(lib):
    assert lib.w4a16_quantize(A, 4, 256, 128, None, A, A, None) == INVALID
    assert lib.w4a16_quantize(A, 4, 250, 128, A, A, A, None) == INVALID
    assert lib.w4a16_quantize(A, 4, 256, 32, A, A, A, None) == UNSUPPORTED
    assert lib.w4a16_quantize(A + 4, 4, 256, 128, A, A, A, None) == MISALIGNED
    assert lib.w4a16_pack(A, 4, 12, A, None) == INVALID
    assert lib.w4a16_pack(A, 0, 16, A, None) == INVALID
    assert lib.w4a16_pack(A + 1, 4, 16, A, None) == MISALIGNED
    assert lib.q4b32_quantize(A, 4, 48, A, A, None) == INVALID
    assert lib.q4b32_quantize(A, 4, 64, A, A + 2, None) == MISALIGNED
    assert lib.q4b32_gemv(A, A, A, None, 4, 64, None) == INVALID
    assert lib.q4b32_gemv(A, A, A, B, 4, 40, None) == INVALID
    assert lib.q4b32_gemv(A, A, A + 8, B, 4, 64, None) == MISALIGNED
    assert lib.w4a16_selftest_bounded_wait(0, None) == INVALID
    assert lib.w4a16_selftest_bounded_wait(2_000_000, None) == INVALID


def test_zero_point_entry_points_reject_bad_arguments_on_host(lib):
    q, p, m = lib.w4a16zp_quantize, lib.w4a16zp_prepare, lib.w4a16zp_matmul
    assert q(A, 4, 256, 128, None, A, A, None) == INVALID
    assert q(A, 4, 250, 128, A, A, A, None) == INVALID
    assert q(A, 4, 256, 64, A, A, A, None) == UNSUPPORTED
    assert q(A, 4, 256, 128, A, A + 2, A, None) == MISALIGNED
    assert p(A, A, A, 4, 256, 128, A, A, None, None) == INVALID
    assert p(A, A, A, 0, 256, 128, A, A, A, None) == INVALID
    assert p(A, A, A, 4, 256, 32, A, A, A, None) == UNSUPPORTED
    assert p(A, A, A, 4, 256, 128, A, A + 8, A, None) == MISALIGNED
    good = (A, A, A, A, B)
    assert m(None, A, A, A, B, 1, 256, 512, 128, None, 0, None) == INVALID
    assert m(*good, 1, 256, 500, 128, None, 0, None) == INVALID
    assert m(*good, 1, 260, 512, 128, None, 0, None) == UNSUPPORTED
    assert m(A, A, A, A + 2, B, 1, 256, 512, 128, None, 0, None) == MISALIGNED
    assert m(*good, 1, 256, 512, 128, A, 0, None) == WORKSPACE


def test_w8a16_rejects_bad_arguments_on_host(lib):
    q, g = lib.w8a16_quantize, lib.w8a16_gemv
    assert q(A, 4, 256, None, A, None) == INVALID
    assert q(A, 4, 100, A, A, None) == INVALID          # K % 64
    assert q(A, 0, 256, A, A, None) == INVALID
    assert q(A, 4, 256, A, A + 4, None) == MISALIGNED
    assert g(A, A, A, None, 4, 256, None) == INVALID
    assert g(A, A, A, B, 4, 96, None) == INVALID         # K % 64
    assert g(A, A, A, B, 4, 64 * 4096, None) == UNSUPPORTED  # x does not fit shared memory
    assert g(A + 2, A, A, B, 4, 256, None) == MISALIGNED


def test_nvfp4_rejects_bad_arguments_on_host(lib):
    q, g = lib.nvfp4_quantize, lib.nvfp4_gemv
    assert q(A, 4, 256, A, A, None, None) == INVALID
    assert q(A, 4, 192, A, A, A, None) == INVALID          # K % 128
    assert q(A, 4, 256, A, A, A + 4, None) == MISALIGNED
    assert g(A, A, A, A, None, 4, 256, None) == INVALID
    assert g(A, A, A, A, B, 4, 64, None) == INVALID        # K % 128
    assert g(A, A, A, A, B, 4, 128 * 2048, None) == UNSUPPORTED
    assert g(A, A, A + 1, A, B, 4, 256, None) == MISALIGNED


def test_matmul_host_rejects_bad_arguments_before_copying(lib):
    h = lib.w4a16_matmul_host
    good = (A, A, A, A, B)
    assert h(None, A, A, A, B, 1, 256, 512, 128, A, B, None, 0, None) == INVALID
    assert h(*good, 1, 256, 512, 128, None, B, None, 0, None) == INVALID     # no x_dev
    assert h(*good, 0, 256, 512, 128, A, B, None, 0, None) == INVALID
    assert h(*good, 1, 256, 500, 128, A, B, None, 0, None) == INVALID
    assert h(*good, 1, 260, 512, 128, A, B, None, 0, None) == UNSUPPORTED
    assert h(*good, 1, 256, 512, 128, A + 2, B, None, 0, None) == MISALIGNED
    assert h(*good, 1, 256, 512, 128, A, B, A, 0, None) == WORKSPACE


def test_mxfp4_rejects_bad_arguments_on_host(lib):
    q, g = lib.mxfp4_quantize, lib.mxfp4_gemv
    assert q(A, 4, 256, None, A, None) == INVALID
    assert q(A, 4, 48, A, A, None) == INVALID             # K % 32
    assert q(A, 4, 256, A, A + 4, None) == MISALIGNED
    assert g(A, A, A, None, 4, 256, None) == INVALID
    assert g(A, A, A, B, 4, 96, None) == INVALID          # K % 128
    assert g(A, A, A, B, 4, 128 * 2048, None) == UNSUPPORTED
    assert g(A + 2, A, A, B, 4, 256, None) == MISALIGNED


def test_fp4_matmul_rejects_bad_arguments_on_host(lib):
    """The M > 1 NVFP4 / MXFP4 matmuls: the workspace query (x rows padded to the passes' 8,
    16 or 32, FP16, plus a float per row) and the host-side rejections, before any launch."""
    wb = lib.fp4_matmul_workspace_bytes
    assert wb(1, 512) == 0 and wb(2, 500) == 0
    assert wb(2, 512) == 8 * 512 * 2 + 8 * 4
    assert wb(16, 512) == 16 * 512 * 2 + 16 * 4
    assert wb(40, 512) == 64 * 512 * 2 + 64 * 4
    nv, mx = lib.nvfp4_matmul, lib.mxfp4_matmul
    need = wb(4, 512)
    assert nv(A, A, A, A, B, 4, 8, 512, None, 0, None) == WORKSPACE
    assert nv(A, A, A, A, B, 4, 8, 512, A, need - 16, None) == WORKSPACE
    assert nv(A, A, A, A, B, 4, 8, 512, A + 8, need, None) == MISALIGNED
    assert nv(A, A, A, None, B, 4, 8, 512, A, need, None) == INVALID     # no tensor scale
    assert nv(A, A, A, A, B, 4, 8, 256, A, need, None) == INVALID        # K % 512
    assert nv(A, A, A, A, B, 0, 8, 512, A, need, None) == INVALID
    assert nv(A + 2, A, A, A, B, 4, 8, 512, A, need, None) == MISALIGNED
    assert mx(A, A, A, B, 4, 8, 512, None, 0, None) == WORKSPACE
    assert mx(A, A, None, B, 4, 8, 512, A, need, None) == INVALID
    assert mx(A, A, A, B + 4, 4, 8, 512, A, need, None) == MISALIGNED


def test_prepared_entry_points_reject_bad_arguments_on_host(lib):
    """The prepared layout's size rule (4.25 bits per weight in 128 x 128 records) and the
    host-side checks of w4a16_prepare and w4a16_matmul_prepared."""
    nb = lib.w4a16_prepared_bytes
    assert nb(14336, 4096, 128) == 31_195_136           # the canonical bytes, reordered
    assert nb(136, 256, 128) == 2 * 2 * 8704            # a partial last tile is padded
    assert nb(256, 200, 128) == 0 and nb(256, 256, 64) == 0 and nb(0, 256, 128) == 0
    p = lib.w4a16_prepare
    need = nb(256, 512, 128)
    assert p(A, A, A, 256, 512, 128, None, need, None) == INVALID
    assert p(A, A, A, 256, 500, 128, B, need, None) == INVALID          # K % group
    assert p(A, A, A, 256, 512, 64, B, need, None) == UNSUPPORTED
    assert p(A, A, A, 256, 512, 128, B, need - 16, None) == INVALID     # buffer too small
    assert p(A, A + 4, A, 256, 512, 128, B, need, None) == MISALIGNED
    assert p(A, A, A, 256, 512, 128, B + 8, need, None) == MISALIGNED
    m = lib.w4a16_matmul_prepared
    good = (A, A, A, A, A, B)
    assert m(None, A, A, A, A, B, 64, 256, 512, 128, None, 0, None) == INVALID
    assert m(*good, 64, 256, 500, 128, None, 0, None) == INVALID
    assert m(*good, 64, 260, 512, 128, None, 0, None) == UNSUPPORTED
    assert m(*good, 64, 256, 512, 64, None, 0, None) == UNSUPPORTED
    assert m(A, A, A, A, A + 8, B, 64, 256, 512, 128, None, 0, None) == MISALIGNED
    assert m(*good, 64, 256, 512, 128, A, 0, None) == WORKSPACE
    assert m(*good, 64, 256, 512, 128, A + 4, 64, None) == MISALIGNED
    # below the threshold (and with no prepared copy) it is w4a16_matmul's checks
    assert m(A, A, A, A, None, B, 1, 260, 512, 128, None, 0, None) == UNSUPPORTED


def test_workspace_query_is_host_only(lib):
    assert lib.w4a16_matmul_workspace_bytes(1, 14336, 4096, 128) >= 0


def test_python_binding_refuses_cpu_tensors():
    import torch

    import gemv_w4a16_group_gb300 as w4

    x = torch.zeros(1, 256, dtype=torch.bfloat16)
    qw = torch.zeros(32, 64, dtype=torch.int32)
    s = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.w4a16_matmul(x, qw, s, s)


def test_every_binding_refuses_cpu_tensors():
    """No entry point has a CPU path: each binding rejects host tensors before any call
    (w4a16_matmul_host takes host x and y by design, but its weights must be on the GPU)."""
    import torch

    import gemv_w4a16_group_gb300 as w4

    f32 = torch.zeros(16, 256)
    bf = torch.zeros(256, dtype=torch.bfloat16)
    u8 = torch.zeros(16, 128, dtype=torch.uint8)
    calls = [
        lambda: w4.w4a16zp_quantize(f32),
        lambda: w4.w4a16zp_prepare(torch.zeros(16, 32, dtype=torch.int32),
                                   torch.zeros(16, 2, dtype=torch.float16),
                                   torch.zeros(16, 2, dtype=torch.float16)),
        lambda: w4.w4a16zp_matmul(bf.reshape(1, -1), torch.zeros(32, 16, dtype=torch.int32),
                                  torch.zeros(2, 16, dtype=torch.float16),
                                  torch.zeros(2, 16, dtype=torch.float16)),
        lambda: w4.w8a16_quantize(f32),
        lambda: w4.w8a16_gemv(bf, torch.zeros(16, 256, dtype=torch.int8), torch.zeros(16)),
        lambda: w4.nvfp4_quantize(f32),
        lambda: w4.nvfp4_gemv(bf, u8, torch.zeros(16, 16, dtype=torch.uint8), torch.ones(1)),
        lambda: w4.mxfp4_quantize(f32),
        lambda: w4.mxfp4_gemv(bf, u8, torch.zeros(16, 8, dtype=torch.uint8)),
        lambda: w4.w4a16_matmul_host(bf.reshape(1, -1), torch.zeros(32, 16, dtype=torch.int32),
                                     torch.zeros(2, 16, dtype=torch.bfloat16),
                                     torch.zeros(2, 16, dtype=torch.bfloat16),
                                     x_dev=bf.reshape(1, -1),
                                     y_dev=torch.zeros(1, 16, dtype=torch.bfloat16)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
