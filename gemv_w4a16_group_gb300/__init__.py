"""GB300 (sm_103a) W4A16 group-quantized matmul and Q4 block-32 GEMV.

Thin Python binding over the C ABI declared in ``include/w4a16.h``: every function
checks tensor dtypes, shapes and devices, allocates outputs with PyTorch when the caller
passes none, and hands raw device pointers plus the current CUDA stream to the library.
All arithmetic runs in the library's CUDA kernels; there is no CPU fallback, and this
module raises ImportError when the compiled library is missing (build it with
``python -m gemv_w4a16_group_gb300.build``).

Formats ("Low-Precision Kernels: INT4, INT8 and FP8 Matmuls, Measured", Step 2;
"Why My 4-Bit CUDA Kernel Wasn't Faster"):
  * W4A16: codes uint8 [N, K]; packed ``qw`` int32 [K/8, N] (word (r, n) holds k = 8r + j
    in bits 4j..4j+3); ``scales`` and ``mins`` bfloat16 [K/128, N]; x bfloat16 [M, K];
    y bfloat16 [M, N]; w_hat = q * scale + min.
  * Q4 block-32: codes uint8 [N, K/2] (low nibble = even k); scales float16 [N, K/32];
    x float16 [K]; y float16 [N]; w_hat = (q - 8) * scale.
  * W4A16 with a zero point ("Quantization and GEMV", "The quantization formulas"):
    quantized into words int32 [N, K/8] and float16 scales / zeros [N, K/128] (the page's
    layout), moved by ``w4a16zp_prepare`` into qw [K/8, N] and scales / zeros [K/128, N]
    for ``w4a16zp_matmul``; w_hat = (q - zero) * scale.
  * W8A16 (the page's exercise 1): q int8 [N, K]; scales float32 [N]; x bfloat16 [K];
    y bfloat16 [N]; w_hat = q * scale.
  * NVFP4A16 ("Hardware-invariant NVFP4 progress report 1"): codes uint8 [N, K/2] (E2M1,
    low nibble = even k); scales uint8 [N, K/16] (E4M3 bits); tensor_scale float32 [1];
    x bfloat16 [K]; y bfloat16 [N]; w_hat = e2m1(q) * e4m3(scale) * tensor_scale.
  * MXFP4A16 ("Low-Precision Kernels ...", Step 6): codes as NVFP4; scales uint8 [N, K/32]
    (E8M0 bits); w_hat = e2m1(q) * 2^(scale - 127).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

__all__ = [
    "W4A16Error", "library_path", "w4a16_quantize", "w4a16_pack", "w4a16_matmul",
    "w4a16_matmul_workspace_bytes", "w4a16_matmul_noalloc", "w4a16_matmul_host",
    "q4b32_quantize", "q4b32_gemv", "w4a16_device_status",
    "w4a16_selftest_bounded_wait", "testing_force_kernel", "testing_set_gemv_max_m",
    "testing_set_q4_variant", "testing_set_skinny_range", "w4a16zp_quantize",
    "w4a16zp_prepare", "w4a16zp_matmul", "w8a16_quantize", "w8a16_gemv", "nvfp4_quantize",
    "nvfp4_gemv", "mxfp4_quantize", "mxfp4_gemv", "w4a16_prepared_bytes", "w4a16_prepare",
    "w4a16_matmul_prepared", "w4a16_matmul_prepared_workspace_bytes",
    "testing_set_prepared_min_m", "testing_set_prepared_max_m",
    "w4a16_matmul_prepared_uses_prepared", "testing_set_fp4_variant",
    "fp4_matmul_workspace_bytes", "nvfp4_matmul", "mxfp4_matmul", "testing_set_w8_variant",
]

STATUS_NAMES = {0: "W4A16_OK", 1: "W4A16_ERR_INVALID_ARG", 2: "W4A16_ERR_UNSUPPORTED",
                3: "W4A16_ERR_MISALIGNED", 4: "W4A16_ERR_CUDA", 5: "W4A16_ERR_TIMEOUT",
                6: "W4A16_ERR_WORKSPACE", 7: "W4A16_ERR_LAYOUT"}


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def library_path() -> str:
    return LIB_PATH


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"the GB300 kernel library is not built ({LIB_PATH} missing); run "
            "`python -m gemv_w4a16_group_gb300.build` on a machine with nvcc")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S, U32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint32
    sigs = {
        "w4a16_quantize": [P, I, I, I, P, P, P, P],
        "w4a16_pack": [P, I, I, P, P],
        "w4a16_matmul": [P, P, P, P, P, I, I, I, I, P, S, P],
        "w4a16_matmul_noalloc": [P, P, P, P, P, I, I, I, I, P],
        "w4a16_matmul_host": [P, P, P, P, P, I, I, I, I, P, P, P, S, P],
        "q4b32_quantize": [P, I, I, P, P, P],
        "q4b32_gemv": [P, P, P, P, I, I, P],
        "w4a16_device_status": [P],
        "w4a16_selftest_bounded_wait": [U32, P],
        "w4a16zp_quantize": [P, I, I, I, P, P, P, P],
        "w4a16zp_prepare": [P, P, P, I, I, I, P, P, P, P],
        "w4a16zp_matmul": [P, P, P, P, P, I, I, I, I, P, S, P],
        "w8a16_quantize": [P, I, I, P, P, P],
        "w8a16_gemv": [P, P, P, P, I, I, P],
        "nvfp4_quantize": [P, I, I, P, P, P, P],
        "nvfp4_gemv": [P, P, P, P, P, I, I, P],
        "mxfp4_quantize": [P, I, I, P, P, P],
        "mxfp4_gemv": [P, P, P, P, I, I, P],
        "nvfp4_matmul": [P, P, P, P, P, I, I, I, P, S, P],
        "mxfp4_matmul": [P, P, P, P, I, I, I, P, S, P],
        "w4a16_prepare": [P, P, P, I, I, I, P, S, P],
        "w4a16_matmul_prepared": [P, P, P, P, P, P, I, I, I, I, P, S, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    for name in ("w4a16_matmul_workspace_bytes", "w4a16_matmul_prepared_workspace_bytes"):
        getattr(lib, name).argtypes = [I, I, I, I]
        getattr(lib, name).restype = S
    lib.w4a16_prepared_bytes.argtypes = [I, I, I]
    lib.w4a16_prepared_bytes.restype = S
    lib.fp4_matmul_workspace_bytes.argtypes = [I, I]
    lib.fp4_matmul_workspace_bytes.restype = S
    lib.w4a16_status_string.argtypes = [I]
    lib.w4a16_status_string.restype = ctypes.c_char_p
    for name in ("w4a16_testing_force_kernel", "w4a16_testing_set_gemv_max_m",
                 "w4a16_testing_set_q4_variant", "w4a16_testing_set_prepared_min_m",
                 "w4a16_testing_set_prepared_max_m", "w4a16_testing_set_fp4_variant",
                 "w4a16_testing_set_w8_variant"):
        getattr(lib, name).argtypes = [I]
        getattr(lib, name).restype = I
    lib.w4a16_testing_set_skinny_range.argtypes = [I, I]
    lib.w4a16_testing_set_skinny_range.restype = I
    return lib


_lib = _load()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _check(name: str, status: int):
    if status != 0:
        raise W4A16Error(name, status)


def w4a16_quantize(w: torch.Tensor, group: int = 128, codes=None, scales=None, mins=None,
                   stream=None):
    """fp32 [N, K] -> (codes uint8 [N, K], scales bf16 [K/group, N], mins bf16 [K/group, N])."""
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((K // group, N), dtype=torch.bfloat16, device=w.device)
    if mins is None:
        mins = torch.empty((K // group, N), dtype=torch.bfloat16, device=w.device)
    _check("w4a16_quantize", _lib.w4a16_quantize(
        _dev(w, "w", torch.float32), N, K, group, _dev(codes, "codes", torch.uint8, (N, K)),
        _dev(scales, "scales", torch.bfloat16, (K // group, N)),
        _dev(mins, "mins", torch.bfloat16, (K // group, N)), _stream(stream)))
    return codes, scales, mins


def w4a16_pack(codes: torch.Tensor, qw=None, stream=None) -> torch.Tensor:
    """uint8 codes [N, K] -> int32 [K/8, N]."""
    N, K = codes.shape
    if qw is None:
        qw = torch.empty((K // 8, N), dtype=torch.int32, device=codes.device)
    _check("w4a16_pack", _lib.w4a16_pack(_dev(codes, "codes", torch.uint8), N, K,
                                         _dev(qw, "qw", torch.int32, (K // 8, N)),
                                         _stream(stream)))
    return qw


def w4a16_matmul_workspace_bytes(M: int, N: int, K: int, group: int = 128) -> int:
    return int(_lib.w4a16_matmul_workspace_bytes(M, N, K, group))


def w4a16_matmul(x: torch.Tensor, qw: torch.Tensor, scales: torch.Tensor, mins: torch.Tensor,
                 group: int = 128, y=None, workspace=None, stream=None) -> torch.Tensor:
    """y [M, N] (bf16) = x [M, K] (bf16) . w_hat^T."""
    M, K = x.shape
    N = qw.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check("w4a16_matmul", _lib.w4a16_matmul(
        _dev(x, "x", torch.bfloat16), _dev(qw, "qw", torch.int32, (K // 8, N)),
        _dev(scales, "scales", torch.bfloat16, (K // group, N)),
        _dev(mins, "mins", torch.bfloat16, (K // group, N)),
        _dev(y, "y", torch.bfloat16, (M, N)), M, N, K, group, ws_ptr, ws_bytes, _stream(stream)))
    return y


def _workspace(workspace):
    if workspace is None:
        return None, 0
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def w4a16_prepared_bytes(N: int, K: int, group: int = 128) -> int:
    """Bytes of the prepared (reordered) copy of an N x K weight matrix."""
    return int(_lib.w4a16_prepared_bytes(N, K, group))


def w4a16_prepare(qw: torch.Tensor, scales: torch.Tensor, mins: torch.Tensor, group: int = 128,
                  prepared=None, stream=None) -> torch.Tensor:
    """Packed weights (qw int32 [K/8, N], scales / mins bf16 [K/group, N]) -> the prepared
    copy, uint8 [w4a16_prepared_bytes(N, K)] (records of 128 columns x 128 k; see
    include/w4a16.h)."""
    N = qw.shape[1]
    K = qw.shape[0] * 8
    nbytes = w4a16_prepared_bytes(N, K, group)
    if prepared is None:
        prepared = torch.empty(nbytes, dtype=torch.uint8, device=qw.device)
    if not (isinstance(prepared, torch.Tensor) and prepared.is_cuda and prepared.is_contiguous()):
        raise ValueError("prepared must be a contiguous CUDA tensor")
    _check("w4a16_prepare", _lib.w4a16_prepare(
        _dev(qw, "qw", torch.int32, (K // 8, N)),
        _dev(scales, "scales", torch.bfloat16, (K // group, N)),
        _dev(mins, "mins", torch.bfloat16, (K // group, N)), N, K, group, prepared.data_ptr(),
        prepared.numel() * prepared.element_size(), _stream(stream)))
    return prepared


def w4a16_matmul_prepared_workspace_bytes(M: int, N: int, K: int, group: int = 128) -> int:
    return int(_lib.w4a16_matmul_prepared_workspace_bytes(M, N, K, group))


def w4a16_matmul_prepared(x: torch.Tensor, qw: torch.Tensor, scales: torch.Tensor,
                          mins: torch.Tensor, prepared, group: int = 128, y=None,
                          workspace=None, stream=None) -> torch.Tensor:
    """y [M, N] (bf16) = x [M, K] (bf16) . w_hat^T, reading the prepared copy of the weights
    (from w4a16_prepare) at the batch sizes where the prepared-layout kernel runs, and
    (qw, scales, mins) below them."""
    M, K = x.shape
    N = qw.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    p_prep = None
    if prepared is not None:
        if not (isinstance(prepared, torch.Tensor) and prepared.is_cuda and prepared.is_contiguous()):
            raise ValueError("prepared must be a contiguous CUDA tensor")
        if prepared.numel() * prepared.element_size() < w4a16_prepared_bytes(N, K, group):
            raise ValueError("prepared is smaller than w4a16_prepared_bytes(N, K)")
        p_prep = prepared.data_ptr()
    ws_ptr, ws_bytes = _workspace(workspace)
    _check("w4a16_matmul_prepared", _lib.w4a16_matmul_prepared(
        _dev(x, "x", torch.bfloat16), _dev(qw, "qw", torch.int32, (K // 8, N)),
        _dev(scales, "scales", torch.bfloat16, (K // group, N)),
        _dev(mins, "mins", torch.bfloat16, (K // group, N)), p_prep,
        _dev(y, "y", torch.bfloat16, (M, N)), M, N, K, group, ws_ptr, ws_bytes, _stream(stream)))
    return y


def w4a16_matmul_prepared_uses_prepared(M: int) -> bool:
    """Whether w4a16_matmul_prepared runs the prepared-layout kernel at this M (else it is
    w4a16_matmul on the canonical arrays)."""
    lo = int(_lib.w4a16_testing_set_prepared_min_m(0))
    hi = int(_lib.w4a16_testing_set_prepared_max_m(0))
    return lo <= M <= hi


def testing_set_prepared_min_m(m: int) -> int:
    """Smallest M that w4a16_matmul_prepared sends to the prepared-layout kernel; returns the
    previous value (m < 1 only queries)."""
    return int(_lib.w4a16_testing_set_prepared_min_m(m))


def testing_set_prepared_max_m(m: int) -> int:
    """Largest M that w4a16_matmul_prepared sends to the prepared-layout kernel; returns the
    previous value (m < 1 only queries)."""
    return int(_lib.w4a16_testing_set_prepared_max_m(m))


def w4a16_matmul_host(x_host: torch.Tensor, qw: torch.Tensor, scales: torch.Tensor,
                      mins: torch.Tensor, y_host=None, x_dev=None, y_dev=None, group: int = 128,
                      workspace=None, stream=None) -> torch.Tensor:
    """y_host [M, N] (bf16, host) = x_host [M, K] (bf16, host) . w_hat^T: one library call that
    enqueues the copy of x, the matmul and the copy of y on the stream and returns; synchronize
    the stream before reading y_host, and keep x_host alive until then. Pass page-locked host
    tensors (``pin_memory()``) and the device staging buffers x_dev, y_dev to avoid any
    allocation per call; with a raw stream handle, pass the staging buffers too."""
    if not isinstance(x_host, torch.Tensor) or x_host.is_cuda:
        raise ValueError("x_host must be a host (CPU) tensor")
    if x_host.dtype != torch.bfloat16 or not x_host.is_contiguous():
        raise TypeError("x_host must be a contiguous bfloat16 tensor")
    M, K = x_host.shape
    N = qw.shape[1]
    dev = qw.device
    p_qw = _dev(qw, "qw", torch.int32, (K // 8, N))
    p_s = _dev(scales, "scales", torch.bfloat16, (K // group, N))
    p_m = _dev(mins, "mins", torch.bfloat16, (K // group, N))
    if y_host is None:
        y_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    if y_host.is_cuda or y_host.dtype != torch.bfloat16 or tuple(y_host.shape) != (M, N) \
            or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous host bfloat16 tensor of shape (M, N)")
    if x_dev is None or y_dev is None:
        # staging allocated on the stream the copies run on (the caching allocator reuses a
        # freed block only in that stream's order)
        on = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.current_stream(dev)
        with torch.cuda.stream(on):
            if x_dev is None:
                x_dev = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            if y_dev is None:
                y_dev = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check("w4a16_matmul_host", _lib.w4a16_matmul_host(
        x_host.data_ptr(), p_qw, p_s, p_m, y_host.data_ptr(), M, N, K, group,
        _dev(x_dev, "x_dev", torch.bfloat16, (M, K)), _dev(y_dev, "y_dev", torch.bfloat16, (M, N)),
        ws_ptr, ws_bytes, _stream(stream)))
    return y_host


def w4a16_matmul_noalloc(x: torch.Tensor, qw: torch.Tensor, scales: torch.Tensor,
                         mins: torch.Tensor, y: torch.Tensor, group: int = 128,
                         stream=None) -> torch.Tensor:
    """y = x . w_hat^T without any allocation by the library or this function: the
    caller passes y. For callers that cannot allocate device memory; the scratch is a
    fixed 16 MiB array inside the library, shared by every call on the device, so calls
    that may overlap on the GPU must be ordered. Make the first call on a device before
    any stream capture."""
    M, K = x.shape
    N = qw.shape[1]
    _check("w4a16_matmul_noalloc", _lib.w4a16_matmul_noalloc(
        _dev(x, "x", torch.bfloat16), _dev(qw, "qw", torch.int32, (K // 8, N)),
        _dev(scales, "scales", torch.bfloat16, (K // group, N)),
        _dev(mins, "mins", torch.bfloat16, (K // group, N)),
        _dev(y, "y", torch.bfloat16, (M, N)), M, N, K, group, _stream(stream)))
    return y


def w4a16zp_quantize(w: torch.Tensor, group: int = 128, qw_rows=None, scales=None, zeros=None,
                     stream=None):
    """fp32 [N, K] -> (words int32 [N, K/8], scales fp16 [N, K/group], zeros fp16
    [N, K/group]), the zero-point format in the layout its page stores."""
    N, K = w.shape
    if qw_rows is None:
        qw_rows = torch.empty((N, K // 8), dtype=torch.int32, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // group), dtype=torch.float16, device=w.device)
    if zeros is None:
        zeros = torch.empty((N, K // group), dtype=torch.float16, device=w.device)
    _check("w4a16zp_quantize", _lib.w4a16zp_quantize(
        _dev(w, "w", torch.float32), N, K, group,
        _dev(qw_rows, "qw_rows", torch.int32, (N, K // 8)),
        _dev(scales, "scales", torch.float16, (N, K // group)),
        _dev(zeros, "zeros", torch.float16, (N, K // group)), _stream(stream)))
    return qw_rows, scales, zeros


def w4a16zp_prepare(qw_rows: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                    group: int = 128, qw=None, scales_t=None, zeros_t=None, stream=None):
    """Words [N, K/8] and scales / zeros [N, K/group] -> the matmul's qw int32 [K/8, N] and
    scales / zeros fp16 [K/group, N]."""
    N, K = qw_rows.shape[0], qw_rows.shape[1] * 8
    dev = qw_rows.device
    if qw is None:
        qw = torch.empty((K // 8, N), dtype=torch.int32, device=dev)
    if scales_t is None:
        scales_t = torch.empty((K // group, N), dtype=torch.float16, device=dev)
    if zeros_t is None:
        zeros_t = torch.empty((K // group, N), dtype=torch.float16, device=dev)
    _check("w4a16zp_prepare", _lib.w4a16zp_prepare(
        _dev(qw_rows, "qw_rows", torch.int32, (N, K // 8)),
        _dev(scales, "scales", torch.float16, (N, K // group)),
        _dev(zeros, "zeros", torch.float16, (N, K // group)), N, K, group,
        _dev(qw, "qw", torch.int32, (K // 8, N)),
        _dev(scales_t, "scales_t", torch.float16, (K // group, N)),
        _dev(zeros_t, "zeros_t", torch.float16, (K // group, N)), _stream(stream)))
    return qw, scales_t, zeros_t


def w4a16zp_matmul(x: torch.Tensor, qw: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                   group: int = 128, y=None, workspace=None, stream=None) -> torch.Tensor:
    """y [M, N] (bf16) = x [M, K] (bf16) . w_hat^T, w_hat = (q - zero) * scale; qw, scales
    and zeros as ``w4a16zp_prepare`` returns them. Workspace as for ``w4a16_matmul``."""
    M, K = x.shape
    N = qw.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check("w4a16zp_matmul", _lib.w4a16zp_matmul(
        _dev(x, "x", torch.bfloat16), _dev(qw, "qw", torch.int32, (K // 8, N)),
        _dev(scales, "scales", torch.float16, (K // group, N)),
        _dev(zeros, "zeros", torch.float16, (K // group, N)),
        _dev(y, "y", torch.bfloat16, (M, N)), M, N, K, group, ws_ptr, ws_bytes, _stream(stream)))
    return y


def w8a16_quantize(w: torch.Tensor, q=None, scales=None, stream=None):
    """fp32 [N, K] -> (q int8 [N, K], scales fp32 [N])."""
    N, K = w.shape
    if q is None:
        q = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if scales is None:
        scales = torch.empty((N,), dtype=torch.float32, device=w.device)
    _check("w8a16_quantize", _lib.w8a16_quantize(
        _dev(w, "w", torch.float32), N, K, _dev(q, "q", torch.int8, (N, K)),
        _dev(scales, "scales", torch.float32, (N,)), _stream(stream)))
    return q, scales


def w8a16_gemv(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, y=None,
               stream=None) -> torch.Tensor:
    """y [N] (bf16) = (q * scales[:, None]) . x, x bf16 [K]."""
    N, K = q.shape
    if y is None:
        y = torch.empty((N,), dtype=torch.bfloat16, device=x.device)
    _check("w8a16_gemv", _lib.w8a16_gemv(
        _dev(x, "x", torch.bfloat16, (K,)), _dev(q, "q", torch.int8, (N, K)),
        _dev(scales, "scales", torch.float32, (N,)), _dev(y, "y", torch.bfloat16, (N,)), N, K,
        _stream(stream)))
    return y


def nvfp4_quantize(w: torch.Tensor, codes=None, scales=None, tensor_scale=None, stream=None):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales uint8 E4M3 [N, K/16], tensor_scale
    float32 [1])."""
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    if tensor_scale is None:
        tensor_scale = torch.empty((1,), dtype=torch.float32, device=w.device)
    _check("nvfp4_quantize", _lib.nvfp4_quantize(
        _dev(w, "w", torch.float32), N, K, _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.uint8, (N, K // 16)),
        _dev(tensor_scale, "tensor_scale", torch.float32, (1,)), _stream(stream)))
    return codes, scales, tensor_scale


def nvfp4_gemv(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
               tensor_scale: torch.Tensor, y=None, stream=None) -> torch.Tensor:
    """y [N] (bf16) = W_hat . x, x bf16 [K]."""
    N, K = codes.shape[0], codes.shape[1] * 2
    if y is None:
        y = torch.empty((N,), dtype=torch.bfloat16, device=x.device)
    _check("nvfp4_gemv", _lib.nvfp4_gemv(
        _dev(x, "x", torch.bfloat16, (K,)), _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.uint8, (N, K // 16)),
        _dev(tensor_scale, "tensor_scale", torch.float32, (1,)),
        _dev(y, "y", torch.bfloat16, (N,)), N, K, _stream(stream)))
    return y


def fp4_matmul_workspace_bytes(M: int, K: int) -> int:
    """Workspace bytes nvfp4_matmul / mxfp4_matmul need for M rows of x (0 for M = 1)."""
    return int(_lib.fp4_matmul_workspace_bytes(M, K))


def _fp4_matmul_args(name, x, codes, y, workspace):
    N, K = codes.shape[0], codes.shape[1] * 2
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None and M > 1:
        workspace = torch.empty(max(fp4_matmul_workspace_bytes(M, K), 16), dtype=torch.uint8,
                                device=x.device)
    ws, ws_bytes = _workspace(workspace)
    return M, N, K, y, ws, ws_bytes


def nvfp4_matmul(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                 tensor_scale: torch.Tensor, y=None, workspace=None, stream=None) -> torch.Tensor:
    """y [M, N] (bf16) = x . W_hat^T, x bf16 [M, K]; a workspace of
    fp4_matmul_workspace_bytes(M, K) bytes is allocated when none is given."""
    M, N, K, y, ws, ws_bytes = _fp4_matmul_args("nvfp4_matmul", x, codes, y, workspace)
    _check("nvfp4_matmul", _lib.nvfp4_matmul(
        _dev(x, "x", torch.bfloat16, (M, K)), _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.uint8, (N, K // 16)),
        _dev(tensor_scale, "tensor_scale", torch.float32, (1,)),
        _dev(y, "y", torch.bfloat16, (M, N)), M, N, K, ws, ws_bytes, _stream(stream)))
    return y


def mxfp4_matmul(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y=None,
                 workspace=None, stream=None) -> torch.Tensor:
    """y [M, N] (bf16) = x . W_hat^T, x bf16 [M, K]; a workspace of
    fp4_matmul_workspace_bytes(M, K) bytes is allocated when none is given."""
    M, N, K, y, ws, ws_bytes = _fp4_matmul_args("mxfp4_matmul", x, codes, y, workspace)
    _check("mxfp4_matmul", _lib.mxfp4_matmul(
        _dev(x, "x", torch.bfloat16, (M, K)), _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.uint8, (N, K // 32)), _dev(y, "y", torch.bfloat16, (M, N)),
        M, N, K, ws, ws_bytes, _stream(stream)))
    return y


def mxfp4_quantize(w: torch.Tensor, codes=None, scales=None, stream=None):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales uint8 E8M0 [N, K/32])."""
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 32), dtype=torch.uint8, device=w.device)
    _check("mxfp4_quantize", _lib.mxfp4_quantize(
        _dev(w, "w", torch.float32), N, K, _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.uint8, (N, K // 32)), _stream(stream)))
    return codes, scales


def mxfp4_gemv(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y=None,
               stream=None) -> torch.Tensor:
    """y [N] (bf16) = W_hat . x, x bf16 [K]."""
    N, K = codes.shape[0], codes.shape[1] * 2
    if y is None:
        y = torch.empty((N,), dtype=torch.bfloat16, device=x.device)
    _check("mxfp4_gemv", _lib.mxfp4_gemv(
        _dev(x, "x", torch.bfloat16, (K,)), _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.uint8, (N, K // 32)), _dev(y, "y", torch.bfloat16, (N,)),
        N, K, _stream(stream)))
    return y


def q4b32_quantize(w: torch.Tensor, codes=None, scales=None, stream=None):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales fp16 [N, K/32])."""
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 32), dtype=torch.float16, device=w.device)
    _check("q4b32_quantize", _lib.q4b32_quantize(
        _dev(w, "w", torch.float32), N, K, _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.float16, (N, K // 32)), _stream(stream)))
    return codes, scales


def q4b32_gemv(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y=None,
               stream=None) -> torch.Tensor:
    """y [N] (fp16) = W_hat [N, K] . x [K] (fp16)."""
    N = codes.shape[0]
    K = codes.shape[1] * 2
    if y is None:
        y = torch.empty((N,), dtype=torch.float16, device=x.device)
    _check("q4b32_gemv", _lib.q4b32_gemv(
        _dev(x, "x", torch.float16, (K,)), _dev(codes, "codes", torch.uint8, (N, K // 2)),
        _dev(scales, "scales", torch.float16, (N, K // 32)), _dev(y, "y", torch.float16, (N,)),
        N, K, _stream(stream)))
    return y


def w4a16_device_status(stream=None) -> int:
    """Synchronize and return (and clear) the device status (0 = OK, 5 = a wait expired)."""
    return int(_lib.w4a16_device_status(_stream(stream)))


def w4a16_selftest_bounded_wait(limit_us: int, stream=None) -> int:
    return int(_lib.w4a16_selftest_bounded_wait(limit_us, _stream(stream)))


def testing_force_kernel(kernel: int) -> int:
    """0 = by M, 1 = the small-M GEMV kernel, 2 = the tcgen05 tensor-core kernel, 3 = the
    skinny kernel (M <= 32, needs the workspace reported for an M in the skinny range)."""
    return int(_lib.w4a16_testing_force_kernel(kernel))


def testing_set_gemv_max_m(m: int) -> int:
    return int(_lib.w4a16_testing_set_gemv_max_m(m))


def testing_set_skinny_range(lo: int, hi: int):
    """Range of M sent to the skinny kernel by the by-M choice; negative values only query.
    Returns the previous (lo, hi)."""
    prev = int(_lib.w4a16_testing_set_skinny_range(lo, hi))
    return prev >> 8, prev & 0xFF


def testing_set_q4_variant(v: int) -> int:
    return int(_lib.w4a16_testing_set_q4_variant(v))


def testing_set_w8_variant(v: int) -> int:
    """Kernel of w8a16_gemv: 1 = tensor-pipe ring (default), 0 = plain loads; other values
    only query. Returns the previous value."""
    return int(_lib.w4a16_testing_set_w8_variant(v))


def testing_set_fp4_variant(v: int) -> int:
    """Kernel of nvfp4_gemv / mxfp4_gemv: 1 = tensor-pipe ring (default), 0 = plain loads;
    other values only query. Returns the previous value."""
    return int(_lib.w4a16_testing_set_fp4_variant(v))
