"""CPU oracle for the W4A16 group-quantized matmul and the Q4 block-32 GEMV.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package; the library under ``gemv_w4a16_group_gb300`` never does, and this
package never imports it. The arithmetic lives in ``w4a16_oracle.c`` (plain
scalar C, fp32 steps where the format fixes them, fp64 sums); this module only
compiles it, loads it with ctypes and marshals numpy arrays.

Array conventions (all numpy, C-contiguous):
  * BF16 / FP16 values are carried as their ``uint16`` bit patterns.
  * W4A16: ``w`` fp32 [N, K]; ``codes`` uint8 [N, K]; ``scales``/``mins`` bf16
    bits [K/G, N]; ``qw`` int32 [K/8, N]; ``x`` bf16 bits [M, K].
  * Q4 block-32: ``codes`` uint8 [N, K/2]; ``scales`` fp16 bits [N, K/32];
    ``x`` fp16 bits [K].
  * W4A16 with a zero point: ``qw_rows`` uint32 [N, K/8]; ``scales``/``zeros``
    fp16 bits [N, K/G] (the layout the format's page stores); w_hat = (q - z) s.
  * W8A16: ``q`` int8 [N, K]; ``s`` fp32 [N] (one per row); ``x`` bf16 bits [K];
    w_hat = q s.
  * NVFP4A16: ``codes`` uint8 [N, K/2] (E2M1, low nibble = even k); ``scales`` uint8
    E4M3 [N, K/16]; ``S`` one fp32; ``x`` bf16 bits [K]; w_hat = e2m1 e4m3 S.
  * MXFP4A16: ``codes`` as NVFP4; ``scales`` uint8 E8M0 [N, K/32]; w_hat = e2m1 2^(s - 127).
  * The NVFP4A16 / MXFP4A16 matmuls take ``x`` bf16 bits [M, K] and return [M, N] (or
    [M, len(rows)]): Y[m] = W_hat . x[m], the GEMV of each row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# No FMA contraction, no fast-math: every fp32 step is one IEEE operation.
CFLAGS = ["-O1", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_to(src_path: str, out_path: str) -> str:
    """Compile an oracle source file (used by the mutation tests) to a shared library."""
    subprocess.check_call(["gcc", *CFLAGS, src_path, "-o", out_path, "-lm"])
    return out_path


_lib = None
_override = None


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_fp16_rne.argtypes = [ctypes.c_float]
    lib.oracle_fp16_rne.restype = ctypes.c_uint16
    lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_float.restype = ctypes.c_float
    lib.oracle_fp16_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_float.restype = ctypes.c_float
    L = ctypes.c_long
    lib.oracle_bf16_rne_array.argtypes = [P, P, L]
    lib.oracle_fp16_rne_array.argtypes = [P, P, L]
    lib.oracle_fp16_to_float_array.argtypes = [P, P, L]
    lib.oracle_w4a16_quantize.argtypes = [P, I, I, I, P, P, P]
    lib.oracle_w4a16_pack.argtypes = [P, I, I, P]
    lib.oracle_w4a16_dequant.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_w4a16_matmul.argtypes = [P, P, P, P, I, I, I, I, P, P]
    lib.oracle_w4a16_matmul_cols.argtypes = [P, P, P, P, I, I, I, I, P, I, P, P]
    lib.oracle_w4a16_prepared_words.argtypes = [I, I, I]
    lib.oracle_w4a16_prepared_words.restype = ctypes.c_long
    lib.oracle_w4a16_prepare.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_q4b32_quantize.argtypes = [P, I, I, P, P]
    lib.oracle_q4b32_dequant.argtypes = [P, P, I, I, P]
    lib.oracle_q4b32_gemv.argtypes = [P, P, P, I, I, P, I, P, P]
    lib.oracle_w4a16zp_quantize.argtypes = [P, I, I, I, P, P, P]
    lib.oracle_w4a16zp_dequant.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_w4a16zp_matmul.argtypes = [P, P, P, P, I, I, I, I, P, I, P, P]
    lib.oracle_w8a16_quantize.argtypes = [P, I, I, P, P]
    lib.oracle_w8a16_gemv.argtypes = [P, P, P, I, I, P, I, P, P]
    F = ctypes.c_float
    lib.oracle_e2m1_value.argtypes = [I]
    lib.oracle_e2m1_value.restype = ctypes.c_double
    lib.oracle_e4m3_value.argtypes = [I]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e2m1_rne.argtypes = [F]
    lib.oracle_e2m1_rne.restype = I
    lib.oracle_e4m3_ceil.argtypes = [F]
    lib.oracle_e4m3_ceil.restype = I
    lib.oracle_nvfp4_quantize.argtypes = [P, I, I, P, P, P]
    lib.oracle_nvfp4_dequant.argtypes = [P, P, F, I, I, P]
    lib.oracle_nvfp4_gemv.argtypes = [P, P, P, F, I, I, P, I, P, P]
    lib.oracle_e8m0_value.argtypes = [I]
    lib.oracle_e8m0_value.restype = ctypes.c_double
    lib.oracle_mxfp4_quantize.argtypes = [P, I, I, P, P]
    lib.oracle_mxfp4_dequant.argtypes = [P, P, I, I, P]
    lib.oracle_mxfp4_gemv.argtypes = [P, P, P, I, I, P, I, P, P]
    for name in ("oracle_bf16_rne_array", "oracle_fp16_rne_array", "oracle_fp16_to_float_array",
                 "oracle_w4a16_quantize", "oracle_w4a16_pack", "oracle_w4a16_dequant",
                 "oracle_w4a16_matmul", "oracle_w4a16_matmul_cols", "oracle_w4a16_prepare",
                 "oracle_q4b32_quantize",
                 "oracle_q4b32_dequant", "oracle_q4b32_gemv", "oracle_w4a16zp_quantize",
                 "oracle_w4a16zp_dequant", "oracle_w4a16zp_matmul", "oracle_w8a16_quantize",
                 "oracle_w8a16_gemv", "oracle_nvfp4_quantize", "oracle_nvfp4_dequant",
                 "oracle_nvfp4_gemv", "oracle_mxfp4_quantize", "oracle_mxfp4_dequant",
                 "oracle_mxfp4_gemv"):
        getattr(lib, name).restype = None
    return lib


def _load():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager: route every oracle call to another compiled build of the
    oracle source (the mutation tests plant one mistake per build)."""

    def __init__(self, path: str):
        self.lib = _bind(ctypes.CDLL(path))

    def __enter__(self):
        global _override
        self._prev = _override
        _override = self.lib
        return self

    def __exit__(self, *exc):
        global _override
        _override = self._prev
        return False


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- #
# IEEE helpers
# --------------------------------------------------------------------------- #

def bf16_rne(values) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (element-wise, same shape)."""
    arr = np.asarray(values, dtype=np.float32)
    v = _c(arr.ravel(), np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_array(_ptr(v), _ptr(out), v.size)
    return out.reshape(arr.shape)


def fp16_rne(values) -> np.ndarray:
    """fp32 -> fp16 bit patterns, round to nearest even (element-wise, same shape)."""
    arr = np.asarray(values, dtype=np.float32)
    v = _c(arr.ravel(), np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_fp16_rne_array(_ptr(v), _ptr(out), v.size)
    return out.reshape(arr.shape)


def bf16_to_float(bits) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact: the pattern is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).ravel()
    lib = _load()
    return np.array([lib.oracle_bf16_to_float(int(h)) for h in b], dtype=np.float32)


def fp16_to_float(bits) -> np.ndarray:
    """fp16 bit patterns -> fp32 (exact)."""
    b = _c(np.asarray(bits, dtype=np.uint16).ravel(), np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    _load().oracle_fp16_to_float_array(_ptr(b), _ptr(out), b.size)
    return out


# --------------------------------------------------------------------------- #
# W4A16
# --------------------------------------------------------------------------- #

def w4a16_quantize(w: np.ndarray, group: int = 128):
    """fp32 [N, K] -> (codes u8 [N, K], scales bf16-bits [K/G, N], mins bf16-bits [K/G, N])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % group == 0
    codes = np.empty((N, K), dtype=np.uint8)
    scales = np.empty((K // group, N), dtype=np.uint16)
    mins = np.empty((K // group, N), dtype=np.uint16)
    _load().oracle_w4a16_quantize(_ptr(w), N, K, group, _ptr(codes), _ptr(scales), _ptr(mins))
    return codes, scales, mins


def w4a16_pack(codes: np.ndarray) -> np.ndarray:
    """u8 codes [N, K] -> int32 [K/8, N]."""
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    assert K % 8 == 0
    qw = np.empty((K // 8, N), dtype=np.int32)
    _load().oracle_w4a16_pack(_ptr(codes), N, K, _ptr(qw))
    return qw


def w4a16_dequant(qw: np.ndarray, scales: np.ndarray, mins: np.ndarray, group: int = 128) -> np.ndarray:
    """Packed weights -> w_hat fp64 [N, K]."""
    qw = _c(qw, np.int32)
    scales = _c(scales, np.uint16)
    mins = _c(mins, np.uint16)
    N = qw.shape[1]
    K = qw.shape[0] * 8
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_w4a16_dequant(_ptr(qw), _ptr(scales), _ptr(mins), N, K, group, _ptr(out))
    return out


def w4a16_matmul(x_bits: np.ndarray, qw: np.ndarray, scales: np.ndarray, mins: np.ndarray,
                 group: int = 128, cols=None):
    """y_ref, abs_ref (fp64 [M, N] or [M, len(cols)]) for y = x . w_hat^T."""
    x_bits = _c(x_bits, np.uint16)
    if x_bits.ndim == 1:
        x_bits = x_bits.reshape(1, -1)
    qw = _c(qw, np.int32)
    scales = _c(scales, np.uint16)
    mins = _c(mins, np.uint16)
    M, K = x_bits.shape
    N = qw.shape[1]
    assert qw.shape[0] * 8 == K
    lib = _load()
    if cols is None:
        y = np.empty((M, N), dtype=np.float64)
        a = np.empty((M, N), dtype=np.float64)
        lib.oracle_w4a16_matmul(_ptr(x_bits), _ptr(qw), _ptr(scales), _ptr(mins), M, N, K, group,
                                _ptr(y), _ptr(a))
    else:
        cols = _c(cols, np.int32)
        y = np.empty((M, len(cols)), dtype=np.float64)
        a = np.empty((M, len(cols)), dtype=np.float64)
        lib.oracle_w4a16_matmul_cols(_ptr(x_bits), _ptr(qw), _ptr(scales), _ptr(mins), M, N, K,
                                     group, _ptr(cols), len(cols), _ptr(y), _ptr(a))
    return y, a


def w4a16_prepared_words(N: int, K: int, group: int = 128) -> int:
    """uint32 words of the prepared layout: one 2176-word record per (128-column tile,
    group of 128)."""
    return int(_load().oracle_w4a16_prepared_words(N, K, group))


def w4a16_prepare(qw: np.ndarray, scales: np.ndarray, mins: np.ndarray, group: int = 128) -> np.ndarray:
    """Canonical (qw [K/8, N], BF16 scales and minimums [K/G, N]) -> the prepared layout,
    uint32 [prepared_words] (see oracle_w4a16_prepare in w4a16_oracle.c)."""
    qw = _c(qw, np.int32)
    scales = _c(scales, np.uint16)
    mins = _c(mins, np.uint16)
    N = qw.shape[1]
    K = qw.shape[0] * 8
    assert K % group == 0
    out = np.empty(w4a16_prepared_words(N, K, group), dtype=np.uint32)
    _load().oracle_w4a16_prepare(_ptr(qw), _ptr(scales), _ptr(mins), N, K, group, _ptr(out))
    return out


# --------------------------------------------------------------------------- #
# W4A16 with a zero point
# --------------------------------------------------------------------------- #

def w4a16zp_quantize(w: np.ndarray, group: int = 128):
    """fp32 [N, K] -> (qw_rows uint32 [N, K/8], scales fp16-bits [N, K/G],
    zeros fp16-bits [N, K/G])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % group == 0 and group % 8 == 0
    qw_rows = np.empty((N, K // 8), dtype=np.uint32)
    scales = np.empty((N, K // group), dtype=np.uint16)
    zeros = np.empty((N, K // group), dtype=np.uint16)
    _load().oracle_w4a16zp_quantize(_ptr(w), N, K, group, _ptr(qw_rows), _ptr(scales),
                                    _ptr(zeros))
    return qw_rows, scales, zeros


def w4a16zp_dequant(qw_rows: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                    group: int = 128) -> np.ndarray:
    """w_hat = (q - z) s, fp64 [N, K]."""
    qw_rows = _c(qw_rows, np.uint32)
    scales = _c(scales, np.uint16)
    zeros = _c(zeros, np.uint16)
    N, K = qw_rows.shape[0], qw_rows.shape[1] * 8
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_w4a16zp_dequant(_ptr(qw_rows), _ptr(scales), _ptr(zeros), N, K, group,
                                   _ptr(out))
    return out


def w4a16zp_matmul(x_bits: np.ndarray, qw_rows: np.ndarray, scales: np.ndarray,
                   zeros: np.ndarray, group: int = 128, cols=None):
    """y_ref, abs_ref (fp64 [M, N] or [M, len(cols)]) for y = x . w_hat^T."""
    x_bits = _c(x_bits, np.uint16)
    if x_bits.ndim == 1:
        x_bits = x_bits.reshape(1, -1)
    qw_rows = _c(qw_rows, np.uint32)
    scales = _c(scales, np.uint16)
    zeros = _c(zeros, np.uint16)
    M, K = x_bits.shape
    N = qw_rows.shape[0]
    assert qw_rows.shape[1] * 8 == K
    if cols is None:
        n_out, cols_p = N, None
    else:
        cols = _c(cols, np.int32)
        n_out, cols_p = len(cols), _ptr(cols)
    y = np.empty((M, n_out), dtype=np.float64)
    a = np.empty((M, n_out), dtype=np.float64)
    _load().oracle_w4a16zp_matmul(_ptr(x_bits), _ptr(qw_rows), _ptr(scales), _ptr(zeros), M, N,
                                  K, group, cols_p, n_out, _ptr(y), _ptr(a))
    return y, a


def w4a16zp_kernel_layout(qw_rows: np.ndarray, scales: np.ndarray, zeros: np.ndarray):
    """The same numbers in the matmul's input layout: words [K/8, N] (int32) and
    scales / zeros [K/G, N]: the transpose of each array, nothing else."""
    return (np.ascontiguousarray(_c(qw_rows, np.uint32).T).view(np.int32),
            np.ascontiguousarray(_c(scales, np.uint16).T),
            np.ascontiguousarray(_c(zeros, np.uint16).T))


# --------------------------------------------------------------------------- #
# W8A16 (symmetric per-row INT8)
# --------------------------------------------------------------------------- #

def w8a16_quantize(w: np.ndarray):
    """fp32 [N, K] -> (q int8 [N, K], s fp32 [N])."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.int8)
    s = np.empty(N, dtype=np.float32)
    _load().oracle_w8a16_quantize(_ptr(w), N, K, _ptr(q), _ptr(s))
    return q, s


def w8a16_gemv(x_bits: np.ndarray, q: np.ndarray, s: np.ndarray, rows=None):
    """y_ref, abs_ref (fp64 [N] or [len(rows)]) for y = W_hat . x."""
    x_bits = _c(x_bits, np.uint16).ravel()
    q = _c(q, np.int8)
    s = _c(s, np.float32)
    N, K = q.shape
    assert x_bits.shape[0] == K and s.shape[0] == N
    if rows is None:
        n_out, rows_p = N, None
    else:
        rows = _c(rows, np.int32)
        n_out, rows_p = len(rows), _ptr(rows)
    y = np.empty(n_out, dtype=np.float64)
    a = np.empty(n_out, dtype=np.float64)
    _load().oracle_w8a16_gemv(_ptr(x_bits), _ptr(q), _ptr(s), N, K, rows_p, n_out, _ptr(y),
                              _ptr(a))
    return y, a


# --------------------------------------------------------------------------- #
# NVFP4 weights (E2M1 codes, E4M3 block scales, fp32 tensor scale)
# --------------------------------------------------------------------------- #

def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(int(code)))


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(int(code)))


def e2m1_rne(t: float) -> int:
    return int(_load().oracle_e2m1_rne(float(t)))


def e4m3_ceil(v: float) -> int:
    return int(_load().oracle_e4m3_ceil(float(v)))


def nvfp4_quantize(w: np.ndarray):
    """fp32 [N, K] -> (codes u8 [N, K/2], scales u8 E4M3 [N, K/16], S float)."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 16 == 0
    codes = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 16), dtype=np.uint8)
    S = np.zeros(1, dtype=np.float32)
    _load().oracle_nvfp4_quantize(_ptr(w), N, K, _ptr(codes), _ptr(scales), _ptr(S))
    return codes, scales, float(S[0])


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, S: float) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_nvfp4_dequant(_ptr(codes), _ptr(scales), float(S), N, K, _ptr(out))
    return out


def nvfp4_gemv(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, S: float, rows=None):
    """y_ref, abs_ref (fp64 [N] or [len(rows)]) for y = W_hat . x."""
    x_bits = _c(x_bits, np.uint16).ravel()
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    assert x_bits.shape[0] == K and scales.shape == (N, K // 16)
    if rows is None:
        n_out, rows_p = N, None
    else:
        rows = _c(rows, np.int32)
        n_out, rows_p = len(rows), _ptr(rows)
    y = np.empty(n_out, dtype=np.float64)
    a = np.empty(n_out, dtype=np.float64)
    _load().oracle_nvfp4_gemv(_ptr(x_bits), _ptr(codes), _ptr(scales), float(S), N, K, rows_p,
                              n_out, _ptr(y), _ptr(a))
    return y, a


def nvfp4_matmul(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, S: float,
                 rows=None):
    """y_ref, abs_ref (fp64 [M, N] or [M, len(rows)]) for Y[m] = W_hat . x[m]: the GEMV of
    each row of x (the matmul's definition, a row at a time)."""
    x_bits = _c(x_bits, np.uint16)
    outs = [nvfp4_gemv(x_bits[m], codes, scales, S, rows=rows) for m in range(x_bits.shape[0])]
    return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])


def e8m0_value(code: int) -> float:
    return float(_load().oracle_e8m0_value(int(code)))


def mxfp4_quantize(w: np.ndarray):
    """fp32 [N, K] -> (codes u8 [N, K/2], scales u8 E8M0 [N, K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    codes = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 32), dtype=np.uint8)
    _load().oracle_mxfp4_quantize(_ptr(w), N, K, _ptr(codes), _ptr(scales))
    return codes, scales


def mxfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_mxfp4_dequant(_ptr(codes), _ptr(scales), N, K, _ptr(out))
    return out


def mxfp4_gemv(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, rows=None):
    """y_ref, abs_ref (fp64 [N] or [len(rows)]) for y = W_hat . x."""
    x_bits = _c(x_bits, np.uint16).ravel()
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    assert x_bits.shape[0] == K and scales.shape == (N, K // 32)
    if rows is None:
        n_out, rows_p = N, None
    else:
        rows = _c(rows, np.int32)
        n_out, rows_p = len(rows), _ptr(rows)
    y = np.empty(n_out, dtype=np.float64)
    a = np.empty(n_out, dtype=np.float64)
    _load().oracle_mxfp4_gemv(_ptr(x_bits), _ptr(codes), _ptr(scales), N, K, rows_p, n_out,
                              _ptr(y), _ptr(a))
    return y, a


# --------------------------------------------------------------------------- #
# Q4 block-32
# --------------------------------------------------------------------------- #

def mxfp4_matmul(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, rows=None):
    """y_ref, abs_ref (fp64 [M, N] or [M, len(rows)]) for Y[m] = W_hat . x[m]: the GEMV of
    each row of x."""
    x_bits = _c(x_bits, np.uint16)
    outs = [mxfp4_gemv(x_bits[m], codes, scales, rows=rows) for m in range(x_bits.shape[0])]
    return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])


def q4b32_quantize(w: np.ndarray):
    """fp32 [N, K] -> (codes u8 [N, K/2], scales fp16-bits [N, K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    codes = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 32), dtype=np.uint16)
    _load().oracle_q4b32_quantize(_ptr(w), N, K, _ptr(codes), _ptr(scales))
    return codes, scales


def q4b32_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    N = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_q4b32_dequant(_ptr(codes), _ptr(scales), N, K, _ptr(out))
    return out


def q4b32_gemv(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, rows=None):
    """y_ref, abs_ref (fp64 [N] or [len(rows)]) for y = W_hat . x."""
    x_bits = _c(x_bits, np.uint16).ravel()
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    N = codes.shape[0]
    K = codes.shape[1] * 2
    assert x_bits.shape[0] == K
    if rows is None:
        n_out, rows_p, nrows = N, None, 0
    else:
        rows = _c(rows, np.int32)
        n_out, rows_p, nrows = len(rows), _ptr(rows), len(rows)
    y = np.empty(n_out, dtype=np.float64)
    a = np.empty(n_out, dtype=np.float64)
    _load().oracle_q4b32_gemv(_ptr(x_bits), _ptr(codes), _ptr(scales), N, K, rows_p, nrows,
                              _ptr(y), _ptr(a))
    return y, a


# --------------------------------------------------------------------------- #
# Acceptance rule
# --------------------------------------------------------------------------- #

def within_tolerance(y, y_ref, abs_ref, rel: float = 4e-3, absf: float = 1e-3) -> np.ndarray:
    """Per-output acceptance: |y - y_ref| <= rel*|y_ref| + absf*sum_k|x_k w_hat_k|.

    The bound is the one the W4A16 target states for BF16 output with fp32
    accumulation; the Q4 GEMV (FP16 output) uses the same form.
    """
    y = np.asarray(y, dtype=np.float64)
    return np.abs(y - y_ref) <= rel * np.abs(y_ref) + absf * abs_ref
