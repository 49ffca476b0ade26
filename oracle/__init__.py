"""Python access to the CPU oracle of the LLM.int8() decomposed matmul.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package; the product library never
imports it.  The arithmetic lives in ``llmint8_oracle.c`` (plain C, compiled
here with gcc on first use); this module only marshals numpy arrays.

Step names follow the method's steps:
  A0 quantize_weight   per-output-column absmax int8 codes of W
  A1 outlier_columns   K-columns of X with some |x| > t
  A2 quantize_rows     per-row absmax int8 codes of the non-outlier part of X
  A3 int8_matmul       exact integer product of the codes (int64)
  A4 outlier_matmul    fp16 product of the outlier slice (double)
  A5 merge             C * s_x * s_w / 127^2 + F, rounded to fp16
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "llmint8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread", "-Wall"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc if the shared object is missing or stale."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH) or
             os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_double_to_half.argtypes = [ctypes.c_double]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_scale_factor.argtypes = [ctypes.c_float]
            lib.oracle_scale_factor.restype = ctypes.c_float
            lib.oracle_code.argtypes = [ctypes.c_float, ctypes.c_float]
            lib.oracle_code.restype = ctypes.c_int8
            lib.oracle_quantize_weight.argtypes = [P, I, I, P, P]
            lib.oracle_outlier_columns.argtypes = [P, I, I, ctypes.c_float, P]
            lib.oracle_quantize_per_tensor.argtypes = [P, I, P, P]
            lib.oracle_quantize_rows.argtypes = [P, I, I, P, P, P]
            lib.oracle_int8_matmul.argtypes = [P, P, I, I, I, P, ctypes.c_int]
            lib.oracle_outlier_matmul.argtypes = [P, P, P, I, I, I, P, ctypes.c_int]
            lib.oracle_merge.argtypes = [P, P, P, P, I, I, P]
            lib.oracle_dequantize_weight.argtypes = [P, P, I, I, P]
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            C = ctypes.c_int
            lib.oracle_quantize_weight_fmt.argtypes = [P, I, I, P, P, C]
            lib.oracle_outlier_columns_fmt.argtypes = [P, I, I, ctypes.c_float, P, C]
            lib.oracle_quantize_rows_fmt.argtypes = [P, I, I, P, P, P, C]
            lib.oracle_outlier_matmul_fmt.argtypes = [P, P, P, I, I, I, P, C, C]
            lib.oracle_merge_fmt.argtypes = [P, P, P, P, I, I, P, C]
            lib.oracle_dequantize_weight_fmt.argtypes = [P, P, I, I, P, C]
            for f in ("oracle_quantize_weight", "oracle_outlier_columns", "oracle_quantize_rows",
                      "oracle_quantize_per_tensor", "oracle_dequantize_weight",
                      "oracle_quantize_weight_fmt", "oracle_outlier_columns_fmt", "oracle_quantize_rows_fmt",
                      "oracle_outlier_matmul_fmt", "oracle_merge_fmt", "oracle_dequantize_weight_fmt",
                      "oracle_int8_matmul", "oracle_outlier_matmul", "oracle_merge"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a) -> np.ndarray:
    """fp16 array (or uint16 bit patterns: fp16, or bf16 data) -> contiguous uint16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16 data or uint16 bit patterns, got {a.dtype}")


# 16-bit element formats of X, W and Y: fp16 (numpy float16 or its bits) or
# bf16 (uint16 bit patterns; numpy has no bfloat16)
_FMT = {"fp16": 0, "bf16": 1}


def _out16(bits: np.ndarray, fmt: str) -> np.ndarray:
    return bits.view(np.float16) if fmt == "fp16" else bits


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# -- scalar helpers ---------------------------------------------------------------

def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits))


def double_to_half(v: float) -> int:
    return int(_load().oracle_double_to_half(float(v)))


def scale_factor(absmax: float) -> float:
    return float(_load().oracle_scale_factor(float(absmax)))


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def double_to_bf16(v: float) -> int:
    return _load().oracle_double_to_bf16(float(v))


def code(x: float, sf: float) -> int:
    return int(_load().oracle_code(float(x), float(sf)))


def to_half(values: np.ndarray) -> np.ndarray:
    """Vector form of double_to_half (returns float16)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_double_to_half(float(x)) for x in v), dtype=np.uint16, count=v.size)
    return out.view(np.float16).reshape(np.shape(values))


# -- method steps -------------------------------------------------------------------

def quantize_weight(W: np.ndarray, fmt: str = "fp16"):
    """A0: W [K,N] -> (Wq int8 [K,N], s_w float32 [N] = column absmax)."""
    Wb = _bits(W)
    K, N = Wb.shape
    Wq = np.empty((K, N), np.int8)
    sw = np.empty(N, np.float32)
    _load().oracle_quantize_weight_fmt(_ptr(Wb), K, N, _ptr(Wq), _ptr(sw), _FMT[fmt])
    return Wq, sw


def outlier_columns(X: np.ndarray, t: float, fmt: str = "fp16") -> np.ndarray:
    """A1: bool [K], True where some |X[i,j]| > t."""
    Xb = _bits(X)
    M, K = Xb.shape
    out = np.empty(K, np.uint8)
    _load().oracle_outlier_columns_fmt(_ptr(Xb), M, K, float(t), _ptr(out), _FMT[fmt])
    return out.astype(bool)


def quantize_rows(X: np.ndarray, is_outlier: np.ndarray, fmt: str = "fp16"):
    """A2: (Xq int8 [M,K] with outlier columns zero, s_x float32 [M])."""
    Xb = _bits(X)
    M, K = Xb.shape
    mask = np.ascontiguousarray(is_outlier, dtype=np.uint8)
    Xq = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    _load().oracle_quantize_rows_fmt(_ptr(Xb), M, K, _ptr(mask), _ptr(Xq), _ptr(sx), _FMT[fmt])
    return Xq, sx


def int8_matmul(Xq: np.ndarray, Wq: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """A3: exact C = Xq . Wq in int64."""
    Xq = np.ascontiguousarray(Xq, np.int8)
    Wq = np.ascontiguousarray(Wq, np.int8)
    M, K = Xq.shape
    K2, N = Wq.shape
    assert K == K2
    C = np.empty((M, N), np.int64)
    _load().oracle_int8_matmul(_ptr(Xq), _ptr(Wq), M, K, N, _ptr(C), nthreads or default_threads())
    return C


def outlier_matmul(X: np.ndarray, W: np.ndarray, is_outlier: np.ndarray,
                   nthreads: int | None = None, fmt: str = "fp16") -> np.ndarray:
    """A4: F = X[:, O] . W[O, :] in double."""
    Xb, Wb = _bits(X), _bits(W)
    M, K = Xb.shape
    K2, N = Wb.shape
    assert K == K2
    mask = np.ascontiguousarray(is_outlier, dtype=np.uint8)
    F = np.empty((M, N), np.float64)
    _load().oracle_outlier_matmul_fmt(_ptr(Xb), _ptr(Wb), _ptr(mask), M, K, N, _ptr(F),
                                      nthreads or default_threads(), _FMT[fmt])
    return F


def merge(C: np.ndarray, s_x: np.ndarray, s_w: np.ndarray, F: np.ndarray | None, fmt: str = "fp16") -> np.ndarray:
    """A5: Y = RNE(C * s_x * s_w / 127^2 + F) in the output format (fp16, or bf16 bits)."""
    C = np.ascontiguousarray(C, np.int64)
    M, N = C.shape
    sx = np.ascontiguousarray(s_x, np.float32)
    sw = np.ascontiguousarray(s_w, np.float32)
    Fp = None
    if F is not None:
        F = np.ascontiguousarray(F, np.float64)
        Fp = _ptr(F)
    Y = np.empty((M, N), np.uint16)
    _load().oracle_merge_fmt(_ptr(C), _ptr(sx), _ptr(sw), Fp, M, N, _ptr(Y), _FMT[fmt])
    return _out16(Y, fmt)


def quantize_per_tensor(A: np.ndarray):
    """Ablation: one scale for the whole fp16 tensor -> (codes int8, same shape; absmax float32)."""
    Ab = np.ascontiguousarray(_bits(A))
    q = np.empty(Ab.shape, np.int8)
    s = np.empty(1, np.float32)
    _load().oracle_quantize_per_tensor(_ptr(Ab), Ab.size, _ptr(q), _ptr(s))
    return q, s[0]


def per_tensor_int8_matmul(X: np.ndarray, W: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """Ablation: Y = X.W with one scale per tensor for X and W, no outlier decomposition."""
    Xq, sx = quantize_per_tensor(X)
    Wq, sw = quantize_per_tensor(W)
    C = int8_matmul(Xq, Wq, nthreads)
    M, N = C.shape
    return merge(C, np.full(M, sx, np.float32), np.full(N, sw, np.float32), None)


def dequantize_weight(Wq: np.ndarray, s_w: np.ndarray, fmt: str = "fp16") -> np.ndarray:
    """A4 weight rows when only the int8 codes are kept: RNE(q * (s_w / 127)) [K,N] in fmt."""
    Wq = np.ascontiguousarray(Wq, np.int8)
    K, N = Wq.shape
    sw = np.ascontiguousarray(s_w, np.float32)
    out = np.empty((K, N), np.uint16)
    _load().oracle_dequantize_weight_fmt(_ptr(Wq), _ptr(sw), K, N, _ptr(out), _FMT[fmt])
    return _out16(out, fmt)


def outlier_indices(is_outlier: np.ndarray) -> np.ndarray:
    """Sorted int32 indices of the outlier columns."""
    return np.flatnonzero(np.asarray(is_outlier)).astype(np.int32)


def llmint8_matmul(X: np.ndarray, W: np.ndarray, t: float, rows=None, nthreads: int | None = None,
                   wq=None, cols=None, w16_rows=None, fmt: str = "fp16"):
    """The whole path A0..A5 for Y = X.W with threshold t.

    Outlier detection (A1) always scans all rows of X, because the outlier set
    is a property of the whole activation matrix.  ``rows`` (optional index
    array) restricts A2..A5 to those rows, for spot checks of large problems.
    ``cols`` (optional) restricts the output columns: A0 (one scale per output
    column), A3, A4 and A5 are each local to a column, so the oracle simply
    runs on W[:, cols].  ``wq`` may pass a precomputed (Wq, s_w) from
    quantize_weight of the (restricted) W.  ``w16_rows`` (optional index
    array) selects the mode where only those rows of W are kept in fp16: A4
    then takes every other outlier row from dequantize_weight.  ``fmt="bf16"``
    takes X and W as bfloat16 bit patterns (uint16) and returns Y in bfloat16
    bits.  Returns a dict with every intermediate.
    """
    if cols is not None:
        W = np.ascontiguousarray(W[:, np.asarray(cols)])
    Wq, s_w = wq if wq is not None else quantize_weight(W, fmt)
    is_out = outlier_columns(X, t, fmt)
    Xs = X if rows is None else np.ascontiguousarray(X[np.asarray(rows)])
    Xq, s_x = quantize_rows(Xs, is_out, fmt)
    C = int8_matmul(Xq, Wq, nthreads)
    W4 = W
    if w16_rows is not None:  # fp16 rows only where kept, dequantized codes elsewhere
        keep = np.zeros(W.shape[0], bool)
        keep[np.asarray(w16_rows, np.int64)] = True
        W4 = np.where(keep[:, None], W, dequantize_weight(Wq, s_w, fmt))
    F = outlier_matmul(Xs, W4, is_out, nthreads, fmt) if is_out.any() else np.zeros(C.shape, np.float64)
    Y = merge(C, s_x, s_w, F, fmt)
    return dict(Y=Y, C=C, F=F, Xq=Xq, s_x=s_x, Wq=Wq, s_w=s_w, is_outlier=is_out,
                outliers=outlier_indices(is_out))
