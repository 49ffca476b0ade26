"""Python binding of the LLM.int8() C ABI, same names as include/llmint8.h.

Argument marshalling only: torch tensors supply device pointers, shapes and the
current CUDA stream; every step of the computation runs in libllmint8.so.
Outputs that are not passed in are allocated with torch (device memory is the
one thing PyTorch is used for).
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib


class LLMInt8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {llmint8_status_str(status)} (status {status})")


def llmint8_status_str(status: int) -> str:
    return _lib.load().llmint8_status_str(int(status)).decode()


def _check(status: int, where: str):
    if status != _lib.OK:
        raise LLMInt8Error(status, where)


# The per-call path is kept thin: device pointers and the stream handle cross as
# plain integers (ctypes converts them for the void* arguments).

def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None, like=None):
    """Raw handle of `stream`, else of the current stream of `like`'s device."""
    if stream is not None:
        return stream.cuda_stream
    dev = like.device.index if like is not None else torch.cuda.current_device()
    return torch._C._cuda_getCurrentRawStream(dev)


def _need(t, dtype, shape, name):
    if t is None:
        return
    if t.dtype != dtype or t.shape != shape or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def llmint8_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(_lib.load().llmint8_workspace_bytes(int(M), int(K), int(N)))


def llmint8_kernels_per_call(M: int, K: int, N: int, threshold: float, write_i32: bool = False) -> int:
    """Kernels one llmint8_matmul (or, with write_i32, llmint8_matmul_i32) call launches."""
    n = _lib.load().llmint8_kernels_per_call(M, K, N, float(threshold), 1 if write_i32 else 0)
    if n < 0:
        raise ValueError(f"llmint8_kernels_per_call: invalid arguments M={M} K={K} N={N} t={threshold}")
    return n


def llmint8_workspace_layout(M: int, K: int, N: int) -> dict:
    off = (ctypes.c_size_t * len(_lib.WS_FIELDS))()
    _check(_lib.load().llmint8_workspace_layout(int(M), int(K), int(N), off), "llmint8_workspace_layout")
    return {name: int(off[i]) for i, name in enumerate(_lib.WS_FIELDS)}


def make_workspace(M: int, K: int, N: int, device=None) -> torch.Tensor:
    n = llmint8_workspace_bytes(M, K, N)
    if n == 0:
        raise ValueError(f"unsupported shape M={M} K={K} N={N}")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def llmint8_quantize_weight(W: torch.Tensor, Wq=None, colScaleW=None, stream=None):
    """A0: W fp16 [K, N] -> (Wq int8 [N, K], colScaleW fp32 [N])."""
    K, N = W.shape
    dev = W.device
    if Wq is None:
        Wq = torch.empty((N, K), dtype=torch.int8, device=dev)
    if colScaleW is None:
        colScaleW = torch.empty((N,), dtype=torch.float32, device=dev)
    _need(W, torch.float16, (K, N), "W")
    _need(Wq, torch.int8, (N, K), "Wq")
    _need(colScaleW, torch.float32, (N,), "colScaleW")
    st = _lib.load().llmint8_quantize_weight(_ptr(W), K, N, _ptr(Wq), _ptr(colScaleW), _stream(stream, W))
    _check(st, "llmint8_quantize_weight")
    return Wq, colScaleW


def llmint8_quantize_weight_bf16(W: torch.Tensor, Wq=None, colScaleW=None, stream=None):
    """A0 for bf16 W [K, N] -> (Wq int8 [N, K], colScaleW fp32 [N])."""
    K, N = W.shape
    dev = W.device
    if Wq is None:
        Wq = torch.empty((N, K), dtype=torch.int8, device=dev)
    if colScaleW is None:
        colScaleW = torch.empty((N,), dtype=torch.float32, device=dev)
    _need(W, torch.bfloat16, (K, N), "W")
    _need(Wq, torch.int8, (N, K), "Wq")
    _need(colScaleW, torch.float32, (N,), "colScaleW")
    st = _lib.load().llmint8_quantize_weight_bf16(_ptr(W), K, N, _ptr(Wq), _ptr(colScaleW),
                                                  _stream(stream, W))
    _check(st, "llmint8_quantize_weight_bf16")
    return Wq, colScaleW


def _shapes(X, Wq):
    M, K = X.shape
    N = Wq.shape[0]
    return M, K, N


def llmint8_matmul(X, threshold, Wq, colScaleW, W16, Y=None, workspace=None, stream=None):
    """A1..A5: Y = X.W with the LLM.int8() decomposition at `threshold`."""
    M, K, N = _shapes(X, Wq)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.float16, (M, K), "X")
    _need(Y, torch.float16, (M, N), "Y")
    st = _lib.load().llmint8_matmul(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW), _ptr(W16),
                                    _ptr(Y), _ptr(workspace), workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul")
    return Y


def llmint8_matmul_host(X_host, X, threshold, Wq, colScaleW, W16, Y, Y_host, workspace, stream=None):
    """llmint8_matmul between host tensors: X_host -> X (device), Y = X.W, Y -> Y_host, all
    enqueued on the stream by one call (synchronize before reading Y_host)."""
    M, K, N = _shapes(X, Wq)
    _need(X_host, torch.float16, (M, K), "X_host")
    _need(X, torch.float16, (M, K), "X")
    _need(Y, torch.float16, (M, N), "Y")
    _need(Y_host, torch.float16, (M, N), "Y_host")
    if X_host.is_cuda or Y_host.is_cuda or not X.is_cuda:
        raise ValueError("llmint8_matmul_host: X_host and Y_host are host tensors, X and Y device tensors")
    st = _lib.load().llmint8_matmul_host(_ptr(X_host), _ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW),
                                         _ptr(W16), _ptr(Y), _ptr(Y_host), _ptr(workspace),
                                         workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul_host")
    return Y_host


def llmint8_chain_state_layout(M: int, N: int):
    """(flags offset, partial-maxima offset, total bytes) of a chain state for an activation [M, N]."""
    off = (ctypes.c_size_t * 3)()
    _check(_lib.load().llmint8_chain_state_layout(M, N, off), "llmint8_chain_state_layout")
    return int(off[0]), int(off[1]), int(off[2])


def make_chain_state(M: int, N: int, device=None) -> torch.Tensor:
    n = _lib.load().llmint8_chain_state_bytes(M, N)
    if n == 0:
        raise ValueError(f"no chain state for M={M} N={N}")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _state(S, M, cols, device, name):
    """A chain state buffer: uint8 on `device`, at least llmint8_chain_state_bytes(M, cols) bytes."""
    if S is None:
        return 0
    need = int(_lib.load().llmint8_chain_state_bytes(M, cols))
    if S.dtype != torch.uint8 or S.device != device or not S.is_contiguous() or S.numel() < need:
        raise ValueError(f"{name}: expected a contiguous uint8 tensor on {device} of at least {need} bytes, "
                         f"got {S.dtype} {tuple(S.shape)} on {S.device}")
    return S.numel()


def llmint8_matmul_chain(X, threshold, state_in, Wq, colScaleW, W16, next_threshold=6.0, state_out=None, Y=None,
                         workspace=None, stream=None, C=None):
    """Decode-chain matmul (M <= 4): Y = X.W as llmint8_matmul; with `state_in` (the chain
    state of X from the previous call) no X pass runs; with `state_out` the chain state of Y
    for `next_threshold` is written.  With `C` (int32 [M, N]) the exact accumulator of the
    int8 product is written too (llmint8_matmul_chain_i32)."""
    M, K, N = _shapes(X, Wq)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.float16, (M, K), "X")
    _need(Y, torch.float16, (M, N), "Y")
    _need(C, torch.int32, (M, N), "C")
    nin = _state(state_in, M, K, X.device, "state_in")
    nout = _state(state_out, M, N, X.device, "state_out")
    lib = _lib.load()
    args = (_ptr(X), M, K, N, float(threshold), _ptr(state_in), nin, _ptr(Wq), _ptr(colScaleW), _ptr(W16), _ptr(Y),
            float(next_threshold), _ptr(state_out), nout)
    if C is None:
        st = lib.llmint8_matmul_chain(*args, _ptr(workspace), workspace.numel(), _stream(stream, X))
    else:
        st = lib.llmint8_matmul_chain_i32(*args, _ptr(C), _ptr(workspace), workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul_chain")
    return Y


def llmint8_quantize_x(X, threshold, Xq=None, rowScaleX=None, workspace=None, stream=None):
    """A1 + A2 into caller buffers: (Xq int8 [M, K], rowScaleX fp32 [M], workspace holding the outlier set)."""
    M, K = X.shape
    dev = X.device
    if Xq is None:
        Xq = torch.empty((M, K), dtype=torch.int8, device=dev)
    if rowScaleX is None:
        rowScaleX = torch.empty((M,), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = make_workspace(M, K, 16, dev)
    _need(X, torch.float16, (M, K), "X")
    _need(Xq, torch.int8, (M, K), "Xq")
    _need(rowScaleX, torch.float32, (M,), "rowScaleX")
    st = _lib.load().llmint8_quantize_x(_ptr(X), M, K, float(threshold), _ptr(Xq), _ptr(rowScaleX), _ptr(workspace),
                                        workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_quantize_x")
    return Xq, rowScaleX, workspace


def llmint8_read_outliers(workspace, K: int, stream=None):
    """Synchronize and return the sorted outlier columns (int32 numpy array) left in `workspace`."""
    import numpy as np
    lib = _lib.load()
    count = ctypes.c_int(0)
    _check(lib.llmint8_read_outliers(_ptr(workspace), int(K), ctypes.byref(count), None, 0,
                                     _stream(stream, workspace)), "llmint8_read_outliers")
    out = np.zeros(max(count.value, 1), np.int32)
    _check(lib.llmint8_read_outliers(_ptr(workspace), int(K), ctypes.byref(count),
                                     out.ctypes.data_as(ctypes.c_void_p), out.size, _stream(stream, workspace)),
           "llmint8_read_outliers")
    return out[:count.value]


def llmint8_pack_w16_rows(W16, rows, stream=None):
    """Kept fp16 rows of W for llmint8_matmul_w8: (W16c [R, N], row_map int32 [K])."""
    K, N = W16.shape
    _need(W16, torch.float16, (K, N), "W16")
    rows = torch.as_tensor(rows, dtype=torch.int32, device=W16.device).contiguous()
    R = rows.numel()
    W16c = torch.empty((R, N), dtype=torch.float16, device=W16.device)
    row_map = torch.empty((K,), dtype=torch.int32, device=W16.device)
    st = _lib.load().llmint8_pack_w16_rows(_ptr(W16), K, N, _ptr(rows) if R else None, R,
                                           _ptr(W16c) if R else None, _ptr(row_map), _stream(stream, W16))
    _check(st, "llmint8_pack_w16_rows")
    return W16c, row_map


def llmint8_matmul_w8(X, threshold, Wq, colScaleW, W16c=None, row_map=None, Y=None, workspace=None,
                      stream=None):
    """A1..A5 without a full fp16 copy of W: outlier rows from W16c via row_map, else dequantized codes."""
    M, K, N = _shapes(X, Wq)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.float16, (M, K), "X")
    _need(Y, torch.float16, (M, N), "Y")
    _need(row_map, torch.int32, (K,), "row_map")
    R = 0 if W16c is None else W16c.shape[0]
    _need(W16c, torch.float16, (R, N), "W16c")
    st = _lib.load().llmint8_matmul_w8(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW),
                                       _ptr(W16c) if R else None, _ptr(row_map), R, _ptr(Y), _ptr(workspace),
                                       workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul_w8")
    return Y


def llmint8_matmul_bf16(X, threshold, Wq, colScaleW, W16, Y=None, workspace=None, stream=None):
    """A1..A5 on bf16 X [M, K] and W16 [K, N] -> Y bf16 [M, N]."""
    M, K, N = _shapes(X, Wq)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.bfloat16, (M, K), "X")
    _need(Y, torch.bfloat16, (M, N), "Y")
    _need(W16, torch.bfloat16, (K, N), "W16")
    st = _lib.load().llmint8_matmul_bf16(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW), _ptr(W16),
                                         _ptr(Y), _ptr(workspace), workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul_bf16")
    return Y


def llmint8_matmul_i32_bf16(X, threshold, Wq, colScaleW, C=None, workspace=None, stream=None):
    """The exact int32 accumulator C of llmint8_matmul_bf16 (bf16 X)."""
    M, K, N = _shapes(X, Wq)
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.bfloat16, (M, K), "X")
    _need(C, torch.int32, (M, N), "C")
    st = _lib.load().llmint8_matmul_i32_bf16(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW),
                                             _ptr(C), _ptr(workspace), workspace.numel(),
                                             _stream(stream, X))
    _check(st, "llmint8_matmul_i32_bf16")
    return C


def llmint8_matmul_int8(X, Wq, colScaleW, Y=None, workspace=None, stream=None):
    """Plain vector-wise int8 (threshold = +inf, no fp16 weight)."""
    M, K, N = _shapes(X, Wq)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.float16, (M, K), "X")
    _need(Y, torch.float16, (M, N), "Y")
    st = _lib.load().llmint8_matmul_int8(_ptr(X), M, K, N, _ptr(Wq), _ptr(colScaleW), _ptr(Y),
                                         _ptr(workspace), workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul_int8")
    return Y


def llmint8_matmul_i32(X, threshold, Wq, colScaleW, C=None, workspace=None, stream=None):
    """Same path, but returns the exact int32 accumulator C = Xq . Wq^T of step A3."""
    M, K, N = _shapes(X, Wq)
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=X.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, X.device)
    _need(X, torch.float16, (M, K), "X")
    _need(C, torch.int32, (M, N), "C")
    st = _lib.load().llmint8_matmul_i32(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW), _ptr(C),
                                        _ptr(workspace), workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_matmul_i32")
    return C


def llmint8_xpass(X, threshold, N, workspace, stream=None):
    """A1 + A2 into `workspace` (first half of llmint8_matmul)."""
    M, K = X.shape
    _need(X, torch.float16, (M, K), "X")
    st = _lib.load().llmint8_xpass(_ptr(X), M, K, int(N), float(threshold), _ptr(workspace), workspace.numel(),
                                   _stream(stream, X))
    _check(st, "llmint8_xpass")


def llmint8_gemm_i32(Xq, Wq, C=None, workspace=None, stream=None):
    """A3 on caller codes: Xq int8 [M, K], Wq int8 [N, K] -> exact C int32 [M, N]."""
    M, K = Xq.shape
    N = Wq.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=Xq.device)
    if workspace is None:
        workspace = make_workspace(M, K, N, Xq.device)
    _need(Xq, torch.int8, (M, K), "Xq")
    _need(Wq, torch.int8, (N, K), "Wq")
    _need(C, torch.int32, (M, N), "C")
    st = _lib.load().llmint8_gemm_i32(_ptr(Xq), _ptr(Wq), M, K, N, _ptr(C), _ptr(workspace), workspace.numel(),
                                      _stream(stream, Xq))
    _check(st, "llmint8_gemm_i32")
    return C


def llmint8_gemm(X, threshold, Wq, colScaleW, W16, Y, workspace, stream=None):
    """A3..A5 from a workspace filled by llmint8_xpass (second half of llmint8_matmul)."""
    M, K, N = _shapes(X, Wq)
    _need(Y, torch.float16, (M, N), "Y")
    st = _lib.load().llmint8_gemm(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW), _ptr(W16), _ptr(Y),
                                  _ptr(workspace), workspace.numel(), _stream(stream, X))
    _check(st, "llmint8_gemm")
    return Y


NOALLOC_SCRATCH_BYTES = 8 << 20


def llmint8_matmul_noalloc(X, threshold, Wq, colScaleW, W16, Y, stream=None):
    """llmint8_matmul on the library's static scratch array (no workspace, no allocation).

    Y must be passed in: this call allocates nothing, not even through torch.
    """
    M, K, N = _shapes(X, Wq)
    _need(X, torch.float16, (M, K), "X")
    _need(Y, torch.float16, (M, N), "Y")
    st = _lib.load().llmint8_matmul_noalloc(_ptr(X), M, K, N, float(threshold), _ptr(Wq), _ptr(colScaleW),
                                            _ptr(W16), _ptr(Y), _stream(stream, X))
    _check(st, "llmint8_matmul_noalloc")
    return Y


def llmint8_device_status(workspace, stream=None) -> int:
    """Synchronize and read (then clear) the device error word; returns a status code."""
    return int(_lib.load().llmint8_device_status(_ptr(workspace), _stream(stream, workspace)))


def llmint8_selftest_timeout(workspace, spin_limit: int, stream=None):
    _check(_lib.load().llmint8_selftest_timeout(_ptr(workspace), int(spin_limit), _stream(stream, workspace)),
           "llmint8_selftest_timeout")


def read_intermediates(workspace: torch.Tensor, M: int, K: int, N: int) -> dict:
    """Copy the X-pass results of the last call out of a workspace (tests/diagnostics).

    Returns row_scale (fp32 [M]), codes (int8 [M, K], decoded from the stored
    fp16 values), outliers (sorted int32) and status.
    """
    lay = llmint8_workspace_layout(M, K, N)
    ws = workspace
    count = int(ws[lay["outlier_count"]:lay["outlier_count"] + 4].view(torch.int32).item())
    idx = ws[lay["outlier_idx"]:lay["outlier_idx"] + 4 * count].view(torch.int32).clone()
    row_scale = ws[lay["row_scale"]:lay["row_scale"] + 4 * M].view(torch.float32).clone()
    if M <= _lib.DECODE_MAX_M:  # decode path: int8 codes
        codes = ws[lay["codes"]:lay["codes"] + M * K].view(torch.int8).view(M, K).clone()
        codes16 = None
    else:  # tensor-core path: the codes as exact fp16 values
        codes16 = ws[lay["codes"]:lay["codes"] + 2 * M * K].view(torch.float16).view(M, K).clone()
        codes = codes16.to(torch.int8)
    status = int(ws[lay["status"]:lay["status"] + 4].view(torch.int32).item())
    return dict(row_scale=row_scale, codes=codes, codes_fp16=codes16, outliers=idx,
                outlier_count=count, status=status)


INF = math.inf
