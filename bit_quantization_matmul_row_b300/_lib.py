"""ctypes declarations of the C ABI in include/llmint8.h (no logic here)."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libllmint8.so")

# status codes (llmint8_status)
OK, EINVAL, EALIGN, EWORKSPACE, ECUDA, ETIMEOUT, EUNSUPPORTED = range(7)
DECODE_MAX_M = 16
WS_FIELDS = ("status", "outlier_count", "outlier_idx", "row_scale", "codes")

EXPORTS = (
    "llmint8_status_str",
    "llmint8_quantize_weight",
    "llmint8_workspace_bytes",
    "llmint8_matmul",
    "llmint8_matmul_host",
    "llmint8_matmul_int8",
    "llmint8_matmul_w8",
    "llmint8_pack_w16_rows",
    "llmint8_quantize_weight_bf16",
    "llmint8_matmul_bf16",
    "llmint8_matmul_i32_bf16",
    "llmint8_matmul_i32",
    "llmint8_gemm_i32",
    "llmint8_xpass",
    "llmint8_gemm",
    "llmint8_chain_state_bytes",
    "llmint8_chain_state_layout",
    "llmint8_matmul_chain",
    "llmint8_matmul_chain_i32",
    "llmint8_quantize_x",
    "llmint8_read_outliers",
    "llmint8_matmul_noalloc",
    "llmint8_kernels_per_call",
    "llmint8_workspace_layout",
    "llmint8_device_status",
    "llmint8_selftest_timeout",
)

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libllmint8.so (built in-tree).  Raises if it has not been built."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m bit_quantization_matmul_row_b300.build` "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.llmint8_status_str.argtypes = [I]
        lib.llmint8_status_str.restype = ctypes.c_char_p
        lib.llmint8_quantize_weight.argtypes = [P, I, I, P, P, P]
        lib.llmint8_workspace_bytes.argtypes = [I, I, I]
        lib.llmint8_workspace_bytes.restype = Z
        lib.llmint8_matmul.argtypes = [P, I, I, I, F, P, P, P, P, P, Z, P]
        lib.llmint8_matmul_host.argtypes = [P, P, I, I, I, F, P, P, P, P, P, P, Z, P]
        lib.llmint8_matmul_int8.argtypes = [P, I, I, I, P, P, P, P, Z, P]
        lib.llmint8_matmul_w8.argtypes = [P, I, I, I, F, P, P, P, P, I, P, P, Z, P]
        lib.llmint8_pack_w16_rows.argtypes = [P, I, I, P, I, P, P, P]
        lib.llmint8_quantize_weight_bf16.argtypes = [P, I, I, P, P, P]
        lib.llmint8_matmul_bf16.argtypes = [P, I, I, I, F, P, P, P, P, P, Z, P]
        lib.llmint8_matmul_i32_bf16.argtypes = [P, I, I, I, F, P, P, P, P, Z, P]
        lib.llmint8_matmul_i32.argtypes = [P, I, I, I, F, P, P, P, P, Z, P]
        lib.llmint8_gemm_i32.argtypes = [P, P, I, I, I, P, P, Z, P]
        lib.llmint8_xpass.argtypes = [P, I, I, I, F, P, Z, P]
        lib.llmint8_gemm.argtypes = [P, I, I, I, F, P, P, P, P, P, Z, P]
        lib.llmint8_matmul_noalloc.argtypes = [P, I, I, I, F, P, P, P, P, P]
        lib.llmint8_chain_state_bytes.argtypes = [I, I]
        lib.llmint8_chain_state_bytes.restype = Z
        lib.llmint8_chain_state_layout.argtypes = [I, I, ctypes.POINTER(Z)]
        lib.llmint8_matmul_chain.argtypes = [P, I, I, I, F, P, Z, P, P, P, P, F, P, Z, P, Z, P]
        lib.llmint8_matmul_chain_i32.argtypes = [P, I, I, I, F, P, Z, P, P, P, P, F, P, Z, P, P, Z, P]
        lib.llmint8_quantize_x.argtypes = [P, I, I, F, P, P, P, Z, P]
        lib.llmint8_read_outliers.argtypes = [P, I, ctypes.POINTER(I), P, I, P]
        lib.llmint8_kernels_per_call.argtypes = [I, I, I, F, I]
        lib.llmint8_kernels_per_call.restype = I
        lib.llmint8_workspace_layout.argtypes = [I, I, I, ctypes.POINTER(Z)]
        lib.llmint8_device_status.argtypes = [P, P]
        lib.llmint8_selftest_timeout.argtypes = [P, I, P]
        for f in ("llmint8_quantize_weight", "llmint8_matmul", "llmint8_matmul_host", "llmint8_matmul_int8", "llmint8_matmul_i32",
                  "llmint8_gemm_i32",
                  "llmint8_matmul_w8", "llmint8_pack_w16_rows", "llmint8_quantize_weight_bf16",
                  "llmint8_matmul_bf16", "llmint8_matmul_i32_bf16",
                  "llmint8_xpass", "llmint8_gemm", "llmint8_matmul_noalloc", "llmint8_chain_state_layout",
                  "llmint8_matmul_chain", "llmint8_matmul_chain_i32", "llmint8_quantize_x",
                  "llmint8_read_outliers", "llmint8_workspace_layout", "llmint8_device_status", "llmint8_selftest_timeout"):
            getattr(lib, f).restype = I
        _lib = lib
        return lib
