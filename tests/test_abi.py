"""The C-ABI library loads and exports every entry point include/llmint8.h
declares; host-side argument checks return their documented status before any
device work (no GPU needed)."""
import ctypes
import math
import os
import re

import pytest

from bit_quantization_matmul_row_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "llmint8.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(llmint8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and nothing from torch crosses the boundary: plain C symbols
    out = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), name


def test_status_strings(lib):
    for code in range(7):
        assert lib.llmint8_status_str(code).decode().startswith("LLMINT8")
    assert b"unknown" in lib.llmint8_status_str(99)


def test_workspace_bytes(lib):
    assert lib.llmint8_workspace_bytes(0, 64, 64) == 0
    assert lib.llmint8_workspace_bytes(16, 70000, 64) == 0
    small = lib.llmint8_workspace_bytes(16, 4096, 4096)
    big = lib.llmint8_workspace_bytes(2048, 4096, 4096)
    assert small > 0 and small % 16 == 0
    # prefill adds the gathered outlier operands: M*Kp + N*Kp fp16
    assert big >= 2048 * 4096 * 2 * 2 + 4096 * 4096 * 2


def test_workspace_layout(lib):
    off = (ctypes.c_size_t * 5)()
    assert lib.llmint8_workspace_layout(300, 1088, 400, off) == _lib.OK
    vals = list(off)
    assert vals[0] == 0 and vals[1] == 4
    assert vals[2] < vals[3] < vals[4]
    assert all(v % 4 == 0 for v in vals)
    assert vals[4] + 300 * 1088 * 2 <= lib.llmint8_workspace_bytes(300, 1088, 400)
    assert lib.llmint8_workspace_layout(0, 16, 16, off) == _lib.EINVAL


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails its checks first


def _mm(lib, M=32, K=64, N=64, t=6.0, X=FAKE, Wq=FAKE, sw=FAKE, w16=FAKE, Y=FAKE, ws=FAKE, wsb=None):
    if wsb is None:
        wsb = 1 << 40
    P = ctypes.c_void_p
    return lib.llmint8_matmul(P(X), M, K, N, t, P(Wq), P(sw), P(w16), P(Y), P(ws), wsb, None)


def test_matmul_argument_errors(lib):
    assert _mm(lib, M=0) == _lib.EINVAL
    assert _mm(lib, K=0) == _lib.EINVAL
    assert _mm(lib, N=-16) == _lib.EINVAL
    assert _mm(lib, t=math.nan) == _lib.EINVAL
    assert _mm(lib, X=0) == _lib.EINVAL
    assert _mm(lib, w16=0) == _lib.EINVAL            # finite threshold needs W16
    assert _mm(lib, Wq=0) == _lib.EINVAL
    assert _mm(lib, K=72) == _lib.EALIGN
    assert _mm(lib, N=40) == _lib.EALIGN
    assert _mm(lib, X=FAKE + 8) == _lib.EALIGN
    assert _mm(lib, ws=0) == _lib.EWORKSPACE
    assert _mm(lib, wsb=16) == _lib.EWORKSPACE


def test_int8_variant_needs_no_w16(lib):
    P = ctypes.c_void_p
    # argument checks pass up to the workspace check: W16 is not required
    st = lib.llmint8_matmul_int8(P(FAKE), 32, 64, 64, P(FAKE), P(FAKE), P(FAKE), P(FAKE), 16, None)
    assert st == _lib.EWORKSPACE


def test_quantize_weight_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.llmint8_quantize_weight(P(0), 64, 64, P(FAKE), P(FAKE), None) == _lib.EINVAL
    assert lib.llmint8_quantize_weight(P(FAKE), 0, 64, P(FAKE), P(FAKE), None) == _lib.EINVAL
    assert lib.llmint8_quantize_weight(P(FAKE), 65, 64, P(FAKE), P(FAKE), None) == _lib.EALIGN
    assert lib.llmint8_quantize_weight(P(FAKE), 64, 64, P(FAKE + 4), P(FAKE), None) == _lib.EALIGN


def test_noalloc_argument_errors(lib):
    P = ctypes.c_void_p
    # shapes whose workspace exceeds the static 8 MiB scratch are rejected on the host
    assert lib.llmint8_matmul_noalloc(P(FAKE), 4096, 8192, 8192, 6.0, P(FAKE), P(FAKE), P(FAKE),
                                      P(FAKE), None) == _lib.EWORKSPACE
    assert lib.llmint8_matmul_noalloc(P(FAKE), 0, 64, 64, 6.0, P(FAKE), P(FAKE), P(FAKE),
                                      P(FAKE), None) == _lib.EINVAL


def _chain(lib, M=1, K=4096, N=4096, t=6.0, sin=0, w16=FAKE, nt=6.0, sout=FAKE + 4096, Y=FAKE, wsb=1 << 40,
           sinb=1 << 30, soutb=1 << 30):
    P = ctypes.c_void_p
    return lib.llmint8_matmul_chain(P(FAKE), M, K, N, t, P(sin) if sin else None, sinb, P(FAKE), P(FAKE),
                                    P(w16) if w16 else None, P(Y), nt, P(sout) if sout else None, soutb, P(FAKE),
                                    wsb, None)


def test_chain_state_layout(lib):
    assert lib.llmint8_chain_state_bytes(5, 64) == 0
    assert lib.llmint8_chain_state_bytes(1, 40) == 0
    n = lib.llmint8_chain_state_bytes(4, 11008)
    off = (ctypes.c_size_t * 3)()
    assert lib.llmint8_chain_state_layout(4, 11008, off) == _lib.OK
    flags, parts, total = off[0], off[1], off[2]
    assert flags == 256 and parts >= flags + 11008 and parts % 256 == 0
    assert total == n == parts + (11008 // 16) * 4 * 4
    assert lib.llmint8_chain_state_layout(0, 16, off) == _lib.EINVAL


def test_chain_argument_errors(lib):
    assert _chain(lib, M=5) == _lib.EUNSUPPORTED        # more than 4 rows
    assert _chain(lib, K=256) == _lib.EUNSUPPORTED      # shorter than one 512-wide ring stage
    assert _chain(lib, M=4, K=65536) == _lib.EUNSUPPORTED  # codes do not fit in shared memory
    assert _chain(lib, sin=FAKE + 4096) == _lib.EINVAL  # state in == state out
    assert _chain(lib, nt=math.nan) == _lib.EINVAL
    assert _chain(lib, w16=0) == _lib.EINVAL            # outliers possible, no fp16 weight
    assert _chain(lib, sin=FAKE + 8) == _lib.EALIGN
    assert _chain(lib, t=math.nan) == _lib.EINVAL
    assert _chain(lib, wsb=16) == _lib.EWORKSPACE
    # state buffers smaller than the states the call reads or writes
    need_in = lib.llmint8_chain_state_bytes(1, 4096)
    assert _chain(lib, sin=FAKE + (1 << 20), sinb=need_in - 16) == _lib.EINVAL
    assert _chain(lib, N=11008, soutb=lib.llmint8_chain_state_bytes(1, 11008) - 1) == _lib.EINVAL
    P = ctypes.c_void_p
    assert lib.llmint8_matmul_chain_i32(P(FAKE), 1, 4096, 4096, 6.0, None, 0, P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                        6.0, None, 0, None, P(FAKE), 1 << 40, None) == _lib.EINVAL  # no C
    assert lib.llmint8_matmul_chain_i32(P(FAKE), 1, 4096, 4096, 6.0, None, 0, P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                        6.0, None, 0, P(FAKE + 4), P(FAKE), 1 << 40, None) == _lib.EALIGN


def test_matmul_host_argument_errors(lib):
    P = ctypes.c_void_p
    ws = lib.llmint8_workspace_bytes(4, 64, 64)
    call = lambda xh=FAKE, yh=FAKE, Y=FAKE, M=4, wsb=ws: lib.llmint8_matmul_host(
        P(xh) if xh else None, P(FAKE), M, 64, 64, 6.0, P(FAKE), P(FAKE), P(FAKE), P(Y) if Y else None,
        P(yh) if yh else None, P(FAKE), wsb, None)
    assert call(xh=0) == _lib.EINVAL
    assert call(yh=0) == _lib.EINVAL
    assert call(Y=0) == _lib.EINVAL
    assert call(M=0) == _lib.EINVAL
    assert call(wsb=16) == _lib.EWORKSPACE


def test_quantize_x_and_read_outliers_argument_errors(lib):
    P = ctypes.c_void_p
    ws = lib.llmint8_workspace_bytes(4, 64, 16)
    q = lambda X=FAKE, M=4, K=64, t=6.0, Xq=FAKE, rs=FAKE, wsb=ws: lib.llmint8_quantize_x(
        P(X) if X else None, M, K, t, P(Xq) if Xq else None, P(rs) if rs else None, P(FAKE), wsb, None)
    assert q(X=0) == _lib.EINVAL
    assert q(M=0) == _lib.EINVAL
    assert q(K=70000) == _lib.EINVAL
    assert q(t=math.nan) == _lib.EINVAL
    assert q(Xq=0) == _lib.EINVAL
    assert q(rs=0) == _lib.EINVAL
    assert q(K=72) == _lib.EALIGN
    assert q(Xq=FAKE + 8) == _lib.EALIGN
    assert q(wsb=ws - 16) == _lib.EWORKSPACE
    n = ctypes.c_int(0)
    r = lib.llmint8_read_outliers
    assert r(None, 64, ctypes.byref(n), None, 0, None) == _lib.EINVAL
    assert r(P(FAKE), 64, None, None, 0, None) == _lib.EINVAL
    assert r(P(FAKE), 0, ctypes.byref(n), None, 0, None) == _lib.EINVAL
    assert r(P(FAKE), 70000, ctypes.byref(n), None, 0, None) == _lib.EINVAL
    assert r(P(FAKE), 64, ctypes.byref(n), None, -1, None) == _lib.EINVAL
    assert r(P(FAKE), 64, ctypes.byref(n), None, 4, None) == _lib.EINVAL  # capacity without a buffer


def test_selftest_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.llmint8_selftest_timeout(P(0), 10, None) == _lib.EINVAL
    assert lib.llmint8_selftest_timeout(P(FAKE), 0, None) == _lib.EINVAL
    assert lib.llmint8_selftest_timeout(P(FAKE), 10 ** 8, None) == _lib.EINVAL


def test_kernels_per_call(lib):
    inf = float("inf")
    k = lib.llmint8_kernels_per_call
    # short decode rows (K <= 4096): the row-quantization cluster finds the
    # outlier columns itself, then the GEMV
    for M, K in ((1, 16), (1, 4096), (4, 4096), (9, 64), (16, 4096)):
        assert k(M, K, 4096, 6.0, 0) == 2, (M, K)
        assert k(M, K, 4096, 6.0, 1) == 2
        assert k(M, K, 4096, inf, 0) == 2
    # longer decode rows: outlier scan + row quantization + GEMV
    for M, K in ((1, 4112), (1, 16384), (16, 11008), (16, 65536)):
        assert k(M, K, 4096, 6.0, 0) == 3, (M, K)
        assert k(M, K, 4096, inf, 0) == 2       # no outlier scan
    # prefill: scan + row quantization (which also gathers the outlier rows of W16
    # when rows have at most 4096 columns and its M/8 CTAs cover the N/16 column
    # groups 8 at a time) + widening of the codes + GEMM
    assert k(2048, 4096, 4096, 6.0, 0) == 4
    assert k(2048, 4096, 11008, 6.0, 0) == 4
    assert k(17, 4096, 4096, 6.0, 0) == 5       # 3 row CTAs: separate gather of the outlier rows of W16
    assert k(17, 4112, 4096, 6.0, 0) == 5       # rows too long for the fused gather
    assert k(17, 4096, 4096, 6.0, 1) == 4       # the int32 result leaves out the fp16 slice
    assert k(17, 4096, 4096, inf, 0) == 3
    assert k(0, 64, 64, 6.0, 0) == -1
    assert k(1, 64, 64, math.nan, 0) == -1


def test_w8_argument_errors(lib):
    from bit_quantization_matmul_row_b300 import _lib
    P = ctypes.c_void_p
    ws = lib.llmint8_workspace_bytes(16, 64, 64)
    args = lambda W16c, rmap, rows: (P(FAKE), 16, 64, 64, 6.0, P(FAKE), P(FAKE), W16c, rmap, rows,
                                     P(FAKE), P(FAKE), ws, None)
    assert lib.llmint8_matmul_w8(*args(None, None, -1)) == _lib.EINVAL
    assert lib.llmint8_matmul_w8(*args(None, P(FAKE), 4)) == _lib.EINVAL   # rows kept, no W16c
    assert lib.llmint8_matmul_w8(*args(P(FAKE + 4), P(FAKE), 4)) == _lib.EALIGN
    assert lib.llmint8_pack_w16_rows(None, 64, 64, None, 0, None, P(FAKE), None) == _lib.EINVAL
    assert lib.llmint8_pack_w16_rows(P(FAKE), 64, 64, None, 3, P(FAKE), P(FAKE), None) == _lib.EINVAL
    assert lib.llmint8_pack_w16_rows(P(FAKE), 64, 40, None, 0, None, P(FAKE), None) == _lib.EALIGN


def test_bf16_argument_errors(lib):
    from bit_quantization_matmul_row_b300 import _lib
    P = ctypes.c_void_p
    assert lib.llmint8_quantize_weight_bf16(P(0), 64, 64, P(FAKE), P(FAKE), None) == _lib.EINVAL
    assert lib.llmint8_quantize_weight_bf16(P(FAKE), 65, 64, P(FAKE), P(FAKE), None) == _lib.EALIGN
    ws = lib.llmint8_workspace_bytes(16, 64, 64)
    assert lib.llmint8_matmul_bf16(P(FAKE), 16, 64, 64, 6.0, P(FAKE), P(FAKE), None, P(FAKE), P(FAKE), ws,
                                   None) == _lib.EINVAL  # finite threshold without W16


def test_gemm_i32_argument_errors(lib):
    P = ctypes.c_void_p
    ws = lib.llmint8_workspace_bytes(32, 64, 64)
    call = lambda xq=FAKE, wq=FAKE, C=FAKE, M=32, K=64, N=64, w=FAKE, wsb=ws: lib.llmint8_gemm_i32(
        P(xq) if xq else None, P(wq) if wq else None, M, K, N, P(C) if C else None, P(w) if w else None, wsb, None)
    assert call(xq=0) == _lib.EINVAL
    assert call(wq=0) == _lib.EINVAL
    assert call(C=0) == _lib.EINVAL
    assert call(M=0) == _lib.EINVAL
    assert call(K=40) == _lib.EALIGN
    assert call(N=24) == _lib.EALIGN
    assert call(xq=FAKE + 4) == _lib.EALIGN
    assert call(w=0) == _lib.EWORKSPACE
    assert call(wsb=ws - 16) == _lib.EWORKSPACE
    # the workspace the matmul of the same shape needs is enough (decode and prefill)
    for M in (1, 16, 17, 300):
        assert lib.llmint8_workspace_bytes(M, 1088, 400) > 0
