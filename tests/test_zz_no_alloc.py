"""The allocation-free entry point (llmint8_matmul_noalloc) gives the same results
as llmint8_matmul.

It serves callers that cannot allocate device memory when they run the matmul
(latency-critical loops that must not risk the synchronization of
cudaMalloc/cudaFree, or hosts whose device memory belongs to another
allocator): its scratch space is a static device array inside the library
instead of a caller workspace.  Two calls in a row
check that the second call is not disturbed by what the first one left in the
shared array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_quantization_matmul_row_b300 import _lib, api, synthetic
from parity import y_close

pytestmark = pytest.mark.gpu


def _noalloc_via_c_abi(X, t, Wq, sw, W16, Y):
    lib = _lib.load()
    P = ctypes.c_void_p
    M, K = X.shape
    N = Wq.shape[0]
    st = lib.llmint8_matmul_noalloc(P(X.data_ptr()), M, K, N, float(t), P(Wq.data_ptr()), P(sw.data_ptr()),
                                    P(W16.data_ptr()) if W16 is not None else None, P(Y.data_ptr()),
                                    P(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.OK, lib.llmint8_status_str(st)
    return Y


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (16, 4096, 4096), (300, 1088, 400)])
def test_noalloc_matches_workspace_entry_point_two_calls(M, K, N):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    W, _ = synthetic.make_w(K, N, seed=M + N)
    Wd = torch.from_numpy(W).to(dev)
    Wq, sw = api.llmint8_quantize_weight(Wd)
    for call in range(2):
        X, _ = synthetic.make_x(M, K, frac=0.01 * (call + 1), min_count=3, seed=900 + call)
        Xd = torch.from_numpy(X).to(dev)
        Y_ref = api.llmint8_matmul(Xd, 6.0, Wq, sw, Wd)
        Y = torch.empty((M, N), dtype=torch.float16, device=dev)
        _noalloc_via_c_abi(Xd, 6.0, Wq, sw, Wd, Y)
        torch.cuda.synchronize()
        ok, ratio = y_close(Y.cpu().numpy(), Y_ref.cpu().numpy())
        assert ok, f"call {call}: worst error/tolerance {ratio:.3g}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    M, K, N = 2048, 4096, 4096  # needs far more than the 8 MiB scratch
    X = torch.zeros((M, K), dtype=torch.float16, device=dev)
    Wq = torch.zeros((N, K), dtype=torch.int8, device=dev)
    sw = torch.zeros((N,), dtype=torch.float32, device=dev)
    Y = torch.full((M, N), 7.0, dtype=torch.float16, device=dev)
    lib = _lib.load()
    P = ctypes.c_void_p
    st = lib.llmint8_matmul_noalloc(P(X.data_ptr()), M, K, N, float("inf"), P(Wq.data_ptr()), P(sw.data_ptr()),
                                    None, P(Y.data_ptr()), None)
    assert st == _lib.EWORKSPACE
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())  # nothing was enqueued
