"""The boundary's stand-alone steps against the CPU oracle (needs a B300).

llmint8_quantize_x writes A1 + A2 into caller buffers: its int8 codes and row
scales, and the outlier set read back with llmint8_read_outliers, must equal the
oracle's bit for bit ("LLM.int8() paper walkthrough", sections 2.1 and 2.3).
The same quantities derived inside the decode chain kernel from a chain state
(codes, row scales, outlier set, and the exact int32 accumulator of A3) must
equal the oracle's too.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantization_matmul_row_b300 import api, synthetic
from parity import y_close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@pytest.mark.parametrize("M,K,frac,t", [
    (1, 4096, 0.001, 6.0),      # one clustered row-quantization launch
    (16, 11008, 0.001, 6.0),    # outlier scan + one CTA per row
    (300, 4096, 0.01, 6.0),     # one warp per row (the prefill X pass), int8 codes
    (40, 5136, 0.05, 6.0),      # long rows, ragged
    (8, 1024, 0.0, float("inf")),
    (3, 256, 0.2, 0.0),         # every nonzero column an outlier
])
def test_quantize_x_matches_the_oracle(M, K, frac, t):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=2 if frac else 0, seed=M + 3 * K)
    Xd = torch.from_numpy(X).cuda()
    Xq, sx, ws = api.llmint8_quantize_x(Xd, t)
    out = api.llmint8_read_outliers(ws, K)
    is_out = oracle.outlier_columns(X, t)
    q_ref, sx_ref = oracle.quantize_rows(X, is_out)
    assert np.array_equal(out, oracle.outlier_indices(is_out))
    assert np.array_equal(sx.cpu().numpy(), np.asarray(sx_ref, np.float32))
    assert np.array_equal(Xq.cpu().numpy(), q_ref)


def test_read_outliers_capacity_and_garbage():
    M, K = 4, 2048
    X, _ = synthetic.make_x(M, K, frac=0.005, min_count=8, seed=5)
    Xd = torch.from_numpy(X).cuda()
    _, _, ws = api.llmint8_quantize_x(Xd, 6.0)
    full = api.llmint8_read_outliers(ws, K)
    assert full.size >= 8
    # a bounded copy: the count is the true count, only `capacity` indices are written
    import ctypes
    from bit_quantization_matmul_row_b300 import _lib
    n = ctypes.c_int(0)
    buf = np.full(3, -7, np.int32)
    st = _lib.load().llmint8_read_outliers(ws.data_ptr(), K, ctypes.byref(n), buf.ctypes.data_as(ctypes.c_void_p), 3,
                                           None)
    assert st == _lib.OK and n.value == full.size
    assert np.array_equal(buf, full[:3])
    # a workspace whose stored count is impossible for this K is rejected
    ws.fill_(0xFF)
    with pytest.raises(api.LLMInt8Error):
        api.llmint8_read_outliers(ws, K)


def _state_from_oracle(X, t):
    M, K = X.shape
    is_out = oracle.outlier_columns(X, t)
    _, s_x = oracle.quantize_rows(X, is_out)
    flags_off, parts_off, total = api.llmint8_chain_state_layout(M, K)
    b = np.zeros(total, np.uint8)
    b[:12] = np.array([M, K, 1], np.int32).view(np.uint8)
    b[12:16] = np.array([t], np.float32).view(np.uint8)
    b[flags_off:flags_off + K] = is_out.astype(np.uint8)
    b[parts_off:parts_off + 4 * M] = np.asarray(s_x, np.float32).view(np.uint8)
    return torch.from_numpy(b).cuda()


@pytest.mark.parametrize("M,K,N,frac", [
    (1, 4096, 4096, 0.001),
    (4, 11008, 4096, 0.001),
    (3, 1040, 16 * 130, 0.05),  # ragged K (last ring stage partly outside K)
    (4, 784, 48, 0.3),          # > 64 outliers: past the lanes' registers
])
def test_chain_with_state_derives_the_oracle_codes(M, K, N, frac):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=3, seed=M * 11 + K)
    W, _ = synthetic.make_w(K, N, seed=K + 7 * N)
    Wd = torch.from_numpy(W).cuda()
    Wq, sw = api.llmint8_quantize_weight(Wd)
    ws = api.make_workspace(M, K, N)
    ws.fill_(0x5A)
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    Y = api.llmint8_matmul_chain(torch.from_numpy(X).cuda(), float("nan"), _state_from_oracle(X, 6.0), Wq, sw, Wd,
                                 workspace=ws, C=C)
    torch.cuda.synchronize()
    assert api.llmint8_device_status(ws) == 0
    ref = oracle.llmint8_matmul(X, W, 6.0)
    inter = api.read_intermediates(ws, M, K, N)
    assert np.array_equal(inter["outliers"].cpu().numpy(), oracle.outlier_indices(ref["is_outlier"]))
    assert np.array_equal(inter["row_scale"].cpu().numpy(), np.asarray(ref["s_x"], np.float32))
    assert np.array_equal(inter["codes"].cpu().numpy(), ref["Xq"])
    assert np.array_equal(C.cpu().numpy().astype(np.int64), ref["C"])
    ok, ratio = y_close(Y.cpu().numpy(), ref["Y"])
    assert ok, f"worst error/tolerance {ratio:.3g}"


def test_chain_rejects_a_state_of_another_shape():
    # a hand-built state whose header names another K: nothing is read past the
    # header, Y stays untouched and the error word says EINVAL
    M, K, N = 2, 1024, 256
    X, _ = synthetic.make_x(M, K, frac=0.0, min_count=0, seed=1)
    W, _ = synthetic.make_w(K, N, seed=2)
    Wd = torch.from_numpy(W).cuda()
    Wq, sw = api.llmint8_quantize_weight(Wd)
    for hdr in ([M, 2 * K, 1], [M + 1, K, 1], [M, K, 0], [M, K, K // 16 + 1]):
        S = _state_from_oracle(X, 6.0)
        S[:12] = torch.from_numpy(np.array(hdr, np.int32).view(np.uint8)).cuda()
        Y = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
        ws = api.make_workspace(M, K, N)
        api.llmint8_matmul_chain(torch.from_numpy(X).cuda(), 6.0, S, Wq, sw, Wd, Y=Y, workspace=ws)
        assert api.llmint8_device_status(ws) == 1, hdr  # LLMINT8_EINVAL
        assert bool((Y == 7.0).all()), hdr
    # and the same workspace works again afterwards
    Y = api.llmint8_matmul_chain(torch.from_numpy(X).cuda(), 6.0, _state_from_oracle(X, 6.0), Wq, sw, Wd, workspace=ws)
    assert api.llmint8_device_status(ws) == 0
    ok, _ = y_close(Y.cpu().numpy(), oracle.llmint8_matmul(X, W, 6.0)["Y"])
    assert ok


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (16, 11008, 4096), (300, 1088, 400)])
def test_matmul_host_equals_the_device_call(M, K, N):
    # host X in, host Y out, one call: the same kernels as llmint8_matmul, so the same bits
    X, _ = synthetic.make_x(M, K, frac=0.001, min_count=4, seed=M + K)
    W, _ = synthetic.make_w(K, N, seed=N)
    Wd = torch.from_numpy(W).cuda()
    Wq, sw = api.llmint8_quantize_weight(Wd)
    Xh = torch.from_numpy(X).pin_memory()
    Xd = torch.empty((M, K), dtype=torch.float16, device="cuda")
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    Yh = torch.empty((M, N), dtype=torch.float16).pin_memory()
    ws = api.make_workspace(M, K, N)
    api.llmint8_matmul_host(Xh, Xd, 6.0, Wq, sw, Wd, Y, Yh, ws)
    torch.cuda.synchronize()
    Yref = api.llmint8_matmul(torch.from_numpy(X).cuda(), 6.0, Wq, sw, Wd)
    torch.cuda.synchronize()
    assert torch.equal(Yh, Yref.cpu())
    ok, _ = y_close(Yh.numpy(), oracle.llmint8_matmul(X, W, 6.0)["Y"])
    assert ok
