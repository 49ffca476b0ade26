"""The outlier slice without a full fp16 copy of W (llmint8_matmul_w8), against
the oracle's kept-rows mode, element by element (needs a B300)."""
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


def _rows(keep, X, K, t):
    out = np.flatnonzero(oracle.outlier_columns(X, t))
    if keep == "none":
        return np.array([], np.int32)
    if keep == "some":  # every other outlier row plus a few rows that are not outliers
        return np.unique(np.concatenate([out[::2], [0, K // 2, K - 1]])).astype(np.int32)
    return np.arange(K, dtype=np.int32)


def _run(M, K, N, keep, frac, seed):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=3, seed=seed)
    W, _ = synthetic.make_w(K, N, seed=seed)
    dev = torch.device("cuda")
    Xd, Wd = torch.from_numpy(X).to(dev), torch.from_numpy(W).to(dev)
    Wq, sw = api.llmint8_quantize_weight(Wd)
    rows = _rows(keep, X, K, 6.0)
    W16c, row_map = api.llmint8_pack_w16_rows(Wd, torch.from_numpy(rows).to(dev))
    ws = api.make_workspace(M, K, N, dev)
    Y = api.llmint8_matmul_w8(Xd, 6.0, Wq, sw, W16c, row_map, workspace=ws)
    torch.cuda.synchronize()
    assert api.llmint8_device_status(ws) == 0
    ref = oracle.llmint8_matmul(X, W, 6.0, w16_rows=rows)
    ok, ratio = y_close(Y.cpu().numpy(), ref["Y"])
    assert ok, ratio
    return X, Xd, Wd, Wq, sw, Y


@pytest.mark.parametrize("M,K,N,keep,frac", [
    (1, 1040, 144, "none", 0.01),      # decode, one-tile GEMV
    (4, 1040, 144, "some", 0.09),      # ~94 outliers: more than one staged chunk
    (16, 4096, 272, "some", 0.005),
    (300, 1088, 400, "none", 0.02),    # prefill, CTA pairs
    (300, 1088, 400, "some", 0.02),
    (100, 2112, 512, "some", 0.02),    # prefill, one-CTA tiles
])
def test_w8_against_oracle(M, K, N, keep, frac):
    _run(M, K, N, keep, frac, seed=M + K + N)


@pytest.mark.parametrize("M,keep,frac", [(2, "none", 0.05), (8, "some", 0.05), (4, "some", 0.2)])
def test_w8_persistent_gemv(M, keep, frac):
    # more 16-column tiles than two CTAs per SM: the persistent GEMV stages the
    # outlier rows tile by tile (frac 0.2: ~218 outliers, several chunks per tile,
    # kept and dequantized rows mixed)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _run(M, 1088, 16 * (2 * sms + 60), keep, frac, seed=300 + M)


@pytest.mark.parametrize("M", [3, 200])
def test_w8_with_every_row_kept_is_llmint8_matmul(M):
    X, Xd, Wd, Wq, sw, Y = _run(M, 1088, 272, "all", 0.02, seed=400 + M)
    Yf = api.llmint8_matmul(Xd, 6.0, Wq, sw, Wd)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), Yf.view(torch.int16))


def test_pack_w16_rows_map_and_out_of_range_rows():
    K, N = 64, 32
    W = (np.arange(K * N, dtype=np.float32).reshape(K, N) / 100).astype(np.float16)
    Wd = torch.from_numpy(W).cuda()
    rows = torch.tensor([3, K + 5, 7], dtype=torch.int32, device="cuda")
    W16c, row_map = api.llmint8_pack_w16_rows(Wd, rows)
    torch.cuda.synchronize()
    m = row_map.cpu().numpy()
    expect = np.full(K, -1, np.int32)
    expect[3], expect[7] = 0, 2
    assert np.array_equal(m, expect)
    c = W16c.cpu().numpy()
    assert np.array_equal(c[0], W[3]) and np.array_equal(c[2], W[7]) and not c[1].any()
