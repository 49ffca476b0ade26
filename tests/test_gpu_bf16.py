"""bfloat16 inputs and output (llmint8_matmul_bf16) against the oracle's bf16 mode,
element by element (needs a B300): weight codes and scales, the X-pass results
and the int32 accumulator bit-exact, Y within 1e-3 max|Y_ref| + 1 bf16 ulp."""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_quantization_matmul_row_b300 import api, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16).cuda()


def _values(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16).double().numpy()


def _bf16_ulp(y):
    a = np.abs(np.asarray(y, np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)


def check_bf16(M, K, N, t, frac=0.01, seed=0):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=3 if frac else 0, seed=seed, fmt="bf16")
    W, _ = synthetic.make_w(K, N, seed=seed, fmt="bf16")
    Xd, Wd = _dev(X), _dev(W)
    Wq, sw = api.llmint8_quantize_weight_bf16(Wd)
    ws = api.make_workspace(M, K, N, Xd.device)
    Y = api.llmint8_matmul_bf16(Xd, t, Wq, sw, Wd, workspace=ws)
    inter = api.read_intermediates(ws, M, K, N)
    C = api.llmint8_matmul_i32_bf16(Xd, t, Wq, sw, workspace=api.make_workspace(M, K, N, Xd.device))
    torch.cuda.synchronize()
    assert api.llmint8_device_status(ws) == 0
    ref = oracle.llmint8_matmul(X, W, t, fmt="bf16")
    assert np.array_equal(Wq.cpu().numpy(), ref["Wq"].T), "weight codes"
    assert np.array_equal(sw.cpu().numpy(), ref["s_w"]), "column scales"
    assert np.array_equal(inter["outliers"].cpu().numpy(), ref["outliers"]), "outlier set"
    assert np.array_equal(inter["row_scale"].cpu().numpy(), ref["s_x"]), "row scales"
    assert np.array_equal(inter["codes"].cpu().numpy(), ref["Xq"]), "X codes"
    assert np.array_equal(C.cpu().numpy().astype(np.int64), ref["C"]), "int32 accumulator"
    y = Y.view(torch.int16).cpu().numpy().view(np.uint16)
    yv, rv = _values(y), _values(ref["Y"])
    tol = 1e-3 * np.max(np.abs(rv)) + _bf16_ulp(rv)
    assert np.all(np.abs(yv - rv) <= tol), float(np.max(np.abs(yv - rv) / tol))
    return ref


@pytest.mark.parametrize("M", [1, 4, 9, 16])
def test_bf16_decode(M):
    check_bf16(M, 1040, 144, 6.0, seed=M)


def test_bf16_decode_persistent_tiles():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    check_bf16(4, 1088, 16 * (2 * sms + 30), 6.0, frac=0.02, seed=5)


@pytest.mark.parametrize("M,K,N", [(100, 1088, 400), (300, 2112, 512), (256, 8192, 256)])
def test_bf16_prefill(M, K, N):
    check_bf16(M, K, N, 6.0, seed=M + K)


@pytest.mark.parametrize("M", [2, 140])
def test_bf16_special_thresholds(M):
    ref = check_bf16(M, 512, 256, math.inf, seed=60 + M)
    assert ref["outliers"].size == 0
    ref = check_bf16(M, 512, 256, 0.0, frac=0.0, seed=70 + M)  # every nonzero column an outlier
    assert not ref["C"].any()


def test_bf16_range_beyond_fp16():
    # bf16 keeps values fp16 cannot hold (|x| > 65504): outliers of 1e6 and
    # weights of 1e-6 still give the exact codes and a finite, close Y
    M, K, N = 8, 512, 128
    X, _ = synthetic.make_x(M, K, frac=0.0, seed=80, fmt="bf16")
    X[:, 7] = synthetic.to_bf16_bits(np.full(M, 1.0e6, np.float32))
    W, _ = synthetic.make_w(K, N, sigma=1e-6, seed=80, fmt="bf16")
    Xd, Wd = _dev(X), _dev(W)
    Wq, sw = api.llmint8_quantize_weight_bf16(Wd)
    Y = api.llmint8_matmul_bf16(Xd, 6.0, Wq, sw, Wd)
    torch.cuda.synchronize()
    ref = oracle.llmint8_matmul(X, W, 6.0, fmt="bf16")
    assert 7 in ref["outliers"]
    yv, rv = _values(Y.view(torch.int16).cpu().numpy().view(np.uint16)), _values(ref["Y"])
    assert np.all(np.isfinite(yv))
    tol = 1e-3 * np.max(np.abs(rv)) + _bf16_ulp(rv)
    assert np.all(np.abs(yv - rv) <= tol)
