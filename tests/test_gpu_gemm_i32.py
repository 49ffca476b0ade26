"""llmint8_gemm_i32: the exact int32 product C = Xq . Wq^T of codes the caller
chooses, through the same kernels the matmul runs (int8 GEMV for M <= 16, the
tensor-core GEMM on exact fp16 codes above), compared bit for bit with the
oracle's int64 product (A3; "Lightning Fabric 8-bit" page, section 2.2:
int8 x int8 accumulated in int32).

The codes are built to stress the tensor-core path's exactness argument: the
fp32 TMEM accumulator of one 1024-long chunk must hold every partial sum
exactly.  Inside each chunk a run of 521 same-sign 127*127 products takes the
partial sum past 2^23 (8,403,209), where an fp32 value has no fraction bits
left, and the remaining products are +-1: an accumulator narrower than fp32 (or
one that rounded anywhere on the way) would drop some of them.  A second
pattern swings the partial sum between large positive and negative values in
runs, a third fills a whole chunk with 127*127 (16,516,096, just under 2^24).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantization_matmul_row_b300 import api

pytestmark = pytest.mark.gpu

CHUNK = 1024


def _signs(rng, shape):
    return np.where(rng.random(shape) < 0.5, -1, 1).astype(np.int8)


def prefix_then_units(M, N, K, seed):
    """Per chunk: 521 products of +-127*127 (sign fixed per row and column), then +-1 products."""
    rng = np.random.default_rng(seed)
    Xq = _signs(rng, (M, K))
    Wq = _signs(rng, (N, K))
    rs = _signs(rng, (M, 1))
    cs = _signs(rng, (N, 1))
    for c0 in range(0, K, CHUNK):
        run = slice(c0, min(K, c0 + 521))
        Xq[:, run] = 127 * rs
        Wq[:, run] = 127 * cs
    return Xq, Wq


def alternating_runs(M, N, K, seed):
    """Runs of 127*127 products whose sign flips run by run, separated by +-1 products."""
    rng = np.random.default_rng(seed)
    Xq = _signs(rng, (M, K))
    Wq = _signs(rng, (N, K))
    k, sign = 0, 1
    while k < K:
        r = int(rng.integers(50, 300))
        Xq[:, k:k + r] = 127
        Wq[:, k:k + r] = 127 * sign
        k += r
        gap = int(rng.integers(1, 40))
        k += gap  # +-1 products in between
        sign = -sign
    return Xq, Wq


def full_chunks(M, N, K, seed):
    """Every product 127*127 except a few +-1: chunk sums just under 2^24."""
    rng = np.random.default_rng(seed)
    Xq = np.full((M, K), 127, np.int8)
    Wq = np.full((N, K), 127, np.int8)
    for c0 in range(0, K, CHUNK):
        Xq[:, c0] = _signs(rng, (M,))
        Wq[:, c0] = 1
    return Xq, Wq


def random_codes(M, N, K, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(-127, 128, size=(M, K)).astype(np.int8),
            rng.integers(-127, 128, size=(N, K)).astype(np.int8))


def run(Xq, Wq):
    dev = torch.device("cuda")
    C = api.llmint8_gemm_i32(torch.from_numpy(Xq).to(dev), torch.from_numpy(Wq).to(dev))
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("M", [1, 16, 17, 256, 300])
@pytest.mark.parametrize("pattern", [prefix_then_units, alternating_runs, full_chunks])
def test_adversarial_codes_exact(pattern, M):
    K, N = 4096, 512
    Xq, Wq = pattern(M, N, K, seed=M)
    ref = oracle.int8_matmul(Xq, Wq.T)
    assert np.abs(ref).max() < 2 ** 31
    C = run(Xq, Wq)
    assert np.array_equal(C, ref), f"{int((C != ref).sum())} of {C.size} entries differ"


def test_prefix_pattern_really_crosses_2_23():
    # the premise of the test above: some chunk partial sums lie in [2^23, 2^24)
    Xq, Wq = prefix_then_units(4, 4, 1024, seed=1)
    prods = Xq[0].astype(np.int64) * Wq[0].astype(np.int64)
    partial = np.abs(np.cumsum(prods))
    assert partial.max() >= 2 ** 23 and partial.max() < 2 ** 24
    Xq, Wq = full_chunks(2, 2, 1024, seed=1)
    assert 2 ** 23 < abs(int(Xq[0].astype(np.int64) @ Wq[0].astype(np.int64))) < 2 ** 24


@pytest.mark.parametrize("M,K,N", [(1, 64, 16), (9, 1040, 144), (17, 64, 256), (300, 1088, 400), (130, 65536, 32)])
def test_random_codes_exact(M, K, N):
    Xq, Wq = random_codes(M, N, K, seed=M + K + N)
    assert np.array_equal(run(Xq, Wq), oracle.int8_matmul(Xq, Wq.T))


def test_matches_llmint8_matmul_i32_on_its_own_codes():
    # the codes the X pass derives, fed back through the caller-code entry point
    from bit_quantization_matmul_row_b300 import synthetic
    M, K, N = 200, 2112, 512
    X, _ = synthetic.make_x(M, K, frac=0.01, min_count=3, seed=5)
    W, _ = synthetic.make_w(K, N, seed=6)
    dev = torch.device("cuda")
    Xd, Wd = torch.from_numpy(X).to(dev), torch.from_numpy(W).to(dev)
    Wq, sw = api.llmint8_quantize_weight(Wd)
    Xq = torch.empty((M, K), dtype=torch.int8, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    api.llmint8_quantize_x(Xd, 6.0, Xq, sx)
    C1 = api.llmint8_matmul_i32(Xd, 6.0, Wq, sw)
    C2 = api.llmint8_gemm_i32(Xq, Wq)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
