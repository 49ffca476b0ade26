"""CUDA path vs the CPU oracle, element by element (needs a B300).

Sizes span several tiles and ragged tails of both kernels: the decode GEMV
(M <= 16, 16-column CTAs, K split over 8 warps, exact int32 every 1024 K) and
the tensor-core GEMM (128 x 256 tiles, 64-wide K steps, 1024-long exact
chunks, the outlier slice as a final fp32 chunk).
"""
import math

import numpy as np
import pytest
import torch

from bit_quantization_matmul_row_b300 import api, synthetic
from parity import check, run_gpu, sample_cols, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


def xw(M, K, N, frac=0.01, seed=0, sigma=0.02, mag=(20.0, 60.0), min_count=0):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=min_count, mag=mag, seed=seed)
    W, _ = synthetic.make_w(K, N, sigma=sigma, seed=seed)
    return X, W


# ------------------------------------------------------------------ small, full compare

def test_tiny_config():
    case = synthetic.tiny()[0]
    X, planted = case.x()
    W, _ = case.w()
    g, ref = check(X, W, case.threshold)
    assert set(planted.tolist()) <= set(g["outliers"].tolist())


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_decode_ragged(M):
    # K = 1040: 17 steps of 64 split over 8 warps (ragged last warp, last step 16 wide)
    X, W = xw(M, 1040, 144, frac=0.01, seed=10 + M, min_count=3)
    check(X, W, 6.0)


@pytest.mark.parametrize("M,K,N", [(1, 16384, 272), (2, 8192, 144), (5, 2048, 400), (16, 65536, 32)])
def test_decode_long_k(M, K, N):
    # long rows: many 64-wide steps per warp (ring wrap-around), K = 65536 is the
    # largest accepted (|C| up to 127^2 * 65536 < 2^31)
    X, W = xw(M, K, N, frac=0.01, seed=M * K, min_count=3)
    check(X, W, 6.0)


@pytest.mark.parametrize("M,K,extra_tiles,frac", [
    (1, 1040, 1, 0.01),      # one CTA takes a second tile
    (8, 4096, 150, 0.002),   # two tiles for half the CTAs; the 8-step ring wraps across tiles
    (4, 1040, 400, 0.09),    # ragged K (warps 6, 7 have no steps), ~94 outliers: past the staged chunk
    (1, 64, 600, 0.05),      # one K step: only warp 0 streams; three or four tiles per CTA
    (4, 11008, 40, 0.001),
    (16, 1040, 400, 0.05),   # more than 8 rows: one-tile CTAs in several waves
    (1, 2048, 150, 0.2),     # ~410 outliers: the persistent GEMV stages six more chunks per tile
    (8, 1040, 200, 0.45),    # ~470 outliers, the last chunk partial
])
def test_decode_many_tiles(M, K, extra_tiles, frac):
    # More 16-column tiles than two CTAs per SM.  Up to 8 rows of X this is the
    # persistent GEMV (each CTA walks several tiles, its ring running on across
    # them); compared in full.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = 16 * (2 * sms + extra_tiles)
    X, W = xw(M, K, N, frac=frac, seed=M * 7 + extra_tiles, min_count=3)
    check(X, W, 6.0)
    if extra_tiles == 1:
        check(X, W, 6.0, int8_variant=True)  # no outlier slice (threshold +inf)


@pytest.mark.parametrize("M,frac", [(1, 0.3), (4, 0.45), (16, 0.4)])
def test_decode_outlier_chunks(M, frac):
    # 300-500 outlier columns: more than one 256-column chunk of the fp16 slice
    # in the GEMV epilogue, the last one partial
    X, W = xw(M, 1040, 144, frac=frac, seed=M + 700)
    g, ref = check(X, W, 6.0)
    assert 256 < len(g["outliers"]) < 512


@pytest.mark.parametrize("M,K,N", [(17, 64, 256), (130, 272, 272), (300, 1088, 400), (256, 2112, 512),
                                   (100, 4160, 384), (200, 3136, 1040), (64, 1024, 4096)])
def test_prefill_ragged(M, K, N):
    # ragged M tiles, ragged N tiles (N % 256 != 0), K not a multiple of 64,
    # K crossing the 1024-long exact chunk boundary; the last three: medium M on
    # 128-wide one-CTA and pair tiles over several exact chunks
    X, W = xw(M, K, N, frac=0.02, seed=M + K + N, min_count=2)
    check(X, W, 6.0)


@pytest.mark.parametrize("M", [4, 200])
def test_int8_variant(M):
    X, W = xw(M, 1088, 272, frac=0.02, seed=30 + M)
    check(X, W, math.inf, int8_variant=True)
    # t = +inf through the general entry point is the same computation
    check(X, W, math.inf)


@pytest.mark.parametrize("M", [5, 150])
def test_threshold_zero_all_outliers(M):
    # every nonzero column is an outlier: the int8 part is empty and the fp16
    # slice covers all of K (many 64-wide outlier steps on the GEMM path)
    X, W = xw(M, 1088, 272, frac=0.0, seed=40 + M)
    X[:, 7] = 0
    g, ref = check(X, W, 0.0)
    assert len(g["outliers"]) == 1087
    assert not g["codes"].any() and not g["C"].any()


@pytest.mark.parametrize("M", [2, 140])
def test_negative_threshold(M):
    X, W = xw(M, 256, 256, frac=0.0, seed=50 + M)
    X[:, 3] = 0
    g, ref = check(X, W, -1.0)
    assert len(g["outliers"]) == 256
    assert not g["s_x"].any()


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_rounding_ties_go_away_from_zero(M):
    # Row absmax 127 makes the scale factor exactly 1, so x = k + 1/2 are exact
    # ties of the code rounding: they must go away from zero (decode path for
    # M = 1, 4, 16; tensor-core path for 64).
    K, N = 1024, 64
    rng = np.random.default_rng(M)
    X = (rng.integers(-127, 127, size=(M, K)) + 0.5).astype(np.float16)
    X[:, 0] = 127
    W, _ = synthetic.make_w(K, N, seed=M)
    g, ref = check(X, W, 200.0)
    x = X.astype(np.float64)
    expect = (np.sign(x) * np.floor(np.abs(x) + 0.5)).astype(np.int8)
    assert np.array_equal(g["codes"].astype(np.int8), expect)


@pytest.mark.parametrize("M", [1, 4, 16, 200])
@pytest.mark.parametrize("t", [6.0, 6.001])
def test_threshold_boundary_values(M, t):
    # |x| > t is strict: a column whose largest |x| equals t (or is the fp16
    # value just below a non-representable t) stays in the int8 part; the next
    # fp16 value above t makes it an outlier column.
    K, N = 512, 64
    X, W = xw(M, K, N, frac=0.0, seed=M)
    at = np.float16(6.0)                      # == t, or just below 6.001
    above = np.float16(6.00390625)            # next fp16 above 6.0 (and above 6.001)
    X[M - 1, 10], X[0, 20], X[M // 2, 30] = at, -above, above
    X[0, 40] = -at
    g, ref = check(X, W, t)
    assert set(g["outliers"].tolist()) == {20, 30}


@pytest.mark.parametrize("M", [2, 16, 256])
def test_exactness_beyond_fp32_integer_range(M):
    # All codes +-127 and K = 8192: |C| reaches 127^2 * 8192 = 132,124,672 > 2^24,
    # so any accumulation in plain fp32 beyond 1024 products would round.
    K, N = 8192, 256
    rng = np.random.default_rng(M)
    X = np.ones((M, K), np.float16)
    X[1::2, K // 2:] = -1            # odd rows change sign halfway
    W = np.full((K, N), 0.02, np.float16)
    W[:, 1::3] = -0.02
    signs = rng.choice([-1.0, 1.0], size=(K, 8)).astype(np.float16)
    W[:, -8:] = signs * np.float16(0.02)  # random signs: large cancellations
    g, ref = check(X, W, 6.0)
    assert np.abs(g["C"]).max() == 127 * 127 * K


def test_zero_rows_and_columns():
    X, W = xw(40, 512, 256, frac=0.01, seed=60)
    X[3] = 0
    W[:, 5] = 0
    g, ref = check(X, W, 6.0)
    assert g["s_x"][3] == 0 and g["s_w"][5] == 0
    assert not g["Y"][:, 5].any()


@pytest.mark.parametrize("M", [7, 129])
def test_workspace_contents_do_not_matter(M):
    X, W = xw(M, 512, 256, seed=70 + M)
    a = run_gpu(X, W, 6.0, want_i32=False)
    b = run_gpu(X, W, 6.0, want_i32=False, garbage_workspace=True)
    assert np.array_equal(a["Y"].view(np.uint16), b["Y"].view(np.uint16))


@pytest.mark.parametrize("M,K,N", [(1, 4096, 11008), (16, 4096, 4096), (300, 1088, 400)])
def test_workspace_reused_by_consecutive_calls(M, K, N):
    # Back-to-back calls on one stream and one workspace with different X: the
    # kernels of a call overlap (programmatic dependent launch), so a read of the
    # previous call's codes, scales or outlier list would give a wrong Y here.
    import oracle
    from parity import y_close
    W, _ = synthetic.make_w(K, N, seed=K + N)
    dev = torch.device("cuda")
    Wd = torch.from_numpy(W).to(dev)
    Wq, sw = api.llmint8_quantize_weight(Wd)
    ws = api.make_workspace(M, K, N, dev)
    Xs = [synthetic.make_x(M, K, frac=0.005 * (j + 1), min_count=2 + 3 * j, seed=500 + j)[0] for j in range(3)]
    Ys = []
    for X in Xs:
        Ys.append(api.llmint8_matmul(torch.from_numpy(X).to(dev), 6.0, Wq, sw, Wd, workspace=ws))
    torch.cuda.synchronize()
    assert api.llmint8_device_status(ws) == 0
    wq = oracle.quantize_weight(W)
    for X, Y in zip(Xs, Ys):
        ref = oracle.llmint8_matmul(X, W, 6.0, wq=wq)
        ok, ratio = y_close(Y.cpu().numpy(), ref["Y"])
        assert ok, ratio


@pytest.mark.parametrize("M", [16, 300])
def test_deterministic_and_stream(M):
    X, W = xw(M, 1088, 400, seed=80 + M)
    a = run_gpu(X, W, 6.0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run_gpu(X, W, 6.0, stream=s)
    s.synchronize()
    for k in ("Y", "C", "codes", "s_x"):
        assert np.array_equal(a[k], b[k]), k


def test_bounded_wait_reports_timeout():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.llmint8_selftest_timeout(ws, 1000)
    assert api.llmint8_device_status(ws) == 5  # LLMINT8_ETIMEOUT, read and cleared
    assert api.llmint8_device_status(ws) == 0
    # the context is still usable afterwards
    X, W = xw(16, 256, 256, seed=90)
    check(X, W, 6.0)


# ------------------------------------------------------------------ full-size workloads
# X-pass outputs compared in full; weight codes on sampled columns; C and Y on
# sampled rows x columns (the oracle computes those one by one).  Same entry points and launch configuration
# as the benchmark.

def _full_case(case, nrows=24, ncols=96):
    X, planted = case.x()
    W, _ = case.w()
    rows = sample_rows(case.M, nrows, seed=case.seed)
    cols = sample_cols(case.N, ncols, seed=case.seed)
    g, ref = check(X, W, case.threshold, rows=rows, cols=cols)
    assert set(planted.tolist()) <= set(g["outliers"].tolist())


@pytest.mark.parametrize("case", synthetic.decode_7b(), ids=lambda c: c.name)
def test_decode_7b(case):
    _full_case(case)


@pytest.mark.parametrize("case", synthetic.prefill_7b(), ids=lambda c: c.name)
def test_prefill_7b(case):
    _full_case(case)


@pytest.mark.parametrize("case", synthetic.ffn_13b(), ids=lambda c: c.name)
def test_ffn_13b(case):
    _full_case(case, nrows=16)


SWEEP = [c for c in synthetic.sweep_70b()
         if (c.N == 28672 and c.frac in (0.0, 0.001, 0.05)) or (c.N == 8192 and c.frac == 0.01)]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: c.name)
def test_sweep_70b(case):
    _full_case(case, nrows=12)


@pytest.mark.parametrize("M,K,N", [(4, 4096, 512), (512, 2048, 512)])
def test_decomposition_beats_plain_int8_on_outlier_inputs(M, K, N):
    # With outlier columns present, the LLM.int8() result (threshold 6) is several
    # times closer to the exact product than plain vector-wise int8 (threshold
    # +inf) computed by the same kernels: the claim the pages make for the method.
    X, W = xw(M, K, N, frac=0.01, seed=M + 900, min_count=4)
    exact = X.astype(np.float64) @ W.astype(np.float64)
    g6 = run_gpu(X, W, 6.0, want_i32=False)
    gi = run_gpu(X, W, math.inf, want_i32=False)
    err = lambda Y: np.linalg.norm(Y.astype(np.float64) - exact) / np.linalg.norm(exact)
    assert err(g6["Y"]) * 4 < err(gi["Y"])
