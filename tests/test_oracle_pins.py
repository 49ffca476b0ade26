"""Pins for the CPU oracle: what the pages and the mathematics fix, independent of
the oracle's own code.

Each test is chosen so that a plausible mistake in the oracle (a dropped term, a
wrong sign, a wrong index, a transposed operand, a different rounding rule)
fails at least one of them:

* the worked example of the pitfalls guide (section 2), stored under tests/golden;
* a tie case that separates round-half-away-from-zero from half-to-even;
* the strict "exceeds the threshold" boundary (paper walkthrough, section 2.3);
* brute-force loops and library routines (numpy matmul, numpy fp16 casts);
* the special cases t = 0 (everything is an outlier: the plain fp16 matmul) and
  t = +inf (no outliers: pure vector-wise int8, bounded by the quantization
  error), and a 1x1x1 closed form.
"""
import math
import os

import numpy as np
import pytest

from bit_quantization_matmul_row_b300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = [float(t) for t in v.split()]
    return out


def fp16_ulp(y):
    """Spacing of fp16 numbers at |y| (subnormal spacing below 2^-14)."""
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


# ---------------------------------------------------------------------------------
# fp16 conversions against numpy (an independent library implementation)
# ---------------------------------------------------------------------------------

def test_half_to_double_all_bit_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


def test_double_to_half_matches_numpy(oracle_mod):
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        # exact midpoints between neighbouring fp16 values (ties to even)
        (np.arange(-3000, 3000).astype(np.float16).astype(np.float64) + 0.5),
        np.array([65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -24, 2.0 ** -25,
                  1.5 * 2.0 ** -25, 2.0 ** -14 * (1 - 2.0 ** -11), -0.0, 0.0]),
    ])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.double_to_half(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------------
# The worked example (pitfalls guide, section 2)
# ---------------------------------------------------------------------------------

def test_worked_example_as_weight_column(oracle_mod):
    g = _read_golden("worked_example.txt")
    W = np.array(g["values"], np.float16).reshape(4, 1)
    Wq, sw = oracle_mod.quantize_weight(W)
    assert Wq[:, 0].tolist() == [int(c) for c in g["codes"]]
    assert sw[0] == 12.0
    sf = oracle_mod.scale_factor(sw[0])
    assert round(sf, 2) == g["scale_factor_2dp"][0]
    deq = [round(q / sf, 2) for q in Wq[:, 0]]
    assert deq == g["dequantized_2dp"]


def test_worked_example_as_activation_row_no_outliers(oracle_mod):
    g = _read_golden("worked_example.txt")
    X = np.array(g["values"], np.float16).reshape(1, 4)
    is_out = oracle_mod.outlier_columns(X, math.inf)
    assert not is_out.any()
    Xq, sx = oracle_mod.quantize_rows(X, is_out)
    assert Xq[0].tolist() == [int(c) for c in g["codes"]]
    assert sx[0] == 12.0


def test_worked_example_with_threshold_six(oracle_mod):
    # Same row under the default threshold: 12.0 > 6 makes column 3 an outlier.
    # The row absmax is then |-0.4| (fp16 0.39990234375); by hand:
    # 0.0999755859375/0.39990234375 = 0.25 exactly -> 31.75 -> 32;
    # 0.300048828125/0.39990234375 * 127 = 95.29 -> 95; -0.4 -> -127; outlier -> 0.
    X = np.array([[0.1, 0.3, -0.4, 12.0]], np.float16)
    is_out = oracle_mod.outlier_columns(X, 6.0)
    assert is_out.tolist() == [False, False, False, True]
    Xq, sx = oracle_mod.quantize_rows(X, is_out)
    assert Xq[0].tolist() == [32, 95, -127, 0]
    assert sx[0] == np.float32(np.float16(0.4))


# ---------------------------------------------------------------------------------
# Rounding rule, clamp and code range
# ---------------------------------------------------------------------------------

def test_round_half_away_from_zero(oracle_mod):
    # absmax 254 -> scale factor 127/254 = 0.5 exactly, so x*sf = x/2 and odd x
    # lands exactly on a half: RHAZ gives [127, 1, 3, -3, -1];
    # half-to-even would give [127, 0, 2, -2, 0].
    X = np.array([[254.0, 1.0, 5.0, -5.0, -1.0]], np.float16)
    Xq, sx = oracle_mod.quantize_rows(X, np.zeros(5, bool))
    assert oracle_mod.scale_factor(sx[0]) == 0.5
    assert Xq[0].tolist() == [127, 1, 3, -3, -1]


def test_code_range_and_argmax(oracle_mod):
    X, planted = synthetic.make_x(64, 512, frac=0.01, min_count=4, seed=7)
    is_out = oracle_mod.outlier_columns(X, 6.0)
    Xq, sx = oracle_mod.quantize_rows(X, is_out)
    assert Xq.min() >= -127 and Xq.max() <= 127
    assert np.all(Xq[:, is_out] == 0)
    xa = np.abs(X.astype(np.float32))
    xa[:, is_out] = -1
    arg = np.argmax(xa, axis=1)
    assert np.all(np.abs(Xq[np.arange(64), arg]) == 127)
    # dequantization error of each kept value is at most half a step (plus fp32 slack)
    deq = Xq.astype(np.float64) * sx[:, None].astype(np.float64) / 127.0
    err = np.abs(deq - X.astype(np.float64))[:, ~is_out]
    assert np.all(err <= sx[:, None].astype(np.float64) * (1 / 254 + 1e-6))


def test_zero_scale(oracle_mod):
    X = np.zeros((2, 8), np.float16)
    X[1, 3] = 50.0  # row 1: its only nonzero is an outlier -> absmax over the rest is 0
    is_out = oracle_mod.outlier_columns(X, 6.0)
    Xq, sx = oracle_mod.quantize_rows(X, is_out)
    assert sx.tolist() == [0.0, 0.0]
    assert not Xq.any()
    W = np.zeros((8, 3), np.float16)
    W[:, 1] = 0.5
    Wq, sw = oracle_mod.quantize_weight(W)
    assert sw.tolist() == [0.0, 0.5, 0.0]
    assert Wq[:, 0].tolist() == [0] * 8 and Wq[:, 1].tolist() == [127] * 8


# ---------------------------------------------------------------------------------
# Outlier set: strict threshold, brute force, generator's planted columns
# ---------------------------------------------------------------------------------

def test_threshold_boundary_is_strict(oracle_mod):
    nxt = float(np.nextafter(np.float16(6.0), np.float16(7.0)))  # 6.00390625
    X = np.zeros((3, 4), np.float16)
    X[0, 0] = 6.0
    X[1, 1] = -6.0
    X[2, 2] = nxt
    X[0, 3] = -nxt
    assert oracle_mod.outlier_columns(X, 6.0).tolist() == [False, False, True, True]


def test_outlier_set_brute_force(oracle_mod):
    rng = np.random.default_rng(3)
    X = (rng.standard_normal((9, 37)) * 4).astype(np.float16)
    for t in (0.0, 1.5, 6.0, 9.0, math.inf):
        brute = sorted({j for i in range(9) for j in range(37) if abs(float(X[i, j])) > t})
        got = oracle_mod.outlier_indices(oracle_mod.outlier_columns(X, t)).tolist()
        assert got == brute


def test_row_absmax_excludes_outlier_columns(oracle_mod):
    X = np.array([[1.0, -2.0, 50.0, 0.5],
                  [3.0, 0.25, -40.0, -1.0]], np.float16)
    is_out = oracle_mod.outlier_columns(X, 6.0)
    Xq, sx = oracle_mod.quantize_rows(X, is_out)
    assert sx.tolist() == [2.0, 3.0]
    assert Xq[:, 2].tolist() == [0, 0]
    assert Xq[0].tolist() == [64, -127, 0, 32]  # 63.5 -> 64 (RHAZ), 31.75 -> 32


@pytest.mark.parametrize("case", synthetic.tiny() + synthetic.decode_7b()[:3])
def test_planted_columns_are_found(oracle_mod, case):
    X, planted = case.x()
    is_out = oracle_mod.outlier_columns(X, case.threshold)
    found = set(np.flatnonzero(is_out).tolist())
    assert set(planted.tolist()) <= found
    # N(0,1) draws exceed 6 with probability ~2e-9: strays are rare
    assert len(found) - len(planted) <= 2


# ---------------------------------------------------------------------------------
# Integer matmul and fp16 outlier matmul
# ---------------------------------------------------------------------------------

def test_int8_matmul_brute_force(oracle_mod):
    rng = np.random.default_rng(5)
    A = rng.integers(-127, 128, (5, 7)).astype(np.int8)
    B = rng.integers(-127, 128, (7, 3)).astype(np.int8)
    C = oracle_mod.int8_matmul(A, B, nthreads=2)
    for i in range(5):
        for n in range(3):
            acc = 0
            for k in range(7):
                acc += int(A[i, k]) * int(B[k, n])
            assert C[i, n] == acc


def test_int8_matmul_matches_numpy_and_extremes(oracle_mod):
    rng = np.random.default_rng(6)
    A = rng.integers(-127, 128, (33, 300)).astype(np.int8)
    B = rng.integers(-127, 128, (300, 21)).astype(np.int8)
    assert np.array_equal(oracle_mod.int8_matmul(A, B, 3), A.astype(np.int64) @ B.astype(np.int64))
    K = 20000  # all +-127: |C| = 127^2 * K = 322,580,000 (beyond fp32's exact range)
    A = np.full((2, K), 127, np.int8)
    A[1] = -127
    B = np.full((K, 2), 127, np.int8)
    B[: K // 2, 1] = -127
    C = oracle_mod.int8_matmul(A, B, 1)
    assert C.tolist() == [[16129 * K, 0], [-16129 * K, 0]]


def test_outlier_matmul_matches_numpy(oracle_mod):
    rng = np.random.default_rng(8)
    X = (rng.standard_normal((17, 64)) * 3).astype(np.float16)
    W = (rng.standard_normal((64, 11)) * 0.1).astype(np.float16)
    is_out = np.zeros(64, bool)
    is_out[[3, 10, 63]] = True
    F = oracle_mod.outlier_matmul(X, W, is_out, 2)
    ref = X[:, is_out].astype(np.float64) @ W[is_out].astype(np.float64)
    assert np.allclose(F, ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------------
# Special cases of the whole path
# ---------------------------------------------------------------------------------

def test_threshold_zero_is_the_fp16_matmul(oracle_mod):
    # Every column holding a nonzero value is an outlier, so the int8 part is
    # empty and Y is the fp16 product of X and W (the all-zero columns add 0).
    X, _ = synthetic.make_x(12, 96, seed=11)
    X[:, 5] = 0
    W, _ = synthetic.make_w(96, 40, seed=11)
    r = oracle_mod.llmint8_matmul(X, W, 0.0)
    assert r["outliers"].size == 95 and 5 not in r["outliers"]
    assert not r["C"].any()
    ref = (X.astype(np.float64) @ W.astype(np.float64)).astype(np.float16)
    diff = np.abs(r["Y"].astype(np.float64) - ref.astype(np.float64))
    assert np.all(diff <= fp16_ulp(ref))


@pytest.mark.parametrize("t", [math.inf, 6.0])
def test_quantization_error_bound(oracle_mod, t):
    # Y - X.W = sum_{k not in O} (e_x w + x^ e_w) with |e_x| <= s_x/254, |e_w| <= s_w/254
    # (plus fp32 slack and the final fp16 rounding).  A transposed operand, a wrong
    # scale index or a missing 1/127^2 breaks this bound by orders of magnitude.
    X, _ = synthetic.make_x(24, 200, frac=0.02, seed=12)
    W, _ = synthetic.make_w(200, 72, seed=12)
    r = oracle_mod.llmint8_matmul(X, W, t)
    keep = ~r["is_outlier"]
    if t == math.inf:
        assert keep.all()
    else:
        assert (~keep).sum() >= 4
    Xd, Wd = X.astype(np.float64), W.astype(np.float64)
    xhat = r["Xq"].astype(np.float64) * r["s_x"][:, None].astype(np.float64) / 127
    sx = r["s_x"].astype(np.float64)[:, None]
    sw = r["s_w"].astype(np.float64)[None, :]
    slack = 1 / 254 + 1e-6
    bound = (sx * slack) * np.abs(Wd[keep]).sum(0)[None, :] + (np.abs(xhat[:, keep]).sum(1)[:, None]) * sw * slack
    ref = Xd @ Wd
    err = np.abs(r["Y"].astype(np.float64) - ref)
    assert np.all(err <= bound + fp16_ulp(ref) + 1e-12)
    # the bound is not vacuous: the decomposition is accurate to a few percent
    assert np.max(err) < 0.05 * np.max(np.abs(ref))


def test_one_by_one_closed_form(oracle_mod):
    # M=K=N=1, t=inf: both codes are +-127, C = +-16129, and the merge gives
    # 16129*|x|*|w|/16129 = x*w exactly in double, so Y = fp16(x*w).
    rng = np.random.default_rng(13)
    for _ in range(200):
        x = np.float16(rng.standard_normal() * 3)
        w = np.float16(rng.standard_normal() * 0.05)
        if x == 0 or w == 0:
            continue
        r = oracle_mod.llmint8_matmul(np.array([[x]]), np.array([[w]]), math.inf)
        assert abs(int(r["Xq"][0, 0])) == 127 and abs(int(r["Wq"][0, 0])) == 127
        assert r["Y"][0, 0] == np.float16(np.float64(x) * np.float64(w))


def test_row_subset_matches_full(oracle_mod):
    case = synthetic.tiny()[0]
    X, _ = case.x()
    W, _ = case.w()
    full = oracle_mod.llmint8_matmul(X, W, 6.0)
    rows = np.array([0, 5, 15])
    sub = oracle_mod.llmint8_matmul(X, W, 6.0, rows=rows)
    assert np.array_equal(sub["Y"].view(np.uint16), full["Y"][rows].view(np.uint16))
    assert np.array_equal(sub["C"], full["C"][rows])


# ---------------------------------------------------------------------------
# Ablation (not a step of the path): per-tensor scales and plain int8 without the
# outlier decomposition, the schemes the pages contrast LLM.int8() with.

def test_per_tensor_codes_closed_form(oracle_mod):
    # one scale for the whole tensor: absmax 4 -> factor 127/4 = 31.75;
    # 2 -> 63.5 -> 64 (tie away from zero), -1 -> -31.75 -> -32, 0.5 -> 15.875 -> 16
    X = np.array([[2.0, -1.0], [0.5, 4.0]], np.float16)
    q, s = oracle_mod.quantize_per_tensor(X)
    assert s == np.float32(4.0)
    assert q.tolist() == [[64, -32], [16, 127]]


@pytest.mark.parametrize("M,K,N,frac,seed", [(64, 1024, 256, 0.01, 1), (16, 4096, 256, 0.001, 2),
                                             (128, 2048, 256, 0.05, 3)])
def test_outliers_break_plain_int8_but_not_the_decomposition(oracle_mod, M, K, N, frac, seed):
    # The pitfalls guide's table and the paper walkthrough: without outlier handling
    # int8 loses much more accuracy than LLM.int8(); coarser (per-tensor) scales
    # lose more still.  Relative Frobenius error against the exact product.
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=4, seed=seed)
    W, _ = synthetic.make_w(K, N, seed=seed)
    exact = X.astype(np.float64) @ W.astype(np.float64)
    err = lambda Y: np.linalg.norm(Y.astype(np.float64) - exact) / np.linalg.norm(exact)
    e_llm = err(oracle_mod.llmint8_matmul(X, W, 6.0)["Y"])
    e_naive = err(oracle_mod.llmint8_matmul(X, W, math.inf)["Y"])
    e_tensor = err(oracle_mod.per_tensor_int8_matmul(X, W))
    assert e_llm * 4 < e_naive < e_tensor
    assert e_llm < 0.02


def test_without_outliers_the_decomposition_is_plain_int8(oracle_mod):
    X, _ = synthetic.make_x(32, 1024, frac=0.0, seed=4)
    W, _ = synthetic.make_w(1024, 512, seed=4)
    assert not oracle_mod.outlier_columns(X, 6.0).any()
    y_llm = oracle_mod.llmint8_matmul(X, W, 6.0)["Y"]
    y_naive = oracle_mod.llmint8_matmul(X, W, math.inf)["Y"]
    assert np.array_equal(y_llm.view(np.uint16), y_naive.view(np.uint16))
    exact = X.astype(np.float64) @ W.astype(np.float64)
    err = lambda Y: np.linalg.norm(Y.astype(np.float64) - exact) / np.linalg.norm(exact)
    assert err(y_naive) <= err(oracle_mod.per_tensor_int8_matmul(X, W))


# ---------------------------------------------------------------------------------
# A4 without a full fp16 copy of W: dequantized int8 weight rows
# ---------------------------------------------------------------------------------

def test_dequantized_weight_matches_worked_example(oracle_mod):
    # The page dequantizes the codes [1, 3, -4, 127] of scale 12 back to the
    # printed [0.09, 0.28, -0.38, 12.0]; the dequantized weight rows follow the
    # same rule (code times absmax / 127).
    g = _read_golden("worked_example.txt")
    W = np.array(g["values"], np.float16).reshape(4, 1)
    Wq, sw = oracle_mod.quantize_weight(W)
    w_hat = oracle_mod.dequantize_weight(Wq, sw)[:, 0].astype(np.float64)
    assert [round(v, 2) for v in w_hat] == g["dequantized_2dp"]


def test_dequantized_weight_error_bound_and_argmax(oracle_mod):
    # Each dequantized weight is within half a code step (absmax / 254) plus one
    # fp16 rounding of the original value, and the row holding a column's
    # absmax dequantizes back to exactly that fp16 value (code +-127).
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((256, 96)) * 0.02).astype(np.float16)
    W[:, 5] = 0
    W[7, 9] = 3.0
    Wq, sw = oracle_mod.quantize_weight(W)
    w_hat = oracle_mod.dequantize_weight(Wq, sw).astype(np.float64)
    w = W.astype(np.float64)
    bound = sw.astype(np.float64)[None, :] / 254.0 + fp16_ulp(w_hat) / 2 + 1e-12
    assert np.all(np.abs(w_hat - w) <= bound)
    arg = np.argmax(np.abs(w), axis=0)
    cols = np.arange(w.shape[1])
    nz = sw > 0
    assert np.array_equal(w_hat[arg[nz], cols[nz]], w[arg[nz], cols[nz]])
    assert not w_hat[:, 5].any()  # zero column: scale 0, weights 0


def test_all_rows_kept_in_fp16_is_the_standard_path(oracle_mod):
    rng = np.random.default_rng(12)
    X = rng.standard_normal((9, 192)).astype(np.float16)
    X[:, [3, 70, 150]] *= 30
    W = (rng.standard_normal((192, 64)) * 0.02).astype(np.float16)
    full = oracle_mod.llmint8_matmul(X, W, 6.0)
    kept = oracle_mod.llmint8_matmul(X, W, 6.0, w16_rows=np.arange(192))
    assert np.array_equal(full["Y"].view(np.uint16), kept["Y"].view(np.uint16))
    assert np.array_equal(full["F"], kept["F"])
    # Only the outlier slice depends on which rows are kept: no rows kept
    # changes F (the weights of the outlier rows become their dequantized codes)
    # and leaves the int8 part alone.
    none = oracle_mod.llmint8_matmul(X, W, 6.0, w16_rows=np.array([], np.int64))
    assert np.array_equal(none["C"], full["C"]) and np.array_equal(none["s_x"], full["s_x"])
    assert not np.array_equal(none["F"], full["F"])
    # without outliers the mode changes nothing
    a = oracle_mod.llmint8_matmul(X, W, math.inf)
    b = oracle_mod.llmint8_matmul(X, W, math.inf, w16_rows=np.array([], np.int64))
    assert np.array_equal(a["Y"].view(np.uint16), b["Y"].view(np.uint16))


# ---------------------------------------------------------------------------------
# bfloat16 inputs and output (the same method on bf16 X, W, Y)
# ---------------------------------------------------------------------------------

def _bf16_values(bits):
    """bf16 bit patterns -> float64 values through torch (an independent library)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def bf16_ulp(y):
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def test_bf16_to_double_all_bit_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = _bf16_values(bits)
    got = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    finite = ~np.isnan(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


def test_double_to_bf16_matches_torch(oracle_mod):
    import torch
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000),
        # exact midpoints between neighbouring bf16 values (ties to even)
        (_bf16_values(np.arange(0, 30000, 7, dtype=np.uint16)) * (1 + 2.0 ** -8)).astype(np.float32),
        np.array([3.3895314e38, 3.4e38, 1e-40, 9.2e-41, -0.0, 0.0], np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.double_to_bf16(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_worked_example_in_bf16(oracle_mod):
    # The pitfalls guide's four values rounded to bf16 still give its codes, its
    # scale and its printed dequantized values.
    g = _read_golden("worked_example.txt")
    bits = synthetic.to_bf16_bits(np.array(g["values"], np.float32)).reshape(4, 1)
    Wq, sw = oracle_mod.quantize_weight(bits, "bf16")
    assert Wq[:, 0].tolist() == [int(c) for c in g["codes"]]
    assert sw[0] == 12.0
    deq = oracle_mod.dequantize_weight(Wq, sw, "bf16")[:, 0]
    assert [round(float(v), 2) for v in _bf16_values(deq)] == g["dequantized_2dp"]


def test_bf16_threshold_zero_is_the_bf16_matmul(oracle_mod):
    X, _ = synthetic.make_x(12, 96, seed=21, fmt="bf16")
    X[:, 5] = 0
    W, _ = synthetic.make_w(96, 40, seed=21, fmt="bf16")
    r = oracle_mod.llmint8_matmul(X, W, 0.0, fmt="bf16")
    assert r["outliers"].size == 95 and not r["C"].any()
    ref = _bf16_values(X) @ _bf16_values(W)
    diff = np.abs(_bf16_values(r["Y"]) - ref)
    assert np.all(diff <= bf16_ulp(ref) / 2 + 1e-30)


@pytest.mark.parametrize("t", [math.inf, 6.0])
def test_bf16_quantization_error_bound(oracle_mod, t):
    # the fp16 bound of test_quantization_error_bound, with a bf16 final rounding
    X, _ = synthetic.make_x(24, 200, frac=0.02, seed=22, fmt="bf16")
    W, _ = synthetic.make_w(200, 72, seed=22, fmt="bf16")
    r = oracle_mod.llmint8_matmul(X, W, t, fmt="bf16")
    keep = ~r["is_outlier"]
    Xd, Wd = _bf16_values(X), _bf16_values(W)
    xhat = r["Xq"].astype(np.float64) * r["s_x"][:, None].astype(np.float64) / 127
    sx = r["s_x"].astype(np.float64)[:, None]
    sw = r["s_w"].astype(np.float64)[None, :]
    slack = 1 / 254 + 1e-6
    bound = (sx * slack) * np.abs(Wd[keep]).sum(0)[None, :] + (np.abs(xhat[:, keep]).sum(1)[:, None]) * sw * slack
    ref = Xd @ Wd
    err = np.abs(_bf16_values(r["Y"]) - ref)
    assert np.all(err <= bound + bf16_ulp(ref) + 1e-12)
    assert np.max(err) < 0.05 * np.max(np.abs(ref))


def test_bf16_and_fp16_agree_on_values_both_represent(oracle_mod):
    # Inputs with at most 8 significant bits inside fp16's normal range are the
    # same numbers in both formats: codes, scales, outlier set and C coincide.
    rng = np.random.default_rng(23)
    Xv = (rng.integers(-255, 256, (10, 128)) / 32.0).astype(np.float32)
    Xv[:, [4, 77]] *= 8
    Wv = (rng.integers(-127, 128, (128, 48)) / 4096.0).astype(np.float32)
    a = oracle_mod.llmint8_matmul(Xv.astype(np.float16), Wv.astype(np.float16), 6.0)
    b = oracle_mod.llmint8_matmul(synthetic.to_bf16_bits(Xv), synthetic.to_bf16_bits(Wv), 6.0, fmt="bf16")
    for k in ("Xq", "s_x", "Wq", "s_w", "C", "outliers", "F"):
        assert np.array_equal(a[k], b[k]), k
