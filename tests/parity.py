"""Run the CUDA path and the CPU oracle on the same seeded inputs and compare.

Bit-exact: weight codes and column scales, the outlier column set, row scales,
activation codes and the int32 accumulators.  Y: within the stated tolerance
max|Y - Y_ref| <= 1e-3 * max|Y_ref| + 1 fp16 ulp of Y_ref, element by element.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_quantization_matmul_row_b300 import api


def fp16_ulp(y):
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def y_close(Y, Yref):
    """(ok, worst ratio of error to tolerance) for the Y tolerance rule."""
    Yd = np.asarray(Y, np.float64)
    Rd = np.asarray(Yref, np.float64)
    if not np.all(np.isfinite(Yd)) or not np.all(np.isfinite(Rd)):
        return False, float("inf")
    tol = 1e-3 * np.max(np.abs(Rd)) + fp16_ulp(Rd)
    err = np.abs(Yd - Rd)
    ratio = float(np.max(err / tol)) if err.size else 0.0
    return bool(np.all(err <= tol)), ratio


def sample_rows(M, n=24, seed=0):
    """Row subset for spot checks of large problems: first/last rows, both sides of
    every 128-row tile boundary near the end, and random rows."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    fixed = {0, 1, M - 1, M - 2, min(127, M - 1), min(128, M - 1)}
    fixed |= set(rng.choice(M, size=n, replace=False).tolist())
    return np.array(sorted(fixed))


def run_gpu(X: np.ndarray, W: np.ndarray, t: float, *, int8_variant=False, want_i32=True,
            garbage_workspace=False, stream=None):
    """The whole CUDA path on device copies of X and W; returns numpy results."""
    M, K = X.shape
    N = W.shape[1]
    dev = torch.device("cuda")
    Xd = torch.from_numpy(np.ascontiguousarray(X)).to(dev)
    Wd = torch.from_numpy(np.ascontiguousarray(W)).to(dev)
    Wq, sw = api.llmint8_quantize_weight(Wd, stream=stream)
    ws = api.make_workspace(M, K, N, dev)
    if garbage_workspace:
        ws.fill_(0xA5)
    if int8_variant:
        Y = api.llmint8_matmul_int8(Xd, Wq, sw, workspace=ws, stream=stream)
    else:
        Y = api.llmint8_matmul(Xd, t, Wq, sw, Wd, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    inter = api.read_intermediates(ws, M, K, N)
    out = dict(Y=Y.cpu().numpy(), Wq=Wq.cpu().numpy(), s_w=sw.cpu().numpy(),
               s_x=inter["row_scale"].cpu().numpy(), codes=inter["codes"].cpu().numpy(),
               codes16=None if inter["codes_fp16"] is None else inter["codes_fp16"].cpu().numpy(),
               outliers=inter["outliers"].cpu().numpy())
    status = api.llmint8_device_status(ws)
    if want_i32:
        ws2 = api.make_workspace(M, K, N, dev)
        C = api.llmint8_matmul_i32(Xd, float("inf") if int8_variant else t, Wq, sw, workspace=ws2,
                                   stream=stream)
        torch.cuda.synchronize()
        out["C"] = C.cpu().numpy()
        status = status or api.llmint8_device_status(ws2)
    out["status"] = status
    return out


def sample_cols(N, n=64, seed=0):
    """Output-column subset: edges, both sides of 256-wide tile boundaries, random columns."""
    if N <= n:
        return np.arange(N)
    rng = np.random.default_rng(seed + 1)
    fixed = {0, 1, 15, 16, N - 1, N - 16, min(255, N - 1), min(256, N - 1), (N // 256) * 256 - 1}
    fixed |= set(rng.choice(N, size=n, replace=False).tolist())
    return np.array(sorted(c for c in fixed if 0 <= c < N))


def check(X, W, t, *, rows=None, cols=None, int8_variant=False, g=None, **kw):
    """Compare every intermediate of the CUDA path with the oracle; returns (gpu, ref).

    rows / cols restrict the comparison of the weight codes, C and Y to a sample
    (each is local to its row or column); the X-pass results are compared in full.
    """
    if g is None:
        g = run_gpu(X, W, t, int8_variant=int8_variant, **kw)
    assert g["status"] == 0, f"device status {g['status']}"
    t_eff = float("inf") if int8_variant else t
    M, K = X.shape
    csel = slice(None) if cols is None else np.asarray(cols)
    Wc = W if cols is None else np.ascontiguousarray(W[:, csel])
    Wq_ref, sw_ref = oracle.quantize_weight(Wc)
    # A0: weight codes (GPU layout [N, K]) and column scales, bit-exact
    assert np.array_equal(g["Wq"][csel], Wq_ref.T), "Wq mismatch"
    assert np.array_equal(g["s_w"][csel].view(np.uint32), sw_ref.view(np.uint32)), "colScaleW mismatch"
    # A1: outlier set (sorted list), A2: row scales and codes for every row
    is_out = oracle.outlier_columns(X, t_eff)
    assert np.array_equal(g["outliers"], oracle.outlier_indices(is_out)), "outlier set mismatch"
    Xq_ref, sx_ref = oracle.quantize_rows(X, is_out)
    assert np.array_equal(g["s_x"].view(np.uint32), sx_ref.view(np.uint32)), "rowScaleX mismatch"
    assert np.array_equal(g["codes"], Xq_ref), "Xq mismatch"
    if g["codes16"] is not None:  # tensor-core path keeps the codes as fp16 values
        assert np.array_equal(g["codes16"].astype(np.float32), Xq_ref.astype(np.float32)), "fp16 code values"
    # A3-A5 on the sampled rows x columns
    ref = oracle.llmint8_matmul(X, Wc, t_eff, rows=rows, wq=(Wq_ref, sw_ref))
    rsel = slice(None) if rows is None else np.asarray(rows)
    if "C" in g:
        assert np.abs(ref["C"]).max(initial=0) < 2 ** 31
        assert np.array_equal(g["C"][rsel][:, csel].astype(np.int64), ref["C"]), "int32 accumulator mismatch"
    ok, ratio = y_close(g["Y"][rsel][:, csel], ref["Y"])
    assert ok, f"Y outside tolerance (worst error/tolerance = {ratio:.3g})"
    return g, ref
