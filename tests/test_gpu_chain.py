"""Decode chain (llmint8_matmul_chain) against the CPU oracle (needs a B300).

The chain's GEMV writes, for its output Y, what the next layer's X pass would
find (outlier flags of Y's columns, row absmax over the other columns), and a
call given that "chain state" runs no X pass.  Checked here:
  * a first call (no state in) gives the oracle's Y, and the state it writes
    holds exactly the flags and row maxima of the Y it wrote;
  * a call whose state comes from the oracle (flags = A1 of X, one partial
    maximum = the A2 row scale) gives the oracle's Y: the in-kernel X pass
    (codes, outlier list) follows the pages' steps;
  * chained calls agree with llmint8_matmul on the same inputs.
Shapes cover several 16-column strips per CTA, ragged K (a last ring stage
that is partly outside K), outlier counts past the lanes' registers, no
outliers, and a negative next threshold (every column an outlier).
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


def _weights(K, N, seed):
    W, _ = synthetic.make_w(K, N, seed=seed)
    Wd = torch.from_numpy(W).cuda()
    Wq, sw = api.llmint8_quantize_weight(Wd)
    return W, Wd, Wq, sw


def _read_state(S, M, N):
    flags_off, parts_off, total = api.llmint8_chain_state_layout(M, N)
    b = S.cpu().numpy()
    hdr = b[:16].view(np.int32)
    thr = float(b[12:16].view(np.float32)[0])
    nparts = int(hdr[2])
    flags = b[flags_off:flags_off + N].astype(bool)
    parts = b[parts_off:parts_off + nparts * M * 4].view(np.float32).reshape(nparts, M)
    return dict(M=int(hdr[0]), N=int(hdr[1]), nparts=nparts, threshold=thr, flags=flags, parts=parts)


def _state_from_oracle(X, t):
    """Chain state of X built on the host: flags = A1 of the oracle, one
    partial maximum per row = the oracle's A2 row scale."""
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


@pytest.mark.parametrize("M,K,N,frac,t2", [
    (1, 4096, 4096, 0.001, 6.0),
    (4, 1040, 16 * 700, 0.01, 0.05),  # ragged K; several strips per CTA; many outlier columns in Y
    (3, 2048, 1040, 0.09, 0.02),      # ~180 outliers in X (past the lanes' registers)
    (2, 528, 64, 0.0, -1.0),          # no outliers in X; next threshold < 0: every column flagged
])
def test_first_call_and_the_state_it_writes(M, K, N, frac, t2):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=0 if frac == 0 else 3, seed=M * 31 + K)
    W, Wd, Wq, sw = _weights(K, N, seed=K + N)
    ref = oracle.llmint8_matmul(X, W, 6.0)
    S = api.make_chain_state(M, N)
    Y = api.llmint8_matmul_chain(torch.from_numpy(X).cuda(), 6.0, None, Wq, sw, Wd, next_threshold=t2, state_out=S)
    torch.cuda.synchronize()
    Yg = Y.cpu().numpy()
    ok, ratio = y_close(Yg, ref["Y"])
    assert ok, f"Y: worst error/tolerance {ratio:.3g}"
    st = _read_state(S, M, N)
    assert (st["M"], st["N"], st["nparts"]) == (M, N, N // 16)
    assert st["threshold"] == np.float32(t2)
    # the state is exactly A1 and the A2 row absmax of the Y this call wrote
    a = np.abs(Yg.astype(np.float32))
    flags = (a > np.float32(t2)).any(axis=0)
    assert np.array_equal(st["flags"], flags)
    sx = np.where(flags[None, :], np.float32(0), a).max(axis=1)
    assert np.array_equal(st["parts"].max(axis=0), sx)
    # and the flags are the oracle's A1 of the oracle's Y, except where an element sits within tolerance of t2
    ra = np.abs(ref["Y"].astype(np.float64))
    tol = 1e-3 * ra.max() + 2.0 ** (np.floor(np.log2(np.maximum(ra, 2.0 ** -14))) - 10)
    near = (np.abs(ra - t2) <= tol).any(axis=0)
    oflags = oracle.outlier_columns(ref["Y"], t2)
    assert np.array_equal(st["flags"][~near], oflags[~near])


@pytest.mark.parametrize("M,K,N,frac", [
    (1, 4096, 11008, 0.001),
    (4, 11008, 4096, 0.001),
    (2, 1040, 16 * 640, 0.05),  # ragged K, ~52 outliers, several strips per CTA
    (4, 784, 48, 0.3),          # ~235 outliers (binary search of the bit map past the registers)
    (1, 512, 16, 0.0),          # one stage, one strip, no outliers
])
def test_call_with_a_state_from_the_oracle(M, K, N, frac):
    X, _ = synthetic.make_x(M, K, frac=frac, min_count=0 if frac == 0 else 3, seed=M * 7 + K)
    W, Wd, Wq, sw = _weights(K, N, seed=K * 3 + N)
    S_in = _state_from_oracle(X, 6.0)
    Xg = torch.from_numpy(X).cuda()
    ws = api.make_workspace(M, K, N, Xg.device)
    C = torch.empty((M, N), dtype=torch.int32, device=Xg.device)
    Y = api.llmint8_matmul_chain(Xg, float("nan"), S_in, Wq, sw, Wd, workspace=ws, C=C)
    torch.cuda.synchronize()
    ref = oracle.llmint8_matmul(X, W, 6.0)
    ok, ratio = y_close(Y.cpu().numpy(), ref["Y"])
    assert ok, f"worst error/tolerance {ratio:.3g}"
    # the kernel rebuilt A1 and A2 from the state: outlier set, row scales and codes
    # bit for bit, and the exact int32 product of those codes
    is_out = oracle.outlier_columns(X, 6.0)
    Xq_ref, sx_ref = oracle.quantize_rows(X, is_out)
    inter = api.read_intermediates(ws, M, K, N)
    assert np.array_equal(inter["outliers"].cpu().numpy(), oracle.outlier_indices(is_out)), "outlier set"
    assert np.array_equal(inter["row_scale"].cpu().numpy().view(np.uint32), sx_ref.view(np.uint32)), "row scales"
    assert np.array_equal(inter["codes"].cpu().numpy(), Xq_ref), "codes"
    Wq_ref, _ = oracle.quantize_weight(W)
    assert np.array_equal(C.cpu().numpy().astype(np.int64), oracle.int8_matmul(Xq_ref, Wq_ref)), "int32 product"


@pytest.mark.parametrize("M", [1, 4])
def test_chained_calls_agree_with_llmint8_matmul(M):
    # X0 [M, 4096] -> (4096, 4096) -> (4096, 11008) -> (11008, 4096), each Y the next X
    shapes = [(4096, 4096), (4096, 11008), (11008, 4096)]
    X, _ = synthetic.make_x(M, 4096, frac=0.001, min_count=4, seed=500 + M)
    Xg = torch.from_numpy(X).cuda()
    S_in = None
    for li, (K, N) in enumerate(shapes):
        _, Wd, Wq, sw = _weights(K, N, seed=li + 10)
        S_out = api.make_chain_state(M, N)
        Y = api.llmint8_matmul_chain(Xg, 6.0, S_in, Wq, sw, Wd, next_threshold=4.0, state_out=S_out)
        # the same layer through the workspace path, on the same X, with the threshold the state stands for
        Y_std = api.llmint8_matmul(Xg, 6.0 if li == 0 else 4.0, Wq, sw, Wd)
        torch.cuda.synchronize()
        ok, ratio = y_close(Y.cpu().numpy(), Y_std.cpu().numpy())
        assert ok, f"layer {li}: worst error/tolerance {ratio:.3g}"
        Xg, S_in = Y, S_out


def test_without_any_state_equals_llmint8_matmul():
    M, K, N = 4, 4096, 4096
    X, _ = synthetic.make_x(M, K, frac=0.001, min_count=4, seed=77)
    W, Wd, Wq, sw = _weights(K, N, seed=78)
    Xg = torch.from_numpy(X).cuda()
    for t in (6.0, float("inf")):
        Y = api.llmint8_matmul_chain(Xg, t, None, Wq, sw, Wd)
        torch.cuda.synchronize()
        ref = oracle.llmint8_matmul(X, W, t)
        ok, ratio = y_close(Y.cpu().numpy(), ref["Y"])
        assert ok, f"t={t}: worst error/tolerance {ratio:.3g}"
