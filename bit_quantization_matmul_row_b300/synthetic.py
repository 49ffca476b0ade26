"""Seeded synthetic inputs for the LLM.int8() decomposed matmul.

This module only *draws* inputs.  It holds none of the method's arithmetic (no
thresholding, no scales, no codes), so both the CPU oracle's tests and the CUDA
path's tests and benchmark can take their inputs from here without sharing any
part of the computation.

Value structure follows the pages' description of the workload:

* activations X ~ N(0, 1) in fp16, shaped [tokens, hidden] (LLM.int8() paper
  summary, section 2.3: X is [seq_len, hidden_dim]);
* a few K-columns carry large-magnitude "outlier features" that appear in the
  same hidden dimensions for every token (same page, section 2.2: 20-100x the
  normal values, stable across all tokens), typically 0.1-1 % of the columns
  (section 2.3);
* weights W ~ N(0, sigma) in fp16, shaped [hidden, out] (section 2.3).

Each planted column is rescaled so that its absolute maximum is drawn from
U(lo, hi); this keeps the column an outlier at every M, including M = 1.
Random streams: numpy PCG64 seeded with [seed, stream], stream 0 for X and
stream 1 for W, so X and W of one case are independent and reproducible.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

X_STREAM = 0
W_STREAM = 1


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def planted_count(K: int, frac: float, min_count: int = 0) -> int:
    """Number of planted outlier columns: round(frac*K), at least min_count."""
    n = int(round(frac * K))
    if frac > 0:
        n = max(n, min_count)
    return min(n, K)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), rounded to nearest even.

    The input generators' bf16 cast (numpy has no bfloat16 type): the upper 16
    bits of the binary32 value after adding 0x7fff plus the lowest kept bit.
    Inputs here are finite.
    """
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _cast(x: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "fp16":
        return x.astype(np.float16)
    if fmt == "bf16":
        return to_bf16_bits(x)
    raise ValueError(fmt)


def make_x(M: int, K: int, *, frac: float = 0.0, min_count: int = 0,
           mag: tuple[float, float] = (20.0, 60.0), seed: int = 0, fmt: str = "fp16"):
    """X fp16 [M, K] ~ N(0,1) with planted outlier columns.

    Returns (X, planted) where planted is the sorted int64 array of the
    planted column indices.  Column j in `planted` is rescaled so that
    max_i |X[i, j]| == U(mag) (before the cast).  fmt="bf16" returns X as
    bfloat16 bit patterns (uint16) of the same draws.
    """
    g = _rng(seed, X_STREAM)
    x = g.standard_normal((M, K), dtype=np.float32)
    n = planted_count(K, frac, min_count)
    cols = np.sort(g.choice(K, size=n, replace=False)) if n else np.zeros(0, np.int64)
    if n:
        target = g.uniform(mag[0], mag[1], size=n).astype(np.float32)
        sub = x[:, cols]
        peak = np.max(np.abs(sub), axis=0)
        peak[peak == 0] = 1.0
        x[:, cols] = sub * (target / peak)[None, :]
    return _cast(x, fmt), cols.astype(np.int64)


def make_w(K: int, N: int, *, sigma: float = 0.02, boosted_frac: float = 0.0,
           boost: float = 10.0, seed: int = 0, fmt: str = "fp16"):
    """W fp16 [K, N] ~ N(0, sigma); a fraction of the N-columns is multiplied by `boost`.

    Returns (W, boosted) with boosted the sorted column indices that were scaled.
    """
    g = _rng(seed, W_STREAM)
    w = g.standard_normal((K, N), dtype=np.float32) * np.float32(sigma)
    nb = int(round(boosted_frac * N))
    cols = np.sort(g.choice(N, size=nb, replace=False)) if nb else np.zeros(0, np.int64)
    if nb:
        w[:, cols] *= np.float32(boost)
    return _cast(w, fmt), cols.astype(np.int64)


@dataclass(frozen=True)
class Case:
    """One matmul problem of a workload: shapes, value recipe and seed."""
    name: str
    M: int
    K: int
    N: int
    frac: float = 0.0
    min_count: int = 0
    mag: tuple = (20.0, 60.0)
    sigma: float = 0.02
    boosted_frac: float = 0.0
    threshold: float = 6.0
    seed: int = 0
    tags: tuple = field(default_factory=tuple)

    def x(self):
        return make_x(self.M, self.K, frac=self.frac, min_count=self.min_count,
                      mag=self.mag, seed=self.seed)

    def w(self):
        return make_w(self.K, self.N, sigma=self.sigma,
                      boosted_frac=self.boosted_frac, seed=self.seed)


def tiny():
    """X [16,256] with 2 planted columns of absmax U(20,60); W [256,512] ~N(0,0.02); t = 6; seed 0."""
    return [Case("tiny", 16, 256, 512, frac=2 / 256, min_count=2, seed=0)]


DECODE_KN = ((4096, 4096), (4096, 11008), (11008, 4096))


def decode_7b():
    """7B-like decode: M in {1,4,16} x (K,N) in DECODE_KN, 0.1 % outlier columns (at least 4)."""
    out, j = [], 0
    for M in (1, 4, 16):
        for K, N in DECODE_KN:
            out.append(Case(f"decode7b_M{M}_K{K}_N{N}", M, K, N, frac=0.001,
                            min_count=4, seed=1000 * 1 + j, tags=("decode",)))
            j += 1
    return out


def prefill_7b():
    """7B-like prefill: M=2048, K=4096, N in {4096, 11008}, 0.1 % outlier columns."""
    return [Case(f"prefill7b_M2048_K4096_N{N}", 2048, 4096, N, frac=0.001,
                 min_count=4, seed=1000 * 2 + j, tags=("prefill",))
            for j, N in enumerate((4096, 11008))]


def ffn_13b():
    """13B-like FFN: M=4096, (K,N) in {(5120,13824),(13824,5120)}; 1 % outlier columns of
    absmax U(20,100); 0.5 % of W's output columns scaled x10."""
    return [Case(f"ffn13b_M4096_K{K}_N{N}", 4096, K, N, frac=0.01, mag=(20.0, 100.0),
                 boosted_frac=0.005, seed=1000 * 3 + j, tags=("prefill",))
            for j, (K, N) in enumerate(((5120, 13824), (13824, 5120)))]


def sweep_70b():
    """70B-like sweep: K=8192, N in {8192, 28672}, M in {1,16,256,2048,8192},
    outlier fraction in {0, 0.1 %, 1 %, 5 %}, W ~N(0,0.015)."""
    out, j = [], 0
    for N in (8192, 28672):
        for M in (1, 16, 256, 2048, 8192):
            for f in (0.0, 0.001, 0.01, 0.05):
                tag = "decode" if M <= 16 else "prefill"
                out.append(Case(f"sweep70b_M{M}_N{N}_f{f:g}", M, 8192, N, frac=f,
                                sigma=0.015, seed=1000 * 4 + j, tags=(tag,)))
                j += 1
    return out
