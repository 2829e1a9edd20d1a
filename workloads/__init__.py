"""Seeded synthetic inputs for the S2 Reducer encode -> reduce -> decode path.

This module is the one piece shared by the CUDA path's tests/benchmark and by
the CPU oracle. It draws gradients and nothing else: no bitmap, no hash, no
sketch, no median. Every workload is a deterministic function of its name and
parameters.

The shapes stand in for the workloads of "S2 Reducer: High-Performance Sparse
Communication to Accelerate Distributed Deep Learning" (Section 4, Table 1:
embedding-layer gradients of language models, and block-wise sparsified dense
models). The datasets and trained models of those experiments are not used;
only the sizes and the sparsity structure are imitated.

Layout: a workload holds, per worker k, the ascending flat indices of its
nonzero elements and their values. ``dense()`` expands that into the
worker-major gradient ``grad[W][n]`` the hot path consumes. For bf16 the values
are held as their raw 16-bit patterns (numpy has no bfloat16).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

__all__ = [
    "Workload",
    "tiny",
    "embedding",
    "topk",
    "large_lm",
    "sweep_point",
    "sweep_grid",
    "dense_laplace",
    "by_name",
    "custom",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "random_sketches",
    "random_bitmaps",
]


@dataclasses.dataclass
class Workload:
    """One synthetic problem: W workers, gradient length n, sketch d x w."""

    name: str
    W: int
    n: int
    d: int
    w: int
    seed: int  # hash seed of the count-sketch
    dtype: str  # "f32" or "bf16"
    idx: List[np.ndarray]  # per worker: ascending int64 flat indices of nonzeros
    val: List[np.ndarray]  # per worker: float32 values, or uint16 bf16 bit patterns

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def nnz_per_worker(self) -> List[int]:
        return [int(a.size) for a in self.idx]

    def dense(self) -> np.ndarray:
        """grad[W][n] as float32 (f32) or uint16 bit patterns (bf16)."""
        npdt = np.float32 if self.dtype == "f32" else np.uint16
        g = np.zeros((self.W, self.n), dtype=npdt)
        for k in range(self.W):
            g[k, self.idx[k]] = self.val[k]
        return g

    def dense_torch(self, device):
        """grad[W][n] as a torch tensor on ``device`` (float32 or bfloat16).

        Only the nonzeros travel from the host; the zero fill happens on the
        device. This is input preparation, not part of the method.
        """
        import torch

        tdt = torch.float32 if self.dtype == "f32" else torch.bfloat16
        g = torch.zeros((self.W, self.n), dtype=tdt, device=device)
        for k in range(self.W):
            ix = torch.from_numpy(self.idx[k]).to(device)
            if self.dtype == "f32":
                v = torch.from_numpy(self.val[k]).to(device)
            else:
                v = torch.from_numpy(self.val[k].view(np.int16)).to(device).view(torch.bfloat16)
            g[k].index_copy_(0, ix, v)
        return g

    def union_nnz(self) -> int:
        """Positions that are nonzero in at least one worker."""
        if not self.W:
            return 0
        mark = np.zeros(self.n, dtype=bool)
        for ix in self.idx:
            mark[ix] = True
        return int(np.count_nonzero(mark))

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "W": self.W,
            "n": self.n,
            "d": self.d,
            "w": self.w,
            "hash_seed": self.seed,
            "dtype": self.dtype,
            "nnz_per_worker": self.nnz_per_worker[0] if self.W else 0,
        }


# ---------------------------------------------------------------------------
# small helpers (input preparation only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((b >> 16) & 1) + 0x7FFF
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _nonzero_normal(rng: np.random.Generator, size: int, sigma: float) -> np.ndarray:
    """float32 N(0, sigma) draws, redrawing any value that is exactly zero."""
    v = rng.normal(0.0, sigma, size=size).astype(np.float32)
    while True:
        z = v == 0
        if not z.any():
            return v
        v[z] = rng.normal(0.0, sigma, size=int(z.sum())).astype(np.float32)


def _nonzero_bf16_normal(rng: np.random.Generator, size: int) -> np.ndarray:
    v = f32_to_bf16_bits(rng.normal(0.0, 1.0, size=size).astype(np.float32))
    while True:
        z = (v & 0x7FFF) == 0
        if not z.any():
            return v
        v[z] = f32_to_bf16_bits(rng.normal(0.0, 1.0, size=int(z.sum())).astype(np.float32))


def _bounded_zipf_distinct(rng: np.random.Generator, n_ranks: int, s: float, count: int) -> np.ndarray:
    """Draw ranks 1..n_ranks with P(r) proportional to r^-s until ``count`` are distinct.

    Returns the distinct 0-based ranks (r - 1), in first-drawn order.
    """
    if count > n_ranks:
        raise ValueError("more distinct rows requested than exist")
    p = np.arange(1, n_ranks + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    seen = set()
    order = []
    while len(order) < count:
        u = rng.random(max(4 * (count - len(order)), 1024))
        r = np.searchsorted(cdf, u, side="right")
        r = np.minimum(r, n_ranks - 1)
        for x in r.tolist():
            if x not in seen:
                seen.add(x)
                order.append(x)
                if len(order) == count:
                    break
    return np.asarray(order, dtype=np.int64)


def _uniform_positions(rng: np.random.Generator, n: int, m: int) -> np.ndarray:
    """``m`` distinct positions in [0, n), uniform without replacement, ascending."""
    if m > n:
        raise ValueError("m > n")
    if m == 0:
        return np.zeros(0, dtype=np.int64)
    if m * 4 >= n:
        return np.sort(rng.permutation(n)[:m]).astype(np.int64)
    picked = np.unique(rng.integers(0, n, size=m + m // 8 + 16, dtype=np.int64))
    while picked.size < m:
        more = rng.integers(0, n, size=(m - picked.size) * 2 + 16, dtype=np.int64)
        picked = np.unique(np.concatenate([picked, more]))
    # drop a uniformly random surplus so the set stays uniform
    if picked.size > m:
        keep = np.sort(rng.permutation(picked.size)[:m])
        picked = picked[keep]
    return picked


def _rows_to_flat(rows: np.ndarray, cols: int) -> np.ndarray:
    rows = np.sort(rows.astype(np.int64))
    return (rows[:, None] * cols + np.arange(cols, dtype=np.int64)[None, :]).reshape(-1)


def _children(tag: int, count: int):
    return np.random.SeedSequence(tag).spawn(count)


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def tiny() -> Workload:
    """W=2, n=4096 fp32, 90% zeros at uniform positions, N(0,1) values, d=3, w=256."""
    W, n = 2, 4096
    m = int(round(0.1 * n))
    ch = _children(1000, W)
    idx, val = [], []
    for k in range(W):
        rng = np.random.default_rng(ch[k])
        idx.append(_uniform_positions(rng, n, m))
        val.append(_nonzero_normal(rng, m, 1.0))
    return Workload("tiny", W, n, 3, 256, 0, "f32", idx, val)


def embedding(rows_per_worker: int = 2000, W: int = 8, n_rows: int = 33_278, cols: int = 512,
              d: int = 5, w: int = 1 << 20) -> Workload:
    """Embedding-row sparsity: a 33,278 x 512 fp32 table, 2,000 Zipf(1.1) rows per worker.

    Rows are drawn by popularity rank from a bounded Zipf(1.1) law until 2,000
    are distinct; ranks map to row ids through one fixed permutation shared by
    all workers, so popular rows overlap across workers. Every value of a drawn
    row is N(0, 0.01).
    """
    ch = _children(1001, W + 1)
    perm = np.random.default_rng(ch[W]).permutation(n_rows)
    idx, val = [], []
    for k in range(W):
        rng = np.random.default_rng(ch[k])
        ranks = _bounded_zipf_distinct(rng, n_rows, 1.1, rows_per_worker)
        flat = _rows_to_flat(perm[ranks], cols)
        idx.append(flat)
        val.append(_nonzero_normal(rng, flat.size, 1e-2))
    return Workload("embedding_33278x512", W, n_rows * cols, d, w, 0, "f32", idx, val)


def topk(W: int = 8, n: int = 25_557_032, keep: float = 0.01, d: int = 3, w: int = 1 << 19) -> Workload:
    """Top-k sparsified dense model (ResNet-50 size): per worker a Laplace(0,1)
    draw of n values keeps its floor(0.01 n) largest magnitudes (ties go to the
    lower index) and zeroes the rest."""
    K = int(math.floor(keep * n))
    ch = _children(1002, W)
    idx, val = [], []
    for k in range(W):
        rng = np.random.default_rng(ch[k])
        x = rng.laplace(0.0, 1.0, size=n).astype(np.float32)
        a = np.abs(x)
        if K == 0:
            sel = np.zeros(0, dtype=np.int64)
        else:
            part = np.argpartition(a, n - K)[n - K:]
            thr = a[part].min()
            above = np.flatnonzero(a > thr)
            ties = np.flatnonzero(a == thr)[: K - above.size]
            sel = np.sort(np.concatenate([above, ties])).astype(np.int64)
        v = x[sel]
        if np.any(v == 0):
            raise RuntimeError("top-k kept an exact zero; choose another seed")
        idx.append(sel)
        val.append(v)
    return Workload("topk_resnet50", W, n, d, w, 0, "f32", idx, val)


def large_lm(W: int = 4, n_rows: int = 267_735, cols: int = 1024, row_frac: float = 0.01,
             d: int = 5, w: int = 1 << 22) -> Workload:
    """Large LM embedding: a 267,735 x 1024 fp32 table, 1% of rows per worker.

    Rows come from one Zipf(1.2) popularity law whose rank -> row map is shared
    by all workers (they overlap heavily); values N(0, 1e-3).
    """
    per = int(round(row_frac * n_rows))
    ch = _children(1003, W + 1)
    perm = np.random.default_rng(ch[W]).permutation(n_rows)
    idx, val = [], []
    for k in range(W):
        rng = np.random.default_rng(ch[k])
        ranks = _bounded_zipf_distinct(rng, n_rows, 1.2, per)
        flat = _rows_to_flat(perm[ranks], cols)
        idx.append(flat)
        val.append(_nonzero_normal(rng, flat.size, 1e-3))
    return Workload("large_lm_267735x1024", W, n_rows * cols, d, w, 0, "f32", idx, val)


def sweep_w(nnz: int) -> int:
    """w = nnz_per_worker / 2 rounded to a power of two (sketch ratio about 0.5)."""
    return 1 << max(0, int(round(math.log2(max(nnz, 1) / 2.0))))


def sweep_point(n: int, dtype: str = "f32", density: float = 0.01, d: int = 3, W: int = 8,
                tag: Optional[int] = None) -> Workload:
    """Flat gradient of length n, ``round(density*n)`` uniform nonzeros per worker, N(0,1)."""
    if dtype not in ("f32", "bf16"):
        raise ValueError(dtype)
    m = int(round(density * n))
    if tag is None:
        tag = 1004 * 1_000_003 + n * 7 + int(round(density * 1e4)) * 3 + d + (0 if dtype == "f32" else 11)
    ch = _children(tag, W)
    idx, val = [], []
    for k in range(W):
        rng = np.random.default_rng(ch[k])
        idx.append(_uniform_positions(rng, n, m))
        val.append(_nonzero_normal(rng, m, 1.0) if dtype == "f32" else _nonzero_bf16_normal(rng, m))
    name = f"sweep_n{n}_{dtype}_rho{density:g}_d{d}"
    return Workload(name, W, n, d, sweep_w(m), 0, dtype, idx, val)


def sweep_grid():
    """The 108 sweep points: n = 2^20..2^28, fp32/bf16, density 0.1/1/10 %, d in {3, 5}."""
    for e in range(20, 29):
        for dt in ("f32", "bf16"):
            for rho in (0.001, 0.01, 0.1):
                for d in (3, 5):
                    yield dict(n=1 << e, dtype=dt, density=rho, d=d)


def custom(W: int, n: int, d: int, w: int, density: float, seed: int = 0, dtype: str = "f32",
           tag: int = 7, values: str = "normal", int_max: int = 1024) -> Workload:
    """A free-form uniform-position workload for tests.

    ``values="int"`` draws nonzero integers in [-int_max, int_max] so that
    every fp32 partial sum of a few such values is exact.
    """
    ch = _children(tag, max(W, 1))
    m = int(round(density * n))
    idx, val = [], []
    for k in range(W):
        rng = np.random.default_rng(ch[k])
        ix = _uniform_positions(rng, n, m)
        if values == "int":
            v = rng.integers(1, int_max + 1, size=m) * rng.choice(np.array([-1, 1]), size=m)
            v = v.astype(np.float32)
            if dtype == "bf16":
                v = f32_to_bf16_bits(v)
        elif dtype == "f32":
            v = _nonzero_normal(rng, m, 1.0)
        else:
            v = _nonzero_bf16_normal(rng, m)
        idx.append(ix)
        val.append(v)
    return Workload(f"custom_W{W}_n{n}_d{d}_w{w}", W, n, d, w, seed, dtype, idx, val)


def random_sketches(W: int, d: int, w: int, tag: int = 11, values: str = "normal") -> np.ndarray:
    """float32 [W][d][w] arrays to feed the reduce step on its own."""
    rng = np.random.default_rng(np.random.SeedSequence(tag))
    if values == "int":
        return rng.integers(-4096, 4097, size=(W, d, w)).astype(np.float32)
    return rng.normal(0.0, 1.0, size=(W, d, w)).astype(np.float32)


def random_bitmaps(W: int, n: int, density: float, tag: int = 12) -> np.ndarray:
    """uint32 [W][ceil(n/32)] words with random set bits below n (bit i = word i>>5, bit i&31)."""
    rng = np.random.default_rng(np.random.SeedSequence(tag))
    nw = (n + 31) // 32
    out = np.zeros((W, nw), dtype=np.uint32)
    for k in range(W):
        pos = _uniform_positions(rng, n, int(round(density * n)))
        np.bitwise_or.at(out[k], pos >> 5, (np.uint32(1) << (pos & 31).astype(np.uint32)))
    return out


def dense_laplace(W: int = 8, n: int = 25_557_032, tag: int = 1005) -> np.ndarray:
    """Dense float32 gradients [W][n] of Laplace(0,1) draws (ResNet-50 size),
    the input of the block-wise Top-K sparsifier (one draw per worker)."""
    ch = _children(tag, W)
    out = np.empty((W, n), dtype=np.float32)
    for k in range(W):
        out[k] = np.random.default_rng(ch[k]).laplace(0.0, 1.0, size=n).astype(np.float32)
    return out


_BY_NAME = {
    "tiny": tiny,
    "embedding": embedding,
    "topk": topk,
    "large_lm": large_lm,
}


def by_name(name: str) -> Workload:
    if name not in _BY_NAME:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(_BY_NAME)}")
    return _BY_NAME[name]()
