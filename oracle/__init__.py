"""CPU oracle for the S2 Reducer encode -> reduce -> decode path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(the CUDA library and its binding) never imports it and shares no code with
it.

The arithmetic lives in ``s2_oracle.c`` (plain C loops, fp64 accumulation),
compiled with gcc into ``oracle/_lib/libs2oracle.so`` on first use. This
module only marshals numpy arrays in and out of it.

Source: "S2 Reducer: High-Performance Sparse Communication to Accelerate
Distributed Deep Learning", Section 3.1 and Algorithm 1 (Sparse-Sketch
Reducer). Every function below says which part it follows.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):
  fmix32 / hash      published MurmurHash3 vectors; bucket range, uniformity,
                     sign balance and pairwise collision statistics
  encode             bitmap = exact nonzero support; sparse insertion equals
                     the dense projection A^T g built from an explicit A
  reduce             linearity: reduce(encode(g_k)) = encode(sum_k g_k)
  decode             exact recovery without collisions; median rejects a
                     minority of colliding rows; brute force A A^T g at d = 1;
                     median equals numpy's median on planted sketches
  decode_compact     indices equal numpy's flatnonzero of the bitmap
  encode_blocks /    block bitmap = numpy any() over each block; block size 1
  decode_dense_blocks  equals the element functions; exact recovery of every
                     position of marked blocks (zeros included) without collisions
  block_topk /       norms = numpy's float64 norm of each block; kept blocks =
  block_split        numpy's lexsort (norm desc, index asc) of those norms;
                     a hand-worked four-block case; sparse + residual = grad +
                     residual exactly; the delta-approximate bound of
                     Theorem 2 (K/nb of the energy)
  sparse_list /      indices = numpy flatnonzero of the bit test, capacity keeps
  exact_sum          the true count; exact_sum = float64 numpy sum; equals the
                     S2 decode wherever no row collides
All functions are pinned; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "s2_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libs2oracle.so")
_lock = threading.Lock()
_lib = None

_DT = {"f32": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2; no contraction of a*b+c into fused
    multiply-adds, so every float operation rounds as written)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        u32, u64, i32, dbl = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        lib.s2o_fmix32.argtypes = [u32]
        lib.s2o_fmix32.restype = u32
        lib.s2o_row_keys.argtypes = [u32, u32, vp, vp]
        lib.s2o_row_keys.restype = None
        lib.s2o_bucket.argtypes = [u32, u32, u32]
        lib.s2o_bucket.restype = u32
        lib.s2o_sign.argtypes = [u32, u32]
        lib.s2o_sign.restype = i32
        lib.s2o_hash.argtypes = [vp, u64, u32, u32, u32, vp, vp]
        lib.s2o_hash.restype = None
        lib.s2o_encode.argtypes = [vp, i32, u64, u32, u32, u32, vp, vp, vp]
        lib.s2o_encode.restype = None
        lib.s2o_reduce.argtypes = [u32, u64, u64, vp, vp, vp, vp, vp, vp]
        lib.s2o_reduce.restype = None
        lib.s2o_decode_dense.argtypes = [vp, vp, vp, u64, u32, u32, u32, dbl, vp, vp]
        lib.s2o_decode_dense.restype = None
        lib.s2o_decode_compact.argtypes = [vp, vp, vp, u64, u32, u32, u32, dbl, vp, vp, vp, u64]
        lib.s2o_decode_compact.restype = u64
        lib.s2o_encode_blocks.argtypes = [vp, i32, u64, u64, u32, u32, u32, vp, vp, vp]
        lib.s2o_encode_blocks.restype = None
        lib.s2o_decode_dense_blocks.argtypes = [vp, vp, vp, u64, u64, u32, u32, u32, dbl, vp, vp]
        lib.s2o_decode_dense_blocks.restype = None
        lib.s2o_sparse_list.argtypes = [vp, u64, vp, vp, u64]
        lib.s2o_sparse_list.restype = u64
        lib.s2o_exact_sum.argtypes = [vp, u32, u64, vp]
        lib.s2o_exact_sum.restype = None
        lib.s2o_block_topk.argtypes = [vp, vp, u64, u64, u64, vp, vp, vp]
        lib.s2o_block_topk.restype = None
        lib.s2o_block_split.argtypes = [vp, vp, u64, u64, vp, vp]
        lib.s2o_block_split.restype = None
        _lib = lib
        return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def nwords(n: int) -> int:
    return (n + 31) // 32


# ---- hash family (MurmurHash3 finalizer; the paper leaves h and s open) ----

def fmix32(x: int) -> int:
    return int(_load().s2o_fmix32(x & 0xFFFFFFFF))


def row_keys(seed: int, j: int) -> Tuple[int, int]:
    kh = ctypes.c_uint32()
    ks = ctypes.c_uint32()
    _load().s2o_row_keys(seed, j, ctypes.byref(kh), ctypes.byref(ks))
    return int(kh.value), int(ks.value)


def hash(idx: np.ndarray, d: int, w: int, seed: int) -> Tuple[np.ndarray, np.ndarray]:
    """Buckets h_j(i) (uint32 [d][m]) and signs s_j(i) (int8 [d][m]) of the given indices."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    m = idx.size
    b = np.empty((d, m), dtype=np.uint32)
    s = np.empty((d, m), dtype=np.int8)
    _load().s2o_hash(_ptr(idx), m, d, w, seed, _ptr(b), _ptr(s))
    return b, s


# ---- compression, aggregation, decompression --------------------------------

def encode(grad: np.ndarray, d: int, w: int, seed: int, dtype: str = "f32"):
    """Algorithm 1 compression phase for ONE worker's gradient.

    Returns (bitmap uint32[nw], S float64[d][w], A float64[d][w]) where A holds
    the summed magnitudes of each bucket's contributions (tolerance scale).
    """
    g = np.ascontiguousarray(grad)
    if dtype == "f32":
        assert g.dtype == np.float32
    else:
        assert g.dtype == np.uint16
    n = g.size
    bm = np.empty(nwords(n), dtype=np.uint32)
    S = np.empty((d, w), dtype=np.float64)
    A = np.empty((d, w), dtype=np.float64)
    _load().s2o_encode(_ptr(g), _DT[dtype], n, d, w, seed, _ptr(bm), _ptr(S), _ptr(A))
    return bm, S, A


def reduce(bitmaps: np.ndarray, S: np.ndarray, A: Optional[np.ndarray] = None):
    """AllReduce(S, C) of Algorithm 1: sum of sketches, OR of bitmaps.

    bitmaps: uint32[W][nw]; S, A: float64[W][d][w]. Returns (bitmap, S_sum, A_sum).
    """
    bitmaps = np.ascontiguousarray(bitmaps, dtype=np.uint32)
    S = np.ascontiguousarray(S, dtype=np.float64)
    W = S.shape[0]
    nw = bitmaps.shape[1]
    dw = int(np.prod(S.shape[1:]))
    bm_out = np.empty(nw, dtype=np.uint32)
    S_out = np.empty(S.shape[1:], dtype=np.float64)
    A_out = None
    if A is not None:
        A = np.ascontiguousarray(A, dtype=np.float64)
        A_out = np.empty(S.shape[1:], dtype=np.float64)
    _load().s2o_reduce(W, nw, dw, _ptr(bitmaps), _ptr(S), _ptr(A), _ptr(bm_out), _ptr(S_out), _ptr(A_out))
    return bm_out, S_out, A_out


def decode_dense(bitmap: np.ndarray, S: np.ndarray, n: int, seed: int, scale: float = 1.0,
                 A: Optional[np.ndarray] = None):
    """Algorithm 1 decompression phase, dense output.

    Returns (out float32[n], amax float64[n]); amax[i] = max_j A[j][h_j(i)]
    (zero where A is not given or the bit is unset).
    """
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint32)
    S = np.ascontiguousarray(S, dtype=np.float64)
    d, w = S.shape
    if d > 64:
        raise ValueError("oracle supports d <= 64")
    out = np.empty(n, dtype=np.float32)
    amax = np.empty(n, dtype=np.float64)
    Ap = None if A is None else np.ascontiguousarray(A, dtype=np.float64)
    _load().s2o_decode_dense(_ptr(bitmap), _ptr(S), _ptr(Ap), n, d, w, seed, float(scale), _ptr(out), _ptr(amax))
    return out, amax


def decode_compact(bitmap: np.ndarray, S: np.ndarray, n: int, seed: int, scale: float = 1.0,
                   A: Optional[np.ndarray] = None, capacity: Optional[int] = None):
    """Algorithm 1 decompression phase, compacted output.

    Returns (count, idx uint32[min(count, capacity)], val float32[...], amax float64[...]).
    """
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint32)
    S = np.ascontiguousarray(S, dtype=np.float64)
    d, w = S.shape
    if d > 64:
        raise ValueError("oracle supports d <= 64")
    if capacity is None:
        capacity = n
    idx = np.empty(max(capacity, 1), dtype=np.uint32)
    val = np.empty(max(capacity, 1), dtype=np.float32)
    amax = np.empty(max(capacity, 1), dtype=np.float64)
    Ap = None if A is None else np.ascontiguousarray(A, dtype=np.float64)
    cnt = int(_load().s2o_decode_compact(_ptr(bitmap), _ptr(S), _ptr(Ap), n, d, w, seed, float(scale),
                                         _ptr(idx), _ptr(val), _ptr(amax), capacity))
    m = min(cnt, capacity)
    return cnt, idx[:m].copy(), val[:m].copy(), amax[:m].copy()


def encode_blocks(grad: np.ndarray, block: int, d: int, w: int, seed: int, dtype: str = "f32"):
    """Compression phase with one bitmap bit per block of `block` positions.

    Returns (block bitmap uint32[ceil(nb/32)], S float64[d][w], A float64[d][w]).
    """
    g = np.ascontiguousarray(grad)
    n = g.size
    nb = (n + block - 1) // block
    bm = np.empty(max(nwords(nb), 1), dtype=np.uint32)
    S = np.empty((d, w), dtype=np.float64)
    A = np.empty((d, w), dtype=np.float64)
    _load().s2o_encode_blocks(_ptr(g), _DT[dtype], n, block, d, w, seed, _ptr(bm), _ptr(S), _ptr(A))
    return bm[: nwords(nb)], S, A


def decode_dense_blocks(bitmap: np.ndarray, S: np.ndarray, n: int, block: int, seed: int, scale: float = 1.0,
                        A: Optional[np.ndarray] = None):
    """Decompression with a block bitmap: every position of every marked block is queried."""
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint32)
    S = np.ascontiguousarray(S, dtype=np.float64)
    d, w = S.shape
    out = np.empty(n, dtype=np.float32)
    amax = np.empty(n, dtype=np.float64)
    Ap = None if A is None else np.ascontiguousarray(A, dtype=np.float64)
    _load().s2o_decode_dense_blocks(_ptr(bitmap), _ptr(S), _ptr(Ap), n, block, d, w, seed, float(scale), _ptr(out),
                                    _ptr(amax))
    return out, amax


def pipeline_blocks(grad: np.ndarray, block: int, d: int, w: int, seed: int, dtype: str = "f32", scale: float = 1.0):
    """Every worker compresses with a block bitmap; aggregate; decode every marked block."""
    W, n = grad.shape
    nb = (n + block - 1) // block
    bms = np.zeros((W, nwords(nb)), dtype=np.uint32)
    S = np.empty((W, d, w), dtype=np.float64)
    A = np.empty((W, d, w), dtype=np.float64)
    for k in range(W):
        bms[k], S[k], A[k] = encode_blocks(grad[k], block, d, w, seed, dtype)
    bm, Ssum, Asum = reduce(bms, S, A)
    out, amax = decode_dense_blocks(bm, Ssum, n, block, seed, scale, Asum)
    return dict(bitmaps=bms, S=S, A=A, bitmap=bm, S_sum=Ssum, A_sum=Asum, out=out, amax=amax)


def block_topk(grad: np.ndarray, residual: np.ndarray, block: int, K: int):
    """Block-wise Top-K with error feedback for ONE worker (Section 2.2; Appendix A.2).

    Returns (sparse float32[n], new residual float32[n], squared block norms
    float64[nb], keep uint8[nb]).
    """
    g = np.ascontiguousarray(grad, dtype=np.float32)
    e = np.array(residual, dtype=np.float32, copy=True)
    n = g.size
    nb = (n + block - 1) // block
    sp = np.empty(n, dtype=np.float32)
    nrm = np.empty(max(nb, 1), dtype=np.float64)
    keep = np.empty(max(nb, 1), dtype=np.uint8)
    _load().s2o_block_topk(_ptr(g), _ptr(e), n, block, K, _ptr(sp), _ptr(nrm), _ptr(keep))
    return sp, e, nrm[:nb], keep[:nb]


def block_split(grad: np.ndarray, residual: np.ndarray, block: int, keep: np.ndarray):
    """The error-feedback split of ONE worker for a given kept-block set
    (Appendix A.2): returns (sparse float32[n], new residual float32[n])."""
    g = np.ascontiguousarray(grad, dtype=np.float32)
    e = np.array(residual, dtype=np.float32, copy=True)
    n = g.size
    kp = np.ascontiguousarray(keep, dtype=np.uint8)
    assert kp.size == (n + block - 1) // block
    sp = np.empty(n, dtype=np.float32)
    _load().s2o_block_split(_ptr(g), _ptr(e), n, block, _ptr(kp if kp.size else np.zeros(1, np.uint8)), _ptr(sp))
    return sp, e


def sparse_list(grad: np.ndarray, capacity: Optional[int] = None):
    """AllGather baseline message of one worker: (count, idx uint32[...], val float32[...]) ascending."""
    g = np.ascontiguousarray(grad, dtype=np.float32)
    cap = g.size if capacity is None else capacity
    idx = np.empty(max(cap, 1), dtype=np.uint32)
    val = np.empty(max(cap, 1), dtype=np.float32)
    c = int(_load().s2o_sparse_list(_ptr(g), g.size, _ptr(idx), _ptr(val), cap))
    m = min(c, cap)
    return c, idx[:m].copy(), val[:m].copy()


def exact_sum(grads: np.ndarray) -> np.ndarray:
    """The gathered lists added up (float64 accumulation, one rounding): float32[n]."""
    g = np.ascontiguousarray(grads, dtype=np.float32)
    W, n = g.shape
    out = np.empty(n, dtype=np.float32)
    _load().s2o_exact_sum(_ptr(g), W, n, _ptr(out))
    return out


def encode_all(grad: np.ndarray, d: int, w: int, seed: int, dtype: str = "f32"):
    """Compression phase on every worker of grad[W][n].

    Returns (bitmaps uint32[W][nw], S float64[W][d][w], A float64[W][d][w]).
    """
    W, n = grad.shape
    bms = np.empty((W, nwords(n)), dtype=np.uint32)
    S = np.empty((W, d, w), dtype=np.float64)
    A = np.empty((W, d, w), dtype=np.float64)
    for k in range(W):
        bms[k], S[k], A[k] = encode(grad[k], d, w, seed, dtype)
    return bms, S, A


def pipeline(grad: np.ndarray, d: int, w: int, seed: int, dtype: str = "f32", scale: float = 1.0,
             dense: bool = True):
    """Every worker compresses, the sketches and bitmaps are aggregated, and
    the aggregate is decompressed once (the decode is the same on every worker).

    Returns a dict with per-worker and aggregated structures and the decode.
    """
    n = grad.shape[1]
    bms, S, A = encode_all(grad, d, w, seed, dtype)
    bm, Ssum, Asum = reduce(bms, S, A)
    res = dict(bitmaps=bms, S=S, A=A, bitmap=bm, S_sum=Ssum, A_sum=Asum)
    if dense:
        res["out"], res["amax"] = decode_dense(bm, Ssum, n, seed, scale, Asum)
    else:
        res["count"], res["idx"], res["val"], res["amax"] = decode_compact(bm, Ssum, n, seed, scale, Asum)
    return res


def tolerance(amax: np.ndarray, scale: float = 1.0, rel: float = 1e-5) -> np.ndarray:
    """Allowed |GPU - oracle| for a decoded value: rel * (largest summed
    contribution magnitude among the queried buckets) * |scale|."""
    return rel * amax * abs(scale)
