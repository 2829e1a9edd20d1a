"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare it with the CPU oracle element by element.

Comparison rules (the tolerance is the one the hot path is specified with):
  bitmaps, hash buckets/signs, compaction indices and counts: bit-exact;
  sketch bucket (j, b): |S_gpu - S| <= 1e-5 * A[j][b] + 6 * c[j][b] * FLT_MIN,
      where A is the sum of the magnitudes of the bucket's contributions and c
      their number; exactly +0.0 where A = 0. The second term covers the
      float atomic adds of the GPU, which flush subnormal addends and sums to
      zero (each addition can lose less than FLT_MIN = 2^-126 per operand and
      per result, and a contribution passes through at most two of them: a
      shared-memory add into a block's copy of the sketch, then that copy's
      add into global memory); it is invisible for normal values;
  decoded value: |g_gpu - g| <= (1e-5 * max_j A[j][h_j(i)] + 6 * max_j c * FLT_MIN)
      * |scale| plus one float32 spacing of the oracle's rounded value. The
      median is 1-Lipschitz in the max-norm, so the bucket bound carries over.
"""
import numpy as np
import torch

import oracle
import sketch_compressed_sparse_gb300 as s2

REL = 1e-5
FLT_MIN = 2.0 ** -126
FTZ_TERMS = 6.0  # flushed operands/results per contribution: 3 per atomic add, at most 2 adds


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def contribution_counts(bitmaps: np.ndarray, n: int, d: int, w: int, seed: int) -> np.ndarray:
    """c[k][j][b]: how many nonzeros of worker k land in bucket b of row j."""
    W = bitmaps.shape[0]
    c = np.zeros((W, d, w), dtype=np.int64)
    for k in range(W):
        pos = np.flatnonzero(unpack(bitmaps[k], n)).astype(np.uint32)
        if pos.size:
            b, _ = oracle.hash(pos, d, w, seed)
            for j in range(d):
                c[k, j] = np.bincount(b[j], minlength=w)
    return c


def assert_sketch_close(got: np.ndarray, S: np.ndarray, A: np.ndarray, what="sketch", cnt=None):
    got = np.asarray(got, dtype=np.float32).reshape(S.shape)
    err = np.abs(got.astype(np.float64) - S)
    tol = REL * A + (0.0 if cnt is None else FTZ_TERMS * FLT_MIN * cnt)
    bad = err > tol
    if bad.any():
        k = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} buckets out of tolerance, first at {tuple(k)}: "
                             f"got {got[tuple(k)]!r} want {S[tuple(k)]!r} tol {tol[tuple(k)]!r}")
    empty = A == 0
    assert (got.view(np.uint32)[empty] == 0).all(), f"{what}: a bucket with no contribution is not +0.0"


def assert_decoded_close(got: np.ndarray, want: np.ndarray, amax: np.ndarray, scale: float = 1.0, what="decode",
                         cmax=None):
    got = np.asarray(got, dtype=np.float32)
    tol = (REL * amax + (0.0 if cmax is None else FTZ_TERMS * FLT_MIN * cmax)) * abs(scale) \
        + np.spacing(np.abs(want)).astype(np.float64)
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bad = err > tol
    if bad.any():
        k = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} values out of tolerance, first at {k}: "
                             f"got {got[k]!r} want {want[k]!r} tol {tol[k]!r}")


def unpack(bitmap: np.ndarray, n: int) -> np.ndarray:
    return np.unpackbits(bitmap.astype("<u4").view(np.uint8), bitorder="little")[:n].astype(bool)


def gpu_pipeline(grad: torch.Tensor, d: int, w: int, seed: int, scale: float = 1.0, compact: bool = False,
                 stream=None):
    """encode_batched -> reduce -> decode through the C ABI; returns numpy results."""
    dev = grad.device
    W, n = grad.shape
    bitmaps, sketches = s2.alloc_encode_outputs(W, n, d, w, dev)
    bitmap = torch.empty(s2.nwords(n), dtype=torch.int32, device=dev)
    sketch = torch.empty((d, w), dtype=torch.float32, device=dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    out_ws = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    dws = torch.empty(max(s2.s2_decode_dense_workspace_size(n, d, w), 1), dtype=torch.uint8, device=dev)
    s2.s2_encode_batched(grad, d, w, seed, bitmaps, sketches, stream=stream)
    s2.s2_reduce(bitmaps, sketches, n, d, w, bitmap, sketch, stream=stream)
    s2.s2_decode_dense(bitmap, sketch, n, d, w, seed, out, scale=scale, stream=stream)
    s2.s2_decode_dense_ws(bitmap, sketch, n, d, w, seed, out_ws, dws, scale=scale, stream=stream)
    res = {}
    if compact:
        ws = torch.empty(max(s2.s2_decode_workspace_size(n), 1), dtype=torch.uint8, device=dev)
        idx = torch.full((max(n, 1),), -1, dtype=torch.int32, device=dev)
        val = torch.full((max(n, 1),), float("nan"), dtype=torch.float32, device=dev)
        cnt = torch.full((1,), -1, dtype=torch.int64, device=dev)
        s2.s2_decode_compact(bitmap, sketch, n, d, w, seed, idx[:n], val[:n], cnt, ws, scale=scale, stream=stream)
        res["compact"] = (idx, val, cnt)
    if stream is not None:
        stream.synchronize()
    torch.cuda.synchronize()
    res.update(bitmaps=u32(bitmaps), sketches=sketches.cpu().numpy(), bitmap=u32(bitmap),
               sketch=sketch.cpu().numpy(), out=out.cpu().numpy(), out_ws=out_ws.cpu().numpy())
    if compact:
        idx, val, cnt = res["compact"]
        c = int(cnt.item())
        res["count"] = c
        res["idx"] = u32(idx[: min(c, n)])
        res["val"] = val[: min(c, n)].cpu().numpy()
    return res


def check_pipeline(host_grad: np.ndarray, dtype: str, got: dict, d: int, w: int, seed: int, scale: float = 1.0,
                   exact: bool = False):
    """Compare a gpu_pipeline result with the oracle on the same gradient."""
    scale = float(np.float32(scale))  # the C ABI takes the scale as a float32
    ref = oracle.pipeline(host_grad, d, w, seed, dtype=dtype, scale=scale)
    n = host_grad.shape[1]
    np.testing.assert_array_equal(got["bitmaps"], ref["bitmaps"])
    np.testing.assert_array_equal(got["bitmap"], ref["bitmap"])
    if exact:
        np.testing.assert_array_equal(got["sketches"].astype(np.float64), ref["S"])
        np.testing.assert_array_equal(got["sketch"].astype(np.float64), ref["S_sum"])
        np.testing.assert_array_equal(got["out"], ref["out"] * np.float32(1.0))
    else:
        cnt = contribution_counts(ref["bitmaps"], n, d, w, seed)
        for k in range(host_grad.shape[0]):
            assert_sketch_close(got["sketches"][k], ref["S"][k], ref["A"][k], what=f"sketch of worker {k}",
                                cnt=cnt[k])
        csum = cnt.sum(axis=0)
        assert_sketch_close(got["sketch"], ref["S_sum"], ref["A_sum"], what="summed sketch", cnt=csum)
        union = np.flatnonzero(unpack(ref["bitmap"], n)).astype(np.uint32)
        cmax = np.zeros(n, dtype=np.float64)
        if union.size:
            b, _ = oracle.hash(union, d, w, seed)
            cmax[union] = np.max(np.stack([csum[j][b[j]] for j in range(d)]), axis=0)
        assert_decoded_close(got["out"], ref["out"], ref["amax"], scale, cmax=cmax)
    unset = ~unpack(ref["bitmap"], n)
    assert (got["out"].view(np.uint32)[unset] == 0).all(), "unset positions must be exactly +0.0"
    if "out_ws" in got:  # the dense decode with a workspace (row passes for large sketches) selects the same values
        np.testing.assert_array_equal(got["out_ws"], got["out"])
        assert (got["out_ws"].view(np.uint32)[unset] == 0).all(), "unset positions must be exactly +0.0"
    if "count" in got:
        cnt, idx, val, amax = oracle.decode_compact(ref["bitmap"], ref["S_sum"], n, seed, scale, ref["A_sum"])
        assert got["count"] == cnt
        np.testing.assert_array_equal(got["idx"], idx)
        np.testing.assert_array_equal(got["val"], got["out"][idx])
    return ref
