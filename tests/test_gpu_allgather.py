"""GPU parity of the sparse AllGather baseline (s2_sparse_pack, s2_sparse_sum)
against the oracle: the per-worker (index, value) lists bit for bit, the
summed vector bit for bit against a sequential float32 sum over workers and
within the path's tolerance of the oracle's float64 sum.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sketch_compressed_sparse_gb300 as s2

DEV = "cuda"


def run(G, capacity=None):
    W, n = G.shape
    cap = n if capacity is None else capacity
    g = torch.from_numpy(G).to(DEV)
    idx = torch.full((W, max(cap, 1)), -1, dtype=torch.int32, device=DEV)[:, :cap].contiguous()
    val = torch.full((W, max(cap, 1)), 9.0, device=DEV)[:, :cap].contiguous()
    cnt = torch.full((W,), -1, dtype=torch.int64, device=DEV)
    ws = torch.empty(max(s2.s2_sparse_pack_workspace_size(W, n), 1), dtype=torch.uint8, device=DEV)
    s2.s2_sparse_pack(g, idx, val, cnt, ws)
    out = torch.full((n,), 5.0, device=DEV)
    s2.s2_sparse_sum(idx, val, cnt, n, out)
    torch.cuda.synchronize()
    return idx.cpu().numpy().view(np.uint32), val.cpu().numpy(), cnt.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("kw", [
    dict(W=3, n=10_000, d=3, w=64, density=0.05, tag=501),
    dict(W=8, n=70_001, d=3, w=64, density=0.01, tag=502),   # ragged last tile
    dict(W=1, n=8192, d=3, w=64, density=1.0, tag=503),      # every position nonzero
    dict(W=4, n=100, d=3, w=64, density=0.0, tag=504),       # nothing to send
])
def test_pack_and_sum(kw):
    wl = workloads.custom(**kw)
    G = wl.dense()
    idx, val, cnt, out = run(G)
    for k in range(wl.W):
        c, ri, rv = oracle.sparse_list(G[k])
        assert cnt[k] == c
        np.testing.assert_array_equal(idx[k, :c], ri)
        np.testing.assert_array_equal(val[k, :c].view(np.uint32), rv.view(np.uint32))
    seq = np.zeros(wl.n, dtype=np.float32)
    for k in range(wl.W):
        seq = seq + G[k]
    np.testing.assert_array_equal(out, seq)  # fixed worker order
    ex = oracle.exact_sum(G)
    tol = 1e-5 * np.abs(G.astype(np.float64)).sum(axis=0) + np.spacing(np.abs(ex))
    assert (np.abs(out.astype(np.float64) - ex) <= tol).all()


def test_pack_capacity_truncates_but_counts_all():
    wl = workloads.custom(W=2, n=50_000, d=3, w=64, density=0.1, tag=505)
    G = wl.dense()
    idx, val, cnt, _ = run(G, capacity=1000)
    for k in range(2):
        c, ri, _ = oracle.sparse_list(G[k])
        assert cnt[k] == c > 1000
        np.testing.assert_array_equal(idx[k], ri[:1000])


@pytest.mark.slow
def test_embedding_full_size():
    wl = workloads.embedding()
    G = wl.dense()
    idx, val, cnt, out = run(G, capacity=max(wl.nnz_per_worker))
    ex = oracle.exact_sum(G)
    tol = 1e-5 * np.abs(G.astype(np.float64)).sum(axis=0) + np.spacing(np.abs(ex))
    assert (cnt == np.array(wl.nnz_per_worker)).all()
    assert (np.abs(out.astype(np.float64) - ex) <= tol).all()
