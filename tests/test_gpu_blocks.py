"""GPU parity of the block-granular bitmap (the paper's per-block bitmap):
s2_encode_batched_blocks -> s2_reduce over nb = ceil(n/block) bits ->
s2_decode_dense_blocks, against the oracle's block functions. Block bitmaps
are compared bit for bit; sketches and decoded values with the tolerance of
the element path (the sketch is the same: zeros are never inserted).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sketch_compressed_sparse_gb300 as s2
    from tests._parity import assert_decoded_close, assert_sketch_close, contribution_counts, u32, unpack

DEV = "cuda"


def rows_workload(W, n_rows, cols, rows_per_worker, d, w, tag, dtype="f32"):
    """Whole nonzero rows (embedding-like); rows drawn uniformly per worker."""
    rng = np.random.default_rng(tag)
    idx, val = [], []
    for _ in range(W):
        rows = np.sort(rng.choice(n_rows, size=rows_per_worker, replace=False))
        flat = (rows[:, None] * cols + np.arange(cols)[None, :]).reshape(-1)
        v = rng.normal(size=flat.size).astype(np.float32)
        v[v == 0] = 1.0
        if dtype == "bf16":
            v = workloads.f32_to_bf16_bits(v)
        idx.append(flat.astype(np.int64))
        val.append(v)
    return workloads.Workload(f"rows{tag}", W, n_rows * cols, d, w, 0, dtype, idx, val)


def run_blocks(wl, block, scale=1.0):
    W, n, d, w = wl.W, wl.n, wl.d, wl.w
    grad = wl.dense_torch(DEV)
    nbw = s2.nblockwords(n, block)
    nb = (n + block - 1) // block
    bms = torch.full((W, max(nbw, 1)), -1, dtype=torch.int32, device=DEV)[:, :nbw].contiguous()
    sks = torch.empty((W, d, w), dtype=torch.float32, device=DEV)
    s2.s2_encode_batched_blocks(grad, block, d, w, wl.seed, bms, sks)
    bm = torch.empty(nbw, dtype=torch.int32, device=DEV)
    sk = torch.empty((d, w), dtype=torch.float32, device=DEV)
    s2.s2_reduce(bms, sks, nb, d, w, bm, sk)
    out = torch.full((n,), 9.0, dtype=torch.float32, device=DEV)
    s2.s2_decode_dense_blocks(bm, sk, n, block, d, w, wl.seed, out, scale=scale)
    torch.cuda.synchronize()
    return u32(bms), sks.cpu().numpy(), u32(bm), sk.cpu().numpy(), out.cpu().numpy()


def check_blocks(wl, block, scale=1.0):
    bms, sks, bm, sk, out = run_blocks(wl, block, scale)
    G = wl.dense()
    scale = float(np.float32(scale))
    ref = oracle.pipeline_blocks(G, block, wl.d, wl.w, wl.seed, dtype=wl.dtype, scale=scale)
    np.testing.assert_array_equal(bms, ref["bitmaps"])
    np.testing.assert_array_equal(bm, ref["bitmap"])
    # per-worker element bitmaps give the contribution counts of the tolerance
    elem = np.stack([oracle.encode(G[k], wl.d, wl.w, wl.seed, wl.dtype)[0] for k in range(wl.W)])
    cnt = contribution_counts(elem, wl.n, wl.d, wl.w, wl.seed)
    for k in range(wl.W):
        assert_sketch_close(sks[k], ref["S"][k], ref["A"][k], what=f"sketch of worker {k}", cnt=cnt[k])
    csum = cnt.sum(axis=0)
    assert_sketch_close(sk, ref["S_sum"], ref["A_sum"], what="summed sketch", cnt=csum)
    nb = (wl.n + block - 1) // block
    marked = np.repeat(unpack(ref["bitmap"], nb), block)[: wl.n]
    cmax = np.zeros(wl.n)
    pos = np.flatnonzero(marked).astype(np.uint32)
    if pos.size:
        b, _ = oracle.hash(pos, wl.d, wl.w, wl.seed)
        cmax[pos] = np.max(np.stack([csum[j][b[j]] for j in range(wl.d)]), axis=0)
    assert_decoded_close(out, ref["out"], ref["amax"], scale, cmax=cmax)
    assert (out.view(np.uint32)[~marked] == 0).all()
    return ref


@pytest.mark.parametrize("block", [32, 96, 512, 1024])
def test_rows_with_block_bitmap(block):
    wl = rows_workload(W=3, n_rows=300, cols=512, rows_per_worker=20, d=5, w=1 << 14, tag=block)
    check_blocks(wl, block)


@pytest.mark.parametrize("block,kw", [
    (32, dict(W=3, n=10_000, d=3, w=1000, density=0.02, tag=401)),
    (64, dict(W=2, n=1001, d=3, w=64, density=0.1, tag=402)),          # unaligned rows, ragged last block
    (256, dict(W=4, n=8192, d=5, w=512, density=0.01, dtype="bf16", tag=403)),
    (128, dict(W=2, n=7777, d=7, w=300, density=0.01, dtype="bf16", tag=404)),
])
def test_scattered_with_block_bitmap(block, kw):
    check_blocks(workloads.custom(**kw), block)


def test_block_scale_and_single_block():
    wl = workloads.custom(W=2, n=500, d=3, w=256, density=0.05, tag=405)
    check_blocks(wl, 1024, scale=0.25)  # one block covers everything


def test_block_size_must_be_a_multiple_of_32():
    grad = torch.zeros((1, 100), dtype=torch.float32, device=DEV)
    with pytest.raises(s2.S2Error) as e:
        s2.s2_encode_batched_blocks(grad, 48, 3, 16, 0, torch.zeros(1, dtype=torch.int32, device=DEV),
                                    torch.zeros((1, 3, 16), device=DEV))
    assert e.value.status == 3


@pytest.mark.slow
def test_embedding_rows_block_512_full_size():
    wl = workloads.embedding()
    check_blocks(wl, 512)
