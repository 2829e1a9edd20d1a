"""GPU parity of the block-wise Top-K sparsifier with error feedback
(s2_block_topk) against the oracle.

"S2 Reducer" (Section 2.2) keeps the K blocks of largest l2 norm. The oracle
takes each norm in float64 as defined; the kernel sums the squares in float32
in a fixed order. So the kept set is checked for validity, not copied:
  - exactly K blocks are kept;
  - no dropped block's float64 norm exceeds a kept block's by more than the
    float32 rounding of the kernel's sum can explain. Each element's square
    goes through at most c = ceil(L / 32) fused multiply-adds on its lane and
    5 butterfly additions (L = block length), each with one rounding of
    relative size at most u = 2^-24 on nonnegative terms, so the float32 norm
    f of a block with exact norm x obeys |f - x| <= g x with g = m u / (1 - m u),
    m = c + 5. If the kernel keeps a over b then f_a >= f_b, hence
    x_b <= x_a (1 + g) / (1 - g);
  - where blocks are identical (the same float32 values) their norms are equal
    on both sides and the lower index must win;
  - given the kernel's kept set, the sent part and the new residual match the
    oracle's split bit for bit (float32 additions grad + residual).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sketch_compressed_sparse_gb300 as s2
    from tests._parity import check_pipeline, gpu_pipeline

DEV = "cuda"
U = 2.0 ** -24
SLICE = 4096  # norms per thread block of the kernel's select


def laplace_grads(W, n, tag, scale=1.0):
    rng = np.random.default_rng(tag)
    return (scale * rng.laplace(size=(W, n))).astype(np.float32)


def gpu_topk(G, E, block, K):
    W, n = G.shape
    g = torch.from_numpy(G).to(DEV)
    e = torch.from_numpy(E.copy()).to(DEV)
    sp = torch.full((W, n), 7.0, device=DEV)
    ws = torch.empty(max(s2.s2_block_topk_workspace_size(W, n, block), 1), dtype=torch.uint8, device=DEV)
    s2.s2_block_topk(g, e, block, K, sp, ws)
    torch.cuda.synchronize()
    return sp.cpu().numpy(), e.cpu().numpy()


def kept_blocks(sp, E_new, block):
    """Kept blocks as seen in the outputs: a kept block has its values in the
    sent part and zeros in the residual (inputs here have no all-zero block)."""
    n = sp.size
    nb = (n + block - 1) // block
    pad = nb * block - n
    s = np.concatenate([sp, np.zeros(pad, np.float32)]).reshape(nb, block)
    r = np.concatenate([E_new, np.zeros(pad, np.float32)]).reshape(nb, block)
    keep = (s != 0).any(axis=1)
    assert not ((r != 0).any(axis=1) & keep).any(), "a kept block left values in the residual"
    return keep.astype(np.uint8)


def rounding_ratio(block):
    m = -(-block // 32) + 5
    g = m * U / (1 - m * U)
    return (1 + g) / (1 - g)


def check_worker(G, E, block, K, sp, E_new):
    """Validity of one worker's kept set and exactness of its split."""
    keep = kept_blocks(sp, E_new, block)
    _, _, nrm, want = oracle.block_topk(G, E, block, K)
    assert int(keep.sum()) == K
    if 0 < K < nrm.size:
        lo_kept = nrm[keep == 1].min()
        hi_dropped = nrm[keep == 0].max()
        assert hi_dropped <= lo_kept * rounding_ratio(block), (hi_dropped, lo_kept)
        # blocks that differ from the oracle's choice lie within the rounding band of the K-th norm
        diff = np.flatnonzero(keep != want)
        kth = np.sort(nrm)[::-1][K - 1]
        assert (np.abs(nrm[diff] - kth) <= 2 * kth * (rounding_ratio(block) - 1)).all()
    rsp, re = oracle.block_split(G, E, block, keep)
    np.testing.assert_array_equal(sp.view(np.uint32), rsp.view(np.uint32))
    np.testing.assert_array_equal(E_new.view(np.uint32), re.view(np.uint32))
    return keep, want


@pytest.mark.parametrize("W,n,block,K", [
    (3, 10_000, 32, 10),
    (3, 10_000, 64, 0),
    (2, 10_001, 64, 157),        # K = nb: every block kept; ragged last block
    (4, 65_536, 256, 8),
    (1, 100_000, 96, 33),
    (2, 5_000, 1024, 2),
    (2, 32 * 20_000, 32, 625),   # 20,000 blocks: the select spans 5 thread blocks per worker
    (1, 32 * 70_001 + 7, 32, 2187),  # 17 slices, ragged last block
    (2, 128 * 9_000 + 132, 128, 400),  # 16-byte vector norms; ragged last block of 132
])
def test_block_topk_keeps_a_valid_largest_set(W, n, block, K):
    G = laplace_grads(W, n, tag=W * 7 + K)
    E = (0.05 * np.random.default_rng(K).normal(size=(W, n))).astype(np.float32)
    sp, e = gpu_topk(G, E, block, K)
    for k in range(W):
        check_worker(G[k], E[k], block, K, sp[k], e[k])


def test_block_topk_ties_go_to_the_lower_block():
    G = np.ones((2, 32 * 40), dtype=np.float32)  # 40 equal blocks per worker
    G[1, 32 * 5:32 * 6] = 2.0                      # worker 1: block 5 is the largest
    sp, e = gpu_topk(G, np.zeros_like(G), 32, 3)
    kept0 = np.flatnonzero(sp[0].reshape(40, 32).any(axis=1))
    kept1 = np.flatnonzero(sp[1].reshape(40, 32).any(axis=1))
    np.testing.assert_array_equal(kept0, [0, 1, 2])
    np.testing.assert_array_equal(kept1, [0, 1, 5])


def test_block_topk_ties_across_thread_blocks_of_the_select():
    # 20,000 equal blocks per worker (five select slices of 4096 norms): K =
    # 9000 ends inside the third slice. Worker 1 also has two larger blocks in
    # later slices, which must be kept ahead of the ties.
    nb, block, K = 20_000, 32, 9000
    G = np.ones((2, nb * block), dtype=np.float32)
    G[1, 15_000 * block:15_001 * block] = 2.0
    G[1, 19_999 * block:] = 3.0
    sp, e = gpu_topk(G, np.zeros_like(G), block, K)
    kept0 = np.flatnonzero(sp[0].reshape(nb, block).any(axis=1))
    kept1 = np.flatnonzero(sp[1].reshape(nb, block).any(axis=1))
    np.testing.assert_array_equal(kept0, np.arange(K))
    np.testing.assert_array_equal(kept1, np.concatenate([np.arange(K - 2), [15_000, 19_999]]))
    for k in range(2):
        check_worker(G[k], np.zeros_like(G[k]), block, K, sp[k], e[k])


@pytest.mark.parametrize("block", [64, 256])  # 4-byte and 16-byte loads in the norms
def test_block_topk_repeated_patterns_match_the_oracle_exactly(block):
    # Every block is one of four fixed patterns with well separated norms, so
    # equal norms are exactly equal on both sides and the kept set is unique:
    # K falls inside the group of the second largest pattern, whose members
    # are spread over all of the select's slices.
    nb = 24_000
    rng = np.random.default_rng(77)
    pats = rng.normal(size=(4, block)).astype(np.float32) * np.array([[1.0], [2.0], [3.0], [4.0]], np.float32)
    choice = rng.integers(0, 4, size=nb)
    G = pats[choice].reshape(1, -1)
    K = int((choice == 3).sum()) + int((choice == 2).sum()) // 2
    sp, e = gpu_topk(G, np.zeros_like(G), block, K)
    keep, want = check_worker(G[0], np.zeros_like(G[0]), block, K, sp[0], e[0])
    np.testing.assert_array_equal(keep, want)


def test_block_topk_two_steps_of_error_feedback():
    W, n, block, K = 3, 20_000, 64, 9
    E = np.zeros((W, n), dtype=np.float32)
    sent = np.zeros((W, n), dtype=np.float64)
    total = np.zeros((W, n), dtype=np.float64)
    for step in range(2):
        G = laplace_grads(W, n, tag=100 + step)
        E_in = E.copy()
        sp, E = gpu_topk(G, E_in, block, K)
        for k in range(W):
            check_worker(G[k], E_in[k], block, K, sp[k], E[k])
        sent += sp
        total += G
    # what was sent plus what is still owed equals what was produced (float32 sums)
    np.testing.assert_allclose(sent + E, total, rtol=0, atol=1e-5 * np.abs(total).max())


def test_block_topk_then_s2_path():
    # sparsify, then encode -> reduce -> decode the sparse gradients
    W, n, block, d, w = 4, 65_536, 256, 3, 4096
    nb = n // block
    G = laplace_grads(W, n, tag=5)
    sp, _ = gpu_topk(G, np.zeros_like(G), block, nb // 32)
    got = gpu_pipeline(torch.from_numpy(sp).to(DEV), d, w, 0, compact=True)
    check_pipeline(sp, "f32", got, d, w, 0)


@pytest.mark.slow
def test_block_topk_resnet50_size():
    W, n, block = 8, 25_557_032, 256
    nb = (n + block - 1) // block
    G = laplace_grads(W, n, tag=11)
    E = np.zeros_like(G)
    sp, e = gpu_topk(G, E, block, nb // 32)
    for k in range(W):
        check_worker(G[k], E[k], block, nb // 32, sp[k], e[k])
