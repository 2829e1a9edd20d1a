"""GPU parity of the block-wise Top-K sparsifier with error feedback
(s2_block_topk) against the oracle. The block norms are computed in the same
float32 order on both sides, so the kept blocks, the sparse output and the
new residual must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sketch_compressed_sparse_gb300 as s2
    from tests._parity import check_pipeline, gpu_pipeline

DEV = "cuda"


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


def oracle_topk(G, E, block, K):
    sps, es = [], []
    for k in range(G.shape[0]):
        sp, e, _, _ = oracle.block_topk(G[k], E[k], block, K)
        sps.append(sp)
        es.append(e)
    return np.stack(sps), np.stack(es)


@pytest.mark.parametrize("W,n,block,K", [
    (3, 10_000, 32, 10),
    (3, 10_000, 64, 0),
    (2, 10_001, 64, 157),        # K = nb: every block kept; ragged last block
    (4, 65_536, 256, 8),
    (1, 100_000, 96, 33),
    (2, 5_000, 1024, 2),
])
def test_block_topk_bit_exact(W, n, block, K):
    G = laplace_grads(W, n, tag=W * 7 + K)
    E = (0.05 * np.random.default_rng(K).normal(size=(W, n))).astype(np.float32)
    sp, e = gpu_topk(G, E, block, K)
    rsp, re = oracle_topk(G, E, block, K)
    np.testing.assert_array_equal(sp.view(np.uint32), rsp.view(np.uint32))
    np.testing.assert_array_equal(e.view(np.uint32), re.view(np.uint32))


def test_block_topk_ties_go_to_the_lower_block():
    G = np.ones((2, 32 * 40), dtype=np.float32)  # 40 equal blocks per worker
    G[1, 32 * 5:32 * 6] = 2.0                      # worker 1: block 5 is the largest
    sp, e = gpu_topk(G, np.zeros_like(G), 32, 3)
    kept0 = np.flatnonzero(sp[0].reshape(40, 32).any(axis=1))
    kept1 = np.flatnonzero(sp[1].reshape(40, 32).any(axis=1))
    np.testing.assert_array_equal(kept0, [0, 1, 2])
    np.testing.assert_array_equal(kept1, [0, 1, 5])


def test_block_topk_two_steps_of_error_feedback():
    W, n, block, K = 3, 20_000, 64, 9
    E = np.zeros((W, n), dtype=np.float32)
    Eo = E.copy()
    for step in range(2):
        G = laplace_grads(W, n, tag=100 + step)
        sp, E = gpu_topk(G, E, block, K)
        rsp, Eo = oracle_topk(G, Eo, block, K)
        np.testing.assert_array_equal(sp.view(np.uint32), rsp.view(np.uint32))
        np.testing.assert_array_equal(E.view(np.uint32), Eo.view(np.uint32))


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
    rsp, re = oracle_topk(G, E, block, nb // 32)
    np.testing.assert_array_equal(sp.view(np.uint32), rsp.view(np.uint32))
    np.testing.assert_array_equal(e.view(np.uint32), re.view(np.uint32))
