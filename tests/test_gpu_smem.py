"""GPU parity of the two encode accumulation paths against the oracle:
S2_PATH_SMEM (a per-block copy of the sketch in shared memory, added into the
global sketch at the end) and S2_PATH_L2 (reductions straight into the global
sketch). Bitmaps must match the oracle bit for bit on both paths, sketches
within the stated tolerance, and bit for bit on integer-valued gradients
(where every float32 partial sum is exact, so the two paths and the oracle
agree exactly whatever the order of the adds).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sketch_compressed_sparse_gb300 as s2
    from tests._parity import assert_sketch_close, contribution_counts, u32

DEV = "cuda"


def encode(wl, path, grad=None):
    g = wl.dense_torch(DEV) if grad is None else grad
    W, n = g.shape
    bitmaps = torch.full((W, max(s2.nwords(n), 1)), -1, dtype=torch.int32, device=DEV)[:, : s2.nwords(n)].contiguous()
    sketches = torch.full((W, wl.d, wl.w), 7.0, dtype=torch.float32, device=DEV)
    s2.s2_encode_batched_path(g, wl.d, wl.w, wl.seed, bitmaps, sketches, path=path)
    torch.cuda.synchronize()
    return u32(bitmaps), sketches.cpu().numpy()


def check(wl, path, exact=False):
    bm, sk = encode(wl, path)
    G = wl.dense()
    rbm, S, A = oracle.encode_all(G, wl.d, wl.w, wl.seed, wl.dtype)
    np.testing.assert_array_equal(bm, rbm)
    if exact:
        np.testing.assert_array_equal(sk.astype(np.float64), S)
    else:
        cnt = contribution_counts(rbm, wl.n, wl.d, wl.w, wl.seed)
        for k in range(wl.W):
            assert_sketch_close(sk[k], S[k], A[k], what=f"{path} sketch of worker {k}", cnt=cnt[k])
    return bm, sk


CASES = [
    ("tiny", None),
    ("sweep_n20_rho0.1pct_d3", dict(W=8, n=1 << 20, d=3, w=512, density=0.001, tag=601)),
    ("sweep_n20_rho1pct_d5", dict(W=8, n=1 << 20, d=5, w=4096, density=0.01, tag=602)),
    ("bf16_vec", dict(W=4, n=8192 * 3, d=5, w=512, density=0.05, dtype="bf16", tag=603)),
    ("f32_unaligned_rows", dict(W=3, n=1001, d=3, w=64, density=0.3, tag=604)),
    ("bf16_unaligned_rows", dict(W=2, n=7777, d=3, w=300, density=0.2, dtype="bf16", tag=605)),
    ("d9_generic", dict(W=3, n=9000, d=9, w=2048, density=0.03, tag=606)),
    ("odd_dw", dict(W=2, n=20_000, d=5, w=333, density=0.05, tag=607)),          # d*w not a multiple of 4
    ("largest_sketch_no_merge", dict(W=2, n=1 << 21, d=3, w=16384, density=0.02, tag=608)),  # 192 KiB, w > 4096
    ("one_worker_many_blocks", dict(W=1, n=1 << 22, d=3, w=1024, density=0.01, tag=609)),
    ("many_workers", dict(W=13, n=4100, d=5, w=700, density=0.02, tag=610)),
    ("dense_rows_small_w", dict(W=2, n=50_000, d=3, w=256, density=1.0, tag=611)),  # every lane collides often
]


@pytest.mark.parametrize("path", ["smem", "l2"])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_path_matches_oracle(name, kw, path):
    wl = workloads.tiny() if kw is None else workloads.custom(**kw)
    check(wl, path)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("w", [1, 7, 256, 8192])
def test_paths_exact_on_integers(dtype, w):
    # w = 1: every nonzero of a worker lands in the one bucket of each row,
    # so every lane of every warp hits the same address
    wl = workloads.custom(W=4, n=30_000, d=3, w=w, density=0.05, values="int", int_max=64, dtype=dtype, tag=620 + w)
    bm_s, sk_s = check(wl, "smem", exact=True)
    bm_l, sk_l = check(wl, "l2", exact=True)
    np.testing.assert_array_equal(bm_s, bm_l)
    np.testing.assert_array_equal(sk_s.view(np.uint32), sk_l.view(np.uint32))


def test_auto_takes_either_path_with_the_same_results():
    for kw in (dict(W=2, n=4096, d=3, w=256, density=0.1, tag=630),          # small sketch
               dict(W=2, n=1 << 16, d=5, w=1 << 14, density=0.05, tag=631)):  # 320 KiB: L2 only
        check(workloads.custom(**kw), "auto")


def test_smem_rejects_a_sketch_too_large_for_shared_memory():
    d, w = 5, 1 << 14  # 320 KiB
    g = torch.zeros((1, 1024), device=DEV)
    bm = torch.zeros((1, 32), dtype=torch.int32, device=DEV)
    sk = torch.zeros((1, d, w), device=DEV)
    with pytest.raises(s2.S2Error) as e:
        s2.s2_encode_batched_path(g, d, w, 0, bm, sk, path="smem")
    assert e.value.status == 3
    with pytest.raises(s2.S2Error) as e:
        s2.s2_encode_batched_path(g, d, w, 0, bm, sk, path=7)
    assert e.value.status == 1


def test_smem_empty_inputs():
    for W, n in ((0, 5000), (3, 0)):
        g = torch.zeros((W, n), dtype=torch.float32, device=DEV)
        bm = torch.zeros((W, max(s2.nwords(n), 1)), dtype=torch.int32, device=DEV)
        sk = torch.full((W, 3, 64), 7.0, device=DEV)
        s2.s2_encode_batched_path(g, 3, 64, 0, bm, sk, path="smem")
        torch.cuda.synchronize()
        assert (sk == 0).all()


def test_block_bitmap_through_the_smem_path():
    # 64 buckets a row for 2^20 positions: the automatic choice is the
    # shared-memory path (n >= 4096 w; the block copies' additions are well
    # under the gradient read)
    wl = workloads.custom(W=2, n=1 << 20, d=3, w=64, density=0.01, tag=640)
    block = 64
    G = wl.dense()
    g = wl.dense_torch(DEV)
    nbw = s2.nblockwords(wl.n, block)
    bms = torch.full((wl.W, nbw), -1, dtype=torch.int32, device=DEV)
    sks = torch.empty((wl.W, wl.d, wl.w), device=DEV)
    s2.s2_encode_batched_blocks(g, block, wl.d, wl.w, wl.seed, bms, sks)
    torch.cuda.synchronize()
    for k in range(wl.W):
        rbm, S, A = oracle.encode_blocks(G[k], block, wl.d, wl.w, wl.seed)
        np.testing.assert_array_equal(u32(bms[k]), rbm)
        assert_sketch_close(sks[k].cpu().numpy(), S, A, what=f"block-mode sketch of worker {k}",
                            cnt=contribution_counts(oracle.encode(G[k], wl.d, wl.w, wl.seed)[0][None], wl.n, wl.d,
                                                    wl.w, wl.seed)[0])
