"""GPU parity of the fused single-sketch mode (s2_encode_reduce_fused) against
the oracle's aggregation: the bitmap must equal the OR of the workers' bitmaps
bit for bit, and the sketch the sum of the workers' sketches within the
tolerance of the per-worker path (bit for bit on integer-valued gradients).
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


def run_fused(grad: torch.Tensor, d: int, w: int, seed: int):
    W, n = grad.shape
    bitmap = torch.full((max(s2.nwords(n), 1),), -1, dtype=torch.int32, device=DEV)
    sketch = torch.full((d, w), 7.0, dtype=torch.float32, device=DEV)
    s2.s2_encode_reduce_fused(grad, d, w, seed, bitmap[: s2.nwords(n)], sketch)
    torch.cuda.synchronize()
    return u32(bitmap[: s2.nwords(n)]), sketch.cpu().numpy()


def check(G: np.ndarray, dtype: str, d: int, w: int, seed: int, exact: bool = False):
    grad = torch.from_numpy(G if dtype == "f32" else G.view(np.int16)).to(DEV)
    if dtype == "bf16":
        grad = grad.view(torch.bfloat16)
    bm, sk = run_fused(grad, d, w, seed)
    ref = oracle.pipeline(G, d, w, seed, dtype=dtype)
    np.testing.assert_array_equal(bm, ref["bitmap"])
    if exact:
        np.testing.assert_array_equal(sk.astype(np.float64), ref["S_sum"])
    else:
        cnt = contribution_counts(ref["bitmaps"], G.shape[1], d, w, seed).sum(axis=0)
        assert_sketch_close(sk, ref["S_sum"], ref["A_sum"], what="fused sketch", cnt=cnt)
    return ref, bm, sk


CASES = [
    ("tiny", None),
    ("f32_ragged", dict(W=3, n=10_000, d=5, w=1000, density=0.1, tag=301)),
    ("f32_unaligned_rows", dict(W=3, n=1001, d=3, w=64, density=0.3, tag=302)),
    ("bf16", dict(W=4, n=8192, d=5, w=512, density=0.05, dtype="bf16", tag=303)),
    ("bf16_odd", dict(W=2, n=7777, d=3, w=300, density=0.2, dtype="bf16", tag=304)),
    ("d1", dict(W=2, n=5000, d=1, w=4096, density=0.02, tag=305)),
    ("d4", dict(W=5, n=6000, d=4, w=333, density=0.05, tag=306)),
    ("d9_generic", dict(W=3, n=9000, d=9, w=2048, density=0.03, tag=307)),
    ("many_workers", dict(W=13, n=4100, d=5, w=700, density=0.02, tag=308)),
    ("one_worker", dict(W=1, n=70_000, d=3, w=4096, density=0.05, tag=309)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_oracle_aggregate(name, kw):
    wl = workloads.tiny() if kw is None else workloads.custom(**kw)
    check(wl.dense(), wl.dtype, wl.d, wl.w, wl.seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_exact_on_integers(dtype):
    wl = workloads.custom(W=6, n=20_000, d=5, w=512, density=0.05, values="int", int_max=1024, dtype=dtype, tag=310)
    check(wl.dense(), dtype, wl.d, wl.w, wl.seed, exact=True)


def test_fused_cancellation_keeps_the_bit_and_adds_nothing():
    n, d, w = 4096, 3, 128
    g = np.zeros((2, n), dtype=np.float32)
    g[0, 10], g[1, 10] = 3.0, -3.0  # cancel exactly
    g[0, 20] = 5.0
    ref, bm, sk = check(g, "f32", d, w, 1, exact=True)
    assert unpack(bm, n)[10] and unpack(bm, n)[20]


def test_fused_then_decode_equals_per_worker_path_within_tolerance():
    wl = workloads.custom(W=4, n=50_000, d=5, w=2048, density=0.05, tag=311)
    G = wl.dense()
    bm, sk = run_fused(torch.from_numpy(G).to(DEV), wl.d, wl.w, wl.seed)
    out = torch.empty(wl.n, dtype=torch.float32, device=DEV)
    s2.s2_decode_dense(torch.from_numpy(bm.view(np.int32)).to(DEV), torch.from_numpy(sk).to(DEV), wl.n, wl.d,
                       wl.w, wl.seed, out)
    torch.cuda.synchronize()
    ref = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    cnt = contribution_counts(ref["bitmaps"], wl.n, wl.d, wl.w, wl.seed).sum(axis=0)
    union = np.flatnonzero(unpack(ref["bitmap"], wl.n)).astype(np.uint32)
    cmax = np.zeros(wl.n)
    b, _ = oracle.hash(union, wl.d, wl.w, wl.seed)
    cmax[union] = np.max(np.stack([cnt[j][b[j]] for j in range(wl.d)]), axis=0)
    assert_decoded_close(out.cpu().numpy(), ref["out"], ref["amax"], cmax=cmax)


def test_fused_empty_and_no_workers():
    for W, n in ((0, 5000), (3, 0)):
        grad = torch.zeros((W, n), dtype=torch.float32, device=DEV)
        bm, sk = run_fused(grad, 3, 64, 0)
        assert (bm == 0).all() and (sk == 0).all()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["embedding", "topk"])
def test_fused_full_size(name):
    wl = workloads.by_name(name)
    check(wl.dense(), wl.dtype, wl.d, wl.w, wl.seed)
