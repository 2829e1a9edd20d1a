"""Pins for the CPU oracle: each test ties it to something other than itself.

Source of what is pinned: "S2 Reducer: High-Performance Sparse Communication
to Accelerate Distributed Deep Learning", Section 3.1 (compression, the
AllReduce of the sketch, decompression), Algorithm 1, and Appendix A.1 (the
proof of Theorem 1: the mapping matrix A and the collision probabilities).
The hash family is the MurmurHash3 finalizer, pinned by published vectors.
"""
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def support_bitmap(nonzero_mask: np.ndarray) -> np.ndarray:
    """Pack a boolean mask into LSB-first uint32 words with numpy's packbits."""
    n = nonzero_mask.size
    nw = (n + 31) // 32
    padded = np.zeros(nw * 32, dtype=bool)
    padded[:n] = nonzero_mask
    return np.packbits(padded, bitorder="little").view("<u4").astype(np.uint32)


def unpack_bits(bitmap: np.ndarray, n: int) -> np.ndarray:
    return np.unpackbits(bitmap.astype("<u4").view(np.uint8), bitorder="little")[:n].astype(bool)


def mapping_matrix(n: int, j: int, d: int, w: int, seed: int) -> np.ndarray:
    """A_j in {-1,0,+1}^{n x w}: A_j[i, h_j(i)] = s_j(i) (Section 3.1, mapping matrix)."""
    b, s = oracle.hash(np.arange(n, dtype=np.uint32), d, w, seed)
    A = np.zeros((n, w))
    A[np.arange(n), b[j]] = s[j]
    return A


# ---------------------------------------------------------------- hash family

def test_fmix32_published_vectors():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "murmur3_fmix32.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 3
    for seed, expect in rows:
        assert oracle.fmix32(int(seed, 16)) == int(expect, 16)


def test_fmix32_is_a_bijection_on_a_sample():
    # The finalizer is a composition of invertible steps; no two sampled inputs may collide.
    x = np.random.default_rng(1).integers(0, 2**32, size=20000, dtype=np.uint64)
    x = np.unique(x)
    y = {oracle.fmix32(int(v)) for v in x}
    assert len(y) == x.size


@pytest.mark.parametrize("w", [1, 2, 3, 255, 256, 1000, 1 << 20, (1 << 31) + 12345])
def test_bucket_range_and_signs(w):
    idx = np.random.default_rng(w % 1000).integers(0, 2**32, size=4096, dtype=np.uint64).astype(np.uint32)
    b, s = oracle.hash(idx, 4, w, seed=7)
    assert b.max() < w
    if w == 1:
        assert (b == 0).all()
    assert set(np.unique(s).tolist()) <= {-1, 1}


def test_bucket_uniformity_and_sign_balance():
    m = 1 << 20
    w = 1024
    b, s = oracle.hash(np.arange(m, dtype=np.uint32), 5, w, seed=0)
    for j in range(5):
        cnt = np.bincount(b[j], minlength=w)
        exp = m / w
        chi2 = ((cnt - exp) ** 2 / exp).sum()
        # chi-square with w-1 dof: mean 1023, sd ~45
        assert abs(chi2 - (w - 1)) < 8 * np.sqrt(2 * (w - 1)), chi2
        plus = int((s[j] == 1).sum())
        assert abs(plus - m / 2) < 6 * np.sqrt(m / 4), plus


def test_pairwise_collision_probability():
    # Appendix A.1: for i != i', Pr[A A^T(i,i') = +1] = Pr[= -1] = 0.5/m.
    m = 64
    N = 1 << 20
    rng = np.random.default_rng(5)
    i = rng.integers(0, 2**31, size=N, dtype=np.uint64).astype(np.uint32)
    i2 = (i.astype(np.uint64) + rng.integers(1, 2**20, size=N)).astype(np.uint32)
    b1, s1 = oracle.hash(i, 1, m, seed=3)
    b2, s2 = oracle.hash(i2, 1, m, seed=3)
    coll = b1[0] == b2[0]
    plus = (coll & (s1[0] == s2[0])).sum()
    minus = (coll & (s1[0] != s2[0])).sum()
    exp = N * 0.5 / m
    sd = np.sqrt(exp)
    assert abs(plus - exp) < 6 * sd and abs(minus - exp) < 6 * sd, (plus, minus, exp)


def test_rows_use_independent_hashes():
    w = 256
    m = 1 << 18
    b, s = oracle.hash(np.arange(m, dtype=np.uint32), 4, w, seed=11)
    for j in range(1, 4):
        same = (b[0] == b[j]).mean()
        assert abs(same - 1 / w) < 6 * np.sqrt(1 / w / m)
        agree = (s[0] == s[j]).mean()
        assert abs(agree - 0.5) < 6 * np.sqrt(0.25 / m)


def test_bucket_is_the_high_part_of_a_multiply_shift():
    # Multiply-shift keeps the HIGH bits of hash * w: halving a power-of-two w
    # drops the lowest bit of the bucket (a modulo reduction would keep the low
    # bits instead), and w = 1 maps everything to bucket 0.
    idx = np.random.default_rng(3).integers(0, 2**32, size=50000, dtype=np.uint64).astype(np.uint32)
    prev, _ = oracle.hash(idx, 3, 2, seed=19)
    assert ((prev == 0) | (prev == 1)).all()
    for k in range(2, 32):
        cur, _ = oracle.hash(idx, 3, 1 << k, seed=19)
        np.testing.assert_array_equal(cur >> 1, prev)
        prev = cur
    # a non-power-of-two w is monotone in w for a fixed hash value
    b7, _ = oracle.hash(idx, 1, 7, seed=19)
    b9, _ = oracle.hash(idx, 1, 9, seed=19)
    assert (b7 <= b9).all()


def test_row_keys_use_the_golden_ratio_constant():
    # Row j's keys mix the seed with odd multiples of floor(2^32 / phi). For
    # seed 0 and row 0 the bucket key is fmix32(floor(2^32 / phi)).
    from decimal import Decimal, getcontext

    getcontext().prec = 50
    phi = (1 + Decimal(5).sqrt()) / 2
    golden = int(Decimal(2**32) / phi)
    assert golden == 0x9E3779B9
    kh0, ks0 = oracle.row_keys(0, 0)
    assert kh0 == oracle.fmix32(golden)
    assert ks0 == oracle.fmix32((2 * golden) % 2**32)
    kh3, ks3 = oracle.row_keys(0xABCDEF01, 3)
    assert kh3 == oracle.fmix32(0xABCDEF01 ^ ((7 * golden) % 2**32))
    assert ks3 == oracle.fmix32(0xABCDEF01 ^ ((8 * golden) % 2**32))


def test_seed_changes_hashes():
    idx = np.arange(10000, dtype=np.uint32)
    b0, _ = oracle.hash(idx, 3, 1 << 16, seed=0)
    b1, _ = oracle.hash(idx, 3, 1 << 16, seed=1)
    assert (b0 != b1).mean() > 0.99


# ----------------------------------------------------------------- bitmap

def test_bitmap_is_exact_support_fp32():
    n = 1000  # not a multiple of 32: a ragged last word
    g = np.zeros(n, dtype=np.float32)
    pos = np.array([0, 1, 31, 32, 63, 500, 998, 999])
    vals = np.array([1.0, -2.5, 1e-45, -1e-45, 3e38, -7.0, 1e-38, 0.5], dtype=np.float32)  # incl. subnormals
    g[pos] = vals
    g[[2, 3, 100]] = np.float32(-0.0)  # negative zero is zero
    bm, S, A = oracle.encode(g, 3, 64, 0)
    mask = np.zeros(n, dtype=bool)
    mask[pos] = True
    np.testing.assert_array_equal(bm, support_bitmap(mask))
    assert bm[-1] >> (n % 32) == 0  # tail bits are zero


def test_bitmap_is_exact_support_bf16():
    n = 77
    g = np.zeros(n, dtype=np.uint16)
    pos = np.array([0, 5, 32, 40, 76])
    g[pos] = np.array([0x3F80, 0x0001, 0x8001, 0xBF80, 0x7F7F], dtype=np.uint16)  # incl. subnormals
    g[[1, 2]] = 0x8000  # -0.0
    bm, _, _ = oracle.encode(g, 2, 8, 0, dtype="bf16")
    mask = np.zeros(n, dtype=bool)
    mask[pos] = True
    np.testing.assert_array_equal(bm, support_bitmap(mask))


# ----------------------------------------------------------------- sketch

@pytest.mark.parametrize("d,w,seed", [(1, 16, 0), (3, 16, 5), (5, 7, 123)])
def test_sparse_insertion_equals_dense_projection(d, w, seed):
    # Section 3.1: inserting only the nonzeros gives the sketch of the dense
    # gradient, and bucket b of row j holds A_j^T(b,:) g.
    n = 300
    rng = np.random.default_rng(d * 100 + w)
    g = rng.normal(size=n).astype(np.float32)
    g[rng.random(n) < 0.6] = 0
    bm, S, _ = oracle.encode(g, d, w, seed)
    for j in range(d):
        Aj = mapping_matrix(n, j, d, w, seed)
        np.testing.assert_allclose(S[j], Aj.T @ g.astype(np.float64), rtol=0, atol=1e-12)


def test_contribution_magnitudes():
    n = 200
    rng = np.random.default_rng(2)
    g = rng.normal(size=n).astype(np.float32)
    g[::3] = 0
    _, _, A = oracle.encode(g, 3, 8, 9)
    for j in range(3):
        Aj = np.abs(mapping_matrix(n, j, 3, 8, 9))
        np.testing.assert_allclose(A[j], Aj.T @ np.abs(g.astype(np.float64)), atol=1e-12)


# ----------------------------------------------------------------- reduce

def test_reduce_is_linear_and_bitmaps_union():
    # Section 3.1: A^T sum_k g_k = sum_k A^T g_k; the aggregate bitmap marks the
    # union of the workers' nonzero positions.
    wl = workloads.custom(W=4, n=3000, d=3, w=97, density=0.05, values="int", tag=21)
    G = wl.dense()
    bms, S, A = oracle.encode_all(G, wl.d, wl.w, wl.seed)
    bm, Ssum, Asum = oracle.reduce(bms, S, A)
    gsum = G.astype(np.float64).sum(axis=0).astype(np.float32)  # integers: exact
    _, S_of_sum, _ = oracle.encode(gsum, wl.d, wl.w, wl.seed)
    np.testing.assert_array_equal(Ssum, S_of_sum)
    np.testing.assert_array_equal(bm, support_bitmap((G != 0).any(axis=0)))
    np.testing.assert_allclose(Asum, A.sum(axis=0))


# ----------------------------------------------------------------- decode

def _union_collision_free_rows(idx_union, d, w, seed):
    b, _ = oracle.hash(idx_union.astype(np.uint32), d, w, seed)
    free = np.zeros(idx_union.size, dtype=int)
    for j in range(d):
        cnt = np.bincount(b[j], minlength=w)
        free += cnt[b[j]] == 1
    return free


@pytest.mark.parametrize("d", [1, 3, 5])
def test_decode_is_exact_without_majority_collisions(d):
    # Decompression recovers the summed gradient wherever a strict majority of
    # a key's rows hold no other nonzero (the median then picks the true sum).
    wl = workloads.custom(W=3, n=20000, d=d, w=1 << 12, density=0.004, values="int", tag=31 + d)
    G = wl.dense()
    res = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    union = np.flatnonzero((G != 0).any(axis=0))
    free = _union_collision_free_rows(union, d, wl.w, wl.seed)
    good = union[free * 2 > d]
    assert good.size > 0.9 * union.size
    gsum = G.astype(np.float64).sum(axis=0)
    np.testing.assert_array_equal(res["out"][good], gsum[good].astype(np.float32))
    # nothing outside the union
    off = np.ones(wl.n, dtype=bool)
    off[union] = False
    assert (res["out"][off].view(np.uint32) == 0).all()


def _find_partner(i, rows_wanted, d, w, seed, start=1):
    """Smallest index i' != i that shares h_j(i) exactly in the rows ``rows_wanted``."""
    bi, _ = oracle.hash(np.array([i], dtype=np.uint32), d, w, seed)
    cand = np.arange(start, start + 2_000_000, dtype=np.uint32)
    bc, _ = oracle.hash(cand, d, w, seed)
    same = bc == bi[:, :1]
    want = np.zeros(d, dtype=bool)
    want[list(rows_wanted)] = True
    ok = (same == want[:, None]).all(axis=0) & (cand != i)
    hits = cand[ok]
    assert hits.size, "no partner found"
    return int(hits[0])


def test_median_rejects_a_minority_collision():
    d, w, seed = 3, 64, 4
    i = 5
    p = _find_partner(i, [1], d, w, seed, start=10)
    n = max(i, p) + 1
    g = np.zeros(n, dtype=np.float32)
    g[i], g[p] = 10.0, 1000.0
    res = oracle.pipeline(g[None, :], d, w, seed)
    assert res["out"][i] == 10.0 and res["out"][p] == 1000.0


def test_median_fails_on_a_majority_collision():
    d, w, seed = 3, 64, 4
    i = 5
    p = _find_partner(i, [0, 2], d, w, seed, start=10)
    n = max(i, p) + 1
    g = np.zeros(n, dtype=np.float32)
    g[i], g[p] = 10.0, 1000.0
    res = oracle.pipeline(g[None, :], d, w, seed)
    assert res["out"][i] != 10.0  # two of three estimates carry +-1000


@pytest.mark.parametrize("W", [1, 3])
def test_bruteforce_d1_is_A_At_g(W):
    # Section 3.1: the query of key i is A(i,:) A^T g; with one row the median
    # is that single estimate. Tiny sizes, every set bit checked.
    n, w, seed = 64, 8, 17
    rng = np.random.default_rng(W)
    G = rng.integers(-50, 51, size=(W, n)).astype(np.float32)
    G[rng.random((W, n)) < 0.7] = 0
    res = oracle.pipeline(G, 1, w, seed)
    A = mapping_matrix(n, 0, 1, w, seed)
    ghat = A @ (A.T @ G.astype(np.float64).sum(axis=0))
    setbits = (G != 0).any(axis=0)
    np.testing.assert_array_equal(res["out"][setbits], ghat[setbits].astype(np.float32))
    assert (res["out"][~setbits] == 0).all()


@pytest.mark.parametrize("d", [1, 2, 3, 4, 5, 6, 8, 16])
def test_median_of_planted_estimates(d):
    # Plant sketch values so that key i's estimates are known numbers v_ij; the
    # decode must return numpy's median of them (mean of the middle pair for even d).
    n, w, seed = 4096, 1 << 16, 23
    rng = np.random.default_rng(d)
    keys = np.sort(rng.choice(n, size=60, replace=False)).astype(np.uint32)
    b, _ = oracle.hash(keys, d, w, seed)
    alone = np.ones(keys.size, dtype=bool)
    for j in range(d):  # keep only keys whose buckets belong to no other key
        cnt = np.bincount(b[j], minlength=w)
        alone &= cnt[b[j]] == 1
    keys = keys[alone]
    assert keys.size >= 30
    b, s = oracle.hash(keys, d, w, seed)
    S = np.zeros((d, w))
    V = rng.integers(-1000, 1001, size=(d, keys.size)).astype(np.float64)
    for j in range(d):
        S[j, b[j]] = s[j] * V[j]
    bm = support_bitmap(np.isin(np.arange(n), keys))
    out, _ = oracle.decode_dense(bm, S, n, seed)
    np.testing.assert_array_equal(out[keys], np.median(V, axis=0).astype(np.float32))


def test_decode_scale_and_zero_fill():
    wl = workloads.custom(W=2, n=5000, d=3, w=64, density=0.05, tag=41)
    G = wl.dense()
    bms, S, A = oracle.encode_all(G, wl.d, wl.w, wl.seed)
    bm, Ssum, Asum = oracle.reduce(bms, S, A)
    o1, _ = oracle.decode_dense(bm, Ssum, wl.n, wl.seed, 1.0, Asum)
    o8, _ = oracle.decode_dense(bm, Ssum, wl.n, wl.seed, 0.125, Asum)
    np.testing.assert_array_equal(o8, o1 * np.float32(0.125))
    unset = ~unpack_bits(bm, wl.n)
    assert (o1[unset].view(np.uint32) == 0).all()  # exactly +0.0


def test_compact_matches_flatnonzero_and_dense():
    n, d, w, seed = 10_000, 3, 512, 2
    bm = workloads.random_bitmaps(1, n, 0.03, tag=51)[0]
    S = workloads.random_sketches(1, d, w, tag=52)[0].astype(np.float64)
    dense, _ = oracle.decode_dense(bm, S, n, seed, 0.5)
    cnt, idx, val, _ = oracle.decode_compact(bm, S, n, seed, 0.5)
    expect_idx = np.flatnonzero(unpack_bits(bm, n))
    assert cnt == expect_idx.size
    np.testing.assert_array_equal(idx, expect_idx.astype(np.uint32))
    np.testing.assert_array_equal(val, dense[expect_idx])
    # capacity: the count stays exact, only the first entries are written
    cnt2, idx2, val2, _ = oracle.decode_compact(bm, S, n, seed, 0.5, capacity=17)
    assert cnt2 == cnt and idx2.size == 17
    np.testing.assert_array_equal(idx2, idx[:17])


def test_bf16_inputs_match_the_same_values_in_fp32():
    wl = workloads.custom(W=2, n=3000, d=3, w=128, density=0.1, dtype="bf16", tag=61)
    Gb = wl.dense()
    Gf = workloads.bf16_bits_to_f32(Gb)
    rb = oracle.pipeline(Gb, wl.d, wl.w, wl.seed, dtype="bf16")
    rf = oracle.pipeline(Gf, wl.d, wl.w, wl.seed, dtype="f32")
    np.testing.assert_array_equal(rb["bitmap"], rf["bitmap"])
    np.testing.assert_array_equal(rb["S_sum"], rf["S_sum"])
    np.testing.assert_array_equal(rb["out"], rf["out"])


def test_unbiased_estimate_with_one_row():
    # Theorem 1 / Appendix A.1: with one bucket array, E[g^] = g over the random
    # hash; here the seed is the randomness. Statistical, 1000 seeds.
    n, w = 48, 8
    rng = np.random.default_rng(71)
    g = rng.integers(-20, 21, size=n).astype(np.float32)
    g[g == 0] = 3
    probe = [0, 7, 30]
    errs = []
    for seed in range(1000):
        res = oracle.pipeline(g[None, :], 1, w, seed)
        errs.append(res["out"][probe].astype(np.float64) - g[probe])
    errs = np.array(errs)
    mean = errs.mean(axis=0)
    se = errs.std(axis=0, ddof=1) / np.sqrt(errs.shape[0])
    assert (np.abs(mean) < 4 * se).all(), (mean, se)


def test_tiny_workload_pipeline_invariants():
    wl = workloads.tiny()
    G = wl.dense()
    res = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    union = (G != 0).any(axis=0)
    np.testing.assert_array_equal(unpack_bits(res["bitmap"], wl.n), union)
    assert (res["out"][~union] == 0).all()
    # estimates are finite and bounded by the largest bucket magnitude
    assert np.isfinite(res["out"]).all()
    assert (np.abs(res["out"][union]) <= res["amax"][union] + 1e-6).all()


# ----------------------------------------------------------------- block-granular bitmap

@pytest.mark.parametrize("block", [1, 7, 32, 512])
def test_block_bitmap_marks_blocks_with_a_nonzero(block):
    # Section 3.1: one bit per block, set iff the block holds a nonzero
    n = 5000
    rng = np.random.default_rng(block)
    g = np.zeros(n, dtype=np.float32)
    pos = rng.choice(n, size=40, replace=False)
    g[pos] = rng.normal(size=40).astype(np.float32)
    g[rng.choice(n, size=10)] = np.float32(-0.0)
    bm, S, _ = oracle.encode_blocks(g, block, 3, 64, 5)
    nb = (n + block - 1) // block
    padded = np.zeros(nb * block, dtype=bool)
    padded[:n] = g.view(np.uint32) & 0x7FFFFFFF != 0
    np.testing.assert_array_equal(bm, support_bitmap(padded.reshape(nb, block).any(axis=1)))
    _, S_elem, _ = oracle.encode(g, 3, 64, 5)
    np.testing.assert_array_equal(S, S_elem)  # zeros are never inserted: same sketch


def test_block_size_one_is_the_element_path():
    wl = workloads.custom(W=3, n=3000, d=5, w=97, density=0.05, tag=81)
    G = wl.dense()
    rb = oracle.pipeline_blocks(G, 1, wl.d, wl.w, wl.seed)
    re_ = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    np.testing.assert_array_equal(rb["bitmap"], re_["bitmap"])
    np.testing.assert_array_equal(rb["out"], re_["out"])


def test_block_decode_recovers_whole_blocks_exactly_without_collisions():
    # every position of a marked block is recovered, the zeros in it as 0.0
    n, block, d, w, seed = 8192, 512, 3, 1 << 22, 9
    G = np.zeros((2, n), dtype=np.float32)
    G[0, 512:560] = np.arange(1, 49, dtype=np.float32)
    G[1, 4096 + 100] = -7.0
    res = oracle.pipeline_blocks(G, block, d, w, seed)
    marked = np.zeros(n, dtype=bool)
    marked[512:1024] = True
    marked[4096:4608] = True
    np.testing.assert_array_equal(unpack_bits(res["bitmap"], n // block), [False, True] + [False] * 6 + [True] + [False] * 6 + [False])
    assert (res["out"][~marked] == 0).all()
    np.testing.assert_array_equal(res["out"][marked], G.sum(axis=0)[marked])


# ----------------------------------------------------------------- block-wise Top-K + error feedback

def _topk_case(n=10_000, block=64, tag=0):
    rng = np.random.default_rng(tag)
    g = rng.laplace(size=n).astype(np.float32)
    e = (0.1 * rng.normal(size=n)).astype(np.float32)
    return g, e


@pytest.mark.parametrize("n,block,K", [(10_000, 64, 5), (10_000, 64, 0), (10_000, 64, 157), (1000, 96, 3),
                                        (4096, 256, 1)])
def test_block_topk_keeps_the_largest_blocks(n, block, K):
    # Section 2.2: the K blocks with the largest l2 norms are kept
    g, e = _topk_case(n, block, tag=K)
    sp, e2, nrm, keep = oracle.block_topk(g, e, block, K)
    acc = g + e  # float32 additions, as the method does
    nb = (n + block - 1) // block
    ref = np.array([np.linalg.norm(acc[x * block:(x + 1) * block].astype(np.float64)) ** 2 for x in range(nb)])
    np.testing.assert_allclose(nrm, ref, rtol=1e-13)  # the float64 norm, whatever the summation order
    order = np.lexsort((np.arange(nb), -nrm))
    want = np.zeros(nb, dtype=np.uint8)
    want[order[:K]] = 1
    np.testing.assert_array_equal(keep, want)
    kept = np.repeat(keep.astype(bool), block)[:n]
    np.testing.assert_array_equal(sp, np.where(kept, acc, 0).astype(np.float32))
    np.testing.assert_array_equal(sp + e2, acc)  # residual carries exactly what was not sent
    assert (e2[kept] == 0).all()
    sp3, e3 = oracle.block_split(g, e, block, keep)  # the split alone, given the same kept blocks
    np.testing.assert_array_equal(sp3.view(np.uint32), sp.view(np.uint32))
    np.testing.assert_array_equal(e3.view(np.uint32), e2.view(np.uint32))


def test_block_topk_worked_four_block_case():
    # Blocks of two elements, worked by hand (squared norms of grad + residual):
    #   block 0: [3, -4]            -> 25
    #   block 1: [0, -5]            -> 25
    #   block 2: [4.9, 0] + [0, 1.5] -> 24.01 + 2.25 = 26.26
    #   block 3: [-1, -4.95]        -> 1 + 24.5025 = 25.5025
    # K = 2 keeps blocks 2 and 3; K = 3 adds block 0 (25 = 25, lower index).
    # Ranking by the signed sum, |sum|, max |x|, the gradient without the
    # residual, or ties to the higher index would keep another set.
    g = np.array([3, -4, 0, -5, 4.9, 0, -1, -4.95], dtype=np.float32)
    e = np.array([0, 0, 0, 0, 0, 1.5, 0, 0], dtype=np.float32)
    _, _, nrm, keep = oracle.block_topk(g, e, 2, 2)
    np.testing.assert_allclose(nrm, [25.0, 25.0, 26.26, 25.5025], rtol=1e-6)
    np.testing.assert_array_equal(keep, [0, 0, 1, 1])
    sp, e2, _, keep3 = oracle.block_topk(g, e, 2, 3)
    np.testing.assert_array_equal(keep3, [1, 0, 1, 1])
    np.testing.assert_array_equal(sp, np.array([3, -4, 0, 0, 4.9, 1.5, -1, -4.95], dtype=np.float32))
    np.testing.assert_array_equal(e2, np.array([0, 0, 0, -5, 0, 0, 0, 0], dtype=np.float32))


def test_block_topk_ties_go_to_the_lower_block():
    g = np.ones(4 * 32, dtype=np.float32)  # four equal blocks
    _, _, _, keep = oracle.block_topk(g, np.zeros_like(g), 32, 2)
    np.testing.assert_array_equal(keep, [1, 1, 0, 0])


def test_block_topk_is_a_delta_approximate_compressor():
    # Theorem 2 / Appendix A.2: ||acc - sparse||^2 <= (1 - K/nb) ||acc||^2
    g, e = _topk_case(20_000, 100, tag=7)
    for K in (1, 10, 50, 199):
        sp, _, _, _ = oracle.block_topk(g, e, 100, K)
        acc = (g + e).astype(np.float64)
        lost = np.sum((acc - sp) ** 2)
        assert lost <= (1 - K / 200) * np.sum(acc ** 2) + 1e-9


def test_block_topk_error_feedback_accumulates_what_was_dropped():
    # two steps: the residual of step 1 joins the gradient of step 2
    g1, _ = _topk_case(5000, 50, tag=1)
    g2, _ = _topk_case(5000, 50, tag=2)
    e0 = np.zeros(5000, dtype=np.float32)
    sp1, e1, _, _ = oracle.block_topk(g1, e0, 50, 10)
    sp2, e2, _, _ = oracle.block_topk(g2, e1, 50, 10)
    np.testing.assert_allclose(sp1.astype(np.float64) + sp2 + e2, g1.astype(np.float64) + g2, atol=1e-5)


# ----------------------------------------------------------------- sparse AllGather baseline

def test_sparse_list_is_the_ascending_support():
    g = np.zeros(3000, dtype=np.float32)
    pos = np.array([3, 40, 41, 2999])
    g[pos] = [1.5, -2.0, 1e-45, 7.0]
    g[100] = np.float32(-0.0)
    c, idx, val = oracle.sparse_list(g)
    assert c == 4
    np.testing.assert_array_equal(idx, pos.astype(np.uint32))
    np.testing.assert_array_equal(val, g[pos])
    c2, idx2, _ = oracle.sparse_list(g, capacity=2)
    assert c2 == 4 and idx2.size == 2


def test_exact_sum_and_agreement_with_the_sketch_without_collisions():
    wl = workloads.custom(W=4, n=20_000, d=3, w=1 << 20, density=0.002, values="int", tag=91)
    G = wl.dense()
    ex = oracle.exact_sum(G)
    np.testing.assert_array_equal(ex, G.astype(np.float64).sum(axis=0).astype(np.float32))
    res = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    union = (G != 0).any(axis=0)
    free = _union_collision_free_rows(np.flatnonzero(union), wl.d, wl.w, wl.seed)
    good = np.flatnonzero(union)[free == wl.d]
    assert good.size > 0.95 * union.sum()
    np.testing.assert_array_equal(res["out"][good], ex[good])
