"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU oracle.

Every case draws its inputs from the seeded generators in ``workloads`` and
compares element by element (rules in ``tests/_parity.py``). Sizes span
several 512-position tasks and end in ragged tails; the edge cases are the
empty gradient, all-zero and all-nonzero gradients, -0.0 and subnormals,
one bucket per row, unaligned worker rows (scalar-load kernel), bf16 inputs,
every row count class (templated d = 1, 3, 5 and the generic kernel).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sketch_compressed_sparse_gb300 as s2
    from tests._parity import (assert_decoded_close, assert_sketch_close, check_pipeline, gpu_pipeline, u32,
                               unpack)

DEV = "cuda"


def _grad(wl):
    return wl.dense_torch(DEV)


# ------------------------------------------------------------------ hash

@pytest.mark.parametrize("d,w,seed", [(1, 1, 0), (3, 256, 0), (5, 1 << 20, 7), (16, 3, 123456789),
                                      (4, (1 << 31), 0xFFFFFFFF), (7, 1000003, 42)])
def test_hash_bit_exact(d, w, seed):
    rng = np.random.default_rng(d * 7 + seed % 97)
    idx = np.concatenate([np.array([0, 1, 2**31 - 1, 2**31, 2**32 - 1], dtype=np.uint64),
                          rng.integers(0, 2**32, size=100_000, dtype=np.uint64)]).astype(np.uint32)
    ti = torch.from_numpy(idx.view(np.int32)).to(DEV)
    b = torch.empty((d, idx.size), dtype=torch.int32, device=DEV)
    s = torch.empty((d, idx.size), dtype=torch.int8, device=DEV)
    s2.s2_hash(ti, d, w, seed, b, s)
    rb, rs = oracle.hash(idx, d, w, seed)
    np.testing.assert_array_equal(u32(b), rb)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


# ------------------------------------------------------------------ whole path

PIPELINE_CASES = [
    # name, kwargs for workloads.custom
    ("tiny", None),
    ("f32_vec_ragged", dict(W=3, n=10_000, d=5, w=1000, density=0.1, tag=101)),
    ("f32_scalar_rows", dict(W=3, n=1001, d=3, w=64, density=0.3, tag=102)),      # n*4 % 16 != 0
    ("f32_one_worker_tail", dict(W=1, n=1001, d=3, w=64, density=0.3, tag=103)),  # vector path + tail
    ("bf16_vec", dict(W=4, n=8192, d=5, w=512, density=0.05, dtype="bf16", tag=104)),
    ("bf16_scalar_rows", dict(W=2, n=7777, d=3, w=300, density=0.2, dtype="bf16", tag=105)),
    ("bf16_one_worker_tail", dict(W=1, n=1003, d=5, w=128, density=0.3, dtype="bf16", tag=115)),
    ("f32_bulk_tail", dict(W=3, n=2048 * 3 + 4 * 7, d=3, w=512, density=0.2, tag=116)),  # 2 KB tasks + tail
    ("d1", dict(W=2, n=5000, d=1, w=4096, density=0.02, tag=106)),
    ("d2_even", dict(W=2, n=5000, d=2, w=777, density=0.05, tag=107)),
    ("d4_even", dict(W=5, n=6000, d=4, w=333, density=0.05, tag=108)),
    ("d7_generic", dict(W=3, n=9000, d=7, w=2048, density=0.03, tag=109)),
    ("d16_generic", dict(W=2, n=3000, d=16, w=100, density=0.05, tag=110)),
    ("w1_all_collide", dict(W=3, n=2000, d=3, w=1, density=0.01, tag=111)),
    ("dense_all_nonzero", dict(W=2, n=4096, d=3, w=8192, density=1.0, tag=112)),
    ("many_workers", dict(W=13, n=4100, d=5, w=700, density=0.02, tag=113)),
    ("sparse_large", dict(W=4, n=1 << 20, d=3, w=1 << 12, density=0.002, tag=114)),
]


@pytest.mark.parametrize("name,kw", PIPELINE_CASES, ids=[c[0] for c in PIPELINE_CASES])
def test_pipeline_parity(name, kw):
    wl = workloads.tiny() if kw is None else workloads.custom(**kw)
    got = gpu_pipeline(_grad(wl), wl.d, wl.w, wl.seed, compact=True)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [3, 5, 6])
def test_pipeline_exact_arithmetic(dtype, d):
    # integer values: every fp32 partial sum is exact, so the atomic order
    # cannot matter and sketches and decoded values must match bit for bit.
    wl = workloads.custom(W=6, n=20_000, d=d, w=512, density=0.05, values="int", int_max=1024, dtype=dtype,
                          tag=200 + d)
    got = gpu_pipeline(_grad(wl), wl.d, wl.w, wl.seed, compact=True)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed, exact=True)


@pytest.mark.parametrize("scale", [0.125, -3.7])
def test_pipeline_scale(scale):
    wl = workloads.custom(W=4, n=12_345, d=5, w=999, density=0.05, tag=301)
    got = gpu_pipeline(_grad(wl), wl.d, wl.w, wl.seed, scale=scale, compact=True)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed, scale=scale)


def test_empty_gradient():
    for W in (0, 2):
        n = 0
        grad = torch.empty((W, n), dtype=torch.float32, device=DEV)
        bitmaps, sketches = s2.alloc_encode_outputs(W, n, 3, 16, DEV)
        sketches.fill_(7.0)
        s2.s2_encode_batched(grad, 3, 16, 0, bitmaps, sketches)
        bitmap = torch.empty(0, dtype=torch.int32, device=DEV)
        sketch = torch.full((3, 16), 5.0, device=DEV)
        s2.s2_reduce(bitmaps, sketches, n, 3, 16, bitmap, sketch)
        torch.cuda.synchronize()
        assert (sketches == 0).all() and (sketch == 0).all()


def test_all_zero_gradient_and_signed_zeros():
    n = 5000
    g = np.zeros((2, n), dtype=np.float32)
    g[0, 100:200] = np.float32(-0.0)
    g[1, 7] = np.float32(1e-45)  # smallest subnormal: nonzero
    g[1, 4999] = np.float32(-2.0)
    got = gpu_pipeline(torch.from_numpy(g).to(DEV), 3, 64, 0, compact=True)
    ref = check_pipeline(g, "f32", got, 3, 64, 0)
    assert ref["bitmap"].sum() > 0
    assert unpack(got["bitmap"], n).sum() == 2


def test_single_worker_encode_matches_batched_row():
    wl = workloads.custom(W=3, n=4096 + 77, d=5, w=321, density=0.1, tag=401)
    g = _grad(wl)
    bitmaps, sketches = s2.alloc_encode_outputs(3, wl.n, 5, 321, DEV)
    s2.s2_encode_batched(g, 5, 321, 0, bitmaps, sketches)
    bm1 = torch.empty(s2.nwords(wl.n), dtype=torch.int32, device=DEV)
    sk1 = torch.empty((5, 321), dtype=torch.float32, device=DEV)
    s2.s2_encode(g[1].clone(), 5, 321, 0, bm1, sk1)  # a fresh, 16-byte aligned row
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u32(bm1), u32(bitmaps[1]))
    ref_bm, ref_S, ref_A = oracle.encode(wl.dense()[1], 5, 321, 0)
    np.testing.assert_array_equal(u32(bm1), ref_bm)
    assert_sketch_close(sk1.cpu().numpy(), ref_S, ref_A)


# ------------------------------------------------------------------ reduce alone

@pytest.mark.parametrize("W,n,d,w", [(1, 1000, 3, 64), (3, 4096, 5, 1000), (8, 4097, 3, 257), (13, 31, 2, 3),
                                     (8, 128 * 1000, 5, 1 << 14)])
def test_reduce_parity(W, n, d, w):
    S = workloads.random_sketches(W, d, w, tag=500 + W)
    B = workloads.random_bitmaps(W, n, 0.05, tag=600 + W)
    tb = torch.from_numpy(B.view(np.int32)).to(DEV)
    ts = torch.from_numpy(S).to(DEV)
    bo = torch.empty(s2.nwords(n), dtype=torch.int32, device=DEV)
    so = torch.empty((d, w), dtype=torch.float32, device=DEV)
    s2.s2_reduce(tb, ts, n, d, w, bo, so)
    torch.cuda.synchronize()
    rb, rS, _ = oracle.reduce(B, S.astype(np.float64), None)
    np.testing.assert_array_equal(u32(bo), rb)
    assert_sketch_close(so.cpu().numpy(), rS, np.abs(S.astype(np.float64)).sum(axis=0), what="reduced sketch")
    # the sum order is fixed (k = 0..W-1): bit-identical to a sequential fp32 sum, run to run
    seq = np.zeros((d, w), dtype=np.float32)
    for k in range(W):
        seq = seq + S[k]
    np.testing.assert_array_equal(so.cpu().numpy(), seq)
    so2 = torch.empty_like(so)
    s2.s2_reduce(tb, ts, n, d, w, bo, so2)
    torch.cuda.synchronize()
    assert torch.equal(so, so2)


def test_reduce_integer_bit_exact():
    S = workloads.random_sketches(8, 3, 4096, tag=700, values="int")
    B = workloads.random_bitmaps(8, 100_000, 0.01, tag=701)
    bo = torch.empty(s2.nwords(100_000), dtype=torch.int32, device=DEV)
    so = torch.empty((3, 4096), dtype=torch.float32, device=DEV)
    s2.s2_reduce(torch.from_numpy(B.view(np.int32)).to(DEV), torch.from_numpy(S).to(DEV), 100_000, 3, 4096, bo, so)
    torch.cuda.synchronize()
    _, rS, _ = oracle.reduce(B, S.astype(np.float64), None)
    np.testing.assert_array_equal(so.cpu().numpy().astype(np.float64), rS)


# ------------------------------------------------------------------ decode alone

@pytest.mark.parametrize("d", [1, 2, 3, 4, 5, 7, 16])
@pytest.mark.parametrize("scale", [1.0, 0.125, -3.7])
def test_decode_parity_on_planted_sketches(d, scale):
    # Decode alone on a generated float32 sketch: the median only selects (odd
    # d) or averages two fp32 values (even d), so the result is bit-exact
    # except for even d with a scale other than 1 (two roundings).
    n, w, seed = 100_003, 4099, 17
    S = workloads.random_sketches(1, d, w, tag=800 + d)[0]
    B = workloads.random_bitmaps(1, n, 0.2, tag=801)[0]
    tb = torch.from_numpy(B.view(np.int32)).to(DEV)
    ts = torch.from_numpy(S).to(DEV)
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    s2.s2_decode_dense(tb, ts, n, d, w, seed, out, scale=scale)
    ws = torch.empty(s2.s2_decode_workspace_size(n), dtype=torch.uint8, device=DEV)
    idx = torch.empty(n, dtype=torch.int32, device=DEV)
    val = torch.empty(n, dtype=torch.float32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int64, device=DEV)
    s2.s2_decode_compact(tb, ts, n, d, w, seed, idx, val, cnt, ws, scale=scale)
    torch.cuda.synchronize()
    scale32 = float(np.float32(scale))  # the C ABI takes the scale as a float32
    want, _ = oracle.decode_dense(B, S.astype(np.float64), n, seed, scale32)
    got = out.cpu().numpy()
    if d % 2 == 1 or scale == 1.0:
        np.testing.assert_array_equal(got, want)
    else:
        np.testing.assert_allclose(got, want, rtol=2 ** -22, atol=0)
    c, ridx, rval, _ = oracle.decode_compact(B, S.astype(np.float64), n, seed, scale32)
    assert int(cnt.item()) == c
    np.testing.assert_array_equal(u32(idx[:c]), ridx)
    np.testing.assert_array_equal(val[:c].cpu().numpy(), got[ridx])


def test_decode_ignores_bits_past_n():
    # tail bits beyond n in the last word must not produce output
    n, d, w = 1000, 3, 128
    B = np.full(s2.nwords(n), 0xFFFFFFFF, dtype=np.uint32)
    S = workloads.random_sketches(1, d, w, tag=900)[0]
    out = torch.full((1024,), 9.0, dtype=torch.float32, device=DEV)
    s2.s2_decode_dense(torch.from_numpy(B.view(np.int32)).to(DEV), torch.from_numpy(S).to(DEV), n, d, w, 0, out[:n])
    ws = torch.empty(s2.s2_decode_workspace_size(n), dtype=torch.uint8, device=DEV)
    idx = torch.empty(1024, dtype=torch.int32, device=DEV)
    val = torch.empty(1024, dtype=torch.float32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int64, device=DEV)
    s2.s2_decode_compact(torch.from_numpy(B.view(np.int32)).to(DEV), torch.from_numpy(S).to(DEV), n, d, w, 0,
                         idx, val, cnt, ws)
    torch.cuda.synchronize()
    assert (out[n:] == 9.0).all()
    assert int(cnt.item()) == n


def test_compact_capacity_truncates_but_counts_all():
    n, d, w = 50_000, 5, 1024
    S = workloads.random_sketches(1, d, w, tag=1000)[0]
    B = workloads.random_bitmaps(1, n, 0.1, tag=1001)[0]
    tb = torch.from_numpy(B.view(np.int32)).to(DEV)
    ts = torch.from_numpy(S).to(DEV)
    cap = 1234
    idx = torch.full((cap + 16,), -7, dtype=torch.int32, device=DEV)
    val = torch.full((cap + 16,), -7.0, dtype=torch.float32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int64, device=DEV)
    ws = torch.empty(s2.s2_decode_workspace_size(n), dtype=torch.uint8, device=DEV)
    s2.s2_decode_compact(tb, ts, n, d, w, 3, idx[:cap], val[:cap], cnt, ws)
    torch.cuda.synchronize()
    c, ridx, rval, _ = oracle.decode_compact(B, S.astype(np.float64), n, 3, 1.0)
    assert int(cnt.item()) == c > cap
    np.testing.assert_array_equal(u32(idx[:cap]), ridx[:cap])
    np.testing.assert_array_equal(val[:cap].cpu().numpy(), rval[:cap])
    assert (idx[cap:] == -7).all() and (val[cap:] == -7.0).all()


# ------------------------------------------------------------------ host-buffer pipeline

def test_pipeline_dense_host_matches_oracle():
    wl = workloads.custom(W=4, n=50_000, d=5, w=2048, density=0.05, tag=1100)
    G = wl.dense()
    hg = torch.from_numpy(G).pin_memory()
    ho = torch.empty(wl.n, dtype=torch.float32).pin_memory()
    ws = torch.empty(s2.s2_pipeline_workspace_size(torch.float32, wl.W, wl.n, wl.d, wl.w), dtype=torch.uint8,
                     device=DEV)
    s2.s2_pipeline_dense_host(hg, wl.d, wl.w, wl.seed, ho, ws)
    torch.cuda.synchronize()
    ref = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    assert_decoded_close(ho.numpy(), ref["out"], ref["amax"])


@pytest.mark.parametrize("pin_in,pin_out", [(False, False), (True, False), (False, True)])
def test_pipeline_dense_host_staged_and_in_place(pin_in, pin_out):
    # pinned buffers are read / written in place by the kernels, pageable
    # ones are staged with copies: the results must be the same
    wl = workloads.custom(W=3, n=40_000, d=3, w=1024, density=0.05, dtype="bf16", tag=1101)
    G = wl.dense()
    hg = torch.from_numpy(G.view(np.int16)).view(torch.bfloat16)
    hg = hg.pin_memory() if pin_in else hg.clone()
    ho = torch.full((wl.n,), 3.0, dtype=torch.float32)
    ho = ho.pin_memory() if pin_out else ho
    ws = torch.empty(s2.s2_pipeline_workspace_size(torch.bfloat16, wl.W, wl.n, wl.d, wl.w), dtype=torch.uint8,
                     device=DEV)
    s2.s2_pipeline_dense_host(hg, wl.d, wl.w, wl.seed, ho, ws)
    torch.cuda.synchronize()
    ref = oracle.pipeline(G, wl.d, wl.w, wl.seed, dtype="bf16")
    assert_decoded_close(ho.numpy(), ref["out"], ref["amax"])


def test_pipeline_dense_host_unaligned_pinned_input_is_staged():
    wl = workloads.custom(W=2, n=10_000, d=3, w=512, density=0.05, tag=1102)
    G = wl.dense()
    buf = torch.zeros(G.size + 1, dtype=torch.float32).pin_memory()
    buf[1:] = torch.from_numpy(G.reshape(-1))
    hg = buf[1:].view(wl.W, wl.n)  # 4 bytes past a pinned allocation: not 16-byte aligned
    ho = torch.empty(wl.n, dtype=torch.float32).pin_memory()
    ws = torch.empty(s2.s2_pipeline_workspace_size(torch.float32, wl.W, wl.n, wl.d, wl.w), dtype=torch.uint8,
                     device=DEV)
    s2.s2_pipeline_dense_host(hg, wl.d, wl.w, wl.seed, ho, ws)
    torch.cuda.synchronize()
    ref = oracle.pipeline(G, wl.d, wl.w, wl.seed)
    assert_decoded_close(ho.numpy(), ref["out"], ref["amax"])


def test_non_default_stream():
    wl = workloads.custom(W=3, n=30_000, d=3, w=1000, density=0.05, tag=1200)
    g = _grad(wl)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        got = gpu_pipeline(g, wl.d, wl.w, wl.seed, compact=True, stream=st)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)


# ------------------------------------------------------------------ argument errors on real device memory

def test_alignment_and_overlap_errors():
    g = torch.zeros((2, 1024), dtype=torch.float32, device=DEV)
    bm = torch.empty((2, 32), dtype=torch.int32, device=DEV)
    sk = torch.empty((2, 3, 64), dtype=torch.float32, device=DEV)
    big = torch.zeros(4096, dtype=torch.float32, device=DEV)
    with pytest.raises(s2.S2Error) as e:
        s2.s2_encode_batched(big[1:2049].view(2, 1024), 3, 64, 0, bm, sk)  # base 4 bytes past alignment
    assert e.value.status == 2  # alignment
    with pytest.raises(s2.S2Error) as e:
        s2.s2_encode_batched(g, 3, 64, 0, bm, g.view(-1)[:384].view(2, 3, 64))
    assert e.value.status == 1  # output overlaps input
    with pytest.raises(s2.S2Error) as e:
        s2.s2_encode_batched(g, 0, 64, 0, bm, sk)
    assert e.value.status == 1  # d = 0
