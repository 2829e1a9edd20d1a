"""GPU parity of the dense decode taken in passes over groups of rows
(s2_decode_dense_ws), for summed sketches larger than 2/5 of L2.

The median query of Algorithm 1 ("S2 Reducer", Section 3.1 "Decompressing
Sparse Gradient") only selects among the d row values of a position (odd d),
so on a planted float32 sketch the result must match the oracle bit for bit
whatever the order in which the rows are visited. The cases cover every plan
on a GB300 (L2 of 135.5 MB, 2/5 of it per pass; the smallest group of rows
first): for d = 5, groups of 3 rows (w = 2^22: 16.8 MB rows; rows {0, 1},
then {2, 3, 4} from two carried candidates), 1 row per pass (w = 2^23), 4
rows per pass (w = 3 * 2^20 + 7) and 2 rows per pass (w = 5,000,003); for
d = 3, 1 + 2 rows (w = 5,000,001) and one row per pass (w = 2^23); and the
one-launch form over all rows, which a sketch of at most 96 MB takes when at
least half of the 512-position tasks hold a set position; ragged lengths and
a scale other than one.
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


def _decode_ws(B, S, n, d, w, seed, scale):
    tb = torch.from_numpy(B.view(np.int32)).to(DEV)
    ts = torch.from_numpy(S).to(DEV)
    out = torch.full((n,), float("nan"), dtype=torch.float32, device=DEV)
    ref = torch.full((n,), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.full((max(s2.s2_decode_dense_workspace_size(n, d, w), 1),), 0xAB, dtype=torch.uint8, device=DEV)
    s2.s2_decode_dense_ws(tb, ts, n, d, w, seed, out, ws, scale=scale)
    s2.s2_decode_dense(tb, ts, n, d, w, seed, ref, scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ref.cpu().numpy()


@pytest.mark.parametrize("d,w,n,density,scale", [
    (5, 1 << 22, 3_000_017, 0.2, 1.0),           # every task set: one launch over all rows
    (5, 1 << 22, 3_000_017, 0.0005, 1.0),        # a quarter of the tasks: rows {0,1}, {2,3,4}
    (5, 1 << 23, 1_000_003, 0.3, 0.5),           # 168 MB: one row per pass
    (5, 3 * (1 << 20) + 7, 2_000_000, 0.0005, 1.0),  # rows {0}, {1,2,3,4}
    (5, 5_000_003, 1_500_001, 0.1, 1.0),         # 100 MB: rows {0}, {1,2}, {3,4}
    (3, 5_000_001, 1_048_579, 0.5, 2.0),         # one launch
    (3, 5_000_001, 1_048_579, 0.001, 2.0),       # rows {0}, {1,2}
    (3, 1 << 23, 777_777, 1.0, 1.0),             # every position set; 100 MB: one row per pass
])
def test_row_pass_decode_is_bit_exact(d, w, n, density, scale):
    seed = 21
    S = workloads.random_sketches(1, d, w, tag=6000 + d + w % 97)[0]
    B = workloads.random_bitmaps(1, n, density, tag=6001 + n % 89)[0]
    got, plain = _decode_ws(B, S, n, d, w, seed, scale)
    scale32 = float(np.float32(scale))
    want, _ = oracle.decode_dense(B, S.astype(np.float64), n, seed, scale32)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    np.testing.assert_array_equal(got.view(np.uint32), plain.view(np.uint32))


def test_row_pass_decode_with_clustered_rows_and_empty_tasks():
    # whole 1024-position rows set, most 512-position tasks empty (the
    # large-LM pattern): empty tasks are written by the zero launch only,
    # partly set chunks at the edges of a row by the last pass
    d, w, n, seed = 5, 1 << 22, 1024 * 3000 + 5, 4
    rng = np.random.default_rng(31)
    S = workloads.random_sketches(1, d, w, tag=6100)[0]
    mark = np.zeros(n, dtype=bool)
    for r in rng.choice(3000, size=60, replace=False):
        mark[r * 1024 + 3:(r + 1) * 1024 - 2] = True
    mark[n - 3:] = True
    B = np.zeros((n + 31) // 32, dtype=np.uint32)
    pos = np.flatnonzero(mark)
    np.bitwise_or.at(B, pos >> 5, (np.uint32(1) << (pos & 31).astype(np.uint32)))
    got, plain = _decode_ws(B, S, n, d, w, seed, 1.0)
    want, _ = oracle.decode_dense(B, S.astype(np.float64), n, seed, 1.0)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    assert (got.view(np.uint32)[~mark] == 0).all()


def test_workspace_size_and_small_workspace_rejected():
    n, d, w = 100_000, 5, 1 << 22
    need = s2.s2_decode_dense_workspace_size(n, d, w)
    assert need >= 2 * 4 * n and s2.s2_decode_dense_workspace_size(n, 3, w) >= 4 * n
    assert s2.s2_decode_dense_workspace_size(n, 4, w) == 0
    tb = torch.zeros((n + 31) // 32, dtype=torch.int32, device=DEV)
    ts = torch.zeros((d, w), dtype=torch.float32, device=DEV)
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    ws = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(s2.S2Error):
        s2.s2_decode_dense_ws(tb, ts, n, d, w, 0, out, ws)
