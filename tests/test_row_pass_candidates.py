"""The candidate scheme of the row-pass dense decode, checked on the host.

The median query of Algorithm 1 ("S2 Reducer", Section 3.1 "Decompressing
Sparse Gradient") needs all d row estimates of a position. The row-pass
decode visits the rows in groups and carries, between passes, only the
values that can still be the median: after r of d rows, at most
kept_after(d, r) values (d = 3: 1, 2; d = 5: 1, 2, 3, 2). This test folds
the rows one at a time in that scheme, for every split of the rows into
passes, and compares with numpy's median by brute force over random values
with many ties. It pins the scheme, not the kernel (the GPU tests compare
the kernel with the oracle bit for bit).
"""
import itertools

import numpy as np
import pytest


def kept_after(d, r):
    if d == 3:
        return [0, 1, 2, 1][r]
    return [0, 1, 2, 3, 2, 1][r]


def fold(cands, r, e, d):
    """The candidates after row r (rows counted from 0) given those after r rows."""
    vals = sorted(cands + [e])
    n_seen = r + 1
    if n_seen == d:  # the median of the d values
        assert len(vals) == kept_after(d, r) + 1
        return [vals[len(vals) // 2]]
    keep = kept_after(d, n_seen)
    if len(vals) == keep:
        return vals
    # drop equally from both ends: the values that can no longer be the middle one
    lo = (len(vals) - keep) // 2
    return vals[lo:lo + keep]


def median_by_passes(e, groups, d):
    cands = []
    r = 0
    for g in groups:
        for _ in range(g):
            cands = fold(cands, r, float(e[r]), d)
            assert len(cands) <= 3
            r += 1
        assert len(cands) == (1 if r == d else kept_after(d, r))
    return cands[0]


def splits(d):
    for k in range(1, d + 1):
        for cut in itertools.combinations(range(1, d), k - 1):
            b = (0,) + cut + (d,)
            yield [b[i + 1] - b[i] for i in range(k)]


@pytest.mark.parametrize("d", [3, 5])
def test_carried_candidates_give_the_median_for_every_split(d):
    rng = np.random.default_rng(5)
    for e in itertools.chain(itertools.product(range(3), repeat=d),  # every pattern of ties
                             rng.normal(size=(2000, d))):
        want = float(np.median(np.asarray(e, dtype=np.float64)))
        for groups in splits(d):
            assert median_by_passes(e, groups, d) == want, (e, groups)


def test_candidate_counts_match_the_kernel_plan():
    # d = 5 in groups of 3 rows runs rows {0, 1} then {2, 3, 4}: two values
    # carried between the passes; {0, 1, 2} first would carry three
    assert kept_after(5, 2) == 2 and kept_after(5, 3) == 3 and kept_after(5, 1) == 1
    assert kept_after(3, 1) == 1 and kept_after(3, 2) == 2
