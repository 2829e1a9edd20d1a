"""GPU parity at the full sizes of the benchmark workloads.

The embedding (33,278 x 512, W=8, d=5, w=2^20), top-k (n=25,557,032, W=8,
d=3, w=2^19) and large-LM (267,735 x 1024, W=4, d=5, w=2^22) workloads run
through the same C-ABI calls, in the same launch configuration, as the
benchmark; the oracle computes every output in full and every element is
compared. The sweep's (dtype, density, d) combinations are checked at
n = 2^20, plus one maximum-length point at n = 2^28 and one point whose
sketch is larger than L2 (n = 2^27, 10 %, d = 5) at the sweep's own shape.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    from tests._parity import check_pipeline, gpu_pipeline


@pytest.mark.parametrize("name", ["tiny", "embedding", "topk", "large_lm"])
def test_full_size_workload(name):
    wl = workloads.by_name(name)
    grad = wl.dense_torch("cuda")
    got = gpu_pipeline(grad, wl.d, wl.w, wl.seed, compact=True)
    del grad
    torch.cuda.empty_cache()
    ref = check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)
    assert int(ref["bitmap"].view(np.uint32).astype(np.uint64).sum()) > 0


@pytest.mark.parametrize("pt", [p for p in workloads.sweep_grid() if p["n"] == 1 << 20],
                         ids=lambda p: f"{p['dtype']}-rho{p['density']}-d{p['d']}")
def test_sweep_point(pt):
    wl = workloads.sweep_point(**pt)
    got = gpu_pipeline(wl.dense_torch("cuda"), wl.d, wl.w, wl.seed, compact=True)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)


def test_sweep_maximum_length():
    wl = workloads.sweep_point(n=1 << 28, dtype="bf16", density=0.001, d=5)
    grad = wl.dense_torch("cuda")
    got = gpu_pipeline(grad, wl.d, wl.w, wl.seed)
    del grad
    torch.cuda.empty_cache()
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)


def test_sweep_point_with_a_sketch_larger_than_l2():
    # 8 workers of 2^27 fp32 positions at 10 % density, d = 5: w = 2^23, so
    # each worker's sketch (167.8 MB) is built in two passes over bucket
    # slices, and the summed sketch is decoded in row passes (one 33.5 MB row
    # each)
    wl = workloads.sweep_point(n=1 << 27, dtype="f32", density=0.1, d=5)
    assert 4 * wl.d * wl.w > 128 << 20
    grad = wl.dense_torch("cuda")
    got = gpu_pipeline(grad, wl.d, wl.w, wl.seed)
    del grad
    torch.cuda.empty_cache()
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)
