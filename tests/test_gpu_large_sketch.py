"""GPU parity for sketches larger than the L2 cache can hold while they are
built (more than 3/4 of L2): the encode then builds each worker's sketch in
several passes, each over one slice of the flattened buckets; and for dense
outputs larger than L2, which the decode writes in two launches. The results
must be those of the single-pass definition: bitmaps bit for bit, sketches
and decoded values within the stated tolerance, and bit for bit on
integer-valued gradients.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests._parity import check_pipeline, gpu_pipeline


def l2_bytes():
    return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 << 20))


def run(wl, exact=False):
    sk_bytes = 4 * wl.d * wl.w
    assert sk_bytes > 0.75 * l2_bytes(), "the case must take the multi-pass encode"
    got = gpu_pipeline(wl.dense_torch("cuda"), wl.d, wl.w, wl.seed)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed, exact=exact)


def test_two_passes_fp32():
    # 5 x 2^23 buckets = 160 MiB per worker
    run(workloads.custom(W=2, n=300_000, d=5, w=1 << 23, density=0.2, tag=701))


def test_ragged_slices_bf16_unaligned_rows():
    # one row of 2^26 + 7 buckets (256 MiB): three passes whose last slice is
    # shorter; odd n: scalar loads
    run(workloads.custom(W=1, n=100_003, d=1, w=(1 << 26) + 7, density=0.3, dtype="bf16", tag=702))


def test_multi_pass_exact_on_integers():
    run(workloads.custom(W=3, n=65_536, d=3, w=(1 << 24) + 1, density=0.1, values="int", int_max=256, tag=703),
        exact=True)


def test_dense_output_larger_than_l2_is_written_in_two_phases():
    # 4n bytes of output above the L2 size: tasks without a set position are
    # written (zeros) by a first launch, the others by a second one
    n = (l2_bytes() // 4) + 5_000_003
    wl = workloads.custom(W=2, n=n, d=3, w=1 << 16, density=0.001, tag=704)
    got = gpu_pipeline(wl.dense_torch("cuda"), wl.d, wl.w, wl.seed)
    check_pipeline(wl.dense(), wl.dtype, got, wl.d, wl.w, wl.seed)
