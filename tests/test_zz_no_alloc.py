"""The allocation-free compacted decode, called through the C ABI.

Some callers cannot allocate device memory for a workspace: a framework that
owns all device memory through its own pool and forbids side allocations, a
latency-critical path where a cudaMalloc may synchronise the device, or code
that keeps no state between calls. For them s2_decode_compact_noalloc keeps
its scratch in a fixed array inside the library instead.

Its results are checked against the oracle (Algorithm 1's decompression
phase, compacted) and against s2_decode_compact with a caller workspace. Both
GPU calls run the same kernels, so they must agree bit for bit; on a planted
float32 sketch with an odd number of rows the median only selects, so the
oracle's values match bit for bit as well. Two calls in a row, the second on
a smaller input with fewer tiles, check that what the first call leaves in
the shared scratch does not leak into the second; a call at the largest
length the scratch is sized for (2^30 positions) checks its layout at the
limit.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _decode_both(n, d, w, seed, density, tag, scale, slack=64):
    import sketch_compressed_sparse_gb300 as s2

    dev = "cuda"
    S = workloads.random_sketches(1, d, w, tag=tag)[0]
    B = workloads.random_bitmaps(1, n, density, tag=tag + 1)[0]
    scale32 = float(np.float32(scale))  # the C ABI takes the scale as a float32
    c_or, idx_or, val_or, _ = oracle.decode_compact(B, S.astype(np.float64), n, seed, scale32,
                                                    capacity=int(round(density * n)) + slack)
    cap = c_or + slack
    bitmap = torch.from_numpy(B.view(np.int32)).to(dev)
    sketch = torch.from_numpy(S).to(dev)

    ws = torch.empty(s2.s2_decode_workspace_size(n), dtype=torch.uint8, device=dev)
    idx_ref = torch.full((cap,), -1, dtype=torch.int32, device=dev)
    val_ref = torch.full((cap,), float("nan"), dtype=torch.float32, device=dev)
    cnt_ref = torch.full((1,), -1, dtype=torch.int64, device=dev)
    s2.s2_decode_compact(bitmap, sketch, n, d, w, seed, idx_ref, val_ref, cnt_ref, ws, scale=scale)

    idx = torch.full((cap,), -2, dtype=torch.int32, device=dev)
    val = torch.full((cap,), float("nan"), dtype=torch.float32, device=dev)
    cnt = torch.full((1,), -2, dtype=torch.int64, device=dev)
    s2.s2_decode_compact_noalloc(bitmap, sketch, n, d, w, seed, idx, val, cnt, scale=scale)
    torch.cuda.synchronize()

    c_ref, c = int(cnt_ref.item()), int(cnt.item())
    assert c == c_ref == c_or == int(round(density * n))
    np.testing.assert_array_equal(_u32(idx[:c]), idx_or)
    np.testing.assert_array_equal(val[:c].cpu().numpy().view(np.uint32), val_or.view(np.uint32))
    np.testing.assert_array_equal(_u32(idx[:c]), _u32(idx_ref[:c]))
    np.testing.assert_array_equal(_u32(val[:c]), _u32(val_ref[:c]))
    assert (idx[c:] == -2).all()  # nothing written past the count
    return c


def test_noalloc_decode_matches_oracle_and_workspace_decode_on_two_calls_in_a_row():
    # first call: ~1M positions (123 tiles of 8192 positions); second: fewer tiles
    c1 = _decode_both(n=1_000_003, d=5, w=4099, seed=3, density=0.1, tag=9100, scale=1.0)
    c2 = _decode_both(n=70_001, d=3, w=1024, seed=11, density=0.3, tag=9200, scale=0.5)
    assert c1 > 0 and c2 > 0


def test_noalloc_decode_at_its_largest_length():
    # 2^30 positions: 131,072 tiles, the most the library's scratch holds
    c = _decode_both(n=1 << 30, d=3, w=4096, seed=5, density=1e-5, tag=9300, scale=1.0)
    assert c > 0
