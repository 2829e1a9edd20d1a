"""The allocation-free compacted decode, called through the C ABI.

Some callers cannot allocate device memory for a workspace: a framework that
owns all device memory through its own pool, a latency-critical path where a
cudaMalloc may synchronise the device, or code that keeps no state between
calls. For them s2_decode_compact_noalloc uses a fixed scratch array inside
the library instead. Its results must be those of s2_decode_compact with a
caller workspace. Two calls in a row, the second on a smaller input with
fewer tiles, check that what the first call leaves in the shared scratch does
not leak into the second.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

REL = 1e-5  # the decode tolerance of the other GPU tests, relative to the sketch magnitude


def _decode_both(n, d, w, seed, density, tag, scale):
    import sketch_compressed_sparse_gb300 as s2

    dev = "cuda"
    S = workloads.random_sketches(1, d, w, tag=tag)[0]
    B = workloads.random_bitmaps(1, n, density, tag=tag + 1)[0]
    bitmap = torch.from_numpy(B.view(np.int32)).to(dev)
    sketch = torch.from_numpy(S).to(dev)

    ws = torch.empty(s2.s2_decode_workspace_size(n), dtype=torch.uint8, device=dev)
    idx_ref = torch.full((n,), -1, dtype=torch.int32, device=dev)
    val_ref = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    cnt_ref = torch.full((1,), -1, dtype=torch.int64, device=dev)
    s2.s2_decode_compact(bitmap, sketch, n, d, w, seed, idx_ref, val_ref, cnt_ref, ws, scale=scale)

    idx = torch.full((n,), -2, dtype=torch.int32, device=dev)
    val = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    cnt = torch.full((1,), -2, dtype=torch.int64, device=dev)
    s2.s2_decode_compact_noalloc(bitmap, sketch, n, d, w, seed, idx, val, cnt, scale=scale)
    torch.cuda.synchronize()

    c_ref, c = int(cnt_ref.item()), int(cnt.item())
    assert c == c_ref == int(np.unpackbits(B.view(np.uint8), bitorder="little")[:n].sum())
    np.testing.assert_array_equal(idx[:c].cpu().numpy(), idx_ref[:c].cpu().numpy())
    tol = REL * float(np.abs(S).max()) * abs(scale)
    np.testing.assert_allclose(val[:c].cpu().numpy(), val_ref[:c].cpu().numpy(), rtol=0, atol=tol)
    assert (idx[c:] == -2).all()  # nothing written past the count
    return c


def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    # first call: ~1M positions (123 tiles of 8192 positions); second: fewer tiles
    c1 = _decode_both(n=1_000_003, d=5, w=4099, seed=3, density=0.1, tag=9100, scale=1.0)
    c2 = _decode_both(n=70_001, d=3, w=1024, seed=11, density=0.3, tag=9200, scale=0.5)
    assert c1 > 0 and c2 > 0
