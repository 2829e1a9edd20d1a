"""Host-side logic of bench.py, on CPU: byte accounting, launch counting, the
reference arm's JSON line, and the max-over-ranks / sum-of-units combination
used when N replicas run under torchrun (two gloo ranks here)."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_algorithmic_bytes_embedding():
    wl = workloads.Workload("e", 8, 33_278 * 512, 5, 1 << 20, 0, "f32", [], [])
    by = bench.algorithmic_bytes(wl, nnz_union=4_466_688)
    nw = (wl.n + 31) // 32
    assert by["encode"] == 8 * wl.n * 4 + 8 * nw * 4 + 8 * 5 * (1 << 20) * 4
    assert by["reduce"] == 9 * (5 * (1 << 20) * 4 + nw * 4)
    assert by["decode"] == nw * 4 + 5 * (1 << 20) * 4 + 4 * wl.n  # sketch read capped at one pass
    assert abs(by["total"] / 1e6 - 1029.2) < 0.1


def test_l2_sector_ops_embedding():
    wl = workloads.embedding()
    ops = bench.l2_sector_ops(wl, wl.union_nnz())
    nw = (wl.n + 31) // 32
    assert ops["encode"] == 8 * wl.n * 4 // 32 + 8 * (nw * 4 // 32) + 8 * (5 * (1 << 20) * 4 // 32) + 8 * 1_024_000 * 5
    assert ops["decode"] == nw * 4 // 32 + wl.union_nnz() * 5 + wl.n * 4 // 32
    assert ops["total"] == ops["encode"] + ops["reduce"] + ops["decode"]


def test_select_workers_keeps_a_prefix():
    wl = workloads.custom(W=4, n=1000, d=3, w=64, density=0.1)
    first = [a.copy() for a in wl.idx[:2]]
    wl2 = bench.select_workers(wl, 2)
    assert wl2.W == 2 and len(wl2.idx) == 2 and all((a == b).all() for a, b in zip(wl2.idx, first))
    assert bench.select_workers(workloads.tiny(), None).W == 2


def test_encode_launch_groups():
    wl = workloads.Workload("e", 8, 1000, 5, 1 << 20, 0, "f32", [], [])  # 20 MiB sketch per worker
    assert bench.encode_launches(wl, 126 << 20) == 2 * 3  # three workers per group
    wl = workloads.Workload("e", 4, 1000, 5, 1 << 22, 0, "f32", [], [])  # 80 MiB
    assert bench.encode_launches(wl, 126 << 20) == 2 * 4  # one worker per group
    wl = workloads.Workload("e", 8, 1000, 3, 1 << 19, 0, "f32", [], [])  # 6 MiB
    assert bench.encode_launches(wl, 126 << 20) == 2


def test_encode_launches_follow_the_path_choice():
    L2 = 135_528_448
    # a 3 KiB sketch with 4096 positions per bucket and more: the shared-memory
    # path, a zero fill and one encode
    wl = workloads.Workload("s", 8, 1 << 22, 3, 256, 0, "f32", [], [])
    assert bench.encode_launches(wl, L2) == 2
    # few positions per bucket: the L2 path (one group)
    wl = workloads.Workload("t", 2, 4096, 3, 256, 0, "f32", [], [])
    assert bench.encode_launches(wl, L2) == 2
    # a 160 MiB sketch: one worker at a time in two slice passes
    wl = workloads.Workload("b", 8, 1 << 27, 5, 1 << 23, 0, "f32", [], [])
    assert bench.encode_launches(wl, L2) == 2 * 8 * 2


def test_dense_decode_launches():
    L2 = 135_528_448
    assert bench.dense_decode_launches(33_278 * 512, L2) == 1
    assert bench.dense_decode_launches(267_735 * 1024, L2) == 2  # 1.1 GB of output: zeros first
    # an 84 MB summed sketch of 5 rows: a zero launch, the one-launch form (which
    # works only if most tasks are set) and passes over rows {0,1}, {2,3,4}
    assert bench.dense_decode_launches(267_735 * 1024, L2, 5, 1 << 22) == 4
    assert bench.dense_decode_launches(1 << 27, L2, 5, 1 << 23) == 6  # 168 MB: one 33.5 MB row per pass
    assert bench.dense_decode_launches(1 << 27, L2, 3, 5_000_001) == 4  # 60 MB: one launch or {0,1}, {2}
    assert bench.dense_decode_launches(1 << 27, L2, 3, 1 << 22) == 2  # 50 MB: below 2/5 of L2
    assert bench.dense_decode_launches(1 << 27, L2, 4, 1 << 23) == 2  # even d: no row passes
    assert bench.dense_decode_launches(33_278 * 512, L2, 5, 1 << 20) == 1  # 21 MB sketch: one launch


def test_compact_decode_accounting():
    wl = workloads.Workload("e", 8, 33_278 * 512, 5, 1 << 20, 0, "f32", [], [])
    dense = bench.algorithmic_bytes(wl, 4_466_688)
    comp = bench.algorithmic_bytes(wl, 4_466_688, compact=True)
    assert dense["decode"] - comp["decode"] == 4 * wl.n - 8 * 4_466_688
    assert dense["encode"] == comp["encode"] and dense["reduce"] == comp["reduce"]


def test_reference_arm_line(capsys):
    assert bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "Gelem/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.out = "1965, 2070, 900.1, Not Active, Not Active, Not Active, Active\n1980, 2070, 950, Not Active, Not Active, Not Active, Not Active\n"
    s = c.summary()
    assert s["sm_mhz"] == 1972.5 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        el, units = bench.combine_over_ranks(1.0 + rank, 100.0 * (rank + 1), world)
        q.put((rank, el, units))
    finally:
        dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_combine_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for _, el, units in got:
        assert el == 2.0 and units == 300.0  # max of times, sum of units


def test_physical_gpu_index(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.physical_gpu_index(1) == 5
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.physical_gpu_index(2) == 2
