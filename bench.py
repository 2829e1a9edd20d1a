"""Benchmark of the S2 Reducer hot path: encode -> reduce -> decode on one GPU.

One step = s2_encode_batched over the W resident workers' gradients, s2_reduce
of their bitmaps and sketches, and s2_decode_dense of the aggregate: the whole
path over one batch of synthetic input, with the inputs already in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0). The default workload is the largest one, the
large-LM embedding table (267,735 x 1024 fp32, W=4, d=5, w=2^22); the line's
``per_config`` object carries the same measurements for the embedding
(33,278 x 512) and top-k (ResNet-50 size) workloads, timed in the same run.
``value`` is W*n gradient elements per second (Gelem/s) over the K timed
steps, whole job. L2 is flushed (a 512 MiB write) before every step, outside
the timed events. ``roofline`` is the dominant
kernel (encode) against the measured HBM copy bandwidth; ``path_roofline`` the
whole step. ``e2e`` times the same path from pinned host memory to host memory
through the C-ABI call s2_pipeline_dense_host. ``cpu_baseline`` times the CPU
oracle (test infrastructure, plain C) on the same workload on the host cores.

With ``--impl reference`` the oracle itself is the timed arm (rank 0 only).
For N > 1 (torchrun), every rank runs an independent replica of the workload
(weak scaling): the path has no exchange between GPUs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "S2 encode→reduce→decode Gelem/s and achieved HBM GB/s vs GB300 peak, 1 GPU"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- byte accounting

def bitmap_bytes(n: int, block: int = 0) -> int:
    """Bytes of one bitmap: one bit per position, or per block of `block` positions."""
    bits = n if not block else (n + block - 1) // block
    return 4 * ((bits + 31) // 32)


def algorithmic_bytes(wl: workloads.Workload, nnz_union: int, block: int = 0, compact: bool = False) -> dict:
    """Bytes each stage must move at minimum (each structure read/written once).

    encode: read grad, write W bitmaps and W sketches;
    reduce: read W bitmaps and W sketches, write one bitmap and one sketch;
    decode: read the bitmap, read at most the sketch (d gathers per set bit,
            counted up to one full read), write the dense output (compact:
            an index and a value per set position).
    """
    W, n, d, w = wl.W, wl.n, wl.d, wl.w
    E = wl.elem_bytes
    BM = bitmap_bytes(n, block)
    SK = 4 * d * w
    enc = W * n * E + W * BM + W * SK
    red = W * (SK + BM) + SK + BM
    dec = BM + min(SK, 4 * d * nnz_union) + (8 * nnz_union if compact else 4 * n)
    return {"encode": enc, "reduce": red, "decode": dec, "total": enc + red + dec}


def algorithmic_bytes_fused(wl: workloads.Workload, nnz_union: int) -> dict:
    """Fused single-sketch mode: read grad once, write the aggregate bitmap and
    sketch once; the decode as in the per-worker path."""
    by = algorithmic_bytes(wl, nnz_union)
    BM = 4 * ((wl.n + 31) // 32)
    SK = 4 * wl.d * wl.w
    fused = wl.W * wl.n * wl.elem_bytes + BM + SK
    return {"encode_reduce_fused": fused, "decode": by["decode"], "total": fused + by["decode"]}


def l2_sector_ops_fused(wl: workloads.Workload, nnz_union: int) -> dict:
    sec = lambda b: (b + 31) // 32
    ops = l2_sector_ops(wl, nnz_union)
    fused = sec(wl.W * wl.n * wl.elem_bytes) + sec(4 * ((wl.n + 31) // 32)) + sec(4 * wl.d * wl.w) + nnz_union * wl.d
    return {"encode_reduce_fused": fused, "decode": ops["decode"], "total": fused + ops["decode"]}


def l2_sector_ops(wl: workloads.Workload, nnz_union: int, block: int = 0, compact: bool = False) -> dict:
    """32-byte L2 sector operations each stage issues at minimum.

    Streams count one operation per 32-byte sector; every scattered 4-byte
    sketch reduction (encode) or gather (decode) is one operation of its own.
    encode: read grad, write bitmaps, zero-fill and then update (W nnz d
            reductions) the per-worker sketches;
    reduce: read W bitmaps and sketches, write one of each;
    decode: read the bitmap, d gathers per set position, write the output.
    """
    W, n, d, w = wl.W, wl.n, wl.d, wl.w
    sec = lambda b: (b + 31) // 32
    BM = bitmap_bytes(n, block)
    SK = 4 * d * w
    nnz = sum(wl.nnz_per_worker)
    enc = sec(W * n * wl.elem_bytes) + W * sec(BM) + W * sec(SK) + nnz * d
    red = W * (sec(SK) + sec(BM)) + sec(SK) + sec(BM)
    dec = sec(BM) + nnz_union * d + (sec(8 * nnz_union) if compact else sec(4 * n))
    return {"encode": enc, "reduce": red, "decode": dec, "total": enc + red + dec}


def measured_ceilings():
    """Scattered-operation ceilings measured by `bench.py --ceilings` on this GPU model."""
    p = os.path.join(ROOT, "profiles", "ceilings_gb300.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        return json.load(f)


def encode_launches(wl: workloads.Workload, l2_bytes: int, sms: int = 152) -> int:
    """Kernels one s2_encode_batched call launches: a zero fill and an encode per
    group of workers whose sketches fit in half of L2 together; per worker and
    slice when the sketch is built in passes (above 3/4 of L2); a zero fill and
    one shared-memory encode when the library takes that path."""
    sk = 4 * wl.d * wl.w
    esz = 4 if wl.dtype == "f32" else 2
    tasks = (wl.n + 511) // 512
    per_worker = max(1, min(-(-sms // max(wl.W, 1)), -(-tasks // 32)))
    if sk <= 192 * 1024 and wl.n >= 4096 * wl.w and per_worker * wl.d * wl.w * 16 <= wl.n * esz:
        return 2 if per_worker > 1 else 1
    cap = l2_bytes // 4 * 3
    if sk > cap:
        return 2 * wl.W * (-(-sk // cap))
    group = max(1, min(wl.W, (l2_bytes // 2) // sk)) if sk else wl.W
    return 2 * ((wl.W + group - 1) // group)


def dense_decode_launches(n: int, l2_bytes: int, d: int = 0, w: int = 0, block: int = 0) -> int:
    """Launches of one s2_decode_dense_ws call: a summed sketch larger than 2/5
    of L2 (d = 3 or 5, element bitmap) is decoded by a zero launch and one
    launch per group of rows that fits in 2/5 of L2; otherwise a dense output
    larger than L2 is written in two launches (zeros first), a smaller one in
    one."""
    budget = l2_bytes * 2 // 5
    if not block and d in (3, 5) and 4 * d * w > budget:
        rpp = 1 if 4 * w >= budget else budget // (4 * w)
        one_launch = 1 if 4 * d * w <= 96 << 20 else 0  # queued too, works when most tasks are set
        return 1 + one_launch + -(-d // rpp)
    return 2 if 4 * n > l2_bytes else 1


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


def kernel_source_sha() -> str:
    """Hash of the sources that define the encode stage (its kernels and their helpers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sketch_compressed_sparse_gb300", "csrc")
    for f in ("s2_device.cuh", "s2_internal.h", "s2_tasks.cuh", "s2_encode.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes of one step's encode stage (its zero-fill and encode launches)
    from a committed ncu summary, if it was taken on the current kernel sources
    (else None)."""
    p = os.path.join(ROOT, "profiles", "encode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    if j.get("source_sha") != kernel_source_sha():
        return None
    return j.get("per_workload", {}).get(workload)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def physical_gpu_index(local: int) -> int:
    """nvidia-smi index of CUDA device `local` (honours a numeric CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids) and ids[local].isdigit():
            return int(ids[local])
    return local


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def combine_over_ranks(elapsed_s: float, units: float, world: int, device=None):
    """(max elapsed over ranks, sum of units over ranks). Single process: identity."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist

    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- CPU oracle timing

def time_oracle(wl: workloads.Workload, G: np.ndarray, reps: int) -> dict:
    import oracle

    oracle.build()
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.pipeline(G, wl.d, wl.w, wl.seed, dtype=wl.dtype)
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts)
    return {"seconds": t, "reps": reps, "value": wl.W * wl.n / t / 1e9}


def time_oracle_threads(wl: workloads.Workload, G: np.ndarray) -> dict:
    """The oracle's steps as they stand, with the W workers' encodes on W
    host threads at once (each call runs in C outside the interpreter lock);
    reduce and decode on one thread."""
    import concurrent.futures as cf

    import oracle

    oracle.build()
    threads = max(1, min(wl.W, os.cpu_count() or 1))
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda k: oracle.encode(G[k], wl.d, wl.w, wl.seed, wl.dtype), range(wl.W)))
    bms = np.stack([p[0] for p in parts])
    S = np.stack([p[1] for p in parts])
    A = np.stack([p[2] for p in parts])
    bm, Ssum, Asum = oracle.reduce(bms, S, A)
    oracle.decode_dense(bm, Ssum, wl.n, wl.seed, 1.0, Asum)
    t = time.perf_counter() - t0
    return {"seconds": t, "threads": threads, "value": wl.W * wl.n / t / 1e9}


# ---------------------------------------------------------------- our arm

def run_ours(args, wl, world, rank, local, config_name=None):
    import torch

    import sketch_compressed_sparse_gb300 as s2

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20))
    W, n, d, w, seed = wl.W, wl.n, wl.d, wl.w, wl.seed
    nnz_u = wl.union_nnz()
    grad = wl.dense_torch(dev)
    blk = args.block
    nbits = (n + blk - 1) // blk if blk else n  # bits of one bitmap
    if args.mode == "fused":
        bitmaps = sketches = None
    else:
        bitmaps = torch.empty((W, s2.nwords(nbits)), dtype=torch.int32, device=dev)
        sketches = torch.empty((W, d, w), dtype=torch.float32, device=dev)

    bitmap = torch.empty(s2.nwords(nbits), dtype=torch.int32, device=dev)
    sketch = torch.empty((d, w), dtype=torch.float32, device=dev)
    compact = args.decode == "compact"
    if compact:
        if blk:
            raise SystemExit("--decode compact takes the element bitmap")
        cidx = torch.empty(max(nnz_u, 1), dtype=torch.int32, device=dev)
        cval = torch.empty(max(nnz_u, 1), dtype=torch.float32, device=dev)
        ccnt = torch.empty(1, dtype=torch.int64, device=dev)
        cws = torch.empty(max(s2.s2_decode_workspace_size(n), 1), dtype=torch.uint8, device=dev)
        out = None
    else:
        out = torch.empty(n, dtype=torch.float32, device=dev)
        dws = torch.empty(max(s2.s2_decode_dense_workspace_size(n, d, w), 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    fused = args.mode == "fused"

    def encode():
        if blk:
            s2.s2_encode_batched_blocks(grad, blk, d, w, seed, bitmaps, sketches)
        else:
            s2.s2_encode_batched(grad, d, w, seed, bitmaps, sketches)

    def decode():
        if blk:
            s2.s2_decode_dense_blocks(bitmap, sketch, n, blk, d, w, seed, out)
        elif compact:
            s2.s2_decode_compact(bitmap, sketch, n, d, w, seed, cidx, cval, ccnt, cws)
        else:
            s2.s2_decode_dense_ws(bitmap, sketch, n, d, w, seed, out, dws)

    def step():
        if fused:
            s2.s2_encode_reduce_fused(grad, d, w, seed, bitmap, sketch)
        else:
            encode()
            s2.s2_reduce(bitmaps, sketches, nbits, d, w, bitmap, sketch)
        decode()

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(physical_gpu_index(local)) as clk:
        wall0 = time.perf_counter()
        for k in range(K):
            flush.fill_(float(k & 7))
            e = ev[k]
            e[0].record(stream)
            if fused:
                s2.s2_encode_reduce_fused(grad, d, w, seed, bitmap, sketch)
                e[1].record(stream)
            else:
                encode()
                e[1].record(stream)
                s2.s2_reduce(bitmaps, sketches, nbits, d, w, bitmap, sketch)
            e[2].record(stream)
            decode()
            e[3].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    enc_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    red_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    dec_ms = sum(e[2].elapsed_time(e[3]) for e in ev)
    total_ms = enc_ms + red_ms + dec_ms
    elapsed, units = combine_over_ranks(total_ms / 1e3, float(W * n * K), world, dev)
    value = units / elapsed / 1e9

    by = algorithmic_bytes(wl, nnz_u, blk, compact)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]
    enc_s = enc_ms / 1e3 / K
    n_enc = encode_launches(wl, l2)
    n_dec = 3 if args.decode == "compact" else dense_decode_launches(n, l2, d, w, blk)
    ach_enc = by["encode"] / enc_s / 1e9
    path_gbs = by["total"] / (total_ms / 1e3 / K) / 1e9
    traffic = recorded_traffic(config_name or args.config)

    res = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "Gelem/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if wl.dtype == "f32" else "bf16",
        "data": "synthetic",
        "config": dict(wl.describe(), nnz_union=nnz_u, l2="flushed before every step (512 MiB write)",
                       parallelism=f"replicas{world}" if world > 1 else "single GPU, W workers resident"),
        "stages_ms_per_step": {"encode": round(enc_ms / K, 5), "reduce": round(red_ms / K, 5),
                               "decode": round(dec_ms / K, 5)},
        "roofline": {"kernel": "encode (zero fill + fused bitmap/sketch scatter)", "bound": "hbm",
                     "achieved": round(ach_enc, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(ach_enc / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_step": by["encode"], "launches_per_step": n_enc,
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "path_roofline": {"bound": "hbm", "achieved": round(path_gbs, 1), "peak": peak, "unit": "GB/s",
                          "frac": round(path_gbs / peak, 4), "algorithmic_bytes_per_step": by["total"],
                          "stage_frac": {k: round(by[k] / (v / 1e3 / K) / 1e9 / peak, 4) for k, v in
                                         (("encode", enc_ms), ("reduce", red_ms), ("decode", dec_ms))}},
        "gpu_launches": K * (n_enc + 1 + n_dec),
        "wall_ms_timed_region": round(wall * 1e3, 3),
    }
    ops = l2_sector_ops(wl, nnz_u, blk, compact)
    ceil = measured_ceilings()
    step_s = total_ms / 1e3 / K
    l2 = {"unit": "G sector ops/s", "ops_per_step": ops, "achieved": round(ops["total"] / step_s / 1e9, 1)}
    if ceil:
        c = float(ceil["red_f32"]["Gops_per_s"])
        l2.update(peak=c, frac=round(ops["total"] / step_s / 1e9 / c, 4),
                  peak_source="scattered red.f32 rate measured by bench.py --ceilings (profiles/ceilings_gb300.json)")
    res["l2_roofline"] = l2
    res["config"]["mode"] = ("per_worker (encode_batched + reduce + decode_compact)" if compact else
                             "per_worker (encode_batched + reduce + decode_dense_ws)")
    if blk:
        res["config"]["mode"] = f"per_worker, block bitmap of {blk} positions (encode_batched_blocks + reduce + decode_dense_blocks)"
        res["gpu_launches"] = K * (n_enc + 1 + 1 + n_dec)  # + the block bitmaps' zero fill
    if fused:
        # same step with encode + reduce replaced by the fused single-sketch pass
        byf = algorithmic_bytes_fused(wl, nnz_u)
        fused_s = enc_ms / 1e3 / K
        ach = byf["encode_reduce_fused"] / fused_s / 1e9
        pg = byf["total"] / step_s / 1e9
        res["config"]["mode"] = "fused_single_sketch (encode_reduce_fused + decode_dense_ws)"
        res["stages_ms_per_step"] = {"encode_reduce_fused": round(enc_ms / K, 5), "decode": round(dec_ms / K, 5)}
        res["roofline"] = {"kernel": "encode_reduce_fused (zero fill + one pass over all workers)", "bound": "hbm",
                           "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                           "traffic": None, "algorithmic_bytes_per_step": byf["encode_reduce_fused"],
                           "launches_per_step": 2, "peak_source": res["roofline"]["peak_source"]}
        res["path_roofline"] = {"bound": "hbm", "achieved": round(pg, 1), "peak": peak, "unit": "GB/s",
                                "frac": round(pg / peak, 4), "algorithmic_bytes_per_step": byf["total"]}
        res["gpu_launches"] = K * (2 + n_dec)
        opsf = l2_sector_ops_fused(wl, nnz_u)
        l2 = dict(l2, ops_per_step=opsf, achieved=round(opsf["total"] / step_s / 1e9, 1))
        if ceil:
            l2["frac"] = round(opsf["total"] / step_s / 1e9 / float(ceil["red_f32"]["Gops_per_s"]), 4)
        res["l2_roofline"] = l2
    res["clocks"] = clk.summary()

    if not args.no_e2e:
        res["e2e"] = run_e2e(args, wl, dev, s2)
    if rank == 0 and world == 1 and not args.no_cpu:
        G = wl.dense()
        o = time_oracle(wl, G, reps=1)
        res["cpu_baseline"] = {"value": round(o["value"], 5), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                               "sample": f"one full encode->reduce->decode of this workload on the host "
                                         f"({o['seconds']:.2f} s, single thread, plain C, fp64)"}
        ot = time_oracle_threads(wl, G)
        res["cpu_baseline_threads"] = {
            "value": round(ot["value"], 5), "unit": "Gelem/s", "cores": ot["threads"], "kind": "oracle",
            "sample": f"the same pass with the {wl.W} workers' encodes on {ot['threads']} host threads, reduce and "
                      f"decode on one ({ot['seconds']:.2f} s; host has {os.cpu_count()} cores)"}
    return res


# The workloads whose whole-path HBM fraction is a target, besides the headline.
GATED_CONFIGS = ("embedding", "topk")
PER_CONFIG_KEYS = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "stages_ms_per_step", "roofline",
                   "path_roofline", "l2_roofline", "gpu_launches", "clocks", "e2e", "cpu_baseline",
                   "cpu_baseline_threads")


def run_per_config(args, world, rank, local, names=GATED_CONFIGS) -> dict:
    """The same measurement on the other gated workloads, one after the other
    in this process (each with its own warm-up and timed steps)."""
    import torch

    out = {}
    for name in names:
        wl = workloads.by_name(name)
        r = run_ours(args, wl, world, rank, local, config_name=name)
        out[r["config"]["workload"]] = {k: r[k] for k in PER_CONFIG_KEYS if k in r}
        del wl, r
        torch.cuda.empty_cache()
    return out


def run_blocktopk(args, world, rank, local):
    """Dense ResNet-50-size gradients -> block-wise Top-K (256-element blocks,
    1/32 of the blocks kept, residual carried across steps) -> the per-worker
    encode -> reduce -> decode path."""
    import torch

    import sketch_compressed_sparse_gb300 as s2

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    W, n, block, d, w, seed = 8, 25_557_032, 256, 3, 1 << 19, 0
    nb = (n + block - 1) // block
    K = nb // 32
    grad = torch.from_numpy(workloads.dense_laplace(W, n)).to(dev)
    resid = torch.zeros_like(grad)
    sparse = torch.empty_like(grad)
    ws = torch.empty(s2.s2_block_topk_workspace_size(W, n, block), dtype=torch.uint8, device=dev)
    bitmaps = torch.empty((W, s2.nwords(n)), dtype=torch.int32, device=dev)
    sketches = torch.empty((W, d, w), dtype=torch.float32, device=dev)
    bitmap = torch.empty(s2.nwords(n), dtype=torch.int32, device=dev)
    sketch = torch.empty((d, w), dtype=torch.float32, device=dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def stages(ev=None):
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        s2.s2_block_topk(grad, resid, block, K, sparse, ws)
        rec(1)
        s2.s2_encode_batched(sparse, d, w, seed, bitmaps, sketches)
        rec(2)
        s2.s2_reduce(bitmaps, sketches, n, d, w, bitmap, sketch)
        rec(3)
        s2.s2_decode_dense(bitmap, sketch, n, d, w, seed, out)
        rec(4)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        stages()
    Ksteps = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(Ksteps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(physical_gpu_index(local)) as clk:
        for k in range(Ksteps):
            flush.fill_(float(k & 7))
            stages(evs[k])
        torch.cuda.synchronize(dev)
    t = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / Ksteps for i in range(4)]
    step_ms = sum(t)
    union = int((torch.from_numpy(np.unpackbits(bitmap.cpu().numpy().view(np.uint8), bitorder="little")[:n])).sum())
    peak = measured_peaks()["hbm_gbs"]
    topk_bytes = W * n * 16  # read grad and residual, write sparse output and residual
    SK, BM = 4 * d * w, 4 * ((n + 31) // 32)
    enc_b, red_b = W * n * 4 + W * BM + W * SK, W * (SK + BM) + SK + BM
    dec_b = BM + min(SK, 4 * d * union) + 4 * n
    total_b = topk_bytes + enc_b + red_b + dec_b
    return {
        "metric": METRIC, "value": round(W * n / (step_ms / 1e3) / 1e9, 3), "unit": "Gelem/s", "n_gpus": world,
        "steps": Ksteps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "block_topk_resnet50", "W": W, "n": n, "block": block, "K": K, "d": d, "w": w,
                   "hash_seed": seed, "nnz_union_last_step": union,
                   "mode": "block-wise Top-K with error feedback, then the per-worker path",
                   "l2": "flushed before every step (512 MiB write)"},
        "stages_ms_per_step": {"block_topk": round(t[0], 5), "encode": round(t[1], 5), "reduce": round(t[2], 5),
                               "decode": round(t[3], 5)},
        "roofline": {"kernel": "block_topk (norms + select + apply)", "bound": "hbm",
                     "achieved": round(topk_bytes / (t[0] / 1e3) / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(topk_bytes / (t[0] / 1e3) / 1e9 / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_step": topk_bytes},
        "path_roofline": {"bound": "hbm", "achieved": round(total_b / (step_ms / 1e3) / 1e9, 1), "peak": peak,
                          "unit": "GB/s", "frac": round(total_b / (step_ms / 1e3) / 1e9 / peak, 4),
                          "algorithmic_bytes_per_step": total_b},
        # Top-K: norms, histogram zero fill, 4 radix passes, equal counts, keep, apply
        "gpu_launches": Ksteps * (9 + encode_launches(workloads.Workload("x", W, n, d, w, 0, "f32", [], []),
                                                      int(torch.cuda.get_device_properties(dev).L2_cache_size)) + 2),
        "clocks": clk.summary(),
    }


def run_allgather(args, wl, world, rank, local):
    """The sparse AllGather baseline on the same workload: pack every worker's
    (index, value) list, sum the gathered lists; beside it the bytes each
    worker would send with either method and the S2 decode's error against
    this exact aggregate."""
    import torch

    import sketch_compressed_sparse_gb300 as s2

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    W, n, d, w, seed = wl.W, wl.n, wl.d, wl.w, wl.seed
    if wl.dtype != "f32":
        raise SystemExit("the AllGather baseline takes float32 gradients")
    cap = max(wl.nnz_per_worker)
    grad = wl.dense_torch(dev)
    idx = torch.empty((W, cap), dtype=torch.int32, device=dev)
    val = torch.empty((W, cap), dtype=torch.float32, device=dev)
    cnt = torch.empty(W, dtype=torch.int64, device=dev)
    ws = torch.empty(s2.s2_sparse_pack_workspace_size(W, n), dtype=torch.uint8, device=dev)
    exact = torch.empty(n, dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        s2.s2_sparse_pack(grad, idx, val, cnt, ws)
        s2.s2_sparse_sum(idx, val, cnt, n, exact)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize(dev)
    with ClockSampler(physical_gpu_index(local)) as clk:
        for k in range(K):
            flush.fill_(float(k & 7))
            e = evs[k]
            e[0].record(stream)
            s2.s2_sparse_pack(grad, idx, val, cnt, ws)
            e[1].record(stream)
            s2.s2_sparse_sum(idx, val, cnt, n, exact)
            e[2].record(stream)
        torch.cuda.synchronize(dev)
    pack_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    sum_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    # the S2 path once, untimed, for its error against the exact aggregate
    bitmaps, sketches = s2.alloc_encode_outputs(W, n, d, w, dev)
    bitmap = torch.empty(s2.nwords(n), dtype=torch.int32, device=dev)
    sketch = torch.empty((d, w), dtype=torch.float32, device=dev)
    out = torch.empty(n, dtype=torch.float32, device=dev)
    s2.s2_encode_batched(grad, d, w, seed, bitmaps, sketches)
    s2.s2_reduce(bitmaps, sketches, n, d, w, bitmap, sketch)
    s2.s2_decode_dense(bitmap, sketch, n, d, w, seed, out)
    torch.cuda.synchronize(dev)
    err = (out.double() - exact.double()).norm().item() / max(exact.double().norm().item(), 1e-300)
    nnz = [int(c) for c in cnt.cpu().tolist()]
    bytes_ag = 8 * sum(nnz) // W
    bytes_s2 = 4 * d * w + 4 * ((n + 31) // 32)
    peak = measured_peaks()["hbm_gbs"]
    alg = W * n * 4 + 2 * 8 * sum(nnz) + 4 * n  # read grads, write + read the lists, write the sum
    step_ms = pack_ms + sum_ms
    return {
        "metric": METRIC, "value": round(W * n / (step_ms / 1e3) / 1e9, 3), "unit": "Gelem/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(wl.describe(), mode="sparse AllGather baseline (pack + sum), exact aggregate",
                       l2="flushed before every step (512 MiB write)"),
        "stages_ms_per_step": {"pack": round(pack_ms, 5), "sum": round(sum_ms, 5)},
        "path_roofline": {"bound": "hbm", "achieved": round(alg / (step_ms / 1e3) / 1e9, 1), "peak": peak,
                          "unit": "GB/s", "frac": round(alg / (step_ms / 1e3) / 1e9 / peak, 4),
                          "algorithmic_bytes_per_step": alg},
        "message_bytes_per_worker": {"allgather_lists": bytes_ag, "s2_sketch_and_bitmap": bytes_s2,
                                     "ratio_s2_over_allgather": round(bytes_s2 / max(bytes_ag, 1), 4)},
        # bytes one worker receives in a ring collective over W workers: the
        # AllGather brings every other worker's list, the AllReduce of the
        # sketch and bitmap 2(W-1)/W of the message (reduce-scatter + gather)
        "ring_bytes_received_per_worker": {
            "allgather": (W - 1) * 8 * sum(nnz) // W,
            "s2_allreduce": 2 * (W - 1) * bytes_s2 // W},
        "s2_decode_rel_l2_error_vs_exact": err,
        "gpu_launches": K * (2 + W + 1 + W),
        "clocks": clk.summary(),
    }


def encode_path_points():
    """Workloads of the encode-path comparison: 8 workers of 2^22 uniform
    positions with d = 3 and few buckets per row (16 .. 16384) at 1, 10 and
    50 % density, where the L2 reductions of many nonzeros pile up on few
    buckets; and the sweep points whose sketch fits in shared memory."""
    pts = []
    for w in (16, 64, 256, 1024, 4096, 16384):
        for rho in (0.01, 0.1, 0.5):
            pts.append(("custom", dict(W=8, n=1 << 22, d=3, w=w, density=rho, tag=7)))
    for e in (20, 22, 24):
        for dt in ("f32", "bf16"):
            for d in (3, 5):
                p = dict(n=1 << e, dtype=dt, density=0.001, d=d)
                if 4 * d * workloads.sweep_w(int(round(0.001 * (1 << e)))) <= 192 * 1024:
                    pts.append(("sweep", p))
    return pts


def run_encode_paths(args):
    """Encode alone (s2_encode_batched_path) on each point with the L2 path,
    the shared-memory path and the automatic choice; median of the timed
    repetitions, L2 flushed before each."""
    import torch

    import sketch_compressed_sparse_gb300 as s2

    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(5, min(args.steps, 30))
    rows = []
    want = {}
    for kv in filter(None, (args.paths_select or "").split(",")):
        k, v = kv.split("=")
        want[k.strip()] = float(v)
    with ClockSampler(physical_gpu_index(0)) as clk:
        for kind, p in encode_path_points():
            if kind != "custom" and want:
                continue
            if any(float(p.get(k, -1)) != v for k, v in want.items()):
                continue
            wl = workloads.custom(**p) if kind == "custom" else workloads.sweep_point(**p)
            g = wl.dense_torch(dev)
            W, n = g.shape
            bm, sk = s2.alloc_encode_outputs(W, n, wl.d, wl.w, dev)
            row = {"workload": wl.name, "W": W, "n": n, "d": wl.d, "w": wl.w, "density": p["density"],
                   "dtype": wl.dtype}
            for path in ("l2", "smem", "auto"):
                for _ in range(max(3, args.warmup)):
                    s2.s2_encode_batched_path(g, wl.d, wl.w, wl.seed, bm, sk, path=path)
                ts = []
                for r in range(reps):
                    flush.fill_(float(r & 7))
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    s2.s2_encode_batched_path(g, wl.d, wl.w, wl.seed, bm, sk, path=path)
                    b.record()
                    torch.cuda.synchronize(dev)
                    ts.append(a.elapsed_time(b))
                row[path + "_ms"] = round(statistics.median(ts), 5)
            row["smem_speedup"] = round(row["l2_ms"] / row["smem_ms"], 3)
            rows.append(row)
            del g, bm, sk
    return {"metric": "encode ms per step, L2 vs shared-memory sketch path", "unit": "ms", "n_gpus": 1,
            "repetitions": reps, "data": "synthetic", "l2": "flushed before every repetition (512 MiB write)",
            "points": rows, "clocks": clk.summary()}


def run_sweep(args):
    """The sweep grid (8 workers, n = 2^20 .. 2^max, fp32/bf16, density 0.1 /
    1 / 10 %, d = 3 or 5, w = nnz/2 rounded to a power of two) through the
    per-worker path, one compact row per point."""
    import copy

    import torch

    rows = []
    sub = copy.copy(args)
    sub.no_e2e, sub.no_cpu, sub.block, sub.mode = True, True, 0, "per_worker"
    sub.steps = max(5, min(args.steps, 30))
    sub.warmup = max(3, args.warmup)
    t0 = time.perf_counter()
    for p in workloads.sweep_grid():
        if p["n"] > (1 << args.sweep_max_log2) or p["n"] < (1 << args.sweep_min_log2):
            continue
        if args.sweep_density is not None and p["density"] != args.sweep_density:
            continue
        wl = workloads.sweep_point(**p)
        r = run_ours(sub, wl, 1, 0, 0)
        rows.append({"n": wl.n, "dtype": wl.dtype, "density": p["density"], "d": wl.d, "w": wl.w,
                     "nnz_union": r["config"]["nnz_union"], "ms_per_step": r["ms_per_step"],
                     "gelem_s": r["value"], "stages_ms": r["stages_ms_per_step"],
                     "hbm_frac_path": r["path_roofline"]["frac"],
                     "l2_frac": r["l2_roofline"].get("frac")})
        del wl
        torch.cuda.empty_cache()
    peaks = measured_peaks()
    return {"metric": METRIC + " (sweep grid)", "unit": "Gelem/s", "n_gpus": 1, "steps_per_point": sub.steps,
            "warmup": sub.warmup, "higher_is_better": True, "data": "synthetic",
            "config": {"workload": "sweep: W=8, n=2^%d..2^%d, fp32/bf16, density %s, d in {3,5}, "
                                   "w = 2^round(log2(nnz/2))" % (args.sweep_min_log2, args.sweep_max_log2,
                                                                 "0.1/1/10 %" if args.sweep_density is None
                                                                 else f"{100 * args.sweep_density:g} %"),
                       "l2": "flushed before every step (512 MiB write)"},
            "hbm_peak_gbs": peaks["hbm_gbs"], "points": rows,
            "wall_s": round(time.perf_counter() - t0, 1)}


def run_e2e(args, wl, dev, s2):
    """Host pinned grad -> device -> path -> host out, through s2_pipeline_dense_host."""
    import torch

    G = wl.dense()
    hg = torch.from_numpy(G if wl.dtype == "f32" else G.view(np.int16)).pin_memory()
    if wl.dtype == "bf16":
        hg = hg.view(torch.bfloat16)
    ho = torch.empty(wl.n, dtype=torch.float32).pin_memory()
    ws = torch.empty(s2.s2_pipeline_workspace_size(hg.dtype, wl.W, wl.n, wl.d, wl.w), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        s2.s2_pipeline_dense_host(hg, wl.d, wl.w, wl.seed, ho, ws)
    torch.cuda.synchronize(dev)
    K = max(3, min(args.steps, args.e2e_steps))
    t = 0.0
    for _ in range(K):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s2.s2_pipeline_dense_host(hg, wl.d, wl.w, wl.seed, ho, ws)
        b.record(stream)
        b.synchronize()
        t += a.elapsed_time(b) / 1e3
    h2d, d2h = int(wl.W * wl.n * wl.elem_bytes), int(4 * wl.n)
    res = {"value": round(wl.W * wl.n * K / t / 1e9, 3), "unit": "Gelem/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": K, "ms_per_step": round(t / K * 1e3, 4),
           "transfer": "pinned host gradient and output; the library's kernels read and write them in place "
                       "(mapped page-locked memory), so the host<->device bytes move inside the kernels"}
    ceil = measured_ceilings()
    link = (ceil or {}).get("host")
    if link and link.get("sm_read_GBps") and link.get("sm_write_GBps"):
        # the time the host link alone needs for this step's bytes, at the rates
        # `bench.py --ceilings` measured for kernels reading and writing mapped host memory
        bound_ms = (h2d / link["sm_read_GBps"] + d2h / link["sm_write_GBps"]) / 1e6
        res["host_link"] = {"bound_ms_per_step": round(bound_ms, 4), "frac": round(bound_ms / (t / K * 1e3), 4),
                            "read_GBps": link["sm_read_GBps"], "write_GBps": link["sm_write_GBps"],
                            "source": "bench.py --ceilings (profiles/ceilings_gb300.json)"}
    return res


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, wl):
    G = wl.dense()
    one = time_oracle(wl, G, reps=1)  # also the untimed warm-up
    budget_s = 150.0
    K = max(1, min(args.steps, int(budget_s // max(one["seconds"], 1e-3))))
    o = time_oracle(wl, G, reps=K)
    v = round(o["value"], 5)
    sample = (f"{K} full encode->reduce->decode passes of this workload (of {args.steps} requested; bounded to "
              f"~{budget_s:.0f} s), single thread, plain C, fp64")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": "Gelem/s",
        "n_gpus": 1,
        "steps": K,
        "warmup": 1,
        "ms_per_step": round(o["seconds"] * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": dict(wl.describe(), nnz_union=wl.union_nnz()),
        "cpu_baseline": {"value": v, "unit": "Gelem/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def select_workers(wl: workloads.Workload, k):
    if k is None or k >= wl.W:
        return wl
    wl.W, wl.idx, wl.val = k, wl.idx[:k], wl.val[:k]
    wl.name = f"{wl.name}_W{k}"
    return wl


def run_ceilings(args):
    """Compile ceilings.cu for sm_103a and print its JSON line."""
    import tempfile

    from sketch_compressed_sparse_gb300 import build as b

    with tempfile.TemporaryDirectory() as td:
        exe = os.path.join(td, "ceilings")
        subprocess.check_call([b.nvcc(), *b.ARCH, "-O3", "-o", exe, os.path.join(ROOT, "ceilings.cu")])
        out = subprocess.run([exe], capture_output=True, text=True)
    line = out.stdout.strip().splitlines()[-1] if out.stdout.strip() else json.dumps({"error": out.stderr[-500:]})
    print(line, flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(line + "\n")
    return out.returncode


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="large_lm",
                    choices=["tiny", "embedding", "topk", "large_lm", "blocktopk", "sweep"])
    ap.add_argument("--no-per-config", action="store_true",
                    help="large_lm per-worker run only: skip the embedding and top-k measurements in per_config")
    ap.add_argument("--sweep-max-log2", type=int, default=28,
                    help="--config sweep: largest gradient length as a power of two (20..28)")
    ap.add_argument("--sweep-min-log2", type=int, default=20,
                    help="--config sweep: smallest gradient length as a power of two (20..28)")
    ap.add_argument("--sweep-density", type=float, default=None, choices=[0.001, 0.01, 0.1],
                    help="--config sweep: only the points of this density")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle timing")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--mode", choices=["per_worker", "fused", "allgather"], default="per_worker",
                    help="per_worker: the simulated data-parallel path (default); fused: encode_reduce_fused + "
                         "decode; allgather: the sparse AllGather baseline (exact sum) on the same workload")
    ap.add_argument("--decode", choices=["dense", "compact"], default="dense",
                    help="decode output: dense [n] (default) or compacted (index, value) pairs")
    ap.add_argument("--block", type=int, default=0,
                    help="positions per bitmap bit (a multiple of 32; 0 = one bit per position, the default)")
    ap.add_argument("--workers", type=int, default=None,
                    help="profiling aid: keep only the first K workers of the workload (changes the workload)")
    ap.add_argument("--ceilings", action="store_true",
                    help="build and run ceilings.cu (device ceilings of scattered L2 operations) and exit")
    ap.add_argument("--paths-select", default=None,
                    help="--encode-paths: keep only the small-sketch points matching e.g. 'w=256,density=0.5'")
    ap.add_argument("--encode-paths", action="store_true",
                    help="time encode on the L2 and the shared-memory sketch paths over small-sketch workloads, "
                         "print one JSON line and exit")
    args = ap.parse_args(argv)
    if args.ceilings:
        return run_ceilings(args)
    if args.encode_paths:
        res = run_encode_paths(args)
        print(json.dumps(res), flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(json.dumps(res) + "\n")
        return 0
    if args.warmup < 3 and args.impl == "ours" and args.steps > 5:
        ap.error("use at least 3 warm-up steps")

    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        if args.config in ("blocktopk", "sweep"):
            res = {"impl": "reference", "unavailable": "the CPU reference arm covers the four S2 workloads only"}
        else:
            res = run_reference(args, workloads.by_name(args.config))
    else:
        if world > 1:
            import torch
            import torch.distributed as dist

            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        if args.config == "blocktopk":
            res = run_blocktopk(args, world, rank, local)
        elif args.config == "sweep":
            res = run_sweep(args)
        elif args.mode == "allgather":
            res = run_allgather(args, workloads.by_name(args.config), world, rank, local)
        else:
            res = run_ours(args, select_workers(workloads.by_name(args.config), args.workers), world, rank, local)
            if (args.config == "large_lm" and args.mode == "per_worker" and args.workers is None
                    and not args.no_per_config):
                import torch

                torch.cuda.empty_cache()
                res["per_config"] = run_per_config(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        if rank != 0:
            return 0
    line = json.dumps(res)
    print(line, flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(line + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
