#!/usr/bin/env python3
"""Benchmark of the fused FP4 paged-MQA indexer prefill + exact TopK on GB300.

Workload (default): Q=8192 rows, H=64, D=128, K=1024, C4 context 196,608 (the
V4-Pro-shaped prefill of "[FlyDSL] Add FP4 LiteTopK prefill operator",
ROCm/aiter#5309, Validation table), one request whose rows are its last 8192
raw tokens, causal windows, shuffled page table, seeded synthetic FP4/UE8M0
values.

One step = one idx_topk_fp4_prefill call (plan, page validation, fused
score+select, merge+map, status read-back) on inputs resident in HBM; L2 is
flushed (256 MiB write) before every timed step, outside the step's events.
Metric value = algorithmic FP4 FLOP (2*64*128 per scored (row, slot)) per
second, summed over ranks (each rank runs the whole workload: weak scaling).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused score+TopK ms & FP4 TFLOPS (% peak) at Q=8192, C4=196608, K=1024"
# The pages' own fused-path times for two of the workloads (Q=8192 rows, MI355X;
# "[FlyDSL] Add FP4 LiteTopK prefill operator", Validation table): another
# machine's numbers, the denominator of vs_baseline, not targets.
PAGES_MS = {"pro-R8192-S196608-K1024": 10.6433,    # V4-Pro, K=1024, C4 196,608
            "flash-R8192-S131072-K512": 7.2235}    # V4-Flash, K=512, C4 131,072
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense FP4 : bf16 tensor ratio of GB300
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
EPI_OPS_PER_ELEMENT = 2               # ReLU max + weighted multiply-add per (row, head, slot)
FP32_LANES_PER_SM = 128               # 4 partitions x 32 lanes, one warp instruction per clock each
EPI_OPS_PER_ISSUE = 4.0 / 3.0         # per head pair: two max.f32 + one fma.rn.f32x2 = 4 ops, 3 issues
NOMINAL_SM_MHZ = 2070.0
KERNELS_PER_CALL = 4                  # plan, page check, scorer, finish (row-team sort + multi-unit merge in one launch)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", type=int, default=3, help="workload index (default 3)")
    ap.add_argument("--pairs", type=int, default=15, help="alternating dense/fused pairs")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload lines and the fresh-process repeats")
    ap.add_argument("--decode-only", action="store_true",
                    help="only the decode-shaped batches (graph replay and synchronous call)")
    ap.add_argument("--child-pairs", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "hardware")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def vs_baseline(workload: str, flop: float, value_tflops: float):
    """value / the pages' throughput on the same workload (the same algorithmic
    FLOP over the pages' time), or None where the pages give no time for it."""
    ms = PAGES_MS.get(workload)
    if ms is None:
        return None
    return value_tflops / (flop / (ms * 1e-3) / 1e12)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (the slowest rank's time); x itself
    at world size 1."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs the same workload (weak scaling),
    so the job does world x the work in the slowest rank's time."""
    return world * flop_per_rank / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def score_kernel_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_sparse_attention_tma_gb300", "csrc")
    for name in ("score.cu", "idx_device.cuh", "idx_select.cuh", "idx_internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the scoring kernel from the committed ncu
    summary, only when it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "score_kernel_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_sha") == score_kernel_sha() and d.get("workload") == workload:
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                n += 1
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def cpu_baseline(p, seconds: float):
    """The oracle, as it stands, on a bounded sample of rows of the workload."""
    import numpy as np
    import oracle
    oracle.build()
    K = p.topk
    scored = np.nonzero(p.lengths() > K)[0]
    t0 = time.perf_counter()
    oracle.prefill_rows(p, rows=scored[-1:].astype(np.int32))
    t_row = max(time.perf_counter() - t0, 1e-3)
    n = int(max(1, min(len(scored), seconds / t_row)))
    pick = scored[np.linspace(0, len(scored) - 1, n).astype(np.int64)].astype(np.int32)
    t0 = time.perf_counter()
    oracle.prefill_rows(p, rows=pick)
    dt = time.perf_counter() - t0
    flop = float(p.lengths()[pick].sum()) * 2 * 64 * 128
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
            "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{n} of {len(scored)} scored rows (evenly spaced), full windows, "
                      f"{dt:.1f} s wall",
            "seconds": dt}


def timed_pairs(m, dev, p, n_warm, n_pairs, flush):
    """Alternating dense-then-TopK / fused calls on one stream (L2 flushed before
    each), n_warm pairs untimed then n_pairs timed with CUDA events; the two
    medians and whether the outputs were identical."""
    import torch
    R, K = p.rows, p.topk
    phys = torch.empty((R, K), dtype=torch.int32, device="cuda")
    raw = torch.empty((R, K), dtype=torch.int32, device="cuda")
    d_phys = torch.empty_like(phys)
    d_raw = torch.empty_like(raw)
    ws = torch.empty((R, p.max_end()), dtype=torch.float32, device="cuda")
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def fused():
        m.idx_topk_fp4_prefill(**dev, topk=K, out_phys_slot=phys, out_raw_idx=raw)

    def dense():
        m.idx_dense_topk_fp4_prefill(**dev, topk=K, out_phys_slot=d_phys, out_raw_idx=d_raw,
                                     score_workspace=ws)

    f_ms, d_ms = [], []
    for i in range(n_warm + n_pairs):
        for fn, acc in ((dense, d_ms), (fused, f_ms)):
            flush.zero_()
            ev0.record()
            fn()
            ev1.record()
            ev1.synchronize()
            if i >= n_warm:
                acc.append(ev0.elapsed_time(ev1))
    same = bool(torch.equal(d_raw, raw) and torch.equal(d_phys, phys))
    return {"fused_ms_median": statistics.median(f_ms), "dense_ms_median": statistics.median(d_ms),
            "indices_identical": same, "score_storage_bytes": ws.numel() * 4}


def child_pairs(args):
    """One fresh process of the repeated measurement: 5 warm-up and
    args.pairs timed dense/fused pairs on the workload; prints one JSON line."""
    import numpy as np
    import torch
    import fp4_sparse_attention_tma_gb300 as m
    from fp4_sparse_attention_tma_gb300 import inputs
    torch.cuda.set_device(0)
    p = inputs.config(args.config)
    dev = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).cuda()
           for k in ("q_fp4", "q_scale", "k_cache_fp4", "k_scale", "weights", "page_table",
                     "row_req", "row_start", "row_end")}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    print(json.dumps(timed_pairs(m, dev, p, 5, args.pairs, flush)), flush=True)


def fresh_processes(args, n=3):
    """The dense/fused pair measurement repeated in n fresh processes (each 5
    warm-up + args.pairs timed pairs); the median over processes of each
    process's median."""
    runs = []
    for _ in range(n):
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--child-pairs",
                              "--config", str(args.config), "--pairs", str(args.pairs)],
                             capture_output=True, text=True, timeout=600)
        if out.returncode != 0:
            raise RuntimeError("fresh-process measurement failed:\n" + out.stderr[-2000:])
        runs.append(json.loads(out.stdout.strip().splitlines()[-1]))
    return {"processes": n, "warmup_pairs": 5, "timed_pairs": args.pairs,
            "fused_ms_median": statistics.median(r["fused_ms_median"] for r in runs),
            "dense_ms_median": statistics.median(r["dense_ms_median"] for r in runs),
            "indices_identical": all(r["indices_identical"] for r in runs),
            "per_process": [{"fused_ms": r["fused_ms_median"], "dense_ms": r["dense_ms_median"]}
                            for r in runs]}


def other_workloads(m, local, flush, cfgs=(0, 1, 2, 4), steps=10, warm=3):
    """The other configurations through the same call, timed in this run: per
    workload the call's mean time (L2 flushed before each call; the library's
    per-call phase events off, as in a user's call), its algorithmic TFLOP/s,
    the scorer's time (a second pass with the phase events on) and the scratch
    a call takes."""
    import numpy as np
    import torch
    from fp4_sparse_attention_tma_gb300 import inputs
    out = []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    for c in cfgs:
        p = inputs.config(c)
        dev = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).cuda()
               for k in ("q_fp4", "q_scale", "k_cache_fp4", "k_scale", "weights", "page_table",
                         "row_req", "row_start", "row_end")}
        phys = torch.empty((p.rows, p.topk), dtype=torch.int32, device="cuda")
        raw = torch.empty_like(phys)
        ms, sc = [], []
        m.idx_topk_set_timing(False)
        for i in range(warm + steps):
            flush.zero_()
            ev0.record()
            m.idx_topk_fp4_prefill(**dev, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw)
            ev1.record()
            ev1.synchronize()
            if i >= warm:
                ms.append(ev0.elapsed_time(ev1))
        m.idx_topk_set_timing(True)
        for i in range(steps):
            flush.zero_()
            m.idx_topk_fp4_prefill(**dev, topk=p.topk, out_phys_slot=phys, out_raw_idx=raw)
            sc.append(m.idx_topk_last_timings()["score_ms"])
        m.idx_topk_set_timing(False)
        flop = float(p.algorithmic_flop())
        call = statistics.mean(ms)
        out.append({"workload": p.name, "rows": p.rows, "topk": p.topk,
                    "scored_pairs": p.scored_pairs(), "algorithmic_flop": flop,
                    "call_ms": call, "tflops": flop / (call * 1e-3) / 1e12,
                    "score_ms": statistics.mean(sc),
                    "scratch_bytes": m.idx_topk_fp4_scratch_bytes(p.rows, p.topk, local),
                    "steps": steps})
        del dev, phys, raw
    return out


def decode_latency(m, flush, reps=30):
    """Decode-shaped batches (32 requests x 2 rows, contexts 4K-64K, topk 512
    and 1024): the stream-ordered call captured into a CUDA graph and replayed
    (median over `reps` replays, CUDA events around each; with the L2 flushed
    before each replay, and back to back), and the synchronous call (L2
    flushed before each).  The replay's outputs must equal the synchronous
    call's and its device status must be 0."""
    import numpy as np
    import torch
    from fp4_sparse_attention_tma_gb300 import inputs
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    out = []
    for K in (512, 1024):
        p = inputs.decode_batch(32, K)
        dev = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).cuda()
               for k in ("q_fp4", "q_scale", "k_cache_fp4", "k_scale", "weights", "page_table",
                         "row_req", "row_start", "row_end")}
        ws = torch.empty(m.idx_topk_fp4_scratch_bytes(p.rows, K), dtype=torch.uint8,
                         device="cuda")
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        phys = torch.empty((p.rows, K), dtype=torch.int32, device="cuda")
        raw = torch.empty_like(phys)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                m.idx_topk_fp4_prefill_async(**dev, topk=K, out_phys_slot=phys, workspace=ws,
                                             status=st, out_raw_idx=raw)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            m.idx_topk_fp4_prefill_async(**dev, topk=K, out_phys_slot=phys, workspace=ws,
                                         status=st, out_raw_idx=raw)
        cold, warm, sync = [], [], []
        for i in range(reps + 3):
            flush.zero_()
            ev0.record()
            g.replay()
            ev1.record()
            ev1.synchronize()
            if i >= 3:
                cold.append(ev0.elapsed_time(ev1) * 1e3)
        for i in range(reps + 3):
            ev0.record()
            g.replay()
            ev1.record()
            ev1.synchronize()
            if i >= 3:
                warm.append(ev0.elapsed_time(ev1) * 1e3)
        status = int(st.item())
        g_phys, g_raw = phys.clone(), raw.clone()
        s_phys, s_raw = torch.empty_like(phys), torch.empty_like(raw)
        for i in range(13):
            flush.zero_()
            ev0.record()
            m.idx_topk_fp4_prefill(**dev, topk=K, out_phys_slot=s_phys, out_raw_idx=s_raw)
            ev1.record()
            ev1.synchronize()
            if i >= 3:
                sync.append(ev0.elapsed_time(ev1) * 1e3)
        out.append({"workload": p.name, "rows": p.rows, "topk": K,
                    "graph_replay_us": statistics.median(cold),
                    "graph_replay_warm_l2_us": statistics.median(warm),
                    "sync_call_us": statistics.median(sync), "status": status,
                    "indices_identical": bool(torch.equal(g_phys, s_phys) and
                                              torch.equal(g_raw, s_raw))})
        del g, dev, ws, phys, raw
    return out


def run_reference(args):
    """Reference arm: the CPU oracle on the host cores, same metric and workload."""
    import numpy as np
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from fp4_sparse_attention_tma_gb300 import inputs
    oracle.build()
    p = inputs.config(args.config)
    scored = np.nonzero(p.lengths() > p.topk)[0]
    t0 = time.perf_counter()
    oracle.prefill_rows(p, rows=scored[-1:].astype(np.int32))
    t_row = max(time.perf_counter() - t0, 1e-3)
    budget = 150.0
    per_step = int(max(1, min(64, len(scored), budget / (args.steps + args.warmup) / t_row)))
    rng = np.random.default_rng(0)
    times, flops = [], []
    for i in range(args.warmup + args.steps):
        pick = np.sort(rng.choice(scored, size=per_step, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.prefill_rows(p, rows=pick)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            flops.append(float(p.lengths()[pick].sum()) * 2 * 64 * 128)
    value = sum(flops) / sum(times) / 1e12
    sample = f"{per_step} random scored rows per step (full windows) of the workload"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": vs_baseline(p.name, float(p.algorithmic_flop()), value),
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": p.name, "rows": p.rows, "c4_context": p.max_end(),
                       "topk": p.topk},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.child_pairs:
        child_pairs(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    import numpy as np
    import torch
    import torch.distributed as dist

    import fp4_sparse_attention_tma_gb300 as m
    from fp4_sparse_attention_tma_gb300 import inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    p = inputs.config(args.config)
    R, K = p.rows, p.topk
    flop = float(p.algorithmic_flop())
    host = dict(q_fp4=p.q_fp4, q_scale=p.q_scale, k_cache_fp4=p.k_cache_fp4, k_scale=p.k_scale,
                weights=p.weights, page_table=p.page_table, row_req=p.row_req,
                row_start=p.row_start, row_end=p.row_end)
    dev = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in host.items()}
    phys = torch.empty((R, K), dtype=torch.int32, device="cuda")
    raw = torch.empty((R, K), dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    if args.decode_only:
        if rank == 0:
            print(json.dumps({"decode": decode_latency(m, flush)}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    def fused():
        m.idx_topk_fp4_prefill(**dev, topk=K, out_phys_slot=phys, out_raw_idx=raw)

    m.idx_topk_set_timing(True)
    for _ in range(args.warmup):
        flush.zero_()
        fused()
    barrier()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    step_ms, score_ms, kern_ms = [], [], []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        flush.zero_()
        ev0.record()
        fused()
        ev1.record()
        ev1.synchronize()
        step_ms.append(ev0.elapsed_time(ev1))
        t = m.idx_topk_last_timings()
        score_ms.append(t["score_ms"])
        kern_ms.append(t["kernels_ms"])
    barrier()
    clk = clocks.stop()
    ms_per_step = max_over_ranks(sum(step_ms), world, "cuda") / args.steps
    value = whole_job_tflops(flop, world, ms_per_step)

    # end to end through the C ABI with host buffers: idx_topk_fp4_prefill_host
    # takes the pinned host tensors, copies them in, runs the fused path and
    # copies the outputs back (all inside the timed region)
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in host.items()}
    h_phys = torch.empty((R, K), dtype=torch.int32).pin_memory()
    h_raw = torch.empty((R, K), dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = 2 * R * K * 4
    e2e_ms = []
    n_e2e = max(3, min(args.steps, 20))
    for i in range(n_e2e + 2):
        flush.zero_()
        torch.cuda.synchronize()
        ev0.record()
        m.idx_topk_fp4_prefill_host(**pinned, topk=K, out_phys_slot=h_phys, out_raw_idx=h_raw,
                                    device=torch.cuda.current_device())
        ev1.record()
        ev1.synchronize()
        if i >= 2:
            e2e_ms.append(ev0.elapsed_time(ev1))
    if not (torch.equal(h_phys, phys.cpu()) and torch.equal(h_raw, raw.cpu())):
        raise RuntimeError("host-buffer call and device call disagree")
    barrier()
    e2e_step = max_over_ranks(statistics.mean(e2e_ms), world, "cuda")
    m.idx_topk_set_timing(False)

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": vs_baseline(p.name, flop, value), "dtype": "fp4",
            "data": "synthetic",
            "config": {"workload": p.name, "rows": R, "c4_context": p.max_end(), "topk": K,
                       "heads": 64, "dim": 128, "page": 64, "scored_pairs": p.scored_pairs(),
                       "algorithmic_flop": flop,
                       "l2": "flushed before every timed step (256 MiB write, untimed)",
                       "parallelism": f"replicas x{world} (rows independent; no collective)"},
            "gpu_launches": KERNELS_PER_CALL * args.steps,
            "clocks": clk,
            "e2e": {"value": whole_job_tflops(flop, world, e2e_step), "unit": "TFLOP/s",
                    "ms_per_step": e2e_step, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}}

    peaks, src = measured_peaks()
    fp4_peak = float(peaks["bf16_tflops"]) * NOMINAL_FP4_OVER_BF16
    sc = statistics.mean(score_ms)
    achieved = flop / (sc * 1e-3) / 1e12
    line["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": fp4_peak,
                        "unit": "TFLOP/s", "frac": achieved / fp4_peak,
                        "traffic": ncu_traffic(p.name),
                        "kernel": "score_kernel<select,%d>" % K, "kernel_ms": sc,
                        "peak_source": f"{src} bf16 burst x {NOMINAL_FP4_OVER_BF16:g} "
                                       "(nominal dense FP4/bf16 ratio)"}
    # the epilogue's CUDA-core roof: per (row, head, slot) element one ReLU
    # (max with 0) and one weighted accumulate; a head pair takes two max.f32
    # and one packed fma.rn.f32x2, 4 operations in 3 issue slots, at one warp
    # instruction per clock per SM partition (128 lanes per SM)
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    elem_ops = float(p.scored_pairs()) * 64 * EPI_OPS_PER_ELEMENT
    alu_peak = (sms * FP32_LANES_PER_SM * EPI_OPS_PER_ISSUE *
                float(clk.get("sm_max_mhz") or NOMINAL_SM_MHZ) * 1e6 / 1e12)
    alu_achieved = elem_ops / (sc * 1e-3) / 1e12
    line["roofline_alu"] = {"bound": "alu", "achieved": alu_achieved, "peak": alu_peak,
                            "unit": "Tops/s", "frac": alu_achieved / alu_peak,
                            "ops_per_launch": elem_ops,
                            "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} lanes x 4/3 "
                                           "ops per issue (2 max + 1 packed FMA per head "
                                           "pair) x max SM clock"}
    line["phases_ms"] = {"kernels": statistics.mean(kern_ms), "score": sc}
    line["scratch"] = {"bytes_per_call": m.idx_topk_fp4_scratch_bytes(R, K, local),
                       "pool_high_water": m.idx_topk_scratch_high_water(local),
                       "dense_scores_bytes": m.dense_score_bytes(R, p.max_end())}

    if not args.no_dense:
        pairs = timed_pairs(m, dev, p, 5, args.pairs, flush)
        line["dense_topk"] = {"ms_median": pairs["dense_ms_median"],
                              "fused_ms_median": pairs["fused_ms_median"],
                              "speedup": pairs["dense_ms_median"] / pairs["fused_ms_median"],
                              "pairs": args.pairs, "indices_identical": pairs["indices_identical"],
                              "score_storage_bytes": pairs["score_storage_bytes"]}

    if not args.no_dense:
        # context-tiled comparison path: bounded fp32 chunks of 16384 positions
        tile = 16384
        t_phys = torch.empty_like(phys)
        t_raw = torch.empty_like(raw)
        t_ms = []
        for i in range(2 + 5):
            flush.zero_()
            ev0.record()
            m.idx_tiled_topk_fp4_prefill(**dev, topk=K, out_phys_slot=t_phys, out_raw_idx=t_raw,
                                         context_tile=tile)
            ev1.record()
            ev1.synchronize()
            if i >= 2:
                t_ms.append(ev0.elapsed_time(ev1))
        line["tiled_topk"] = {"ms_median": statistics.median(t_ms), "context_tile": tile,
                              "chunk_buffer_bytes": R * tile * 4,
                              "indices_identical": bool(torch.equal(t_raw, raw) and
                                                        torch.equal(t_phys, phys))}

    if rank == 0 and world == 1 and not args.no_extra:
        line["workloads"] = other_workloads(m, local, flush)
        line["decode"] = decode_latency(m, flush)
        if not args.no_dense:
            line["fresh_processes"] = fresh_processes(args)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(p, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
