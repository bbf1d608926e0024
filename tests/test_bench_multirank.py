"""Multi-rank logic of bench.py on CPU: two gloo ranks, each with its own step
time, agree on the slowest rank's time and report the whole-job throughput of
N replicas of the workload (rows are independent; no data-path collective).
The reference arm (the oracle) prints its line on rank 0 only."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank           # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        out.put((rank, ms, bench.whole_job_tflops(2.0e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in res:
        assert ms == pytest.approx(15.0)
        # 2 replicas x 2e12 FLOP in 15 ms
        assert value == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)


def _run_bench(args, env_extra):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, cwd=root, env=env,
                       capture_output=True, text=True, timeout=300)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return r.returncode, [json.loads(l) for l in lines], r.stderr


def test_reference_arm_prints_one_line_on_rank_zero():
    """The reference arm (the oracle on the host cores) on the smallest workload,
    whose 30 scored rows are fewer than the arm's per-step sample cap."""
    import bench
    code, lines, err = _run_bench(["--impl", "reference", "--config", "0", "--steps", "2",
                                   "--warmup", "3"], {"RANK": "0", "WORLD_SIZE": "1"})
    assert code == 0, err
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny-R32-S4096-K512" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert isinstance(d["cpu_baseline"]["cpu_model"], str) and d["cpu_baseline"]["cpu_model"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["vs_baseline"] is None          # the pages give no time for this workload


def test_reference_arm_other_ranks_exit_without_work():
    code, lines, err = _run_bench(["--impl", "reference", "--config", "0", "--steps", "1",
                                   "--warmup", "3"], {"RANK": "1", "WORLD_SIZE": "2"})
    assert code == 0, err
    assert lines == []


def test_vs_baseline_divides_by_the_pages_throughput_on_the_same_workload():
    import bench
    flop = 2.6251e13
    # the pages' fused-path time on this workload (MI355X): 10.6433 ms
    same = flop / 10.6433e-3 / 1e12
    assert bench.vs_baseline("pro-R8192-S196608-K1024", flop, same) == pytest.approx(1.0)
    assert bench.vs_baseline("pro-R8192-S196608-K1024", flop, same / 2) == pytest.approx(0.5)
    assert bench.vs_baseline("flash-R8192-S131072-K512", 1.7455e13,
                             1.7455e13 / 7.2235e-3 / 1e12) == pytest.approx(1.0)
    assert bench.vs_baseline("mid-R1024-4req-8k..64k-K512", 5.15e11, 1.0) is None
