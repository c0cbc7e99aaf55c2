"""The multi-rank path of bench.py (replicas only: no collective on the layer's
path; the ranks only agree on the slowest rank's time).  Two gloo ranks on CPU."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, results):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(times[rank], world)
        results[rank] = (m, bench.job_tokens_per_s(1, 10, world, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    times = [120.0, 250.0]  # ms of work per rank
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        m, v = results[r]
        assert m == 250.0
        assert abs(v - 2 * 10 / 0.25) < 1e-9  # 20 tokens over the slowest 0.25 s


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(8, 5, 1, 1000.0) == 40.0


def test_reference_arm_json_contract():
    """`bench.py --impl reference` (the oracle on host cores) prints one JSON
    line with the keys the driver reads."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny"
    # config names the workload only: the same dictionary the GPU arm prints
    # (run details such as the number of token batches sit beside it)
    import bench

    assert d["config"] == bench.workload_config(bench.synth.CONFIGS["tiny"])
    assert d["token_batches"] == 3
