"""The N > 1 path of bench.py: every rank runs an independent replica of the layer (the layer has
no cross-token exchange), the timings are reduced with a max over ranks, and the whole-job
throughput is N * T / max time. Checked with two gloo ranks on the CPU."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.0 + rank, 5.0 - rank]  # rank 0: (1, 5); rank 1: (2, 4)
    got = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, got, bench.replica_throughput(world, 4096, got[0])))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, thr in out:
        assert got == [2.0, 5.0]
        assert thr == pytest.approx(2 * 4096 / 2e-3)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.replica_throughput(1, 128, 0.5) == pytest.approx(256000.0)


def test_reference_arm_other_ranks_exit_without_output():
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_follows_the_bench_contract():
    """Rank 0 of the reference arm (the float64 oracle on the host cores) prints one JSON line
    with the keys the bench contract names, its e2e equal to its own value with no copies."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 1 and j["steps"] == 3
    assert j["warmup"] >= 3 and j["higher_is_better"] is True and j["scaling"] == "weak"
    assert j["unit"] == "tokens/s" and j["value"] > 0 and j["ms_per_step"] > 0
    assert j["config"]["workload"].startswith("tiny") and j["config"]["T"] == 128
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == j["value"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
