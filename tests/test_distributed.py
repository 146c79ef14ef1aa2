"""Host-side multi-rank logic of the benchmark, on CPU with the gloo backend.

With N GPUs every rank runs an independent replica of the emulated R-rank
workload (no data-path collective); the benchmark brackets the timed region
with barriers and reports the whole job against the slowest rank.  These
tests run that logic as two gloo ranks; the reference arm (the CPU oracle)
runs here too, rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(1.5 + rank)
        job = bench.whole_job(1000, 10, got, world)
        q.put((rank, got, job))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, got, job in res:
        assert got == 2.5  # the slowest rank's time, on every rank
        # two replicas of 1000 bytes / 10 tokens each in 2.5 ms
        assert job["gbs"] == pytest.approx(2 * 1000 / 2.5e-3 / 1e9)
        assert job["tokens_per_s"] == pytest.approx(2 * 10 / 2.5e-3)


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25) == 3.25


def _bench(*args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         env=env, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    return lines


def test_reference_arm_prints_one_line_on_cpu():
    lines = _bench("--impl", "reference", "--steps", "2", "--warmup", "1", "--reference-seconds", "2")
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    # the largest single-GPU workload by default, with the GPU arm's config block
    assert d["config"]["workload"].startswith("r32-e256-t2048-h7168")
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W

    args = bench.parse_args([])
    assert d["config"] == bench.config_block(W.WORKLOADS[bench.DEFAULT_WORKLOAD], args)


def test_reference_arm_nonzero_ranks_exit_quietly():
    lines = _bench("--impl", "reference", "--steps", "1", "--warmup", "0",
                   env_extra={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert lines == []
