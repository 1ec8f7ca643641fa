"""Host logic of multi-process runs, on CPU with the gloo backend (world size 2).

The path shards by batch with no exchange between ranks ("replicas": each rank runs its own
batch on its own GPU), so the only cross-rank step is the timing: the job's throughput is every
rank's units over the slowest rank's time.  The oracle reference arm runs on rank 0 alone."""
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


def _rank_main(rank, world, port, local_ms, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    value, total_ms = bench.job_throughput(local_ms[rank], 32, 100, world, dist, "cpu")
    out.put((rank, value, total_ms))
    dist.barrier()
    dist.destroy_process_group()


def test_job_throughput_is_set_by_the_slowest_rank():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    local_ms = [10.0, 15.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, total_ms in got:
        assert total_ms == 15.0
        assert value == pytest.approx(32 * 100 * 2 / 15e-3)


def test_job_throughput_single_process():
    sys.path.insert(0, ROOT)
    import bench

    value, total_ms = bench.job_throughput(20.0, 8, 50, 1)
    assert total_ms == 20.0 and value == pytest.approx(8 * 50 / 20e-3)


def _bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _bench(["--impl", "reference", "--workload", "1", "--steps", "3", "--warmup", "3"],
                {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _bench(["--impl", "reference", "--workload", "1", "--steps", "3", "--warmup", "3"],
                {"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["gpu_launches"] == 0
    assert line["unit"] == "queries/s" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
