"""Host logic of bench.py runs on more than one GPU, on CPU.

The library runs on one GPU: its decode attention kernel's clusters multicast their row
gathers within this GPU's memory, and nothing in the path exchanges data between GPUs.  So
bench.py refuses a multi-GPU run (torchrun with WORLD_SIZE > 1, or --gpus > 1): rank 0 prints
one line saying so, every rank exits 0, and none touches a GPU or starts a process group.  The
reference arm (the CPU oracle) still runs, on rank 0 alone."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    env.pop("STI_LIB", None)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


@pytest.mark.parametrize("rank", [0, 1])
def test_multi_gpu_run_is_refused_without_touching_a_gpu(rank):
    # CUDA_VISIBLE_DEVICES="" : were any rank to reach torch.cuda, it would fail
    r = _bench(["--steps", "3", "--warmup", "3"],
               {"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank), "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    if rank != 0:
        assert r.stdout.strip() == ""
        return
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 2 and "single-GPU" in line["unavailable"]


def test_gpus_flag_above_one_is_refused():
    r = _bench(["--gpus", "4", "--steps", "3", "--warmup", "3"], {"CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 4 and "unavailable" in line


def test_job_throughput_single_process():
    sys.path.insert(0, ROOT)
    import bench

    value, total_ms = bench.job_throughput(20.0, 8, 50)
    assert total_ms == 20.0 and value == pytest.approx(8 * 50 / 20e-3)


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


def test_step_roofline_sums_kernel_floors():
    """The headline roofline is the whole step: sum of each kernel's floor over the step time."""
    sys.path.insert(0, ROOT)
    import bench

    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0, "source": "test"}
    wk = {"a": {"bytes": 1e6, "flops": 0.0}, "b": {"bytes": 2e6, "flops": 1e9}}   # 1 us + max(2 us, 1 us)
    r = bench.step_roofline(["a", "b"], wk, 6e-6, pk, "none")
    assert r["bound"] == "hbm" and r["floor_us"] == pytest.approx(3.0)
    assert r["frac"] == pytest.approx(0.5) and r["achieved"] == pytest.approx(500.0)
    wk["c"] = {"bytes": 1e6, "flops": 8e9}                                             # 8 us on the tensor cores
    r = bench.step_roofline(["a", "b", "c"], wk, 22e-6, pk, "none")
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(0.5)
