"""Host-side checks of bench.py: the one-GPU guard, the reference arm, peaks and digest."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_multi_gpu_launch_prints_unavailable_and_does_no_work():
    """The library is one-GPU only: --gpus 2 prints one 'unavailable' line without
    touching a GPU or loading the library."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert "unavailable" in line and line["n_gpus"] == 2


def test_torchrun_ranks_of_the_gemm_arm_exit_without_work():
    for rank, want_line in (("0", True), ("1", False)):
        env = dict(os.environ, RANK=rank, WORLD_SIZE="2", LOCAL_RANK=rank)
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                            "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                           timeout=300, cwd=ROOT, env=env)
        assert r.returncode == 0, r.stderr
        assert bool(r.stdout.strip()) == want_line


def test_bench_has_no_collective_or_process_group():
    text = open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read()
    for word in ("init_process_group", "nccl", "all_reduce", "torch.distributed"):
        assert word not in text, word


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "4", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_peaks_and_digest():
    sys.path.insert(0, ROOT)
    import bench
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 100
    assert len(bench.source_digest()) == 16
