"""Host-side checks of bench.py: rank bookkeeping (gloo, world size 2) and the reference arm."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(backend="gloo")
    d.barrier()
    got = d.max(float(rank + 1) * 1.5)
    d.barrier()
    d.close()
    with open(os.path.join(out_dir, "r%d" % rank), "w") as f:
        f.write(repr(got))


def test_dist_max_over_ranks_gloo(tmp_path):
    world = 2
    port = 29500 + (os.getpid() % 2000)
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        assert float((tmp_path / ("r%d" % r)).read_text()) == 3.0


def test_single_process_dist_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.max(4.25) == 4.25
    d.barrier()
    d.close()


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
