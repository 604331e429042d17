"""bench.py under a multi-rank launch, on the CPU.

The library runs on one GPU per process and nothing launches it on more
than one GPU.  When bench.py is started with --gpus N > 1 (the driver runs
it under torchrun, one process per rank), no rank touches a GPU: rank 0
prints one JSON line that says the path is single-GPU and every rank exits
0.  The reference arm (the CPU oracle) runs on rank 0 only; other ranks
return at once."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(rank, world, *extra):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555", CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", str(world), "--steps", "3",
                           "--warmup", "3", *extra], env=env, capture_output=True, text=True, timeout=120)


def test_two_ranks_skip_without_touching_a_gpu():
    r0, r1 = _run(0, 2), _run(1, 2)
    assert r0.returncode == 0, r0.stderr
    assert r1.returncode == 0, r1.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["value"] is None
    assert "single-GPU" in line["skipped"]
    assert r1.stdout.strip() == ""
    # no rank imported torch's CUDA runtime or the library
    assert "libmq" not in r0.stderr + r1.stderr


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run(1, 2, "--impl", "reference")
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
