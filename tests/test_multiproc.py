"""bench.py under torchrun-style launches, on the CPU.

Every call of the library runs on one GPU, so the benchmark of our arm is single-GPU:
a launch with WORLD_SIZE > 1 (or --gpus > 1) prints one error line from rank 0 and
exits with status 2 before touching a device.  The reference arm (the fp64 oracle on
the host cores) prints one line from rank 0 and lets the other ranks exit without work.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(rank, world, *extra):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *extra], env=env,
                          capture_output=True, text=True, timeout=600, cwd=ROOT)


def test_our_arm_refuses_more_than_one_gpu():
    for rank in (0, 1):
        r = _run(rank, 2, "--steps", "1", "--warmup", "3")
        assert r.returncode == 2, r.stderr[-2000:]
        if rank == 0:
            line = json.loads(r.stdout.strip())
            assert "single-GPU" in line["error"] and line["n_gpus"] == 2
        else:
            assert r.stdout.strip() == ""
    r = _run(0, 1, "--gpus", "4", "--steps", "1")
    assert r.returncode == 2 and json.loads(r.stdout.strip())["n_gpus"] == 4


def test_reference_arm_world2_prints_once():
    """Under torchrun-style env vars the oracle arm runs on rank 0 only."""
    outs = []
    for rank in (0, 1):
        r = _run(rank, 2, "--impl", "reference", "--steps", "1", "--warmup", "3")
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip())
    assert outs[1] == ""
    line = json.loads(outs[0])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
