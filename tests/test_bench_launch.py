"""bench.py's launch contract on CPU: the reference arm (the fp64 oracle on
the host cores) under torchrun with two ranks prints exactly one JSON line,
from rank 0; the other rank exits 0 without work."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_two_ranks_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29533", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--workload", "tiny_4x256x512"]
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=300, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 3
    assert d["higher_is_better"] is False and d["unit"] == "ms" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_4x256x512"


def test_reference_arm_single_process():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3", "--warmup", "3",
           "--workload", "tiny_4x512x256"]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads(p.stdout.strip().splitlines()[-1])
    assert d["cpu_baseline"]["cores"] >= 1 and d["metric"].startswith("ms per NS call")


def test_cuda_arm_refuses_more_than_one_gpu():
    # The library is for 1-GPU processes (its multicast tensor maps cover the
    # calling GPU's own buffers): bench.py --impl ours stops before touching a
    # GPU, whether N comes from --gpus or from a launcher's WORLD_SIZE.
    script = os.path.join(ROOT, "bench.py")
    for extra, env in ((["--gpus", "2"], {}), ([], {"WORLD_SIZE": "2", "RANK": "1"})):
        p = subprocess.run([sys.executable, script, "--steps", "3", "--warmup", "3"] + extra,
                           stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=120, cwd=ROOT,
                           env=dict(os.environ, **env))
        assert p.returncode == 2, p.stderr
        assert "one GPU only" in p.stderr and p.stdout.strip() == ""
