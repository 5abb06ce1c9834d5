"""World-size-2 tests of the replica (weak-scaling) path on the CPU with gloo.

The layer step needs no collective: layers and sequences are independent,
so N GPUs run N replicas and the only cross-rank traffic is the timing
barrier and the max over ranks.  These tests launch two ranks with
torch.distributed.run exactly as a multi-GPU bench run is launched."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=300):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}"] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_replica_plumbing_two_ranks():
    r = _torchrun([os.path.join(ROOT, "tests", "multirank_worker.py")])
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "rank 0 ok" in r.stdout and "rank 1 ok" in r.stdout


def test_reference_arm_two_ranks_prints_one_line():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--workload", "tiny_verify_f32",
                   "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
