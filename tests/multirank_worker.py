"""One rank of the world-size-2 replica test, launched by torch.distributed.run
on the CPU (gloo).  Exercises bench.py's multi-rank plumbing: process-group
setup from the launcher's environment, the timing barrier, the max over ranks,
whole-job accounting, per-rank input seeds, and the reference arm running on
rank 0 alone."""
import contextlib
import io
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
from workloads import WORKLOADS, make_layer  # noqa: E402


def main():
    world, rank, local = bench.dist_setup(None)
    assert world == 2 and dist.is_initialized() and dist.get_backend() == "gloo", (world, dist.get_backend())
    assert rank == int(os.environ["RANK"]) and local == int(os.environ["LOCAL_RANK"])

    # The slowest rank's time decides; the rate counts every rank's units.
    ms = bench.max_over_ranks(100.0 + 25.0 * rank, world)
    assert ms == 125.0, ms
    assert bench.whole_job_rate(12 * 10, world, ms) == 12 * 10 * 2 / 0.125

    # Replicas draw different inputs (bench seeds each rank with its rank).
    x = make_layer(L=64, M=4, seed=rank, layer=0, device="cpu")
    mine = torch.tensor([float(x.q.sum())], dtype=torch.float64)
    both = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(both, mine)
    assert both[0].item() != both[1].item()

    # The reference arm: rank 1 returns at once and prints nothing.
    if rank == 1:
        class A:
            layers, warmup, steps, workload = 0, 0, 1, "tiny_verify_f32"
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            r = bench.run_reference(A, WORKLOADS["tiny_verify_f32"], world, rank)
        assert r is None and out.getvalue() == "", out.getvalue()

    bench.barrier(world)
    dist.destroy_process_group()
    print(f"rank {rank} ok", flush=True)


if __name__ == "__main__":
    main()
