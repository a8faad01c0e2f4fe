"""The benchmark's multi-rank path on the CPU: world size 2 over gloo.

N GPUs run N independent replicas (no data exchange). The collective work is a barrier on both sides of
the timed region and the maximum of the timings over the ranks; the whole-job rate counts every rank's
tokens. The reference arm runs on rank 0 only.
"""
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


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.rank_barrier(world)
    # rank r times (1 + r) s on the device and (5 - r) s end to end: the job takes the slowest of each
    got = bench.max_over_ranks([1.0 + rank, 5.0 - rank], world, device="cpu")
    bench.rank_barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(" ".join(repr(v) for v in got))
    torch.distributed.destroy_process_group()


def test_timings_are_the_maximum_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        vals = [float(x) for x in (tmp_path / f"rank{r}.txt").read_text().split()]
        assert vals == [2.0, 5.0]                  # device: max(1, 2); end to end: max(5, 4)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 4], 1) == [3.0, 4.0]
    bench.rank_barrier(1)


def test_whole_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(1, 32, 256, 0.64) == pytest.approx(12800.0)
    assert bench.whole_job_rate(8, 32, 256, 0.64) == pytest.approx(8 * 12800.0)   # weak scaling: per-rank work fixed


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
