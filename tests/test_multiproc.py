"""The bench's multi-process path on CPU: ranks are independent replicas
(no collective on the data path); the job's time is the slowest rank's,
taken by one all-reduce (max) over gloo here and NCCL on GPUs, and the
value counts every rank's verified positions.  The reference arm runs on
rank 0 alone."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 + 7.0 * rank          # rank 1 is the slower one
    total = bench.max_over_ranks(torch, local_ms, dist, "cpu")
    dist.barrier()
    value = bench.whole_job_value(10, world, total)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{total} {value}\n")
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo(tmp_path):
    world = 2
    port = _free_port()
    torch.multiprocessing.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                                join=True)
    import bench
    for r in range(world):
        total, value = map(float, (tmp_path / f"r{r}.txt").read_text().split())
        assert total == 107.0                   # every rank sees the slowest rank's time
        # 2 ranks x 10 steps x 96 positions in 107 ms
        assert value == pytest.approx(bench.B * bench.GAMMA * 10 * 2 / 0.107)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(torch, 12.5, None, "cpu") == 12.5
    assert bench.whole_job_value(200, 1, 1000.0) == pytest.approx(bench.B * bench.GAMMA * 200)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
