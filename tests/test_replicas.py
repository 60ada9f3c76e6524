"""The multi-GPU path of the benchmark is N independent replicas (nothing of the data path
crosses ranks).  Its host logic: a barrier on every rank around the timed region, the time
taken as the maximum over ranks, the job's figure counting every rank's work, and the
reference arm printing from rank 0 only.  Checked here as world-size-2 gloo runs on the CPU."""
import json
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
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.ranks_barrier(world, cuda=False)
        t = bench.ranks_max(1.5 + rank, world, "cpu")  # rank 1 is the slow one
        gbs = bench.job_gbs(10**9, 4, world, t)
        bench.ranks_barrier(world, cuda=False)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t": t, "gbs": gbs}, f)
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["t"] == 2.5  # the maximum over ranks, on every rank
        assert r["gbs"] == pytest.approx(10**9 * 4 * 2 / 2.5 / 1e9)  # both ranks' work / the slowest time


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.ranks_barrier(1, cuda=False)
    assert bench.ranks_max(3.25, 1, "cpu") == 3.25
    assert bench.job_gbs(2 * 10**9, 3, 1, 2.0) == pytest.approx(3.0)


def test_reference_arm_prints_from_rank_zero_only():
    """Launched as rank 1 of 2, the reference arm exits 0 without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1", MASTER_PORT="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--cpu-seconds", "0.1"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
