"""The bench's multi-GPU bookkeeping on CPU: two gloo ranks, as torchrun would
start them, agree on the slowest rank's time and on the whole-job throughput,
and the reference arm runs on rank 0 only."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_setup(world)
    own_ms = 100.0 + 50.0 * r               # rank 1 is the slow one
    bench.barrier(w)
    slowest = bench.max_over_ranks(own_ms, w)
    value = bench.throughput(w, 32, 10, slowest)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "slowest": slowest, "value": value,
                   "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_agree_on_slowest_time_and_throughput(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world
        assert d["backend"] == "gloo"
        assert d["slowest"] == 150.0                       # max over ranks, on every rank
        assert d["value"] == pytest.approx(2 * 32 * 10 / 0.150)   # all ranks' tokens / slowest time


def _ref_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(world), "--config", "tiny",
                "--cpu-sample-tokens", "2"]
    out = os.path.join(out_dir, f"ref{rank}.txt")
    fd = os.open(out, os.O_WRONLY | os.O_CREAT | os.O_TRUNC)
    os.dup2(fd, 1)
    bench.main()
    sys.stdout.flush()


@pytest.mark.timeout(600)
def test_reference_arm_prints_on_rank0_only(tmp_path):
    sys.path.insert(0, ROOT)
    import oracle
    oracle.build()
    world = 2
    mp.start_processes(_ref_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    lines0 = [l for l in open(tmp_path / "ref0.txt").read().splitlines() if l.startswith("{")]
    lines1 = [l for l in open(tmp_path / "ref1.txt").read().splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
