"""The multi-process plumbing of bench.py on CPU: two gloo ranks, launched the
way torchrun would (RANK / WORLD_SIZE / MASTER_* in the environment), start
and stop the clock together, every rank learns the slowest rank's time, and
only rank 0 reports.  The reference arm does no work on ranks other than 0."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    r = bench.Replicas("gloo")
    assert (r.world, r.rank) == (world, rank)
    r.barrier()
    slowest = r.max(10.0 * (rank + 1))
    r.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{slowest} {int(r.reports)}\n")
    r.close()


def test_two_gloo_ranks_share_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    assert got == [["20.0", "1"], ["20.0", "0"]]


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    r = bench.Replicas("gloo")
    assert (r.world, r.rank, r.reports, r.dist) == (1, 0, True, None)
    r.barrier()
    assert r.max(3.5) == 3.5


def test_reference_arm_idles_on_other_ranks(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    import workloads as W

    args = argparse.Namespace(steps=3, warmup=1)
    bench.reference_arm(args, W.WORKLOADS["tiny_f32"])
    assert capsys.readouterr().out == ""
