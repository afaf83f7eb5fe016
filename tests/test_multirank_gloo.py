"""The multi-rank (N > 1) host logic of bench.py, as two gloo ranks on CPU.

The path shards with no exchange step: each rank casts its own batch (its
own seed), the job's time is the slowest rank's (MAX over the process
group) and the whole-job rate counts every rank's bytes over that time;
under the reference arm only rank 0 works and prints.  No GPU is involved.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synthetic
    local = [1.5, 2.0, 0.5][rank]
    t = bench.slowest_rank_seconds(local, world, "cpu")
    rate = bench.job_gbs(1e9, world, t)
    gate, _, _ = synthetic.large(M=64, N=64, device="cpu",
                                 seed=synthetic.SEEDS["large_131072x8192"] + rank)
    # the reference arm: ranks other than 0 return at once, printing nothing
    class A:
        warmup, steps, ref_blocks = 0, 1, 1
    quiet = None
    if rank != 0:
        quiet = bench.run_reference(A(), world, rank)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"t": t, "rate": rate, "sum": float(gate.float().sum()), "quiet": quiet}, f)


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_take_the_slowest_time_and_count_every_rank(world, tmp_path, capfd):
    mp.start_processes(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    slowest = max([1.5, 2.0, 0.5][:world])
    for r in res:
        assert r["t"] == slowest
        assert r["rate"] == pytest.approx(1e9 * world / slowest / 1e9)
    # independent shards: every rank drew its own batch
    assert len({r["sum"] for r in res}) == world
    assert all(r["quiet"] == 0 for r in res[1:])
    assert "impl" not in capfd.readouterr().out
