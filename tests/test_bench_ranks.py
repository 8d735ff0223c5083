"""The multi-rank plumbing of bench.py on the CPU: two gloo ranks (one
process per GPU on a GPU node; here the gloo backend stands in for NCCL).
Every rank runs the whole workload; only the barrier and the max of the
ranks' times cross ranks, and the reported value is the whole job's bytes
over the slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.rank_context()
    assert (w, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    barrier, max_over_ranks = bench.rank_ops(world, "cpu")
    barrier()
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    m = max_over_ranks(ms)
    value = bench.aggregate_gbs(1e9, 3, world, m)
    barrier()
    dist.destroy_process_group()
    out[rank] = (m, value)


def test_two_gloo_ranks_barrier_max_and_aggregate():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == 15.0  # both ranks see the slowest time
    # 2 ranks x 3 steps x 1 GB in 15 ms
    assert out[0][1] == pytest.approx(2 * 3 * 1e9 / 15e-3 / 1e9)
    assert out[0][1] == out[1][1]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup = 5, 3

    bench.run_reference(A())  # returns at once: no oracle work, no output
    assert capsys.readouterr().out == ""
