"""The bench's multi-rank logic on CPU with world_size 2 over gloo: the timing
barrier, the max-over-ranks step time, the whole-job aggregate (weak scaling:
each rank runs its own copy of the workload, no data-path collective), and the
reference arm running on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    bench.barrier(True)
    step_ms = bench.max_over_ranks(local_ms, True, "cpu")
    value = bench.aggregate_value(1.0e12, step_ms, world)
    results[rank] = (step_ms, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        step_ms, value = results[r]
        assert step_ms == 15.0                      # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 1.0e12 / 15e-3 / 1e12)


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(steps=1, warmup=0, gpus=2, workload="single")
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_decode_step_appends_the_newest_tokens():
    import bench
    # sequences of 5, 3 and 4 keys with 1, 3 and 2 new query tokens
    rows = bench.newest_token_rows([0, 1, 4, 6], [0, 5, 8, 12])
    assert rows.tolist() == [4, 5, 6, 7, 10, 11]
    assert bench.newest_token_rows([0], [0]).size == 0
