"""Host logic of the multi-GPU bench (weak scaling) on CPU: two gloo ranks.

Each rank of `bench.py --gpus N` runs the step on its own share of the minibatch and all-reduces
the weight gradients (block_sparse_matrix_gb300.dp; tests/test_data_parallel.py checks the sum).
The job's step time is the slowest rank's, its value the sum of the ranks' work over that time;
the reference arm runs on rank 0 only.
"""
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


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_env() == (ws, rank, rank)
        dev_ms = 10.0 + 5.0 * rank                    # rank 1 is the slower replica
        t = bench.max_over_ranks(dev_ms, ws, torch.device("cpu"))
        v = bench.job_value(ws, 1e12, 100, t)
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_value():
    ws, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
    for r in range(ws):
        t, v = out[r]
        assert t == 15.0                              # every rank sees the slowest time
        assert v == pytest.approx(2 * 1e12 * 100 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_value(1, 2e12, 10, 20.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args) is None         # returns before any oracle work
    assert capsys.readouterr().out == ""
