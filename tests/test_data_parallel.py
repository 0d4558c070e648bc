"""Data parallelism over the minibatch (block_sparse_matrix_gb300.dp) on CPU with two gloo ranks.

Each rank takes its shard of the minibatch and computes the shard's weight gradient through a
compute callback -- here the float64 oracle stands in for the library's GPU updat, in this test
only -- then the gradients are summed with one all-reduce.  The result must equal the oracle's
weight gradient of the whole minibatch, and the shards must cover every minibatch entry once.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_sparse_matrix_gb300 import dp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("N,world,align", [(200, 2, 1), (7, 3, 1), (136, 4, 8), (0, 2, 1), (3, 8, 1), (64, 3, 8)])
def test_shards_cover_the_minibatch_once(N, world, align):
    seen = np.zeros(N, np.int64)
    prev_hi = 0
    for r in range(world):
        lo, hi = dp.shard_bounds(N, r, world, align)
        assert lo == prev_hi and lo <= hi
        assert lo % align == 0 or lo == N
        seen[lo:hi] += 1
        prev_hi = hi
    assert prev_hi == N and np.all(seen == 1)


def test_shard_layouts():
    a = torch.arange(24.).reshape(4, 6)
    assert torch.equal(dp.shard(a, 1, 3, 1), a[1:3])                # (N, F): rows
    s = dp.shard(a, 2, 5, 0)                                          # (F, N): columns, contiguous
    assert torch.equal(s, a[:, 2:5]) and s.is_contiguous()


def _worker(rank, ws, port, fa, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    from block_sparse_matrix_gb300 import dp as dpm, workloads as wk
    from oracle import oracle as o
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        R, S, bs, N = 7, 6, 16, 104
        L = (np.random.default_rng(3).random((R, S)) < 0.5).astype(np.uint8)
        x = wk.normals(wk.act_shape(R * bs, N, fa), 21, 1.0, "bf16")     # every rank draws the same minibatch
        dy = wk.normals(wk.act_shape(S * bs, N, fa), 22, 1.0, "bf16")
        lo, hi = dpm.shard_bounds(N, rank, ws, 8)
        xs, dys = dpm.shard(x, lo, hi, fa), dpm.shard(dy, lo, hi, fa)

        def updat(a, b):                                                 # the oracle as compute callback
            return torch.from_numpy(o.updat(L, bs, a, b, fa))

        dw = dpm.data_parallel_updat(xs, dys, updat)
        out[rank] = (dw.numpy(), o.updat(L, bs, x, dy, fa), hi - lo)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fa", [1, 0])
def test_two_rank_gradient_equals_whole_minibatch(fa):
    ws, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(ws, port, fa, out), nprocs=ws, join=True)
    sizes = [out[r][2] for r in range(ws)]
    assert sum(sizes) == 104 and min(sizes) > 0
    for r in range(ws):
        got, ref, _ = out[r]
        # float64 sums of the same products in another order
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(out[0][0], out[1][0])                      # every rank holds the same sum
