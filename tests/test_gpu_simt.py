"""The IEEE float32 SIMT kernels (the float32 path, and the second implementation of the 16-bit
passes) against the float64 oracle, through the C ABI.

The fprop/bprop kernel stages its LUT entries in groups (4 entries, or 3 for 64-row tiles at
block size 32), so the layout gives block columns and rows every length from 0 to 9 entries:
empty, one partial group, exactly one group, a group plus one, and several groups.  Both tile
heights run: a minibatch small enough that a CTA takes 256 / bs rows, and 64-row tiles with a
ragged last tile.  Integer inputs check the sums bit for bit; normal inputs at the float32 bound.
"""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import workloads as wk
from block_sparse_matrix_gb300.bsmm import BlocksparseMatMul
from oracle import oracle as o

from _util import cpu64, rel_fro

pytestmark = pytest.mark.gpu

TIGHT = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}
DT = wk.DTYPES


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def staircase(n=10):
    """L[i, k] = 1 for i < k: block column k has k entries, block row i has n - 1 - i."""
    return np.triu(np.ones((n, n), np.uint8), 1)


def _run(L, bs, fa, dtype, x, w, dy, N):
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    m.set_kernel("simt")
    y = torch.full(m.o_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
    dx = torch.full(m.i_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
    m.fprop(x.cuda(), w.cuda(), y)
    m.bprop(dy.cuda(), w.cuda(), dx)
    dw = m.updat(x.cuda(), dy.cuda())
    m.sync_status()
    m.close()
    return cpu64(y), cpu64(dx), cpu64(dw)


# N = 40: 10 block columns x 1 tile of 64 < the SM count, so each CTA takes 256 / bs rows.
# N = 1000: 10 x 16 tiles >= the SM count, so 64-row tiles; 1000 = 15 x 64 + 40 leaves a ragged tile.
@pytest.mark.parametrize("N", [40, 1000])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("fa", [0, 1])
def test_simt_group_boundaries_integer_exact(N, bs, fa):
    L = staircase()
    nnz = int(L.sum())
    x = wk.small_ints(wk.act_shape(10 * bs, N, fa), 31 + bs, "f32")
    dy = wk.small_ints(wk.act_shape(10 * bs, N, fa), 32 + bs, "f32")
    w = wk.small_ints((nnz, bs, bs), 33 + bs, "f32")
    y, dx, dw = _run(L, bs, fa, "f32", x, w, dy, N)
    assert np.array_equal(y, o.fprop(L, bs, x, w, fa))
    assert np.array_equal(dx, o.bprop(L, bs, dy, w, fa))
    assert np.array_equal(dw, o.updat(L, bs, x, dy, fa))


@pytest.mark.parametrize("N", [40, 1000])
@pytest.mark.parametrize("bs,fa,dtype", [(32, 1, "f32"), (32, 0, "f32"), (16, 0, "f32"), (8, 1, "f32"),
                                         (32, 1, "bf16"), (16, 0, "f16")])
def test_simt_group_boundaries_normal(N, bs, fa, dtype):
    L = staircase()
    nnz = int(L.sum())
    x = wk.normals(wk.act_shape(10 * bs, N, fa), 41 + bs, 1.0, dtype)
    dy = wk.normals(wk.act_shape(10 * bs, N, fa), 42 + bs, 1.0, dtype)
    w = wk.normals((nnz, bs, bs), 43 + bs, float(1 / np.sqrt(5 * bs)), dtype)
    y, dx, dw = _run(L, bs, fa, dtype, x, w, dy, N)
    assert rel_fro(y, o.fprop(L, bs, x, w, fa)) <= TIGHT[dtype]
    assert rel_fro(dx, o.bprop(L, bs, dy, w, fa)) <= TIGHT[dtype]
    assert rel_fro(dw, o.updat(L, bs, x, dy, fa)) <= 1e-5
