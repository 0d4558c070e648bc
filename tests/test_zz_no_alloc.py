"""The allocation-free weight gradient (bsmm_updat_noalloc) against the float64 oracle and
against the ordinary weight gradient (bsmm_updat).

It exists for callers that must not allocate device memory, e.g. code running under a
framework's memory budget or caching allocator, or a latency-critical loop: it computes
with a fixed device array instead of tables the handle allocates.  This file is collected
last so that a failure here cannot stop the other GPU tests.  Each test passes on its own
in a fresh process and after all other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import bsmm, workloads as wk
from oracle import oracle as o

from _util import TOL_DW, cpu64, rand_layout, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(R, S, bs, N, fa, dtype, seed):
    x = wk.normals(wk.act_shape(R * bs, N, fa), seed, 1.0, dtype)
    dy = wk.normals(wk.act_shape(S * bs, N, fa), seed + 1, 1.0, dtype)
    return x, dy


@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", [(32, 1, "bf16", 24, 20, 0.5, 200),
                                                 (16, 0, "f16", 30, 28, 0.2, 136),
                                                 (8, 0, "bf16", 40, 36, 0.1, 96)])
def test_noalloc_matches_oracle_twice(bs, fa, dtype, R, S, p, N):
    L = rand_layout(R, S, p, 31 + bs)
    m = bsmm.BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    for call, seed in enumerate((41, 43)):           # two calls in a row share the device array
        x, dy = _inputs(R, S, bs, N, fa, dtype, seed)
        ref = o.updat(L, bs, x, dy, fa)
        xc, dyc = x.cuda(), dy.cuda()
        got = torch.full(m.w_shape, float("nan"), dtype=torch.float32, device="cuda")
        bsmm.bsmm_updat_noalloc(m.handle, xc, dyc, got, N)
        m.sync_status()
        assert rel_fro(cpu64(got), ref) <= TOL_DW[dtype], call
        # the ordinary entry point gives the same gradient within the same tolerance
        assert rel_fro(cpu64(got), cpu64(m.updat(xc, dyc))) <= TOL_DW[dtype], call
        acc = got.clone()
        m.updat_noalloc(xc, dyc, dw=acc, accumulate=True)
        m.sync_status()
        assert rel_fro(cpu64(acc), 2 * ref) <= TOL_DW[dtype], call


def test_noalloc_alternating_handles():
    """A larger table followed by a smaller one in the shared array, and back: each call
    rewrites what it uses, so no stale entries of the other handle are read."""
    big = (rand_layout(48, 40, 0.6, 5), 32, 1, "bf16", 136)
    small = (rand_layout(6, 5, 0.5, 6), 32, 1, "bf16", 72)
    cases = []
    for L, bs, fa, dtype, N in (big, small):
        m = bsmm.BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
        x, dy = _inputs(L.shape[0], L.shape[1], bs, N, fa, dtype, 300 + L.shape[0])
        cases.append((m, L, bs, fa, x, dy, o.updat(L, bs, x, dy, fa), N))
    for m, L, bs, fa, x, dy, ref, N in cases + cases:
        got = torch.full(m.w_shape, float("nan"), dtype=torch.float32, device="cuda")
        bsmm.bsmm_updat_noalloc(m.handle, x.cuda(), dy.cuda(), got, N)
        m.sync_status()
        assert rel_fro(cpu64(got), ref) <= TOL_DW["bf16"]


def test_noalloc_rejects_oversized_layout_on_host():
    """A layout whose tables need more than the fixed array (102,400 blocks of 32 x 32) is
    refused before anything is copied or launched."""
    L = np.ones((320, 320), np.uint8)
    m = bsmm.BlocksparseMatMul(L, block_size=32, feature_axis=1)
    buf = torch.zeros(64, dtype=torch.bfloat16, device="cuda")    # never touched: refused first
    dw = torch.zeros(64, dtype=torch.float32, device="cuda")
    n0 = bsmm.launch_count()
    code = bsmm.lib().bsmm_updat_noalloc(m.handle, ctypes.c_void_p(buf.data_ptr()), ctypes.c_void_p(buf.data_ptr()),
                                         ctypes.c_void_p(dw.data_ptr()), 64, bsmm.BF16, 0,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == bsmm.ERR_UNSUPPORTED
    assert bsmm.launch_count() == n0
    m.sync_status()


def test_noalloc_refuses_a_capturing_stream():
    """Called while its stream captures a graph it returns UNSUPPORTED without enqueuing
    anything, and the capture stays valid."""
    L = rand_layout(6, 6, 0.5, 7)
    m = bsmm.BlocksparseMatMul(L, block_size=32, feature_axis=1)
    x, dy = _inputs(6, 6, 32, 64, 1, "bf16", 77)
    xc, dyc = x.cuda(), dy.cuda()
    dw = torch.zeros(m.w_shape, dtype=torch.float32, device="cuda")
    y = torch.zeros(16, device="cuda")
    codes = []
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        codes.append(bsmm.lib().bsmm_updat_noalloc(m.handle, ctypes.c_void_p(xc.data_ptr()),
                                                   ctypes.c_void_p(dyc.data_ptr()), ctypes.c_void_p(dw.data_ptr()),
                                                   64, bsmm.BF16, 0, ctypes.c_void_p(s.cuda_stream)))
        y.add_(1.0)
    g.replay()
    torch.cuda.synchronize()
    assert codes == [bsmm.ERR_UNSUPPORTED]
    assert torch.equal(y, torch.ones_like(y))
    assert not torch.any(dw != 0)
    m.sync_status()


def test_noalloc_rejects_fp32_bad_alignment_and_wrong_dw():
    L = np.eye(3, dtype=np.uint8)
    m = bsmm.BlocksparseMatMul(L, block_size=32, feature_axis=1)
    x = torch.zeros((64, 96), dtype=torch.float32, device="cuda")
    dw = torch.zeros(m.w_shape, dtype=torch.float32, device="cuda")
    with pytest.raises(bsmm.BsmmError) as e:
        bsmm.bsmm_updat_noalloc(m.handle, x, x, dw, 64)
    assert e.value.code == bsmm.ERR_UNSUPPORTED
    xb = torch.zeros(64 * 96 + 8, dtype=torch.bfloat16, device="cuda")
    code = bsmm.lib().bsmm_updat_noalloc(m.handle, ctypes.c_void_p(xb[1:].data_ptr()),
                                         ctypes.c_void_p(xb[1:].data_ptr()), ctypes.c_void_p(dw.data_ptr()), 64,
                                         bsmm.BF16, 0, None)
    assert code == bsmm.ERR_ALIGN
    # the binding refuses a dw that is not float32 (nnz, bs, bs) before the C call
    xh = torch.zeros((64, 96), dtype=torch.bfloat16, device="cuda")
    n0 = bsmm.launch_count()
    with pytest.raises(ValueError):
        bsmm.bsmm_updat_noalloc(m.handle, xh, xh, torch.zeros(m.w_shape, dtype=torch.bfloat16, device="cuda"), 64)
    with pytest.raises(ValueError):
        bsmm.bsmm_updat_noalloc(m.handle, xh[:32], xh, dw, 64)
    assert bsmm.launch_count() == n0
    m.sync_status()
