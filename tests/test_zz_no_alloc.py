"""The allocation-free weight gradient (bsmm_updat_noalloc) against the ordinary one.

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

from _util import TOL_DW, cpu64, rand_layout, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", [(32, 1, "bf16", 24, 20, 0.5, 200),
                                                 (16, 0, "f16", 30, 28, 0.2, 136),
                                                 (8, 0, "bf16", 40, 36, 0.1, 96)])
def test_noalloc_matches_updat_twice(bs, fa, dtype, R, S, p, N):
    L = rand_layout(R, S, p, 31 + bs)
    m = bsmm.BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    for call, seed in enumerate((41, 43)):           # two calls in a row share the device array
        x = wk.normals(wk.act_shape(R * bs, N, fa), seed, 1.0, dtype).cuda()
        dy = wk.normals(wk.act_shape(S * bs, N, fa), seed + 1, 1.0, dtype).cuda()
        ref = m.updat(x, dy)
        got = torch.full(m.w_shape, float("nan"), dtype=torch.float32, device="cuda")
        bsmm.bsmm_updat_noalloc(m.handle, x, dy, got, N)
        m.sync_status()
        assert rel_fro(cpu64(got), cpu64(ref)) <= TOL_DW[dtype], call
        acc = got.clone()
        bsmm.bsmm_updat_noalloc(m.handle, x, dy, acc, N, accumulate=True)
        m.sync_status()
        assert rel_fro(cpu64(acc), 2 * cpu64(ref)) <= TOL_DW[dtype], call


def test_noalloc_rejects_fp32_and_bad_alignment():
    L = np.eye(3, dtype=np.uint8)
    m = bsmm.BlocksparseMatMul(L, block_size=32, feature_axis=1)
    x = torch.zeros((64, 96), dtype=torch.float32, device="cuda")
    dw = torch.zeros(m.w_shape, dtype=torch.float32, device="cuda")
    with pytest.raises(bsmm.BsmmError) as e:
        bsmm.bsmm_updat_noalloc(m.handle, x, x, dw, 64)
    assert e.value.code == bsmm.ERR_UNSUPPORTED
    xb = torch.zeros(64 * 96 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bsmm.BsmmError) as e:
        bsmm.bsmm_updat_noalloc(m.handle, xb[1:], xb[1:], dw, 64)
    assert e.value.code == bsmm.ERR_ALIGN
    m.sync_status()
