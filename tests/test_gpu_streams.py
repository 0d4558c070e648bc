"""One handle driven from two CUDA streams at once: the schedules are read-only and built once,
scratch is kept per stream, so the passes of both streams, interleaved, give the same bits as
the same calls made one after another on one stream -- for every kernel family."""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import workloads as wk
from block_sparse_matrix_gb300.bsmm import BlocksparseMatMul

from _util import rand_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", [(32, 1, "bf16", 32, 32, 0.5, 1024), (32, 1, "bf16", 32, 32, 0.5, 64),
                                                 (32, 1, "bf16", 24, 24, 0.15, 128), (16, 0, "f16", 64, 64, 0.1, 512),
                                                 (8, 0, "bf16", 64, 64, 0.05, 256), (32, 1, "f32", 8, 8, 0.5, 64)])
def test_two_streams_share_one_handle(bs, fa, dtype, R, S, p, N):
    L = rand_layout(R, S, p, 3 + bs + N)
    L[0, 0] = 1
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    dt = wk.DTYPES[dtype]
    K = 3
    xs = [wk.normals(wk.act_shape(R * bs, N, fa), 10 + i, 1.0, dtype).cuda() for i in range(2 * K)]
    dys = [wk.normals(wk.act_shape(S * bs, N, fa), 20 + i, 1.0, dtype).cuda() for i in range(2 * K)]
    w = wk.normals(m.w_shape, 30, float(1 / np.sqrt(R * bs * p)), dtype).cuda()

    def run(i, stream):
        y = m.fprop(xs[i], w, stream=stream)
        dx = m.bprop(dys[i], w, stream=stream)
        dw = m.updat(xs[i], dys[i], stream=stream)
        return y, dx, dw

    torch.cuda.synchronize()
    serial = [run(i, None) for i in range(2 * K)]
    torch.cuda.synchronize()
    m.sync_status()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [None] * (2 * K)
    for i in range(K):                                   # interleaved enqueue on two streams
        with torch.cuda.stream(s1):
            outs[2 * i] = run(2 * i, s1)
        with torch.cuda.stream(s2):
            outs[2 * i + 1] = run(2 * i + 1, s2)
    torch.cuda.synchronize()
    m.sync_status()
    for a, b in zip(serial, outs):
        for u, v in zip(a, b):
            assert torch.equal(u, v)
    m.close()
