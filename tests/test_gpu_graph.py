"""The passes captured in a CUDA graph (tensor-core kernels, and the float32 SIMT kernels, which
also launch with programmatic dependent launch): a recurrent-style layer -- per-step fprop and
bprop and the grouped weight gradient of the steps -- is warmed up on one stream (the handle
builds its schedules and per-stream scratch there), captured on that stream, replayed twice,
and must equal eager execution bit for bit; the eager results match the float64 oracle."""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import workloads as wk
from block_sparse_matrix_gb300.bsmm import BlocksparseMatMul
from oracle import oracle as o

from _util import TOL_DW, cpu64, rand_layout, rel_fro

pytestmark = pytest.mark.gpu
TIGHT = {"f16": 2e-3, "bf16": 8e-3, "f32": 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _layer(m, w, xs, dys, ys, dxs, dw):
    for t in range(len(xs)):
        m.fprop(xs[t], w, ys[t])
        m.bprop(dys[t], w, dxs[t])
    m.updat_grouped(xs[: len(xs) // 2], dys[: len(xs) // 2], dw=dw)
    m.updat_grouped(xs[len(xs) // 2:], dys[len(xs) // 2:], dw=dw, accumulate=True)


@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", [(32, 1, "bf16", 24, 24, 0.2, 128), (32, 1, "bf16", 16, 16, 0.5, 64),
                                                 (32, 1, "bf16", 16, 16, 0.5, 256), (16, 0, "f16", 40, 36, 0.1, 256),
                                                 (8, 0, "bf16", 41, 37, 0.08, 136), (32, 1, "f32", 8, 8, 0.5, 64),
                                                 (16, 0, "f32", 12, 10, 0.4, 200)])
def test_layer_replays_in_a_cuda_graph(bs, fa, dtype, R, S, p, N):
    T = 4
    L = rand_layout(R, S, p, 60 + bs + N)
    np.fill_diagonal(L[:min(R, S), :min(R, S)], 1)
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    xs_h = [wk.normals(wk.act_shape(R * bs, N, fa), 70 + t, 1.0, dtype) for t in range(T)]
    dys_h = [wk.normals(wk.act_shape(S * bs, N, fa), 80 + t, 1.0, dtype) for t in range(T)]
    w_h = wk.normals(m.w_shape, 90, float(1 / np.sqrt(R * bs * p)), dtype)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xs = [a.cuda() for a in xs_h]
        dys = [a.cuda() for a in dys_h]
        w = w_h.cuda()
        ys = [torch.full(m.o_shape(N), float("nan"), dtype=wk.DTYPES[dtype], device="cuda") for _ in range(T)]
        dxs = [torch.full(m.i_shape(N), float("nan"), dtype=wk.DTYPES[dtype], device="cuda") for _ in range(T)]
        dw = torch.full(m.w_shape, float("nan"), device="cuda")
        _layer(m, w, xs, dys, ys, dxs, dw)                   # eager, and the warm-up of the stream
        eager = [a.clone() for a in ys + dxs + [dw]]
    s.synchronize()
    m.sync_status()
    for a in ys + dxs + [dw]:
        a.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _layer(m, w, xs, dys, ys, dxs, dw)
    for _ in range(2):
        for a in ys + dxs + [dw]:
            a.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ys + dxs + [dw], eager):
            assert torch.equal(a, b)
    m.sync_status()
    for t in range(T):
        assert rel_fro(cpu64(eager[t]), o.fprop(L, bs, xs_h[t], w_h, fa)) <= TIGHT[dtype]
        assert rel_fro(cpu64(eager[T + t]), o.bprop(L, bs, dys_h[t], w_h, fa)) <= TIGHT[dtype]
    assert rel_fro(cpu64(eager[2 * T]), o.updat_grouped(L, bs, xs_h, dys_h, fa)) <= TOL_DW[dtype]
    m.close()


def _bptt_layer(m, w, xs, dys, ys, dxs, dw, side, G):
    """fprops, then bprops in reverse step order; each group's weight gradient on `side` once the
    backward pass has reached the group's first step, the latest group first (writes dw), the
    others accumulating; `side` joined back at the end."""
    T = len(xs)
    cur = torch.cuda.current_stream()
    groups = list(range(0, T, G))[::-1]
    for t in range(T):
        m.fprop(xs[t], w, ys[t])
    for t in reversed(range(T)):
        m.bprop(dys[t], w, dxs[t])
        if t in groups:
            ev = torch.cuda.Event()
            ev.record(cur)
            side.wait_event(ev)
            with torch.cuda.stream(side):
                m.updat_grouped(xs[t:t + G], dys[t:t + G], dw=dw, accumulate=t != groups[0])
    ev = torch.cuda.Event()
    ev.record(side)
    cur.wait_event(ev)


@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", [(32, 1, "bf16", 24, 24, 0.2, 128), (16, 0, "f16", 40, 36, 0.1, 256),
                                                 (32, 1, "f32", 8, 8, 0.5, 64)])
def test_two_stream_layer_replays_in_a_cuda_graph(bs, fa, dtype, R, S, p, N):
    """The backpropagation-through-time layer with its weight-gradient groups forked to a second
    stream (as the recurrent benchmark runs it): captured across both streams, replayed twice, equal
    to eager execution bit for bit; the eager results match the float64 oracle."""
    T, G = 6, 2
    L = rand_layout(R, S, p, 160 + bs + N)
    np.fill_diagonal(L[:min(R, S), :min(R, S)], 1)
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    xs_h = [wk.normals(wk.act_shape(R * bs, N, fa), 170 + t, 1.0, dtype) for t in range(T)]
    dys_h = [wk.normals(wk.act_shape(S * bs, N, fa), 180 + t, 1.0, dtype) for t in range(T)]
    w_h = wk.normals(m.w_shape, 190, float(1 / np.sqrt(R * bs * p)), dtype)
    s, side = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s):
        xs = [a.cuda() for a in xs_h]
        dys = [a.cuda() for a in dys_h]
        w = w_h.cuda()
        ys = [torch.full(m.o_shape(N), float("nan"), dtype=wk.DTYPES[dtype], device="cuda") for _ in range(T)]
        dxs = [torch.full(m.i_shape(N), float("nan"), dtype=wk.DTYPES[dtype], device="cuda") for _ in range(T)]
        dw = torch.full(m.w_shape, float("nan"), device="cuda")
        _bptt_layer(m, w, xs, dys, ys, dxs, dw, side, G)    # eager, and the warm-up of both streams
        eager = [a.clone() for a in ys + dxs + [dw]]
    s.synchronize()
    m.sync_status()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _bptt_layer(m, w, xs, dys, ys, dxs, dw, side, G)
    for _ in range(2):
        for a in ys + dxs + [dw]:
            a.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ys + dxs + [dw], eager):
            assert torch.equal(a, b)
    m.sync_status()
    for t in range(T):
        assert rel_fro(cpu64(eager[t]), o.fprop(L, bs, xs_h[t], w_h, fa)) <= TIGHT[dtype]
        assert rel_fro(cpu64(eager[T + t]), o.bprop(L, bs, dys_h[t], w_h, fa)) <= TIGHT[dtype]
    assert rel_fro(cpu64(eager[2 * T]), o.updat_grouped(L, bs, xs_h, dys_h, fa)) <= TOL_DW[dtype]
    m.close()
