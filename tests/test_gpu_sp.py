"""The sparse-window fprop/bprop kernel (k_tc_sp) against the
float64 oracle, through the C ABI: every block size and activation layout, pinned window sizes
and both split settings (one CTA per window, or two CTAs of a cluster summing their halves),
ragged minibatches, ragged layouts (odd block counts for block size 8, whose kernel works on
16 x 16 coarse blocks), empty block rows and columns; and against the window kernel."""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import workloads as wk
from block_sparse_matrix_gb300.bsmm import BlocksparseMatMul
from oracle import oracle as o

from _util import cpu64, rand_layout, rel_fro

pytestmark = pytest.mark.gpu

# relative Frobenius bound for one float32-accumulated sum rounded once to the output type
TIGHT = {"f16": 2e-3, "bf16": 8e-3}
DT = wk.DTYPES

CASES = [  # bs, feature_axis, dtype, R, S, density, N
    (16, 0, "f16", 40, 36, 0.10, 392),
    (16, 1, "bf16", 33, 29, 0.20, 200),
    (8, 0, "bf16", 41, 37, 0.08, 264),
    (8, 1, "f16", 30, 35, 0.15, 136),
    (32, 1, "bf16", 20, 22, 0.15, 520),
    (32, 0, "f16", 18, 21, 0.30, 136),
]


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _problem(bs, fa, dtype, R, S, p, N):
    L = rand_layout(R, S, p, 1000 + R * S + bs)
    L[:, 3] = 0                                          # an empty output block column
    L[2, :] = 0                                          # an empty input block row
    nnz = int(L.sum())
    x = wk.normals(wk.act_shape(R * bs, N, fa), 11 + R, 1.0, dtype)
    dy = wk.normals(wk.act_shape(S * bs, N, fa), 12 + S, 1.0, dtype)
    w = wk.normals((nnz, bs, bs), 13 + bs, float(1 / np.sqrt(R * bs * p)), dtype)
    return L, x, w, dy


def _run(L, bs, fa, dtype, x, w, dy, N):
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    y = torch.full(m.o_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
    dx = torch.full(m.i_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
    m.fprop(x.cuda(), w.cuda(), y)
    m.bprop(dy.cuda(), w.cuda(), dx)
    m.sync_status()
    m.close()
    return cpu64(y), cpu64(dx)


@pytest.mark.parametrize("W,split", [(None, None), (1, 1), (3, 2), (13, 1), (28, 2), (32, 1), (32, 2)])
@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", CASES)
def test_sp_matches_oracle(monkeypatch, W, split, bs, fa, dtype, R, S, p, N):
    monkeypatch.setenv("BSMM_TC_FB", "sp")
    if W:
        monkeypatch.setenv("BSMM_SP_W", str(W))
    if split:
        monkeypatch.setenv("BSMM_SP_SPLIT", str(split))
    L, x, w, dy = _problem(bs, fa, dtype, R, S, p, N)
    y, dx = _run(L, bs, fa, dtype, x, w, dy, N)
    assert rel_fro(y, o.fprop(L, bs, x, w, fa)) <= TIGHT[dtype]
    assert rel_fro(dx, o.bprop(L, bs, dy, w, fa)) <= TIGHT[dtype]


@pytest.mark.parametrize("bs,fa,dtype,R,S,p,N", CASES[:4])
def test_sp_split_and_window_kernel_agree(monkeypatch, bs, fa, dtype, R, S, p, N):
    """One CTA per window, two CTAs per window and the window kernel (activation operand read from
    shared memory) all accumulate in float32 and round once: they agree to output rounding."""
    L, x, w, dy = _problem(bs, fa, dtype, R, S, p, N)
    outs = {}
    for name, env in (("sp1", {"BSMM_TC_FB": "sp", "BSMM_SP_SPLIT": "1", "BSMM_SP_W": "8"}),
                      ("sp2", {"BSMM_TC_FB": "sp", "BSMM_SP_SPLIT": "2", "BSMM_SP_W": "8"}),
                      ("window", {"BSMM_TC_FB": "window"})):
        for k in ("BSMM_TC_FB", "BSMM_SP_SPLIT", "BSMM_SP_W"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        outs[name] = _run(L, bs, fa, dtype, x, w, dy, N)
    for other in ("sp2", "window"):
        for a, b in zip(outs["sp1"], outs[other]):
            assert rel_fro(a, b) <= TIGHT[dtype], other


@pytest.mark.parametrize("bs,fa,dtype", [(16, 0, "f16"), (8, 0, "bf16"), (32, 1, "bf16"), (8, 1, "bf16")])
@pytest.mark.parametrize("split", [1, 2])
def test_sp_integer_inputs_exact(monkeypatch, bs, fa, dtype, split):
    """Inputs in {-1, 0, 1}: every product and partial sum is a small integer, exact in float32 and
    in the 16-bit output, so the kernel equals the oracle bit for bit, with and without the split."""
    monkeypatch.setenv("BSMM_TC_FB", "sp")
    monkeypatch.setenv("BSMM_SP_SPLIT", str(split))
    monkeypatch.setenv("BSMM_SP_W", "4")
    R, S, N = 13, 11, 136
    L = rand_layout(R, S, 0.3, 77 + bs)
    nnz = int(L.sum())
    x = wk.small_ints(wk.act_shape(R * bs, N, fa), 5, dtype)
    dy = wk.small_ints(wk.act_shape(S * bs, N, fa), 6, dtype)
    w = wk.small_ints((nnz, bs, bs), 7, dtype)
    y, dx = _run(L, bs, fa, dtype, x, w, dy, N)
    assert np.array_equal(y, o.fprop(L, bs, x, w, fa))
    assert np.array_equal(dx, o.bprop(L, bs, dy, w, fa))


@pytest.mark.parametrize("bs,fa", [(16, 0), (8, 1), (32, 1)])
def test_sp_refuses_an_out_of_range_block_id(monkeypatch, bs, fa):
    """Fault injection on the host: a test hook makes the schedule name block nnz + 5.  The kernel
    checks every block id before its copy, zero-fills that block and records BSMM_ERR_BOUNDS; no
    memory past w is read, and the next call on a fresh schedule is correct again."""
    from block_sparse_matrix_gb300 import bsmm
    monkeypatch.setenv("BSMM_TC_FB", "sp")
    L, x, w, dy = _problem(bs, fa, "bf16", 12, 11, 0.4, 136)
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    monkeypatch.setenv("BSMM_SP_TEST_BAD_ID", "1")
    y = m.fprop(x.cuda(), w.cuda())
    with pytest.raises(bsmm.BsmmError) as e:
        m.sync_status()
    assert e.value.code == bsmm.ERR_BOUNDS
    assert torch.isfinite(y.float()).all()
    m.close()
    monkeypatch.delenv("BSMM_SP_TEST_BAD_ID")
    y2, _ = _run(L, bs, fa, "bf16", x, w, dy, 136)
    assert rel_fro(y2, o.fprop(L, bs, x, w, fa)) <= TIGHT["bf16"]
