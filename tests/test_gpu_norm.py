"""GPU parity of layer_norm (README "blocksparse.norms") against the float64 oracle, through
the C ABI, for both activation layouts (axis = the matmul's feature_axis)."""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import bsmm, workloads as wk
from oracle import oracle as o

from _util import cpu64, rel_fro

pytestmark = pytest.mark.gpu
DT = wk.DTYPES
# one float32 normalisation rounded once to the output type (RMS rounding of bf16 ~1e-3)
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(N, C, axis, dtype, seed):
    shape = (N, C) if axis == 1 else (C, N)
    x = wk.normals(shape, seed, 1.0, dtype) * 2.0 + 0.75
    x = x.to(DT[dtype])
    rng = np.random.default_rng(seed + 1)
    g = torch.from_numpy(rng.standard_normal(C).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal(C).astype(np.float32))
    return x, g, b


@pytest.mark.parametrize("axis", [1, 0])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("relu", [False, True])
@pytest.mark.parametrize("N,C", [(200, 4096), (72, 256), (136, 8192), (8, 4104), (1032, 24)])
def test_layer_norm_parity(axis, dtype, relu, N, C):
    x, g, b = _case(N, C, axis, dtype, 31 * N + C + axis)
    eps = 1e-6 if dtype != "f16" else 1e-5
    y = bsmm.layer_norm(x.cuda(), g.cuda(), b.cuda(), axis=axis, epsilon=eps, relu=relu)
    torch.cuda.synchronize()
    ref = o.layer_norm(x, g, b, axis=axis, epsilon=eps, relu=relu)
    assert rel_fro(cpu64(y), ref) <= TOL[dtype]


@pytest.mark.parametrize("rpc", ["1", "2", "4"])
@pytest.mark.parametrize("dtype,C", [("bf16", 4096), ("f32", 24), ("f16", 2056)])
def test_layer_norm_rows_per_cta(monkeypatch, rpc, dtype, C):
    """(N, C) rows normalised 1, 2 or 4 per CTA, with a minibatch that is not a multiple of 4."""
    monkeypatch.setenv("BSMM_LN_RPC", rpc)
    N = 1030
    x, g, b = _case(N, C, 1, dtype, 77 + C)
    y = bsmm.layer_norm(x.cuda(), g.cuda(), b.cuda(), relu=True)
    torch.cuda.synchronize()
    assert rel_fro(cpu64(y), o.layer_norm(x, g, b, relu=True)) <= TOL[dtype]


@pytest.mark.parametrize("axis", [1, 0])
def test_layer_norm_constant_samples_give_shift_exactly(axis):
    N, C = 64, 4096
    x = torch.full((N, C) if axis == 1 else (C, N), 0.5, dtype=torch.bfloat16)
    g = torch.linspace(-2, 2, C, dtype=torch.float32)
    b = torch.linspace(-1, 3, C, dtype=torch.float32)
    y = bsmm.layer_norm(x.cuda(), g.cuda(), b.cuda(), axis=axis, relu=True).cpu()
    want = torch.clamp(b, min=0).to(torch.bfloat16)
    want = want.expand(N, C) if axis == 1 else want[:, None].expand(C, N)
    assert torch.equal(y, want)


@pytest.mark.parametrize("axis", [1, 0])
def test_layer_norm_in_place_and_empty(axis):
    x, g, b = _case(96, 512, axis, "bf16", 5)
    xc = x.cuda()
    want = bsmm.layer_norm(xc, g.cuda(), b.cuda(), axis=axis)
    bsmm.layer_norm(xc, g.cuda(), b.cuda(), axis=axis, y=xc)
    torch.cuda.synchronize()
    assert torch.equal(xc, want)
    e = torch.empty((0, 512) if axis == 1 else (512, 0), dtype=torch.bfloat16, device="cuda")
    bsmm.layer_norm(e, g.cuda(), b.cuda(), axis=axis)


def test_layer_norm_limits():
    C = 16384
    x, g, b = _case(4, C, 1, "bf16", 9)
    y = bsmm.layer_norm(x.cuda(), g.cuda(), b.cuda())
    assert rel_fro(cpu64(y), o.layer_norm(x, g, b)) <= TOL["bf16"]
    x2 = torch.zeros((4, C + 8), dtype=torch.bfloat16, device="cuda")
    g2 = torch.zeros(C + 8, device="cuda")
    with pytest.raises(bsmm.BsmmError):
        bsmm.layer_norm(x2, g2, g2)


# ---- gradient --------------------------------------------------------------------------------
# dx: one float32 evaluation rounded once to the input type; dg, db: float32 sums over samples
GTOL = {"f32": 2e-5, "f16": 2e-3, "bf16": 8e-3}
SUMTOL = 1e-4


def _grad_case(N, C, axis, dtype, seed, relu, eps):
    x, g, b = _case(N, C, axis, dtype, seed)
    dy = wk.normals(x.shape, seed + 7, 1.0, dtype)
    y = bsmm.layer_norm(x.cuda(), g.cuda(), b.cuda(), axis=axis, epsilon=eps, relu=relu) if relu else None
    return x, g, dy, y


@pytest.mark.parametrize("axis", [1, 0])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("relu", [False, True])
@pytest.mark.parametrize("N,C", [(200, 4096), (72, 256), (136, 8192), (8, 4104), (1304, 24), (400, 1000)])
def test_layer_norm_grad_parity(axis, dtype, relu, N, C):
    eps = 1e-6 if dtype != "f16" else 1e-5
    x, g, dy, y = _grad_case(N, C, axis, dtype, 17 * N + C + axis, relu, eps)
    dx = torch.full(x.shape, float("nan"), dtype=DT[dtype], device="cuda")
    dx, dg, db = bsmm.layer_norm_grad(x.cuda(), g.cuda(), dy.cuda(), y=y, axis=axis, epsilon=eps, relu=relu,
                                      dx=dx)
    torch.cuda.synchronize()
    rdx, rdg, rdb = o.layer_norm_grad(x, g, dy, y=cpu64(y) if relu else None, axis=axis, epsilon=eps, relu=relu)
    assert rel_fro(cpu64(dx), rdx) <= GTOL[dtype]
    assert rel_fro(cpu64(dg), rdg) <= SUMTOL
    assert rel_fro(cpu64(db), rdb) <= SUMTOL


@pytest.mark.parametrize("form", ["fused", "split"])
@pytest.mark.parametrize("dtype,N,C", [("bf16", 1030, 4096), ("f32", 7, 1000), ("f16", 5000, 64)])
def test_layer_norm_grad_rows_forms(monkeypatch, form, dtype, N, C):
    """(N, C) gradient in one pass (rows in chunks, partials in registers) and in the three-kernel
    form (dx, then chunked column sums), including chunks of more than 8 samples (N > 4096)."""
    if form == "split":
        monkeypatch.setenv("BSMM_LNG_SPLIT", "1")
    x, g, dy, y = _grad_case(N, C, 1, dtype, 91 + N, True, 1e-5)
    dx, dg, db = bsmm.layer_norm_grad(x.cuda(), g.cuda(), dy.cuda(), y=y, relu=True, epsilon=1e-5)
    torch.cuda.synchronize()
    rdx, rdg, rdb = o.layer_norm_grad(x, g, dy, y=cpu64(y), relu=True, epsilon=1e-5)
    assert rel_fro(cpu64(dx), rdx) <= GTOL[dtype]
    assert rel_fro(cpu64(dg), rdg) <= SUMTOL
    assert rel_fro(cpu64(db), rdb) <= SUMTOL


@pytest.mark.parametrize("axis", [1, 0])
def test_layer_norm_grad_large(axis):
    """The largest supported rows (C = 16384 for axis 1, with more samples than chunks of 8; a
    (C, N) slice that no longer fits shared memory for axis 0)."""
    N, C = (4100, 16384) if axis == 1 else (64, 12288)
    x, g, dy, y = _grad_case(N, C, axis, "bf16", 3 + axis, True, 1e-6)
    dx, dg, db = bsmm.layer_norm_grad(x.cuda(), g.cuda(), dy.cuda(), y=y, axis=axis, relu=True)
    torch.cuda.synchronize()
    rdx, rdg, rdb = o.layer_norm_grad(x, g, dy, y=cpu64(y), axis=axis, relu=True)
    assert rel_fro(cpu64(dx), rdx) <= GTOL["bf16"]
    assert rel_fro(cpu64(dg), rdg) <= SUMTOL
    assert rel_fro(cpu64(db), rdb) <= SUMTOL


@pytest.mark.parametrize("axis", [1, 0])
def test_layer_norm_grad_small_integers_exact_db(axis):
    """Constant g = 1, dy in {-1, 0, 1} and x whose samples have mean 0 and variance 1 exactly:
    db is a sum of small integers, exact in float32 in any order."""
    N, C = 96, 64
    rng = np.random.default_rng(5)
    base = np.tile(np.array([-1.0, 1.0]), C // 2)              # mean 0, biased variance 1
    xs = np.stack([rng.permutation(base) for _ in range(N)])    # (N, C)
    x = torch.from_numpy(xs.astype(np.float32)).to(torch.bfloat16)
    dy = wk.small_ints((N, C), 6, "bf16")
    if axis == 0:
        x, dy = x.T.contiguous(), dy.T.contiguous()
    g = torch.ones(C)
    dx, dg, db = bsmm.layer_norm_grad(x.cuda(), g.cuda(), dy.cuda(), axis=axis, epsilon=0.0)
    rdx, rdg, rdb = o.layer_norm_grad(x, g, dy, axis=axis, epsilon=0.0)
    assert np.array_equal(cpu64(db), rdb)
    assert rel_fro(cpu64(dg), rdg) <= 1e-6
    assert rel_fro(cpu64(dx), rdx) <= GTOL["bf16"]


@pytest.mark.parametrize("axis", [1, 0])
def test_layer_norm_grad_empty_minibatch(axis):
    C = 256
    x = torch.empty((0, C) if axis == 1 else (C, 0), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(C, device="cuda")
    dx, dg, db = bsmm.layer_norm_grad(x, g, torch.empty_like(x), axis=axis)
    torch.cuda.synchronize()
    assert dx.numel() == 0 and torch.equal(dg, torch.zeros(C, device="cuda")) and torch.equal(db, dg)


def test_layer_norm_grad_refuses_dx_over_an_input():
    x, g, dy, _ = _grad_case(16, 256, 1, "bf16", 8, False, 1e-6)
    xc, dyc = x.cuda(), dy.cuda()
    with pytest.raises(ValueError):
        bsmm.layer_norm_grad(xc, g.cuda(), dyc, dx=dyc)
