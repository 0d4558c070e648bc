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
