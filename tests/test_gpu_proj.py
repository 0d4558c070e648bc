"""GPU parity of SparseProj (README "API Documentation: blocksparse.matmul", class SparseProj)
against the float64 oracle, through the C ABI.  Copies are exact, and each sum or product of two
inputs is formed in float32 and rounded once; for bf16 / fp16 / fp32 inputs that equals the exact
result rounded once to the type, so every comparison is bit-exact."""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import bsmm, workloads as wk
from oracle import oracle as o

pytestmark = pytest.mark.gpu
DT = wk.DTYPES


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


MAPS = {   # name: (nhidden, SparseProj keyword arguments)
    "random": (4096, lambda: {"gather_lut": np.random.default_rng(1).permutation(4096)[:1000]}),
    "default": (4096, lambda: {"nproj": 2048, "proj_stride": 64, "block_size": 32}),
    "permutation": (520, lambda: {"gather_lut": np.random.default_rng(2).permutation(520)}),
    "single": (72, lambda: {"gather_lut": [71]}),
    "mixed": (4096, lambda: {"gather_lut": _mixed_lut()}),
}


def _mixed_lut():
    """Runs of 32 every 64 features, with a swapped pair and one reversed run: some 16-byte groups
    of the map are aligned runs and some are not."""
    lut = o.proj_default_lut(2048, 64, 32)
    lut[[5, 6]] = lut[[6, 5]]
    lut[64:96] = lut[64:96][::-1].copy()
    return lut


def _exact(ref, dtype):
    """The float64 oracle result rounded once to dtype."""
    return torch.from_numpy(ref).to(DT[dtype])


def _arr(shape, seed, dtype):
    return wk.normals(shape, seed, 1.0, dtype)


@pytest.mark.parametrize("name", list(MAPS))
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("axis", [1, 0])
@pytest.mark.parametrize("N", [8, 1032])
def test_sparse_proj_parity(name, dtype, axis, N):
    nhidden, kw = MAPS[name]
    sp = bsmm.SparseProj(nhidden, feature_axis=axis, **kw())
    lut = sp.lut
    shape = lambda F: (N, F) if axis == 1 else (F, N)
    x = _arr(shape(nhidden), 10 + N, dtype)
    z = _arr(shape(nhidden), 11 + N, dtype)
    s = _arr(shape(sp.nproj), 12 + N, dtype)
    xd, zd, sd = x.cuda(), z.cuda(), s.cuda()
    checks = [
        (sp.gather(xd), o.sparse_proj("gather", lut, x, axis=axis)),
        (sp.scatter(sd), o.sparse_proj("scatter", lut, s, nhidden=nhidden, axis=axis)),
        (sp.scatter_add(xd, sd), o.sparse_proj("scatter_add", lut, x, s, axis=axis)),
        (sp.scatter_mul(xd, sd), o.sparse_proj("scatter_mul", lut, x, s, axis=axis)),
        (sp.gather_mul(xd, zd), o.sparse_proj("gather_mul", lut, x, z, axis=axis)),
    ]
    torch.cuda.synchronize()
    for got, ref in checks:
        assert torch.equal(got.cpu(), _exact(ref, dtype))
    # in place: only the mapped features change
    xi = xd.clone()
    sp.scatter_add(xi, sd, out=xi)
    assert torch.equal(xi.cpu(), _exact(o.sparse_proj("scatter_add", lut, x, s, axis=axis), dtype))
    xi = xd.clone()
    sp.scatter_mul(xi, sd, out=xi)
    assert torch.equal(xi.cpu(), _exact(o.sparse_proj("scatter_mul", lut, x, s, axis=axis), dtype))
    sp.close()


@pytest.mark.parametrize("axis", [1, 0])
def test_sparse_proj_ragged_and_empty(axis):
    """N not a multiple of anything for (N, F); N = 0 is a no-op; the default map's shape."""
    sp = bsmm.SparseProj(300, proj_stride=40, block_size=16, feature_axis=axis)
    assert sp.nproj == 16 * ((300 - 16) // 40 + 1)
    assert sp.lut.tolist() == o.proj_default_lut(sp.nproj, 40, 16).tolist()
    N = 37 if axis == 1 else 40
    shape = lambda F: (N, F) if axis == 1 else (F, N)
    x = _arr(shape(300), 3, "bf16")
    got = sp.gather(x.cuda()).cpu()
    assert torch.equal(got, _exact(o.sparse_proj("gather", sp.lut, x, axis=axis), "bf16"))
    e = torch.empty((0, 300) if axis == 1 else (300, 0), dtype=torch.bfloat16, device="cuda")
    assert sp.gather(e).numel() == 0
    sp.close()


def test_sparse_proj_gradients_are_adjoint():
    """gather_grad = scatter and scatter_grad = gather, so <gather(x), dy> = <x, gather_grad(dy)>."""
    sp = bsmm.SparseProj(1024, gather_lut=np.random.default_rng(3).permutation(1024)[:333])
    x = torch.randn(64, 1024, device="cuda", dtype=torch.float64).float()
    dy = torch.randn(64, 333, device="cuda").float()
    lhs = (sp.gather(x).double() * dy.double()).sum()
    rhs = (x.double() * sp.gather_grad(dy).double()).sum()
    assert torch.allclose(lhs, rhs, rtol=1e-10)
    dx, dys = sp.scatter_mul_grad(dy.new_ones(64, 1024), x, sp.gather(x))
    assert torch.equal(dys, sp.gather(x))
    sp.close()


def test_sparse_proj_rejects_bad_calls():
    sp = bsmm.SparseProj(64, gather_lut=[3, 9])
    x = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bsmm.BsmmError):               # gather in place
        bsmm.bsmm_proj(sp._h, "gather", x, None, x, 8)
    with pytest.raises(bsmm.BsmmError):               # (F, N) with N * 2 bytes not a multiple of 16
        bsmm.bsmm_proj(sp._h, "gather", torch.zeros(64, 12, dtype=torch.bfloat16, device="cuda"), None,
                       torch.zeros(2, 12, dtype=torch.bfloat16, device="cuda"), 12, axis=0)
    sp.close()
