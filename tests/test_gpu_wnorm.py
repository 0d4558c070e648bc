"""GPU parity of l2_normalize (weight normalisation, README "API Documentation:
blocksparse.matmul") and of its gradient against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import bsmm, workloads as wk
from oracle import oracle as o

from _util import cpu64, rel_fro

pytestmark = pytest.mark.gpu
DT = wk.DTYPES
# float32 sums over a feature's vector, one rounding of y to the output type
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}
TOL_GRAD = 1e-5          # dw, dgain are float32 from exact inputs


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(R, S, bs, p, seed, scale=1.0, zero_col=None, kind="bernoulli"):
    L = wk.make_layout(R, S, kind, p, False, seed)
    if zero_col is not None:
        L[:, zero_col] = 0
    m = bsmm.BlocksparseMatMul(L, block_size=bs)
    w = wk.normals(m.w_shape, seed + 1, scale, "f32")
    rng = np.random.default_rng(seed + 2)
    gain = torch.from_numpy((rng.uniform(0.5, 2.0, S * bs) * np.where(rng.random(S * bs) < 0.2, -1, 1))
                            .astype(np.float32))
    return L, m, w, gain


SHAPES = [  # R, S, bs, density: several CTAs per cluster, ragged columns, long columns (the
    # last two exceed the persistent kernel's shared memory for float32 gradients / at bs 32 and
    # stream in the register kernel), more columns than resident clusters (1024 x 8)
    (8, 8, 32, 0.5), (128, 128, 32, 0.5), (40, 24, 16, 0.3), (512, 64, 8, 0.05), (16, 1024, 8, 0.2),
    (1, 5, 16, 1.0), (256, 3, 32, 1.0), (2048, 2, 8, 1.0),
]


# "auto": the library's choice; "registers": the one-pass register kernel everywhere;
# "persistent": the persistent shared-memory kernel wherever a column share fits (the register
# kernel beyond).
FORMS = ["auto", "registers", "persistent"]


@pytest.fixture(params=FORMS)
def form(request, monkeypatch):
    if request.param == "auto":
        monkeypatch.delenv("BSMM_WN_KERNEL", raising=False)
    else:
        monkeypatch.setenv("BSMM_WN_KERNEL", request.param)
    return request.param


@pytest.mark.parametrize("R,S,bs,p", SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("with_gain", [False, True])
def test_l2_normalize_parity(R, S, bs, p, dtype, with_gain, form):
    L, m, w, gain = _case(R, S, bs, p, 7 * R + S + bs, zero_col=S // 2 if S > 2 else None)
    g = gain if with_gain else None
    y = m.l2_normalize(w.cuda(), None if g is None else g.cuda(), dtype=DT[dtype])
    torch.cuda.synchronize()
    ref = o.l2_normalize(L, bs, w, g)
    assert rel_fro(cpu64(y), ref) <= TOL[dtype]
    m.close()


@pytest.mark.parametrize("R,S,bs,p", SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_gain", [False, True])
def test_l2_normalize_grad_parity(R, S, bs, p, dtype, with_gain, form):
    L, m, w, gain = _case(R, S, bs, p, 11 * R + S + bs, zero_col=S // 2 if S > 2 else None)
    g = gain if with_gain else None
    dy = wk.normals(m.w_shape, 3 * R + 1, 1.0, dtype)
    dw, dgain = m.l2_normalize_grad(w.cuda(), dy.cuda(), None if g is None else g.cuda())
    torch.cuda.synchronize()
    rdw, rdg = o.l2_normalize_grad(L, bs, w, dy, g)
    assert rel_fro(cpu64(dw), rdw) <= TOL_GRAD
    assert rel_fro(cpu64(dgain), rdg) <= TOL_GRAD
    m.close()


@pytest.mark.parametrize("bs", [32, 8])
def test_l2_normalize_epsilon_branch(bs, form):
    """Features whose squared norm is below epsilon (tiny weights), forward and gradient."""
    L, m, w, gain = _case(16, 6, bs, 0.5, 5, scale=1e-4)
    eps = 1e-2
    dy = wk.normals(m.w_shape, 6, 1.0, "f32")
    y = m.l2_normalize(w.cuda(), gain.cuda(), epsilon=eps)
    dw, dgain = m.l2_normalize_grad(w.cuda(), dy.cuda(), gain.cuda(), epsilon=eps)
    torch.cuda.synchronize()
    assert rel_fro(cpu64(y), o.l2_normalize(L, bs, w, gain, epsilon=eps)) <= TOL["f32"]
    rdw, rdg = o.l2_normalize_grad(L, bs, w, dy, gain, epsilon=eps)
    assert rel_fro(cpu64(dw), rdw) <= TOL_GRAD and rel_fro(cpu64(dgain), rdg) <= TOL_GRAD
    m.close()


def test_l2_normalize_exact_cases():
    """identity_init weights: a feature with one unit entry has norm 1, so y = gain * w exactly;
    all-ones blocks over 4 rows of 32 give norm sqrt(128) per feature."""
    L = np.eye(6, dtype=np.uint8)
    m = bsmm.BlocksparseMatMul(L, block_size=32)
    w = m.identity_init()
    gain = torch.linspace(-3, 3, m.K, dtype=torch.float32, device="cuda")
    y = m.l2_normalize(w, gain)
    want = torch.diag_embed(gain.view(6, 32))
    assert torch.equal(y, want)
    m.close()
    L = np.zeros((4, 2), np.uint8)
    L[:, 1] = 1
    m = bsmm.BlocksparseMatMul(L, block_size=32)
    y = m.l2_normalize(torch.ones(m.w_shape, device="cuda") * 4.0, dtype=torch.bfloat16)
    assert torch.equal(y.float(), torch.full(m.w_shape, 1 / np.sqrt(128.0), dtype=torch.bfloat16).float().cuda())
    m.close()


def test_l2_normalize_in_place_deterministic_and_empty(form):
    L, m, w, gain = _case(64, 16, 32, 0.5, 9)
    wd = w.cuda()
    y1 = m.l2_normalize(wd, gain.cuda())
    y2 = m.l2_normalize(wd, gain.cuda())
    assert torch.equal(y1, y2)                         # fixed summation order
    m.l2_normalize(wd, gain.cuda(), y=wd)              # in place (float32)
    assert torch.equal(wd, y1)
    dy = wk.normals(m.w_shape, 4, 1.0, "f32").cuda()
    a = m.l2_normalize_grad(w.cuda(), dy)
    b = m.l2_normalize_grad(w.cuda(), dy)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    with pytest.raises(bsmm.BsmmError):                # 16-bit output over the float32 input
        bsmm.bsmm_l2_normalize(m.handle, wd, None, wd.view(torch.bfloat16)[..., :32])
    m.close()
    m = bsmm.BlocksparseMatMul(np.zeros((3, 4), np.uint8), block_size=16)
    w0 = torch.empty((0, 16, 16), device="cuda")
    assert m.l2_normalize(w0).shape == (0, 16, 16)
    dw, dgain = m.l2_normalize_grad(w0, torch.empty((0, 16, 16), device="cuda"))
    assert dw.numel() == 0 and torch.equal(dgain, torch.zeros(64, device="cuda"))
    m.sync_status()
    m.close()
