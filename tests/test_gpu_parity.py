"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Bit-exact for the lookup tables, block_coord, identity_init, the all-zero and
identity cases and small-integer inputs; relative Frobenius error within the
stated tolerance otherwise.  Every compute test runs both kernel families:
"simt" (IEEE fp32 FFMA) and "auto" (tcgen05 tensor cores for 16-bit inputs).
"""
import functools

import numpy as np
import pytest
import torch

from block_sparse_matrix_gb300 import bsmm, workloads as wk
from block_sparse_matrix_gb300.bsmm import BlocksparseMatMul
from oracle import oracle as o

from _util import TOL, TOL_DW, act_nf, cpu64, problem, rand_layout, rel_fro

pytestmark = pytest.mark.gpu

# Tighter bound than TOL for one float32-accumulated dot product rounded once
# to the output type (RMS relative rounding error of bf16 ~1e-3, fp16 ~1.5e-4).
TIGHT = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}
KERNELS = ["simt", "auto"]
DT = wk.DTYPES


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def make(L, bs, fa, kernel="auto"):
    m = BlocksparseMatMul(L, block_size=bs, feature_axis=fa)
    m.set_kernel(kernel)
    return m


# ---- tables -----------------------------------------------------------------------

@pytest.mark.parametrize("R,S,p,seed", [(8, 8, 0.5, 0), (5, 9, 0.3, 1), (33, 17, 0.7, 2), (1, 1, 1.0, 3),
                                         (6, 6, 0.0, 4), (512, 512, 0.1, 5), (192, 192, 0.05, 6)])
def test_luts_bit_exact(R, S, p, seed):
    L = rand_layout(R, S, p, seed)
    m = make(L, 16, 1)
    got = m.get_luts()
    ref = o.luts(L)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)
    for b in np.random.default_rng(seed).integers(0, max(1, m.nnz), 20) if m.nnz else []:
        assert m.block_coord(int(b)) == tuple(ref[4][b])
    with pytest.raises(bsmm.BsmmError):
        m.block_coord(m.nnz)


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_identity_init_bit_exact(bs, dtype):
    L = rand_layout(7, 7, 0.4, bs, diag=True)
    L[3, 3] = 0
    m = make(L, bs, 1)
    w = m.identity_init(dtype=DT[dtype])
    assert np.array_equal(cpu64(w), o.identity_init(L, bs))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("bs,fa,dtype", [(32, 1, "bf16"), (16, 0, "f16"), (8, 0, "bf16"), (32, 1, "f32"),
                                         (8, 1, "f16"), (16, 1, "bf16"), (32, 0, "f16")])
def test_identity_layer_is_exact(kernel, bs, fa, dtype):
    """identity_init on a block-diagonal layout: y = x and dx = dy bit for bit."""
    R, N = 6, 136
    L = np.eye(R, dtype=np.uint8)
    m = make(L, bs, fa, kernel)
    w = m.identity_init(dtype=DT[dtype])
    x = wk.normals(wk.act_shape(R * bs, N, fa), 5, 1.0, dtype).cuda()
    assert torch.equal(m.fprop(x, w), x)
    assert torch.equal(m.bprop(x, w), x)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("bs,fa,dtype", [(32, 1, "bf16"), (16, 0, "f16"), (8, 0, "bf16"), (8, 1, "f32")])
def test_all_zero_layout(kernel, bs, fa, dtype):
    L = np.zeros((4, 5), np.uint8)
    m = make(L, bs, fa, kernel)
    assert m.nnz == 0
    N = 72
    x = wk.normals(wk.act_shape(4 * bs, N, fa), 1, 1.0, dtype).cuda()
    dy = wk.normals(wk.act_shape(5 * bs, N, fa), 2, 1.0, dtype).cuda()
    w = torch.empty((0, bs, bs), dtype=DT[dtype], device="cuda")
    y = torch.full(m.o_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
    dx = torch.full(m.i_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
    m.fprop(x, w, y)
    m.bprop(dy, w, dx)
    assert not torch.any(y != 0) and not torch.any(dx != 0)
    m.updat(x, dy)
    m.sync_status()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("fa", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_brute_force_2x2_integer_exact(kernel, bs, fa, dtype):
    """All 16 patterns of a 2x2-block layout with entries in {-1,0,1}: every product
    and partial sum is an integer below 2^8, exact in every dtype, so GPU == oracle."""
    N = 144
    for pattern in range(16):
        L = np.array([(pattern >> q) & 1 for q in range(4)], np.uint8).reshape(2, 2)
        m = make(L, bs, fa, kernel)
        seed = 100 * pattern + bs + fa
        x = wk.small_ints(wk.act_shape(2 * bs, N, fa), seed, dtype).cuda()
        dy = wk.small_ints(wk.act_shape(2 * bs, N, fa), seed + 1, dtype).cuda()
        w = wk.small_ints((m.nnz, bs, bs), seed + 2, dtype).cuda()
        y = m.fprop(x, w)
        dx = m.bprop(dy, w)
        dw = m.updat(x, dy)
        m.sync_status()
        assert np.array_equal(cpu64(y), o.fprop(L, bs, x.cpu(), w.cpu(), fa)), pattern
        assert np.array_equal(cpu64(dx), o.bprop(L, bs, dy.cpu(), w.cpu(), fa)), pattern
        assert np.array_equal(cpu64(dw), o.updat(L, bs, x.cpu(), dy.cpu(), fa)), pattern


# ---- seeded random problems spanning several tiles with a ragged tail ---------------

@functools.lru_cache(maxsize=None)
def small_case(bs, fa, dtype):
    R = S = {32: 12, 16: 20, 8: 36}[bs]
    N = 200                                   # 200 = 128 + 72: a full tile plus a ragged tail
    L, x, w, dy = problem(R, S, bs, N, fa, dtype, p=0.4, seed=7 * bs + fa)
    L[:, 1] = 0                               # an empty output block column
    L[2, :] = 0                               # an empty input block row
    nnz = int(L.sum())
    w = w[:nnz] if w.shape[0] >= nnz else wk.normals((nnz, bs, bs), 9, 0.05, dtype)
    w = wk.normals((nnz, bs, bs), 7 * bs + fa + 2, float(1 / np.sqrt(R * bs * 0.4)), dtype)
    ref_y = o.fprop(L, bs, x, w, fa)
    ref_dx = o.bprop(L, bs, dy, w, fa)
    ref_dw = o.updat(L, bs, x, dy, fa)
    return L, x, w, dy, ref_y, ref_dx, ref_dw


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("fa", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_parity_small(kernel, bs, fa, dtype):
    L, x, w, dy, ref_y, ref_dx, ref_dw = small_case(bs, fa, dtype)
    m = make(L, bs, fa, kernel)
    xc, wc, dyc = x.cuda(), w.cuda(), dy.cuda()
    y = torch.full(m.o_shape(200), float("nan"), dtype=DT[dtype], device="cuda")
    dx = torch.full(m.i_shape(200), float("nan"), dtype=DT[dtype], device="cuda")
    m.fprop(xc, wc, y)
    m.bprop(dyc, wc, dx)
    dw = m.updat(xc, dyc)
    m.sync_status()
    for got, ref in ((y, ref_y), (dx, ref_dx)):
        e = rel_fro(cpu64(got), ref)
        assert e <= TOL[dtype] and e <= TIGHT[dtype], e
    e = rel_fro(cpu64(dw), ref_dw)
    assert e <= TOL_DW[dtype], e
    # accumulate: dw += updat
    dw2 = dw.clone()
    m.updat(xc, dyc, dw=dw2, accumulate=True)
    m.sync_status()
    assert rel_fro(cpu64(dw2), 2 * ref_dw) <= TOL_DW[dtype]
    # 16-bit dW output (dw_dtype of the README): float32 sums rounded once to the input type, on the
    # tensor-core kernels under "auto"; accumulating adds in float32 and rounds once more
    if dtype != "f32":
        dwh = m.updat(xc, dyc, dw_dtype=DT[dtype])
        m.sync_status()
        assert dwh.dtype == DT[dtype]
        assert rel_fro(cpu64(dwh), ref_dw) <= TIGHT[dtype]
        m.updat(xc, dyc, dw=dwh, accumulate=True)
        m.sync_status()
        assert rel_fro(cpu64(dwh), 2 * ref_dw) <= TIGHT[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fa,bs,dtype", [(1, 32, "bf16"), (0, 16, "f16"), (0, 8, "bf16"), (1, 8, "f32")])
@pytest.mark.parametrize("G", [1, 3, 8])
def test_grouped_updat(kernel, fa, bs, dtype, G):
    R, S, N = 10, 9, 96
    L = rand_layout(R, S, 0.5, G + bs)
    m = make(L, bs, fa, kernel)
    xs = [wk.normals(wk.act_shape(R * bs, N, fa), 50 + t, 1.0, dtype) for t in range(G)]
    dys = [wk.normals(wk.act_shape(S * bs, N, fa), 70 + t, 1.0, dtype) for t in range(G)]
    ref = o.updat_grouped(L, bs, xs, dys, fa)
    dw = m.updat_grouped([a.cuda() for a in xs], [a.cuda() for a in dys])
    m.sync_status()
    assert rel_fro(cpu64(dw), ref) <= TOL_DW[dtype]
    m.updat_grouped([a.cuda() for a in xs], [a.cuda() for a in dys], dw=dw, accumulate=True)
    m.sync_status()
    assert rel_fro(cpu64(dw), 2 * ref) <= TOL_DW[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
def test_deterministic(kernel):
    L, x, w, dy, *_ = small_case(16, 0, "f16")
    m = make(L, 16, 0, kernel)
    xc, wc, dyc = x.cuda(), w.cuda(), dy.cuda()
    a = (m.fprop(xc, wc), m.bprop(dyc, wc), m.updat(xc, dyc))
    b = (m.fprop(xc, wc), m.bprop(dyc, wc), m.updat(xc, dyc))
    for p, q in zip(a, b):
        assert torch.equal(p, q)


# ---- the five benchmark configurations, full size, sampled outputs -------------------

def _sample_check(m, L, bs, fa, dtype, x, w, dy, y, dx, dw, rng, n_samples=384):
    N = x.shape[0] if fa == 1 else x.shape[1]
    C, K = L.shape[0] * bs, L.shape[1] * bs
    n = rng.integers(0, N, n_samples)
    fk = rng.integers(0, K, n_samples)
    fc = rng.integers(0, C, n_samples)
    y_nf, dx_nf = act_nf(y, fa), act_nf(dx, fa)
    gy = y_nf[torch.from_numpy(n).cuda(), torch.from_numpy(fk).cuda()].double().cpu().numpy()
    gdx = dx_nf[torch.from_numpy(n).cuda(), torch.from_numpy(fc).cuda()].double().cpu().numpy()
    ry = o.fprop_at(L, bs, w, x, fa, n, fk)
    rdx = o.bprop_at(L, bs, w, dy, fa, n, fc)
    assert rel_fro(gy, ry) <= min(TOL[dtype], TIGHT[dtype] * 2)
    assert rel_fro(gdx, rdx) <= min(TOL[dtype], TIGHT[dtype] * 2)
    if dw is not None:
        b = rng.integers(0, m.nnz, n_samples)
        i = rng.integers(0, bs, n_samples)
        j = rng.integers(0, bs, n_samples)
        gdw = dw[torch.from_numpy(b).cuda(), torch.from_numpy(i).cuda(), torch.from_numpy(j).cuda()]
        rdw = o.updat_at(L, bs, x, dy, fa, b, i, j)
        assert rel_fro(gdw.double().cpu().numpy(), rdw) <= TOL_DW[dtype]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", ["h256_b32_fp32", "h4096_b32_p50_n64", "h4096_b32_p50_n1024", "h8192_b16_p10", "h4096_b8_p5"])
def test_config_full_size(kernel, name):
    wl = wk.CONFIGS[name]
    inp = wk.make_inputs(wl)
    L = inp.layout
    m = make(L, wl.bs, wl.feature_axis, kernel)
    x, w, dy = inp.x.cuda(), inp.w.cuda(), inp.dy.cuda()
    y, dx, dw = m.fprop(x, w), m.bprop(dy, w), m.updat(x, dy)
    m.sync_status()
    _sample_check(m, L, wl.bs, wl.feature_axis, wl.dtype, inp.x, inp.w, inp.dy, y, dx, dw,
                  np.random.default_rng(wl.seed_ns))
    if name == "h256_b32_fp32":   # small enough for the full oracle
        assert rel_fro(cpu64(y), o.fprop(L, wl.bs, inp.x, inp.w, 1)) <= TOL["f32"]
        assert rel_fro(cpu64(dx), o.bprop(L, wl.bs, inp.dy, inp.w, 1)) <= TOL["f32"]
        assert rel_fro(cpu64(dw), o.updat(L, wl.bs, inp.x, inp.dy, 1)) <= TOL["f32"]


def test_headline_config_every_output():
    """hidden 4096, block 32, 50% dense, minibatch 1024, bf16: every output of the three passes on
    the tensor-core path against the float64 oracle over the whole tensors (not a sample)."""
    wl = wk.CONFIGS["h4096_b32_p50_n1024"]
    inp = wk.make_inputs(wl)
    L = inp.layout
    m = make(L, wl.bs, 1, "auto")
    x, w, dy = inp.x.cuda(), inp.w.cuda(), inp.dy.cuda()
    y, dx, dw = m.fprop(x, w), m.bprop(dy, w), m.updat(x, dy)
    m.sync_status()
    assert rel_fro(cpu64(y), o.fprop(L, wl.bs, inp.x, inp.w, 1)) <= TIGHT["bf16"]
    assert rel_fro(cpu64(dx), o.bprop(L, wl.bs, inp.dy, inp.w, 1)) <= TIGHT["bf16"]
    assert rel_fro(cpu64(dw), o.updat(L, wl.bs, inp.x, inp.dy, 1)) <= TOL_DW["bf16"]


@pytest.mark.parametrize("kernel", KERNELS)
def test_config5_recurrent_grouped(kernel):
    """16 timesteps share W: per-step fprop/bprop, weight gradient grouped 8 steps per
    call and summed into one float32 dW (group_param_grads)."""
    wl = wk.CONFIGS["h6144_b32_recurrent"]
    inp = wk.make_inputs(wl)
    L, bs = inp.layout, wl.bs
    m = make(L, bs, 1, kernel)
    w = inp.w.cuda()
    xs = [a.cuda() for a in inp.xs]
    dys = [a.cuda() for a in inp.dys]
    rng = np.random.default_rng(55)
    for t in (0, 15):
        y, dx = m.fprop(xs[t], w), m.bprop(dys[t], w)
        _sample_check(m, L, bs, 1, wl.dtype, inp.xs[t], inp.w, inp.dys[t], y, dx, None, rng)
    dw = bsmm.group_param_grads(m, xs, dys, group_size=8)
    m.sync_status()
    b = rng.integers(0, m.nnz, 256)
    i = rng.integers(0, bs, 256)
    j = rng.integers(0, bs, 256)
    ref = sum(o.updat_at(L, bs, inp.xs[t], inp.dys[t], 1, b, i, j) for t in range(16))
    got = dw[torch.from_numpy(b).cuda(), torch.from_numpy(i).cuda(), torch.from_numpy(j).cuda()]
    assert rel_fro(got.double().cpu().numpy(), ref) <= TOL_DW[wl.dtype]


# ---- host-side argument errors with a live handle --------------------------------------

def test_errors_reported():
    L = rand_layout(4, 4, 0.6, 1, diag=True)
    m = make(L, 16, 0)
    x = torch.zeros((64, 72), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(m.w_shape, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((64, 72), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bsmm.BsmmError) as e:           # fa=0 row pitch 70*2 bytes: not 16B aligned
        bsmm.bsmm_fprop(m.handle, x, w, y, 70)
    assert e.value.code == bsmm.ERR_ALIGN
    flat = torch.zeros(64 * 72 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bsmm.BsmmError) as e:           # base pointer off by 2 bytes
        bsmm.bsmm_fprop(m.handle, flat[1:], w, y, 72)
    assert e.value.code == bsmm.ERR_ALIGN
    with pytest.raises(bsmm.BsmmError) as e:
        bsmm.bsmm_updat_grouped(m.handle, [x] * 9, [x] * 9, torch.zeros(m.w_shape, device="cuda"), 72)
    assert e.value.code == bsmm.ERR_INVALID
    with pytest.raises(bsmm.BsmmError) as e:           # dW as fp16 for bf16 inputs
        bsmm.bsmm_updat(m.handle, x, x, torch.zeros(m.w_shape, dtype=torch.float16, device="cuda"), 72)
    assert e.value.code == bsmm.ERR_UNSUPPORTED
    m.sync_status()


@pytest.mark.parametrize("bs,fa,dtype", [(32, 1, "bf16"), (16, 0, "f16"), (8, 0, "bf16"), (8, 1, "f16")])
def test_window_sizes_bit_identical(monkeypatch, bs, fa, dtype):
    """The tensor-core fprop/bprop split output blocks into windows, the minibatch into tiles of
    128 or 64 rows and a window's sources into chunks of 1 to 8 panels; each output is
    accumulated over its source blocks in the same order for every window size, tile height and
    chunk size, so all give the same bits (and match the oracle).  N = 200 leaves a ragged last
    tile either way."""
    L, x, w, dy, ref_y, ref_dx, _ = small_case(bs, fa, dtype)
    xc, wc, dyc = x.cuda(), w.cuda(), dy.cuda()
    outs = []
    monkeypatch.setenv("BSMM_TC_FB", "window")
    for rows in (128, 64):
        monkeypatch.setenv("BSMM_TC_ROWS", str(rows))
        for wlog in range(0, 5):
            monkeypatch.setenv("BSMM_TC_WLOG", str(wlog))
            m = make(L, bs, fa, "auto")
            outs.append((m.fprop(xc, wc), m.bprop(dyc, wc)))
            m.sync_status()
    monkeypatch.delenv("BSMM_TC_ROWS")
    for eslots in (1, 3, 8):                   # activation panels per chunk
        monkeypatch.setenv("BSMM_TC_ESLOTS", str(eslots))
        m = make(L, bs, fa, "auto")
        outs.append((m.fprop(xc, wc), m.bprop(dyc, wc)))
        m.sync_status()
    for y, dx in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(dx, outs[0][1])
    assert rel_fro(cpu64(outs[0][0]), ref_y) <= TIGHT[dtype]
    assert rel_fro(cpu64(outs[0][1]), ref_dx) <= TIGHT[dtype]


@pytest.mark.parametrize("bs,fa,dtype,R,N", [(32, 1, "bf16", 200, 136), (16, 0, "f16", 200, 200),
                                             (8, 0, "bf16", 400, 136), (32, 0, "bf16", 170, 72),
                                             (16, 1, "f16", 200, 40), (32, 0, "bf16", 170, 64)])
def test_window_bins_bit_identical(monkeypatch, bs, fa, dtype, R, N):
    """With more output blocks than SMs per minibatch tile, the window kernel may deal the blocks
    to one bin per SM (heaviest first) and treat each bin as a window of arbitrary output blocks.
    Every output still sums its sources in increasing order, so binned and plain one-block windows
    give the same bits, and both match the oracle.  Columns and rows of 1 to ~30 blocks."""
    L = rand_layout(R, R, 0.05, 900 + bs)
    L[:, 5] = 0                                          # an empty output block column
    L[7, :] = 0                                          # an empty input block row
    L[:, 9] = 1                                          # a full block column
    nnz = int(L.sum())
    x = wk.normals(wk.act_shape(R * bs, N, fa), 61 + bs, 1.0, dtype)
    dy = wk.normals(wk.act_shape(R * bs, N, fa), 62 + bs, 1.0, dtype)
    w = wk.normals((nnz, bs, bs), 63 + bs, float(1 / np.sqrt(R * bs * 0.05)), dtype)
    xc, wc, dyc = x.cuda(), w.cuda(), dy.cuda()
    monkeypatch.setenv("BSMM_TC_FB", "window")
    monkeypatch.setenv("BSMM_TC_WLOG", "0")
    outs = []
    for bins in ("0", "1"):
        monkeypatch.setenv("BSMM_TC_BINS", bins)
        m = make(L, bs, fa, "auto")
        y = torch.full(m.o_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
        dx = torch.full(m.i_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
        m.fprop(xc, wc, y)
        m.bprop(dyc, wc, dx)
        m.sync_status()
        outs.append((y, dx))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert rel_fro(cpu64(outs[1][0]), o.fprop(L, bs, x, w, fa)) <= TIGHT[dtype]
    assert rel_fro(cpu64(outs[1][1]), o.bprop(L, bs, dy, w, fa)) <= TIGHT[dtype]


def test_bounded_wait_times_out_and_context_survives():
    """A device wait that nothing satisfies gives up after its limit, the status word
    reports TIMEOUT, and the same handle keeps computing correct results afterwards."""
    L = np.eye(4, dtype=np.uint8)
    m = make(L, 32, 1)
    bsmm.bsmm_selftest_wait_timeout(m.handle, 20_000_000)        # 20 ms
    with pytest.raises(bsmm.BsmmError) as e:
        m.sync_status()
    assert e.value.code == bsmm.ERR_TIMEOUT
    m.sync_status()                                              # the sticky word was cleared
    w = m.identity_init(dtype=torch.bfloat16)
    x = wk.normals((128, 128), 3, 1.0, "bf16").cuda()
    assert torch.equal(m.fprop(x, w), x)
    m.sync_status()


@pytest.mark.parametrize("variant", ["stack", "dense1", "dense"])
@pytest.mark.parametrize("fa", [0, 1])
@pytest.mark.parametrize("p,G", [(0.5, 1), (0.2, 3), (0.9, 8)])
def test_updat_variants_bs32(monkeypatch, variant, fa, p, G):
    """The tensor-core weight-gradient schemes against the oracle: blocks of a column stacked
    along M ("stack"), dense 128x256 tiles of x^T.dy on one CTA ("dense1"), dense 256x256
    tiles on a CTA pair with two-SM MMAs ("dense"), the present blocks extracted; ragged
    layouts (R, S not multiples of the tile) and a ragged minibatch."""
    monkeypatch.setenv("BSMM_TC_UPDAT", variant)
    bs, R, S, N = 32, 10, 13, 136
    L = rand_layout(R, S, p, 17 + G)
    m = make(L, bs, fa, "auto")
    xs = [wk.normals(wk.act_shape(R * bs, N, fa), 500 + t, 1.0, "bf16") for t in range(G)]
    dys = [wk.normals(wk.act_shape(S * bs, N, fa), 600 + t, 1.0, "bf16") for t in range(G)]
    ref = o.updat_grouped(L, bs, xs, dys, fa)
    dw = m.updat_grouped([a.cuda() for a in xs], [a.cuda() for a in dys])
    m.sync_status()
    assert rel_fro(cpu64(dw), ref) <= TOL_DW["bf16"]
    m.updat_grouped([a.cuda() for a in xs], [a.cuda() for a in dys], dw=dw, accumulate=True)
    m.sync_status()
    assert rel_fro(cpu64(dw), 2 * ref) <= TOL_DW["bf16"]
    if G == 1:
        ref1 = o.updat(L, bs, xs[0], dys[0], fa)
        dw1 = m.updat(xs[0].cuda(), dys[0].cuda())
        m.sync_status()
        assert rel_fro(cpu64(dw1), ref1) <= TOL_DW["bf16"]
        # bf16 dW from the same kernel: one rounding of the float32 sums
        dwh = m.updat(xs[0].cuda(), dys[0].cuda(), dw_dtype=torch.bfloat16)
        m.sync_status()
        assert rel_fro(cpu64(dwh), ref1) <= TIGHT["bf16"]
        assert np.array_equal(cpu64(dwh), cpu64(dw1.bfloat16()))


@pytest.mark.parametrize("fa", [0, 1])
def test_updat_pair_tail_split(monkeypatch, fa):
    """A layout with more 256x256 tiles than CTA pairs, so the last round of tiles is split
    into 256x128 units: the CTA-pair kernel equals the one-CTA dense kernel bit for bit (same
    products, same order) and the oracle within tolerance."""
    bs, R, S, N = 32, 72, 72, 136
    L = rand_layout(R, S, 0.5, 31 + fa)
    x = wk.normals(wk.act_shape(R * bs, N, fa), 900 + fa, 1.0, "bf16")
    dy = wk.normals(wk.act_shape(S * bs, N, fa), 910 + fa, 1.0, "bf16")
    outs = {}
    for variant in ("dense1", "dense"):
        monkeypatch.setenv("BSMM_TC_UPDAT", variant)
        m = make(L, bs, fa, "auto")
        outs[variant] = cpu64(m.updat(x.cuda(), dy.cuda()))
        m.sync_status()
    assert np.array_equal(outs["dense1"], outs["dense"])
    assert rel_fro(outs["dense"], o.updat(L, bs, x, dy, fa)) <= TOL_DW["bf16"]


@pytest.mark.parametrize("variant,bs,fa", [("stack", 32, 1), ("stack", 32, 0), ("stack", 16, 1), ("stack", 16, 0),
                                            ("stack", 8, 1), ("dense1", 32, 1), ("dense1", 32, 0), ("dense", 32, 1),
                                            ("dense", 32, 0)])
@pytest.mark.parametrize("N,G", [(64, 1), (136, 3), (8, 1)])
def test_updat_epilogue_forms_bit_identical(monkeypatch, variant, bs, fa, N, G):
    """The weight-gradient kernels (stacked, dense one-CTA, CTA pair) write dW blocks either by TMA
    (store, or reduce-add in L2 when accumulating) from a swizzled staging tile, or by per-thread
    stores: the same float32 sums, the same single rounding, so the same bits -- float32 dW written
    and accumulated, a bf16 dW written -- and the oracle within tolerance."""
    monkeypatch.setenv("BSMM_TC_UPDAT", variant)
    R, S = 11, 9
    L = rand_layout(R, S, 0.45, 90 + bs + N)
    L[0, 0] = 1
    xs = [wk.normals(wk.act_shape(R * bs, N, fa), 300 + t + N, 1.0, "bf16") for t in range(G)]
    dys = [wk.normals(wk.act_shape(S * bs, N, fa), 400 + t + N, 1.0, "bf16") for t in range(G)]
    xg, dyg = [a.cuda() for a in xs], [a.cuda() for a in dys]
    outs = {}
    for form in ("tma", "stores"):
        monkeypatch.setenv("BSMM_UP_EPI", form)
        m = make(L, bs, fa, "auto")
        dw = m.updat_grouped(xg, dyg)
        dw_first = dw.clone()
        m.updat_grouped(xg, dyg, dw=dw, accumulate=True)
        dwh = m.updat(xg[0], dyg[0], dw_dtype=torch.bfloat16)
        m.sync_status()
        outs[form] = (dw_first, dw, dwh)
    for a, b in zip(outs["tma"], outs["stores"]):
        assert torch.equal(a, b)
    ref = o.updat_grouped(L, bs, xs, dys, fa)
    assert rel_fro(cpu64(outs["tma"][0]), ref) <= TOL_DW["bf16"]
    assert rel_fro(cpu64(outs["tma"][1]), 2 * ref) <= TOL_DW["bf16"]
    assert rel_fro(cpu64(outs["tma"][2]), o.updat(L, bs, xs[0], dys[0], fa)) <= TIGHT["bf16"]


@pytest.mark.parametrize("variant,bs,fa", [("stack", 32, 1), ("stack", 16, 0), ("stack", 8, 1),
                                            ("dense1", 32, 0), ("dense", 32, 1)])
def test_updat_refuses_an_out_of_range_block_id(monkeypatch, variant, bs, fa):
    """Fault injection on the host: a test hook makes the weight-gradient table name block
    nnz + 5.  The epilogue checks every block id before its store, skips that block and records
    BSMM_ERR_BOUNDS.  dW sits at the start of a larger buffer, so an unchecked store would land
    in the guard blocks after it (inside the allocation): they must keep their sentinel, every
    other block must match the oracle, and the next call on a fresh table is correct again."""
    monkeypatch.setenv("BSMM_TC_UPDAT", variant)
    R, S, N = 10, 13, 136
    L = rand_layout(R, S, 0.5, 41 + bs)
    L[0, 0] = 1
    nnz = int(L.sum())
    x = wk.normals(wk.act_shape(R * bs, N, fa), 950 + bs, 1.0, "bf16")
    dy = wk.normals(wk.act_shape(S * bs, N, fa), 960 + bs, 1.0, "bf16")
    ref = o.updat(L, bs, x, dy, fa)
    monkeypatch.setenv("BSMM_UP_TEST_BAD_ID", "1")
    m = make(L, bs, fa, "auto")
    buf = torch.full((nnz + 8, bs, bs), 7.0, device="cuda")
    m.updat(x.cuda(), dy.cuda(), dw=buf[:nnz])
    with pytest.raises(bsmm.BsmmError) as e:
        m.sync_status()
    assert e.value.code == bsmm.ERR_BOUNDS
    got = cpu64(buf)
    m.close()
    assert np.all(got[nnz:] == 7.0)
    err = np.abs(got[:nnz] - ref).max(axis=(1, 2))
    off = np.flatnonzero(err > 1e-3 * (np.abs(ref).max() + 1.0))
    assert len(off) <= 1                         # only the block whose id was replaced
    assert all(np.all(got[b] == 7.0) for b in off)
    monkeypatch.delenv("BSMM_UP_TEST_BAD_ID")
    m = make(L, bs, fa, "auto")
    dw = m.updat(x.cuda(), dy.cuda())
    m.sync_status()
    assert rel_fro(cpu64(dw), ref) <= TOL_DW["bf16"]


@pytest.mark.parametrize("fa,dtype", [(1, "bf16"), (0, "f16")])
@pytest.mark.parametrize("R,S,p,N", [(10, 13, 0.5, 392), (7, 9, 0.9, 264), (12, 6, 0.3, 136),
                                     (20, 37, 0.5, 520), (10, 13, 0.5, 64), (9, 7, 0.8, 40)])
def test_fprop_bprop_variants_bs32(monkeypatch, fa, dtype, R, S, p, N):
    """The tensor-core fprop/bprop schemes against the oracle: windows of output blocks over
    128-row tiles; dense tiles of 4 output blocks x 256 rows with absent blocks as zero tiles
    on one CTA ("dense1"); dense tiles of 8 output blocks x 256 rows on a CTA pair with
    two-SM MMAs ("dense"; for a minibatch of at most 64 rows the dense tile is instead split
    over a cluster of 4 CTAs and summed in distributed shared memory).  Layouts whose block
    counts are not multiples of the tile, and ragged minibatches."""
    bs = 32
    L = rand_layout(R, S, p, R * 31 + S)
    L[:, 2] = 0                                           # an empty output block column
    L[1, :] = 0                                           # an empty input block row
    nnz = int(L.sum())
    x = wk.normals(wk.act_shape(R * bs, N, fa), 700 + R, 1.0, dtype)
    dy = wk.normals(wk.act_shape(S * bs, N, fa), 800 + S, 1.0, dtype)
    w = wk.normals((nnz, bs, bs), 900 + R + S, float(1 / np.sqrt(R * bs * p)), dtype)
    ref_y, ref_dx = o.fprop(L, bs, x, w, fa), o.bprop(L, bs, dy, w, fa)
    outs = {}
    for variant in ("window", "sp", "dense1", "dense"):
        monkeypatch.setenv("BSMM_TC_FB", variant)
        m = make(L, bs, fa, "auto")
        y = torch.full(m.o_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
        dx = torch.full(m.i_shape(N), float("nan"), dtype=DT[dtype], device="cuda")
        m.fprop(x.cuda(), w.cuda(), y)
        m.bprop(dy.cuda(), w.cuda(), dx)
        m.sync_status()
        assert rel_fro(cpu64(y), ref_y) <= TIGHT[dtype]
        assert rel_fro(cpu64(dx), ref_dx) <= TIGHT[dtype]
        outs[variant] = (cpu64(y), cpu64(dx))
    # every scheme accumulates in fp32 and rounds once: they agree to a few output ulps
    for other in ("sp", "dense"):
        for a, b in zip(outs["window"], outs[other]):
            assert rel_fro(a, b) <= TIGHT[dtype]
    # one-CTA and CTA-pair dense tiles add the same products in the same order
    for a, b in zip(outs["dense1"], outs["dense"]):
        assert np.array_equal(a, b)
