"""Pins for the CPU oracle: facts fixed by the blocksparse README and by plain
mathematics, checked by routes that do not go through the oracle's own code.

Each test names the passage or the property it relies on.  A plausible slip
in the oracle (a transposed block, a wrong block order, a dropped block, a
swapped feature_axis) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as o
from block_sparse_matrix_gb300 import workloads as wk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_layout(R, S, p, seed):
    return (np.random.default_rng(seed).random((R, S)) < p).astype(np.uint8)


def act(a, fa):
    """(N, F) view of an activation stored in feature_axis `fa` layout."""
    return a if fa == 1 else a.T


def from_nf(a_nf, fa):
    return a_nf if fa == 1 else np.ascontiguousarray(a_nf.T)


def blocks_of_dense(L, bs, Wfull):
    """Weight blocks cut out of a dense matrix, one per nonzero, in np.argwhere order."""
    return np.stack([Wfull[c * bs:(c + 1) * bs, k * bs:(k + 1) * bs] for c, k in np.argwhere(L)]) \
        if L.any() else np.zeros((0, bs, bs))


def mask(L, bs):
    return np.kron(L.astype(np.float64), np.ones((bs, bs)))


# -- lookup tables / block_coord ("block_coord(block)" in the API listing) ----------

@pytest.mark.parametrize("R,S,p,seed", [(8, 8, 0.5, 0), (5, 9, 0.3, 1), (16, 3, 0.7, 2),
                                         (1, 1, 1.0, 3), (7, 7, 0.0, 4), (32, 32, 0.1, 5)])
def test_luts_match_brute_force(R, S, p, seed):
    L = rand_layout(R, S, p, seed)
    row_ptr, row_ent, col_ptr, col_ent, coord = o.luts(L)
    ref = np.argwhere(L)                          # row-major scan order
    assert np.array_equal(coord, ref.astype(np.int32).reshape(-1, 2))
    assert np.array_equal(row_ptr, np.concatenate([[0], np.cumsum(L.sum(1))]).astype(np.int32))
    assert np.array_equal(col_ptr, np.concatenate([[0], np.cumsum(L.sum(0))]).astype(np.int32))
    assert np.array_equal(row_ent, ref[:, 1].astype(np.int32))
    ids = {tuple(ck): b for b, ck in enumerate(ref)}
    for k in range(S):
        seg = col_ent[col_ptr[k]:col_ptr[k + 1]]
        cs = np.nonzero(L[:, k])[0]
        assert np.array_equal(seg[:, 1], cs)
        assert all(seg[i, 0] == ids[(c, k)] for i, c in enumerate(cs))


# -- the dense special cases ----------------------------------------------------

@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("fa", [0, 1])
def test_all_ones_layout_is_dense_matmul(bs, fa):
    """An all-ones layout makes W dense; y = x.W, dx = dy.W^T, dW = x^T.dy (numpy)."""
    R, S, N = 3, 2, 5
    rng = np.random.default_rng(bs + fa)
    L = np.ones((R, S), np.uint8)
    C, K = R * bs, S * bs
    Wfull = rng.standard_normal((C, K))
    w = Wfull.reshape(R, bs, S, bs).transpose(0, 2, 1, 3).reshape(R * S, bs, bs)
    x_nf, dy_nf = rng.standard_normal((N, C)), rng.standard_normal((N, K))
    x, dy = from_nf(x_nf, fa), from_nf(dy_nf, fa)
    np.testing.assert_allclose(act(o.fprop(L, bs, x, w, fa), fa), x_nf @ Wfull, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(act(o.bprop(L, bs, dy, w, fa), fa), dy_nf @ Wfull.T, rtol=1e-12, atol=1e-12)
    G = x_nf.T @ dy_nf
    dw_ref = G.reshape(R, bs, S, bs).transpose(0, 2, 1, 3).reshape(R * S, bs, bs)
    np.testing.assert_allclose(o.updat(L, bs, x, dy, fa), dw_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bs,fa,seed", [(8, 1, 0), (16, 0, 1), (32, 1, 2), (8, 0, 3)])
def test_random_layout_equals_masked_dense(bs, fa, seed):
    """W = (dense matrix) * (layout expanded to bs x bs); blocks in block_coord order."""
    R, S, N = 6, 5, 7
    rng = np.random.default_rng(100 + seed)
    L = rand_layout(R, S, 0.45, seed)
    L[0, :] = 0          # an empty block row
    L[:, 2] = 0          # an empty block column
    Wfull = rng.standard_normal((R * bs, S * bs))
    w = blocks_of_dense(L, bs, Wfull)
    Wm = Wfull * mask(L, bs)
    x_nf, dy_nf = rng.standard_normal((N, R * bs)), rng.standard_normal((N, S * bs))
    x, dy = from_nf(x_nf, fa), from_nf(dy_nf, fa)
    np.testing.assert_allclose(o.densify(L, bs, w), Wm, rtol=0, atol=0)
    np.testing.assert_allclose(act(o.fprop(L, bs, x, w, fa), fa), x_nf @ Wm, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(act(o.bprop(L, bs, dy, w, fa), fa), dy_nf @ Wm.T, rtol=1e-12, atol=1e-12)
    dw_ref = blocks_of_dense(L, bs, x_nf.T @ dy_nf)
    np.testing.assert_allclose(o.updat(L, bs, x, dy, fa), dw_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fa", [0, 1])
def test_all_zero_layout_gives_zeros(fa):
    L = np.zeros((4, 3), np.uint8)
    bs, N = 16, 6
    x = np.random.default_rng(0).standard_normal(wk.act_shape(4 * bs, N, fa))
    dy = np.random.default_rng(1).standard_normal(wk.act_shape(3 * bs, N, fa))
    w = np.zeros((0, bs, bs))
    assert not o.fprop(L, bs, x, w, fa).any()
    assert not o.bprop(L, bs, dy, w, fa).any()
    assert o.updat(L, bs, x, dy, fa).shape == (0, bs, bs)


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("fa", [0, 1])
def test_identity_init_block_diagonal_is_identity(bs, fa):
    """identity_init ("identity_init + layernorm is all you need") on a block-diagonal
    layout gives y = x and dx = dy exactly; with off-diagonal blocks present they are 0."""
    R = 4
    N = 9
    L = np.eye(R, dtype=np.uint8)
    w = o.identity_init(L, bs)
    x = np.random.default_rng(bs).standard_normal(wk.act_shape(R * bs, N, fa))
    assert np.array_equal(o.fprop(L, bs, x, w, fa), x)
    assert np.array_equal(o.bprop(L, bs, x, w, fa), x)
    L2 = L.copy()
    L2[0, 3] = L2[2, 1] = 1
    w2 = o.identity_init(L2, bs)
    assert np.array_equal(o.fprop(L2, bs, x, w2, fa), x)
    assert np.array_equal(o.densify(L2, bs, w2), np.eye(R * bs))
    # a missing diagonal block leaves its output block zero
    L3 = L.copy()
    L3[1, 1] = 0
    y3 = act(o.fprop(L3, bs, x, o.identity_init(L3, bs), fa), fa)
    assert not y3[:, bs:2 * bs].any()
    assert np.array_equal(y3[:, :bs], act(x, fa)[:, :bs])


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("fa", [0, 1])
def test_brute_force_2x2_layouts_integers(bs, fa):
    """All 16 patterns of a 2x2-block layout, small-integer inputs (exact in fp32),
    against a block-by-block accumulation written independently here."""
    N = 4
    for bits in itertools.product([0, 1], repeat=4):
        L = np.array(bits, np.uint8).reshape(2, 2)
        z = int(L.sum())
        rng = np.random.default_rng(int("".join(map(str, bits)), 2) + 10 * bs + fa)
        w = rng.integers(-1, 2, (z, bs, bs)).astype(np.float64)
        x_nf = rng.integers(-1, 2, (N, 2 * bs)).astype(np.float64)
        dy_nf = rng.integers(-1, 2, (N, 2 * bs)).astype(np.float64)
        y = np.zeros((N, 2 * bs))
        dx = np.zeros((N, 2 * bs))
        dw = np.zeros((z, bs, bs))
        b = 0
        for c in range(2):
            for k in range(2):
                if not L[c, k]:
                    continue
                xs, ks = slice(c * bs, (c + 1) * bs), slice(k * bs, (k + 1) * bs)
                for n in range(N):
                    for i in range(bs):
                        for j in range(bs):
                            y[n, k * bs + j] += x_nf[n, c * bs + i] * w[b, i, j]
                            dx[n, c * bs + i] += dy_nf[n, k * bs + j] * w[b, i, j]
                            dw[b, i, j] += x_nf[n, c * bs + i] * dy_nf[n, k * bs + j]
                b += 1
        x, dy = from_nf(x_nf, fa), from_nf(dy_nf, fa)
        assert np.array_equal(act(o.fprop(L, bs, x, w, fa), fa), y)
        assert np.array_equal(act(o.bprop(L, bs, dy, w, fa), fa), dx)
        assert np.array_equal(o.updat(L, bs, x, dy, fa), dw)


# -- invariants -----------------------------------------------------------------

@pytest.mark.parametrize("bs,fa", [(8, 0), (16, 1), (32, 0)])
def test_adjoint_identity(bs, fa):
    """<x.W, dy> = <x, dy.W^T> = <dW, w> where dW = updat(x, dy)."""
    R, S, N = 5, 4, 6
    rng = np.random.default_rng(7 * bs + fa)
    L = rand_layout(R, S, 0.5, bs)
    w = rng.standard_normal((int(L.sum()), bs, bs))
    x = rng.standard_normal(wk.act_shape(R * bs, N, fa))
    dy = rng.standard_normal(wk.act_shape(S * bs, N, fa))
    a = np.sum(o.fprop(L, bs, x, w, fa) * dy)
    b = np.sum(x * o.bprop(L, bs, dy, w, fa))
    c = np.sum(o.updat(L, bs, x, dy, fa) * w)
    assert abs(a - b) <= 1e-10 * abs(a) + 1e-10
    assert abs(a - c) <= 1e-10 * abs(a) + 1e-10


@pytest.mark.parametrize("bs", [8, 32])
def test_feature_axis_transpose(bs):
    """feature_axis=0 on transposed activations gives the transposed feature_axis=1 result."""
    R, S, N = 3, 4, 5
    rng = np.random.default_rng(bs)
    L = rand_layout(R, S, 0.6, 9)
    w = rng.standard_normal((int(L.sum()), bs, bs))
    x = rng.standard_normal((N, R * bs))
    dy = rng.standard_normal((N, S * bs))
    assert np.array_equal(o.fprop(L, bs, x.T.copy(), w, 0), o.fprop(L, bs, x, w, 1).T)
    assert np.array_equal(o.bprop(L, bs, dy.T.copy(), w, 0), o.bprop(L, bs, dy, w, 1).T)
    assert np.array_equal(o.updat(L, bs, x.T.copy(), dy.T.copy(), 0), o.updat(L, bs, x, dy, 1))


@pytest.mark.parametrize("fa", [0, 1])
def test_grouped_is_sum_of_steps_and_concat(fa):
    """group_param_grads: the grouped weight gradient equals the per-step sum and the
    single updat over the minibatch concatenation of the steps."""
    bs, R, S, N, G = 8, 4, 3, 5, 5
    rng = np.random.default_rng(fa)
    L = rand_layout(R, S, 0.5, 11)
    xs = [rng.standard_normal(wk.act_shape(R * bs, N, fa)) for _ in range(G)]
    dys = [rng.standard_normal(wk.act_shape(S * bs, N, fa)) for _ in range(G)]
    g = o.updat_grouped(L, bs, xs, dys, fa)
    s = sum(o.updat(L, bs, a, d, fa) for a, d in zip(xs, dys))
    ax = 0 if fa == 1 else 1
    cat = o.updat(L, bs, np.concatenate(xs, axis=ax), np.concatenate(dys, axis=ax), fa)
    np.testing.assert_allclose(g, s, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g, cat, rtol=1e-12, atol=1e-12)
    init = rng.standard_normal(g.shape)
    np.testing.assert_allclose(o.updat_grouped(L, bs, xs, dys, fa, dw_init=init), g + init,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o.updat(L, bs, xs[0], dys[0], fa, dw_init=init),
                               o.updat(L, bs, xs[0], dys[0], fa) + init, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bs,fa", [(8, 1), (16, 0), (32, 1)])
def test_sampled_outputs_equal_full(bs, fa):
    R, S, N = 4, 5, 6
    rng = np.random.default_rng(3 * bs + fa)
    L = rand_layout(R, S, 0.5, 21)
    w = rng.standard_normal((int(L.sum()), bs, bs))
    x = rng.standard_normal(wk.act_shape(R * bs, N, fa))
    dy = rng.standard_normal(wk.act_shape(S * bs, N, fa))
    y, dx, dw = o.fprop(L, bs, x, w, fa), o.bprop(L, bs, dy, w, fa), o.updat(L, bs, x, dy, fa)
    n = rng.integers(0, N, 50)
    fk = rng.integers(0, S * bs, 50)
    fc = rng.integers(0, R * bs, 50)
    np.testing.assert_allclose(o.fprop_at(L, bs, w, x, fa, n, fk), act(y, fa)[n, fk], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o.bprop_at(L, bs, w, dy, fa, n, fc), act(dx, fa)[n, fc], rtol=1e-13, atol=1e-13)
    b = rng.integers(0, len(w), 50)
    i = rng.integers(0, bs, 50)
    j = rng.integers(0, bs, 50)
    np.testing.assert_allclose(o.updat_at(L, bs, x, dy, fa, b, i, j), dw[b, i, j], rtol=1e-13, atol=1e-13)


def test_golden_usage_example_ones():
    """Hand-worked values for the README 'Usage' example pattern (x = ones)."""
    with open(os.path.join(GOLDEN, "usage_ones.json")) as f:
        g = json.load(f)
    L = np.array(g["layout"], np.uint8)
    bs, N = g["block_size"], g["N"]
    w = np.stack([np.full((bs, bs), float((b + 1) ** 2)) for b in range(int(L.sum()))])
    C, K = L.shape[0] * bs, L.shape[1] * bs
    for fa in (0, 1):
        y = act(o.fprop(L, bs, np.ones(wk.act_shape(C, N, fa)), w, fa), fa)
        assert np.array_equal(y, np.tile(g["fprop_x_ones_expected_row"], (N, 1)))
        dx = act(o.bprop(L, bs, np.ones(wk.act_shape(K, N, fa)), w, fa), fa)
        assert np.array_equal(dx, np.tile(g["bprop_dy_ones_expected_row"], (N, 1)))
        dw = o.updat(L, bs, np.ones(wk.act_shape(C, N, fa)), np.ones(wk.act_shape(K, N, fa)), fa)
        assert np.all(dw == g["updat_ones_expected"])


def test_workload_layouts():
    """The synthetic layouts have the stated structure (diagonal forced, 8 extra per row)."""
    for name in ("h256_b32_fp32", "h8192_b16_p10", "h4096_b8_p5"):
        wl = wk.CONFIGS[name]
        L = wk.make_layout(wl.R, wl.S, wl.layout_kind, wl.density, wl.force_diag, 1000 * wl.seed_ns)
        assert np.all(np.diag(L) == 1)
    wl = wk.CONFIGS["h6144_b32_recurrent"]
    L = wk.make_layout(wl.R, wl.S, wl.layout_kind, wl.density, wl.force_diag, 5000)
    assert np.all(L.sum(1) == 9) and np.all(np.diag(L) == 1)


# ---- layer_norm (README "blocksparse.norms"): pins independent of the oracle's code ----------

def _ln_inputs(N, C, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, C)) * 3.0 + 1.5, rng.standard_normal(C), rng.standard_normal(C)


def test_layer_norm_hand_example():
    """x = (1, 2, 3, 4): mean 5/2 and biased variance 5/4 by hand, so the normalised values
    are (x - 5/2) / sqrt(5/4); then scale, shift and relu elementwise."""
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    g = np.array([1.0, 2.0, 0.5, -1.0])
    b = np.array([0.0, 1.0, -1.0, 0.25])
    z = (x[0] - 2.5) / math.sqrt(1.25)
    want = g * z + b
    got = o.layer_norm(x, g, b, axis=1, epsilon=0.0)
    assert np.allclose(got[0], want, rtol=0, atol=1e-15)
    got_r = o.layer_norm(x, g, b, axis=1, epsilon=0.0, relu=True)
    assert np.array_equal(got_r[0], np.maximum(got[0], 0.0))


def test_layer_norm_output_statistics():
    """With g = 1, b = 0 every sample's output has mean 0 and mean square var / (var + eps)
    (numpy's biased variance of the input)."""
    x, _, _ = _ln_inputs(7, 37, 1)
    eps = 1e-3
    y = o.layer_norm(x, np.ones(37), np.zeros(37), axis=1, epsilon=eps)
    var = np.var(x, axis=1)
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-13)
    assert np.allclose((y * y).mean(axis=1), var / (var + eps), rtol=1e-12)


def test_layer_norm_constant_sample_gives_shift():
    x = np.full((3, 16), 0.5)
    x[1] = -2.0
    g, b = np.arange(16.0) - 3, np.linspace(-1, 1, 16)
    for relu in (False, True):
        y = o.layer_norm(x, g, b, axis=1, epsilon=1e-6, relu=relu)
        assert np.array_equal(y, np.tile(np.maximum(b, 0.0) if relu else b, (3, 1)))


def test_layer_norm_affine_invariance():
    """layer_norm(a x + c) with epsilon scaled by a^2 equals layer_norm(x): a wrong centring,
    a wrong variance divisor or epsilon outside the square root breaks this."""
    x, g, b = _ln_inputs(5, 64, 2)
    a, c, eps = 3.0, -7.0, 1e-2
    y1 = o.layer_norm(x, g, b, axis=1, epsilon=eps)
    y2 = o.layer_norm(a * x + c, g, b, axis=1, epsilon=eps * a * a)
    assert np.allclose(y1, y2, rtol=1e-11, atol=1e-12)


def test_layer_norm_axis_layouts_agree():
    x, g, b = _ln_inputs(6, 40, 3)
    y1 = o.layer_norm(x, g, b, axis=1, epsilon=1e-6, relu=True)
    y0 = o.layer_norm(x.T.copy(), g, b, axis=0, epsilon=1e-6, relu=True)
    assert np.array_equal(y0, y1.T)


def test_layer_norm_matches_numpy_definition():
    """Against numpy's own mean / biased variance, written independently of the oracle."""
    x, g, b = _ln_inputs(9, 33, 4)
    eps = 1e-6
    want = g * (x - x.mean(axis=1, keepdims=True)) / np.sqrt(x.var(axis=1, keepdims=True) + eps) + b
    assert np.allclose(o.layer_norm(x, g, b, axis=1, epsilon=eps), want, rtol=1e-12, atol=1e-12)


# ---- layer_norm gradient: pinned to the (pinned) forward pass by finite differences ----------

def _ln_loss(x, g, b, dy, axis, eps, relu):
    return float((dy * o.layer_norm(x, g, b, axis=axis, epsilon=eps, relu=relu)).sum())


@pytest.mark.parametrize("axis", [1, 0])
@pytest.mark.parametrize("relu", [False, True])
def test_layer_norm_grad_finite_differences(axis, relu):
    """dx, dg and db against central differences of sum(dy * layer_norm(x, g, b)); with relu the
    inputs keep every pre-activation at least 1e-3 from zero, so the mask is locally constant."""
    N, C, eps = 5, 11, 1e-3
    x, g, b = _ln_inputs(N, C, 21)
    if axis == 0:
        x = x.T.copy()
    dy = np.random.default_rng(22).standard_normal(x.shape)
    y = o.layer_norm(x, g, b, axis=axis, epsilon=eps, relu=relu)
    if relu:
        z = o.layer_norm(x, g, b, axis=axis, epsilon=eps)
        assert np.abs(z).min() > 1e-3 and (z < 0).any() and (z > 0).any()
    dx, dg, db = o.layer_norm_grad(x, g, dy, y=y, axis=axis, epsilon=eps, relu=relu)
    h = 1e-6
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = (_ln_loss(xp, g, b, dy, axis, eps, relu) - _ln_loss(xm, g, b, dy, axis, eps, relu)) / (2 * h)
        assert abs(fd - dx[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, dx[idx])
    for f in range(C):
        for v, grad in ((g, dg), (b, db)):
            vp, vm = v.copy(), v.copy()
            vp[f] += h
            vm[f] -= h
            args_p = (vp, b) if v is g else (g, vp)
            args_m = (vm, b) if v is g else (g, vm)
            fd = (_ln_loss(x, *args_p, dy, axis, eps, relu) - _ln_loss(x, *args_m, dy, axis, eps, relu)) / (2 * h)
            assert abs(fd - grad[f]) <= 1e-6 * max(1.0, abs(fd)), (f, fd, grad[f])


def test_layer_norm_grad_invariances():
    """The output ignores a shift of a sample, and (epsilon = 0) a scaling of it, so every row
    of dx sums to zero and is orthogonal to the centred sample; without relu db is the plain sum
    of dy over samples."""
    x, g, b = _ln_inputs(7, 29, 23)
    dy = np.random.default_rng(24).standard_normal(x.shape)
    dx, dg, db = o.layer_norm_grad(x, g, dy, axis=1, epsilon=0.0)
    assert np.allclose(dx.sum(axis=1), 0.0, atol=1e-12)
    xc = x - x.mean(axis=1, keepdims=True)
    assert np.allclose((dx * xc).sum(axis=1), 0.0, atol=1e-11)
    assert np.allclose(db, dy.sum(axis=0), rtol=1e-14, atol=1e-14)
    xh = xc / np.sqrt((xc * xc).mean(axis=1, keepdims=True))
    assert np.allclose(dg, (dy * xh).sum(axis=0), rtol=1e-12, atol=1e-12)


def test_layer_norm_grad_relu_mask_zeroes_and_layouts_agree():
    """Where the forward output is 0 the gradient does not pass: dy there changes nothing; the
    (C, N) layout gives the transposed result of the (N, C) one."""
    x, g, b = _ln_inputs(6, 17, 25)
    y = o.layer_norm(x, g, b, axis=1, epsilon=1e-6, relu=True)
    assert (y == 0).any()
    dy = np.random.default_rng(26).standard_normal(x.shape)
    dy2 = np.where(y > 0, dy, 100.0)
    r1 = o.layer_norm_grad(x, g, dy, y=y, axis=1, relu=True)
    r2 = o.layer_norm_grad(x, g, dy2, y=y, axis=1, relu=True)
    for a, c in zip(r1, r2):
        assert np.array_equal(a, c)
    r0 = o.layer_norm_grad(x.T.copy(), g, dy.T.copy(), y=y.T.copy(), axis=0, relu=True)
    assert np.allclose(r0[0], r1[0].T, rtol=1e-13, atol=1e-13)
    assert np.allclose(r0[1], r1[1], rtol=1e-13, atol=1e-13)
    assert np.allclose(r0[2], r1[2], rtol=1e-13, atol=1e-13)


# --- l2_normalize (README, "API Documentation: blocksparse.matmul": weight normalisation) ---

def _wn_inputs(R, S, bs, p, seed, scale=1.0):
    L = rand_layout(R, S, p, seed)
    L[0, 0] = 1                                   # at least one block
    rng = np.random.default_rng(seed + 100)
    w = rng.standard_normal((int(L.sum()), bs, bs)) * scale
    gain = rng.uniform(0.5, 2.0, S * bs) * np.where(rng.random(S * bs) < 0.2, -1.0, 1.0)
    return L, w, gain


def test_l2_normalize_hand_example():
    """Block column 0 holds two all-ones 8x8 blocks: each of its features has 16 ones, norm 4.
    Block column 1 holds 2*I: each feature has the single entry 2, norm 2."""
    L = np.array([[1, 0], [1, 1]], np.uint8)      # ids: (0,0) -> 0, (1,0) -> 1, (1,1) -> 2
    w = np.stack([np.ones((8, 8)), np.ones((8, 8)), 2.0 * np.eye(8)])
    gain = np.arange(16.0) + 1.0
    y = o.l2_normalize(L, 8, w)
    assert np.array_equal(y[0], np.full((8, 8), 0.25)) and np.array_equal(y[1], y[0])
    assert np.array_equal(y[2], np.eye(8))
    yg = o.l2_normalize(L, 8, w, gain)
    assert np.array_equal(yg[0], np.tile(0.25 * gain[:8], (8, 1)))
    assert np.array_equal(yg[2], np.diag(gain[8:]))


def test_l2_normalize_unit_feature_norms():
    """Without a gain every output feature of the dense weight has unit norm; features of empty
    block columns stay absent (zero)."""
    L, w, _ = _wn_inputs(9, 7, 8, 0.4, 1)
    L2 = L.copy()
    L2[:, 3] = 0                                   # one empty block column
    w2 = w[: int(L2.sum())]
    Yd = o.densify(L2, 8, o.l2_normalize(L2, 8, w2))
    norms = np.linalg.norm(Yd, axis=0)
    present = np.repeat(L2.any(axis=0), 8)
    assert np.allclose(norms[present], 1.0, rtol=1e-13) and np.array_equal(norms[~present], np.zeros((~present).sum()))


def test_l2_normalize_matches_dense_numpy():
    """Against column norms of the dense weight computed by numpy (a route through densify, not
    through the oracle's block loop): a norm over rows instead of features, or a block of the
    wrong column, fails here."""
    for bs, seed in ((8, 2), (16, 3), (32, 4)):
        L, w, gain = _wn_inputs(5, 6, bs, 0.5, seed)
        eps = 1e-6
        Wd = o.densify(L, bs, w)
        want = Wd * gain / np.sqrt(np.maximum((Wd ** 2).sum(axis=0), eps))
        got = o.densify(L, bs, o.l2_normalize(L, bs, w, gain, epsilon=eps))
        assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


def test_l2_normalize_epsilon_bounds_the_squared_norm():
    """A feature whose squared norm is below epsilon is divided by sqrt(epsilon) instead."""
    L, w, gain = _wn_inputs(4, 4, 8, 0.6, 5, scale=1e-4)   # squared norms ~ 1e-7 * 32
    eps = 0.25
    assert np.allclose(o.l2_normalize(L, 8, w, gain, epsilon=eps),
                       w * gain.reshape(-1, 8)[np.argwhere(L)[:, 1]][:, None, :] / 0.5, rtol=1e-15, atol=0)


def test_l2_normalize_scale_invariance():
    L, w, gain = _wn_inputs(6, 5, 16, 0.5, 6)
    assert np.allclose(o.l2_normalize(L, 16, 37.5 * w, gain), o.l2_normalize(L, 16, w, gain), rtol=1e-13)


def _wn_loss(L, bs, w, dy, gain, eps):
    return float((o.l2_normalize(L, bs, w, gain, epsilon=eps) * dy).sum())


@pytest.mark.parametrize("regime", ["norm", "epsilon"])
def test_l2_normalize_grad_finite_differences(regime):
    """dw and dgain against central differences of sum(dy * l2_normalize(w, gain)), in both
    branches of the max (squared norm above and below epsilon)."""
    scale, eps = (1.0, 1e-6) if regime == "norm" else (1e-3, 1.0)
    L, w, gain = _wn_inputs(4, 3, 8, 0.6, 7, scale=scale)
    dy = np.random.default_rng(8).standard_normal(w.shape)
    dw, dgain = o.l2_normalize_grad(L, 8, w, dy, gain, epsilon=eps)
    rng = np.random.default_rng(9)
    h = 1e-6 * scale
    for _ in range(12):
        idx = tuple(rng.integers(0, n) for n in w.shape)
        wp, wm = w.copy(), w.copy()
        wp[idx] += h
        wm[idx] -= h
        fd = (_wn_loss(L, 8, wp, dy, gain, eps) - _wn_loss(L, 8, wm, dy, gain, eps)) / (2 * h)
        assert abs(fd - dw[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, dw[idx])
    for f in rng.integers(0, gain.size, 8):
        gp, gm = gain.copy(), gain.copy()
        gp[f] += 1e-6
        gm[f] -= 1e-6
        fd = (_wn_loss(L, 8, w, dy, gp, eps) - _wn_loss(L, 8, w, dy, gm, eps)) / 2e-6
        assert abs(fd - dgain[f]) <= 1e-6 * max(1.0, abs(fd))


def test_l2_normalize_grad_orthogonal_to_w():
    """Without a gain and above epsilon, the output does not change along w itself, so each
    feature's dw is orthogonal to its weights; dgain does not depend on whether a gain was given."""
    L, w, _ = _wn_inputs(7, 6, 8, 0.5, 10)
    dy = np.random.default_rng(11).standard_normal(w.shape)
    dw, dgain = o.l2_normalize_grad(L, 8, w, dy)
    dots = (o.densify(L, 8, dw) * o.densify(L, 8, w)).sum(axis=0)
    assert np.allclose(dots, 0.0, atol=1e-12)
    _, dgain1 = o.l2_normalize_grad(L, 8, w, dy, np.ones(6 * 8))
    assert np.array_equal(dgain, dgain1)


# --- SparseProj (README, "API Documentation: blocksparse.matmul", class SparseProj) ---

def _proj_inputs(N, nhidden, nproj, seed):
    rng = np.random.default_rng(seed)
    lut = rng.permutation(nhidden)[:nproj].astype(np.int32)       # distinct: one to one
    return lut, rng.standard_normal((N, nhidden)), rng.standard_normal((N, nproj))


def test_sparse_proj_hand_example():
    lut = [4, 1, 3]
    x = np.array([[10., 11., 12., 13., 14., 15.]])
    s = np.array([[2., 3., 5.]])
    assert np.array_equal(o.sparse_proj("gather", lut, x), [[14., 11., 13.]])
    assert np.array_equal(o.sparse_proj("scatter", lut, s, nhidden=6), [[0., 3., 0., 5., 2., 0.]])
    assert np.array_equal(o.sparse_proj("scatter_add", lut, x, s), [[10., 14., 12., 18., 16., 15.]])
    assert np.array_equal(o.sparse_proj("scatter_mul", lut, x, s), [[10., 33., 12., 65., 28., 15.]])
    assert np.array_equal(o.sparse_proj("gather_mul", lut, x, x), [[196., 121., 169.]])


def test_sparse_proj_default_lut():
    """Runs of block_size features, one every proj_stride features (the reading of the defaults)."""
    assert o.proj_default_lut(8, 6, 4).tolist() == [0, 1, 2, 3, 6, 7, 8, 9]
    assert o.proj_default_lut(6, 2, 2).tolist() == [0, 1, 2, 3, 4, 5]
    assert o.proj_default_lut(96, 64, 32).tolist() == list(range(32)) + list(range(64, 96)) + list(range(128, 160))


def test_sparse_proj_against_numpy_indexing():
    """Against numpy fancy indexing, a route independent of the oracle's loops."""
    lut, x, s = _proj_inputs(5, 40, 17, 1)
    assert np.array_equal(o.sparse_proj("gather", lut, x), x[:, lut])
    want = np.zeros((5, 40))
    want[:, lut] = s
    assert np.array_equal(o.sparse_proj("scatter", lut, s, nhidden=40), want)
    want = x.copy()
    want[:, lut] += s
    assert np.array_equal(o.sparse_proj("scatter_add", lut, x, s), want)
    want = x.copy()
    want[:, lut] *= s
    assert np.array_equal(o.sparse_proj("scatter_mul", lut, x, s), want)
    z = np.random.default_rng(2).standard_normal((5, 40))
    assert np.array_equal(o.sparse_proj("gather_mul", lut, x, z), x[:, lut] * z[:, lut])


def test_sparse_proj_adjoint_and_round_trips():
    """gather and scatter are adjoint (so each is the other's gradient, with no collisions to
    sum); scatter then gather is the identity; gather then scatter keeps only the mapped features."""
    lut, x, s = _proj_inputs(7, 33, 12, 3)
    g = o.sparse_proj("gather", lut, x)
    sc = o.sparse_proj("scatter", lut, s, nhidden=33)
    assert np.isclose((g * s).sum(), (x * sc).sum(), rtol=1e-13)
    assert np.array_equal(o.sparse_proj("gather", lut, sc), s)
    mask = np.zeros(33)
    mask[lut] = 1
    assert np.array_equal(o.sparse_proj("scatter", lut, g, nhidden=33), x * mask)


def test_sparse_proj_scatter_mul_gradient():
    """<dout, scatter_mul(x, y)> is affine in y with slope gather_mul(dout, x): the sparse-operand
    gradient of scatter_mul."""
    lut, x, s = _proj_inputs(4, 20, 9, 4)
    dout = np.random.default_rng(5).standard_normal((4, 20))
    f = lambda y: (dout * o.sparse_proj("scatter_mul", lut, x, y)).sum()
    gm = o.sparse_proj("gather_mul", lut, dout, x)
    d = np.random.default_rng(6).standard_normal(s.shape)
    assert np.isclose(f(s + d) - f(s), (gm * d).sum(), rtol=1e-12)


def test_sparse_proj_axis_layouts_agree():
    lut, x, s = _proj_inputs(6, 24, 10, 7)
    for op, a, b, kw in (("gather", x, None, {}), ("scatter", s, None, {"nhidden": 24}),
                         ("scatter_add", x, s, {}), ("scatter_mul", x, s, {}), ("gather_mul", x, x, {})):
        r1 = o.sparse_proj(op, lut, a, b, axis=1, **kw)
        r0 = o.sparse_proj(op, lut, a.T.copy(), None if b is None else b.T.copy(), axis=0, **kw)
        assert np.array_equal(r0, r1.T), op
