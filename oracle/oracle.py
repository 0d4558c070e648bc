"""Python face of the float64 CPU oracle (``bsmm_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA library.  Every function follows the blocksparse README, section
"API Documentation: blocksparse.matmul" (BlocksparseMatMul, block_coord,
identity_init, l2_normalize, __call__, group_param_grads, SparseProj), or its "blocksparse.norms" section
(layer_norm); the C file states the readings taken where the page is silent.

Inputs are numpy arrays; floating-point inputs are converted to float64
exactly (bf16/fp16/fp32 values widen without rounding).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsmm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_d = ctypes.POINTER(ctypes.c_double)
_u8 = ctypes.POINTER(ctypes.c_uint8)
_i32 = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.POINTER(ctypes.c_int64)
_c = ctypes.c_int
_l = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_nnz.restype = _l
        lib.oracle_nnz.argtypes = [_u8, _c, _c]
        lib.oracle_luts.argtypes = [_u8, _c, _c, _i32, _i32, _i32, _i32, _i32]
        lib.oracle_densify.argtypes = [_u8, _c, _c, _c, _d, _d]
        lib.oracle_identity_init.argtypes = [_u8, _c, _c, _c, _d]
        lib.oracle_fprop.argtypes = [_d, _d, _d, _c, _c, _c, _c, _c, _c, _c]
        lib.oracle_bprop.argtypes = [_d, _d, _d, _c, _c, _c, _c, _c, _c, _c]
        lib.oracle_updat.argtypes = [_u8, _c, _c, _c, _d, _d, _d, _c, _c, _c, _l, _l, _c]
        lib.oracle_updat_grouped.argtypes = [_u8, _c, _c, _c, ctypes.POINTER(_d), ctypes.POINTER(_d),
                                             _c, _d, _c, _c, _c, _c]
        lib.oracle_fprop_at.argtypes = [_u8, _c, _c, _c, _d, _d, _c, _c, _i64, _i64, _l, _d]
        lib.oracle_bprop_at.argtypes = [_u8, _c, _c, _c, _d, _d, _c, _c, _i64, _i64, _l, _d]
        lib.oracle_updat_at.argtypes = [_u8, _c, _c, _c, _d, _d, _c, _c, _i64, _i64, _i64, _l, _d]
        lib.oracle_layer_norm.argtypes = [_d, _d, _d, _d, _c, _c, _c, ctypes.c_double, _c]
        lib.oracle_layer_norm_grad.argtypes = [_d, _d, _d, _d, _d, _d, _d, _c, _c, _c, ctypes.c_double, _c]
        lib.oracle_l2_normalize.argtypes = [_u8, _c, _c, _c, _d, _d, ctypes.c_double, _d]
        lib.oracle_l2_normalize_grad.argtypes = [_u8, _c, _c, _c, _d, _d, ctypes.c_double, _d, _d, _d]
        lib.oracle_proj_default_lut.argtypes = [_c, _c, _c, _i32]
        lib.oracle_sparse_proj.argtypes = [_c, _d, _d, _d, _i32, _c, _c, _c, _c]
        lib.oracle_max_threads.restype = _c
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):            # torch tensor -> exact float64
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _lay(L) -> np.ndarray:
    L = np.ascontiguousarray(np.asarray(L) != 0, dtype=np.uint8)
    assert L.ndim == 2
    return L


def _p(a, t):
    return a.ctypes.data_as(t)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def nnz(L) -> int:
    L = _lay(L)
    return int(_load().oracle_nnz(_p(L, _u8), L.shape[0], L.shape[1]))


def luts(L):
    """(row_ptr, row_ent, col_ptr, col_ent, coord) as int32 arrays (see the C file)."""
    L = _lay(L)
    R, S = L.shape
    z = nnz(L)
    row_ptr = np.zeros(R + 1, np.int32)
    row_ent = np.zeros(max(z, 1), np.int32)
    col_ptr = np.zeros(S + 1, np.int32)
    col_ent = np.zeros(max(2 * z, 1), np.int32)
    coord = np.zeros(max(2 * z, 1), np.int32)
    _load().oracle_luts(_p(L, _u8), R, S, _p(row_ptr, _i32), _p(row_ent, _i32),
                        _p(col_ptr, _i32), _p(col_ent, _i32), _p(coord, _i32))
    return row_ptr, row_ent[:z], col_ptr, col_ent[:2 * z].reshape(z, 2), coord[:2 * z].reshape(z, 2)


def densify(L, bs: int, w) -> np.ndarray:
    L = _lay(L)
    R, S = L.shape
    w = _f64(w)
    assert w.size == nnz(L) * bs * bs
    Wd = np.zeros((R * bs, S * bs), np.float64)
    _load().oracle_densify(_p(L, _u8), R, S, bs, _p(w, _d), _p(Wd, _d))
    return Wd


def identity_init(L, bs: int) -> np.ndarray:
    L = _lay(L)
    w = np.zeros((nnz(L), bs, bs), np.float64)
    _load().oracle_identity_init(_p(L, _u8), L.shape[0], L.shape[1], bs, _p(w, _d))
    return w


def fprop(L, bs: int, x, w, feature_axis: int, rows=None, nthreads: int = 0) -> np.ndarray:
    """y = x . W.  x: (N,C) for feature_axis=1, (C,N) for 0.  `rows` = (n_lo, n_hi) subset."""
    L = _lay(L)
    R, S = L.shape
    C, K = R * bs, S * bs
    x = _f64(x)
    N = x.shape[0] if feature_axis == 1 else x.shape[1]
    Wd = densify(L, bs, w)
    y = np.zeros((N, K) if feature_axis == 1 else (K, N), np.float64)
    lo, hi = rows if rows is not None else (0, N)
    _load().oracle_fprop(_p(x, _d), _p(Wd, _d), _p(y, _d), N, C, K, feature_axis, lo, hi, nthreads)
    return y


def bprop(L, bs: int, dy, w, feature_axis: int, rows=None, nthreads: int = 0) -> np.ndarray:
    """dx = dy . W^T.  dy: (N,K) for feature_axis=1, (K,N) for 0."""
    L = _lay(L)
    R, S = L.shape
    C, K = R * bs, S * bs
    dy = _f64(dy)
    N = dy.shape[0] if feature_axis == 1 else dy.shape[1]
    Wd = densify(L, bs, w)
    dx = np.zeros((N, C) if feature_axis == 1 else (C, N), np.float64)
    lo, hi = rows if rows is not None else (0, N)
    _load().oracle_bprop(_p(dy, _d), _p(Wd, _d), _p(dx, _d), N, C, K, feature_axis, lo, hi, nthreads)
    return dx


def updat(L, bs: int, x, dy, feature_axis: int, dw_init=None, blocks=None, nthreads: int = 0) -> np.ndarray:
    """dw[b] = x[:, c_b-block]^T . dy[:, k_b-block] (+ dw_init when given)."""
    L = _lay(L)
    R, S = L.shape
    x, dy = _f64(x), _f64(dy)
    N = x.shape[0] if feature_axis == 1 else x.shape[1]
    z = nnz(L)
    acc = dw_init is not None
    dw = _f64(dw_init).reshape(z, bs, bs).copy() if acc else np.zeros((z, bs, bs), np.float64)
    lo, hi = blocks if blocks is not None else (0, z)
    _load().oracle_updat(_p(L, _u8), R, S, bs, _p(x, _d), _p(dy, _d), _p(dw, _d), N, feature_axis,
                         int(acc), lo, hi, nthreads)
    return dw


def updat_grouped(L, bs: int, xs, dys, feature_axis: int, dw_init=None, nthreads: int = 0) -> np.ndarray:
    """group_param_grads: sum over the G <= 8 timesteps of updat(x_t, dy_t) (+ dw_init)."""
    L = _lay(L)
    R, S = L.shape
    xs = [_f64(a) for a in xs]
    dys = [_f64(a) for a in dys]
    G = len(xs)
    assert G == len(dys) and G >= 1
    N = xs[0].shape[0] if feature_axis == 1 else xs[0].shape[1]
    z = nnz(L)
    acc = dw_init is not None
    dw = _f64(dw_init).reshape(z, bs, bs).copy() if acc else np.zeros((z, bs, bs), np.float64)
    xa = (_d * G)(*[_p(a, _d) for a in xs])
    da = (_d * G)(*[_p(a, _d) for a in dys])
    _load().oracle_updat_grouped(_p(L, _u8), R, S, bs, xa, da, G, _p(dw, _d), N, feature_axis,
                                 int(acc), nthreads)
    return dw


def fprop_at(L, bs: int, w, x, feature_axis: int, n_idx, f_idx) -> np.ndarray:
    """Sampled y[n, f] (activation coordinates, any feature_axis)."""
    L = _lay(L)
    x, w = _f64(x), _f64(w)
    N = x.shape[0] if feature_axis == 1 else x.shape[1]
    n_idx = np.ascontiguousarray(n_idx, np.int64)
    f_idx = np.ascontiguousarray(f_idx, np.int64)
    out = np.zeros(len(n_idx), np.float64)
    _load().oracle_fprop_at(_p(L, _u8), L.shape[0], L.shape[1], bs, _p(w, _d), _p(x, _d), N,
                            feature_axis, _p(n_idx, _i64), _p(f_idx, _i64), len(n_idx), _p(out, _d))
    return out


def bprop_at(L, bs: int, w, dy, feature_axis: int, n_idx, f_idx) -> np.ndarray:
    L = _lay(L)
    dy, w = _f64(dy), _f64(w)
    N = dy.shape[0] if feature_axis == 1 else dy.shape[1]
    n_idx = np.ascontiguousarray(n_idx, np.int64)
    f_idx = np.ascontiguousarray(f_idx, np.int64)
    out = np.zeros(len(n_idx), np.float64)
    _load().oracle_bprop_at(_p(L, _u8), L.shape[0], L.shape[1], bs, _p(w, _d), _p(dy, _d), N,
                            feature_axis, _p(n_idx, _i64), _p(f_idx, _i64), len(n_idx), _p(out, _d))
    return out


def updat_at(L, bs: int, x, dy, feature_axis: int, b_idx, i_idx, j_idx) -> np.ndarray:
    L = _lay(L)
    x, dy = _f64(x), _f64(dy)
    N = x.shape[0] if feature_axis == 1 else x.shape[1]
    b_idx = np.ascontiguousarray(b_idx, np.int64)
    i_idx = np.ascontiguousarray(i_idx, np.int64)
    j_idx = np.ascontiguousarray(j_idx, np.int64)
    out = np.zeros(len(b_idx), np.float64)
    _load().oracle_updat_at(_p(L, _u8), L.shape[0], L.shape[1], bs, _p(x, _d), _p(dy, _d), N,
                            feature_axis, _p(b_idx, _i64), _p(i_idx, _i64), _p(j_idx, _i64),
                            len(b_idx), _p(out, _d))
    return out


def layer_norm(x, g, b, axis: int = 1, epsilon: float = 1e-6, relu: bool = False) -> np.ndarray:
    """layer_norm of the README's "blocksparse.norms" section (the readings are stated in the
    C source): x is (N, C) for axis = 1 or (C, N) for axis = 0; g, b have C entries."""
    x, g, b = _f64(x), _f64(g).reshape(-1), _f64(b).reshape(-1)
    assert x.ndim == 2 and axis in (0, 1)
    C = x.shape[1] if axis == 1 else x.shape[0]
    N = x.shape[0] if axis == 1 else x.shape[1]
    assert g.size == C and b.size == C
    y = np.empty_like(x)
    _load().oracle_layer_norm(_p(x, _d), _p(g, _d), _p(b, _d), _p(y, _d), N, C, axis, float(epsilon), int(relu))
    return y


def layer_norm_grad(x, g, dy, y=None, axis: int = 1, epsilon: float = 1e-6, relu: bool = False):
    """Gradient of layer_norm with respect to (x, g, b) for the output gradient dy; with relu the
    mask is y > 0 for the forward output y (readings in the C source).  Returns (dx, dg, db)."""
    x, g, dy = _f64(x), _f64(g).reshape(-1), _f64(dy)
    assert x.ndim == 2 and axis in (0, 1) and dy.shape == x.shape
    C = x.shape[1] if axis == 1 else x.shape[0]
    N = x.shape[0] if axis == 1 else x.shape[1]
    assert g.size == C
    yv = _f64(y) if relu else np.zeros_like(x)
    assert yv.shape == x.shape
    dx = np.empty_like(x)
    dg, db = np.empty(C), np.empty(C)
    _load().oracle_layer_norm_grad(_p(x, _d), _p(yv, _d), _p(g, _d), _p(dy, _d), _p(dx, _d), _p(dg, _d),
                                   _p(db, _d), N, C, axis, float(epsilon), int(relu))
    return dx, dg, db


def _gain(gain, S: int, bs: int):
    if gain is None:
        return None
    g = _f64(gain).reshape(-1)
    assert g.size == S * bs
    return g


def l2_normalize(L, bs: int, w, gain=None, epsilon: float = 1e-6) -> np.ndarray:
    """BlocksparseMatMul.l2_normalize (README, "API Documentation: blocksparse.matmul"): each
    output feature's incoming weights, over every block of its block column, scaled to unit L2
    norm (squared norm bounded below by epsilon) and multiplied by gain[f] (K values, or 1)."""
    L = _lay(L)
    w = _f64(w)
    assert w.shape == (nnz(L), bs, bs)
    g = _gain(gain, L.shape[1], bs)
    y = np.empty_like(w)
    _load().oracle_l2_normalize(_p(L, _u8), L.shape[0], L.shape[1], bs, _p(w, _d),
                                None if g is None else _p(g, _d), float(epsilon), _p(y, _d))
    return y


def l2_normalize_grad(L, bs: int, w, dy, gain=None, epsilon: float = 1e-6):
    """Gradient of l2_normalize: (dw, dgain) for the upstream gradient dy of its output; dgain
    has one entry per output feature (the derivative with respect to gain, also without one)."""
    L = _lay(L)
    w, dy = _f64(w), _f64(dy)
    assert w.shape == (nnz(L), bs, bs) and dy.shape == w.shape
    g = _gain(gain, L.shape[1], bs)
    dw = np.empty_like(w)
    dgain = np.empty(L.shape[1] * bs)
    _load().oracle_l2_normalize_grad(_p(L, _u8), L.shape[0], L.shape[1], bs, _p(w, _d),
                                     None if g is None else _p(g, _d), float(epsilon), _p(dy, _d),
                                     _p(dw, _d), _p(dgain, _d))
    return dw, dgain


PROJ_OPS = {"gather": 0, "scatter": 1, "scatter_add": 2, "scatter_mul": 3, "gather_mul": 4}


def proj_default_lut(nproj: int, proj_stride: int, block_size: int) -> np.ndarray:
    """SparseProj's map without gather_lut (README, class SparseProj; the reading is stated in
    the C source): runs of block_size features, one starting every proj_stride features."""
    lut = np.empty(nproj, np.int32)
    _load().oracle_proj_default_lut(nproj, proj_stride, block_size, _p(lut, _i32))
    return lut


def sparse_proj(op: str, lut, x, y=None, nhidden: int = None, axis: int = 1) -> np.ndarray:
    """SparseProj.gather / scatter / scatter_add / scatter_mul (and gather_mul, the sparse-operand
    gradient of scatter_mul), float64.  Activations are (N, F) for axis = 1, (F, N) for axis = 0;
    x is dense (nhidden features) except for scatter, whose x is sparse (nproj features)."""
    lut = np.ascontiguousarray(lut, dtype=np.int32)
    x = _f64(x)
    nproj = lut.size
    N = x.shape[0] if axis == 1 else x.shape[1]
    if op == "scatter":
        assert nhidden is not None
    else:
        nhidden = x.shape[1] if axis == 1 else x.shape[0]
    dense = (N, nhidden) if axis == 1 else (nhidden, N)
    sparse = (N, nproj) if axis == 1 else (nproj, N)
    yv = _f64(y) if y is not None else np.zeros(1)
    out = np.empty(sparse if op in ("gather", "gather_mul") else dense)
    _load().oracle_sparse_proj(PROJ_OPS[op], _p(x, _d), _p(yv, _d), _p(out, _d), _p(lut, _i32), N, nhidden,
                               nproj, axis)
    return out
