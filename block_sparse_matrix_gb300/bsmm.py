"""Thin ctypes binding of libbsmm (include/bsmm.h).

Argument marshalling only: every step of every pass runs in the CUDA library.
Torch tensors supply device memory and the current stream.  There is no CPU
fallback: if libbsmm.so is missing or fails to load, every call raises.

Module-level functions carry the C names (bsmm_create, bsmm_fprop, ...);
``BlocksparseMatMul`` wraps them with the shape helpers of the blocksparse
README ("API Documentation: blocksparse.matmul": w_shape, i_shape, o_shape,
block_coord, identity_init, __call__) and of group_param_grads.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsmm.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_ALIGN, ERR_CUDA, ERR_TIMEOUT, ERR_OOM, ERR_BOUNDS = range(8)
F32, F16, BF16 = 0, 1, 2
KERNELS = {"auto": 0, "simt": 1, "tc": 2}
_DT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

_lib = None


class BsmmError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s (status %d)" % (what, status_string(code), code))


def lib():
    """Load libbsmm.so (build it first with __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libbsmm.so not built at %s; run block_sparse_matrix_gb300/build.py" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        pi, pi64, pi32 = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
        sig = {
            "bsmm_create": [ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_uint8), i, i, i, i, vp],
            "bsmm_destroy": [vp],
            "bsmm_w_shape": [vp, pi64, pi],
            "bsmm_layout_info": [vp, pi, pi, pi],
            "bsmm_block_coord": [vp, i64, pi, pi],
            "bsmm_get_luts": [vp, pi32, pi32, pi32, pi32, pi32],
            "bsmm_identity_init": [vp, vp, i, vp],
            "bsmm_fprop": [vp, vp, vp, vp, i, i, vp],
            "bsmm_bprop": [vp, vp, vp, vp, i, i, vp],
            "bsmm_updat": [vp, vp, vp, vp, i, i, i, i, vp],
            "bsmm_updat_grouped": [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), i, i, i, vp, i, vp],
            "bsmm_set_kernel": [vp, i],
            "bsmm_sync_status": [vp, vp],
            "bsmm_selftest_wait_timeout": [vp, ctypes.c_uint64, vp],
            "bsmm_selftest_empty_launch": [vp, ctypes.c_int, ctypes.c_int, vp],
            "bsmm_updat_noalloc": [vp, vp, vp, vp, i, i, i, vp],
            "bsmm_layer_norm": [vp, vp, vp, vp, i, i, i, ctypes.c_float, i, i, vp],
            "bsmm_layer_norm_grad": [vp, vp, vp, vp, vp, vp, vp, i, i, i, ctypes.c_float, i, i, vp,
                                     ctypes.c_size_t, vp],
            "bsmm_l2_normalize": [vp, vp, vp, vp, ctypes.c_float, i, vp],
            "bsmm_l2_normalize_grad": [vp, vp, vp, vp, vp, vp, ctypes.c_float, i, vp],
            "bsmm_proj_create": [ctypes.POINTER(vp), i, i, i, i, pi32],
            "bsmm_proj_destroy": [vp],
            "bsmm_proj_info": [vp, pi, pi],
            "bsmm_proj_get_lut": [vp, pi32],
            "bsmm_proj": [vp, i, vp, vp, vp, i, i, i, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.bsmm_status_string.argtypes = [ctypes.c_int]
        L.bsmm_status_string.restype = ctypes.c_char_p
        L.bsmm_layer_norm_grad_workspace.argtypes = [i, i, i]
        L.bsmm_layer_norm_grad_workspace.restype = ctypes.c_size_t
        L.bsmm_launch_count.argtypes = []
        L.bsmm_launch_count.restype = ctypes.c_int64
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().bsmm_status_string(code).decode()


def launch_count() -> int:
    return int(lib().bsmm_launch_count())


def _check(code, what):
    if code != OK:
        raise BsmmError(code, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _want(t, what, shape, dtype=None, device=None):
    """A caller's tensor must have exactly the shape (and dtype, device) the call reads or writes:
    the C calls see only pointers, so a mismatch would read or write outside the tensor."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (what, tuple(shape), tuple(t.shape)))
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if t.dtype not in _DT:
        raise ValueError("%s has unsupported dtype %s" % (what, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s must be on %s, got %s" % (what, device, t.device))
    _dev(t, what)


def _dev(t, what):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)


# ---- C-named wrappers --------------------------------------------------------------

def bsmm_create(layout, block_size: int = 32, feature_axis: int = 1, stream=None):
    lay = np.ascontiguousarray(np.asarray(layout) != 0, dtype=np.uint8)
    if lay.ndim != 2:
        raise ValueError("layout must be 2-D")
    h = ctypes.c_void_p()
    _check(lib().bsmm_create(ctypes.byref(h), lay.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                             lay.shape[0], lay.shape[1], block_size, feature_axis, _stream(stream)),
           "bsmm_create")
    return h


def bsmm_destroy(h):
    _check(lib().bsmm_destroy(h), "bsmm_destroy")


def bsmm_identity_init(h, w, stream=None):
    _dev(w, "w")
    _check(lib().bsmm_identity_init(h, _ptr(w), _DT[w.dtype], _stream(stream)), "bsmm_identity_init")


def bsmm_fprop(h, x, w, y, N: int, stream=None):
    _check(lib().bsmm_fprop(h, _ptr(x), _ptr(w), _ptr(y), N, _DT[x.dtype], _stream(stream)), "bsmm_fprop")


def bsmm_bprop(h, dy, w, dx, N: int, stream=None):
    _check(lib().bsmm_bprop(h, _ptr(dy), _ptr(w), _ptr(dx), N, _DT[dy.dtype], _stream(stream)), "bsmm_bprop")


def bsmm_updat(h, x, dy, dw, N: int, accumulate: bool = False, stream=None):
    _check(lib().bsmm_updat(h, _ptr(x), _ptr(dy), _ptr(dw), N, _DT[x.dtype], _DT[dw.dtype], int(accumulate),
                            _stream(stream)), "bsmm_updat")


def bsmm_updat_grouped(h, xs, dys, dw, N: int, accumulate: bool = False, stream=None):
    G = len(xs)
    xa = (ctypes.c_void_p * max(G, 1))(*[t.data_ptr() for t in xs])
    da = (ctypes.c_void_p * max(G, 1))(*[t.data_ptr() for t in dys])
    dt = _DT[xs[0].dtype] if G else F32
    _check(lib().bsmm_updat_grouped(h, xa, da, G, N, dt, _ptr(dw), int(accumulate), _stream(stream)),
           "bsmm_updat_grouped")


def _handle_shapes(h):
    """(nnz, bs, C, K, feature_axis) of a handle, read through the C ABI."""
    nnz, bs = ctypes.c_int64(), ctypes.c_int()
    R, S, fa = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().bsmm_w_shape(h, ctypes.byref(nnz), ctypes.byref(bs)), "bsmm_w_shape")
    _check(lib().bsmm_layout_info(h, ctypes.byref(R), ctypes.byref(S), ctypes.byref(fa)), "bsmm_layout_info")
    return int(nnz.value), bs.value, R.value * bs.value, S.value * bs.value, fa.value


def bsmm_updat_noalloc(h, x, dy, dw, N: int, accumulate: bool = False, stream=None):
    """Weight gradient that allocates no device memory (see include/bsmm.h): for callers
    whose allocator or memory budget forbids cudaMalloc.  x and dy are 16-bit activations
    of minibatch N in the handle's layout, dw is float32 (nnz, bs, bs) on the same device:
    the C call sees only pointers, so every shape is checked here first."""
    nnz, bs, C, K, fa = _handle_shapes(h)
    act = (lambda F: (N, F)) if fa == 1 else (lambda F: (F, N))
    _dev(x, "x")
    _want(x, "x", act(C), None, x.device)
    _want(dy, "dy", act(K), x.dtype, x.device)
    _want(dw, "dw", (nnz, bs, bs), torch.float32, x.device)
    _check(lib().bsmm_updat_noalloc(h, _ptr(x), _ptr(dy), _ptr(dw), N, _DT[x.dtype], int(accumulate),
                                    _stream(stream)), "bsmm_updat_noalloc")


def bsmm_l2_normalize(h, w, gain, y, epsilon: float = 1e-6, stream=None):
    _check(lib().bsmm_l2_normalize(h, _ptr(w), _ptr(gain), _ptr(y), float(epsilon), _DT[y.dtype], _stream(stream)),
           "bsmm_l2_normalize")


def bsmm_l2_normalize_grad(h, w, gain, dy, dw, dgain, epsilon: float = 1e-6, stream=None):
    _check(lib().bsmm_l2_normalize_grad(h, _ptr(w), _ptr(gain), _ptr(dy), _ptr(dw), _ptr(dgain), float(epsilon),
                                        _DT[dy.dtype], _stream(stream)), "bsmm_l2_normalize_grad")


def bsmm_sync_status(h, stream=None):
    _check(lib().bsmm_sync_status(h, _stream(stream)), "bsmm_sync_status")


def bsmm_selftest_wait_timeout(h, limit_ns: int, stream=None):
    _check(lib().bsmm_selftest_wait_timeout(h, int(limit_ns), _stream(stream)), "bsmm_selftest_wait_timeout")


def bsmm_selftest_empty_launch(h, ctas: int, tensor_memory: bool, stream=None):
    _check(lib().bsmm_selftest_empty_launch(h, int(ctas), int(bool(tensor_memory)), _stream(stream)),
           "bsmm_selftest_empty_launch")


# ---- README-style object -------------------------------------------------------------

class BlocksparseMatMul:
    """BlocksparseMatMul(layout, block_size=32, feature_axis=1) on the current CUDA device."""

    def __init__(self, layout, block_size: int = 32, feature_axis: int = 1):
        self.layout = np.ascontiguousarray(np.asarray(layout) != 0, dtype=np.uint8)
        self.block_size = block_size
        self.feature_axis = feature_axis
        self._h = bsmm_create(self.layout, block_size, feature_axis)
        nnz = ctypes.c_int64()
        bs = ctypes.c_int()
        _check(lib().bsmm_w_shape(self._h, ctypes.byref(nnz), ctypes.byref(bs)), "bsmm_w_shape")
        self.nnz = int(nnz.value)
        self.C = self.layout.shape[0] * block_size
        self.K = self.layout.shape[1] * block_size

    def close(self):
        if getattr(self, "_h", None):
            bsmm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # shape helpers
    @property
    def w_shape(self):
        return (self.nnz, self.block_size, self.block_size)

    def i_shape(self, N):
        return (N, self.C) if self.feature_axis == 1 else (self.C, N)

    def o_shape(self, N):
        return (N, self.K) if self.feature_axis == 1 else (self.K, N)

    def _N(self, a, F):
        if a.dim() != 2:
            raise ValueError("activations must be 2-D")
        if self.feature_axis == 1:
            if a.shape[1] != F:
                raise ValueError("activation shape %s does not match feature size %d" % (tuple(a.shape), F))
            return a.shape[0]
        if a.shape[0] != F:
            raise ValueError("activation shape %s does not match feature size %d" % (tuple(a.shape), F))
        return a.shape[1]

    def block_coord(self, block: int):
        c, k = ctypes.c_int(), ctypes.c_int()
        _check(lib().bsmm_block_coord(self._h, int(block), ctypes.byref(c), ctypes.byref(k)), "bsmm_block_coord")
        return c.value, k.value

    def get_luts(self):
        R, S = self.layout.shape
        z = max(self.nnz, 1)
        row_ptr = np.zeros(R + 1, np.int32)
        col_ptr = np.zeros(S + 1, np.int32)
        row_ent = np.zeros(z, np.int32)
        col_ent = np.zeros(2 * z, np.int32)
        coord = np.zeros(2 * z, np.int32)
        p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        _check(lib().bsmm_get_luts(self._h, p(row_ptr), p(row_ent), p(col_ptr), p(col_ent), p(coord)),
               "bsmm_get_luts")
        n = self.nnz
        return row_ptr, row_ent[:n], col_ptr, col_ent[:2 * n].reshape(n, 2), coord[:2 * n].reshape(n, 2)

    def set_kernel(self, which: str):
        _check(lib().bsmm_set_kernel(self._h, KERNELS[which]), "bsmm_set_kernel")

    def sync_status(self, stream=None):
        bsmm_sync_status(self._h, stream)

    def identity_init(self, w=None, dtype=torch.float32, device="cuda"):
        if w is None:
            w = torch.empty(self.w_shape, dtype=dtype, device=device)
        _want(w, "w", self.w_shape)
        bsmm_identity_init(self._h, w)
        return w

    def _wn_args(self, w, gain):
        _want(w, "w", self.w_shape, torch.float32)
        if gain is not None:
            _want(gain, "gain", (self.K,), torch.float32, w.device)

    def l2_normalize(self, w, gain=None, epsilon=1e-6, dtype=torch.float32, y=None, stream=None):
        """Weight normalisation (README: l2_normalize(W, gain=None, epsilon=1e-6, dtype)): every
        output feature's incoming weights scaled to unit L2 norm (squared norm at least epsilon),
        times gain[f]; returned in dtype.  y may be w for float32."""
        self._wn_args(w, gain)
        if y is None:
            y = torch.empty(self.w_shape, dtype=dtype, device=w.device)
        _want(y, "y", self.w_shape, None, w.device)
        bsmm_l2_normalize(self._h, w, gain, y, epsilon, stream)
        return y

    def l2_normalize_grad(self, w, dy, gain=None, epsilon=1e-6, dw=None, dgain=None, stream=None):
        """(dw, dgain): gradient of l2_normalize for the gradient dy of its output (dy in the
        output's dtype, dw and dgain float32; dgain has K values)."""
        self._wn_args(w, gain)
        _want(dy, "dy", self.w_shape, None, w.device)
        if dw is None:
            dw = torch.empty(self.w_shape, dtype=torch.float32, device=w.device)
        if dgain is None:
            dgain = torch.empty(self.K, dtype=torch.float32, device=w.device)
        _want(dw, "dw", self.w_shape, torch.float32, w.device)
        _want(dgain, "dgain", (self.K,), torch.float32, w.device)
        bsmm_l2_normalize_grad(self._h, w, gain, dy, dw, dgain, epsilon, stream)
        return dw, dgain

    def fprop(self, x, w, y=None, stream=None):
        _dev(x, "x")
        N = self._N(x, self.C)
        _want(w, "w", self.w_shape, x.dtype, x.device)
        if y is None:
            y = torch.empty(self.o_shape(N), dtype=x.dtype, device=x.device)
        _want(y, "y", self.o_shape(N), x.dtype, x.device)
        bsmm_fprop(self._h, x, w, y, N, stream)
        return y

    __call__ = fprop

    def bprop(self, dy, w, dx=None, stream=None):
        _dev(dy, "dy")
        N = self._N(dy, self.K)
        _want(w, "w", self.w_shape, dy.dtype, dy.device)
        if dx is None:
            dx = torch.empty(self.i_shape(N), dtype=dy.dtype, device=dy.device)
        _want(dx, "dx", self.i_shape(N), dy.dtype, dy.device)
        bsmm_bprop(self._h, dy, w, dx, N, stream)
        return dx

    def updat(self, x, dy, dw=None, accumulate=False, dw_dtype=torch.float32, stream=None):
        _dev(x, "x")
        _dev(dy, "dy")
        N = self._N(x, self.C)
        if self._N(dy, self.K) != N:
            raise ValueError("x and dy minibatch sizes differ")
        _want(dy, "dy", self.o_shape(N), x.dtype, x.device)
        if dw is None:
            dw = torch.empty(self.w_shape, dtype=dw_dtype, device=x.device)
        _want(dw, "dw", self.w_shape, None, x.device)
        bsmm_updat(self._h, x, dy, dw, N, accumulate, stream)
        return dw

    def updat_noalloc(self, x, dy, dw=None, accumulate=False, stream=None):
        """updat with dw_dtype float32 through bsmm_updat_noalloc: the library allocates no
        device memory for it (dw is allocated here only when not given)."""
        _dev(x, "x")
        _dev(dy, "dy")
        N = self._N(x, self.C)
        if self._N(dy, self.K) != N:
            raise ValueError("x and dy minibatch sizes differ")
        if dw is None:
            dw = torch.empty(self.w_shape, dtype=torch.float32, device=x.device)
        bsmm_updat_noalloc(self._h, x, dy, dw, N, accumulate, stream)
        return dw

    def updat_grouped(self, xs, dys, dw=None, accumulate=False, stream=None):
        if len(xs) != len(dys) or not 1 <= len(xs) <= 8:
            raise ValueError("need 1..8 (x, dy) pairs")
        for a in list(xs) + list(dys):
            _dev(a, "activation")
        N = self._N(xs[0], self.C)
        x0 = xs[0]
        for a in xs:
            _want(a, "x", self.i_shape(N), x0.dtype, x0.device)
        for a in dys:
            _want(a, "dy", self.o_shape(N), x0.dtype, x0.device)
        if dw is None:
            dw = torch.empty(self.w_shape, dtype=torch.float32, device=x0.device)
        _want(dw, "dw", self.w_shape, torch.float32, x0.device)
        bsmm_updat_grouped(self._h, xs, dys, dw, N, accumulate, stream)
        return dw


def group_param_grads(bsmm: BlocksparseMatMul, xs, dys, group_size: int = 8, dw=None, accumulate=False):
    """Sum of the weight gradients of all timesteps (x_t, dy_t) sharing one weight,
    computed group_size (<= 8) timesteps per call into one float32 dW."""
    if not 1 <= group_size <= 8:
        raise ValueError("group_size must be in 1..8")
    for g0 in range(0, len(xs), group_size):
        dw = bsmm.updat_grouped(xs[g0:g0 + group_size], dys[g0:g0 + group_size], dw=dw,
                                accumulate=accumulate or g0 > 0)
    return dw


def bsmm_layer_norm(x, g, b, y, N: int, C: int, axis: int = 1, epsilon: float = 1e-6, relu: bool = False,
                    stream=None):
    _check(lib().bsmm_layer_norm(_ptr(x), _ptr(g), _ptr(b), _ptr(y), N, C, axis, float(epsilon), int(relu),
                                 _DT[x.dtype], _stream(stream)), "bsmm_layer_norm")


def layer_norm(x, g, b, axis: int = 1, epsilon: float = 1e-6, relu: bool = False, y=None, stream=None):
    """layer_norm(x, g, b, axis=1, epsilon=1e-6, relu=False) of the README's
    "blocksparse.norms" section: x is (N, C) for axis = 1 or (C, N) for axis = 0 (the
    matmul's feature_axis), g and b are float32 vectors of C values; returns y (x's dtype).
    y may be x (in place)."""
    for t, what in ((x, "x"), (g, "g"), (b, "b")):
        _dev(t, what)
    if x.dim() != 2 or axis not in (0, 1):
        raise ValueError("x must be 2-D and axis 0 or 1")
    C = x.shape[1] if axis == 1 else x.shape[0]
    N = x.shape[0] if axis == 1 else x.shape[1]
    if g.dtype != torch.float32 or b.dtype != torch.float32 or g.numel() != C or b.numel() != C:
        raise ValueError("g and b must be float32 with C = %d values" % C)
    if g.device != x.device or b.device != x.device:
        raise ValueError("g and b must be on %s" % x.device)
    if y is None:
        y = torch.empty_like(x)
    _want(y, "y", x.shape, x.dtype, x.device)
    bsmm_layer_norm(x, g, b, y, N, C, axis, epsilon, relu, stream)
    return y


def bsmm_layer_norm_grad(x, y, g, dy, dx, dg, db, N: int, C: int, axis: int, epsilon: float, relu: bool,
                         workspace, stream=None):
    _check(lib().bsmm_layer_norm_grad(_ptr(x), _ptr(y) if y is not None else None, _ptr(g), _ptr(dy), _ptr(dx),
                                      _ptr(dg), _ptr(db), N, C, axis, float(epsilon), int(relu), _DT[x.dtype],
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "bsmm_layer_norm_grad")


def layer_norm_grad(x, g, dy, y=None, axis: int = 1, epsilon: float = 1e-6, relu: bool = False, dx=None,
                    stream=None):
    """Gradient of layer_norm(x, g, b, axis, epsilon, relu) for the output gradient dy: returns
    (dx, dg, db), dx in x's dtype, dg and db float32 vectors of C values.  With relu the forward
    output y is needed (the gradient passes where y > 0).  dx must not share memory with x, y or
    dy (they are read again after dx is written)."""
    for t, what in ((x, "x"), (g, "g"), (dy, "dy")):
        _dev(t, what)
    if x.dim() != 2 or axis not in (0, 1):
        raise ValueError("x must be 2-D and axis 0 or 1")
    C = x.shape[1] if axis == 1 else x.shape[0]
    N = x.shape[0] if axis == 1 else x.shape[1]
    if g.dtype != torch.float32 or g.numel() != C or g.device != x.device:
        raise ValueError("g must be float32 with C = %d values on %s" % (C, x.device))
    _want(dy, "dy", x.shape, x.dtype, x.device)
    if relu:
        if y is None:
            raise ValueError("relu needs the forward output y")
        _want(y, "y", x.shape, x.dtype, x.device)
    else:
        y = None
    if dx is None:
        dx = torch.empty_like(x)
    _want(dx, "dx", x.shape, x.dtype, x.device)
    if any(t is not None and t.data_ptr() == dx.data_ptr() for t in (x, y, dy)) and dx.numel() > 0:
        raise ValueError("dx must not share memory with x, y or dy")
    dg = torch.empty(C, dtype=torch.float32, device=x.device)
    db = torch.empty(C, dtype=torch.float32, device=x.device)
    nbytes = int(lib().bsmm_layer_norm_grad_workspace(N, C, axis))
    ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device=x.device)
    bsmm_layer_norm_grad(x, y, g, dy, dx, dg, db, N, C, axis, epsilon, relu, ws, stream)
    return dx, dg, db


# ---- SparseProj -------------------------------------------------------------------------

PROJ_OPS = {"gather": 0, "scatter": 1, "scatter_add": 2, "scatter_mul": 3, "gather_mul": 4}


def bsmm_proj_create(nhidden: int, nproj=None, proj_stride=None, block_size: int = 32, gather_lut=None):
    h = ctypes.c_void_p()
    lut = None
    if gather_lut is not None:
        lut = np.ascontiguousarray(np.asarray(gather_lut), dtype=np.int32).reshape(-1)
        nproj = lut.size
    _check(lib().bsmm_proj_create(ctypes.byref(h), int(nhidden), int(nproj or 0), int(proj_stride or 0),
                                  int(block_size), None if lut is None else
                                  lut.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))), "bsmm_proj_create")
    return h


def bsmm_proj_destroy(h):
    _check(lib().bsmm_proj_destroy(h), "bsmm_proj_destroy")


def bsmm_proj(h, op: str, x, y, out, N: int, axis: int = 1, stream=None):
    _check(lib().bsmm_proj(h, PROJ_OPS[op], _ptr(x), _ptr(y), _ptr(out), int(N), int(axis), _DT[x.dtype],
                           _stream(stream)), "bsmm_proj")


class SparseProj:
    """SparseProj(nhidden, nproj=None, proj_stride=None, block_size=32, gather_lut=None) of the
    README ("API Documentation: blocksparse.matmul"): dense <-> sparse feature projections over a
    one-to-one map.  Sparse feature p is dense feature lut[p]; without gather_lut the map keeps
    runs of block_size features, one run every proj_stride (default block_size) features.
    Activations are (N, F) for feature_axis = 1 and (F, N) for feature_axis = 0."""

    def __init__(self, nhidden, nproj=None, proj_stride=None, block_size=32, gather_lut=None, feature_axis=1):
        if feature_axis not in (0, 1):
            raise ValueError("feature_axis must be 0 or 1")
        self.feature_axis = feature_axis
        self._h = bsmm_proj_create(nhidden, nproj, proj_stride, block_size, gather_lut)
        a, b = ctypes.c_int(), ctypes.c_int()
        _check(lib().bsmm_proj_info(self._h, ctypes.byref(a), ctypes.byref(b)), "bsmm_proj_info")
        self.nhidden, self.nproj = a.value, b.value

    def close(self):
        if getattr(self, "_h", None):
            bsmm_proj_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def lut(self):
        out = np.empty(self.nproj, np.int32)
        _check(lib().bsmm_proj_get_lut(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
               "bsmm_proj_get_lut")
        return out

    def _n(self, a, F, what):
        _dev(a, what)
        if a.dim() != 2:
            raise ValueError("%s must be 2-D" % what)
        f, n = (a.shape[1], a.shape[0]) if self.feature_axis == 1 else (a.shape[0], a.shape[1])
        if f != F:
            raise ValueError("%s has %d features, expected %d" % (what, f, F))
        return n

    def _shape(self, N, F):
        return (N, F) if self.feature_axis == 1 else (F, N)

    def _run(self, op, x, y, out, N, stream):
        bsmm_proj(self._h, op, x, y, out, N, self.feature_axis, stream)
        return out

    def _out(self, out, x, N, F):
        if out is None:
            return torch.empty(self._shape(N, F), dtype=x.dtype, device=x.device)
        _want(out, "out", self._shape(N, F), x.dtype, x.device)
        return out

    def _operand(self, y, x, N, F):
        _want(y, "y", self._shape(N, F), x.dtype, x.device)

    def gather(self, x, out=None, stream=None):
        N = self._n(x, self.nhidden, "x")
        return self._run("gather", x, None, self._out(out, x, N, self.nproj), N, stream)

    def scatter(self, x, out=None, stream=None):
        N = self._n(x, self.nproj, "x")
        return self._run("scatter", x, None, self._out(out, x, N, self.nhidden), N, stream)

    def scatter_add(self, x, y, out=None, stream=None):
        """x (dense) with y (sparse) added at the mapped features; out may be x (in place)."""
        N = self._n(x, self.nhidden, "x")
        self._operand(y, x, N, self.nproj)
        return self._run("scatter_add", x, y, self._out(out, x, N, self.nhidden), N, stream)

    def scatter_mul(self, x, y, out=None, stream=None):
        """x (dense) with its mapped features multiplied by y (sparse); out may be x (in place)."""
        N = self._n(x, self.nhidden, "x")
        self._operand(y, x, N, self.nproj)
        return self._run("scatter_mul", x, y, self._out(out, x, N, self.nhidden), N, stream)

    def gather_mul(self, x, y, out=None, stream=None):
        """gather(x) * gather(y) for two dense operands, in one pass."""
        N = self._n(x, self.nhidden, "x")
        self._operand(y, x, N, self.nhidden)
        return self._run("gather_mul", x, y, self._out(out, x, N, self.nproj), N, stream)

    # Gradients: with a one-to-one map gather and scatter are each other's adjoint.
    def gather_grad(self, dy):
        return self.scatter(dy)

    def scatter_grad(self, dout):
        return self.gather(dout)

    def scatter_add_grad(self, dout):
        """(dx, dy) of scatter_add(x, y)."""
        return dout, self.gather(dout)

    def scatter_mul_grad(self, dout, x, y):
        """(dx, dy) of scatter_mul(x, y)."""
        return self.scatter_mul(dout, y), self.gather_mul(dout, x)
