"""The C-ABI library loads, exports every symbol include/bsmm.h declares, and
rejects bad arguments on the host (no GPU needed: these checks run before any
CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

from block_sparse_matrix_gb300 import bsmm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "bsmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsmm_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("bsmm_create", "bsmm_destroy", "bsmm_fprop", "bsmm_bprop", "bsmm_updat",
                     "bsmm_updat_grouped", "bsmm_identity_init", "bsmm_block_coord", "bsmm_w_shape",
                     "bsmm_get_luts", "bsmm_sync_status", "bsmm_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(bsmm.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings():
    for code in range(8):
        assert bsmm.status_string(code)
    assert "align" in bsmm.status_string(bsmm.ERR_ALIGN)


def _create(layout, bs, fa, R=None, S=None):
    L = bsmm.lib()
    lay = np.ascontiguousarray(layout, dtype=np.uint8)
    h = ctypes.c_void_p()
    R = lay.shape[0] if R is None else R
    S = lay.shape[1] if S is None else S
    return L.bsmm_create(ctypes.byref(h), lay.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), R, S, bs, fa, None)


def test_create_rejects_bad_arguments_on_host():
    lay = np.ones((2, 2), np.uint8)
    assert _create(lay, 12, 1) == bsmm.ERR_UNSUPPORTED        # block size not in {32,16,8}
    assert _create(lay, 64, 1) == bsmm.ERR_UNSUPPORTED
    assert _create(lay, 32, 2) == bsmm.ERR_INVALID            # feature_axis not 0/1
    assert _create(lay, 32, 1, R=0) == bsmm.ERR_INVALID
    assert _create(lay, 32, 1, S=-1) == bsmm.ERR_INVALID
    L = bsmm.lib()
    assert L.bsmm_create(None, None, 2, 2, 32, 1, None) == bsmm.ERR_INVALID


def test_null_handle_rejected():
    L = bsmm.lib()
    assert L.bsmm_fprop(None, None, None, None, 4, 0, None) == bsmm.ERR_INVALID
    assert L.bsmm_updat_grouped(None, None, None, 1, 4, 0, None, 0, None) == bsmm.ERR_INVALID
    assert L.bsmm_destroy(None) == bsmm.OK
    assert L.bsmm_set_kernel(None, 0) == bsmm.ERR_INVALID


def test_selftest_rejects_bad_arguments_on_host():
    L = bsmm.lib()
    assert L.bsmm_selftest_wait_timeout(None, 1000, None) == bsmm.ERR_INVALID
    assert L.bsmm_selftest_empty_launch(None, 1, 1, None) == bsmm.ERR_INVALID


def test_layer_norm_rejects_bad_arguments_on_host():
    """Every case fails validation before anything is enqueued (the pointers are never used)."""
    L = bsmm.lib()
    A, B = 0x10000, 0x20000                     # 16-byte aligned stand-ins, never dereferenced
    assert L.bsmm_layer_norm(None, A, A, A, 4, 8, 1, 1e-6, 0, 2, None) == bsmm.ERR_INVALID
    assert L.bsmm_layer_norm(None, None, None, None, 0, 8, 1, 1e-6, 0, 2, None) == bsmm.OK   # N = 0
    assert L.bsmm_layer_norm(A, A, A, B, 4, 0, 1, 1e-6, 0, 2, None) == bsmm.ERR_INVALID      # C < 1
    assert L.bsmm_layer_norm(A, A, A, B, -1, 8, 1, 1e-6, 0, 2, None) == bsmm.ERR_INVALID     # N < 0
    assert L.bsmm_layer_norm(A, A, A, B, 4, 8, 2, 1e-6, 0, 2, None) == bsmm.ERR_INVALID      # axis
    assert L.bsmm_layer_norm(A, A, A, B, 4, 8, 1, -1.0, 0, 2, None) == bsmm.ERR_INVALID      # epsilon
    assert L.bsmm_layer_norm(A, A, A, B, 4, 8, 1, float("nan"), 0, 2, None) == bsmm.ERR_INVALID
    assert L.bsmm_layer_norm(A + 8, A, A, B, 4, 8, 1, 1e-6, 0, 2, None) == bsmm.ERR_ALIGN   # x
    assert L.bsmm_layer_norm(A, A, A + 4, B, 4, 8, 1, 1e-6, 0, 2, None) == bsmm.ERR_ALIGN   # b
    assert L.bsmm_layer_norm(A, A, A, B, 4, 12, 1, 1e-6, 0, 2, None) == bsmm.ERR_ALIGN      # C * 2 % 16
    assert L.bsmm_layer_norm(A, A, A, B, 12, 8, 0, 1e-6, 0, 2, None) == bsmm.ERR_ALIGN      # N * 2 % 16
    assert L.bsmm_layer_norm(A, A, A, B, 12, 8, 0, 1e-6, 0, 0, None) == bsmm.ERR_ALIGN      # fp32, N % 8
    assert L.bsmm_layer_norm(A, A, A, B, 4, 16392, 1, 1e-6, 0, 2, None) == bsmm.ERR_UNSUPPORTED


def test_layer_norm_grad_rejects_bad_arguments_on_host():
    """Every case fails validation before anything is enqueued (the pointers are never used)."""
    L = bsmm.lib()
    A, B, D, W = 0x10000, 0x20000, 0x30000, 0x40000   # 16-byte aligned stand-ins, never dereferenced
    ws = L.bsmm_layer_norm_grad_workspace(4, 8, 1)
    assert ws == (8 + 1 * 2 * 8) * 4                     # 2N statistics + one chunk of 2C partials
    assert L.bsmm_layer_norm_grad_workspace(1000, 64, 1) == (2000 + 250 * 2 * 64) * 4   # 4-sample chunks
    assert L.bsmm_layer_norm_grad_workspace(8000, 64, 1) == (16000 + 1000 * 2 * 64) * 4  # at most 1024 chunks
    assert L.bsmm_layer_norm_grad_workspace(1000, 64, 0) == 32 * 2 * 64 * 4             # 32-sample tiles
    assert L.bsmm_layer_norm_grad_workspace(-1, 8, 1) == 0

    def call(x=A, y=None, g=A, dy=A, dx=B, dg=D, db=D + 0x1000, N=4, C=8, axis=1, eps=1e-6, relu=0, t=2,
             w=W, wb=ws):
        return L.bsmm_layer_norm_grad(x, y, g, dy, dx, dg, db, N, C, axis, eps, relu, t, w, wb, None)
    assert call(x=None) == bsmm.ERR_INVALID
    assert call(dx=A) == bsmm.ERR_INVALID                   # dx over x (and dy)
    assert call(relu=1, y=B) == bsmm.ERR_INVALID            # dx over y
    assert call(relu=1) == bsmm.ERR_INVALID                 # relu needs y
    assert call(dg=None) == bsmm.ERR_INVALID
    assert call(db=D) == bsmm.ERR_INVALID                   # dg == db
    assert call(w=None) == bsmm.ERR_INVALID
    assert call(wb=ws - 4) == bsmm.ERR_INVALID              # workspace too small
    assert call(N=-1) == bsmm.ERR_INVALID
    assert call(C=0) == bsmm.ERR_INVALID
    assert call(axis=2) == bsmm.ERR_INVALID
    assert call(eps=-1.0) == bsmm.ERR_INVALID
    assert call(eps=float("nan")) == bsmm.ERR_INVALID
    assert call(t=7) == bsmm.ERR_INVALID
    assert call(x=A + 8) == bsmm.ERR_ALIGN
    assert call(dx=B + 2) == bsmm.ERR_ALIGN
    assert call(relu=1, y=A + 4) == bsmm.ERR_ALIGN
    assert call(w=W + 4) == bsmm.ERR_ALIGN
    assert call(dg=D + 4) == bsmm.ERR_ALIGN
    assert call(C=12, wb=1 << 20) == bsmm.ERR_ALIGN          # C * 2 % 16
    assert call(N=12, axis=0, wb=1 << 20) == bsmm.ERR_ALIGN  # N * 2 % 16
    assert call(C=16392, wb=1 << 30) == bsmm.ERR_UNSUPPORTED


def test_l2_normalize_rejects_null_handle_on_host():
    L = bsmm.lib()
    A = 0x10000
    assert L.bsmm_l2_normalize(None, A, None, A, 1e-6, 0, None) == bsmm.ERR_INVALID
    assert L.bsmm_l2_normalize_grad(None, A, None, A, A + 0x1000, None, 1e-6, 0, None) == bsmm.ERR_INVALID


def test_proj_create_rejects_bad_maps_on_host():
    """The map is validated on the host before any CUDA call."""
    L = bsmm.lib()
    h = ctypes.c_void_p()

    def create(nhidden, nproj, stride, bs, lut=None):
        arr = None
        if lut is not None:
            lut = np.ascontiguousarray(lut, dtype=np.int32)
            arr = lut.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        return L.bsmm_proj_create(ctypes.byref(h), nhidden, nproj, stride, bs, arr)

    assert create(8, 3, 0, 1, [1, 5, 1]) == bsmm.ERR_INVALID          # repeated feature
    assert create(8, 3, 0, 1, [1, 5, 8]) == bsmm.ERR_INVALID          # out of range
    assert create(8, 3, 0, 1, [1, -1, 2]) == bsmm.ERR_INVALID
    assert create(2, 3, 0, 1, [0, 1, 2]) == bsmm.ERR_INVALID          # nproj > nhidden
    assert create(0, 0, 0, 32) == bsmm.ERR_INVALID                    # nhidden < 1
    assert create(100, 96, 64, 32) == bsmm.ERR_INVALID                # third run ends at 160 > 100
    assert create(256, 48, 64, 32) == bsmm.ERR_INVALID                # nproj not a multiple of block_size
    assert create(256, 64, 16, 32) == bsmm.ERR_INVALID                # runs would overlap
    assert create(16, 0, 0, 32) == bsmm.ERR_INVALID                   # no run fits
    assert L.bsmm_proj_create(None, 8, 0, 0, 4, None) == bsmm.ERR_INVALID
    A = 0x10000
    assert L.bsmm_proj(None, 0, A, None, A + 0x100, 4, 1, 2, None) == bsmm.ERR_INVALID
    assert L.bsmm_proj_destroy(None) == bsmm.OK


def test_binding_checks_caller_tensors_before_any_call():
    """The object API refuses a caller's tensor whose shape, dtype or device differs from what the
    C call will read or write (the C ABI sees only pointers)."""
    import torch
    t = torch.zeros(4, 6, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        bsmm._want(t, "y", (4, 7))
    with pytest.raises(ValueError, match="must be torch.float32"):
        bsmm._want(t, "dw", (4, 6), torch.float32)
    with pytest.raises(ValueError, match="unsupported dtype"):
        bsmm._want(torch.zeros(4, 6, dtype=torch.float64), "x", (4, 6))
    with pytest.raises(ValueError, match="must be on"):
        bsmm._want(t, "y", (4, 6), torch.bfloat16, torch.device("cuda", 0))
    with pytest.raises(ValueError, match="CUDA tensor"):           # right shape and dtype, host memory
        bsmm._want(t, "y", (4, 6), torch.bfloat16)


def test_noalloc_binding_checks_every_tensor_before_the_c_call(monkeypatch):
    """bsmm_updat_noalloc's binding checks x, dy and dw against the handle's shapes (the C call
    sees only pointers): a wrong dtype or shape raises before the library is reached."""
    import torch

    class _NoLib:
        def __getattr__(self, name):
            raise AssertionError("C call reached: " + name)

    monkeypatch.setattr(bsmm, "_handle_shapes", lambda h: (3, 32, 96, 128, 1))   # nnz, bs, C, K, fa
    monkeypatch.setattr(bsmm, "_dev", lambda t, what: None)                      # CPU tensors stand in
    monkeypatch.setattr(bsmm, "lib", lambda: _NoLib())
    x = torch.zeros((64, 96), dtype=torch.bfloat16)
    dy = torch.zeros((64, 128), dtype=torch.bfloat16)
    dw = torch.zeros((3, 32, 32), dtype=torch.float32)
    bad = [(x, dy, dw.bfloat16()),                       # dw not float32
           (x, dy, dw[:2]),                              # dw shape
           (x[:32], dy, dw),                             # x minibatch
           (x, dy[:, :96], dw),                          # dy features
           (x, dy.half(), dw)]                           # dy dtype differs from x
    for a, b, c in bad:
        with pytest.raises(ValueError):
            bsmm.bsmm_updat_noalloc(None, a, b, c, 64)
    with pytest.raises(AssertionError, match="C call reached"):
        bsmm.bsmm_updat_noalloc(None, x, dy, dw, 64)
