"""Shared helpers for the GPU parity tests (comparison metrics, problem setup)."""
import numpy as np
import torch

from block_sparse_matrix_gb300 import workloads as wk

# Tolerances on the relative Frobenius error ||O - R|| / ||R|| against the
# float64 oracle: IEEE fp32 path 1e-5; 16-bit inputs with float32 accumulation
# and one rounding of the output 2e-2.
TOL = {"f32": 1e-5, "f16": 2e-2, "bf16": 2e-2}
# updat writes float32 dW from exact 16-bit inputs, so only float32 summation error remains.
TOL_DW = {"f32": 1e-5, "f16": 1e-5, "bf16": 1e-5}


def rel_fro(out, ref):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    nr = np.linalg.norm(ref)
    if nr == 0:
        return 0.0 if not np.any(out) else np.inf
    return float(np.linalg.norm(out - ref) / nr)


def cpu64(t):
    return t.detach().float().cpu().double().numpy()


def rand_layout(R, S, p, seed, diag=False):
    L = (np.random.default_rng(seed).random((R, S)) < p).astype(np.uint8)
    if diag:
        for i in range(min(R, S)):
            L[i, i] = 1
    return L


def problem(R, S, bs, N, fa, dtype, p=0.5, seed=0, diag=False, w_std=None):
    L = rand_layout(R, S, p, seed, diag)
    nnz = int(L.sum())
    C, K = R * bs, S * bs
    if w_std is None:
        w_std = float(1.0 / np.sqrt(max(1.0, C * p)))
    x = wk.normals(wk.act_shape(C, N, fa), seed + 1, 1.0, dtype)
    w = wk.normals((nnz, bs, bs), seed + 2, w_std, dtype)
    dy = wk.normals(wk.act_shape(K, N, fa), seed + 3, 1.0, dtype)
    return L, x, w, dy


def act_nf(a, fa):
    """(N, F) view of an activation array stored in feature_axis layout fa."""
    return a if fa == 1 else a.T
