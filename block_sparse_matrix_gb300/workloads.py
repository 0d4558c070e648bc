"""Seeded synthetic inputs for block-sparse matmul workloads.

This module only draws random numbers and builds 0/1 layouts.  It holds none of
the method's arithmetic, so both the CUDA path's tests/benchmarks and the CPU
oracle can take their inputs from it without sharing any computation.

Workloads follow the usage example of the blocksparse README (hidden 4096,
block size 32, minibatch 64, random 0/1 layout: "Usage" section) and the
benchmark workloads of this library (named by their sizes, below).  All draws use
numpy's PCG64 generator (``numpy.random.default_rng(seed)``) with
``seed = 1000 * seed_ns + stream`` where stream 0 = layout, 1 = x, 2 = w, 3 = dy,
10 + t = x of timestep t, 30 + t = dy of timestep t.  Normals are drawn in
float32 and rounded to nearest-even into the compute dtype by torch.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed_ns: int           # seed namespace: inputs draw from seeds 1000 * seed_ns + stream
    C: int                 # input features
    K: int                 # output features
    bs: int                # block size (32, 16 or 8)
    layout_kind: str       # "bernoulli" | "blockdiag_plus"
    density: float         # Bernoulli probability (bernoulli) or extra blocks per row (blockdiag_plus)
    force_diag: bool
    N: int                 # minibatch per call
    dtype: str             # "f32" | "f16" | "bf16"
    feature_axis: int      # 1: (N,C) activations, 0: (C,N)
    w_var: float           # variance of the weight normals
    steps: int = 1         # timesteps sharing W (grouped weight gradient)
    group: int = 1         # timesteps summed per grouped-updat call

    @property
    def R(self) -> int:
        return self.C // self.bs

    @property
    def S(self) -> int:
        return self.K // self.bs


# The benchmark workloads, named by hidden size, block size and density; the 4096-wide, block 32,
# 50% dense one is quoted at N=64 and at N=1024.
CONFIGS = {
    "h256_b32_fp32": Workload("h256_b32_fp32", 1, 256, 256, 32, "bernoulli", 0.5, True, 64, "f32", 1,
                              1.0 / 256),
    "h4096_b32_p50_n64": Workload("h4096_b32_p50_n64", 2, 4096, 4096, 32, "bernoulli", 0.5, False, 64, "bf16",
                                  1, 1.0 / (4096 * 0.5)),
    "h4096_b32_p50_n1024": Workload("h4096_b32_p50_n1024", 2, 4096, 4096, 32, "bernoulli", 0.5, False, 1024,
                                    "bf16", 1, 1.0 / (4096 * 0.5)),
    "h8192_b16_p10": Workload("h8192_b16_p10", 3, 8192, 8192, 16, "bernoulli", 0.10, True, 512, "f16", 0,
                              1.0 / (8192 * 0.10)),
    "h4096_b8_p5": Workload("h4096_b8_p5", 4, 4096, 4096, 8, "bernoulli", 0.05, True, 2048, "bf16", 0,
                            1.0 / (4096 * 0.05)),
    "h6144_b32_recurrent": Workload("h6144_b32_recurrent", 5, 6144, 6144, 32, "blockdiag_plus", 8, True, 128,
                                    "bf16", 1, 1.0 / (9 * 32), steps=16, group=8),
}


def make_layout(R: int, S: int, kind: str, density: float, force_diag: bool, seed: int) -> np.ndarray:
    """0/1 uint8 layout of shape (R, S) (rows = input blocks c, cols = output blocks k)."""
    rng = np.random.default_rng(seed)
    if kind == "bernoulli":
        lay = (rng.random((R, S)) < density).astype(np.uint8)
    elif kind == "blockdiag_plus":
        # block diagonal plus `density` distinct random off-diagonal blocks per row
        extra = int(density)
        lay = np.zeros((R, S), dtype=np.uint8)
        for c in range(R):
            picks = rng.choice(S - 1, size=extra, replace=False)
            picks = np.where(picks >= c, picks + 1, picks)   # skip the diagonal column
            lay[c, picks] = 1
    elif kind == "ones":
        lay = np.ones((R, S), dtype=np.uint8)
    elif kind == "zeros":
        lay = np.zeros((R, S), dtype=np.uint8)
    else:
        raise ValueError(kind)
    if force_diag:
        for i in range(min(R, S)):
            lay[i, i] = 1
    return lay


def normals(shape, seed: int, std: float = 1.0, dtype: str = "f32") -> torch.Tensor:
    """float32 N(0, std^2) draws from PCG64(seed), rounded RNE into `dtype` (CPU tensor)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(DTYPES[dtype])


def device_normals(shape, seed: int, std: float = 1.0, dtype: str = "f32", device="cuda") -> torch.Tensor:
    """N(0, std^2) draws made on the device by torch's seeded CUDA generator (for inputs of several
    GB, where host generation and upload would dominate), in `dtype`.  Deterministic per seed."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(DTYPES[dtype])


def small_ints(shape, seed: int, dtype: str = "f32", lo: int = -1, hi: int = 1) -> torch.Tensor:
    """Integers uniform in [lo, hi] (exactly representable in every dtype here)."""
    rng = np.random.default_rng(seed)
    a = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return torch.from_numpy(a).to(DTYPES[dtype])


def act_shape(C: int, N: int, feature_axis: int):
    """Activation shape: (N, C) for feature_axis=1, (C, N) for feature_axis=0."""
    return (N, C) if feature_axis == 1 else (C, N)


@dataclasses.dataclass
class Inputs:
    layout: np.ndarray
    nnz: int
    x: torch.Tensor
    w: torch.Tensor
    dy: torch.Tensor
    xs: Optional[list] = None     # per-timestep x (grouped weight gradient)
    dys: Optional[list] = None


def make_inputs(wl: Workload, N: Optional[int] = None, steps: Optional[int] = None) -> Inputs:
    """All inputs of a workload on the CPU, in the workload's dtype."""
    N = wl.N if N is None else N
    lay = make_layout(wl.R, wl.S, wl.layout_kind, wl.density, wl.force_diag, 1000 * wl.seed_ns + 0)
    nnz = int(lay.sum())
    base = 1000 * wl.seed_ns
    x = normals(act_shape(wl.C, N, wl.feature_axis), base + 1, 1.0, wl.dtype)
    w = normals((nnz, wl.bs, wl.bs), base + 2, float(np.sqrt(wl.w_var)), wl.dtype)
    dy = normals(act_shape(wl.K, N, wl.feature_axis), base + 3, 1.0, wl.dtype)
    xs = dys = None
    T = wl.steps if steps is None else steps
    if T > 1:
        xs = [normals(act_shape(wl.C, N, wl.feature_axis), base + 10 + t, 1.0, wl.dtype) for t in range(T)]
        dys = [normals(act_shape(wl.K, N, wl.feature_axis), base + 30 + t, 1.0, wl.dtype) for t in range(T)]
    return Inputs(lay, nnz, x, w, dy, xs, dys)


def effective_flops(N: int, nnz: int, bs: int) -> int:
    """Effective FLOPs of one pass: 2*N*nnz*bs^2 (multiply-adds of the nonzero blocks only)."""
    return 2 * N * nnz * bs * bs
