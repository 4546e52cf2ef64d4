"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and nothing else: it holds none of the
block's or the schedules' arithmetic, and it imports neither the CUDA binding
nor the oracle.  Draws are fp32 from numpy's PCG64 generator; a caller that
wants bf16 rounds them (ties to even) itself, so both sides see identical
input bits.

Draw order for a P-stage pipeline (one generator, one seed): for each stage s
its W1_s, W2_s (and b1_s, b2_s when biases are on); then X_{0,j} for
j = 0..m-1; then dY_{P-1,j} for j = 0..m-1.

Workload shapes follow the GPT-3-style configurations the pages describe
([ZB-PP summary] §5 "Base model(s)": hidden sizes up to 6144, sequence 1024 in
the paper; the block sizes here are h, f = 4h, M tokens per microbatch).
Weights are N(0, 0.02^2); inputs and the last stage's output gradient are
N(0, 1), unless a case overrides the scales.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class StageDraws:
    W1: np.ndarray
    W2: np.ndarray | None
    b1: np.ndarray | None = None
    b2: np.ndarray | None = None


def normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """fp32 N(0, std^2) draws."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def pipeline_draws(P: int, m: int, M: int, h: int, f: int, *, seed: int = 0,
                   w_std: float = 0.02, x_std: float = 1.0, g_std: float = 1.0,
                   bias: bool = False, b_std: float = 0.02, single_linear: bool = False):
    """Draw weights, stage-0 inputs and last-stage output gradients.

    single_linear: one weight W1[h, f] per stage and no W2 (Y = X W1).
    Returns (stages, X0, dY_last) with X0[j] of shape [M, h] and dY_last[j]
    of shape [M, h] (or [M, f] for a single linear layer).
    """
    rng = np.random.default_rng(seed)
    stages = []
    for _ in range(P):
        W1 = normal(rng, (h, f), w_std)
        W2 = None if single_linear else normal(rng, (f, h), w_std)
        b1 = b2 = None
        if bias:
            b1 = normal(rng, (f,), b_std)
            b2 = None if single_linear else normal(rng, (h,), b_std)
        stages.append(StageDraws(W1, W2, b1, b2))
    X0 = [normal(rng, (M, h), x_std) for _ in range(m)]
    out_w = f if single_linear else h
    dY = [normal(rng, (M, out_w), g_std) for _ in range(m)]
    return stages, X0, dY


def matrix(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """One seeded fp32 N(0, std^2) matrix (standalone kernel cases)."""
    return normal(np.random.default_rng(seed), shape, std)


def optimizer_draws(sizes_per_stage, *, seed: int = 0, grad_std=None, theta_std: float = 0.02):
    """Optimizer state for P stages: per stage a list of (theta, m, v, grad)
    fp32 arrays of the given sizes.  theta ~ N(0, theta_std^2), m ~ N(0, 1e-4),
    v = (N(0, 1e-2))^2 (a second moment, so non-negative), grad ~ N(0,
    grad_std[s]^2) (1 for every stage by default).  Draw order: stage by
    stage, tensor by tensor, theta, m, v, grad."""
    rng = np.random.default_rng(seed)
    out = []
    for s, sizes in enumerate(sizes_per_stage):
        gs = 1.0 if grad_std is None else float(grad_std[s])
        st = []
        for n in sizes:
            theta = normal(rng, (n,), theta_std)
            m = normal(rng, (n,), 1e-2)
            v = np.square(normal(rng, (n,), 1e-1))
            g = normal(rng, (n,), gs)
            st.append((theta, m, v, g))
        out.append(st)
    return out
