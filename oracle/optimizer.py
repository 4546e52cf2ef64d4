"""fp64 oracle of post-update validation with an AdamW step and its inverse.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Plain numpy, float64.

Followed: [ZB-PP summary] §4 "The Optimizer Synchronization Bypass" and
"Why rollback is feasible":
  * staged reduce: stage i combines its local state (gradient norm squared,
    NaN/Inf flag) with the partial state received from stage i-1 and passes
    the result on; the last stage holds the global state;
  * optimistic step: each stage steps with its partially reduced state —
    clipping when the partial norm exceeds the threshold, skipping the update
    when a NaN/Inf has been seen;
  * validation: the global state travels back; a stage whose step used a
    different clip factor or skip decision rolls its step back and redoes it
    with the global state;
  * AdamW (the summary's update formula):
        m_t = b1 m_{t-1} + (1 - b1) g,   v_t = b2 v_{t-1} + (1 - b2) g^2,
        theta_{t+1} = theta_t - lr wd theta_t
                      - lr (m_t / (1 - b1^t)) / (sqrt(v_t / (1 - b2^t)) + eps)
    and its inverse given g, (m_t, v_t, theta_{t+1}):
        m_{t-1} = (m_t - (1 - b1) g) / b1,  v_{t-1} = (v_t - (1 - b2) g^2) / b2,
        theta_t = (theta_{t+1} + lr mhat / (sqrt(vhat) + eps)) / (1 - lr wd).
    (Algorithm 1's listing is not on the pages; the inverse is the algebraic
    inverse of the formula above.)
Clip factor for a norm n and threshold c: c / n when n > c, else 1.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01


def adamw_step(theta, m, v, g, t: int, hp: AdamW):
    """One AdamW update at step t >= 1.  Returns new (theta, m, v)."""
    theta, m, v, g = (np.asarray(a, dtype=np.float64) for a in (theta, m, v, g))
    m1 = hp.beta1 * m + (1.0 - hp.beta1) * g
    v1 = hp.beta2 * v + (1.0 - hp.beta2) * g * g
    mhat = m1 / (1.0 - hp.beta1 ** t)
    vhat = v1 / (1.0 - hp.beta2 ** t)
    th1 = theta - hp.lr * hp.weight_decay * theta - hp.lr * mhat / (np.sqrt(vhat) + hp.eps)
    return th1, m1, v1


def adamw_rollback(theta1, m1, v1, g, t: int, hp: AdamW):
    """Inverse of adamw_step given the same gradient: returns (theta, m, v)."""
    theta1, m1, v1, g = (np.asarray(a, dtype=np.float64) for a in (theta1, m1, v1, g))
    mhat = m1 / (1.0 - hp.beta1 ** t)
    vhat = v1 / (1.0 - hp.beta2 ** t)
    theta = (theta1 + hp.lr * mhat / (np.sqrt(vhat) + hp.eps)) / (1.0 - hp.lr * hp.weight_decay)
    m = (m1 - (1.0 - hp.beta1) * g) / hp.beta1
    v = (v1 - (1.0 - hp.beta2) * g * g) / hp.beta2
    return theta, m, v


def clip_factor(norm_sq: float, max_norm: float) -> float:
    n = float(np.sqrt(norm_sq))
    return max_norm / n if n > max_norm else 1.0


def local_state(grads):
    """(sum of squares, non-finite count) over a stage's gradient arrays."""
    sq = 0.0
    bad = 0
    for g in grads:
        g = np.asarray(g, dtype=np.float64)
        bad += int(np.sum(~np.isfinite(g)))
        sq += float(np.sum(g * g))
    return sq, bad


def staged_reduce(states):
    """Partial states along the stages: partial[i] = state[0] + ... + state[i]."""
    out = []
    sq, bad = 0.0, 0
    for s_sq, s_bad in states:
        sq += s_sq
        bad += s_bad
        out.append((sq, bad))
    return out


def post_validated_step(stage_params, stage_grads, t: int, hp: AdamW, max_norm: float):
    """Replay the protocol for P stages.

    stage_params: per stage a list of (theta, m, v) arrays (one per tensor);
    stage_grads:  per stage a list of gradient arrays (same order).
    Returns (new params per stage, report) where report per stage holds the
    (scale, skip) used optimistically, the global (scale, skip) and whether
    the stage rolled back.
    """
    states = [local_state(gs) for gs in stage_grads]
    partial = staged_reduce(states)
    g_sq, g_bad = partial[-1]
    g_scale, g_skip = clip_factor(g_sq, max_norm), g_bad > 0
    out, report = [], []
    for s, (params, grads) in enumerate(zip(stage_params, stage_grads)):
        p_sq, p_bad = partial[s]
        scale, skip = clip_factor(p_sq, max_norm), p_bad > 0
        new = []
        for (th, m, v), g in zip(params, grads):
            new.append((th, m, v) if skip else adamw_step(th, m, v, scale * np.asarray(g, np.float64), t, hp))
        rolled = (scale != g_scale) or (skip != g_skip)
        if rolled:
            fixed = []
            for (th1, m1, v1), (th, m, v), g in zip(new, params, grads):
                if not skip:
                    th, m, v = adamw_rollback(th1, m1, v1, scale * np.asarray(g, np.float64), t, hp)
                fixed.append((th, m, v) if g_skip else
                             adamw_step(th, m, v, g_scale * np.asarray(g, np.float64), t, hp))
            new = fixed
        out.append(new)
        report.append({"scale": scale, "skip": skip, "global_scale": g_scale,
                       "global_skip": g_skip, "rolled_back": rolled})
    return out, report


def synchronous_step(stage_params, stage_grads, t: int, hp: AdamW, max_norm: float):
    """The baseline: all-reduce the global state first, then step every stage."""
    states = [local_state(gs) for gs in stage_grads]
    g_sq, g_bad = staged_reduce(states)[-1]
    scale, skip = clip_factor(g_sq, max_norm), g_bad > 0
    out = []
    for params, grads in zip(stage_params, stage_grads):
        out.append([(th, m, v) if skip else adamw_step(th, m, v, scale * np.asarray(g, np.float64), t, hp)
                    for (th, m, v), g in zip(params, grads)])
    return out
