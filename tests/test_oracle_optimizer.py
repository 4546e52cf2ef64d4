"""Pins of the post-update-validation oracle.

* AdamW against torch.optim.AdamW (a library routine) in fp64;
* the first step's textbook property: with zero moments, bias correction
  makes the update lr * g / (|g| + eps) (about lr in magnitude);
* rollback(step(x)) = x (the inverse the summary's "Why rollback is
  feasible" relies on);
* the staged reduce ends at the global state;
* post-validated results equal the synchronous (all-reduce first) step, with
  exactly the stages whose optimistic decision differed rolled back.
"""

import numpy as np
import pytest
import torch

from oracle import optimizer as O

HP = O.AdamW(lr=2e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def test_adamw_matches_torch():
    rng = np.random.default_rng(0)
    th0 = rng.standard_normal(1000)
    p = torch.nn.Parameter(torch.tensor(th0, dtype=torch.float64))
    opt = torch.optim.AdamW([p], lr=HP.lr, betas=(HP.beta1, HP.beta2), eps=HP.eps,
                            weight_decay=HP.weight_decay)
    th, m, v = th0.copy(), np.zeros(1000), np.zeros(1000)
    for t in range(1, 6):
        g = rng.standard_normal(1000)
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        th, m, v = O.adamw_step(th, m, v, g, t, HP)
        assert np.allclose(th, p.detach().numpy(), rtol=1e-13, atol=1e-15)


def test_first_step_is_lr_times_sign():
    g = np.array([3.0, -0.5, 1e-3])
    hp = O.AdamW(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    th1, m1, v1 = O.adamw_step(np.zeros(3), np.zeros(3), np.zeros(3), g, 1, hp)
    assert np.allclose(th1, -hp.lr * g / (np.abs(g) + hp.eps), rtol=1e-12)
    assert np.allclose(m1, 0.1 * g) and np.allclose(v1, 0.001 * g * g)


@pytest.mark.parametrize("t", [1, 2, 7, 1000])
def test_rollback_inverts_step(t):
    rng = np.random.default_rng(t)
    th, m, v, g = rng.standard_normal((4, 500))
    v = np.abs(v)
    th1, m1, v1 = O.adamw_step(th, m, v, g, t, HP)
    th0, m0, v0 = O.adamw_rollback(th1, m1, v1, g, t, HP)
    assert np.allclose(th0, th, rtol=1e-12, atol=1e-12)
    assert np.allclose(m0, m, rtol=1e-12, atol=1e-12)
    assert np.allclose(v0, v, rtol=1e-9, atol=1e-12)


def test_staged_reduce_reaches_global_state():
    states = [(1.0, 0), (2.5, 0), (0.5, 1), (4.0, 0)]
    part = O.staged_reduce(states)
    assert part == [(1.0, 0), (3.5, 0), (4.0, 1), (8.0, 1)]
    assert O.clip_factor(16.0, 2.0) == 0.5 and O.clip_factor(3.0, 2.0) == 1.0


def _stages(rng, P, scales, nan_stage=None):
    params, grads = [], []
    for s in range(P):
        shapes = [(7, 5), (11,)]
        params.append([(rng.standard_normal(sh), 0.1 * rng.standard_normal(sh),
                        np.abs(0.01 * rng.standard_normal(sh))) for sh in shapes])
        gs = [scales[s] * rng.standard_normal(sh) for sh in shapes]
        if nan_stage == s:
            gs[0][1, 2] = np.nan
        grads.append(gs)
    return params, grads


@pytest.mark.parametrize("case", ["no_clip", "clip_late", "nan_late", "nan_first"])
def test_post_validated_equals_synchronous(case):
    rng = np.random.default_rng(11)
    P = 4
    scales = {"no_clip": [0.01] * 4, "clip_late": [0.05, 0.05, 0.05, 3.0],
              "nan_late": [0.01] * 4, "nan_first": [0.01] * 4}[case]
    nan_stage = {"nan_late": 2, "nan_first": 0}.get(case)
    params, grads = _stages(rng, P, scales, nan_stage)
    max_norm = 1.0
    got, rep = O.post_validated_step(params, grads, 3, HP, max_norm)
    ref = O.synchronous_step(params, grads, 3, HP, max_norm)
    for s in range(P):
        for a, b in zip(got[s], ref[s]):
            for x, y in zip(a, b):
                assert np.allclose(x, y, rtol=1e-10, atol=1e-12)
    rolled = [r["rolled_back"] for r in rep]
    assert rolled[-1] is False  # the last stage already holds the global state
    expect = {"no_clip": [False] * 4, "clip_late": [True, True, True, False],
              "nan_late": [True, True, False, False], "nan_first": [False] * 4}[case]
    assert rolled == expect
