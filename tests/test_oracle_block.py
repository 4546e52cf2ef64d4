"""Pins of the fp64 block oracle against things other than itself.

* finite differences of L = sum(Y * G) on tiny shapes (calculus fixes B and W);
* textbook special cases (linear layer rules of "Pipeline Schedules", section
  "Zero bubble: split the backward pass"; GeLU values of the normal CDF);
* the split-backward invariant of "Zero-Bubble Pipeline Parallelism, Proven",
  section "Split backward without changing the update";
* bf16 rounding against torch's own round-to-nearest-even cast.
"""

import math

import numpy as np
import pytest
import torch

from oracle import block as ob
from oracle import schedules as osch

RNG = np.random.default_rng(1234)


def _rand(*shape, std=1.0):
    return RNG.standard_normal(shape) * std


def _loss_fn(X, W1, W2, b1, b2, G, act):
    _, _, Y = ob.forward(X, W1, W2, b1, b2, act)
    return float(np.sum(Y * G))


def _fd_grad(fun, P, eps=1e-6):
    g = np.zeros_like(P)
    it = np.nditer(P, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = P[i]
        P[i] = old + eps
        lp = fun()
        P[i] = old - eps
        lm = fun()
        P[i] = old
        g[i] = (lp - lm) / (2 * eps)
    return g


@pytest.mark.parametrize("act", ["gelu_erf", "gelu_tanh"])
@pytest.mark.parametrize("bias", [False, True])
def test_block_gradients_match_finite_differences(act, bias):
    M, h, f = 5, 3, 7
    X, W1, W2, G = _rand(M, h), _rand(h, f, std=0.7), _rand(f, h, std=0.7), _rand(M, h)
    b1 = _rand(f, std=0.3) if bias else None
    b2 = _rand(h, std=0.3) if bias else None
    H, A, Y = ob.forward(X, W1, W2, b1, b2, act)
    _, dH, dX = ob.backward_input(G, W1, W2, H, act)
    dW1, dW2, db1, db2 = ob.backward_weight(X, A, dH, G, act)
    L = lambda: _loss_fn(X, W1, W2, b1, b2, G, act)  # noqa: E731
    for got, param in ((dX, X), (dW1, W1), (dW2, W2)):
        fd = _fd_grad(L, param)
        assert ob.rel_fro(got, fd) < 1e-7
    if bias:
        assert ob.rel_fro(db1, _fd_grad(L, b1)) < 1e-7
        assert ob.rel_fro(db2, _fd_grad(L, b2)) < 1e-7


def test_single_linear_matches_textbook_rules_and_fd():
    # Y = X W: Xbar = Ybar W^T, Wbar = X^T Ybar (linear-layer split).
    M, h, n = 4, 3, 5
    X, W, G = _rand(M, h), _rand(h, n), _rand(M, n)
    _, _, Y = ob.forward(X, W, None, act="none")
    assert np.array_equal(Y, X @ W)
    _, _, dX = ob.backward_input(G, W, None, None, act="none")
    dW, _, _, _ = ob.backward_weight(X, None, None, G, act="none")
    L = lambda: float(np.sum(ob.forward(X, W, None, act="none")[2] * G))  # noqa: E731
    assert ob.rel_fro(dX, _fd_grad(L, X)) < 1e-7
    assert ob.rel_fro(dW, _fd_grad(L, W)) < 1e-7


def test_gelu_special_values():
    # GeLU(x) = x Phi(x); Phi(1) = 0.8413447460685429 (standard normal CDF).
    phi1 = 0.8413447460685429
    assert ob.gelu(0.0) == 0.0
    assert math.isclose(float(ob.gelu(1.0)), phi1, rel_tol=1e-15)
    assert math.isclose(float(ob.gelu(-1.0)), -(1 - phi1), rel_tol=1e-14)
    assert math.isclose(float(ob.gelu_prime(0.0)), 0.5, rel_tol=1e-15)
    # GeLU'(1) = Phi(1) + phi(1), phi(1) = exp(-1/2)/sqrt(2 pi) = 0.24197072451914337
    assert math.isclose(float(ob.gelu_prime(1.0)), phi1 + 0.24197072451914337, rel_tol=1e-14)
    big = np.array([12.0, 30.0])
    assert np.allclose(ob.gelu(big), big, rtol=0, atol=1e-12)
    assert np.allclose(ob.gelu_prime(big), 1.0, rtol=0, atol=1e-12)
    assert np.allclose(ob.gelu(-big), 0.0, atol=1e-12)
    assert np.allclose(ob.gelu_prime(-big), 0.0, atol=1e-12)
    # the tanh form is within its known ~1e-3 absolute distance of the erf form
    x = np.linspace(-6, 6, 1001)
    assert np.max(np.abs(ob.gelu(x, "gelu_tanh") - ob.gelu(x))) < 1e-3
    assert float(ob.gelu(0.0, "gelu_tanh")) == 0.0
    assert math.isclose(float(ob.gelu_prime(0.0, "gelu_tanh")), 0.5, rel_tol=1e-15)


def test_identity_weight_gives_h_equals_x():
    M, h = 6, 4
    X = _rand(M, h)
    W2 = _rand(h, h)
    H, A, _ = ob.forward(X, np.eye(h), W2)
    assert np.array_equal(H, X)
    assert np.allclose(A, ob.gelu(X))


def test_rel_fro_hand_value():
    ref = np.array([[3.0, 4.0]])
    got = np.array([[3.0, 4.5]])
    assert math.isclose(ob.rel_fro(got, ref), 0.5 / 5.0)
    assert ob.rel_fro(ref, ref) == 0.0


def test_bf16_round_matches_torch_rne():
    x = np.concatenate([_rand(4096) * 10.0 ** RNG.integers(-6, 6, 4096),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, -3.0e38])])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = ob.bf16_round(x32)
    assert np.array_equal(got, ref)


def _chain_inputs(P=2, m=3, M=4, h=3, f=5, act="gelu_erf"):
    stages = [{"W1": _rand(h, f, std=0.6), "W2": _rand(f, h, std=0.6)} for _ in range(P)]
    X0 = [_rand(M, h) for _ in range(m)]
    G = [_rand(M, h) for _ in range(m)]
    return stages, X0, G


def test_pipeline_chain_matches_finite_differences():
    # Two chained stages: loss = sum_j sum(Y_last_j * G_j).
    P, m = 2, 3
    stages, X0, G = _chain_inputs(P, m)
    _, ops = osch.make_schedule("ZBH1", P, m)
    out = ob.run_pipeline(stages, X0, G, ops)

    def loss():
        tot = 0.0
        for j in range(m):
            x = X0[j]
            for st in stages:
                _, _, x = ob.forward(x, st["W1"], st["W2"])
            tot += float(np.sum(x * G[j]))
        return tot

    for s in range(P):
        assert ob.rel_fro(out["dW1"][s], _fd_grad(loss, stages[s]["W1"])) < 1e-7
        assert ob.rel_fro(out["dW2"][s], _fd_grad(loss, stages[s]["W2"])) < 1e-7
    for j in range(m):
        assert ob.rel_fro(out["dX0"][j], _fd_grad(loss, X0[j])) < 1e-7


@pytest.mark.parametrize("P,m", [(2, 3), (4, 8)])
def test_deferred_w_equals_fused_backward_exactly(P, m):
    stages, X0, G = _chain_inputs(P, m)
    res = {}
    for kind in osch.SCHEDULES:
        _, ops = osch.make_schedule(kind, P, m)
        res[kind] = ob.run_pipeline(stages, X0, G, ops)
    for kind in ("ZBH1", "ZBH2"):
        for key in ("dW1", "dW2", "db1", "db2"):
            for s in range(P):
                assert np.array_equal(res[kind][key][s], res["1F1B"][key][s])
        for j in range(m):
            assert np.array_equal(res[kind]["dX0"][j], res["1F1B"]["dX0"][j])
            assert np.array_equal(res[kind]["Y_last"][j], res["1F1B"]["Y_last"][j])
