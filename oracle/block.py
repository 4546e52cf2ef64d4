"""fp64 oracle of one pipeline stage's MLP block, split into F, B and W.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Plain numpy in float64;
the only library primitives are ``@`` (matrix product) and ``scipy.special.erf``.
No blocking, fusion or reordering beyond the definitions below.

Definitions followed
--------------------
* [ZB-PP summary] §2 "The Unexploited Opportunity" and §3.4 "The Backward Pass
  Decomposition": a layer's backward splits into the input gradient
  B = (d f / d x)^T dl/dy and the parameter gradient W = (d f / d W)^T dl/dy;
  W of stage i, microbatch j depends only on B of the same (i, j).
* [Pipeline schedules] "Zero bubble: split the backward pass": for a linear
  map Y = X W the two halves are  Xbar = Ybar W^T  (B) and  Wbar = X^T Ybar (W).
* [ZB-PP summary] §2, Figure 1 names an MLP layer as the worked example; the
  block here is  H = X W1 (+ b1),  A = GeLU(H),  Y = A W2 (+ b2),  row-major,
  X[M,h], W1[h,f], W2[f,h].  GeLU(x) = x Phi(x) = x/2 (1 + erf(x / sqrt 2)),
  with the tanh approximation selectable; the pages name no activation, so
  the exact-erf form is the default reading.
* Chain rule through the block (plain calculus, no reading needed):
      dA = dY W2^T,   dH = dA * GeLU'(H),   dX = dH W1^T         (B)
      dW2 += A^T dY,  dW1 += X^T dH,  db2 += colsum dY,  db1 += colsum dH   (W)
  with GeLU'(x) = Phi(x) + x phi(x).
* Pipeline chain ([ZB-PP summary] §3.4, dependencies of B; §3 "Dependency
  constraints", Eqs. 4-5): the input of stage s+1 for microbatch j is the
  output of stage s; the output gradient of stage s is the input gradient of
  stage s+1.  Weight gradients accumulate over microbatches in the order the
  W passes run ([ZB proven] "Split backward without changing the update").
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)
_TANH_K = math.sqrt(2.0 / math.pi)
_TANH_C = 0.044715

ACTS = ("none", "gelu_erf", "gelu_tanh")


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# activation
# --------------------------------------------------------------------------
def gelu(x, act: str = "gelu_erf"):
    """GeLU(x) = x * Phi(x) (erf form) or the tanh approximation."""
    x = _f64(x)
    if act == "gelu_erf":
        return 0.5 * x * (1.0 + erf(x / _SQRT2))
    if act == "gelu_tanh":
        return 0.5 * x * (1.0 + np.tanh(_TANH_K * (x + _TANH_C * x ** 3)))
    if act == "none":
        return x.copy()
    raise ValueError(act)


def gelu_prime(x, act: str = "gelu_erf"):
    """d GeLU / dx.  erf form: Phi(x) + x phi(x)."""
    x = _f64(x)
    if act == "gelu_erf":
        phi_cdf = 0.5 * (1.0 + erf(x / _SQRT2))
        phi_pdf = _INV_SQRT_2PI * np.exp(-0.5 * x * x)
        return phi_cdf + x * phi_pdf
    if act == "gelu_tanh":
        u = _TANH_K * (x + _TANH_C * x ** 3)
        t = np.tanh(u)
        du = _TANH_K * (1.0 + 3.0 * _TANH_C * x * x)
        return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * du
    if act == "none":
        return np.ones_like(x)
    raise ValueError(act)


# --------------------------------------------------------------------------
# the three passes of one block
# --------------------------------------------------------------------------
def forward(X, W1, W2, b1=None, b2=None, act: str = "gelu_erf"):
    """F: H = X W1 (+b1); A = GeLU(H); Y = A W2 (+b2).  Returns (H, A, Y).

    With act == "none" the block is the single linear map Y = X W1 and
    (H, A) are X W1 as well; W2 / b2 are ignored.
    """
    X, W1 = _f64(X), _f64(W1)
    H = X @ W1
    if b1 is not None:
        H = H + _f64(b1)[None, :]
    if act == "none":
        return H, H, H
    A = gelu(H, act)
    Y = A @ _f64(W2)
    if b2 is not None:
        Y = Y + _f64(b2)[None, :]
    return H, A, Y


def backward_input(dY, W1, W2, H, act: str = "gelu_erf"):
    """B: dA = dY W2^T; dH = dA * GeLU'(H); dX = dH W1^T.  Returns (dA, dH, dX).

    act == "none": dX = dY W1^T (textbook linear input gradient); dA = dH = dY.
    """
    dY, W1 = _f64(dY), _f64(W1)
    if act == "none":
        return dY, dY, dY @ W1.T
    dA = dY @ _f64(W2).T
    dH = dA * gelu_prime(H, act)
    dX = dH @ W1.T
    return dA, dH, dX


def backward_weight(X, A, dH, dY, act: str = "gelu_erf"):
    """W (one microbatch's contribution): returns (dW1, dW2, db1, db2).

    dW2 = A^T dY, dW1 = X^T dH, db2 = colsum dY, db1 = colsum dH.
    act == "none": dW1 = X^T dY (textbook linear weight gradient), the rest None.
    """
    X, dY = _f64(X), _f64(dY)
    if act == "none":
        return X.T @ dY, None, dY.sum(axis=0), None
    A, dH = _f64(A), _f64(dH)
    return X.T @ dH, A.T @ dY, dH.sum(axis=0), dY.sum(axis=0)


# --------------------------------------------------------------------------
# errors
# --------------------------------------------------------------------------
def rel_fro(got, ref) -> float:
    """Relative Frobenius error ||got - ref||_F / ||ref||_F in fp64."""
    got, ref = _f64(got), _f64(ref)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


# --------------------------------------------------------------------------
# fp64 pipeline chain
# --------------------------------------------------------------------------
def run_pipeline(stages, X0, dY_last, ops, act: str = "gelu_erf", round_fn=None):
    """Replay an F/B/W(/BW/OPT) op list over P stages in fp64.

    stages  : list of dicts with "W1", "W2" (and optional "b1", "b2").
    X0      : list of m stage-0 inputs [M,h].
    dY_last : list of m output gradients entering stage P-1 [M,h].
    ops     : iterable of (kind, stage, micro), kind in {"F","B","W","BW","OPT"}.
    round_fn: optional callable applied where a stored tensor would be
              rounded (H, A, Y, dH, dX); None keeps everything in fp64.

    Returns dict with "dW1", "dW2", "db1", "db2" per stage (accumulated in
    op order), "Y_last" and "dX0" per microbatch.
    """
    P = len(stages)
    m = len(X0)
    rnd = round_fn if round_fn is not None else (lambda a: a)
    X = {(0, j): _f64(X0[j]) for j in range(m)}
    dY = {(P - 1, j): _f64(dY_last[j]) for j in range(m)}
    H, A, dH = {}, {}, {}
    out = {"dW1": [None] * P, "dW2": [None] * P, "db1": [None] * P,
           "db2": [None] * P, "Y_last": [None] * m, "dX0": [None] * m}

    def acc(key, s, val):
        if val is None:
            return
        out[key][s] = val if out[key][s] is None else out[key][s] + val

    def do_b(s, j):
        st = stages[s]
        _, dh, dx = backward_input(dY[(s, j)], st["W1"], st.get("W2"), H[(s, j)], act)
        dH[(s, j)] = rnd(dh)
        dx = rnd(dx)
        if s == 0:
            out["dX0"][j] = dx
        else:
            dY[(s - 1, j)] = dx

    def do_w(s, j):
        dw1, dw2, db1, db2 = backward_weight(X[(s, j)], A[(s, j)], dH[(s, j)], dY[(s, j)], act)
        acc("dW1", s, dw1)
        acc("dW2", s, dw2)
        acc("db1", s, db1)
        acc("db2", s, db2)

    for kind, s, j in ops:
        if kind == "F":
            st = stages[s]
            h_, a_, y_ = forward(X[(s, j)], st["W1"], st.get("W2"), st.get("b1"), st.get("b2"), act)
            H[(s, j)] = rnd(h_)
            A[(s, j)] = rnd(a_)
            y_ = rnd(y_)
            if s == P - 1:
                out["Y_last"][j] = y_
            else:
                X[(s + 1, j)] = y_
        elif kind == "B":
            do_b(s, j)
        elif kind == "W":
            do_w(s, j)
        elif kind == "BW":
            do_b(s, j)
            do_w(s, j)
        elif kind == "OPT":
            pass
        else:
            raise ValueError(kind)
    return out


def bf16_round(a):
    """Round fp64 values to the nearest bfloat16 value (ties to even), via fp32.

    Used only by the optional rounding-emulating chain; rounding through fp32
    first can differ from a direct fp64 -> bf16 rounding in rare halfway cases.
    """
    a32 = np.asarray(a, dtype=np.float32)
    bits = a32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    out = rounded.astype(np.uint32).view(np.float32)
    nan = np.isnan(a32)
    if nan.any():
        out = np.where(nan, a32, out)
    return out.astype(np.float64)
