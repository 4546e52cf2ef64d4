"""Seeded random shapes through every GEMM path, against the fp64 oracle.

Twenty (M, h, f) triples drawn from a fixed seed — M in [1, 3000], h and f
multiples of 8 in [8, 2048] and [8, 8192], at most ~2 GFLOP per GEMM — with
bias on or off and the erf or tanh GeLU, so that one-CTA tiles, CTA pairs and
split K (S = 2 and 4) all occur with ragged M, N and K.  Each stored value of
the F and B passes lies within its own bf16 rounding (2^-8 relative, covering
the fp32 accumulation and the GeLU approximation) plus 1e-4 of the largest
magnitude; the fp32 weight gradients within 5e-3 relative Frobenius error.
"""

import numpy as np
import pytest

from oracle import block as ob
from split_backward_gemms_gb300 import inputs as I
from tests.gpu_util import dev_bf16, empty_bf16, empty_f32, f64, have_gpu, sync

pytestmark = pytest.mark.gpu

ACTS = {"gelu_erf": 1, "gelu_tanh": 2}


def _shapes(n=20, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M = int(rng.integers(1, 3001))
        h = 8 * int(rng.integers(1, 257))
        f = 8 * int(rng.integers(1, 1025))
        if 2.0 * M * h * f > 2e9:
            continue
        bias = bool(rng.integers(0, 2))
        act = "gelu_tanh" if rng.integers(0, 4) == 0 else "gelu_erf"
        out.append((M, h, f, bias, act))
    return out


@pytest.fixture(scope="module")
def zb():
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def _close(got, ref, what):
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * np.max(np.abs(ref))
    bad = err > bound
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:3].tolist())


@pytest.mark.parametrize("M,h,f,bias,act", _shapes())
def test_random_shapes_match_oracle(zb, M, h, f, bias, act):
    stages, X0, dY = I.pipeline_draws(1, 1, M, h, f, seed=M ^ (h << 3) ^ (f << 7), bias=bias)
    st = stages[0]
    X, G = dev_bf16(X0[0]), dev_bf16(dY[0])
    W1, W2 = dev_bf16(st.W1), dev_bf16(st.W2)
    b1 = dev_bf16(st.b1) if bias else None
    b2 = dev_bf16(st.b2) if bias else None
    blk = zb.make_block(M, h, f, zb.ZB_DT_BF16, ACTS[act], bias)
    H, A, Y = empty_bf16(M, f), empty_bf16(M, f), empty_bf16(M, h)
    zb.zb_forward(blk, X, W1, W2, b1, b2, H, A, Y)
    dH, dX = empty_bf16(M, f), empty_bf16(M, h)
    zb.zb_backward_input(blk, G, W1, W2, H, dH, dX)
    dW1, dW2 = empty_f32(h, f), empty_f32(f, h)
    db1 = empty_f32(f) if bias else None
    db2 = empty_f32(h) if bias else None
    zb.zb_backward_weight(blk, X, A, dH, G, dW1, dW2, db1, db2, 0)
    sync(zb)
    Xd, W1d, W2d, Gd = f64(X), f64(W1), f64(W2), f64(G)
    b1d = f64(b1) if bias else None
    b2d = f64(b2) if bias else None
    Hr, Ar, _ = ob.forward(Xd, W1d, W2d, b1d, b2d, act)
    _close(f64(H), Hr, "H")
    _close(f64(A), Ar, "A")
    _close(f64(Y), f64(A) @ W2d + (b2d[None, :] if bias else 0.0), "Y")
    _, dHr, _ = ob.backward_input(Gd, W1d, W2d, f64(H), act)
    _close(f64(dH), dHr, "dH")
    _close(f64(dX), f64(dH) @ W1d.T, "dX")
    dW1r, dW2r, db1r, db2r = ob.backward_weight(Xd, f64(A), f64(dH), Gd, act)
    assert ob.rel_fro(f64(dW1), dW1r) < 5e-3
    assert ob.rel_fro(f64(dW2), dW2r) < 5e-3
    if bias:
        assert ob.rel_fro(f64(db1), db1r) < 5e-3
        assert ob.rel_fro(f64(db2), db2r) < 5e-3
