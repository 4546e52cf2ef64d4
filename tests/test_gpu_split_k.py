"""Split-K GEMMs: shapes with too few output tiles to occupy the GPU.

When a bf16-output GEMM of the F or B pass has few 128x256 tiles and a long K
loop, the library computes each tile with a cluster of S CTAs (S = 2 or 4),
one per K range; the fp32 partial tiles are exchanged through distributed
shared memory and summed in rank order before the epilogue.  The shapes below
take each S on the F and B GEMMs (every epilogue: bf16 store, GeLU dual
store, GeLU' product; ragged M, N and K), checked element by element against
the fp64 oracle from the GPU's own saved tensors: every stored value must lie
within its own bf16 rounding (2^-9 relative, taken as 2^-8 to cover the fp32
accumulation and the GeLU approximation) plus 1e-4 of the largest magnitude.
A dropped, doubled or misplaced K range or column slice breaks that bound by
orders of magnitude.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import block as ob
from split_backward_gemms_gb300 import inputs as I
from tests.gpu_util import dev_bf16, empty_bf16, f64, have_gpu, sync

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

ACTS = {"gelu_erf": 1, "gelu_tanh": 2}

# (M, h, f): split factors of (F1 H = X W1, F2 Y = A W2) with 152 SMs and at
# least 16 K blocks of 64 per CTA; the B GEMMs dA = dY W2^T (GeLU' epilogue)
# and dX = dH W1^T have the shapes of F1 and F2.
#   (256, 1024, 4096):  32 tiles, 16 K blocks -> no split;  8 tiles, 64 K blocks -> S=4
#   (200, 520, 2056):   18 tiles, 9 K blocks -> no split;
#                       6 tiles, 33 K blocks (ragged K, N and M) -> S=2 (ranges of 16 and 17)
#   (256, 2048, 8192):  64 tiles, 32 K blocks -> S=2;  16 tiles, 128 K blocks -> S=4
#   (200, 2056, 2104):  18 tiles, 33 K blocks -> S=2;  18 tiles, 33 K blocks -> S=2 (all ragged)
#   (2048, 1024, 4096): CTA-pair tiles for F1;  64 tiles, 64 K blocks -> S=2
# degenerate shapes:
#   (1, 1024, 4096) and (3, 520, 4104): one or three rows, F2 S=4 (4 and 3 tiles)
#   (130, 8, 4096):     F2 two tiles of 8 live columns, S=4 (three owners hold no column)
#   (1, 2048, 8):       F1 one tile of 8 live columns, 32 K blocks -> S=2
SHAPES = [(256, 1024, 4096), (200, 520, 2056), (256, 2048, 8192), (200, 2056, 2104), (2048, 1024, 4096),
          (1, 1024, 4096), (3, 520, 4104), (130, 8, 4096), (1, 2048, 8)]


@pytest.fixture(scope="module")
def zb():
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def _assert_close_elementwise(got, ref, what):
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * np.max(np.abs(ref))
    bad = err > bound
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:5].tolist(), float(err.max()))


def _passes(zb, M, h, f, act, bias, seed):
    stages, X0, dY = I.pipeline_draws(1, 1, M, h, f, seed=seed, bias=bias)
    st = stages[0]
    t = {"X": dev_bf16(X0[0]), "dY": dev_bf16(dY[0]), "W1": dev_bf16(st.W1), "W2": dev_bf16(st.W2)}
    if bias:
        t["b1"], t["b2"] = dev_bf16(st.b1), dev_bf16(st.b2)
    blk = zb.make_block(M, h, f, zb.ZB_DT_BF16, ACTS[act], bias)
    H, A, Y = empty_bf16(M, f), empty_bf16(M, f), empty_bf16(M, h)
    zb.zb_forward(blk, t["X"], t["W1"], t["W2"], t.get("b1"), t.get("b2"), H, A, Y)
    dH, dX = empty_bf16(M, f), empty_bf16(M, h)
    zb.zb_backward_input(blk, t["dY"], t["W1"], t["W2"], H, dH, dX)
    sync(zb)
    return t, {"H": H, "A": A, "Y": Y, "dH": dH, "dX": dX}


@pytest.mark.parametrize("M,h,f", SHAPES)
@pytest.mark.parametrize("act,bias", [("gelu_erf", False), ("gelu_tanh", True), ("gelu_erf", True)])
def test_split_k_passes_match_oracle_elementwise(zb, M, h, f, act, bias):
    t, o = _passes(zb, M, h, f, act, bias, seed=M + h + f)
    X, W1, W2, dY = (f64(t[k]) for k in ("X", "W1", "W2", "dY"))
    b1 = f64(t["b1"]) if bias else None
    b2 = f64(t["b2"]) if bias else None
    Hr, Ar, _ = ob.forward(X, W1, W2, b1, b2, act)
    _assert_close_elementwise(f64(o["H"]), Hr, "H")
    _assert_close_elementwise(f64(o["A"]), Ar, "A")
    Yr = f64(o["A"]) @ W2 + (b2[None, :] if bias else 0.0)
    _assert_close_elementwise(f64(o["Y"]), Yr, "Y")
    _, dHr, _ = ob.backward_input(dY, W1, W2, f64(o["H"]), act)
    _assert_close_elementwise(f64(o["dH"]), dHr, "dH")
    _assert_close_elementwise(f64(o["dX"]), f64(o["dH"]) @ W1.T, "dX")


def test_split_k_same_inputs_same_bits(zb):
    M, h, f = 200, 520, 2056
    _, a = _passes(zb, M, h, f, "gelu_erf", True, seed=3)
    _, b = _passes(zb, M, h, f, "gelu_erf", True, seed=3)
    for k in a:
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k


def _child(out_path, M, h, f):
    """Runs the F and B passes in this process and saves the outputs."""
    from split_backward_gemms_gb300 import zb as _zb
    _, o = _passes(_zb, M, h, f, "gelu_erf", True, seed=11)
    np.savez(out_path, **{k: v.view(torch.int16).cpu().numpy() for k, v in o.items()})


def test_split_and_unsplit_agree_up_to_summation_order(zb, tmp_path):
    """ZB_GEMM_SPLIT_K=1 turns the split off (read once per process, so each
    variant runs in a fresh process).  The two results differ in the order of
    the fp32 additions only: close to each other, and not bit-identical (which
    shows that the default run took the split path)."""
    M, h, f = 256, 1024, 4096
    res = {}
    for cap in ("4", "1"):
        out = str(tmp_path / f"cap{cap}.npz")
        env = dict(os.environ, ZB_GEMM_SPLIT_K=cap)
        code = f"import tests.test_gpu_split_k as t; t._child({out!r}, {M}, {h}, {f})"
        r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
        res[cap] = np.load(out)
    any_diff = False
    for k in ("H", "A", "Y", "dH", "dX"):
        a = torch.from_numpy(res["4"][k]).view(torch.bfloat16).double().numpy()
        b = torch.from_numpy(res["1"][k]).view(torch.bfloat16).double().numpy()
        assert ob.rel_fro(a, b) < 5e-3, k
        any_diff |= bool((res["4"][k] != res["1"][k]).any())
    assert any_diff
