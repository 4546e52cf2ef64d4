"""The GPU parity suite with each GEMM tile shape forced.

The library picks the CTA-pair kernel (256 x 256 tiles on two SMs) for large
problems and the one-CTA kernel (128 x 256 tiles) for small ones; forcing
each shape in a fresh process (the choice is read once, from
ZB_GEMM_CTA_GROUP) runs both kernels over the ragged small shapes and the
full-size ones of the parity file.

A second test compares the bits of the two shapes: with K never split,
every output element is the same ascending-K sum of the same bf16 products
in both (only the MMA's M and its CTA group differ), so the outputs are
bit-identical, and the results do not depend on which shape the problem's
size selects.
"""

import os
import subprocess
import sys

import numpy as np
import pytest

from tests.gpu_util import have_gpu

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

SHAPES = ["1", "2"]


@pytest.mark.parametrize("cg", SHAPES)
def test_parity_suite_with_forced_cta_group(cg):
    if not have_gpu():
        pytest.skip("no CUDA device")
    env = dict(os.environ, ZB_GEMM_CTA_GROUP=cg)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_gpu_parity.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-4000:] + r.stderr[-2000:])


def _child(out_path):
    """Every pass at a few shapes (ragged edges included), bits saved."""
    import torch

    from split_backward_gemms_gb300 import inputs as I
    from split_backward_gemms_gb300 import zb
    from tests.gpu_util import dev_bf16, empty_bf16, empty_f32, sync
    res = {}
    for M, h, f in ((520, 264, 1048), (2048, 1024, 4096), (136, 72, 200)):
        stages, X0, dY = I.pipeline_draws(1, 1, M, h, f, seed=3 * M + h, bias=True)
        st = stages[0]
        X, G = dev_bf16(X0[0]), dev_bf16(dY[0])
        W1, W2, b1, b2 = dev_bf16(st.W1), dev_bf16(st.W2), dev_bf16(st.b1), dev_bf16(st.b2)
        blk = zb.make_block(M, h, f, has_bias=True, split_k=False)
        H, A, Y = empty_bf16(M, f), empty_bf16(M, f), empty_bf16(M, h)
        zb.zb_forward(blk, X, W1, W2, b1, b2, H, A, Y)
        dH, dX = empty_bf16(M, f), empty_bf16(M, h)
        zb.zb_backward_input(blk, G, W1, W2, H, dH, dX)
        dW1, dW2, db1, db2 = empty_f32(h, f), empty_f32(f, h), empty_f32(f), empty_f32(h)
        zb.zb_backward_weight(blk, X, A, dH, G, dW1, dW2, db1, db2, 0)
        zb.zb_backward_weight(blk, X, A, dH, G, dW1, dW2, db1, db2, 1)
        sync(zb)
        for name, t in (("H", H), ("A", A), ("Y", Y), ("dH", dH), ("dX", dX), ("dW1", dW1), ("dW2", dW2)):
            v = t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)
            res[f"{M}x{h}x{f}/{name}"] = v.cpu().numpy()
    np.savez(out_path, **res)


def test_cta_groups_give_identical_bits(tmp_path):
    if not have_gpu():
        pytest.skip("no CUDA device")
    outs = []
    for cg in SHAPES:
        out = str(tmp_path / f"bits_{cg}.npz")
        env = dict(os.environ, ZB_GEMM_CTA_GROUP=cg)
        code = f"import sys; sys.path.insert(0, {ROOT!r}); from tests.test_gpu_cta_groups import _child; _child({out!r})"
        r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
        outs.append(np.load(out))
    ref = outs[0]
    for cg, got in zip(SHAPES[1:], outs[1:]):
        for k in ref.files:
            assert np.array_equal(ref[k], got[k]), f"{k}: CTA group {cg} differs"
