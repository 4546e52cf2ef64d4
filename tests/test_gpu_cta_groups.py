"""The GPU parity suite with each GEMM CTA-group shape forced.

The library picks the CTA-pair kernel (256x256 tiles on two SMs) for large
problems and the one-CTA kernel (128x256 tiles) for small ones; forcing each
shape in a fresh process (the choice is read once, from ZB_GEMM_CTA_GROUP)
runs both kernels over the ragged small shapes and the full-size ones.
"""

import os
import subprocess
import sys

import pytest

from tests.gpu_util import have_gpu

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_parity_suite_with_forced_cta_group(cg):
    if not have_gpu():
        pytest.skip("no CUDA device")
    env = dict(os.environ, ZB_GEMM_CTA_GROUP=cg)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_gpu_parity.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-4000:] + r.stderr[-2000:])
