"""The allocation-free replay (zb_run_stage_schedule_static) against the
workspace replay (zb_run_stage_schedule).

Some callers cannot allocate device memory: a custom operator inside a
framework that owns every byte through its own pool, or a latency-critical
loop that must not call cudaMalloc / cudaFree because they can synchronise
the device.  For them the library keeps the replay's activation arena in a
static device array.  This file is collected last on purpose, so a failure
here comes after every other test has run.
"""

import pytest
import torch

from oracle import block as ob
from split_backward_gemms_gb300 import inputs as I
from tests.gpu_util import dev_bf16, empty_bf16, empty_f32, f64, have_gpu, sync

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3


@pytest.fixture(scope="module")
def zb():
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def _outputs(P, m, M, h, f, wts):
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    return stages, dX0, Yl


def _same(a, b):
    assert ob.rel_fro(f64(a), f64(b)) < TOL_BF16
    ia = a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16)
    ib = b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)
    assert torch.equal(ia, ib)


def test_static_arena_replay_matches_workspace_replay(zb):
    P, m, M, h, f = 2, 4, 256, 256, 1024
    draws, X0n, dYn = I.pipeline_draws(P, m, M, h, f, seed=21)
    wts = [{"W1": dev_bf16(s.W1), "W2": dev_bf16(s.W2)} for s in draws]
    X0 = [dev_bf16(x) for x in X0n]
    dY = [dev_bf16(g) for g in dYn]
    ops = zb.zb_make_schedule("ZBH1", P, m)
    pl = zb.make_pipeline(P, m, zb.make_block(M, h, f))
    need, _ = zb.zb_schedule_workspace_size(pl, ops)
    assert need <= zb.ZB_STATIC_ARENA_BYTES

    ref_st, ref_dx, ref_y = _outputs(P, m, M, h, f, wts)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    zb.zb_run_stage_schedule(pl, ref_st, X0, dY, ref_dx, ref_y, ops, ws, need)
    sync(zb)

    for _ in range(2):  # two calls in a row share (and reuse) the static arena
        st, dx, y = _outputs(P, m, M, h, f, wts)
        zb.zb_run_stage_schedule_static(pl, st, X0, dY, dx, y, ops)
        sync(zb)
        for s in range(P):
            _same(st[s]["dW1"], ref_st[s]["dW1"])
            _same(st[s]["dW2"], ref_st[s]["dW2"])
        for j in range(m):
            _same(dx[j], ref_dx[j])
            _same(y[j], ref_y[j])


def test_static_arena_rejects_oversized_lists(zb):
    P, m, M, h, f = 4, 8, 2048, 1024, 4096
    ops = zb.zb_make_schedule("ZBH1", P, m)
    pl = zb.make_pipeline(P, m, zb.make_block(M, h, f))
    need, _ = zb.zb_schedule_workspace_size(pl, ops)
    assert need > zb.ZB_STATIC_ARENA_BYTES
    X = [torch.empty(16, dtype=torch.uint8, device="cuda")] * m
    stages = [{"W1": X[0], "W2": X[0], "dW1": X[0], "dW2": X[0]} for _ in range(P)]
    with pytest.raises(zb.ZBError) as e:
        zb.zb_run_stage_schedule_static(pl, stages, X, X, None, None, ops)
    assert e.value.status == zb.ZB_ERR_WORKSPACE
    assert "static arena" in zb.zb_last_error()
