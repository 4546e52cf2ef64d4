"""Launch modes and copy policies change timing only, never bits.

GEMMs that follow each other on one stream launch as programmatic dependents
(their setup overlaps the previous GEMM's tail, their first global access
waits for it to complete; the W pass's second GEMM, independent of the
first, runs beside it and waits for it before exiting).  ZB_GEMM_PDL=0 turns that off and ZB_GEMM_PDL=1
turns it on inside every replay lane; the setting is read once per process,
so each mode runs in a fresh process on the same seeded inputs: single passes
(with and without split K) and replays on one lane, on an F/B lane beside a W
lane, on four stage lanes and on an F, a B and a W lane per stage must give
the same bits in every mode (and long-K passes with and without the GeLU
epilogues' hand-off between warps).  And a
process whose first library calls are made inside a CUDA graph capture (the
split-K occupancy query and the programmatic launches among them) replays
the graph to the bits of the same passes run eagerly.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from split_backward_gemms_gb300 import inputs as I
from tests.gpu_util import dev_bf16, empty_bf16, empty_f32, have_gpu, sync

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _bits(t):
    return (t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)).cpu().numpy()


def _child(out_path):
    """Runs the passes and replays of this file and saves every output's bits."""
    from split_backward_gemms_gb300 import zb
    res = {}
    # single passes: one shape that splits K (F2 / B2), one that does not
    for M, h, f in ((256, 1024, 4096), (640, 512, 2048)):
        stages, X0, dY = I.pipeline_draws(1, 1, M, h, f, seed=M + h, bias=True)
        st = stages[0]
        X, G = dev_bf16(X0[0]), dev_bf16(dY[0])
        W1, W2, b1, b2 = dev_bf16(st.W1), dev_bf16(st.W2), dev_bf16(st.b1), dev_bf16(st.b2)
        blk = zb.make_block(M, h, f, has_bias=True)
        H, A, Y = empty_bf16(M, f), empty_bf16(M, f), empty_bf16(M, h)
        zb.zb_forward(blk, X, W1, W2, b1, b2, H, A, Y)
        dH, dX = empty_bf16(M, f), empty_bf16(M, h)
        zb.zb_backward_input(blk, G, W1, W2, H, dH, dX)
        dW1, dW2, db1, db2 = empty_f32(h, f), empty_f32(f, h), empty_f32(f), empty_f32(h)
        zb.zb_backward_weight(blk, X, A, dH, G, dW1, dW2, db1, db2, 0)
        # fifteen accumulating W passes right behind the first, on alternating
        # operands: each pass's dW1 GEMM starts beside its dW2 GEMM and must
        # still follow the previous pass's dW1 GEMM (a lost or reordered
        # update changes the fp32 bits)
        dH_alt, G_alt = dH.flip(0).contiguous(), G.flip(0).contiguous()
        for k in range(15):
            if k % 2:
                zb.zb_backward_weight(blk, X, A, dH, G, dW1, dW2, db1, db2, 1)
            else:
                zb.zb_backward_weight(blk, X, A, dH_alt, G_alt, dW1, dW2, db1, db2, 1)
        sync(zb)
        for k, v in dict(H=H, A=A, Y=Y, dH=dH, dX=dX, dW1=dW1, dW2=dW2, db1=db1, db2=db2).items():
            res[f"pass{M}_{k}"] = _bits(v)
    # long K (>= 64 blocks of 64) on CTA pairs: the GeLU and GeLU' epilogues
    # hand raw accumulator chunks from one warp to another (ragged edges,
    # bias, both activations)
    for M, h, f, act, bias in ((520, 4104, 1048, zb.ZB_ACT_GELU_ERF, True),
                               (392, 4096, 776, zb.ZB_ACT_GELU_TANH, False)):
        stages, X0, dY = I.pipeline_draws(1, 1, M, h, f, seed=M + h, bias=True)
        st = stages[0]
        X, G = dev_bf16(X0[0]), dev_bf16(dY[0])
        W1, W2 = dev_bf16(st.W1), dev_bf16(st.W2)
        b1, b2 = (dev_bf16(st.b1), dev_bf16(st.b2)) if bias else (None, None)
        blk = zb.make_block(M, h, f, act=act, has_bias=bias, split_k=False)
        H, A, Y = empty_bf16(M, f), empty_bf16(M, f), empty_bf16(M, h)
        zb.zb_forward(blk, X, W1, W2, b1, b2, H, A, Y)
        dH, dX = empty_bf16(M, f), empty_bf16(M, h)
        zb.zb_backward_input(blk, G, W1, W2, H, dH, dX)
        sync(zb)
        for k, v in dict(H=H, A=A, Y=Y, dH=dH, dX=dX).items():
            res[f"longk{M}_{k}"] = _bits(v)
    # replays: one lane, F/B lane + W lane (one stage), four stage lanes
    for name, P, m, streams, kind in (("serial", 2, 4, 1, "ZBH1"), ("wlane", 1, 6, 2, "ZBH2"),
                                      ("stages", 4, 8, 4, "ZBH1"), ("fbw", 4, 8, 12, "ZBH2")):
        M, h, f = 512, 256, 1024
        stages, X0, dY = I.pipeline_draws(P, m, M, h, f, seed=P * 10 + m)
        wts = [{"W1": dev_bf16(s.W1), "W2": dev_bf16(s.W2), "dW1": empty_f32(h, f), "dW2": empty_f32(f, h)}
               for s in stages]
        X0 = [dev_bf16(x) for x in X0]
        dY = [dev_bf16(g) for g in dY]
        ops = zb.zb_make_schedule(kind, max(P, 8) if P == 1 else P, m)
        if P == 1:
            ops = [(k, 0, j) for k, s, j in ops if s == 0]
        pl = zb.make_pipeline(P, m, zb.make_block(M, h, f), streams=streams)
        ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        dX0 = [empty_bf16(M, h) for _ in range(m)]
        Yl = [empty_bf16(M, h) for _ in range(m)]
        zb.zb_run_stage_schedule(pl, wts, X0, dY, dX0, Yl, ops, ws, ws.numel())
        sync(zb)
        for s in range(P):
            res[f"{name}_dW1_{s}"] = _bits(wts[s]["dW1"])
            res[f"{name}_dW2_{s}"] = _bits(wts[s]["dW2"])
        for j in range(m):
            res[f"{name}_dX0_{j}"] = _bits(dX0[j])
            res[f"{name}_Y_{j}"] = _bits(Yl[j])
    np.savez(out_path, **res)


# Each mode: environment settings of a fresh process.  The L2 eviction
# priorities of the GEMM's copies (ZB_GEMM_L2_HINTS=0 turns them off) only
# decide where data sits in L2, the W pass's paced reduce-adds only decide
# when each is issued, its two GEMMs in one grouped launch
# (ZB_GEMM_GROUP_W=0: two launches) compute every tile as before, and the
# long-K GeLU epilogues' hand-off (ZB_GEMM_HANDOFF=0: every warp does its
# own rows) only moves the same fp32 sums between warps: none may change a
# bit either.
MODES = {"default": {}, "pdl0": {"ZB_GEMM_PDL": "0"}, "pdl1": {"ZB_GEMM_PDL": "1"},
         "nohints": {"ZB_GEMM_L2_HINTS": "0"}, "twolaunchw": {"ZB_GEMM_GROUP_W": "0"},
         "nohandoff": {"ZB_GEMM_HANDOFF": "0"}}


def test_launch_modes_change_no_bits(tmp_path):
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    res = {}
    for mode, extra in MODES.items():
        out = str(tmp_path / f"mode_{mode}.npz")
        env = dict(os.environ)
        for k in ("ZB_GEMM_PDL", "ZB_GEMM_L2_HINTS", "ZB_GEMM_GROUP_W", "ZB_GEMM_HANDOFF"):
            env.pop(k, None)
        env.update(extra)
        code = f"import tests.test_gpu_launch_modes as t; t._child({out!r})"
        r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
        res[mode] = np.load(out)
    keys = res["default"].files
    assert len(keys) > 40
    for mode in MODES:
        assert res[mode].files == keys
        for k in keys:
            assert np.array_equal(res[mode][k], res["default"][k]), (mode, k)


def _graph_child(out_path):
    """The first library calls of the process happen inside a CUDA graph
    capture: single passes at a split-K shape (its occupancy query and
    programmatic launches included), then the graph is replayed and
    compared with the same passes run eagerly afterwards."""
    from split_backward_gemms_gb300 import zb
    M, h, f = 256, 1024, 4096
    stages, X0, dY = I.pipeline_draws(1, 1, M, h, f, seed=21, bias=True)
    st = stages[0]
    X, G = dev_bf16(X0[0]), dev_bf16(dY[0])
    W1, W2, b1, b2 = dev_bf16(st.W1), dev_bf16(st.W2), dev_bf16(st.b1), dev_bf16(st.b2)
    blk = zb.make_block(M, h, f, has_bias=True)

    def outs():
        return dict(H=empty_bf16(M, f), A=empty_bf16(M, f), Y=empty_bf16(M, h), dH=empty_bf16(M, f),
                    dX=empty_bf16(M, h))

    def run(o, stream):
        zb.zb_forward(blk, X, W1, W2, b1, b2, o["H"], o["A"], o["Y"], stream)
        zb.zb_backward_input(blk, G, W1, W2, o["H"], o["dH"], o["dX"], stream)

    torch.cuda.synchronize()
    g_out = outs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            run(g_out, side)
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    e_out = outs()
    run(e_out, torch.cuda.current_stream())
    sync(zb)
    np.savez(out_path, **{f"g_{k}": _bits(v) for k, v in g_out.items()},
             **{f"e_{k}": _bits(v) for k, v in e_out.items()})


def test_first_calls_inside_graph_capture(tmp_path):
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    out = str(tmp_path / "graph.npz")
    code = f"import tests.test_gpu_launch_modes as t; t._graph_child({out!r})"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    res = np.load(out)
    for k in ("H", "A", "Y", "dH", "dX"):
        assert np.array_equal(res[f"g_{k}"], res[f"e_{k}"]), k
        assert not np.array_equal(res[f"g_{k}"], np.full_like(res[f"g_{k}"], res[f"g_{k}"].flat[0])), k
