"""GPU replays of the multi-chunk orderings (ZB-V and interleaved 1F1B).

A stage holding v chunks makes the model a chain of v P virtual stages
("ZB-PP" summary, §6 "ZB-V"; "Pipeline Schedules", "Interleaved stages").
The replay of a chunked list must compute exactly what the plain replay of
that chain computes: every virtual stage's weight gradients are accumulated
in ascending microbatch order in both, so outputs and gradients are
bit-identical.  They are also compared with the fp64 oracle chain that
rounds at the same five storage points, and the stage-parallel replay (one
stream per stage) with the serial one.

Chain tolerance: 5e-3 is the bound of one pass (bf16 operands, fp32
accumulation).  End to end, stage 0's gradients sit at the end of a path of
2L passes, and wherever the GPU's fp32 value and the oracle's fp64 value fall
on different sides of a bf16 rounding boundary the two chains carry
independent one-ulp differences onward; those add in quadrature, so the
bound grows with the square root of the depth: 5e-3 sqrt(L / 2) (equal to
the one-pass bound for a two-stage chain).
"""

import numpy as np
import pytest
import torch

from oracle import block as ob
from oracle import interleaved as IL
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


def _setup(L, m, M, h, f, seed):
    stages, X0, dY = I.pipeline_draws(L, m, M, h, f, seed=seed)
    wts = [{"W1": dev_bf16(st.W1), "W2": dev_bf16(st.W2)} for st in stages]
    return wts, [dev_bf16(x) for x in X0], [dev_bf16(g) for g in dY]


def _replay(zb, pl, wts, X0, dY, ops, M, h, f):
    m = len(X0)
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    zb.zb_run_stage_schedule(pl, stages, X0, dY, dX0, Yl, ops, ws, ws.numel())
    sync(zb)
    return stages, dX0, Yl


def _same(a, b):
    sa, xa, ya = a
    sb, xb, yb = b
    for p, q in zip(sa, sb):
        assert torch.equal(p["dW1"], q["dW1"]) and torch.equal(p["dW2"], q["dW2"])
    for p, q in zip(xa + ya, xb + yb):
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))


CASES = [("ZBV", 2, 2, 4), ("ZBV", 3, 2, 5), ("1F1B-I", 2, 2, 4), ("1F1B-I", 2, 3, 2)]


@pytest.mark.parametrize("kind,P,v,m", CASES)
def test_chunked_replay_is_the_chain_replay(zb, kind, P, v, m):
    M, h, f = 136, 72, 200
    L = v * P
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(L, m, M, h, f, seed=31 + L + m)
    ops = zb.zb_make_interleaved_schedule(kind, P, v, m)
    got = _replay(zb, zb.make_pipeline(P, m, blk, chunks=v, layout=kind), wts, X0, dY, ops, M, h, f)
    ref = _replay(zb, zb.make_pipeline(L, m, blk), wts, X0, dY, zb.zb_make_schedule("1F1B", L, m), M, h, f)
    _same(got, ref)
    # and the oracle chain, replaying the same list on the virtual stages
    st64 = [{"W1": f64(w["W1"]), "W2": f64(w["W2"])} for w in wts]
    emul = ob.run_pipeline(st64, [f64(x) for x in X0], [f64(g) for g in dY], IL.to_virtual(kind, P, ops),
                           round_fn=ob.bf16_round)
    stages, dX0, Yl = got
    tol = TOL_BF16 * np.sqrt(L / 2)
    for k in range(L):
        assert ob.rel_fro(f64(stages[k]["dW1"]), emul["dW1"][k]) < tol
        assert ob.rel_fro(f64(stages[k]["dW2"]), emul["dW2"][k]) < tol
    for j in range(m):
        assert ob.rel_fro(f64(Yl[j]), emul["Y_last"][j]) < tol
        assert ob.rel_fro(f64(dX0[j]), emul["dX0"][j]) < tol


@pytest.mark.parametrize("kind,P,v,m", [("ZBV", 2, 2, 4), ("1F1B-I", 2, 2, 4)])
def test_stage_parallel_chunked_replay_is_bit_identical(zb, kind, P, v, m):
    M, h, f = 136, 72, 200
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(v * P, m, M, h, f, seed=77)
    ops = zb.zb_make_interleaved_schedule(kind, P, v, m)
    serial = _replay(zb, zb.make_pipeline(P, m, blk, chunks=v, layout=kind), wts, X0, dY, ops, M, h, f)
    par = _replay(zb, zb.make_pipeline(P, m, blk, chunks=v, layout=kind, streams=P), wts, X0, dY, ops, M, h, f)
    _same(serial, par)


def test_zbv_replay_at_measured_times_and_stats(zb):
    """A list simulated with unequal pass times (and T_comm) replays the same
    chain; the replay's OPT markers write each virtual stage's state."""
    P, v, m, M, h, f = 2, 2, 5, 136, 72, 200
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(v * P, m, M, h, f, seed=5)
    _, ops = zb.zb_simulate_interleaved_schedule("ZBV", P, v, m, 1.0, 1.3, 0.7, 0.1, want_ops=True)
    pl = zb.make_pipeline(P, m, blk, chunks=v, layout="ZBV")
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h),
                   grad_stats=torch.full((2,), -1.0, dtype=torch.float64, device="cuda")) for w in wts]
    zb.zb_run_stage_schedule(pl, stages, X0, dY, None, None, ops, ws, ws_bytes)
    sync(zb)
    ref = _replay(zb, zb.make_pipeline(v * P, m, blk), wts, X0, dY, zb.zb_make_schedule("ZBH1", v * P, m),
                  M, h, f)
    for k in range(v * P):
        assert torch.equal(stages[k]["dW1"], ref[0][k]["dW1"])
        st = stages[k]["grad_stats"].cpu().numpy()
        g = np.concatenate([f64(stages[k]["dW1"]).ravel(), f64(stages[k]["dW2"]).ravel()])
        assert st[1] == 0 and abs(st[0] - float(np.sum(g * g))) <= 1e-6 * st[0]


def test_zbv_replay_with_bias_is_the_chain_replay(zb):
    P, v, m, M, h, f = 2, 2, 3, 136, 72, 200
    L = v * P
    blk = zb.make_block(M, h, f, has_bias=True)
    stages_d, X0, dY = I.pipeline_draws(L, m, M, h, f, seed=8, bias=True)
    wts = [{"W1": dev_bf16(st.W1), "W2": dev_bf16(st.W2), "b1": dev_bf16(st.b1), "b2": dev_bf16(st.b2)}
           for st in stages_d]
    X0 = [dev_bf16(x) for x in X0]
    dY = [dev_bf16(g) for g in dY]

    def run(pl, ops):
        ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h), db1=empty_f32(f), db2=empty_f32(h))
                  for w in wts]
        Yl = [empty_bf16(M, h) for _ in range(m)]
        zb.zb_run_stage_schedule(pl, stages, X0, dY, None, Yl, ops, ws, ws_bytes)
        sync(zb)
        return stages, Yl

    a = run(zb.make_pipeline(P, m, blk, chunks=2, layout="ZBV"), zb.zb_make_interleaved_schedule("ZBV", P, 2, m))
    b = run(zb.make_pipeline(L, m, blk), zb.zb_make_schedule("ZBH1", L, m))
    for p, q in zip(a[0], b[0]):
        for key in ("dW1", "dW2", "db1", "db2"):
            assert torch.equal(p[key], q[key])
    for p, q in zip(a[1], b[1]):
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))


@pytest.mark.parametrize("kind,P,v,m", [("ZBV", 2, 2, 4), ("ZBV", 3, 2, 5), ("1F1B-I", 2, 2, 4)])
def test_chunked_replay_per_pass_against_oracle(zb, kind, P, v, m):
    """Every pass of a chunked replay at the one-pass bound (5e-3).

    Single-pass calls along the chain of virtual stages reproduce the
    chunked replay bit for bit; each of their passes is then compared with
    the fp64 oracle from the exact bf16 tensors it consumed, so no part of
    the replay is checked only through the chain bound above.
    """
    from tests.test_gpu_parity import _hand_chain
    M, h, f = 136, 72, 200
    L = v * P
    wts, X0, dY = _setup(L, m, M, h, f, seed=41 + L + m)
    ops = zb.zb_make_interleaved_schedule(kind, P, v, m)
    blk = zb.make_block(M, h, f)
    stages, dX0, Yl = _replay(zb, zb.make_pipeline(P, m, blk, chunks=v, layout=kind), wts, X0, dY, ops,
                              M, h, f)
    rec, Xs, dYs, dWs = _hand_chain(zb, zb.make_block(M, h, f, split_k=False), L, m, wts, X0, dY)
    for k in range(L):
        assert torch.equal(stages[k]["dW1"], dWs[k][0]) and torch.equal(stages[k]["dW2"], dWs[k][1])
    for j in range(m):
        assert torch.equal(dX0[j].view(torch.int16), rec[("B", 0, j)][1].view(torch.int16))
        assert torch.equal(Yl[j].view(torch.int16), rec[("F", L - 1, j)][2].view(torch.int16))
    for k in range(L):
        W1, W2 = f64(wts[k]["W1"]), f64(wts[k]["W2"])
        for j in (0, m - 1):
            H, A, Y = rec[("F", k, j)]
            Hr, Ar, Yr = ob.forward(f64(Xs[(k, j)]), W1, W2)
            assert ob.rel_fro(f64(H), Hr) < TOL_BF16
            assert ob.rel_fro(f64(A), Ar) < TOL_BF16
            assert ob.rel_fro(f64(Y), f64(A) @ W2) < TOL_BF16
            dH, dX = rec[("B", k, j)]
            _, dHr, _ = ob.backward_input(f64(dYs[(k, j)]), W1, W2, f64(H))
            assert ob.rel_fro(f64(dH), dHr) < TOL_BF16
            assert ob.rel_fro(f64(dX), f64(dH) @ W1.T) < TOL_BF16
        r1 = np.zeros((h, f))
        r2 = np.zeros((f, h))
        for j in range(m):
            _, A, _ = rec[("F", k, j)]
            dH, _ = rec[("B", k, j)]
            a, b, _, _ = ob.backward_weight(f64(Xs[(k, j)]), f64(A), f64(dH), f64(dYs[(k, j)]))
            r1 += a
            r2 += b
        assert ob.rel_fro(f64(stages[k]["dW1"]), r1) < TOL_BF16
        assert ob.rel_fro(f64(stages[k]["dW2"]), r2) < TOL_BF16


@pytest.mark.parametrize("kind", ["ZBV", "1F1B-I"])
def test_chunked_pipeline_as_benchmarked(zb, kind):
    """The two-chunk P=4, h=1024 pipeline (8 blocks, 4 x 512 tokens per
    microbatch, m=8) in the launch configuration the benchmark times: 12
    streams, one step captured into a CUDA graph and replayed twice, bit for
    bit the serial eager replay of the same list."""
    P, v, m, M, h = 4, 2, 8, 2048, 1024
    f = 4 * h
    L = P * v
    blk = zb.make_block(M, h, f)
    gen = torch.Generator(device="cuda").manual_seed(17)
    bf = torch.bfloat16
    wts = [{"W1": (torch.randn(h, f, device="cuda", generator=gen) * 0.02).to(bf),
            "W2": (torch.randn(f, h, device="cuda", generator=gen) * 0.02).to(bf)} for _ in range(L)]
    X0 = [torch.randn(M, h, device="cuda", generator=gen).to(bf) for _ in range(m)]
    dY = [torch.randn(M, h, device="cuda", generator=gen).to(bf) for _ in range(m)]
    ops = zb.zb_make_interleaved_schedule(kind, P, v, m)
    ref = _replay(zb, zb.make_pipeline(P, m, blk, chunks=v, layout=kind), wts, X0, dY, ops, M, h, f)
    pl = zb.make_pipeline(P, m, blk, chunks=v, layout=kind, streams=3 * P)
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    ops_c = zb.ops_array(ops)
    zb.zb_run_stage_schedule(pl, stages, X0, dY, dX0, Yl, ops_c, ws, ws_bytes)  # eager: makes the lanes
    sync(zb)
    for s in stages:
        s["dW1"].fill_(float("nan"))
        s["dW2"].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            zb.zb_run_stage_schedule(pl, stages, X0, dY, dX0, Yl, ops_c, ws, ws_bytes, None, side)
    for _ in range(2):
        g.replay()
        sync(zb)
        _same((stages, dX0, Yl), ref)
