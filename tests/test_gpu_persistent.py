"""The persistent replay executor: every GEMM of an op list in one kernel.

With zb_pipeline.executor = ZB_EXEC_PERSISTENT the executor records the GEMMs
an op list would launch and runs them all in one persistent kernel on CTA
pairs; a GEMM's tiles start once the earlier GEMMs whose buffers conflict
with its own have stored all of theirs (counters in the workspace).  Every
tile is the one-launch kernel's tile and the accumulating weight-gradient
GEMMs of a stage keep their list order, so outputs and gradients are the
serial replay's bit for bit: handcrafted and heuristic orderings, one stage
and several, plans by longest chain and in list order, ragged shapes and M
below one 128-row block (a one-CTA tile in the serial replay), chunked (ZB-V
and interleaved 1F1B) lists, both GeLU forms, gradient statistics at OPT,
accumulation into existing gradients, the allocation-free entry point, and a
CUDA graph.  The serial replay
is checked against the fp64 oracle elsewhere; one case here is also
compared with the rounding-emulating oracle chain directly.
"""

import numpy as np
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


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _setup(L, m, M, h, f, seed):
    stages, X0, dY = I.pipeline_draws(L, m, M, h, f, seed=seed)
    wts = [{"W1": dev_bf16(st.W1), "W2": dev_bf16(st.W2)} for st in stages]
    return wts, [dev_bf16(x) for x in X0], [dev_bf16(g) for g in dY]


def _ops(zb, kind, P, m, chunks):
    if chunks > 1:
        return zb.zb_make_interleaved_schedule(kind, P, chunks, m)
    if kind in ("ZB1P", "ZB2P"):
        limit = P if kind == "ZB1P" else 2 * P
        _, ops, _ = zb.zb_auto_schedule(P, m, 1.0, 1.0, 1.0, 0.0, limit, 1.0)
        return ops
    if P == 1:
        return [op for op in zb.zb_make_schedule(kind, 8, m) if op[1] == 0]
    return zb.zb_make_schedule(kind, P, m)


def _replay(zb, pl, wts, X0, dY, ops, M, h, f, stats_bufs=False, init=None, stats=None):
    m = len(X0)
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.full((max(ws_bytes, 256),), 255, dtype=torch.uint8, device="cuda")
    stages = []
    for k, w in enumerate(wts):
        d = dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h))
        if init is not None:
            d["dW1"].copy_(init[k][0])
            d["dW2"].copy_(init[k][1])
        if stats_bufs:
            d["grad_stats"] = torch.zeros(2, dtype=torch.float64, device="cuda")
        stages.append(d)
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    zb.zb_run_stage_schedule(pl, stages, X0, dY, dX0, Yl, ops, ws, ws.numel(), stats)
    sync(zb)
    return stages, dX0, Yl


def _same_bits(a, b, stats=False):
    sa, xa, ya = a
    sb, xb, yb = b
    for p, q in zip(sa, sb):
        assert torch.equal(_bits(p["dW1"]), _bits(q["dW1"]))
        assert torch.equal(_bits(p["dW2"]), _bits(q["dW2"]))
        if stats:
            assert torch.equal(p["grad_stats"], q["grad_stats"])
    for p, q in zip(xa + ya, xb + yb):
        assert torch.equal(_bits(p), _bits(q))


CASES = [
    # kind, P, m, M, h, f, chunks
    ("ZBH1", 4, 8, 512, 256, 1024, 1),
    ("ZB1P", 4, 8, 512, 256, 1024, 1),
    ("ZBH2", 8, 16, 256, 256, 512, 1),
    ("1F1B-I", 2, 4, 512, 256, 1024, 2),  # two chunks per stage, cyclic
    ("ZBH2", 4, 8, 512, 256, 1024, 1),
    ("1F1B", 4, 8, 512, 256, 1024, 1),
    ("ZB2P", 4, 8, 512, 256, 1024, 1),
    ("ZBH1", 2, 4, 520, 264, 1048, 1),   # ragged rows and columns
    ("ZBH1", 2, 3, 96, 256, 1024, 1),    # M below one 128-row block
    ("ZBH2", 1, 6, 512, 256, 1024, 1),   # one stage, its ZB-H2 list
    ("ZBV", 2, 4, 512, 256, 1024, 2),    # two chunks per stage, V-shaped
    ("ZBH1", 4, 8, 2048, 1024, 4096, 1),  # the 4-stage h=1024 pipeline
]


@pytest.mark.parametrize("kind,P,m,M,h,f,chunks", CASES)
def test_persistent_replay_is_the_serial_replay(zb, kind, P, m, M, h, f, chunks):
    L = P * chunks
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(L, m, M, h, f, seed=7 * P + m + M)
    ops = _ops(zb, kind, P, m, chunks)
    extra = dict(chunks=chunks, layout=kind) if chunks > 1 else {}
    ref = _replay(zb, zb.make_pipeline(P, m, blk, **extra), wts, X0, dY, ops, M, h, f, stats_bufs=True)
    st = zb.zb_run_stats()
    got = _replay(zb, zb.make_pipeline(P, m, blk, executor="persistent", **extra), wts, X0, dY, ops, M, h, f,
                  stats_bufs=True, stats=st)
    _same_bits(ref, got, stats=any(op[0] in ("OPT", 4) for op in ops))
    assert 2 <= st.n_gemm_launches <= 64  # the replay kernel and its table uploads
    # a second run over the same (reused) tables and counters
    got2 = _replay(zb, zb.make_pipeline(P, m, blk, executor="persistent", **extra), wts, X0, dY, ops, M, h, f,
                   stats_bufs=True)
    _same_bits(ref, got2)


def test_persistent_replay_in_list_order(zb):
    # GEMMs of two or more waves of tiles (M=2048, h=2048, f=8192: H/A, dH,
    # dW1 and dW2 have 256 tiles of 256 x 256 for 76 CTA pairs) make the plan
    # give priority to list order, as for the large one-stage steps, instead
    # of the longest chain; the replay is still the serial replay bit for bit
    P, m, M, h, f = 1, 6, 2048, 2048, 8192
    blk = zb.make_block(M, h, f)
    ops = _ops(zb, "ZBH2", P, m, 1)
    info, _ = zb.zb_persistent_plan(zb.make_pipeline(P, m, blk), ops, pairs=76)
    assert info.by_chain == 0 and info.gemms == 6 * m
    wts, X0, dY = _setup(P, m, M, h, f, seed=91)
    ref = _replay(zb, zb.make_pipeline(P, m, blk), wts, X0, dY, ops, M, h, f)
    got = _replay(zb, zb.make_pipeline(P, m, blk, executor="persistent"), wts, X0, dY, ops, M, h, f)
    _same_bits(ref, got)


@pytest.mark.parametrize("act", ["tanh", "erf"])
def test_persistent_replay_activation_forms(zb, act):
    # the runtime-selected GeLU / GeLU' epilogues, both activation forms
    P, m, M, h, f = 2, 4, 520, 264, 1048
    blk = zb.make_block(M, h, f, act=zb.ZB_ACT_GELU_TANH if act == "tanh" else zb.ZB_ACT_GELU_ERF)
    wts, X0, dY = _setup(P, m, M, h, f, seed=17)
    ops = zb.zb_make_schedule("ZBH2", P, m)
    ref = _replay(zb, zb.make_pipeline(P, m, blk), wts, X0, dY, ops, M, h, f)
    got = _replay(zb, zb.make_pipeline(P, m, blk, executor="persistent"), wts, X0, dY, ops, M, h, f)
    _same_bits(ref, got)


def test_persistent_replay_single_linear_block(zb):
    # the single-linear block (no activation): plain-store and fp32 GEMMs only
    P, m, M, h = 2, 4, 520, 264
    blk = zb.make_block(M, h, h, act=zb.ZB_ACT_NONE)
    wts, X0, dY = _setup(P, m, M, h, h, seed=29)
    ops = zb.zb_make_schedule("ZBH1", P, m)
    ref = _replay(zb, zb.make_pipeline(P, m, blk), wts, X0, dY, ops, M, h, h)
    got = _replay(zb, zb.make_pipeline(P, m, blk, executor="persistent"), wts, X0, dY, ops, M, h, h)
    for p_, q_ in zip(ref[0], got[0]):
        assert torch.equal(_bits(p_["dW1"]), _bits(q_["dW1"]))
    for p_, q_ in zip(ref[1] + ref[2], got[1] + got[2]):
        assert torch.equal(_bits(p_), _bits(q_))


def test_persistent_replay_without_workspace_argument(zb):
    # the allocation-free entry point (library-owned static arena) with the
    # persistent executor: its tables fit the static arena too
    P, m, M, h, f = 2, 4, 256, 256, 1024
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(P, m, M, h, f, seed=23)
    ops = zb.zb_make_schedule("ZBH1", P, m)
    ref = _replay(zb, zb.make_pipeline(P, m, blk), wts, X0, dY, ops, M, h, f)
    pl = zb.make_pipeline(P, m, blk, executor="persistent")
    need, _ = zb.zb_schedule_workspace_size(pl, ops)
    assert need <= zb.ZB_STATIC_ARENA_BYTES
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    st = zb.zb_run_stats()
    zb.zb_run_stage_schedule_static(pl, stages, X0, dY, dX0, Yl, ops, st)
    sync(zb)
    assert 2 <= st.n_gemm_launches <= 64
    _same_bits(ref, (stages, dX0, Yl))


def test_persistent_replay_accumulates_into_existing_gradients(zb):
    P, m, M, h, f = 2, 4, 512, 256, 1024
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(P, m, M, h, f, seed=11)
    ops = zb.zb_make_schedule("ZBH2", P, m)
    g = torch.Generator(device="cpu").manual_seed(5)
    init = [(torch.randn(h, f, generator=g).cuda(), torch.randn(f, h, generator=g).cuda()) for _ in range(P)]
    ref = _replay(zb, zb.make_pipeline(P, m, blk, zero_grads=False), wts, X0, dY, ops, M, h, f, init=init)
    got = _replay(zb, zb.make_pipeline(P, m, blk, zero_grads=False, executor="persistent"), wts, X0, dY, ops,
                  M, h, f, init=init)
    _same_bits(ref, got)


def test_persistent_replay_against_the_oracle_chain(zb):
    # the rounding-emulating fp64 chain (bf16 at the five storage points)
    P, m, M, h, f = 3, 3, 256, 256, 1024
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(P, m, M, h, f, seed=3)
    ops = zb.zb_make_schedule("ZBH1", P, m)
    stages, dX0, Yl = _replay(zb, zb.make_pipeline(P, m, blk, executor="persistent"), wts, X0, dY, ops, M, h, f)
    st64 = [{"W1": f64(w["W1"]), "W2": f64(w["W2"])} for w in wts]
    emul = ob.run_pipeline(st64, [f64(x) for x in X0], [f64(g) for g in dY], ops, round_fn=ob.bf16_round)
    for s in range(P):
        assert ob.rel_fro(f64(stages[s]["dW1"]), emul["dW1"][s]) < TOL_BF16
        assert ob.rel_fro(f64(stages[s]["dW2"]), emul["dW2"][s]) < TOL_BF16
    for j in range(m):
        assert ob.rel_fro(f64(Yl[j]), emul["Y_last"][j]) < TOL_BF16
        assert ob.rel_fro(f64(dX0[j]), emul["dX0"][j]) < TOL_BF16


def test_persistent_replay_captured_in_a_cuda_graph(zb):
    P, m, M, h, f = 4, 8, 512, 256, 1024
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(P, m, M, h, f, seed=61)
    ops = zb.zb_make_schedule("ZBH1", P, m)
    ref = _replay(zb, zb.make_pipeline(P, m, blk), wts, X0, dY, ops, M, h, f)
    pl = zb.make_pipeline(P, m, blk, executor="persistent")
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    ops_c = zb.ops_array(ops)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            zb.zb_run_stage_schedule(pl, stages, X0, dY, dX0, Yl, ops_c, ws, ws_bytes, None, side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        for s in stages:
            s["dW1"].fill_(float("nan"))
            s["dW2"].fill_(float("nan"))
        ws.fill_(255)  # the tables are rewritten by the graph itself
        graph.replay()
        sync(zb)
        _same_bits(ref, (stages, dX0, Yl))


def test_persistent_replay_errors(zb):
    P, m, M, h, f = 2, 2, 256, 256, 1024
    ops = zb.zb_make_schedule("ZBH1", P, m)
    wts, X0, dY = _setup(P, m, M, h, f, seed=1)
    # bias: the W pass's column sums are not part of the kernel
    blk_b = zb.make_block(M, h, f, has_bias=True)
    pl = zb.make_pipeline(P, m, blk_b, executor="persistent")
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stages = [dict(w, b1=torch.zeros(f, dtype=torch.bfloat16, device="cuda"),
                   b2=torch.zeros(h, dtype=torch.bfloat16, device="cuda"), dW1=empty_f32(h, f),
                   dW2=empty_f32(f, h), db1=empty_f32(f), db2=empty_f32(h)) for w in wts]
    with pytest.raises(zb.ZBError) as e:
        zb.zb_run_stage_schedule(pl, stages, X0, dY, None, None, ops, ws, ws_bytes)
    assert e.value.status == zb.ZB_ERR_UNSUPPORTED
    # the workspace must hold the tables as well as the arena
    blk = zb.make_block(M, h, f)
    pl_s = zb.make_pipeline(P, m, blk)
    pl_p = zb.make_pipeline(P, m, blk, executor="persistent")
    arena, _ = zb.zb_schedule_workspace_size(pl_s, ops)
    need, _ = zb.zb_schedule_workspace_size(pl_p, ops)
    assert need > arena
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    with pytest.raises(zb.ZBError) as e:
        zb.zb_run_stage_schedule(pl_p, stages, X0, dY, None, None, ops, ws, arena)
    assert e.value.status == zb.ZB_ERR_WORKSPACE
    # an unknown executor
    pl_x = zb.make_pipeline(P, m, blk, executor=7)
    with pytest.raises(zb.ZBError) as e:
        zb.zb_run_stage_schedule(pl_x, stages, X0, dY, None, None, ops, ws, need)
    assert e.value.status == zb.ZB_ERR_INVALID_ARG
    sync(zb)


def test_persistent_replay_timing_fields(zb):
    P, m, M, h, f = 2, 4, 512, 256, 1024
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _setup(P, m, M, h, f, seed=2)
    ops = zb.zb_make_schedule("ZBH1", P, m)
    st = zb.zb_run_stats()
    _replay(zb, zb.make_pipeline(P, m, blk, timing=True, executor="persistent"), wts, X0, dY, ops, M, h, f,
            stats=st)
    assert 2 <= st.n_gemm_launches <= 64 and st.total_ms > 0 and st.gemm_ms == st.total_ms
    assert st.workspace_bytes > 0 and st.n_ops == len(ops)
