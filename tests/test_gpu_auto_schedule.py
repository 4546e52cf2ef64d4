"""GPU replays of the heuristic orderings ZB-1p and ZB-2p.

"Zero Bubble Pipeline Parallelism" (summary of arXiv 2401.10241), §3 "The
Heuristic Scheduling Algorithm": the scheduler places F, B and W on a
simulated timeline under a memory limit (p M_B for ZB-1p, 2p M_B for ZB-2p)
and inserts W where memory forces it or a gap fits it.  Its lists differ
from the handcrafted ones: several B in a row with their W pending,
memory-triggered W right before an F, warm-ups of more than P forwards.

The executor must accept every such list, and because each stage's W still
run in ascending microbatch order, the replay must reproduce the 1F1B replay
of the same inputs bit for bit (split backward leaves the update unchanged:
"Zero-Bubble Pipeline Parallelism, Proven", "Split backward without changing
the update").  Every pass is also compared with the fp64 oracle from the
exact bf16 tensors it consumed (relative Frobenius 5e-3), and the arena's
peak with an independent count of the bytes the executor must hold.

Memory unit: for this block a microbatch's forward state M_B (H and A) and
its weight-gradient state M_W (A and dH) are both two [M, f] buffers, so the
heuristic runs with M_W / M_B = 1.
"""

import numpy as np
import pytest
import torch

from oracle import block as ob
from oracle import schedules as S
from tests.gpu_util import f64, have_gpu
from tests.test_gpu_parity import _bits, _hand_chain, _pipeline_setup, _run_schedule

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3
MW_RATIO = 1.0

# pass times: equal; Table 9's 1.5B row (ms, with T_comm); W slower than F/B
TIMES = {
    "equal": (1.0, 1.0, 1.0, 0.0),
    "table9_1.5B": (18.522, 18.086, 9.337, 0.601),
    "slow_w": (1.0, 1.0, 1.2, 0.0),
}


@pytest.fixture(scope="module")
def zb():
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def _arena_peak_model(ops, P, M, h, f):
    """Bytes of saved activations the executor holds, counted op by op.

    F(s,j) saves H and A ([M, f] each) and hands Y to stage s+1 as its X
    ([M, h], not for the last stage, whose Y is the caller's); B(s,j) saves
    dH and hands dX to stage s-1 as its dY (not for stage 0), then frees H;
    W(s,j) frees X (s > 0), A, dH and dY (s < P-1).  A running op holds its
    new outputs and its inputs at once, so the peak is read after the takes
    and before the releases of each op.
    """
    row, ffn = M * h * 2, M * f * 2
    live = peak = 0
    for k, s, _ in ops:
        if k == "F":
            live += 2 * ffn + (row if s < P - 1 else 0)
            peak = max(peak, live)
        elif k in ("B", "BW"):
            live += ffn + (row if s > 0 else 0)
            peak = max(peak, live)
            live -= ffn
        if k in ("W", "BW"):
            live -= (row if s > 0 else 0) + 2 * ffn + (row if s < P - 1 else 0)
    assert live == 0
    return peak


@pytest.mark.parametrize("times", list(TIMES))
@pytest.mark.parametrize("limit_x", [1, 2])
def test_heuristic_lists_replay_bit_exact_and_match_oracle(zb, limit_x, times):
    # The P=4, h=1024, ffn=4096 pipeline at 512 tokens per microbatch, m=8.
    P, m, M, h, f = 4, 8, 512, 1024, 4096
    tf, tb, tw, tc = TIMES[times]
    limit = limit_x * P
    res, ops, hyper = zb.zb_auto_schedule(P, m, tf, tb, tw, tc, limit, MW_RATIO)
    # the library's list is the oracle's, op for op, and legal
    ev, ref_ops, ref_hyper = S.auto_schedule_search(P, m, S.Times(tf, tb, tw, tc), limit, MW_RATIO)
    assert ops == ref_ops and hyper == ref_hyper
    assert S.validate_ops(ops, P, m)
    assert max(S.mem_peaks(ev, P, MW_RATIO)) <= limit + 1e-9
    handcrafted = zb.zb_make_schedule("ZBH1" if limit_x == 1 else "ZBH2", P, m)
    assert ops != handcrafted  # a list of its own, not a copy of ZB-H1 / ZB-H2

    blk = zb.make_block(M, h, f)
    wts, X0, dY = _pipeline_setup(zb, P, m, M, h, f, seed=11 + limit_x)
    auto = _run_schedule(zb, blk, P, m, wts, X0, dY, ops)
    base = _run_schedule(zb, blk, P, m, wts, X0, dY, zb.zb_make_schedule("1F1B", P, m))
    for s in range(P):
        for key in ("dW1", "dW2"):
            assert torch.equal(_bits(auto[0][s][key]), _bits(base[0][s][key]))
    for j in range(m):
        assert torch.equal(_bits(auto[1][j]), _bits(base[1][j]))
        assert torch.equal(_bits(auto[2][j]), _bits(base[2][j]))

    # the arena holds exactly what the lifetime rules say, within the limit
    peak = auto[4]
    assert peak == _arena_peak_model(ops, P, M, h, f)
    row, ffn = M * h * 2, M * f * 2
    # per stage at most `limit` microbatches of (H, A) or (A, dH) plus their
    # two row buffers, and one running B's dH and dX on top
    assert peak <= P * (limit * (2 * ffn + 2 * row)) + ffn + row

    # single passes in plain order reproduce the replay; every pass of two
    # microbatches per stage against the oracle from its own inputs
    rec, Xs, dYs, dWs = _hand_chain(zb, zb.make_block(M, h, f, split_k=False), P, m, wts, X0, dY)
    for s in range(P):
        assert torch.equal(_bits(auto[0][s]["dW1"]), _bits(dWs[s][0]))
        assert torch.equal(_bits(auto[0][s]["dW2"]), _bits(dWs[s][1]))
    for j in range(m):
        assert torch.equal(_bits(auto[1][j]), _bits(rec[("B", 0, j)][1]))
        assert torch.equal(_bits(auto[2][j]), _bits(rec[("F", P - 1, j)][2]))
    for j in (0, m - 1):
        for s in range(P):
            W1, W2 = f64(wts[s]["W1"]), f64(wts[s]["W2"])
            H, A, Y = rec[("F", s, j)]
            Hr, Ar, _ = ob.forward(f64(Xs[(s, j)]), W1, W2)
            assert ob.rel_fro(f64(H), Hr) < TOL_BF16
            assert ob.rel_fro(f64(A), Ar) < TOL_BF16
            assert ob.rel_fro(f64(Y), f64(A) @ W2) < TOL_BF16
            dH, dX = rec[("B", s, j)]
            _, dHr, _ = ob.backward_input(f64(dYs[(s, j)]), W1, W2, f64(H))
            assert ob.rel_fro(f64(dH), dHr) < TOL_BF16
            assert ob.rel_fro(f64(dX), f64(dH) @ W1.T) < TOL_BF16
    for s in range(P):
        r1 = np.zeros((h, f))
        r2 = np.zeros((f, h))
        for j in range(m):
            _, A, _ = rec[("F", s, j)]
            dH, _ = rec[("B", s, j)]
            a, b, _, _ = ob.backward_weight(f64(Xs[(s, j)]), f64(A), f64(dH), f64(dYs[(s, j)]))
            r1 += a
            r2 += b
        assert ob.rel_fro(f64(auto[0][s]["dW1"]), r1) < TOL_BF16
        assert ob.rel_fro(f64(auto[0][s]["dW2"]), r2) < TOL_BF16


@pytest.mark.parametrize("limit_x", [1, 2])
def test_heuristic_list_stage_parallel_and_budget(zb, limit_x):
    # The same list on stage lanes with W lanes (8 streams) gives the serial
    # bits, and a byte budget just below the replay's peak is refused.
    P, m, M, h, f = 4, 8, 512, 1024, 4096
    _, ops, _ = zb.zb_auto_schedule(P, m, *TIMES["table9_1.5B"], limit_x * P, MW_RATIO)
    blk = zb.make_block(M, h, f)
    wts, X0, dY = _pipeline_setup(zb, P, m, M, h, f, seed=21)
    serial = _run_schedule(zb, blk, P, m, wts, X0, dY, ops)
    pl = zb.make_pipeline(P, m, blk, streams=2 * P)
    ws_bytes, peak = zb.zb_schedule_workspace_size(pl, ops)
    assert peak == serial[4]
    from tests.gpu_util import empty_bf16, empty_f32, sync
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stages = [dict(w, dW1=empty_f32(h, f), dW2=empty_f32(f, h)) for w in wts]
    dX0 = [empty_bf16(M, h) for _ in range(m)]
    Yl = [empty_bf16(M, h) for _ in range(m)]
    zb.zb_run_stage_schedule(pl, stages, X0, dY, dX0, Yl, ops, ws, ws_bytes)
    sync(zb)
    for s in range(P):
        assert torch.equal(_bits(stages[s]["dW1"]), _bits(serial[0][s]["dW1"]))
        assert torch.equal(_bits(stages[s]["dW2"]), _bits(serial[0][s]["dW2"]))
    for j in range(m):
        assert torch.equal(_bits(dX0[j]), _bits(serial[1][j]))
        assert torch.equal(_bits(Yl[j]), _bits(serial[2][j]))
    tight = zb.make_pipeline(P, m, blk, mem_limit_bytes=peak - 1)
    with pytest.raises(zb.ZBError) as e:
        zb.zb_schedule_workspace_size(tight, ops)
    assert e.value.status == zb.ZB_ERR_BUDGET
