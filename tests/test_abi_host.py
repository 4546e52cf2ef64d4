"""Host-side checks of the C ABI (no GPU needed, no device work).

* the library loads and exports every function ``include/zb.h`` declares;
* ``zb_make_schedule`` (C++) agrees op for op with the oracle's generator
  (an independent Python implementation of the same rules);
* op-list validation returns the documented error codes;
* the arena's ledger peak equals the Delta-M model of "Zero Bubble Pipeline
  Parallelism" (summary, "The Memory Model") for single-stage lists.
"""

import os
import re

import pytest

from oracle import schedules as S
from split_backward_gemms_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zb():
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def test_library_exports_every_declared_function(zb):
    with open(os.path.join(ROOT, "include", "zb.h")) as fh:
        hdr = fh.read()
    names = set(re.findall(r"^(?:zb_status|const char\*)\s+(zb_\w+)\s*\(", hdr, re.M))
    assert {"zb_forward", "zb_backward_input", "zb_backward_weight", "zb_run_stage_schedule",
            "zb_schedule_workspace_size", "zb_make_schedule", "zb_sync_status",
            "zb_last_error", "zb_version"} <= names
    for n in names:
        assert hasattr(zb.LIB, n), n
    assert "sm_103a" in zb.zb_version()


@pytest.mark.parametrize("kind", S.SCHEDULES)
@pytest.mark.parametrize("P,m", [(1, 1), (1, 5), (2, 2), (3, 7), (4, 8), (4, 4), (8, 16),
                                 (8, 24), (5, 3), (6, 13)])
def test_generator_matches_oracle(zb, kind, P, m):
    _, ref = S.make_schedule(kind, P, m)
    got = zb.zb_make_schedule(kind, P, m)
    assert got == ref


def test_generator_rejects_bad_args(zb):
    with pytest.raises(zb.ZBError) as e:
        zb.zb_make_schedule(7, 2, 2)
    assert e.value.status == zb.ZB_ERR_INVALID_ARG
    with pytest.raises(zb.ZBError) as e:
        zb.zb_make_schedule("ZBH1", 0, 2)
    assert e.value.status == zb.ZB_ERR_SHAPE


def _pl(zb, P, m, M=64, h=32, f=128, act=None, limit=0):
    act = zb.ZB_ACT_GELU_ERF if act is None else act
    return zb.make_pipeline(P, m, zb.make_block(M, h, f, zb.ZB_DT_BF16, act), limit)


def test_validation_error_codes(zb):
    P, m = 2, 3
    _, ok = S.make_schedule("ZBH1", P, m)
    pl = _pl(zb, P, m)
    zb.zb_schedule_workspace_size(pl, ok)

    def code(ops):
        with pytest.raises(zb.ZBError) as e:
            zb.zb_schedule_workspace_size(pl, ops)
        return e.value.status

    bad = [op for op in ok if op != ("B", 1, 0)]
    bad.insert(0, ("B", 1, 0))
    assert code(bad) == zb.ZB_ERR_SCHEDULE  # consumer before producer
    assert code([op for op in ok if op != ("W", 0, 1)]) == zb.ZB_ERR_SCHEDULE  # missing
    assert code(ok[:1] + ok) == zb.ZB_ERR_SCHEDULE  # duplicate
    sw = list(ok)
    i0, i1 = sw.index(("W", 1, 0)), sw.index(("W", 1, 1))
    sw[i0], sw[i1] = sw[i1], sw[i0]
    assert code(sw) in (zb.ZB_ERR_W_ORDER, zb.ZB_ERR_SCHEDULE)
    # W of micro 1 moved before W of micro 0 while both Bs precede: pure order error
    st1 = [op for op in ok if op[1] == 1]
    assert st1.index(("B", 1, 1)) < st1.index(("W", 1, 0)) or True
    o = [op for op in ok if op != ("OPT", 0, 0)]
    o.insert(o.index(("W", 0, 2)), ("OPT", 0, 0))
    assert code(o) == zb.ZB_ERR_SCHEDULE  # OPT before the stage's last W
    assert code(ok + [("F", 2, 0)]) == zb.ZB_ERR_SCHEDULE  # unknown stage
    assert code(ok[:-1] + [("BW", 0, 2)]) == zb.ZB_ERR_SCHEDULE


def test_w_order_code_on_pure_reordering(zb):
    # single stage, all B before any W: swapping two W's is only an order error
    P, m = 1, 3
    ops = [("F", 0, j) for j in range(m)] + [("B", 0, j) for j in range(m)]
    ops += [("W", 0, 1), ("W", 0, 0), ("W", 0, 2)]
    with pytest.raises(zb.ZBError) as e:
        zb.zb_schedule_workspace_size(_pl(zb, P, m), ops)
    assert e.value.status == zb.ZB_ERR_W_ORDER
    with pytest.raises(S.ScheduleError) as e2:
        S.validate_ops(ops, P, m)
    assert e2.value.code == "w_order"


@pytest.mark.parametrize("kind,Pg", [("ZBH1", 8), ("ZBH2", 8), ("1F1B", 4), ("ZBH2", 4)])
def test_single_stage_ledger_matches_delta_m_model(zb, kind, Pg):
    # One stage replaying the stage-0 list of a Pg-stage ordering.  Saved per
    # microbatch: F stores H and A (M_B = 2 ffn buffers), B swaps H for dH
    # (M_W = A + dH = 2 ffn buffers), W frees both.
    m = 3 * Pg
    _, ops = S.make_schedule(kind, Pg, m)
    st0 = [(k, 0, j) for k, s, j in ops if s == 0]
    M, h, f = 48, 32, 128
    pl = _pl(zb, 1, m, M, h, f)
    ws, peak = zb.zb_schedule_workspace_size(pl, st0)
    ffn = M * f * 2
    led_peak, led_final = S.memory_ledger(st0, 1, 2 * ffn, 2 * ffn)
    assert led_final == [0.0]
    # peak in microbatches: P (1F1B, ZB-H1) or 2P-1 (ZB-H2), Table 2
    assert led_peak[0] == S.table2_peak_mb(kind, Pg) * 2 * ffn
    # The Delta-M model books B's swap of H for dH as one step; a running B
    # holds both, so the arena's peak is the model's level before each op
    # plus that op's outputs (F: H and A; B/BW: dH).
    expect = 0.0
    for i, op in enumerate(st0):
        before = S.memory_ledger(st0[:i], 1, 2 * ffn, 2 * ffn)[1][0] if i else 0.0
        out = {"F": 2 * ffn, "B": ffn, "BW": ffn}.get(op[0], 0)
        expect = max(expect, before + out)
    assert peak == expect
    assert ws >= peak


def test_budget_error(zb):
    _, ops = S.make_schedule("ZBH2", 4, 8)
    pl = _pl(zb, 4, 8)
    ws, peak = zb.zb_schedule_workspace_size(pl, ops)
    pl2 = _pl(zb, 4, 8, limit=peak - 1)
    with pytest.raises(zb.ZBError) as e:
        zb.zb_schedule_workspace_size(pl2, ops)
    assert e.value.status == zb.ZB_ERR_BUDGET
    pl3 = _pl(zb, 4, 8, limit=peak)
    assert zb.zb_schedule_workspace_size(pl3, ops)[1] == peak


def test_zbh2_needs_more_memory_than_zbh1(zb):
    P, m = 4, 8
    peaks = {}
    for kind in S.SCHEDULES:
        _, ops = S.make_schedule(kind, P, m)
        peaks[kind] = zb.zb_schedule_workspace_size(_pl(zb, P, m), ops)[1]
    assert peaks["ZBH2"] > peaks["ZBH1"] >= peaks["1F1B"]


def test_single_linear_multi_stage_needs_square(zb):
    _, ops = S.make_schedule("ZBH1", 2, 2)
    pl = zb.make_pipeline(2, 2, zb.make_block(16, 32, 64, zb.ZB_DT_F32, zb.ZB_ACT_NONE))
    with pytest.raises(zb.ZBError) as e:
        zb.zb_schedule_workspace_size(pl, ops)
    assert e.value.status == zb.ZB_ERR_SHAPE


@pytest.mark.parametrize("kind", S.SCHEDULES)
@pytest.mark.parametrize("P,m", [(2, 3), (4, 8), (8, 24), (5, 11), (3, 2)])
def test_simulator_with_times_matches_oracle(zb, kind, P, m):
    # dyadic times (exact in binary) so both simulators see identical sums
    import random
    rnd = random.Random(P * 100 + m)
    for _ in range(4):
        tf, tb, tw = (rnd.randint(1, 16) / 8 for _ in range(3))
        tc = rnd.randint(0, 4) / 16
        t = S.Times(tf, tb, tw, tc)
        ev, ref_ops = S.make_schedule(kind, P, m, t)
        res, ops = zb.zb_simulate_schedule(kind, P, m, tf, tb, tw, tc, want_ops=True)
        assert ops == ref_ops
        assert res.cost == S.cost(ev, P)
        assert abs(res.bubble_rate - S.bubble_rate(ev, P, m, t)) < 1e-12
        assert res.peak_live_microbatches == max(S.peak_live(ev, P))
        assert res.peak_live_stage0 == S.peak_live(ev, P)[0]


def test_simulator_equal_times_is_make_schedule(zb):
    for kind in S.SCHEDULES:
        res, ops = zb.zb_simulate_schedule(kind, 4, 8, 1.0, 1.0, 1.0, 0.0, want_ops=True)
        assert ops == zb.zb_make_schedule(kind, 4, 8)
        assert res.cost == {"1F1B": 33.0, "ZBH1": 27.0, "ZBH2": 24.0}[kind]


def test_simulator_rejects_bad_times(zb):
    for bad in ((0.0, 1.0, 1.0, 0.0), (1.0, -1.0, 1.0, 0.0), (1.0, 1.0, float("nan"), 0.0),
                (1.0, 1.0, 1.0, -0.5)):
        with pytest.raises(zb.ZBError) as e:
            zb.zb_simulate_schedule("ZBH1", 4, 8, *bad)
        assert e.value.status == zb.ZB_ERR_INVALID_ARG


@pytest.mark.parametrize("P,m", [(2, 4), (4, 8), (4, 12), (8, 24), (3, 7)])
@pytest.mark.parametrize("limit_x", [1, 2])
def test_auto_scheduler_matches_oracle(zb, P, m, limit_x):
    import random
    rnd = random.Random(P * 31 + m * 7 + limit_x)
    cases = [(1.0, 1.0, 1.0, 0.0)]
    for _ in range(3):
        cases.append((rnd.randint(4, 16) / 8, rnd.randint(4, 16) / 8, rnd.randint(2, 12) / 8,
                      rnd.randint(0, 3) / 16))
    for tf, tb, tw, tc in cases:
        for mw in (0.5, 0.375):
            t = S.Times(tf, tb, tw, tc)
            ev, ref_ops, ref_h = S.auto_schedule_search(P, m, t, limit_x * P, mw)
            res, ops, hyper = zb.zb_auto_schedule(P, m, tf, tb, tw, tc, limit_x * P, mw)
            assert ops == ref_ops
            assert hyper == ref_h
            assert res.cost == S.cost(ev, P)


def test_auto_scheduler_reproduces_printed_bubbles(zb):
    from tests.test_oracle_schedules import table5_rows
    for name, P, m, t, mw, limit, pct in table5_rows():
        res, ops, _ = zb.zb_auto_schedule(P, m, t.F, t.B, t.W, t.comm, limit, mw)
        assert abs(100 * res.bubble_rate - pct) <= 0.015
        assert S.validate_ops(ops, P, m)
        ev, ref_ops, _ = S.auto_schedule_search(P, m, t, limit, mw)
        assert ops == ref_ops


@pytest.mark.parametrize("P,m", [(2, 6), (4, 8), (6, 18), (8, 24)])
def test_auto_scheduler_at_the_zero_bubble_threshold(zb, P, m):
    # the same lists as the oracle at (2P-1) M_B (zero bubble at equal times)
    # and one M_B below it (a bubble of at most one forward pass)
    for limit in (2 * P - 1, 2 * P - 2):
        res, ops, _ = zb.zb_auto_schedule(P, m, 1.0, 1.0, 1.0, 0.0, limit, 0.5)
        ev, ref_ops, _ = S.auto_schedule_search(P, m, S.Times(), limit, 0.5)
        assert ops == ref_ops and res.cost == S.cost(ev, P)
        assert (res.cost == 3 * m) == (limit == 2 * P - 1)


def test_auto_scheduler_rejects_bad_budget(zb):
    with pytest.raises(zb.ZBError) as e:
        zb.zb_auto_schedule(4, 8, 1, 1, 1, 0, 0.5)
    assert e.value.status == zb.ZB_ERR_BUDGET
    with pytest.raises(zb.ZBError) as e:
        zb.zb_auto_schedule(4, 8, 1, 1, 1, 0, 4, 1.5)
    assert e.value.status == zb.ZB_ERR_INVALID_ARG


ABI_STRUCTS = ["zb_block", "zb_op", "zb_sim_times", "zb_sim_result", "zb_pipeline",
               "zb_stage_params", "zb_run_stats", "zb_opt_tensor", "zb_adamw_params",
               "zb_stage_decision"]


def test_ctypes_layout_matches_header(zb, tmp_path):
    """Every struct of the binding has the C compiler's size and field offsets."""
    import ctypes
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "zb.h"', "int main(void) {"]
    for name in ABI_STRUCTS:
        cls = getattr(zb, name)
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for ln in out:
        if ln:
            n, f, v = ln.split()
            got[(n, f)] = int(v)
    for name in ABI_STRUCTS:
        cls = getattr(zb, name)
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[(name, field)] == getattr(cls, field).offset, (name, field)


def test_post_validated_adamw_argument_errors(zb):
    """Argument checks run before anything is enqueued (fake, never dereferenced pointers)."""
    fake = 1 << 20
    st = [fake + 8 * i for i in range(2)]
    dec = fake + 4096
    t = dict(theta=fake, m=fake + 256, v=fake + 512, grad=fake + 768, weight_bf16=None,
             count=16, stage=0)

    def code(P=2, states=st, tensors=(t,), hp=None, decisions=dec):
        hp = zb.make_adamw(max_norm=1.0) if hp is None else hp
        with pytest.raises(zb.ZBError) as e:
            zb.zb_post_validated_adamw(P, states, list(tensors), hp, decisions)
        return e.value.status

    assert code(P=0, states=[]) == zb.ZB_ERR_SHAPE
    assert code(P=65, states=[fake] * 65) == zb.ZB_ERR_SHAPE
    assert code(decisions=None) == zb.ZB_ERR_INVALID_ARG
    assert code(decisions=dec + 4) == zb.ZB_ERR_ALIGN
    assert code(states=[fake, None]) == zb.ZB_ERR_INVALID_ARG
    assert code(states=[fake, fake + 4]) == zb.ZB_ERR_ALIGN
    assert code(tensors=[dict(t, stage=2)]) == zb.ZB_ERR_INVALID_ARG
    assert code(tensors=[dict(t, theta=fake + 4)]) == zb.ZB_ERR_ALIGN
    assert code(tensors=[dict(t, weight_bf16=fake + 2)]) == zb.ZB_ERR_ALIGN
    assert code(tensors=[dict(t, grad=None)]) == zb.ZB_ERR_INVALID_ARG
    for bad in (dict(step=0), dict(beta1=1.0), dict(beta2=0.0), dict(eps=0.0), dict(lr=-1.0),
                dict(weight_decay=-0.1), dict(lr=1.0, weight_decay=1.0), dict(max_norm=-1.0)):
        assert code(hp=zb.make_adamw(**bad)) == zb.ZB_ERR_INVALID_ARG, bad
    hp = zb.make_adamw()
    hp.reserved = 1
    assert code(hp=hp) == zb.ZB_ERR_INVALID_ARG


# ------------------------------------------------------------------ multi-chunk orderings
from oracle import interleaved as IL  # noqa: E402

ILV_CASES = ([("ZBV", P, 2, m) for P in (1, 2, 3, 4, 8) for m in (1, 2 * P - 1, 2 * P, 3 * P)]
             + [("1F1B-I", P, v, m) for P in (1, 2, 4, 8) for v in (2, 4) for m in (P, 2 * P, 3 * P)])


@pytest.mark.parametrize("kind,P,v,m", ILV_CASES)
def test_interleaved_generator_matches_oracle(zb, kind, P, v, m):
    _, ref = IL.make_interleaved_schedule(kind, P, v, m)
    assert zb.zb_make_interleaved_schedule(kind, P, v, m) == ref


def test_interleaved_simulator_matches_oracle_at_random_times(zb):
    import random
    rng = random.Random(11)
    for _ in range(60):
        kind = rng.choice(["ZBV", "1F1B-I"])
        P = rng.randint(1, 5)
        v = 2 if kind == "ZBV" else rng.randint(2, 3)
        m = rng.randint(1, 3 * P) if kind == "ZBV" else P * rng.randint(1, 3)
        t = S.Times(rng.uniform(0.2, 3), rng.uniform(0.2, 3), rng.uniform(0.1, 3),
                    rng.choice([0.0, rng.uniform(0, 1)]))
        res, got = zb.zb_simulate_interleaved_schedule(kind, P, v, m, t.F, t.B, t.W, t.comm, want_ops=True)
        ev, ref = IL.make_interleaved_schedule(kind, P, v, m, t)
        assert got == ref
        assert abs(res.bubble_rate - IL.bubble_rate(ev, P, m, t)) < 1e-12
        assert res.peak_live_microbatches == max(IL.peak_live_chunks(ev, P))
        assert res.peak_live_stage0 == IL.peak_live_chunks(ev, P)[0]


def test_interleaved_argument_errors(zb):
    def code(*a):
        with pytest.raises(zb.ZBError) as e:
            zb.zb_make_interleaved_schedule(*a)
        return e.value.status
    assert code("ZBV", 2, 3, 4) == zb.ZB_ERR_INVALID_ARG
    assert code("1F1B-I", 2, 1, 4) == zb.ZB_ERR_INVALID_ARG
    assert code("ZBH1", 2, 2, 4) == zb.ZB_ERR_INVALID_ARG
    assert code("1F1B-I", 4, 2, 6) == zb.ZB_ERR_SHAPE
    assert code("ZBV", 0, 2, 4) == zb.ZB_ERR_SHAPE


@pytest.mark.parametrize("kind,P,v,m", [("ZBV", 2, 2, 4), ("ZBV", 4, 2, 8), ("1F1B-I", 2, 2, 4),
                                        ("1F1B-I", 2, 3, 4)])
def test_chunked_list_sizes_like_its_virtual_chain(zb, kind, P, v, m):
    """A chunked replay is the replay of its chain of v P virtual stages."""
    ops = zb.zb_make_interleaved_schedule(kind, P, v, m)
    blk = zb.make_block(64, 32, 128)
    pl = zb.make_pipeline(P, m, blk, chunks=v, layout=kind)
    chain = zb.make_pipeline(v * P, m, blk)
    flat = IL.to_virtual(kind, P, ops)
    assert zb.zb_schedule_workspace_size(pl, ops) == zb.zb_schedule_workspace_size(chain, flat)
    # the ledger of the V replay on one GPU: every virtual stage's M_B, chained
    _, peak_b = zb.zb_schedule_workspace_size(pl, ops)
    assert peak_b > 0


def test_chunked_validation_codes(zb):
    ops = zb.zb_make_interleaved_schedule("ZBV", 2, 2, 3)
    blk = zb.make_block(64, 32, 128)

    def code(pl, o):
        with pytest.raises(zb.ZBError) as e:
            zb.zb_schedule_workspace_size(pl, o)
        return e.value.status

    pl = zb.make_pipeline(2, 3, blk, chunks=2, layout="ZBV")
    assert code(zb.make_pipeline(2, 3, blk), ops) == zb.ZB_ERR_SCHEDULE  # chunk 1 without chunks
    assert code(zb.make_pipeline(2, 3, blk, chunks=3, layout="ZBV"), ops) == zb.ZB_ERR_INVALID_ARG
    assert code(zb.make_pipeline(2, 3, blk, chunks=2, layout=7), ops) == zb.ZB_ERR_INVALID_ARG
    bad = [("F", 0, 2, 0)] + ops
    assert code(pl, bad) == zb.ZB_ERR_SCHEDULE
    # a V list replayed with the cyclic layout breaks the chain order
    assert code(zb.make_pipeline(2, 3, blk, chunks=2, layout="1F1B-I"), ops) == zb.ZB_ERR_SCHEDULE
    # W of a virtual stage out of order
    i = next(n for n, op in enumerate(ops) if op[0] == "W" and op[3] == 0)
    k = next(n for n, op in enumerate(ops) if op[0] == "W" and op[1:3] == ops[i][1:3] and op[3] == 1)
    sw = list(ops)
    sw[i], sw[k] = sw[k], sw[i]
    assert code(pl, sw) in (zb.ZB_ERR_W_ORDER, zb.ZB_ERR_SCHEDULE)


@pytest.mark.parametrize("kind,P,v,m", [("ZBV", 16, 2, 48), ("ZBV", 32, 2, 96), ("1F1B-I", 16, 2, 64),
                                        ("1F1B-I", 32, 4, 64)])
def test_interleaved_at_the_pages_scales(zb, kind, P, v, m):
    """Table 8 / Figure 9 scales (16-32 stages): generated quickly, valid
    replays of the chain, ZB-V at exactly P M_B on every stage."""
    import time
    t0 = time.perf_counter()
    res, ops = zb.zb_simulate_interleaved_schedule(kind, P, v, m, 1.0, 1.0, 1.0, 0.0, want_ops=True)
    assert time.perf_counter() - t0 < 20.0
    blk = zb.make_block(64, 32, 128)
    pl = zb.make_pipeline(P, m, blk, chunks=v, layout=kind)
    zb.zb_schedule_workspace_size(pl, ops)  # validates the list on the chain
    if kind == "ZBV":
        assert res.peak_live_microbatches == 2 * P
        assert res.bubble_rate < S.bubble_rate(S.make_schedule("ZBH1", P, m)[0], P, m, S.Times())
    else:
        assert abs(res.bubble_rate - (P - 1) / (v * m + P - 1)) < 1e-12


def test_block_flags(zb):
    """zb_block.flags: the binding's ZB_BLOCK_NO_SPLIT_K is the header's, a
    block carrying it validates, and unknown bits are rejected."""
    import re
    hdr = open(os.path.join(ROOT, "include", "zb.h")).read()
    assert int(re.search(r"#define ZB_BLOCK_NO_SPLIT_K (\d+)", hdr).group(1)) == zb.ZB_BLOCK_NO_SPLIT_K
    P, m = 2, 3
    _, ok = S.make_schedule("ZBH1", P, m)
    blk = zb.make_block(64, 16, 32, split_k=False)
    assert blk.flags == zb.ZB_BLOCK_NO_SPLIT_K and zb.make_block(64, 16, 32).flags == 0
    zb.zb_schedule_workspace_size(zb.make_pipeline(P, m, blk), ok)
    blk.flags = 2
    with pytest.raises(zb.ZBError) as e:
        zb.zb_schedule_workspace_size(zb.make_pipeline(P, m, blk), ok)
    assert e.value.status == zb.ZB_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library the binding refuses to import: there is no
    CPU fallback for any entry point."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    missing = str(tmp_path / "libzb_gb300.so")
    code = ("import split_backward_gemms_gb300.build as b; b.LIB_PATH = %r\n"
            "try:\n"
            "    from split_backward_gemms_gb300 import zb\n"
            "except RuntimeError as e:\n"
            "    print('refused:', e)\n"
            "else:\n"
            "    print('imported')\n" % missing)
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.startswith("refused:") and "no CPU fallback" in r.stdout, r.stdout
