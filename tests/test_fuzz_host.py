"""Property-based tests of the host schedulers, the planner and the oracle.

Random pipeline depths, microbatch counts, pass times and communication
times (dyadic, so both sides add exactly the same floating-point values):
the C++ simulators of the handcrafted and the multi-chunk orderings and the
C++ heuristic scheduler return the oracle's op lists and costs, every list
passes the oracle's validator, and the heuristic respects its memory limit;
the persistent executor's host plan of random lists, for any number of CTA
pairs, keeps every data dependency (and passes its own deadlock check); the
oracle's trace checker accepts every simulated step and rejects it once one
pass starts before a producer has ended; the fp64 block's gradients match
central differences on random tiny shapes.  CPU only (hypothesis; skipped
where it is not installed).
"""

import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import schedules as S  # noqa: E402
from split_backward_gemms_gb300 import build as B  # noqa: E402

B.build()
from split_backward_gemms_gb300 import zb  # noqa: E402

dyadic = st.integers(min_value=1, max_value=24).map(lambda k: k / 8)
comm = st.integers(min_value=0, max_value=8).map(lambda k: k / 16)


@st.composite
def pipelines(draw):
    P = draw(st.integers(min_value=1, max_value=8))
    m = draw(st.integers(min_value=1, max_value=3 * P + 3))
    return P, m


@settings(max_examples=400, deadline=None)
@given(pipelines(), st.sampled_from(S.SCHEDULES), dyadic, dyadic, dyadic, comm)
def test_simulator_matches_oracle(pm, kind, tf, tb, tw, tc):
    P, m = pm
    t = S.Times(tf, tb, tw, tc)
    ev, ref_ops = S.make_schedule(kind, P, m, t)
    res, ops = zb.zb_simulate_schedule(kind, P, m, tf, tb, tw, tc, want_ops=True)
    assert ops == ref_ops
    assert res.cost == S.cost(ev, P)
    assert S.validate_ops(ops, P, m)


@settings(max_examples=300, deadline=None)
@given(pipelines(), st.integers(min_value=0, max_value=8), dyadic, dyadic, dyadic, comm,
       st.sampled_from([0.25, 0.375, 0.5, 0.75, 1.0]))
def test_auto_scheduler_matches_oracle(pm, extra, tf, tb, tw, tc, mw):
    P, m = pm
    limit = P + extra * P / 8  # between the 1F1B budget and twice it
    t = S.Times(tf, tb, tw, tc)
    ev, ref_ops, ref_h = S.auto_schedule_search(P, m, t, limit, mw)
    res, ops, hyper = zb.zb_auto_schedule(P, m, tf, tb, tw, tc, limit, mw)
    assert ops == ref_ops and hyper == ref_h
    assert res.cost == S.cost(ev, P)
    assert S.validate_ops(ops, P, m)
    assert max(S.mem_peaks(ev, P, mw)) <= limit + 1e-9


@settings(max_examples=300, deadline=None)
@given(st.sampled_from(["ZBV", "1F1B-I"]), st.integers(min_value=1, max_value=6),
       st.integers(min_value=2, max_value=3), st.integers(min_value=1, max_value=4),
       dyadic, dyadic, dyadic, comm)
def test_interleaved_simulator_matches_oracle(kind, P, v, k, tf, tb, tw, tc):
    from oracle import interleaved as IL
    if kind == "ZBV":
        v, m = 2, k * P - (k % 2)  # odd and even microbatch counts, from P - 1 up
        m = max(m, 1)
    else:
        m = k * P  # whole groups of P microbatches
    t = S.Times(tf, tb, tw, tc)
    ev, ref_ops = IL.make_interleaved_schedule(kind, P, v, m, t)
    res, ops = zb.zb_simulate_interleaved_schedule(kind, P, v, m, tf, tb, tw, tc, want_ops=True)
    assert ops == ref_ops
    assert abs(res.bubble_rate - IL.bubble_rate(ev, P, m, t)) < 1e-12
    assert IL.validate_interleaved(kind, P, v, m, ops)


@settings(max_examples=60, deadline=None)
@given(st.sampled_from(["1F1B", "ZBH1", "ZBH2", "ZB1P", "ZB2P"]), pipelines(),
       st.sampled_from([(96, 256, 512), (256, 256, 1024), (520, 264, 1048), (2048, 1024, 4096)]),
       st.integers(min_value=1, max_value=76))
def test_persistent_plan_keeps_every_data_dependency(kind, pm, shape, pairs):
    # the persistent executor's host plan on random lists: every data
    # dependency of the split backward implied by its kept edges
    from tests.test_persistent_plan import _gemms, _reach
    P, m = pm
    M, h, f = shape
    if kind in ("ZB1P", "ZB2P"):
        limit = P if kind == "ZB1P" else 2 * P
        _, ops, _ = zb.zb_auto_schedule(P, m, 1.0, 1.0, 1.0, 0.0, limit, 1.0)
    else:
        ops = zb.zb_make_schedule(kind, P, m)
    info, edges = zb.zb_persistent_plan(zb.make_pipeline(P, m, zb.make_block(M, h, f)), ops, pairs=pairs)
    g = _gemms(ops)
    assert info.gemms == len(g) == 6 * P * m and all(p < c for c, p in edges)
    clo = _reach(len(g), edges)
    at = {x: i for i, x in enumerate(g)}
    for (name, s, j), i in at.items():
        need = {"F1": [("F2", s - 1, j)] if s > 0 else [],
                "F2": [("F1", s, j)],
                "B1": [("F1", s, j)] + ([("B2", s + 1, j)] if s < P - 1 else []),
                "B2": [("B1", s, j)],
                "W2": [("F1", s, j)] + ([("B2", s + 1, j)] if s < P - 1 else []),
                "W1": [("B1", s, j)] + ([("F2", s - 1, j)] if s > 0 else [])}[name]
        for x in need:
            assert at[x] in clo[i], (kind, (name, s, j), x)


@settings(max_examples=150, deadline=None)
@given(pipelines(), st.sampled_from(S.SCHEDULES), dyadic, dyadic, dyadic, comm, st.data())
def test_trace_checker_accepts_simulated_and_rejects_early_starts(pm, kind, tf, tb, tw, tc, data):
    # every simulated step passes the oracle's trace checker, with and without
    # the trace's own dependency claims; moving one pass so that it starts
    # before one of its producers has ended (same length) is rejected
    P, m = pm
    t = S.Times(tf, tb, tw, tc)
    ev, _ = S.make_schedule(kind, P, m, t)
    evs = S.events_as_dicts(ev)
    r = S.check_trace(evs, P)
    assert abs(r["bubble_eq3"] - S.bubble_rate(ev, P, m, t)) < 1e-12
    bare = [{k: v for k, v in e.items() if k != "dependsOn"} for e in evs]
    assert S.check_trace(bare, P) == r
    with_producer = [e for e in evs if e["dependsOn"]]
    if not with_producer:
        return
    victim = data.draw(st.sampled_from(with_producer))
    ends = {e["id"]: e["end"] for e in evs}
    latest = max(ends[p] for p in victim["dependsOn"])
    shift = victim["start"] - latest + data.draw(st.sampled_from([0.0625, 0.25, 1.0]))
    moved = []
    for e in bare:
        e = dict(e)
        if e["id"] == victim["id"]:
            e["start"], e["end"] = e["start"] - shift, e["end"] - shift
        moved.append(e)
    if victim["start"] - shift < 0:
        return  # the move would leave the trace's time range
    with pytest.raises(S.ScheduleError) as ei:
        S.check_trace(moved, P)
    assert ei.value.code in ("early_consumer", "stage_collision")


@settings(max_examples=60, deadline=None)
@given(st.integers(1, 6), st.integers(1, 5), st.integers(1, 8), st.sampled_from(["gelu_erf", "gelu_tanh"]),
       st.booleans(), st.integers(0, 2**31 - 1))
def test_block_oracle_gradients_match_finite_differences(M, h, f, act, bias, seed):
    # the fp64 block's B and W against central differences of L = sum(Y * G)
    # on random tiny shapes (calculus, not the oracle, fixes the gradients)
    import numpy as np
    from oracle import block as ob
    rng = np.random.default_rng(seed)
    X, G = rng.standard_normal((M, h)), rng.standard_normal((M, h))
    W1, W2 = rng.standard_normal((h, f)) * 0.7, rng.standard_normal((f, h)) * 0.7
    b1 = rng.standard_normal(f) * 0.3 if bias else None
    b2 = rng.standard_normal(h) * 0.3 if bias else None
    H, A, _ = ob.forward(X, W1, W2, b1, b2, act)
    _, dH, dX = ob.backward_input(G, W1, W2, H, act)
    dW1, dW2, db1, db2 = ob.backward_weight(X, A, dH, G, act)

    def loss():
        return float(np.sum(ob.forward(X, W1, W2, b1, b2, act)[2] * G))

    params = [(dX, X), (dW1, W1), (dW2, W2)] + ([(db1, b1), (db2, b2)] if bias else [])
    for got, p in params:
        fd = np.zeros_like(p)
        for i in np.ndindex(p.shape):
            old = p[i]
            p[i] = old + 1e-6
            lp = loss()
            p[i] = old - 1e-6
            lm = loss()
            p[i] = old
            fd[i] = (lp - lm) / 2e-6
        assert np.abs(got - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max())
