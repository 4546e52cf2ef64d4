"""bench.py's op lists: every ordering it can replay (--schedule) on every
workload is a legal list for the executor, checked against the oracle's
validator, with the shape the workload states (the whole P-stage pipeline,
or the stage-0 list of an 8-stage ordering replayed as one stage).  Host
logic only: the lists come from the library's host generators."""

import pytest

import bench
from oracle import schedules as S


@pytest.fixture(scope="module")
def zb():
    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


@pytest.mark.parametrize("sched", ["1F1B", "ZBH1", "ZBH2", "ZB1P", "ZB2P"])
@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_bench_op_lists_are_legal(zb, name, sched):
    h, f, M, m, _, Pl, _ = bench.WORKLOADS[name]
    multi = name == "c2"
    ops = bench.make_ops(zb, sched, Pl, m, multi)
    P = Pl if multi else 1
    assert S.validate_ops(ops, P, m)
    per_micro = 2 if sched == "1F1B" else 3
    assert len(ops) == P * m * per_micro + P  # every pass once, one OPT per stage
    if sched in ("ZB1P", "ZB2P"):
        limit = Pl if sched == "ZB1P" else 2 * Pl
        _, ref, _ = S.auto_schedule_search(Pl, m, S.Times(), limit, 1.0)
        if not multi:
            ref = [(k, 0, j) for k, s, j in ref if s == 0]
        assert ops == ref
    else:
        _, ref = S.make_schedule(sched, Pl, m)
        if not multi:
            ref = [(k, 0, j) for k, s, j in ref if s == 0]
        assert ops == ref
