"""Pins of the multi-chunk orderings oracle (1F1B-I and ZB-V).

* the V assignment is the one the pages state (stage i holds chunks i and
  2p-i+1) and the cyclic one (stage i holds i, p+i, ...);
* 1F1B-I reproduces the bubble table printed in "Pipeline Schedules: GPipe,
  1F1B and Zero Bubble", section "Interleaved stages", and the closed form
  (P-1)/(vm+P-1) it comes from, exactly, at other sizes too; it needs more
  memory than 1F1B ("ZB-PP" summary, §6.2: 1F1B-I "requires more memory");
* ZB-V peaks at exactly p M_B on every device ("ZB-PP" summary, §6) and
  its bubble lies below ZB-H1's and 1F1B-I's at equal times (Table 8's
  ordering);
* exhaustive search: gap-free V schedules exist at p M_B and not below --
  the pages' zero-bubble claim -- and the search itself is pinned by the
  one-device case;
* every generated list is a valid replay of the virtual chain, with and
  without communication time.
"""

import os

import numpy as np
import pytest

from oracle import interleaved as I
from oracle import schedules as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bubble_table.txt")


def _rows():
    out = []
    with open(GOLDEN) as fh:
        for ln in fh:
            if ln.strip() and not ln.startswith("#"):
                P, m, v1, v2, v4 = ln.split()
                out.append((int(P), int(m), float(v1), float(v2), float(v4)))
    return out


@pytest.mark.parametrize("P", [1, 2, 3, 4, 7, 8])
def test_v_assignment_is_the_pages(P):
    for i in range(1, P + 1):  # 1-indexed stage, 1-indexed chunks
        got = {I.virtual_stage("V", P, i - 1, c) + 1 for c in (0, 1)}
        assert got == {i, 2 * P - i + 1}
    for k in range(2 * P):
        s, c = I.device_chunk("V", P, k)
        assert I.virtual_stage("V", P, s, c) == k


@pytest.mark.parametrize("P,v", [(1, 2), (4, 2), (4, 4), (3, 3)])
def test_cyclic_assignment(P, v):
    for i in range(1, P + 1):
        got = sorted(I.virtual_stage("cyclic", P, i - 1, c) + 1 for c in range(v))
        assert got == [i + c * P for c in range(v)]


@pytest.mark.parametrize("row", _rows())
def test_1f1b_i_reproduces_the_printed_table(row):
    P, m, _v1, v2, v4 = row
    t = S.Times()
    for v, printed in ((2, v2), (4, v4)):
        ev = I.simulate_interleaved("1F1B-I", P, v, m, t)
        b = I.bubble_rate(ev, P, m, t)
        assert round(100 * b, 1) == printed
        assert abs(b - (P - 1) / (v * m + P - 1)) < 1e-12


@pytest.mark.parametrize("P,m,v", [(2, 2, 2), (2, 6, 3), (3, 9, 2), (4, 4, 2), (5, 10, 4), (6, 12, 2),
                                   (8, 24, 2), (1, 3, 2)])
def test_1f1b_i_closed_form(P, m, v):
    t = S.Times()
    ev = I.simulate_interleaved("1F1B-I", P, v, m, t)
    assert abs(I.bubble_rate(ev, P, m, t) - (P - 1) / (v * m + P - 1)) < 1e-12


@pytest.mark.parametrize("P,m", [(4, 8), (8, 16), (4, 12)])
def test_1f1b_i_needs_more_memory_than_1f1b(P, m):
    ev = I.simulate_interleaved("1F1B-I", P, 2, m)
    peaks = I.peak_live_chunks(ev, P)
    assert peaks[0] / 2 > P  # in units of M_B (a chunk activation is M_B / v)
    ev1, _ = S.make_schedule("1F1B", P, m)
    assert max(S.peak_live(ev1, P)) == P


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 8])
def test_zbv_peak_is_p_mb_on_every_device(P):
    for m in sorted({max(1, 2 * P - 1), 2 * P, 3 * P}):
        ev = I.simulate_interleaved("ZBV", P, 2, m)
        assert I.peak_live_chunks(ev, P) == [2 * P] * P  # 2P chunks of M_B / 2


@pytest.mark.parametrize("P", [2, 3, 4, 5, 6, 8])
def test_zbv_bubble_below_zbh1_and_1f1b_i(P):
    t = S.Times()
    for m in (2 * P, 3 * P, 4 * P):
        zbv = I.bubble_rate(I.simulate_interleaved("ZBV", P, 2, m, t), P, m, t)
        h1 = S.bubble_rate(S.make_schedule("ZBH1", P, m, t)[0], P, m, t)
        ilv = I.bubble_rate(I.simulate_interleaved("1F1B-I", P, 2, m, t), P, m, t)
        assert zbv < h1 and zbv < ilv


def test_search_pinned_by_one_device():
    # one device holds both chunks: something is always ready once two
    # activations fit, and nothing can run past the first F with one
    for m in (1, 2, 3):
        assert I.v_zero_bubble_exists(1, m, 2)
        assert not I.v_zero_bubble_exists(1, m, 1)


@pytest.mark.parametrize("P,m", [(2, 3), (2, 4), (3, 5)])
def test_gap_free_v_schedules_exist_at_p_mb_and_not_below(P, m):
    assert I.v_zero_bubble_exists(P, m, 2 * P)
    assert not I.v_zero_bubble_exists(P, m, 2 * P - 1)


@pytest.mark.parametrize("P", [2, 3])
def test_gap_free_v_needs_m_at_least_2p_minus_1(P):
    assert not I.v_zero_bubble_exists(P, 2 * P - 2, 2 * P)


@pytest.mark.parametrize("P,m,limit", [(1, 3, 2), (1, 2, 1), (2, 2, 4), (2, 3, 4), (2, 4, 4), (2, 4, 3),
                                       (3, 4, 6), (3, 5, 6), (3, 5, 5)])
def test_integer_program_agrees_with_the_search(P, m, limit):
    # two independent methods on the same model: depth-first search over
    # slots and a 0/1 program; every schedule found passes the checker
    sched = I.v_gap_free_schedule_ilp(P, m, limit)
    assert (sched is not None) == I.v_zero_bubble_exists(P, m, limit)
    if sched is not None:
        I.check_gap_free_v(P, m, limit, sched)


@pytest.mark.parametrize("P", list(range(1, 9)))
def test_zbv_rule_is_gap_free_at_equal_times(P):
    # the summary's ZB-V properties: no bubble at T_F = T_B = T_W with peak
    # p M_B (2P chunk activations); the rule's schedule, in unit slots of
    # one chunk pass, also passes the independent gap-free checker
    t = S.Times()
    for m in sorted({max(1, 2 * P - 1), 2 * P, 3 * P, 3 * P + 1, 4 * P + 3}):
        ev = I.simulate_zbv(P, m, t)
        assert I.bubble_rate(ev, P, m, t) == 0.0, (P, m)
        assert max(I.peak_live_chunks(ev, P)) == min(2 * P, 2 * m)
        sched = {s: [] for s in range(P)}
        for kind, s, c, j, st, en in ev:
            k = I.virtual_stage("V", P, s, c)
            sched[s].append((int(round(st * 2)), kind, k, j))
        for s in sched:
            sched[s].sort()
        I.check_gap_free_v(P, m, 2 * P, sched)


def test_zbv_rule_never_deadlocks_at_random_times():
    rng = np.random.default_rng(5)
    for _ in range(40):
        t = S.Times(*rng.uniform(0.3, 2.0, 3), float(rng.choice([0.0, rng.uniform(0.0, 0.6)])))
        P = int(rng.integers(1, 9))
        m = int(rng.integers(1, 4 * P + 4))
        ev = I.simulate_zbv(P, m, t)
        assert len(ev) == 6 * P * m
        assert max(I.peak_live_chunks(ev, P)) <= 2 * P


def test_gap_free_checker_rejects_planted_mistakes():
    P, m, limit = 2, 4, 4
    good = I.v_gap_free_schedule_ilp(P, m, limit)
    I.check_gap_free_v(P, m, limit, good)

    def planted(edit):
        bad = {s: list(row) for s, row in good.items()}
        edit(bad)
        with pytest.raises(AssertionError):
            I.check_gap_free_v(P, m, limit, bad)

    # an idle slot: shift the last pass of device 0 one slot later
    planted(lambda b: b[0].__setitem__(-1, (b[0][-1][0] + 1,) + b[0][-1][1:]))
    # a dependency broken: device 0's first B trades slots with its first
    # pass, so it runs no later than the F it needs (same device, later)
    def swap(b):
        row = b[0]
        p = next(i for i, (_, kd, _, _) in enumerate(row) if kd == "B")
        (t0, *o0), (tp, *op) = row[0], row[p]
        row[0], row[p] = (t0, *op), (tp, *o0)
    planted(swap)
    # a pass missing (and another duplicated)
    planted(lambda b: b[0].__setitem__(-1, (b[0][-1][0],) + b[0][-2][1:]))
    # too little memory for this schedule
    with pytest.raises(AssertionError):
        I.check_gap_free_v(P, m, limit - 1, good)


TIMES = [S.Times(), S.Times(1.0, 1.2, 0.6, 0.0), S.Times(18.522, 18.086, 9.337, 0.601),
         S.Times(1.0, 1.0, 1.5, 0.1)]


@pytest.mark.parametrize("t", TIMES)
@pytest.mark.parametrize("kind,P,v,m", [("ZBV", 1, 2, 3), ("ZBV", 2, 2, 5), ("ZBV", 4, 2, 8),
                                        ("ZBV", 3, 2, 2), ("1F1B-I", 2, 2, 4), ("1F1B-I", 4, 2, 8),
                                        ("1F1B-I", 3, 3, 6)])
def test_lists_are_valid_replays(t, kind, P, v, m):
    ev, ops = I.make_interleaved_schedule(kind, P, v, m, t)
    assert I.validate_interleaved(kind, P, v, m, ops)
    # events respect dependencies (+ T_comm across devices) and never overlap on a device
    layout = I.layout_of(kind)
    end = {(e[0], I.virtual_stage(layout, P, e[1], e[2]), e[3]): e for e in ev}
    for e in ev:
        k = I.virtual_stage(layout, P, e[1], e[2])
        for d in I._deps(e[0], k, e[3], v * P, kind == "1F1B-I"):
            de = end[d]
            gap = t.comm if de[1] != e[1] else 0.0
            assert e[4] >= de[5] + gap - 1e-9
    for s in range(P):
        mine = sorted((e for e in ev if e[1] == s), key=lambda e: e[4])
        for a, b in zip(mine, mine[1:]):
            assert b[4] >= a[5] - 1e-9


def test_validator_rejects_bad_chunk_and_order():
    _, ops = I.make_interleaved_schedule("ZBV", 2, 2, 3)
    with pytest.raises(S.ScheduleError) as e:
        I.validate_interleaved("ZBV", 2, 2, 3, [("F", 0, 2, 0)] + ops)
    assert e.value.code == "chunk"
    bad = list(ops)
    i = bad.index(("F", 1, 0, 0))  # virtual stage 1 needs virtual stage 0 first
    bad.insert(0, bad.pop(i))
    with pytest.raises(S.ScheduleError) as e:
        I.validate_interleaved("ZBV", 2, 2, 3, bad)
    assert e.value.code == "dependency"


def test_bad_arguments():
    with pytest.raises(ValueError):
        I.simulate_interleaved("ZBV", 2, 3, 4)
    with pytest.raises(ValueError):
        I.simulate_interleaved("1F1B-I", 4, 2, 6)  # m not a multiple of P
    with pytest.raises(ValueError):
        I.simulate_interleaved("1F1B-I", 4, 1, 8)


def test_zbv_random_times_valid_and_within_p_mb():
    import random
    rng = random.Random(7)
    for _ in range(150):
        P = rng.randint(1, 6)
        m = rng.randint(1, 3 * P + 2)
        t = S.Times(rng.uniform(0.2, 3), rng.uniform(0.2, 3), rng.uniform(0.1, 3),
                    rng.choice([0.0, rng.uniform(0, 1)]))
        ev, ops = I.make_interleaved_schedule("ZBV", P, 2, m, t)
        assert I.validate_interleaved("ZBV", P, 2, m, ops)
        assert max(I.peak_live_chunks(ev, P)) <= 2 * P
