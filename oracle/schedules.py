"""Oracle of the pipeline orderings: 1F1B, ZB-H1, ZB-H2 event graphs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Plain Python.

What is followed, and the readings taken where the pages leave a step open
--------------------------------------------------------------------------
Dependencies ([ZB-PP summary] §3.4 "critical dependency"; §3 Eqs. 4-5;
[ZB proven] "Draw the event graph before the Gantt"):
    F(s,j) after F(s-1,j) (+ T_comm);
    B(s,j) after F(s,j) and after B(s+1,j) (+ T_comm);
    W(s,j) after B(s,j) only;  the optimizer marker OPT(s) after every W of s.
1F1B ([Pipeline schedules] "1F1B: same bubble, bounded memory"; [ZB-PP summary]
§2 "Synchronous 1F1B"): stage s (0-indexed) runs min(P-1-s, m) warm-up
forwards, then alternates one forward (while any remain) with one backward,
then drains.  Its backward is the monolithic B+W, modelled as one fused op BW
whose input gradient is released only at its end.
ZB-H1 ([ZB-PP summary] §3.4 "Handcrafted Schedule ZB-H1", Table 2): 1F1B's F/B
order (warm-up min(P-s, m) forwards counting the first steady one), with W
split off and placed later.
ZB-H2 ([ZB-PP summary] §3.4 "Handcrafted Schedule ZB-H2"): stage 0 runs 2P-1
forwards before its first B; reading: stage s runs min(2(P-1-s)+1, m).
W placement for both ZB orderings (reading of [ZB-PP summary] §3.4 and the
heuristic's phases 2 and 4, "W insertion to fill bubbles", "Memory-triggered W
insertion", "Cool-down"): on a simulated timeline each stage runs its next F/B
the moment its dependencies are met; when the next F/B is not ready it runs
its oldest pending W; a W is forced before an F when the stage's live
microbatches (F done, W not done) reach L = P (H1, peak p M_B) or 2P-1 (H2,
peak (2p-1) M_B); leftover W's drain in ascending microbatch order.
With T_F = T_B = T_W this reproduces Table 2's bubbles exactly
((p-1)(T_F+T_B+T_W), (p-1)(T_F+T_B-T_W), (p-1)(T_F+T_B-2T_W)); with unequal
times it is a reading, not the paper's Figure 3 (which the pages do not show).
Global serial order for a one-GPU replay: (simulated start, stage index).

Metrics: per-stage span (Eq. 3: last end - first start), cost = max over
stages, bubble rate = (cost - m (T_F+T_B+T_W)) / cost ([ZB-PP summary] §5
"Metrics").  The [ZB proven] checker's denominator (global span x stages) is
also computed, labelled separately.  Closed forms (P-1)/(m+P-1) and
(P-1)/(v m + P-1) ([Pipeline schedules] "Interleaved stages").
Memory model ([ZB-PP summary] "The Memory Model"): F: +M_B, B: +M_W - M_B,
W: -M_W (BW: -M_B).
"""

from __future__ import annotations

import itertools
from collections import deque
from dataclasses import dataclass, field

KINDS = ("F", "B", "W", "BW", "OPT")
SCHEDULES = ("1F1B", "ZBH1", "ZBH2")


@dataclass(frozen=True)
class Times:
    F: float = 1.0
    B: float = 1.0
    W: float = 1.0
    comm: float = 0.0

    def dur(self, kind: str) -> float:
        if kind == "BW":
            return self.B + self.W
        if kind == "OPT":
            return 0.0
        return getattr(self, kind)


@dataclass
class Event:
    kind: str
    stage: int
    micro: int
    start: float
    end: float
    deps: tuple = field(default_factory=tuple)

    @property
    def id(self):
        return (self.kind, self.stage, self.micro)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def bubble_fraction(P: int, m: int, v: int = 1) -> float:
    """(P-1) / (v m + P-1): GPipe / 1F1B (v = 1) and interleaved 1F1B."""
    return (P - 1) / (v * m + P - 1)


def table2_bubble(kind: str, P: int, t: Times) -> float:
    """Bubble size of [ZB-PP summary] Table 2 (total idle per stage span)."""
    if kind == "1F1B":
        return (P - 1) * (t.F + t.B + t.W)
    if kind == "ZBH1":
        return (P - 1) * (t.F + t.B - t.W)
    if kind == "ZBH2":
        return (P - 1) * (t.F + t.B - 2 * t.W)
    raise ValueError(kind)


def table2_peak_mb(kind: str, P: int) -> int:
    """Peak activation memory in units of M_B ([ZB-PP summary] Table 2)."""
    return {"1F1B": P, "ZBH1": P, "ZBH2": 2 * P - 1}[kind]


# --------------------------------------------------------------------------
# per-stage F/B sequences
# --------------------------------------------------------------------------
def warmup_forwards(kind: str, P: int, m: int, s: int) -> int:
    if kind == "1F1B":
        return min(P - 1 - s, m)
    if kind == "ZBH1":
        return min(P - s, m)
    if kind == "ZBH2":
        return min(2 * (P - 1 - s) + 1, m)
    raise ValueError(kind)


def fb_sequence(kind: str, P: int, m: int, s: int):
    """The fixed F/B (or F/BW) order of stage s; W's are placed by simulate()."""
    w = warmup_forwards(kind, P, m, s)
    seq = [("F", j) for j in range(w)]
    nxt = w
    for b in range(m):
        if kind == "1F1B":
            if nxt < m:
                seq.append(("F", nxt))
                nxt += 1
            seq.append(("BW", b))
        else:
            seq.append(("B", b))
            if nxt < m:
                seq.append(("F", nxt))
                nxt += 1
    return seq


def live_limit(kind: str, P: int):
    return {"1F1B": None, "ZBH1": P, "ZBH2": 2 * P - 1}[kind]


# --------------------------------------------------------------------------
# dependencies
# --------------------------------------------------------------------------
def op_deps(kind: str, s: int, j: int, P: int, fused: bool):
    """Ids this op waits for.  B(s+1,j) is BW(s+1,j) when backward is fused."""
    bk = "BW" if fused else "B"
    if kind == "F":
        return (("F", s - 1, j),) if s > 0 else ()
    if kind in ("B", "BW"):
        d = [("F", s, j)]
        if s < P - 1:
            d.append((bk, s + 1, j))
        return tuple(d)
    if kind == "W":
        return (("B", s, j),)
    raise ValueError(kind)


def _is_cross_stage(dep, s):
    return dep[1] != s


# --------------------------------------------------------------------------
# list-scheduling simulator
# --------------------------------------------------------------------------
def simulate(kind: str, P: int, m: int, t: Times = Times()):
    """Simulate one ordering; returns the list of Events (no OPT markers)."""
    if P < 1 or m < 1:
        raise ValueError("P and m must be >= 1")
    fused = kind == "1F1B"
    seqs = [fb_sequence(kind, P, m, s) for s in range(P)]
    limit = live_limit(kind, P)
    ptr = [0] * P
    pending = [deque() for _ in range(P)]
    live = [0] * P
    t_free = [0.0] * P
    waiting = [False] * P
    end = {}
    events = []

    def has_work(s):
        return ptr[s] < len(seqs[s]) or bool(pending[s])

    def ready_at(s, k, j):
        tt = 0.0
        for d in op_deps(k, s, j, P, fused):
            if d not in end:
                return None
            tt = max(tt, end[d] + (t.comm if _is_cross_stage(d, s) else 0.0))
        return tt

    def run(s, k, j, start):
        e = start + t.dur(k)
        deps = op_deps(k, s, j, P, fused)
        events.append(Event(k, s, j, start, e, deps))
        end[(k, s, j)] = e
        t_free[s] = e
        if k == "F":
            live[s] += 1
        elif k == "B":
            pending[s].append(j)
        elif k in ("W", "BW"):
            live[s] -= 1

    while any(has_work(s) for s in range(P)):
        cands = [s for s in range(P) if has_work(s) and not waiting[s]]
        if not cands:
            raise RuntimeError("deadlock in simulate")
        s = min(cands, key=lambda x: (t_free[x], x))
        now = t_free[s]
        nxt = seqs[s][ptr[s]] if ptr[s] < len(seqs[s]) else None
        r = ready_at(s, nxt[0], nxt[1]) if nxt is not None else None
        acted = True
        if nxt is not None and r is not None and r <= now:
            if (nxt[0] == "F" and limit is not None and live[s] >= limit
                    and pending[s]):
                run(s, "W", pending[s].popleft(), now)
            else:
                run(s, nxt[0], nxt[1], now)
                ptr[s] += 1
        elif pending[s]:
            run(s, "W", pending[s].popleft(), now)
        else:
            acted = False
            if r is not None:
                t_free[s] = r
            else:
                later = [e for e in end.values() if e > now]
                later += [t_free[o] for o in range(P)
                          if o != s and has_work(o) and t_free[o] > now]
                if later:
                    t_free[s] = min(later)
                else:
                    waiting[s] = True
        if acted:
            for o in range(P):
                waiting[o] = False
    return events


def global_order(events):
    """One-GPU serial replay order: (start, stage), then append OPT markers."""
    evs = sorted(events, key=lambda e: (e.start, e.stage))
    ops = [(e.kind, e.stage, e.micro) for e in evs]
    P = 1 + max(e.stage for e in events)
    last = {}
    for i, (k, s, j) in enumerate(ops):
        last[s] = i
    # insert OPT(s) right after the last op of stage s, keeping relative order
    out = []
    for i, op in enumerate(ops):
        out.append(op)
        for s in range(P):
            if last.get(s) == i:
                out.append(("OPT", s, 0))
    return out


def make_schedule(kind: str, P: int, m: int, t: Times = Times()):
    """Events and the global op list (with OPT markers) of one ordering."""
    evs = simulate(kind, P, m, t)
    return evs, global_order(evs)


def stage_lists(ops, P: int):
    """Per-stage op sequences (kind, micro) from a global op list."""
    out = [[] for _ in range(P)]
    for k, s, j in ops:
        out[s].append((k, j))
    return out


# --------------------------------------------------------------------------
# metrics
# --------------------------------------------------------------------------
def stage_spans(events, P: int):
    spans = []
    for s in range(P):
        ev = [e for e in events if e.stage == s]
        spans.append(max(e.end for e in ev) - min(e.start for e in ev))
    return spans


def cost(events, P: int) -> float:
    """Eq. 3: max over stages of (end of last pass - start of first pass)."""
    return max(stage_spans(events, P))


def bubble_rate(events, P: int, m: int, t: Times) -> float:
    """(cost - m (T_F + T_B + T_W)) / cost  ([ZB-PP summary] §5 Metrics)."""
    c = cost(events, P)
    return (c - m * (t.F + t.B + t.W)) / c


def peak_live(events, P: int):
    """Peak live microbatches per stage (F done, W / BW not yet done)."""
    peaks = []
    for s in range(P):
        ev = sorted((e for e in events if e.stage == s), key=lambda e: e.start)
        cur = pk = 0
        for e in ev:
            if e.kind == "F":
                cur += 1
                pk = max(pk, cur)
            elif e.kind in ("W", "BW"):
                cur -= 1
        peaks.append(pk)
    return peaks


def memory_ledger(ops, P: int, M_B: float, M_W: float):
    """Running activation memory per stage under the Delta-M model.

    F: +M_B;  B: +M_W - M_B;  W: -M_W;  BW (B then W): -M_B.
    Returns (peak per stage, final per stage).
    """
    cur = [0.0] * P
    peak = [0.0] * P
    for k, s, j in ops:
        if k == "F":
            cur[s] += M_B
        elif k == "B":
            cur[s] += M_W - M_B
        elif k == "W":
            cur[s] -= M_W
        elif k == "BW":
            cur[s] -= M_B
        peak[s] = max(peak[s], cur[s])
    return peak, cur


# --------------------------------------------------------------------------
# validators
# --------------------------------------------------------------------------
class ScheduleError(ValueError):
    """Raised by the validators; ``code`` names the rule that failed."""

    def __init__(self, code: str, detail: str = ""):
        super().__init__(f"{code}: {detail}" if detail else code)
        self.code = code


def validate_ops(ops, P: int, m: int):
    """Check a global op list for legal one-GPU replay.

    Rules ([ZB-PP summary] §3.4 dependencies; [ZB proven] "Draw the event
    graph before the Gantt"): every (s, j) has exactly one F and either one B
    and one W or one fused BW; each op appears after its producers in list
    order; W/BW of a stage run in ascending microbatch order (so fp32
    accumulation follows a fixed order); OPT(s), if present, appears once and
    after every W/BW of stage s, and nothing of stage s follows it.
    Raises ScheduleError with code in {"kind", "stage", "micro", "duplicate",
    "mixed", "missing", "dependency", "w_order", "opt"}.
    """
    seen = {}
    last_w = [-1] * P
    opt_done = [False] * P
    for idx, op in enumerate(ops):
        if len(op) != 3:
            raise ScheduleError("kind", str(op))
        k, s, j = op
        if k not in KINDS:
            raise ScheduleError("kind", str(op))
        if not (0 <= s < P):
            raise ScheduleError("stage", str(op))
        if k != "OPT" and not (0 <= j < m):
            raise ScheduleError("micro", str(op))
        if opt_done[s]:
            raise ScheduleError("opt", f"{op} after OPT of its stage")
        if k == "OPT":
            opt_done[s] = True
            continue
        if (k, s, j) in seen:
            raise ScheduleError("duplicate", str(op))
        if k == "BW" and (("B", s, j) in seen or ("W", s, j) in seen):
            raise ScheduleError("mixed", str(op))
        if k in ("B", "W") and ("BW", s, j) in seen:
            raise ScheduleError("mixed", str(op))
        fused_next = ("BW", s + 1, j) in seen
        if k == "F":
            need = [("F", s - 1, j)] if s > 0 else []
        elif k in ("B", "BW"):
            need = [("F", s, j)]
            if s < P - 1:
                need.append(("BW", s + 1, j) if fused_next else ("B", s + 1, j))
        else:  # W
            need = [("B", s, j)]
        for d in need:
            if d not in seen:
                raise ScheduleError("dependency", f"{op} before {d}")
        if k in ("W", "BW"):
            if j <= last_w[s]:
                raise ScheduleError("w_order", str(op))
            last_w[s] = j
        seen[(k, s, j)] = idx
    for s in range(P):
        for j in range(m):
            has_f = ("F", s, j) in seen
            split = ("B", s, j) in seen and ("W", s, j) in seen
            fused = ("BW", s, j) in seen
            if not has_f or not (split or fused):
                raise ScheduleError("missing", f"stage {s} micro {j}")
    return True


def _producers(kind, s, j, stages, present):
    """The passes an event needs before it may start, by the dependency rules.

    [ZB proven] "Draw the event graph before the Gantt": a forward consumes
    the previous stage's forward output; an input-gradient pass consumes its
    own forward context and the next stage's input gradient (that stage's BW
    when its backward is fused); a weight-gradient pass consumes its own B;
    the optimizer consumes every weight gradient of its stage that the trace
    began (a forward without its W leaves the update waiting).
    ``present`` is the set of (kind, stage, micro) keys in the trace.
    """
    if kind == "F":
        return [] if s == 0 else [("F", s - 1, j)]
    if kind == "W":
        return [("B", s, j)]
    if kind in ("B", "BW"):
        need = [("F", s, j)]
        if s + 1 < stages:
            nxt = "BW" if ("BW", s + 1, j) in present else "B"
            need.append((nxt, s + 1, j))
        return need
    # OPT
    began = sorted(i for (k, t, i) in present if k == "F" and t == s)
    return [("BW" if ("BW", s, i) in present else "W", s, i) for i in began]


def check_trace(events, stages: int):
    """Legality and bubble accounting of a timed event trace of one step.

    Written from the prose of [ZB proven] "Draw the event graph before the
    Gantt" and "Validate the schedule as data".  A trace is a list of dicts
    {id, stage, micro, kind, start, end, dependsOn (optional)} with kind in
    F, B, W, BW (fused backward) or OPT (the stage's optimizer barrier, which
    may take no time).  The check builds the event graph: one node per
    (kind, stage, micro), producer edges both from the trace's own
    ``dependsOn`` claims and from the dependency rules (``_producers``), and
    resource edges that keep one stage's passes apart.  Failures raise
    ScheduleError with these codes:
        "stages"           the stage count is not a positive integer;
        "duplicate_id"     two events carry one id;
        "unknown_kind", "unknown_stage", "bad_interval"  (start < 0, end before
                           start, or a pass of zero length);
        "duplicate_work"   two events for one (kind, stage, micro);
        "missing_producer" a claimed or required producer is not in the trace;
        "early_consumer"   an event starts before a producer has ended;
        "stage_collision"  two events of one stage overlap in time.
    Producer edges are checked event by event in order of start time (ties
    by id), the trace's claims before the rules' requirements, so the error
    names the earliest offending consumer.

    Returns a dict:
        makespan           last end - first start;
        busy               the summed length of every pass;
        bubble_global      1 - busy / (stages x makespan): the checker's
                           denominator of [ZB proven];
        bubble_eq3         1 - busy / (stages x cost), cost = the longest
                           per-stage span (Eq. 3 of the summary, §5 Metrics);
        open_after_b       (stage, micro) pairs with a forward and no B / BW:
                           activations the input-gradient pass never released;
        open_after_w       pairs with a forward and no W / BW: activations of
                           the memory model ("The Memory Model") still held.
    """
    if isinstance(stages, bool) or not isinstance(stages, int) or stages < 1:
        raise ScheduleError("stages", repr(stages))
    by_id = {}
    for ev in events:
        if ev["id"] in by_id:
            raise ScheduleError("duplicate_id", str(ev["id"]))
        by_id[ev["id"]] = ev
    by_key = {}
    for ident, ev in by_id.items():
        kind, s = ev["kind"], ev["stage"]
        if kind not in KINDS:
            raise ScheduleError("unknown_kind", f"{ident}: {kind!r}")
        if isinstance(s, bool) or not isinstance(s, int) or not 0 <= s < stages:
            raise ScheduleError("unknown_stage", f"{ident}: {s!r}")
        a, b = float(ev["start"]), float(ev["end"])
        zero_ok = kind == "OPT"
        if not (0.0 <= a and (b > a or (zero_ok and b == a))) or b == float("inf"):
            raise ScheduleError("bad_interval", f"{ident}: [{a}, {b}]")
        key = (kind, s, 0 if kind == "OPT" else ev["micro"])
        if key in by_key:
            raise ScheduleError("duplicate_work", f"{by_key[key]} and {ident}")
        by_key[key] = ident
    present = set(by_key)

    # producer edges, in order of the consumers' start times
    for ident in sorted(by_id, key=lambda i: (float(by_id[i]["start"]), str(i))):
        ev = by_id[ident]
        claimed = list(ev.get("dependsOn") or ())
        key = (ev["kind"], ev["stage"], 0 if ev["kind"] == "OPT" else ev["micro"])
        required = [by_key.get(p, p) for p in _producers(*key, stages, present)]
        for p in claimed + required:
            if p not in by_id:
                raise ScheduleError("missing_producer", f"{ident} needs {p}")
            if float(by_id[p]["end"]) > float(ev["start"]):
                raise ScheduleError("early_consumer", f"{ident} starts before {p} ends")

    # resource edges: one pass at a time per stage
    lanes = {}
    for ident, ev in by_id.items():
        lanes.setdefault(ev["stage"], []).append((float(ev["start"]), float(ev["end"]), str(ident)))
    first = float("inf")
    last = float("-inf")
    longest_span = 0.0
    busy = 0.0
    for s, lane in lanes.items():
        lane.sort()
        free_at, holder = float("-inf"), None
        for a, b, ident in lane:
            if a < free_at:
                raise ScheduleError("stage_collision", f"{holder} and {ident} on stage {s}")
            free_at, holder = b, ident
            busy += b - a
        first = min(first, lane[0][0])
        last = max(last, free_at)
        longest_span = max(longest_span, free_at - lane[0][0])

    began = {(ev["stage"], ev["micro"]) for ev in by_id.values() if ev["kind"] == "F"}
    done_b = {(ev["stage"], ev["micro"]) for ev in by_id.values() if ev["kind"] in ("B", "BW")}
    done_w = {(ev["stage"], ev["micro"]) for ev in by_id.values() if ev["kind"] in ("W", "BW")}
    makespan = last - first if by_id else 0.0
    return {
        "makespan": makespan,
        "busy": busy,
        "bubble_global": 1.0 - busy / (stages * makespan) if makespan > 0 else 0.0,
        "bubble_eq3": 1.0 - busy / (stages * longest_span) if longest_span > 0 else 0.0,
        "open_after_b": len(began - done_b),
        "open_after_w": len(began - done_w),
    }


def events_as_dicts(events):
    """Convert simulator Events to validator dicts (ids as 'k:s:j' strings)."""
    def sid(i):
        return f"{i[0]}:{i[1]}:{i[2]}"
    return [{"id": sid(e.id), "stage": e.stage, "micro": e.micro, "kind": e.kind,
             "start": e.start, "end": e.end, "dependsOn": [sid(d) for d in e.deps]}
            for e in events]


# --------------------------------------------------------------------------
# brute force (tiny cases only)
# --------------------------------------------------------------------------
def _stage_orders(P, m, s, split=True):
    """All per-stage orders of F/B/W (or F/BW) for stage s obeying local deps."""
    ops = []
    for j in range(m):
        ops.append(("F", j))
        if split:
            ops += [("B", j), ("W", j)]
        else:
            ops.append(("BW", j))
    res = []
    for perm in itertools.permutations(ops):
        pos = {o: i for i, o in enumerate(perm)}
        ok = True
        for j in range(m):
            if split:
                if not (pos[("F", j)] < pos[("B", j)] < pos[("W", j)]):
                    ok = False
                    break
            elif not pos[("F", j)] < pos[("BW", j)]:
                ok = False
                break
        if ok:
            res.append(list(perm))
    return res


def evaluate_orders(orders, P, m, t: Times, fused=False):
    """As-soon-as-possible timeline of fixed per-stage orders; returns cost or
    None if the orders deadlock."""
    end = {}
    ptr = [0] * P
    t_free = [0.0] * P
    total = sum(len(o) for o in orders)
    done = 0
    progress = True
    while done < total and progress:
        progress = False
        for s in range(P):
            while ptr[s] < len(orders[s]):
                k, j = orders[s][ptr[s]]
                deps = op_deps(k, s, j, P, fused)
                if any(d not in end for d in deps):
                    break
                r = max([t_free[s]] + [end[d] + (t.comm if d[1] != s else 0.0) for d in deps])
                end[(k, s, j)] = r + t.dur(k)
                t_free[s] = end[(k, s, j)]
                ptr[s] += 1
                done += 1
                progress = True
    if done < total:
        return None
    spans = []
    for s in range(P):
        st = [end[(k, s, j)] - t.dur(k) for k, j in orders[s]]
        en = [end[(k, s, j)] for k, j in orders[s]]
        spans.append(max(en) - min(st))
    return max(spans)


def brute_force_min_cost(P, m, t: Times, split=True):
    """Minimum Eq. 3 cost over all per-stage orders (P, m tiny)."""
    per_stage = [_stage_orders(P, m, s, split) for s in range(P)]
    best = None
    for combo in itertools.product(*per_stage):
        c = evaluate_orders(list(combo), P, m, t, fused=not split)
        if c is not None and (best is None or c < best):
            best = c
    return best


# --------------------------------------------------------------------------
# heuristic automatic scheduler (ZB-1p / ZB-2p)
# --------------------------------------------------------------------------
def auto_schedule(P: int, m: int, t: Times, mem_limit: float, mw_ratio: float = 0.5,
                  h1: int = 1, h2: int = 0):
    """One run of the heuristic scheduler ([ZB-PP summary] §3 "The Heuristic
    Scheduling Algorithm", phases 1-4, and "The Memory Model").

    Memory is counted in units of M_B: F adds 1, B adds mw_ratio - 1
    (M_W = mw_ratio * M_B), W subtracts mw_ratio; a stage never starts a pass
    that would take it above mem_limit.  Reading of the phases, applied by a
    stage whenever it is free, in time order:
      * B first: a stage runs its next B as soon as it is ready (the critical
        path, "Schedule B promptly").
      * Warm-up / steady F: otherwise it runs its next F if that F is ready,
        fits in memory, and (h2 = 1) the stage is not already more than one
        forward ahead of the next stage (phase 3's skip hyperparameter).
        Before its first B, with h1 = 0 it stops adding forwards once one
        more F would delay that B (phase 1's hyperparameter); with h1 = 1 it
        keeps filling until memory stops it.
      * W: otherwise, with a W pending, it runs the oldest one when memory is
        what blocks the F (memory-triggered W), when the idle gap before the
        next F/B is at least T_W, or when idling the gap would make this
        stage's accumulated idle time the largest of all stages (the greedy
        "cumulative maximum bubble" rule); else it idles until the next pass
        becomes ready.  Idle time counts from a stage's first pass (a
        stage's span, Eq. 3, starts there).
      * Cool-down: remaining W's run in ascending order.
    Returns the list of Events.
    """
    nF = [0] * P
    nB = [0] * P
    pending = [deque() for _ in range(P)]
    mem = [0.0] * P
    idle = [0.0] * P
    t_free = [0.0] * P
    waiting = [False] * P
    endF, endB = {}, {}
    ends = []
    events = []
    eps = 1e-9

    def has_work(s):
        return nF[s] < m or nB[s] < m or bool(pending[s])

    def ready_f(s):
        j = nF[s]
        if j >= m:
            return None
        if s == 0:
            return 0.0
        e = endF.get((s - 1, j))
        return None if e is None else e + t.comm

    def ready_b(s):
        j = nB[s]
        if j >= m or j >= nF[s]:
            return None
        e = endF.get((s, j))
        if e is None:
            return None
        if s == P - 1:
            return e
        u = endB.get((s + 1, j))
        return None if u is None else max(e, u + t.comm)

    def run(s, k, j, start):
        d = t.dur(k)
        e = start + d
        deps = op_deps(k, s, j, P, False)
        events.append(Event(k, s, j, start, e, deps))
        ends.append(e)
        t_free[s] = e
        if k == "F":
            endF[(s, j)] = e
            nF[s] += 1
            mem[s] += 1.0
        elif k == "B":
            endB[(s, j)] = e
            nB[s] += 1
            mem[s] += mw_ratio - 1.0
            pending[s].append(j)
        else:
            mem[s] -= mw_ratio

    while any(has_work(s) for s in range(P)):
        cands = [s for s in range(P) if has_work(s) and not waiting[s]]
        if not cands:
            raise RuntimeError("deadlock in auto_schedule")
        s = min(cands, key=lambda x: (t_free[x], x))
        now = t_free[s]
        rb = ready_b(s)
        rf = ready_f(s)
        f_fits = mem[s] + 1.0 <= mem_limit + eps
        f_skip = h2 and s < P - 1 and nF[s] - nF[s + 1] > 1
        if (nB[s] == 0 and not h1 and rf is not None and rb is not None
                and rb < max(now, rf) + t.F):
            f_skip = True  # one more warm-up F would delay the first B
        f_ok = rf is not None and f_fits and not f_skip
        acted = True
        if rb is not None and rb <= now:
            run(s, "B", nB[s], now)
        elif f_ok and rf <= now:
            run(s, "F", nF[s], now)
        elif pending[s]:
            nxt = [x for x in (rb, rf if f_ok else None) if x is not None]
            gap = (min(nxt) - now) if nxt else float("inf")
            mem_block = rf is not None and rf <= now and not f_fits
            tail = nF[s] == m and nB[s] == m
            if (tail or mem_block or gap >= t.W - eps
                    or idle[s] + gap > max(idle) + eps):
                run(s, "W", pending[s].popleft(), now)
            else:
                if nF[s] > 0:
                    idle[s] += gap
                t_free[s] = min(nxt)
        else:
            acted = False
            nxt = [x for x in (rb, rf if f_ok else None) if x is not None and x > now]
            if nxt:
                if nF[s] > 0:
                    idle[s] += min(nxt) - now
                t_free[s] = min(nxt)
            else:
                later = [e for e in ends if e > now]
                later += [t_free[o] for o in range(P) if o != s and has_work(o) and t_free[o] > now]
                if later:
                    if nF[s] > 0:
                        idle[s] += min(later) - now
                    t_free[s] = min(later)
                else:
                    waiting[s] = True
        if acted:
            for o in range(P):
                waiting[o] = False
    return events


def auto_schedule_search(P: int, m: int, t: Times, mem_limit: float, mw_ratio: float = 0.5):
    """Grid search over the two binary hyperparameters; the smallest Eq. 3
    cost wins (ties: the first of (0,0), (0,1), (1,0), (1,1)).
    Returns (events, ops, (h1, h2))."""
    best = None
    for h1 in (0, 1):
        for h2 in (0, 1):
            ev = auto_schedule(P, m, t, mem_limit, mw_ratio, h1, h2)
            c = cost(ev, P)
            if best is None or c < best[0] - 1e-12:
                best = (c, ev, (h1, h2))
    return best[1], global_order(best[1]), best[2]


def mem_peaks(events, P: int, mw_ratio: float):
    """Peak activation memory per stage (units of M_B) of an event list."""
    peaks = []
    for s in range(P):
        cur = pk = 0.0
        for e in sorted((e for e in events if e.stage == s), key=lambda e: e.start):
            cur += {"F": 1.0, "B": mw_ratio - 1.0, "W": -mw_ratio, "BW": -1.0}[e.kind]
            pk = max(pk, cur)
        peaks.append(pk)
    return peaks
