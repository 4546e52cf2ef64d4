"""Oracle of the multi-chunk orderings: interleaved 1F1B (1F1B-I) and ZB-V.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Plain Python.

A device (pipeline stage) s holds v model chunks; the model is a chain of
L = v P virtual stages k = 0 .. L-1 (forward order) and chunk c of device s is
virtual stage k(s, c):
  * cyclic assignment, 1F1B-I ([Pipeline schedules] "Interleaved stages";
    [ZB-PP summary] §5 "1F1B-I", §6 ZB-V paragraph on interleaving): stage i
    gets chunks i, p+i, 2p+i, ...  ->  k = c P + s;
  * V assignment, ZB-V ([ZB-PP summary] §6 "ZB-V"): exactly 2p chunks, stage
    i (1-indexed) gets chunks i and 2p-i+1  ->  k = s (c = 0) or 2P-1-s
    (c = 1).
Dependencies are those of the one-chunk orderings on the virtual chain:
F(k,j) after F(k-1,j); B(k,j) after F(k,j) and B(k+1,j); W(k,j) after B(k,j)
(T_comm added when the two virtual stages sit on different devices).  A
chunk pass takes T/v of the device's per-microbatch time T, so the ideal
per-device time stays m (T_F + T_B + T_W) and bubble rates are comparable
with the one-chunk orderings ([ZB-PP summary] §5 "Metrics", Eq. 3).

1F1B-I (reading of the interleaved schedule the pages cite, Narayanan et
al. 2021, as the pages describe it: cyclic chunks, 1F1B steady state, fused
backward): device s runs min(2(P-1-s) + (v-1) P, v m) warm-up chunk
forwards, then alternates one forward with one fused backward BW, then
drains the backwards.  Its i-th forward is chunk (i mod vP) div P of
microbatch (i div vP) P + (i mod P) -- microbatches enter in groups of P,
each group visiting the chunks in order -- and its i-th backward the same
microbatch of chunk v-1-(that chunk).  Requires m to be a multiple of P.
At equal times this reproduces the printed bubble (P-1)/(vm+P-1).

ZB-V (reading; the pages give the assignment and the properties -- zero
bubble at T_F = T_B = T_W with peak activation memory p M_B -- but not the
layout of its figure): the V assignment on a simulated timeline.  Whenever a
device is free it takes, among the passes that can start at the earliest
moment: a W when it holds 2P live chunk activations (F done, W not done;
P M_B, since a chunk activation is M_B/2), as only a W frees one; else an F
before a B before a W; within a kind the oldest microbatch first, then the
later virtual stage.  An F needs fewer than 2P live activations, and a
chunk-a forward (new work entering the device) fewer than 2P-1 unless a W of
the device is pending: the last slot either stays free for a chunk-b
forward or is freed by that W next, so the forward of the oldest unfinished
microbatch can always advance (no deadlock at any pass times, T_comm
included).  A W comes from the device's pending ones, oldest first.  At
equal times this leaves no device idle between its first and last pass and
peaks at exactly P M_B -- both properties the pages state (pinned for P up
to 8).  ``v_zero_bubble_exists`` shows by exhaustive search that no gap-free
V schedule holds less memory and none exists below m = 2P-1;
``v_gap_free_schedule_ilp`` asks the same question of the same model as a
0/1 integer program (scipy's HiGHS) and reaches larger P;
``check_gap_free_v`` checks any unit-slot schedule independently.
"""

from __future__ import annotations

from .schedules import KINDS, ScheduleError, Times, validate_ops

LAYOUTS = ("cyclic", "V")
INTERLEAVED = ("1F1B-I", "ZBV")


def virtual_stage(layout: str, P: int, s: int, c: int) -> int:
    if layout == "cyclic":
        return c * P + s
    if layout == "V":
        return s if c == 0 else 2 * P - 1 - s
    raise ValueError(layout)


def device_chunk(layout: str, P: int, k: int):
    """Inverse of virtual_stage: (device, chunk) of virtual stage k."""
    if layout == "cyclic":
        return k % P, k // P
    return (k, 0) if k < P else (2 * P - 1 - k, 1)


def layout_of(kind: str) -> str:
    return {"1F1B-I": "cyclic", "ZBV": "V"}[kind]


# --------------------------------------------------------------------------
# 1F1B-I: fixed per-device sequences
# --------------------------------------------------------------------------
def ilv_forward(P: int, v: int, i: int):
    """(chunk, micro) of a device's i-th chunk forward."""
    g, r = divmod(i, P * v)
    return r // P, g * P + i % P


def ilv_sequence(P: int, v: int, m: int, s: int):
    """Device s's op sequence [(kind, chunk, micro)] of 1F1B-I."""
    total = v * m
    warm = min(2 * (P - 1 - s) + (v - 1) * P, total)
    seq = [("F",) + ilv_forward(P, v, i) for i in range(warm)]
    for i in range(total - warm):
        seq.append(("F",) + ilv_forward(P, v, warm + i))
        c, j = ilv_forward(P, v, i)
        seq.append(("BW", v - 1 - c, j))
    for i in range(total - warm, total):
        c, j = ilv_forward(P, v, i)
        seq.append(("BW", v - 1 - c, j))
    return seq


def _check_args(kind, P, v, m):
    if kind not in INTERLEAVED:
        raise ValueError(kind)
    if P < 1 or m < 1:
        raise ValueError("P and m must be >= 1")
    if kind == "ZBV" and v != 2:
        raise ValueError("ZB-V has exactly two chunks per device")
    if kind == "1F1B-I":
        if v < 2:
            raise ValueError("1F1B-I needs v >= 2 chunks per device")
        if m % P:
            raise ValueError("1F1B-I needs m to be a multiple of P")


def _deps(kind, k, j, L, fused):
    """Virtual-stage dependencies (ids (kind, k, j))."""
    if kind == "F":
        return (("F", k - 1, j),) if k > 0 else ()
    if kind in ("B", "BW"):
        d = [("F", k, j)]
        if k < L - 1:
            d.append(("BW" if fused else "B", k + 1, j))
        return tuple(d)
    return (("B", k, j),)


def _dur(t: Times, kind: str, v: int) -> float:
    if kind == "BW":
        return (t.B + t.W) / v
    return {"F": t.F, "B": t.B, "W": t.W}[kind] / v


def simulate_ilv(P: int, v: int, m: int, t: Times = Times()):
    """Events [(kind, s, c, j, start, end)] of 1F1B-I: each device runs its
    sequence in order, every pass as soon as its producers have ended."""
    layout, L = "cyclic", v * P
    seqs = [ilv_sequence(P, v, m, s) for s in range(P)]
    pos, free = [0] * P, [0.0] * P
    end, events = {}, []
    progress = True
    while progress:
        progress = False
        for s in range(P):
            while pos[s] < len(seqs[s]):
                kind, c, j = seqs[s][pos[s]]
                k = virtual_stage(layout, P, s, c)
                ready = 0.0
                ok = True
                for d in _deps(kind, k, j, L, True):
                    if d not in end:
                        ok = False
                        break
                    cross = device_chunk(layout, P, d[1])[0] != s
                    ready = max(ready, end[d] + (t.comm if cross else 0.0))
                if not ok:
                    break
                st = max(ready, free[s])
                e = st + _dur(t, kind, v)
                end[(kind, k, j)] = e
                free[s] = e
                events.append((kind, s, c, j, st, e))
                pos[s] += 1
                progress = True
    if any(pos[s] < len(seqs[s]) for s in range(P)):
        raise RuntimeError("1F1B-I sequences deadlocked")
    return events


# --------------------------------------------------------------------------
# ZB-V: rule-based simulation
# --------------------------------------------------------------------------
def simulate_zbv(P: int, m: int, t: Times = Times(), limit: int | None = None):
    """Events [(kind, s, c, j, start, end)] of the ZB-V reading above."""
    layout, v, L = "V", 2, 2 * P
    limit = 2 * P if limit is None else limit
    nF, nB = [0] * L, [0] * L
    end = {}
    free = [0.0] * P
    live = [0] * P
    pend = [[] for _ in range(P)]  # pending W ids (j, k) per device
    events = []
    todo = 3 * L * m
    mine = [(virtual_stage(layout, P, s, 0), virtual_stage(layout, P, s, 1)) for s in range(P)]
    while todo:
        best = None
        for s in range(P):
            cands = []  # (start, kind rank, j, -k, kind, k)
            for k in mine[s]:
                j = nB[k]
                if j < nF[k]:
                    dep = ("F", k, j) if k == L - 1 else ("B", k + 1, j)
                    if dep in end:
                        r = end[dep]
                        if k < L - 1 and device_chunk(layout, P, k + 1)[0] != s:
                            r += t.comm
                        cands.append((max(r, free[s]), 2, j, -k, "B", k))
                j = nF[k]
                # a chunk-a forward leaves the last slot to chunk b unless a W
                # is pending (a full device runs that W next)
                room = live[s] < limit and (k >= P or live[s] < limit - 1 or bool(pend[s]))
                if j < m and room and (k == 0 or ("F", k - 1, j) in end):
                    r = 0.0
                    if k > 0:
                        r = end[("F", k - 1, j)]
                        if device_chunk(layout, P, k - 1)[0] != s:
                            r += t.comm
                    cands.append((max(r, free[s]), 1, j, -k, "F", k))
            if pend[s]:
                j, k = min(pend[s], key=lambda x: (x[0], -x[1]))
                wrank = 0 if live[s] >= limit else 3
                cands.append((max(end[("B", k, j)], free[s]), wrank, j, -k, "W", k))
            if not cands:
                continue
            s0 = min(c[0] for c in cands)
            pick = min((c for c in cands if c[0] == s0), key=lambda c: (c[1], c[2], c[3]))
            if best is None or (pick[0], s) < (best[0][0], best[1]):
                best = (pick, s)
        if best is None:
            raise RuntimeError("ZB-V simulation deadlocked (memory limit too small)")
        (st, _r, j, _nk, kind, k), s = best
        e = st + _dur(t, kind, v)
        end[(kind, k, j)] = e
        free[s] = e
        c = device_chunk(layout, P, k)[1]
        events.append((kind, s, c, j, st, e))
        if kind == "F":
            nF[k] += 1
            live[s] += 1
        elif kind == "B":
            nB[k] += 1
            pend[s].append((j, k))
        else:
            pend[s].remove((j, k))
            live[s] -= 1
        todo -= 1
    return events


# --------------------------------------------------------------------------
# lists and metrics
# --------------------------------------------------------------------------
def simulate_interleaved(kind: str, P: int, v: int, m: int, t: Times = Times()):
    _check_args(kind, P, v, m)
    if kind == "1F1B-I":
        return simulate_ilv(P, v, m, t)
    return simulate_zbv(P, m, t)


def global_order(kind: str, P: int, v: int, events):
    """One-GPU replay order (start, device), then OPT(s, c) after the last op
    of each virtual stage."""
    layout = layout_of(kind)
    evs = sorted(events, key=lambda e: (e[4], e[1]))
    ops = [(e[0], e[1], e[2], e[3]) for e in evs]
    last = {}
    for i, (kd, s, c, j) in enumerate(ops):
        last[virtual_stage(layout, P, s, c)] = i
    out = []
    for i, op in enumerate(ops):
        out.append(op)
        for k in range(v * P):
            if last.get(k) == i:
                s, c = device_chunk(layout, P, k)
                out.append(("OPT", s, c, 0))
    return out


def make_interleaved_schedule(kind: str, P: int, v: int, m: int, t: Times = Times()):
    evs = simulate_interleaved(kind, P, v, m, t)
    return evs, global_order(kind, P, v, evs)


def to_virtual(kind: str, P: int, ops):
    """(kind, s, c, j) ops -> (kind, k, j) ops on the virtual chain."""
    layout = layout_of(kind)
    return [(kd, virtual_stage(layout, P, s, c), j) for kd, s, c, j in ops]


def validate_interleaved(kind: str, P: int, v: int, m: int, ops):
    for op in ops:
        if len(op) != 4 or op[0] not in KINDS:
            raise ScheduleError("kind", str(op))
        if not (0 <= op[1] < P):
            raise ScheduleError("stage", str(op))
        if not (0 <= op[2] < v):
            raise ScheduleError("chunk", str(op))
    return validate_ops(to_virtual(kind, P, ops), v * P, m)


def device_spans(events, P: int):
    out = []
    for s in range(P):
        ev = [e for e in events if e[1] == s]
        out.append(max(e[5] for e in ev) - min(e[4] for e in ev))
    return out


def bubble_rate(events, P: int, m: int, t: Times) -> float:
    """(cost - m (T_F + T_B + T_W)) / cost, cost = max per-device span (Eq. 3)."""
    c = max(device_spans(events, P))
    return (c - m * (t.F + t.B + t.W)) / c


def peak_live_chunks(events, P: int):
    """Per device: peak live chunk activations (F done, W / BW not done)."""
    out = []
    for s in range(P):
        cur = pk = 0
        for e in sorted((e for e in events if e[1] == s), key=lambda e: e[4]):
            if e[0] == "F":
                cur += 1
                pk = max(pk, cur)
            elif e[0] in ("W", "BW"):
                cur -= 1
        out.append(pk)
    return out


# --------------------------------------------------------------------------
# exhaustive search: do gap-free V schedules exist?
# --------------------------------------------------------------------------
def v_zero_bubble_exists(P: int, m: int, limit: int, max_nodes: int = 2_000_000) -> bool:
    """Exhaustive search over unit-time V schedules (every chunk pass takes one
    slot, no T_comm): is there a schedule in which no device idles between its
    first and last pass while holding at most `limit` live chunk activations?
    F and B of a virtual stage run in microbatch order, W in any order.
    A device may delay its first pass.  Small P and m only."""
    L = 2 * P
    mine = [[k for k in range(L) if device_chunk("V", P, k)[0] == s] for s in range(P)]
    per_dev = 6 * m
    seen = set()
    nodes = [0]

    def rec(nF, nB, wdone, started, count):
        nodes[0] += 1
        if nodes[0] > max_nodes:
            raise RuntimeError("search too large")
        if all(c == per_dev for c in count):
            return True
        key = (nF, nB, wdone, started)
        if key in seen:
            return False
        choices = []
        for s in range(P):
            if count[s] == per_dev:
                choices.append([None])
                continue
            live = sum(nF[k] for k in mine[s]) - sum(bin(wdone[k]).count("1") for k in mine[s])
            c = []
            for k in mine[s]:
                j = nB[k]
                if j < nF[k] and (k == L - 1 or nB[k + 1] > j):
                    c.append(("B", k, j))
            for k in mine[s]:
                j = nF[k]
                if j < m and live < limit and (k == 0 or nF[k - 1] > j):
                    c.append(("F", k, j))
            for k in mine[s]:
                for j in range(nB[k]):
                    if not (wdone[k] >> j) & 1:
                        c.append(("W", k, j))
            if not c:
                if (started >> s) & 1:
                    seen.add(key)
                    return False
                c = [None]
            elif not (started >> s) & 1:
                c.append(None)
            choices.append(c)

        def prod(s, acc):
            if s == P:
                if all(a is None for a in acc):
                    return False
                nF2, nB2, w2 = list(nF), list(nB), list(wdone)
                st2, cnt2 = started, list(count)
                for dd, op in enumerate(acc):
                    if op is None:
                        continue
                    st2 |= 1 << dd
                    cnt2[dd] += 1
                    kd, k, j = op
                    if kd == "F":
                        nF2[k] += 1
                    elif kd == "B":
                        nB2[k] += 1
                    else:
                        w2[k] |= 1 << j
                return rec(tuple(nF2), tuple(nB2), tuple(w2), st2, tuple(cnt2))
            for op in choices[s]:
                if prod(s + 1, acc + [op]):
                    return True
            return False

        ok = prod(0, [])
        if not ok:
            seen.add(key)
        return ok

    z = tuple([0] * L)
    return rec(z, z, z, 0, tuple([0] * P))


# --------------------------------------------------------------------------
# the same question as an integer program (larger P than the search reaches)
# --------------------------------------------------------------------------
def v_gap_free_schedule_ilp(P: int, m: int, limit: int, max_delay: int | None = None,
                            time_limit: float = 60.0):
    """The model of ``v_zero_bubble_exists`` (unit slots, no T_comm, F and B
    of a virtual stage in microbatch order, W in any order; a device may
    delay its first pass, here by at most ``max_delay`` slots, default 4P) as
    a 0/1 integer program solved by scipy's HiGHS: x[op, t] = 1 when op
    starts in slot t; each op once; a device's slots from its first pass on
    hold exactly one op each for 6m slots (gap-free); every dependency ends
    before its consumer starts; at every slot a device holds at most `limit`
    live chunk activations (F done, W not done).  Returns {device: [(slot,
    kind, k, j), ...]} for a schedule, None when there is none, and raises
    RuntimeError when the solver stops at its time limit."""
    import numpy as np
    from scipy.optimize import Bounds, LinearConstraint, milp
    from scipy.sparse import coo_matrix

    L = 2 * P
    dmax = 4 * P if max_delay is None else max_delay
    T = dmax + 6 * m
    dev = [device_chunk("V", P, k)[0] for k in range(L)]
    ops = [(kd, k, j) for j in range(m) for k in range(L) for kd in "FBW"]
    # earliest and latest starts along each microbatch's chain
    es, ls = {}, {}
    for j in range(m):
        for k in range(L):
            es[("F", k, j)] = k
            es[("B", k, j)] = L + (L - 1 - k)
            es[("W", k, j)] = L + (L - 1 - k) + 1
            ls[("W", k, j)] = T - 1
            ls[("B", k, j)] = T - 2 - k
        for k in range(L):
            ls[("F", k, j)] = ls[("B", L - 1, j)] - 1 - (L - 1 - k)
    var = [(op, t) for op in ops for t in range(es[op], ls[op] + 1)]
    nx = len(var)
    n = nx + P * (dmax + 1)  # then one-hot first-slot offsets per device
    byop = {}
    for i, (op, t) in enumerate(var):
        byop.setdefault(op, []).append((i, t))
    rows, cols, vals, lo, hi = [], [], [], [], []

    def add(coefs, a, b):
        r = len(lo)
        for i, v in coefs.items():
            rows.append(r)
            cols.append(i)
            vals.append(v)
        lo.append(a)
        hi.append(b)

    for op in ops:
        add({i: 1 for i, _ in byop[op]}, 1, 1)
    for s in range(P):
        add({nx + s * (dmax + 1) + o: 1 for o in range(dmax + 1)}, 1, 1)
    bydt = {}
    for i, ((kd, k, j), t) in enumerate(var):
        bydt.setdefault((dev[k], t), []).append(i)
    for s in range(P):
        for t in range(T):
            c = {i: 1 for i in bydt.get((s, t), [])}
            for o in range(max(0, t - 6 * m + 1), min(t, dmax) + 1):
                c[nx + s * (dmax + 1) + o] = -1
            add(c, 0, 0)

    def before(a, b):  # start(a) + 1 <= start(b)
        c = {i: t for i, t in byop[b]}
        for i, t in byop[a]:
            c[i] = c.get(i, 0) - t
        add(c, 1, np.inf)

    for j in range(m):
        for k in range(L):
            if k > 0:
                before(("F", k - 1, j), ("F", k, j))
            before(("F", k, j), ("B", k, j))
            if k < L - 1:
                before(("B", k + 1, j), ("B", k, j))
            before(("B", k, j), ("W", k, j))
            if j + 1 < m:
                before(("F", k, j), ("F", k, j + 1))
                before(("B", k, j), ("B", k, j + 1))
    for s in range(P):
        fs = [(i, t) for i, ((kd, k, j), t) in enumerate(var) if kd == "F" and dev[k] == s]
        ws = [(i, t) for i, ((kd, k, j), t) in enumerate(var) if kd == "W" and dev[k] == s]
        for t in range(T):
            c = {i: 1 for i, tt in fs if tt <= t}
            for i, tt in ws:
                if tt < t:
                    c[i] = c.get(i, 0) - 1
            add(c, -np.inf, limit)
    A = coo_matrix((vals, (rows, cols)), shape=(len(lo), n)).tocsr()
    res = milp(c=np.zeros(n), constraints=LinearConstraint(A, np.array(lo, float), np.array(hi, float)),
               integrality=np.ones(n), bounds=Bounds(0, 1), options={"time_limit": time_limit})
    if res.status == 2:
        return None
    if res.status != 0 or res.x is None:
        raise RuntimeError(f"integer program not decided: {res.message}")
    out = {s: [] for s in range(P)}
    for i, ((kd, k, j), t) in enumerate(var):
        if res.x[i] > 0.5:
            out[dev[k]].append((t, kd, k, j))
    for s in out:
        out[s].sort()
    return out


def check_gap_free_v(P: int, m: int, limit: int, sched) -> None:
    """Independent check of a unit-slot V schedule {device: [(slot, kind, k,
    j)]}: every pass once on its own device, one pass per slot with no idle
    slot between a device's first and last, each dependency in an earlier
    slot, at most `limit` live chunk activations on a device at any slot.
    Raises AssertionError on the first violation."""
    L = 2 * P
    when = {}
    for s, row in sched.items():
        slots = [t for t, *_ in row]
        assert slots == list(range(slots[0], slots[0] + len(slots))), f"device {s} idles"
        assert len(row) == 6 * m, f"device {s} runs {len(row)} passes"
        live = peak = 0
        for t, kd, k, j in row:
            assert device_chunk("V", P, k)[0] == s, f"{kd}{k},{j} on device {s}"
            assert (kd, k, j) not in when, f"{kd}{k},{j} twice"
            when[(kd, k, j)] = t
            if kd == "F":
                live += 1
                peak = max(peak, live)
            elif kd == "W":
                live -= 1
        assert peak <= limit, f"device {s} holds {peak} > {limit}"
    assert len(when) == 3 * L * m
    for (kd, k, j), t in when.items():
        deps = []
        if kd == "F" and k > 0:
            deps.append(("F", k - 1, j))
        if kd == "B":
            deps.append(("F", k, j))
            if k < L - 1:
                deps.append(("B", k + 1, j))
        if kd == "W":
            deps.append(("B", k, j))
        for d in deps:
            assert when[d] < t, f"{kd}{k},{j} at {t} before {d} at {when[d]}"
