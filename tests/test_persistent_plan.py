"""Host plans of the persistent executor (no GPU needed, no device work).

zb_persistent_plan records the GEMMs an op list would run, derives their
dependencies from conflicting byte ranges (with the arena the library plans),
reduces them, assigns the tiles to CTA pairs by simulation and checks that
the assignment cannot deadlock.  These tests check, for every ordering the
library generates, that

* the GEMM and tile counts are those of the list (6 GEMMs per stage and
  microbatch of the MLP block: H/A, Y, dH, dX, dW2, dW1);
* every data dependency of the split backward is implied by the kept edges,
  each pointing backwards in list order: the next stage's forward after
  this stage's Y, B after the stage's own F (H) and after the next stage's B
  (its dX is this stage's dY), dX after dH, W after the F and B it reads, the
  fp32 accumulation of a stage's W GEMMs in list order; for the two- and
  three-chunk ZB-V and interleaved 1F1B lists the same along the chain of
  virtual stages;
* the priority rule follows the GEMM sizes (list order for multi-wave GEMMs,
  longest chain for small ones), and the plan holds for one pair as well;
* the workspace size query counts the kernel's tables on top of the arena.
The order-safety check itself runs inside the library on every plan.
"""

import pytest

from split_backward_gemms_gb300 import build as B


@pytest.fixture(scope="module")
def zb():
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def _gemms(ops):
    """GEMM index -> (name, stage, micro) in list order."""
    out = []
    for op in ops:
        k, s, j = op[0], op[1], op[-1]
        if k == "F":
            out += [("F1", s, j), ("F2", s, j)]
        elif k == "B":
            out += [("B1", s, j), ("B2", s, j)]
        elif k == "W":
            out += [("W2", s, j), ("W1", s, j)]
        elif k == "BW":
            out += [("B1", s, j), ("B2", s, j), ("W2", s, j), ("W1", s, j)]
    return out


def _reach(n, edges):
    """closure[j] = set of GEMMs j transitively depends on."""
    deps = [[] for _ in range(n)]
    for c, p in edges:
        deps[c].append(p)
    clo = [set() for _ in range(n)]
    for j in range(n):
        for p in deps[j]:
            clo[j] |= {p} | clo[p]
    return clo


def _ops(zb, kind, P, m):
    if kind in ("ZB1P", "ZB2P"):
        limit = P if kind == "ZB1P" else 2 * P
        _, ops, _ = zb.zb_auto_schedule(P, m, 1.0, 1.0, 1.0, 0.0, limit, 1.0)
        return ops
    return zb.zb_make_schedule(kind, P, m)


@pytest.mark.parametrize("kind", ["1F1B", "ZBH1", "ZBH2", "ZB1P", "ZB2P"])
@pytest.mark.parametrize("P,m,M,h,f", [(4, 8, 2048, 1024, 4096), (3, 5, 520, 264, 1048), (2, 2, 96, 256, 512)])
def test_plan_keeps_every_data_dependency(zb, kind, P, m, M, h, f):
    ops = _ops(zb, kind, P, m)
    pl = zb.make_pipeline(P, m, zb.make_block(M, h, f))
    info, edges = zb.zb_persistent_plan(pl, ops, pairs=76)
    g = _gemms(ops)
    n = len(g)
    assert info.gemms == n == 6 * P * m
    t = lambda a, b: ((a + 255) // 256) * ((b + 255) // 256)
    assert info.tiles == P * m * (2 * t(M, f) + 2 * t(M, h) + t(f, h) + t(h, f))
    assert info.deps == len(edges) and all(p < c for c, p in edges)
    clo = _reach(n, edges)
    at = {x: i for i, x in enumerate(g)}
    for (name, s, j), i in at.items():
        need = []
        if name == "F1" and s > 0:
            need.append(("F2", s - 1, j))
        if name == "F2":
            need.append(("F1", s, j))
        if name == "B1":
            need.append(("F1", s, j))
            if s < P - 1:
                need.append(("B2", s + 1, j))
        if name == "B2":
            need.append(("B1", s, j))
        if name == "W2":
            need.append(("F1", s, j))
            if s < P - 1:
                need.append(("B2", s + 1, j))
        if name == "W1":
            need.append(("B1", s, j))
            if s > 0:
                need.append(("F2", s - 1, j))
        for x in need:
            assert at[x] in clo[i], (kind, (name, s, j), x)
    # a stage's weight-gradient GEMMs accumulate in list order
    for name in ("W2", "W1"):
        for s in range(P):
            seq = [i for i, x in enumerate(g) if x[0] == name and x[1] == s]
            for a, b in zip(seq, seq[1:]):
                assert a in clo[b], (kind, name, s)


def test_plan_priority_follows_gemm_sizes(zb):
    # the h=6144 one-stage step: multi-wave GEMMs, list order
    ops = [op for op in zb.zb_make_schedule("ZBH2", 8, 24) if op[1] == 0]
    info, _ = zb.zb_persistent_plan(zb.make_pipeline(1, 24, zb.make_block(3072, 6144, 24576)), ops)
    assert info.by_chain == 0 and info.gemms == 144 and info.tiles == 24 * 7488
    # the P=4, h=1024 pipeline: GEMMs of at most 128 tiles, longest chain first
    ops = zb.zb_make_schedule("ZBH1", 4, 8)
    info, _ = zb.zb_persistent_plan(zb.make_pipeline(4, 8, zb.make_block(2048, 1024, 4096)), ops)
    assert info.by_chain == 1 and info.gemms == 192 and info.tiles == 14336
    # makespan: no better than all tiles spread perfectly over the pairs
    assert info.est_makespan_kblocks * 76 >= 14336 * 16


def test_plan_on_one_pair_and_chunked_lists(zb):
    ops = zb.zb_make_schedule("ZBH2", 2, 4)
    pl = zb.make_pipeline(2, 4, zb.make_block(512, 256, 1024))
    info, _ = zb.zb_persistent_plan(pl, ops, pairs=1)
    assert info.max_tiles_per_pair == info.tiles
    ops = zb.zb_make_interleaved_schedule("ZBV", 2, 2, 4)
    pl = zb.make_pipeline(2, 4, zb.make_block(512, 256, 1024), chunks=2, layout="ZBV")
    info, edges = zb.zb_persistent_plan(pl, ops, pairs=76)
    assert info.gemms == 6 * 4 * 4 and all(p < c for c, p in edges)


def test_plan_errors(zb):
    ops = zb.zb_make_schedule("ZBH1", 2, 2)
    with pytest.raises(zb.ZBError) as e:
        zb.zb_persistent_plan(zb.make_pipeline(2, 2, zb.make_block(256, 256, 1024, has_bias=True)), ops)
    assert e.value.status == zb.ZB_ERR_UNSUPPORTED
    with pytest.raises(zb.ZBError) as e:
        zb.zb_persistent_plan(zb.make_pipeline(2, 2, zb.make_block(256, 256, 1024)), ops, pairs=0)
    assert e.value.status == zb.ZB_ERR_INVALID_ARG
    bad = [op for op in ops if op[0] != "W"]  # W missing: not a legal replay
    with pytest.raises(zb.ZBError):
        zb.zb_persistent_plan(zb.make_pipeline(2, 2, zb.make_block(256, 256, 1024)), bad)


def test_workspace_holds_the_replay_tables(zb):
    # the persistent executor's workspace is the stream executor's arena plus
    # the kernel's tables: per GEMM up to four tensor maps (128 bytes each),
    # a 128-byte job record, up to 16 dependency entries and a counter; per
    # tile one entry of the order
    for (P, m, M, h, f) in ((4, 8, 2048, 1024, 4096), (2, 4, 520, 264, 1048)):
        ops = zb.zb_make_schedule("ZBH1", P, m)
        blk = zb.make_block(M, h, f)
        ws_s, peak_s = zb.zb_schedule_workspace_size(zb.make_pipeline(P, m, blk), ops)
        ws_p, peak_p = zb.zb_schedule_workspace_size(zb.make_pipeline(P, m, blk, executor="persistent"), ops)
        info, _ = zb.zb_persistent_plan(zb.make_pipeline(P, m, blk), ops)
        nj, nt = info.gemms, info.tiles
        assert peak_p == peak_s
        extra = ws_p - ws_s
        assert extra >= nj * (4 * 128 + 128 + 16 * 4 + 4) + nt * 4
        assert extra <= nj * (4 * 128 + 128 + 16 * 4 + 4) + nt * 4 + 8 * 256


def _vstage(kind, P, op):
    """Virtual stage of a chunked op: cyclic (chunk c of stage s is c P + s)
    or V (chunk 0 of stage s is s, chunk 1 is 2P - 1 - s)."""
    _, s, c, _ = op
    if kind == "ZBV":
        return s if c == 0 else 2 * P - 1 - s
    return c * P + s


@pytest.mark.parametrize("kind,P,v,m", [("ZBV", 2, 2, 4), ("ZBV", 3, 2, 6), ("1F1B-I", 2, 2, 4), ("1F1B-I", 2, 3, 4)])
def test_chunked_plan_keeps_every_data_dependency(zb, kind, P, v, m):
    # the same rules along the chain of L = v P virtual stages
    M, h, f = 256, 256, 1024
    ops = zb.zb_make_interleaved_schedule(kind, P, v, m)
    L = v * P
    pl = zb.make_pipeline(P, m, zb.make_block(M, h, f), chunks=v, layout=kind)
    info, edges = zb.zb_persistent_plan(pl, ops, pairs=76)
    g = []
    for op in ops:
        if op[0] == "OPT":  # no GEMM
            continue
        k, s, j = op[0], _vstage(kind, P, op), op[3]
        g += {"F": [("F1", s, j), ("F2", s, j)], "B": [("B1", s, j), ("B2", s, j)],
              "W": [("W2", s, j), ("W1", s, j)],
              "BW": [("B1", s, j), ("B2", s, j), ("W2", s, j), ("W1", s, j)]}[k]
    assert info.gemms == len(g) == 6 * L * m
    assert all(p < c for c, p in edges)
    clo = _reach(len(g), edges)
    at = {x: i for i, x in enumerate(g)}
    for (name, s, j), i in at.items():
        need = {"F1": [("F2", s - 1, j)] if s > 0 else [],
                "F2": [("F1", s, j)],
                "B1": [("F1", s, j)] + ([("B2", s + 1, j)] if s < L - 1 else []),
                "B2": [("B1", s, j)],
                "W2": [("F1", s, j)] + ([("B2", s + 1, j)] if s < L - 1 else []),
                "W1": [("B1", s, j)] + ([("F2", s - 1, j)] if s > 0 else [])}[name]
        for x in need:
            assert at[x] in clo[i], (kind, (name, s, j), x)
    for name in ("W2", "W1"):
        for s in range(L):
            seq = [i for i, x in enumerate(g) if x[0] == name and x[1] == s]
            for a, b in zip(seq, seq[1:]):
                assert a in clo[b], (kind, name, s)
