"""GPU parity of post-update validation with AdamW against the fp64 oracle.

"Zero Bubble Pipeline Parallelism" (paper-graph-ui summary), §4 "The Optimizer
Synchronization Bypass" and "Why rollback is feasible": stages step with their
staged-reduce partial state, and a stage whose clip / skip decision differs
from the global one inverts its step and redoes it.  The library's result is
compared, tensor by tensor, with ``oracle.optimizer.post_validated_step`` and
with the synchronous step it must equal; its per-stage decisions with the
oracle's report.  The round trip step -> rollback is checked on its own: a
NaN in a late stage makes every earlier stage roll back to its starting
values.  Tolerance: 1e-5 relative Frobenius (fp32 arithmetic).
"""

import numpy as np
import pytest
import torch

from oracle import block as ob
from oracle import optimizer as oo
from split_backward_gemms_gb300 import inputs as I
from tests.gpu_util import dev_bf16, dev_f32, empty_f32, f64, have_gpu, sync

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
HP = oo.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
STEP = 3


@pytest.fixture(scope="module")
def zb():
    if not have_gpu():
        pytest.skip("no CUDA device")
    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb as _zb
    return _zb


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def hp_c(zb, max_norm, step=STEP):
    return zb.make_adamw(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, max_norm, step)


def _device_state(zb, draws, with_bf16):
    """Device tensors for every (theta, m, v, g); returns (tensors, dev)."""
    dev, tensors = [], []
    for s, st in enumerate(draws):
        ds = []
        for k, (th, m, v, g) in enumerate(st):
            d = {"theta": dev_f32(th), "m": dev_f32(m), "v": dev_f32(v), "grad": dev_f32(g)}
            d["weight_bf16"] = d["theta"].to(torch.bfloat16) if with_bf16(s, k) else None
            ds.append(d)
            tensors.append(dict(d, stage=s))
        dev.append(ds)
    return tensors, dev


def _stage_states(zb, dev):
    """Each stage's {sum of squares, NaN/Inf count} from zb_grad_stats, four
    gradient buffers per call (its limit), the calls' results added."""
    nbytes = zb.zb_grad_stats_scratch_bytes()
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = []
    for ds in dev:
        total = torch.zeros(2, dtype=torch.float64, device="cuda")
        gs = [d["grad"] for d in ds if d["grad"].numel() > 0]
        for i in range(0, len(gs), 4):
            o = torch.zeros(2, dtype=torch.float64, device="cuda")
            zb.zb_grad_stats(gs[i:i + 4], [g.numel() for g in gs[i:i + 4]], o, scratch, nbytes)
            sync(zb)  # the scratch is reused by the next call
            total += o
        out.append(total)
    return out


def _run(zb, draws, max_norm, with_bf16=lambda s, k: k == 0):
    P = len(draws)
    tensors, dev = _device_state(zb, draws, with_bf16)
    states = _stage_states(zb, dev)
    dec = torch.empty(P * 40, dtype=torch.uint8, device="cuda")
    zb.zb_post_validated_adamw(P, states, tensors, hp_c(zb, max_norm), dec)
    sync(zb)
    return dev, zb.decisions_from_bytes(dec.cpu().numpy().tobytes(), P)


def _oracle(draws, max_norm):
    # the library's max_norm = 0 switches clipping off: an infinite threshold
    max_norm = np.inf if max_norm == 0 else max_norm
    params = [[(th, m, v) for th, m, v, _ in st] for st in draws]
    grads = [[g for *_, g in st] for st in draws]
    new, report = oo.post_validated_step(params, grads, STEP, HP, max_norm)
    sync_new = oo.synchronous_step(params, grads, STEP, HP, max_norm)
    return new, report, sync_new


SIZES = [72 * 200, 200 * 72, 200, 72, 1001, 3]  # ragged tails, one not a multiple of 4
N_STAGE = sum(SIZES)


def _draws(P=4, seed=11, grad_std=None):
    return I.optimizer_draws([SIZES] * P, seed=seed, grad_std=grad_std)


def _partial_norms(draws):
    sq = np.cumsum([sum(float(np.sum(g.astype(np.float64) ** 2)) for *_, g in st) for st in draws])
    return np.sqrt(sq)


def _check(zb, draws, max_norm, expect_rollback):
    dev, dec = _run(zb, draws, max_norm)
    new, report, sync_new = _oracle(draws, max_norm)
    assert [d["rolled_back"] for d in dec] == [int(r["rolled_back"]) for r in report] == \
        [int(x) for x in expect_rollback]
    for s, (d, r) in enumerate(zip(dec, report)):
        assert d["skip_used"] == int(r["skip"]) and d["skip_global"] == int(r["global_skip"])
        assert abs(d["scale_used"] - r["scale"]) <= 1e-6 * r["scale"]
        assert abs(d["scale_global"] - r["global_scale"]) <= 1e-6 * r["global_scale"]
    worst = 0.0
    for s, ds in enumerate(dev):
        for k, d in enumerate(ds):
            got = [f64(d[n]) for n in ("theta", "m", "v")]
            for gv, want, want_sync in zip(got, new[s][k], sync_new[s][k]):
                e = rel(gv, want)
                worst = max(worst, e)
                assert e <= TOL_F32, (s, k, e)
                assert rel(gv, want_sync) <= TOL_F32
            if d["weight_bf16"] is not None:
                assert torch.equal(d["weight_bf16"], d["theta"].to(torch.bfloat16))
    return dev, dec, worst


def test_no_clip_no_rollback(zb):
    _check(zb, _draws(), 0.0, [0, 0, 0, 0])
    _check(zb, _draws(seed=12), 1e9, [0, 0, 0, 0])


def test_clip_decided_by_last_stage_rolls_back_earlier_stages(zb):
    draws = _draws()
    n = _partial_norms(draws)
    c = float(np.sqrt(n[2] * n[3]))  # between the 3-stage and the global norm
    _, dec, _ = _check(zb, draws, c, [1, 1, 1, 0])
    assert all(d["scale_used"] == 1.0 for d in dec[:3]) and dec[3]["scale_used"] < 1.0


def test_clip_everywhere_with_different_partial_scales(zb):
    draws = _draws(grad_std=[1.0, 0.5, 2.0, 0.25])
    n = _partial_norms(draws)
    c = float(0.5 * n[0])
    _, dec, _ = _check(zb, draws, c, [1, 1, 1, 0])
    assert len({d["scale_used"] for d in dec}) == 4


def test_single_stage_never_rolls_back(zb):
    draws = _draws(P=1)
    n = _partial_norms(draws)
    _check(zb, draws, float(0.5 * n[0]), [0])


@pytest.mark.parametrize("bad_stage,value", [(2, np.nan), (3, np.inf), (1, -np.inf)])
def test_nonfinite_late_rolls_back_to_start(zb, bad_stage, value):
    """Round trip: stages before the bad one stepped, then inverted their step."""
    draws = _draws(seed=20 + bad_stage)
    draws[bad_stage][1][3][17] = value
    start = [[tuple(a.copy() for a in t[:3]) for t in st] for st in draws]
    expect = [1 if s < bad_stage else 0 for s in range(4)]
    dev, dec, _ = _check(zb, draws, 1e4, expect)  # no clipping: only the skip differs
    for s, ds in enumerate(dev):
        for k, d in enumerate(ds):
            for name, want in zip(("theta", "m", "v"), start[s][k]):
                got = d[name].cpu().numpy()
                if s < bad_stage:
                    assert rel(got, want) <= TOL_F32, (s, k, name)
                else:
                    assert np.array_equal(got, want)  # never written


def test_nonfinite_first_stage_skips_everything(zb):
    draws = _draws(seed=30)
    draws[0][0][3][5] = np.nan
    dev, dec, _ = _check(zb, draws, 1e4, [0, 0, 0, 0])
    assert all(d["skip_used"] == 1 and d["skip_global"] == 1 for d in dec)
    for s, ds in enumerate(dev):
        for k, d in enumerate(ds):
            assert np.array_equal(d["theta"].cpu().numpy(), draws[s][k][0])


def test_many_tensors_span_several_launch_tables(zb):
    """More than 64 tensors (and empty ones) split over several launches."""
    rng = np.random.default_rng(4)
    sizes = [[int(x) for x in rng.integers(0, 3000, size=45)] for _ in range(3)]
    sizes[1][7] = 0
    draws = I.optimizer_draws(sizes, seed=5)
    n = _partial_norms(draws)
    c = float(np.sqrt(n[1] * n[2]))
    dev, dec = _run(zb, draws, c, with_bf16=lambda s, k: k % 3 == 0)
    new, report, _ = _oracle(draws, c)
    assert [d["rolled_back"] for d in dec] == [1, 1, 0]
    for s, ds in enumerate(dev):
        for k, d in enumerate(ds):
            for name, want in zip(("theta", "m", "v"), new[s][k]):
                if want.size:
                    assert rel(f64(d[name]), want) <= TOL_F32, (s, k, name)


def test_repeatable_bits(zb):
    draws = _draws(seed=40)
    n = _partial_norms(draws)
    c = float(np.sqrt(n[1] * n[2]))
    a, _ = _run(zb, draws, c)
    b, _ = _run(zb, draws, c)
    for da, db in zip(a, b):
        for x, y in zip(da, db):
            for name in ("theta", "m", "v"):
                assert torch.equal(x[name], y[name])


def test_replay_then_post_validated_step(zb):
    """The training step's tail: the replay's OPT markers write each stage's
    gradient state, the optimizer consumes it and refreshes the bf16 weights
    the next F reads.  Per-op parity: the oracle steps from the fp32
    gradients this step consumed."""
    P, m, M, h, f = 2, 3, 136, 72, 200
    blk = zb.make_block(M, h, f)
    stages_d, X0, dY = I.pipeline_draws(P, m, M, h, f, seed=9)
    ops = zb.zb_make_schedule("ZBH1", P, m)
    pl = zb.make_pipeline(P, m, blk)
    ws_bytes, _ = zb.zb_schedule_workspace_size(pl, ops)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stages, masters = [], []
    for st in stages_d:
        W1, W2 = dev_bf16(st.W1), dev_bf16(st.W2)
        stages.append(dict(W1=W1, W2=W2, dW1=empty_f32(h, f), dW2=empty_f32(f, h),
                           grad_stats=torch.zeros(2, dtype=torch.float64, device="cuda")))
        masters.append([(W1.float().contiguous(), torch.zeros_like(W1, dtype=torch.float32),
                         torch.zeros_like(W1, dtype=torch.float32)),
                        (W2.float().contiguous(), torch.zeros_like(W2, dtype=torch.float32),
                         torch.zeros_like(W2, dtype=torch.float32))])
    zb.zb_run_stage_schedule(pl, stages, [dev_bf16(x) for x in X0], [dev_bf16(g) for g in dY],
                             None, None, ops, ws, ws_bytes)
    sync(zb)
    grads = [[f64(s["dW1"]).ravel(), f64(s["dW2"]).ravel()] for s in stages]
    start = [[tuple(f64(a).ravel() for a in t) for t in ms] for ms in masters]
    norms = np.sqrt(np.cumsum([sum(float(np.sum(g ** 2)) for g in gs) for gs in grads]))
    c = float(np.sqrt(norms[0] * norms[1]))
    tensors = []
    for s in range(P):
        for k, (name, gname) in enumerate((("W1", "dW1"), ("W2", "dW2"))):
            th, mm, vv = masters[s][k]
            tensors.append(dict(theta=th, m=mm, v=vv, grad=stages[s][gname], weight_bf16=stages[s][name],
                                stage=s))
    dec = torch.empty(P * 40, dtype=torch.uint8, device="cuda")
    zb.zb_post_validated_adamw(P, [s["grad_stats"] for s in stages], tensors,
                               zb.make_adamw(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay, c, 1), dec)
    sync(zb)
    d = zb.decisions_from_bytes(dec.cpu().numpy().tobytes(), P)
    assert [x["rolled_back"] for x in d] == [1, 0]
    new, _ = oo.post_validated_step(start, grads, 1, HP, c)
    for s in range(P):
        for k, name in enumerate(("W1", "W2")):
            th = f64(masters[s][k][0]).ravel()
            assert rel(th, new[s][k][0]) <= TOL_F32
            assert torch.equal(stages[s][name], masters[s][k][0].to(torch.bfloat16))
    # the refreshed weights feed the next forward (one block, checked against the oracle)
    X = dev_bf16(X0[0])
    H = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
    A, Y = torch.empty_like(H), torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    zb.zb_forward(blk, X, stages[0]["W1"], stages[0]["W2"], None, None, H, A, Y)
    sync(zb)
    _, _, Yr = ob.forward(f64(X), f64(stages[0]["W1"]), f64(stages[0]["W2"]), act="gelu_erf")
    assert rel(f64(Y), Yr) <= 5e-3


def test_decisions_only_without_tensors(zb):
    """No tensors: the call still writes every stage's decision."""
    draws = _draws(seed=50)
    n = _partial_norms(draws)
    c = float(np.sqrt(n[2] * n[3]))
    _, dev = _device_state(zb, draws, lambda s, k: False)
    states = _stage_states(zb, dev)
    dec = torch.empty(4 * 40, dtype=torch.uint8, device="cuda")
    zb.zb_post_validated_adamw(4, states, [], hp_c(zb, c), dec)
    sync(zb)
    d = zb.decisions_from_bytes(dec.cpu().numpy().tobytes(), 4)
    _, report, _ = _oracle(draws, c)
    assert [x["rolled_back"] for x in d] == [int(r["rolled_back"]) for r in report] == [1, 1, 1, 0]
    for x, r in zip(d, report):
        assert abs(x["norm_sq_global"] - n[3] ** 2) <= 1e-6 * n[3] ** 2
