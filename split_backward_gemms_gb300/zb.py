"""Thin ctypes binding of the C ABI in ``include/zb.h`` (same names).

Argument marshalling only: every pass runs in the CUDA library
``libzb_gb300.so`` built in-tree by ``split_backward_gemms_gb300.build``.
Importing this module loads the library and fails loudly if it is missing;
there is no CPU fallback.

Pointers may be given as torch tensors (their ``data_ptr()``), plain ints or
None.  ``stream`` may be a ``torch.cuda.Stream``, an int handle or None (the
current torch stream when torch's CUDA is initialised, else the legacy
default stream).  A non-OK status raises ``ZBError`` carrying the status and
``zb_last_error()``.
"""

from __future__ import annotations

import ctypes as C
import os

from . import build as _build

# ---------------------------------------------------------------- constants
ZB_OK = 0
ZB_ERR_INVALID_ARG = 1
ZB_ERR_SHAPE = 2
ZB_ERR_ALIGN = 3
ZB_ERR_DTYPE = 4
ZB_ERR_SCHEDULE = 5
ZB_ERR_W_ORDER = 6
ZB_ERR_BUDGET = 7
ZB_ERR_WORKSPACE = 8
ZB_ERR_CUDA = 9
ZB_ERR_TIMEOUT = 10
ZB_ERR_UNSUPPORTED = 11
STATUS_NAMES = {v: k for k, v in list(globals().items()) if k.startswith("ZB_ERR_") or k == "ZB_OK"}

ZB_DT_F32 = 0
ZB_DT_BF16 = 1
ZB_ACT_NONE = 0
ZB_ACT_GELU_ERF = 1
ZB_ACT_GELU_TANH = 2
ZB_BLOCK_NO_SPLIT_K = 1  # zb_block.flags: single passes never split K

ZB_OP_F, ZB_OP_B, ZB_OP_W, ZB_OP_BW, ZB_OP_OPT = range(5)
OP_NAMES = ("F", "B", "W", "BW", "OPT")
ZB_SCHED_1F1B, ZB_SCHED_ZBH1, ZB_SCHED_ZBH2, ZB_SCHED_1F1B_I, ZB_SCHED_ZBV = range(5)
SCHED_IDS = {"1F1B": ZB_SCHED_1F1B, "ZBH1": ZB_SCHED_ZBH1, "ZBH2": ZB_SCHED_ZBH2,
             "1F1B-I": ZB_SCHED_1F1B_I, "ZBV": ZB_SCHED_ZBV}
ZB_LAYOUT_CYCLIC, ZB_LAYOUT_V = range(2)
ZB_EXEC_STREAMS, ZB_EXEC_PERSISTENT = range(2)
EXECUTOR_OF = {"streams": ZB_EXEC_STREAMS, "persistent": ZB_EXEC_PERSISTENT}
LAYOUT_OF = {"1F1B-I": ZB_LAYOUT_CYCLIC, "ZBV": ZB_LAYOUT_V}


# ---------------------------------------------------------------- structs
class zb_block(C.Structure):
    _fields_ = [("M", C.c_int64), ("h", C.c_int64), ("f", C.c_int64), ("dtype", C.c_int32),
                ("act", C.c_int32), ("has_bias", C.c_int32), ("flags", C.c_int32)]


class zb_op(C.Structure):
    _fields_ = [("kind", C.c_uint8), ("chunk", C.c_uint8), ("stage", C.c_uint16), ("micro", C.c_uint32)]


class zb_pipeline(C.Structure):
    _fields_ = [("P", C.c_int32), ("m", C.c_int32), ("blk", zb_block),
                ("mem_limit_bytes", C.c_uint64), ("zero_grads", C.c_int32), ("timing", C.c_int32),
                ("streams", C.c_int32), ("chunks", C.c_int32), ("layout", C.c_int32),
                ("executor", C.c_int32)]


class zb_stage_params(C.Structure):
    _fields_ = [("W1", C.c_void_p), ("W2", C.c_void_p), ("b1", C.c_void_p), ("b2", C.c_void_p),
                ("dW1", C.c_void_p), ("dW2", C.c_void_p), ("db1", C.c_void_p), ("db2", C.c_void_p),
                ("grad_stats", C.c_void_p)]


class zb_run_stats(C.Structure):
    _fields_ = [("workspace_bytes", C.c_uint64), ("peak_live_bytes", C.c_uint64),
                ("n_ops", C.c_uint32), ("n_gemm_launches", C.c_uint32), ("total_ms", C.c_double),
                ("kind_ms", C.c_double * 4), ("gemm_ms", C.c_double), ("op_ms", C.POINTER(C.c_float))]


class zb_sim_times(C.Structure):
    _fields_ = [("t_f", C.c_double), ("t_b", C.c_double), ("t_w", C.c_double), ("t_comm", C.c_double)]


class zb_sim_result(C.Structure):
    _fields_ = [("cost", C.c_double), ("ideal", C.c_double), ("bubble_rate", C.c_double),
                ("peak_live_microbatches", C.c_uint32), ("peak_live_stage0", C.c_uint32)]


class zb_opt_tensor(C.Structure):
    _fields_ = [("theta", C.c_void_p), ("m", C.c_void_p), ("v", C.c_void_p), ("grad", C.c_void_p),
                ("weight_bf16", C.c_void_p), ("count", C.c_uint64), ("stage", C.c_int32),
                ("reserved", C.c_int32)]


class zb_adamw_params(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("max_norm", C.c_float), ("step", C.c_int32),
                ("reserved", C.c_int32)]


class zb_stage_decision(C.Structure):
    _fields_ = [("norm_sq_partial", C.c_double), ("norm_sq_global", C.c_double),
                ("scale_used", C.c_float), ("scale_global", C.c_float), ("skip_used", C.c_int32),
                ("skip_global", C.c_int32), ("rolled_back", C.c_int32), ("reserved", C.c_int32)]


class ZBError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


# ---------------------------------------------------------------- loading
def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run split_backward_gemms_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = C.CDLL(path)
    vp, sz = C.c_void_p, C.c_size_t
    sig = {
        "zb_forward": [C.POINTER(zb_block), vp, vp, vp, vp, vp, vp, vp, vp, vp],
        "zb_backward_input": [C.POINTER(zb_block), vp, vp, vp, vp, vp, vp, vp],
        "zb_backward_weight": [C.POINTER(zb_block), vp, vp, vp, vp, vp, vp, vp, vp, C.c_int, vp],
        "zb_make_schedule": [C.c_int32, C.c_int32, C.c_int32, C.POINTER(zb_op), C.POINTER(sz)],
        "zb_make_interleaved_schedule": [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.POINTER(zb_op),
                                         C.POINTER(sz)],
        "zb_simulate_interleaved_schedule": [C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                             C.POINTER(zb_sim_times), C.POINTER(zb_op), C.POINTER(sz),
                                             C.POINTER(zb_sim_result)],
        "zb_schedule_workspace_size": [C.POINTER(zb_pipeline), C.POINTER(zb_op), sz, C.POINTER(sz),
                                       C.POINTER(sz)],
        "zb_run_stage_schedule": [C.POINTER(zb_pipeline), C.POINTER(zb_stage_params), C.POINTER(vp),
                                  C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), C.POINTER(zb_op), sz,
                                  vp, sz, C.POINTER(zb_run_stats), vp],
        "zb_run_stage_schedule_static": [C.POINTER(zb_pipeline), C.POINTER(zb_stage_params),
                                         C.POINTER(vp), C.POINTER(vp), C.POINTER(vp),
                                         C.POINTER(vp), C.POINTER(zb_op), sz,
                                         C.POINTER(zb_run_stats), vp],
        "zb_simulate_schedule": [C.c_int32, C.c_int32, C.c_int32, C.POINTER(zb_sim_times),
                                 C.POINTER(zb_op), C.POINTER(sz), C.POINTER(zb_sim_result)],
        "zb_selftest_wait_timeout": [C.c_uint64, vp],
        "zb_auto_schedule": [C.c_int32, C.c_int32, C.POINTER(zb_sim_times), C.c_double, C.c_double,
                             C.POINTER(zb_op), C.POINTER(sz), C.POINTER(zb_sim_result),
                             C.POINTER(C.c_int32)],
        "zb_grad_stats": [C.POINTER(vp), C.POINTER(C.c_uint64), C.c_int32, vp, vp, sz, vp],
        "zb_sync_status": [vp],
        "zb_post_validated_adamw": [C.c_int32, C.POINTER(vp), C.POINTER(zb_opt_tensor), C.c_int32,
                                    C.POINTER(zb_adamw_params), vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_int
    lib.zb_last_error.argtypes = []
    lib.zb_last_error.restype = C.c_char_p
    lib.zb_grad_stats_scratch_bytes.argtypes = []
    lib.zb_grad_stats_scratch_bytes.restype = C.c_size_t
    lib.zb_version.argtypes = []
    lib.zb_version.restype = C.c_char_p
    return lib


LIB = _load()


# ---------------------------------------------------------------- helpers
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    raise TypeError(f"cannot take a device pointer of {type(x)!r}")


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream or None
        except Exception:  # pragma: no cover - torch missing
            pass
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _check(st: int, where: str):
    if st != ZB_OK:
        raise ZBError(st, where, zb_last_error())


def make_block(M: int, h: int, f: int, dtype: int = ZB_DT_BF16, act: int = ZB_ACT_GELU_ERF,
               has_bias: bool = False, split_k: bool = True) -> zb_block:
    """split_k=False sets ZB_BLOCK_NO_SPLIT_K (single passes sum K in the
    replay's order)."""
    return zb_block(M, h, f, dtype, act, 1 if has_bias else 0, 0 if split_k else ZB_BLOCK_NO_SPLIT_K)


def ops_array(ops):
    """(kind, stage, micro) or (kind, stage, chunk, micro) tuples (kind as name
    or id) -> ctypes zb_op array."""
    arr = (zb_op * len(ops))()
    for i, op in enumerate(ops):
        k, s, c, j = op if len(op) == 4 else (op[0], op[1], 0, op[2])
        arr[i].kind = OP_NAMES.index(k) if isinstance(k, str) else int(k)
        arr[i].chunk = c
        arr[i].stage = s
        arr[i].micro = j
    return arr


def ops_tuples(arr, n=None, chunks=False):
    """ctypes zb_op array -> (kind_name, stage, micro) tuples, or (kind_name,
    stage, chunk, micro) with chunks=True."""
    n = len(arr) if n is None else n
    if chunks:
        return [(OP_NAMES[arr[i].kind], arr[i].stage, arr[i].chunk, arr[i].micro) for i in range(n)]
    return [(OP_NAMES[arr[i].kind], arr[i].stage, arr[i].micro) for i in range(n)]


# ---------------------------------------------------------------- ABI
def zb_last_error() -> str:
    return LIB.zb_last_error().decode()


def zb_version() -> str:
    return LIB.zb_version().decode()


def zb_forward(blk, X, W1, W2, b1, b2, H_save, A_save, Y, stream=None):
    _check(LIB.zb_forward(C.byref(blk), _ptr(X), _ptr(W1), _ptr(W2), _ptr(b1), _ptr(b2),
                          _ptr(H_save), _ptr(A_save), _ptr(Y), _stream(stream)), "zb_forward")


def zb_backward_input(blk, dY, W1, W2, H_save, dH_out, dX, stream=None):
    _check(LIB.zb_backward_input(C.byref(blk), _ptr(dY), _ptr(W1), _ptr(W2), _ptr(H_save),
                                 _ptr(dH_out), _ptr(dX), _stream(stream)), "zb_backward_input")


def zb_backward_weight(blk, X, A_save, dH, dY, dW1, dW2, db1, db2, accumulate, stream=None):
    _check(LIB.zb_backward_weight(C.byref(blk), _ptr(X), _ptr(A_save), _ptr(dH), _ptr(dY),
                                  _ptr(dW1), _ptr(dW2), _ptr(db1), _ptr(db2),
                                  1 if accumulate else 0, _stream(stream)), "zb_backward_weight")


def zb_make_schedule(kind, P: int, m: int):
    """Generated op list as (kind_name, stage, micro) tuples."""
    kid = SCHED_IDS[kind] if isinstance(kind, str) else int(kind)
    n = C.c_size_t(0)
    _check(LIB.zb_make_schedule(kid, P, m, None, C.byref(n)), "zb_make_schedule")
    arr = (zb_op * n.value)()
    _check(LIB.zb_make_schedule(kid, P, m, arr, C.byref(n)), "zb_make_schedule")
    return ops_tuples(arr, n.value)


def zb_simulate_schedule(kind, P: int, m: int, t_f: float, t_b: float, t_w: float,
                         t_comm: float = 0.0, want_ops: bool = False):
    """Simulated ordering with the given pass times: returns (result, ops or None)."""
    kid = SCHED_IDS[kind] if isinstance(kind, str) else int(kind)
    t = zb_sim_times(t_f, t_b, t_w, t_comm)
    res = zb_sim_result()
    if not want_ops:
        _check(LIB.zb_simulate_schedule(kid, P, m, C.byref(t), None, None, C.byref(res)),
               "zb_simulate_schedule")
        return res, None
    n = C.c_size_t(0)
    _check(LIB.zb_make_schedule(kid, P, m, None, C.byref(n)), "zb_make_schedule")
    arr = (zb_op * n.value)()
    _check(LIB.zb_simulate_schedule(kid, P, m, C.byref(t), arr, C.byref(n), C.byref(res)),
           "zb_simulate_schedule")
    return res, ops_tuples(arr, n.value)


def zb_make_interleaved_schedule(kind, P: int, v: int, m: int):
    """Multi-chunk ordering ("1F1B-I" or "ZBV") as (kind_name, stage, chunk, micro)."""
    kid = SCHED_IDS[kind] if isinstance(kind, str) else int(kind)
    n = C.c_size_t(0)
    _check(LIB.zb_make_interleaved_schedule(kid, P, v, m, None, C.byref(n)), "zb_make_interleaved_schedule")
    arr = (zb_op * n.value)()
    _check(LIB.zb_make_interleaved_schedule(kid, P, v, m, arr, C.byref(n)), "zb_make_interleaved_schedule")
    return ops_tuples(arr, n.value, chunks=True)


def zb_simulate_interleaved_schedule(kind, P: int, v: int, m: int, t_f: float, t_b: float, t_w: float,
                                     t_comm: float = 0.0, want_ops: bool = False):
    """Simulated multi-chunk ordering: (result, ops or None); peaks count chunk activations."""
    kid = SCHED_IDS[kind] if isinstance(kind, str) else int(kind)
    t = zb_sim_times(t_f, t_b, t_w, t_comm)
    res = zb_sim_result()
    if not want_ops:
        _check(LIB.zb_simulate_interleaved_schedule(kid, P, v, m, C.byref(t), None, None, C.byref(res)),
               "zb_simulate_interleaved_schedule")
        return res, None
    n = C.c_size_t(0)
    _check(LIB.zb_make_interleaved_schedule(kid, P, v, m, None, C.byref(n)), "zb_make_interleaved_schedule")
    arr = (zb_op * n.value)()
    _check(LIB.zb_simulate_interleaved_schedule(kid, P, v, m, C.byref(t), arr, C.byref(n), C.byref(res)),
           "zb_simulate_interleaved_schedule")
    return res, ops_tuples(arr, n.value, chunks=True)


def zb_grad_stats_scratch_bytes() -> int:
    return LIB.zb_grad_stats_scratch_bytes()


def zb_grad_stats(bufs, counts, out, scratch, scratch_bytes, stream=None):
    """out (device double[2]) <- [sum of squares, non-finite count] over bufs."""
    arr = (C.c_void_p * len(bufs))(*[_ptr(b) for b in bufs])
    cnt = (C.c_uint64 * len(bufs))(*[int(c) for c in counts])
    _check(LIB.zb_grad_stats(arr, cnt, len(bufs), _ptr(out), _ptr(scratch), scratch_bytes,
                             _stream(stream)), "zb_grad_stats")


def make_adamw(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_norm=0.0,
               step=1) -> zb_adamw_params:
    return zb_adamw_params(lr, beta1, beta2, eps, weight_decay, max_norm, int(step), 0)


def zb_post_validated_adamw(P: int, stage_state, tensors, hp, decisions, stream=None):
    """One post-validated AdamW step of P stages.

    stage_state: P device pointers (tensors) to double[2] gradient states;
    tensors: sequence of dicts with theta, m, v, grad, weight_bf16 (or None),
    stage (count defaults to theta.numel()); decisions: device buffer of P
    zb_stage_decision records (40 bytes each)."""
    st = (C.c_void_p * P)(*[_ptr(x) for x in stage_state])
    arr = (zb_opt_tensor * max(len(tensors), 1))()
    for i, t in enumerate(tensors):
        count = t.get("count")
        if count is None:
            count = t["theta"].numel()
        arr[i] = zb_opt_tensor(_ptr(t["theta"]), _ptr(t["m"]), _ptr(t["v"]), _ptr(t["grad"]),
                               _ptr(t.get("weight_bf16")), int(count), int(t["stage"]), 0)
    _check(LIB.zb_post_validated_adamw(P, st, arr, len(tensors), C.byref(hp), _ptr(decisions),
                                       _stream(stream)), "zb_post_validated_adamw")


def decisions_from_bytes(raw: bytes, P: int):
    """Decode P zb_stage_decision records copied back from the device."""
    recs = (zb_stage_decision * P).from_buffer_copy(raw[:P * C.sizeof(zb_stage_decision)])
    return [{name: getattr(r, name) for name, _ in zb_stage_decision._fields_ if name != "reserved"}
            for r in recs]


def zb_auto_schedule(P: int, m: int, t_f: float, t_b: float, t_w: float, t_comm: float,
                     mem_limit: float, mw_ratio: float = 0.5):
    """Heuristic schedule: returns (result, ops, (h1, h2))."""
    t = zb_sim_times(t_f, t_b, t_w, t_comm)
    res = zb_sim_result()
    n = C.c_size_t(0)
    _check(LIB.zb_make_schedule(SCHED_IDS["ZBH1"], P, m, None, C.byref(n)), "zb_make_schedule")
    arr = (zb_op * n.value)()
    hyper = (C.c_int32 * 2)()
    _check(LIB.zb_auto_schedule(P, m, C.byref(t), mem_limit, mw_ratio, arr, C.byref(n), C.byref(res),
                                hyper), "zb_auto_schedule")
    return res, ops_tuples(arr, n.value), (hyper[0], hyper[1])


def zb_selftest_wait_timeout(limit_ns: int, stream=None):
    _check(LIB.zb_selftest_wait_timeout(int(limit_ns), _stream(stream)), "zb_selftest_wait_timeout")


def make_pipeline(P, m, blk, mem_limit_bytes=0, zero_grads=True, timing=False,
                  streams=1, chunks=1, layout=ZB_LAYOUT_CYCLIC, executor=ZB_EXEC_STREAMS) -> zb_pipeline:
    if isinstance(layout, str):
        layout = LAYOUT_OF[layout]
    if isinstance(executor, str):
        executor = EXECUTOR_OF[executor]
    return zb_pipeline(P, m, blk, mem_limit_bytes, 1 if zero_grads else 0, 1 if timing else 0,
                       int(streams), int(chunks), int(layout), int(executor))


class zb_persistent_plan_info(C.Structure):
    _fields_ = [("gemms", C.c_uint64), ("tiles", C.c_uint64), ("deps", C.c_uint64), ("pairs", C.c_uint64),
                ("est_makespan_kblocks", C.c_double), ("by_chain", C.c_int32), ("reserved", C.c_int32),
                ("max_tiles_per_pair", C.c_uint64)]


def zb_persistent_plan(pl, ops, pairs=76):
    """Host plan of a persistent replay: (info, [(consumer, producer), ...])."""
    arr = ops if isinstance(ops, C.Array) else ops_array(ops)
    info = zb_persistent_plan_info()
    n = C.c_size_t(0)
    _check(LIB.zb_persistent_plan(C.byref(pl), arr, len(arr), int(pairs), C.byref(info), None, C.byref(n)),
           "zb_persistent_plan")
    edges = (C.c_int32 * (2 * max(n.value, 1)))()
    _check(LIB.zb_persistent_plan(C.byref(pl), arr, len(arr), int(pairs), C.byref(info), edges, C.byref(n)),
           "zb_persistent_plan")
    return info, [(edges[2 * k], edges[2 * k + 1]) for k in range(n.value)]


def zb_schedule_workspace_size(pl, ops):
    """Returns (workspace_bytes, peak_live_bytes)."""
    arr = ops if isinstance(ops, C.Array) else ops_array(ops)
    b = C.c_size_t(0)
    pk = C.c_size_t(0)
    _check(LIB.zb_schedule_workspace_size(C.byref(pl), arr, len(arr), C.byref(b), C.byref(pk)),
           "zb_schedule_workspace_size")
    return b.value, pk.value


def _ptr_array(xs):
    if xs is None:
        return None
    arr = (C.c_void_p * len(xs))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def zb_run_stage_schedule(pl, stages, X0, dY_last, dX0_out, Y_last_out, ops, workspace,
                          ws_bytes, stats=None, stream=None):
    """stages: list of dicts/objects with W1, W2, b1, b2, dW1, dW2, db1, db2 pointers."""
    sp = (zb_stage_params * len(stages))()
    for i, st in enumerate(stages):
        get = st.get if isinstance(st, dict) else (lambda k, _s=st: getattr(_s, k, None))
        for k in ("W1", "W2", "b1", "b2", "dW1", "dW2", "db1", "db2", "grad_stats"):
            setattr(sp[i], k, _ptr(get(k)))
    arr = ops if isinstance(ops, C.Array) else ops_array(ops)
    st_ptr = C.byref(stats) if stats is not None else None
    _check(LIB.zb_run_stage_schedule(C.byref(pl), sp, _ptr_array(X0), _ptr_array(dY_last),
                                     _ptr_array(dX0_out), _ptr_array(Y_last_out), arr, len(arr),
                                     _ptr(workspace), ws_bytes, st_ptr, _stream(stream)),
           "zb_run_stage_schedule")


ZB_STATIC_ARENA_BYTES = 64 << 20


def zb_run_stage_schedule_static(pl, stages, X0, dY_last, dX0_out, Y_last_out, ops, stats=None,
                                 stream=None):
    """zb_run_stage_schedule with the arena in the library's static device
    array (no workspace argument; allocates nothing)."""
    sp = (zb_stage_params * len(stages))()
    for i, st in enumerate(stages):
        get = st.get if isinstance(st, dict) else (lambda k, _s=st: getattr(_s, k, None))
        for k in ("W1", "W2", "b1", "b2", "dW1", "dW2", "db1", "db2", "grad_stats"):
            setattr(sp[i], k, _ptr(get(k)))
    arr = ops if isinstance(ops, C.Array) else ops_array(ops)
    st_ptr = C.byref(stats) if stats is not None else None
    _check(LIB.zb_run_stage_schedule_static(C.byref(pl), sp, _ptr_array(X0), _ptr_array(dY_last),
                                            _ptr_array(dX0_out), _ptr_array(Y_last_out), arr,
                                            len(arr), st_ptr, _stream(stream)),
           "zb_run_stage_schedule_static")


def zb_sync_status(stream=None):
    _check(LIB.zb_sync_status(_stream(stream)), "zb_sync_status")
