/*
 * zb.h — C ABI of the GB300 split-backward MLP stage library.
 *
 * One pipeline stage's transformer MLP block with its backward split in two,
 * after "Zero Bubble Pipeline Parallelism" (paper-graph-ui summary of arXiv
 * 2401.10241, §2 "The Unexploited Opportunity" and §3.4 "The Backward Pass
 * Decomposition"):
 *   F  (forward):           H = X W1 (+b1);  A = GeLU(H);  Y = A W2 (+b2)
 *   B  (input gradient):    dA = dY W2^T;  dH = dA * GeLU'(H);  dX = dH W1^T
 *   W  (weight gradient):   dW2 += A^T dY;  dW1 += X^T dH  (fp32, accumulated)
 * For a linear map the two halves are Xbar = Ybar W^T and Wbar = X^T Ybar
 * ("Pipeline Schedules: GPipe, 1F1B and Zero Bubble", section "Zero bubble:
 * split the backward pass").  A per-stage F/B/W executor replays 1F1B, ZB-H1
 * and ZB-H2 orderings for all P stages serially on one GPU (summary §3.4
 * "Handcrafted Schedule ZB-H1 / ZB-H2", Table 2): one launch per GEMM on
 * streams and events, or every GEMM of the list in one persistent kernel
 * that orders them on the device (zb_pipeline.executor).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Layout: row-major.  X[M,h], W1[h,f], W2[f,h], H/A/dH[M,f], Y/dY/dX[M,h],
 *    dW1[h,f] and dW2[f,h] in fp32, b1[f], b2[h] in the block dtype, db1[f],
 *    db2[h] in fp32.  Leading dimensions are the row widths (dense tensors).
 *  - Ownership: the caller owns every buffer (device memory unless stated).
 *    The library never allocates device memory; the schedule executor works
 *    inside the caller's workspace.  Pointers are not retained after return.
 *  - Alignment: device pointers must be 16-byte aligned; for bf16 blocks h and
 *    f must be multiples of 8 (16-byte rows for the tensor-memory-access
 *    copies).  Violations return ZB_ERR_ALIGN.  M may be any value >= 1.
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream) and the call returns without
 *    waiting.  A device-side wait that gives up (bounded spin in the GEMM
 *    pipeline) sets a device error word; it is reported as ZB_ERR_TIMEOUT by
 *    zb_sync_status().  Launch failures are reported as ZB_ERR_CUDA at once.
 *    A GEMM that follows another of this library's GEMMs on the same stream
 *    may start its setup before that one ends (programmatic dependent
 *    launch); it touches no memory until every earlier work item of the
 *    stream has completed, so stream order holds as usual.  One exception:
 *    zb_backward_weight's dW1 and dW2 GEMMs run at once (one grouped
 *    launch, or the second launched beside the first), since neither reads
 *    or writes what the other writes; when the caller's buffers overlap
 *    (the library checks) they run one after the other.  Environment:
 *    ZB_GEMM_PDL=0 disables this, ZB_GEMM_SPLIT_K=1 disables split K (see
 *    zb_block.flags), ZB_GEMM_CTA_GROUP=1|2 forces a GEMM tile shape,
 *    ZB_GEMM_L2_HINTS=0 removes the L2 eviction priorities of the GEMMs'
 *    copies, ZB_GEMM_GROUP_W=0 runs the W pass's two GEMMs as two launches
 *    (by default one persistent launch runs both), ZB_GEMM_HANDOFF=0 keeps
 *    the long-K GeLU / GeLU' epilogues on every warp's own rows (by default
 *    the warps that share SM schedulers with the copy and MMA warps hand
 *    their accumulator chunks to the others).  For the persistent executor
 *    (zb_pipeline.executor): ZB_REPLAY_PRIORITY=list|level forces the rule
 *    that orders its tiles, ZB_REPLAY_PARAM_MAPS=0 keeps its tensor maps in
 *    the workspace instead of the launch parameters, ZB_REPLAY_TRACE=1 writes
 *    per-tile timestamps at the end of the workspace (eager replays; the
 *    size query then counts them).  All are read once per process and none
 *    changes a result.
 *  - Errors: every call returns a zb_status; zb_last_error() returns a
 *    thread-local, human-readable message for the last failing call.
 *  - Threads and devices: calls may come from several host threads and for
 *    several devices; each works on the device current on its thread.  Per
 *    device and shared by all threads: kernel configuration (made on first
 *    use), the helper streams of multi-lane replays (two threads replaying at
 *    once on one device interleave on them, in order, so correctly but not
 *    concurrently) and the device error word read by zb_sync_status().  Per
 *    thread and device: the events that order a replay's lanes and time its
 *    ops.  zb_run_stage_schedule_static's arena is one per device.
 *  - Determinism: for fixed shapes the same inputs give the same output bits;
 *    the W pass adds each microbatch's product into the fp32 gradient with a
 *    fixed tile order, so deferred-W and fused-backward replays that visit
 *    microbatches in the same (ascending) order are bit-identical.  Without
 *    split K every output element is the ascending-K sum of its products in
 *    either GEMM tile shape, so the bits do not depend on the shape the
 *    problem's size selects either.
 */
#ifndef ZB_GB300_H
#define ZB_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zb_status {
    ZB_OK = 0,
    ZB_ERR_INVALID_ARG = 1,  /* NULL where a pointer is required, bad enum   */
    ZB_ERR_SHAPE = 2,        /* M, h, f, P or m out of range                 */
    ZB_ERR_ALIGN = 3,        /* pointer not 16-byte aligned, h/f not mult. 8 */
    ZB_ERR_DTYPE = 4,        /* dtype / activation combination unsupported   */
    ZB_ERR_SCHEDULE = 5,     /* op list not a legal replay (dependency,
                                duplicate, missing op, OPT misplaced)        */
    ZB_ERR_W_ORDER = 6,      /* W / BW of a stage not in ascending micro     */
    ZB_ERR_BUDGET = 7,       /* peak live activation bytes > mem limit       */
    ZB_ERR_WORKSPACE = 8,    /* workspace missing or too small               */
    ZB_ERR_CUDA = 9,         /* a CUDA runtime call or launch failed         */
    ZB_ERR_TIMEOUT = 10,     /* a bounded device-side wait gave up           */
    ZB_ERR_UNSUPPORTED = 11  /* no kernel for this device / configuration    */
} zb_status;

typedef enum zb_dtype { ZB_DT_F32 = 0, ZB_DT_BF16 = 1 } zb_dtype;

/* GeLU(x) = x Phi(x) (exact erf form, the default) or its tanh approximation;
 * NONE makes the block the single linear map Y = X W1 (W2, H, A unused). */
typedef enum zb_act { ZB_ACT_NONE = 0, ZB_ACT_GELU_ERF = 1, ZB_ACT_GELU_TANH = 2 } zb_act;

typedef struct zb_block {
    int64_t M;        /* tokens per microbatch (rows of X)                     */
    int64_t h;        /* hidden width                                          */
    int64_t f;        /* ffn width; for ZB_ACT_NONE the output width of W1     */
    int32_t dtype;    /* zb_dtype of X, W, H, A, Y, dY, dH, dX, b              */
    int32_t act;      /* zb_act                                                */
    int32_t has_bias; /* 1: b1/b2 added in F, db1/db2 accumulated in W         */
    int32_t flags;    /* ZB_BLOCK_* bits; others must be 0                     */
} zb_block;

/* zb_block.flags.  Split K: when a bf16-output GEMM of zb_forward or
 * zb_backward_input has too few output tiles to occupy the GPU, those
 * entry points split its K loop over a cluster of 2 or 4 CTAs and add the
 * fp32 partial sums in a fixed order (deterministic: the same inputs give
 * the same bits; the sums differ from the unsplit ones in rounding order
 * only).  The replay (zb_run_stage_schedule) never splits, so its results
 * do not depend on how many streams it spreads over; a caller that compares
 * single passes with a replay bit for bit sets ZB_BLOCK_NO_SPLIT_K. */
#define ZB_BLOCK_NO_SPLIT_K 1

/* Supported combinations: BF16 with any zb_act (tensor-core path, fp32
 * accumulation); F32 with ZB_ACT_NONE (true fp32 FFMA path, no TF32). */

/* ------------------------------------------------------------------------ */
/* Single passes                                                            */
/* ------------------------------------------------------------------------ */

/* F of one microbatch.  Writes H_save and A_save ([M,f], kept for B and W)
 * and Y ([M,h]).  b1/b2 are read only when has_bias (else may be NULL).
 * ZB_ACT_NONE: Y = X W1 ([M,f]); W2, b2, H_save, A_save may be NULL. */
zb_status zb_forward(const zb_block* blk, const void* X, const void* W1,
                     const void* W2, const void* b1, const void* b2,
                     void* H_save, void* A_save, void* Y, void* stream);

/* B of one microbatch (the critical-path input gradient).  Reads dY [M,h],
 * W1, W2 and H_save; writes dH_out ([M,f], kept for W) and dX ([M,h]).
 * dA = dY W2^T stays in fp32 inside the kernel and is never stored.
 * ZB_ACT_NONE: dX = dY W1^T with dY [M,f]; W2, H_save, dH_out unused. */
zb_status zb_backward_input(const zb_block* blk, const void* dY, const void* W1,
                            const void* W2, const void* H_save, void* dH_out,
                            void* dX, void* stream);

/* W of one microbatch (the deferrable weight gradient).
 * accumulate = 0: dW1 = X^T dH, dW2 = A^T dY (db1 = colsum dH, db2 = colsum dY)
 * accumulate = 1: the same products are added to the fp32 buffers.
 * ZB_ACT_NONE: dW1 (+)= X^T dY with dY [M,f]; A_save, dH, dW2 unused. */
zb_status zb_backward_weight(const zb_block* blk, const void* X, const void* A_save,
                             const void* dH, const void* dY, float* dW1, float* dW2,
                             float* db1, float* db2, int accumulate, void* stream);

/* ------------------------------------------------------------------------ */
/* Schedules                                                                */
/* ------------------------------------------------------------------------ */

typedef enum zb_op_kind {
    ZB_OP_F = 0, ZB_OP_B = 1, ZB_OP_W = 2,
    ZB_OP_BW = 3,  /* fused B then W of one (stage, micro): 1F1B's backward  */
    ZB_OP_OPT = 4  /* optimizer marker of a stage: after all its W, no-op    */
} zb_op_kind;

/* Pass id (i, j, c) of the summary's ILP formulation (Appendix G), plus the
 * model chunk for multi-chunk orderings. */
typedef struct zb_op {
    uint8_t kind;    /* zb_op_kind                                        */
    uint8_t chunk;   /* 0 .. chunks-1 (0 for one-chunk orderings)          */
    uint16_t stage;  /* 0 .. P-1: the pipeline stage (device) running it   */
    uint32_t micro;  /* 0 .. m-1 (ignored for OPT)                         */
} zb_op;

typedef enum zb_schedule_kind {
    ZB_SCHED_1F1B = 0, ZB_SCHED_ZBH1 = 1, ZB_SCHED_ZBH2 = 2,
    ZB_SCHED_1F1B_I = 3, /* interleaved 1F1B: v chunks per stage, cyclic    */
    ZB_SCHED_ZBV = 4     /* ZB-V: two chunks per stage, V-shaped            */
} zb_schedule_kind;

/* Model-chunk layouts of multi-chunk pipelines.  With v chunks per stage the
 * model is a chain of L = v P virtual stages k = 0 .. L-1 (forward order):
 *   CYCLIC: chunk c of stage s is k = c P + s (stage i holds chunks i, p+i,
 *           2p+i, ...: "Pipeline Schedules: GPipe, 1F1B and Zero Bubble",
 *           section "Interleaved stages");
 *   V:      v = 2, chunk 0 of stage s is k = s and chunk 1 is k = 2P-1-s
 *           (stage i holds chunks i and 2p-i+1: summary §6 "ZB-V"). */
typedef enum zb_layout { ZB_LAYOUT_CYCLIC = 0, ZB_LAYOUT_V = 1 } zb_layout;

/* How zb_run_stage_schedule runs an op list's GEMMs (zb_pipeline.executor). */
typedef enum zb_executor {
    ZB_EXEC_STREAMS = 0,    /* one launch per GEMM, ordered by streams and
                               events (zb_pipeline.streams)                  */
    ZB_EXEC_PERSISTENT = 1  /* one persistent kernel for every GEMM of the
                               list, ordered on the device                   */
} zb_executor;

/* Generate the one-GPU replay list of a handcrafted ordering for P stages and
 * m microbatches at equal pass times (T_F = T_B = T_W, no communication):
 *   1F1B : warm-up min(P-1-s, m) forwards, then F / fused BW alternation;
 *   ZB-H1: 1F1B's F/B order, W split off; a W runs when the next F/B is not
 *          ready, and before an F when P microbatches are live on the stage;
 *   ZB-H2: warm-up min(2(P-1-s)+1, m) forwards, live limit 2P-1.
 * Ops are ordered by simulated start time, then stage; OPT(s) follows the
 * last op of stage s.  out may be NULL to query the length; otherwise *n_ops
 * holds its capacity on entry and the length on return (ZB_ERR_INVALID_ARG
 * if too small).  Host only, no device work. */
zb_status zb_make_schedule(int32_t kind, int32_t P, int32_t m, zb_op* out, size_t* n_ops);

/* Multi-chunk orderings for P stages, v chunks per stage, m microbatches.
 * A chunk pass takes T/v of the stage's per-microbatch pass time T, so the
 * ideal per-stage time stays m (T_F + T_B + T_W).
 *   ZB_SCHED_1F1B_I (cyclic layout, v >= 2, m a multiple of P): the
 *     interleaved 1F1B the pages cite ("Pipeline Schedules", "Interleaved
 *     stages"; summary §5 "1F1B-I"): stage s runs min(2(P-1-s) + (v-1) P, vm)
 *     warm-up chunk forwards, then alternates a forward with a fused backward
 *     BW, then drains; its i-th forward is chunk (i mod vP) div P of
 *     microbatch (i div vP) P + i mod P, its i-th backward the same
 *     microbatch of chunk v-1-(that chunk).  At equal times its bubble is
 *     (P-1)/(vm+P-1).
 *   ZB_SCHED_ZBV (V layout, v = 2): on a simulated timeline a free stage
 *     takes, among its passes that can start earliest, a W when it holds 2P
 *     live chunk activations, else an F before a B before a W (oldest
 *     microbatch first, then the later virtual stage); an F only while it
 *     holds fewer than 2P (P M_B: summary §6), a chunk-0 forward only while
 *     it holds fewer than 2P-1 or has a W pending; a W from its pending
 *     ones, oldest first.  Peak: exactly P M_B per stage; at equal times no
 *     stage idles between its first and last pass (summary §6: zero bubble
 *     at T_F = T_B = T_W) for any m >= 2P-1; it never deadlocks.
 * Ops carry (stage, chunk); OPT(stage, chunk) follows the last op of each
 * virtual stage; list order = (simulated start, stage).
 * zb_make_interleaved_schedule uses equal times; the simulate variant takes
 * measured ones (T_comm added between chunks on different stages) and fills
 * `result`, whose peak_live fields then count chunk activations (M_B / v
 * each).  out / n_ops as for zb_make_schedule.  Host only.  Errors:
 * ZB_ERR_INVALID_ARG (kind, v, times), ZB_ERR_SHAPE (P, m, or m not a
 * multiple of P for 1F1B-I). */
zb_status zb_make_interleaved_schedule(int32_t kind, int32_t P, int32_t v, int32_t m, zb_op* out,
                                       size_t* n_ops);

/* Pass times for zb_simulate_schedule (any one unit, e.g. ms). */
typedef struct zb_sim_times { double t_f, t_b, t_w, t_comm; } zb_sim_times;

typedef struct zb_sim_result {
    double cost;                     /* max over stages of (end of last pass -
                                        start of first pass), summary Eq. 3     */
    double ideal;                    /* m (T_F + T_B + T_W)                     */
    double bubble_rate;              /* (cost - ideal) / cost, summary §5       */
    uint32_t peak_live_microbatches; /* max over stages: F done, W not done     */
    uint32_t peak_live_stage0;       /* the same on stage 0                     */
} zb_sim_result;

/* Simulate an ordering for P stages, m microbatches and the given pass times
 * with the same rules as zb_make_schedule (T_comm is added to every
 * cross-stage dependency, summary Eqs. 4-5): the projected bubble of a
 * P-GPU pipeline from measured per-pass times.  `out`/`n_ops` may be NULL;
 * when given they receive the op list ordered by simulated start as in
 * zb_make_schedule.  Host only.  ZB_ERR_INVALID_ARG for non-positive or
 * non-finite pass times (T_comm may be 0). */
zb_status zb_simulate_schedule(int32_t kind, int32_t P, int32_t m, const zb_sim_times* times,
                               zb_op* out, size_t* n_ops, zb_sim_result* result);

zb_status zb_simulate_interleaved_schedule(int32_t kind, int32_t P, int32_t v, int32_t m,
                                           const zb_sim_times* times, zb_op* out, size_t* n_ops,
                                           zb_sim_result* result);

/* Heuristic automatic scheduler for measured pass times (summary §3 "The
 * Heuristic Scheduling Algorithm" with "The Memory Model"): memory counted in
 * units of M_B per stage (F +1, B + r - 1, W -r with r = mw_ratio = M_W/M_B),
 * never above mem_limit (ZB-1p: P, ZB-2p: 2P).  Whenever a stage is free it
 * runs its next B if ready; else its next F if ready, within memory, and
 * allowed by two binary hyperparameters (h1: keep adding warm-up forwards
 * even when one would delay the first B; h2: never run more than one F
 * ahead of the next stage); else its oldest W if memory blocks the F, the
 * idle gap is at least T_W, or idling would make the stage's accumulated
 * idle time the largest of all stages; remaining W drain at the end.  All
 * four (h1, h2) are simulated and the smallest Eq. 3 cost is returned
 * (hyper[0..1], may be NULL).  out / n_ops as for zb_simulate_schedule.
 * Host only.  ZB_ERR_BUDGET if mem_limit < 1; ZB_ERR_INVALID_ARG for bad
 * times or mw_ratio outside (0, 1]. */
zb_status zb_auto_schedule(int32_t P, int32_t m, const zb_sim_times* times, double mem_limit,
                           double mw_ratio, zb_op* out, size_t* n_ops, zb_sim_result* result,
                           int32_t* hyper);

typedef struct zb_pipeline {
    int32_t P;                 /* stages (devices of the pipeline)           */
    int32_t m;                 /* microbatches                               */
    zb_block blk;              /* every stage has the same block shape; for
                                  P > 1 the block must map [M,h] to [M,h]    */
    uint64_t mem_limit_bytes;  /* 0 = unlimited; else ZB_ERR_BUDGET when the
                                  peak live activation bytes exceed it       */
    int32_t zero_grads;        /* 1: the first W/BW of each stage overwrites
                                  dW/db (accumulate = 0); 0: always add      */
    int32_t timing;            /* 1: record CUDA events around every op and
                                  GEMM launch, synchronise at the end and
                                  fill the timing fields of zb_run_stats     */
    int32_t streams;           /* 0 or 1: every op on `stream`, in list
                                  order.  n > 1: stage s runs on stream
                                  s mod min(n, P, 8) (the caller's stream and
                                  library-owned streams), ordered by events:
                                  F(s-1,j) -> F(s,j), B(s+1,j) -> B(s,j), and
                                  an arena slot's next writer after its last
                                  reader.  The stages' passes then share the
                                  GPU the way pipeline stages share time; a
                                  stage's W still run in list order on its
                                  stream, so results are bit-identical to the
                                  serial replay.  n >= 2 P (2 P <= 8): each
                                  stage's W and OPT ops also get a stream of
                                  their own, ordered after the stage's B by
                                  events and kept in list order, so a weight
                                  gradient GEMM fills the SMs that an F/B
                                  kernel's last partial wave leaves idle (the
                                  one-stage replay with n = 2).  P > 1 and
                                  n >= 3 P (3 P <= 12): each stage's B and
                                  BW ops also leave its F stream for one of
                                  their own (ordered after F(s,j) by an
                                  event), so a stage's forwards do not queue
                                  behind its backwards.  P = 1 and
                                  n >= 3: the F/B/BW ops of consecutive
                                  microbatches also alternate over n - 1
                                  streams (at most 7).  The call forks from
                                  and joins back into `stream`.
                                  With chunks, lanes follow the stage
                                  (device) of an op.                         */
    int32_t chunks;            /* model chunks per stage: 0 or 1 = one; v > 1
                                  makes the model a chain of L = v P virtual
                                  stages placed by `layout`; every per-stage
                                  array (zb_stage_params, OPT, the arena) is
                                  then per virtual stage, in chain order     */
    int32_t layout;            /* zb_layout (V requires chunks = 2); ignored
                                  for one chunk                              */
    int32_t executor;          /* zb_executor.  ZB_EXEC_PERSISTENT: one
                                  persistent kernel on CTA pairs (every SM)
                                  runs all GEMMs of the list; a GEMM's
                                  tiles start once every earlier GEMM whose
                                  buffers it reads or overwrites (or that
                                  reads what it overwrites) has stored all
                                  of its tiles, tracked by counters in the
                                  workspace.  Same bits as the serial
                                  replay.  bf16 blocks without bias only
                                  (else ZB_ERR_UNSUPPORTED); `streams` is
                                  ignored; OPT statistics follow the kernel
                                  on `stream`; the workspace also holds the
                                  kernel's tables (zb_schedule_workspace_size
                                  counts them), written on `stream` by
                                  small kernels before it.  Kernels of
                                  other streams delay it (it waits for all
                                  of its CTA pairs' SMs); its waits are
                                  bounded like every device wait.  With
                                  timing, total_ms and gemm_ms cover the
                                  kernel and its table upload; the per-op
                                  times are 0; n_gemm_launches counts the
                                  replay kernel and the upload kernels.  */
} zb_pipeline;

typedef struct zb_stage_params {
    const void* W1; const void* W2; const void* b1; const void* b2;
    float* dW1; float* dW2; float* db1; float* db2;
    double* grad_stats;  /* optional device double[2]: at the stage's OPT op,
                            [0] = sum of squares and [1] = count of non-finite
                            values over dW1, dW2 (db1, db2) — the stage's local
                            state for a post-update check of the global
                            gradient norm and NaN/Inf (summary §4 "Staged
                            reduce").  NULL: not computed.               */
} zb_stage_params;

typedef struct zb_run_stats {
    uint64_t workspace_bytes;   /* arena bytes used by this op list            */
    uint64_t peak_live_bytes;   /* ledger peak of live saved activations       */
    uint32_t n_ops;             /* ops replayed (OPT included)                 */
    uint32_t n_gemm_launches;   /* tensor-core / FFMA GEMM launches enqueued
                                   (persistent executor: its replay kernel and
                                   the kernels that write its tables)         */
    double total_ms;            /* timing: first op start to last op end       */
    double kind_ms[4];          /* timing: summed op time per F, B, W, BW      */
    double gemm_ms;             /* timing: summed GEMM kernel time             */
    float* op_ms;               /* caller array of n_ops floats or NULL        */
} zb_run_stats;

/* Validate an op list and size its arena.  Checks: every (stage, micro) has
 * one F and either one B and one W or one BW; producers precede consumers
 * (F(s-1,j) -> F(s,j) -> B(s,j) <- B(s+1,j); B(s,j) -> W(s,j)); W/BW of a
 * stage in ascending micro; OPT at most once per stage, after all its W.
 * Lifetimes (the deferred-W activation store): F saves X, H, A; B frees H and
 * saves dH; W frees X, A, dH and dY; a stage's Y is the next stage's X and a
 * stage's dX the previous stage's dY (pointer hand-off inside the arena).
 * The arena also holds zb_grad_stats scratch for each stage (at its end).
 * With chunks > 1 every op's (stage, chunk) names the virtual stage of the
 * pipeline's layout and the rules apply to the chain of virtual stages
 * (ZB_ERR_SCHEDULE for a chunk >= chunks or a stage >= P; ZB_ERR_INVALID_ARG
 * for a layout other than CYCLIC / V, or V with chunks != 2).
 * Returns the arena size (*bytes) and the ledger peak (*peak_live_bytes,
 * may be NULL).  Host only. */
zb_status zb_schedule_workspace_size(const zb_pipeline* pl, const zb_op* ops, size_t n_ops,
                                     size_t* bytes, size_t* peak_live_bytes);

/* The host plan of a persistent replay (zb_pipeline.executor =
 * ZB_EXEC_PERSISTENT; `pl->executor` itself is ignored here), for inspection
 * and tests; host only, no device is touched.  The op list is validated and
 * its GEMMs recorded as zb_run_stage_schedule would run them, with every
 * stage parameter, input and workspace buffer at a distinct stand-in
 * address (no caller output buffers), for `pairs` CTA pairs (1..128; a
 * GB300 has 76).  GEMMs are numbered in list order: an F op gives H = X W1
 * (with A = GeLU(H)) then Y = A W2, a B op dH then dX, a W op dW2 then dW1,
 * a BW op its B then its W (a single-linear block: one GEMM per pass).
 *   info   counts: GEMMs, 256 x 256 tiles, dependency edges kept after the
 *          transitive reduction, pairs, the simulated makespan in K blocks
 *          of one pair, the priority rule (by_chain 1: longest chain of work
 *          after the GEMM; 0: list order), the longest tile list of a pair.
 *   edges  optional, 2 * (*n_edges) int32: (consumer, producer) GEMM index
 *          pairs of the kept dependencies; *n_edges holds the capacity on
 *          entry and the count on return (ZB_ERR_INVALID_ARG if the
 *          capacity is smaller; n_edges NULL: edges not returned).
 * Errors as zb_run_stage_schedule (list, shapes, bias: ZB_ERR_UNSUPPORTED),
 * and ZB_ERR_UNSUPPORTED if the plan fails its deadlock-freedom check (every
 * tile must start, in the simulation, after every tile of the GEMMs it
 * depends on and after its pair's earlier tiles). */
typedef struct zb_persistent_plan_info {
    uint64_t gemms, tiles, deps, pairs;
    double est_makespan_kblocks;
    int32_t by_chain;
    int32_t reserved;
    uint64_t max_tiles_per_pair;
} zb_persistent_plan_info;
zb_status zb_persistent_plan(const zb_pipeline* pl, const zb_op* ops, size_t n_ops, int32_t pairs,
                             zb_persistent_plan_info* info, int32_t* edges, size_t* n_edges);

/* Replay an op list over P stages on one GPU.
 *   stages[L]       weights and fp32 gradient buffers per (virtual) stage,
 *                   in chain order; L = P, or chunks * P with chunks > 1;
 *   X0[m]           inputs of the first (virtual) stage [M,h] (device
 *                   pointers);
 *   dY_last[m]      output gradients entering the last (virtual) stage
 *                   [M,h];
 *   dX0_out[m]      optional (array or entries may be NULL): the first
 *                   stage's dX;
 *   Y_last_out[m]   optional: the last stage's outputs Y;
 *   workspace       device buffer of >= zb_schedule_workspace_size bytes,
 *                   256-byte aligned;
 *   stats           optional (NULL to skip).
 * Kernels are enqueued on `stream` in list order. */
zb_status zb_run_stage_schedule(const zb_pipeline* pl, const zb_stage_params* stages,
                                const void* const* X0, const void* const* dY_last,
                                void* const* dX0_out, void* const* Y_last_out,
                                const zb_op* ops, size_t n_ops, void* workspace,
                                size_t ws_bytes, zb_run_stats* stats, void* stream);

/* Allocation-free replay.  No counterpart in the paper: this is a library
 * convenience for callers that cannot allocate device memory themselves
 * (a custom operator inside a framework that owns all device memory through
 * its own pool, or a latency-critical loop that must never call cudaMalloc /
 * cudaFree, which can synchronise the whole device).  Same arguments and
 * semantics as zb_run_stage_schedule, minus the workspace: the activation
 * arena is a static device array of ZB_STATIC_ARENA_BYTES (64 MiB).  Under
 * CUDA's default lazy module loading a device holds it from this entry
 * point's first call on that device until the process exits; under eager
 * loading (CUDA_MODULE_LOADING=EAGER) every process that loads the library
 * holds it on each device from that device's context creation, whether or
 * not it ever calls this entry point.  Op lists whose arena
 * (zb_schedule_workspace_size) is larger are
 * rejected with ZB_ERR_WORKSPACE; pl->timing must be 0 and pl->streams at
 * most 1 (ZB_ERR_INVALID_ARG otherwise).  No device memory is allocated by the call.  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current and caches it for the life of the process; make
 * that first call before any stream capture.  The cache is not refreshed
 * after cudaDeviceReset (which ends the context the address belongs to), so
 * do not call this entry point on a device after resetting it in the same
 * process.  All calls share the one array: calls whose work overlaps on the GPU (e.g.
 * on two streams at once) race on it.  The arena needs no clearing (every
 * buffer is written before it is read); the caller's dW/db follow
 * pl->zero_grads exactly as in zb_run_stage_schedule. */
#define ZB_STATIC_ARENA_BYTES (64ull << 20)
zb_status zb_run_stage_schedule_static(const zb_pipeline* pl, const zb_stage_params* stages,
                                       const void* const* X0, const void* const* dY_last,
                                       void* const* dX0_out, void* const* Y_last_out,
                                       const zb_op* ops, size_t n_ops, zb_run_stats* stats,
                                       void* stream);

/* Gradient statistics of fp32 buffers: out[0] = sum of squares, out[1] =
 * number of NaN/Inf values (as a double), over every element of the nbufs
 * device buffers (bufs[i] holds counts[i] floats, 16-byte aligned).  The
 * reduction order is fixed (per-thread fp32 partial sums over fixed ranges,
 * then fp64 sums in a fixed tree), so the same inputs give the same bits.
 * `scratch` is a device buffer of at least zb_grad_stats_scratch_bytes();
 * `out` is device memory (double[2]).  HBM-bound: reads 4 bytes per element. */
size_t zb_grad_stats_scratch_bytes(void);
zb_status zb_grad_stats(const float* const* bufs, const uint64_t* counts, int32_t nbufs,
                        double* out, void* scratch, size_t scratch_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Post-update validation: staged reduce, optimistic AdamW step, rollback    */
/* ------------------------------------------------------------------------ */

/* One fp32 tensor of the optimizer: master weights theta, first and second
 * moments m and v, and its gradient (for example a stage's dW1 after the
 * schedule ran), all `count` floats, device memory, 16-byte aligned.
 * weight_bf16, if not NULL, receives bf16(theta) (round to nearest even)
 * wherever theta is written: the copy the F/B passes read.  `stage` names the
 * pipeline stage whose decision applies.  reserved must be 0. */
typedef struct zb_opt_tensor {
    float* theta;
    float* m;
    float* v;
    const float* grad;
    void* weight_bf16;
    uint64_t count;
    int32_t stage;
    int32_t reserved;
} zb_opt_tensor;

/* AdamW hyperparameters for update number `step` (>= 1):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   theta -= lr wd theta + lr (m / (1-b1^step)) / (sqrt(v / (1-b2^step)) + eps)
 * with g = clip * grad.  max_norm > 0 enables clipping by the global gradient
 * norm (clip = max_norm / ||g|| when ||g|| > max_norm, else 1); 0 disables it.
 * Requires 0 < beta1, beta2 < 1, eps > 0, wd >= 0, lr >= 0, lr*wd < 1. */
typedef struct zb_adamw_params {
    float lr, beta1, beta2, eps, weight_decay, max_norm;
    int32_t step;
    int32_t reserved; /* must be 0 */
} zb_adamw_params;

/* Per-stage record of one post-validated step (device memory, written by
 * zb_post_validated_adamw).  norm_sq_partial is the staged-reduce state the
 * stage stepped with (sum of squares of stages 0..s), norm_sq_global that of
 * all stages; scale_* are the clip factors, skip_* are 1 when a NaN/Inf was
 * seen (no update); rolled_back is 1 when the optimistic decision differed
 * from the global one and the stage inverted and redid its step. */
typedef struct zb_stage_decision {
    double norm_sq_partial;
    double norm_sq_global;
    float scale_used;
    float scale_global;
    int32_t skip_used;
    int32_t skip_global;
    int32_t rolled_back;
    int32_t reserved;
} zb_stage_decision;

/* One optimizer step of P stages with post-update validation, after "Zero
 * Bubble Pipeline Parallelism" (paper-graph-ui summary, §4 "The Optimizer
 * Synchronization Bypass" and "Why rollback is feasible"):
 *   1. staged reduce: stage s's partial state is the sum of the local states
 *      (sum of squares, NaN/Inf count) of stages 0..s; stage P-1's is global;
 *   2. optimistic step: each stage runs AdamW with its partial clip factor,
 *      or leaves its tensors untouched if its partial state saw a NaN/Inf;
 *   3. validation: a stage whose clip factor or skip decision differs from
 *      the global one inverts its step (the algebraic inverse of the update
 *      above, given the same gradient) and applies the global decision.
 * stage_state: host array of P device pointers, each to double[2] = {sum of
 * squares, NaN/Inf count} of that stage's gradients (what zb_grad_stats and
 * the executor's OPT marker write).  tensors: host array of n_tensors
 * descriptors.  decisions: device array of P records (the report).
 * All decisions are made on the device: the call enqueues work on `stream`
 * (three kernels per 64 tensors at most) and never waits.  The result equals
 * the synchronous step (global state first, then one update per stage) up to
 * fp32 rounding of the inverse.  Errors: ZB_ERR_SHAPE (P outside [1, 64],
 * n_tensors < 0), ZB_ERR_INVALID_ARG (NULL, bad stage index or
 * hyperparameters), ZB_ERR_ALIGN; nothing is enqueued on error. */
zb_status zb_post_validated_adamw(int32_t P, const double* const* stage_state,
                                  const zb_opt_tensor* tensors, int32_t n_tensors,
                                  const zb_adamw_params* hp, zb_stage_decision* decisions,
                                  void* stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                   */
/* ------------------------------------------------------------------------ */

/* Synchronise `stream`, then report (and clear) the device error word of the
 * current device: ZB_ERR_TIMEOUT if a bounded device wait gave up,
 * ZB_ERR_CUDA if the stream reported an error, else ZB_OK.  zb_last_error()
 * then gives the word, whose bits name the role whose wait gave up: 1 a TMA
 * producer (or the persistent replay's tile scheduler), 2 an MMA issuer, 4
 * an epilogue warp, 8 the persistent replay's wait for a GEMM it depends on,
 * 1 << 31 zb_selftest_wait_timeout. */
zb_status zb_sync_status(void* stream);

/* Self-test of the device-side timeout path: launches one thread that waits
 * on an mbarrier nothing will ever arrive on, bounded by limit_ns (clamped to
 * [1 ms, 2 s]); when the bound expires it sets the device error word and
 * returns.  The next zb_sync_status() then reports ZB_ERR_TIMEOUT (and clears
 * the word); the context stays usable.  Nothing faults, traps or hangs. */
zb_status zb_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* zb_last_error(void);

/* Library version string, e.g. "zb-gb300 0.1 sm_103a". */
const char* zb_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ZB_GB300_H */
