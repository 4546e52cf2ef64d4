// api.cu — the C ABI: single passes F / B / W of the MLP block and the
// serial one-GPU replay of a pipeline op list (the per-stage F/B/W executor
// with its deferred-W activation arena).
//
// The block and its split backward follow "Zero Bubble Pipeline Parallelism"
// (paper-graph-ui summary of arXiv 2401.10241), §3.4 "The Backward Pass
// Decomposition"; the replay honours the dependencies of §3.4 / Eqs. 4-5:
// F(s,j) after F(s-1,j); B(s,j) after F(s,j) and B(s+1,j); W(s,j) after B(s,j).
#include <cuda_runtime.h>

#include <cstdlib>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "zb_internal.h"

namespace zb {

namespace {
thread_local std::string g_last_error;
}

zb_status fail(zb_status st, const std::string& msg) {
    g_last_error = msg;
    return st;
}

void clear_error() { g_last_error.clear(); }

namespace {

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

zb_status check_block(const zb_block* b) {
    if (!b) return fail(ZB_ERR_INVALID_ARG, "block is NULL");
    if (b->flags & ~ZB_BLOCK_NO_SPLIT_K) return fail(ZB_ERR_INVALID_ARG, "unknown bits in block.flags");
    if (b->M <= 0 || b->h <= 0 || b->f <= 0) return fail(ZB_ERR_SHAPE, "M, h and f must be >= 1");
    if (b->M > (1LL << 30) || b->h > (1LL << 30) || b->f > (1LL << 30))
        return fail(ZB_ERR_SHAPE, "M, h and f must be <= 2^30");
    if (b->act < ZB_ACT_NONE || b->act > ZB_ACT_GELU_TANH) return fail(ZB_ERR_INVALID_ARG, "unknown activation");
    if (b->dtype == ZB_DT_BF16) {
        if (b->h % 8 || b->f % 8) return fail(ZB_ERR_ALIGN, "bf16 blocks need h and f to be multiples of 8");
    } else if (b->dtype == ZB_DT_F32) {
        if (b->act != ZB_ACT_NONE) return fail(ZB_ERR_DTYPE, "fp32 blocks support the single linear map only (act NONE)");
        if (b->has_bias) return fail(ZB_ERR_DTYPE, "fp32 blocks have no bias path");
    } else {
        return fail(ZB_ERR_DTYPE, "unknown dtype");
    }
    return ZB_OK;
}

// Events bracketing kernel launches of one replay (timing mode only).
struct Recorder {
    cudaStream_t st = nullptr;
    bool on = false;
    std::vector<cudaEvent_t>* pool = nullptr;
    size_t used = 0;
    // (before, after, is_gemm) event indices of every launch
    struct Span { size_t a, b; bool gemm; };
    std::vector<Span> spans;
    zb_status mark(size_t* idx) {
        if (used == pool->size()) {
            cudaEvent_t e;
            cudaError_t r = cudaEventCreate(&e);
            if (r != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("cudaEventCreate: ") + cudaGetErrorString(r));
            pool->push_back(e);
        }
        cudaError_t r = cudaEventRecord((*pool)[used], st);
        if (r != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("cudaEventRecord: ") + cudaGetErrorString(r));
        *idx = used++;
        return ZB_OK;
    }
};

// The current device's ordinal, in [0, 64).  Events belong to the device
// that was current when they were created, so the pools below keep one list
// per device.
zb_status current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (*dev < 0 || *dev >= 64) return fail(ZB_ERR_CUDA, "device ordinal out of range");
    return ZB_OK;
}

// Timing events of this thread on the current device.
zb_status event_pool(std::vector<cudaEvent_t>** out) {
    static thread_local std::vector<cudaEvent_t> pools[64];
    int dev = 0;
    zb_status s = current_device(&dev);
    if (s != ZB_OK) return s;
    *out = &pools[dev];
    return ZB_OK;
}

// Events without timing that order ops across streams (one per op), this
// thread's on the current device.
zb_status sync_events(size_t n, std::vector<cudaEvent_t>** out) {
    static thread_local std::vector<cudaEvent_t> pools[64];
    int dev = 0;
    zb_status s = current_device(&dev);
    if (s != ZB_OK) return s;
    std::vector<cudaEvent_t>& pool = pools[dev];
    while (pool.size() < n) {
        cudaEvent_t e;
        cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
        if (r != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("cudaEventCreate: ") + cudaGetErrorString(r));
        pool.push_back(e);
    }
    *out = &pool;
    return ZB_OK;
}

// Library-owned non-blocking streams of the current device (created once).
zb_status helper_streams(int count, std::vector<cudaStream_t>* out) {
    static std::mutex mu;
    static std::vector<cudaStream_t> per_dev[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(ZB_ERR_CUDA, "cudaGetDevice failed");
    std::lock_guard<std::mutex> lk(mu);
    auto& v = per_dev[dev];
    while (static_cast<int>(v.size()) < count) {
        cudaStream_t st;
        e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
        if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("cudaStreamCreate: ") + cudaGetErrorString(e));
        v.push_back(st);
    }
    out->assign(v.begin(), v.begin() + count);
    return ZB_OK;
}

template <typename F>
zb_status timed(Recorder* rec, bool gemm, F&& launch) {
    if (!rec || !rec->on) return launch();
    size_t a = 0, b = 0;
    zb_status s = rec->mark(&a);
    if (s != ZB_OK) return s;
    s = launch();
    if (s != ZB_OK) return s;
    s = rec->mark(&b);
    if (s != ZB_OK) return s;
    rec->spans.push_back({a, b, gemm});
    return ZB_OK;
}

thread_local int* g_gemm_counter = nullptr;  // GEMM launch count of the running replay
// A replay is running: its GEMMs never split K, so its results do not depend
// on the number of lanes.  With several lanes an under-filled GEMM's idle
// SMs are taken by other lanes' GEMMs anyway, and splitting would only add
// the partial-tile exchange (measured on the 4-stage h=1024 replay on four
// streams: 963 TF/s unsplit, 898 split).
thread_local bool g_in_replay = false;
// The running replay's GEMMs may launch as programmatic dependents: one lane,
// or one F/B lane beside the W lane(s) of a one-stage replay (measured: the
// h=6144 and h=4096 one-stage steps +0.3 % and +1.0 %).  Not with
// stage-parallel lanes, whose small GEMMs share the SMs: a GEMM's waiting
// CTAs keep other stages' GEMMs off free SMs there (the P=4, h=1024 pipeline
// on four streams: 956 -> 938 TF/s).
thread_local bool g_pdl_lanes = true;
// A persistent replay is being planned: GEMMs are recorded, not launched.
thread_local std::vector<GemmBf16>* g_record = nullptr;
// zb_persistent_plan: stop after the host plan (no device work at all).
struct PlanOnly {
    int pairs = 0;
    ReplayPlan plan;
};
thread_local PlanOnly* g_plan_only = nullptr;

zb_status run_gemm(const GemmBf16& g, void* stream, Recorder* rec) {
    if (g_record) {
        g_record->push_back(g);
        g_record->back().second = nullptr;
        return ZB_OK;
    }
    if (g_gemm_counter) ++*g_gemm_counter;
    GemmBf16 h = g;
    // programmatic dependent launch where the lanes allow it, and with no
    // events between launches (per-op timing)
    // ZB_GEMM_PDL=0 turns it off, =1 on inside every lane (else the rule above)
    static const int pdl_env = [] {
        const char* v = std::getenv("ZB_GEMM_PDL");
        return v && (v[0] == '0' || v[0] == '1') ? v[0] - '0' : -1;
    }();
    const bool lanes_ok = pdl_env < 0 ? g_pdl_lanes : pdl_env == 1;
    h.allow_pdl = lanes_ok && !(rec && rec->on);
    return timed(rec, true, [&] { return gemm_bf16_tc(h, stream); });
}

// Byte ranges [a, a + na) and [b, b + nb) do not overlap.
bool disjoint(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa + na <= pb || pb + nb <= pa;
}

int split_allowed(const zb_block& b) { return !g_in_replay && !(b.flags & ZB_BLOCK_NO_SPLIT_K); }

zb_status run_gemm32(const GemmF32& g, void* stream, Recorder* rec) {
    if (g_record) return fail(ZB_ERR_UNSUPPORTED, "fp32 GEMM in a persistent replay");
    if (g_gemm_counter) ++*g_gemm_counter;
    return timed(rec, true, [&] { return gemm_f32_simt(g, stream); });
}

zb_status forward_impl(const zb_block& b, const void* X, const void* W1, const void* W2, const void* b1,
                       const void* b2, void* H, void* A, void* Y, void* stream, Recorder* rec) {
    if (b.dtype == ZB_DT_F32) {
        GemmF32 g;
        g.Mg = b.M; g.Ng = b.f; g.Kg = b.h;
        g.A = static_cast<const float*>(X); g.sam = b.h; g.sak = 1;
        g.B = static_cast<const float*>(W1); g.sbk = b.f; g.sbn = 1;
        g.C = static_cast<float*>(Y); g.ldc = b.f;
        return run_gemm32(g, stream, rec);
    }
    if (b.act == ZB_ACT_NONE) {
        GemmBf16 g;
        g.Mg = b.M; g.Ng = b.f; g.Kg = b.h;
        g.A = X; g.lda = b.h; g.a_mn = 0;
        g.B = W1; g.ldb = b.f; g.b_mn = 1;
        g.epi = EPI_STORE_BF16; g.out0 = Y; g.ld0 = b.f;
        g.bias = b.has_bias ? b1 : nullptr; g.allow_split = split_allowed(b);
        return run_gemm(g, stream, rec);
    }
    GemmBf16 g1;  // H = X W1 (+b1), A = GeLU(H)
    g1.Mg = b.M; g1.Ng = b.f; g1.Kg = b.h;
    g1.A = X; g1.lda = b.h; g1.a_mn = 0;
    g1.B = W1; g1.ldb = b.f; g1.b_mn = 1;
    g1.epi = EPI_GELU_DUAL; g1.out0 = H; g1.ld0 = b.f; g1.out1 = A; g1.ld1 = b.f;
    g1.bias = b.has_bias ? b1 : nullptr; g1.act = b.act; g1.allow_split = split_allowed(b);
    zb_status s = run_gemm(g1, stream, rec);
    if (s != ZB_OK) return s;
    GemmBf16 g2;  // Y = A W2 (+b2)
    g2.Mg = b.M; g2.Ng = b.h; g2.Kg = b.f;
    g2.A = A; g2.lda = b.f; g2.a_mn = 0;
    g2.B = W2; g2.ldb = b.h; g2.b_mn = 1;
    g2.epi = EPI_STORE_BF16; g2.out0 = Y; g2.ld0 = b.h;
    g2.bias = b.has_bias ? b2 : nullptr; g2.allow_split = split_allowed(b);
    return run_gemm(g2, stream, rec);
}

zb_status backward_input_impl(const zb_block& b, const void* dY, const void* W1, const void* W2,
                              const void* H, void* dH, void* dX, void* stream, Recorder* rec) {
    if (b.dtype == ZB_DT_F32) {
        GemmF32 g;  // dX = dY W1^T
        g.Mg = b.M; g.Ng = b.h; g.Kg = b.f;
        g.A = static_cast<const float*>(dY); g.sam = b.f; g.sak = 1;
        g.B = static_cast<const float*>(W1); g.sbk = 1; g.sbn = b.f;
        g.C = static_cast<float*>(dX); g.ldc = b.h;
        return run_gemm32(g, stream, rec);
    }
    if (b.act == ZB_ACT_NONE) {
        GemmBf16 g;
        g.Mg = b.M; g.Ng = b.h; g.Kg = b.f;
        g.A = dY; g.lda = b.f; g.a_mn = 0;
        g.B = W1; g.ldb = b.f; g.b_mn = 0;
        g.epi = EPI_STORE_BF16; g.out0 = dX; g.ld0 = b.h; g.allow_split = split_allowed(b);
        return run_gemm(g, stream, rec);
    }
    GemmBf16 g3;  // dH = (dY W2^T) * GeLU'(H); dA stays in fp32 in TMEM
    g3.Mg = b.M; g3.Ng = b.f; g3.Kg = b.h;
    g3.A = dY; g3.lda = b.h; g3.a_mn = 0;
    g3.B = W2; g3.ldb = b.h; g3.b_mn = 0;
    g3.epi = EPI_GELU_BWD; g3.out0 = dH; g3.ld0 = b.f; g3.aux = H; g3.ldaux = b.f; g3.act = b.act;
    g3.allow_split = split_allowed(b);
    zb_status s = run_gemm(g3, stream, rec);
    if (s != ZB_OK) return s;
    GemmBf16 g4;  // dX = dH W1^T
    g4.Mg = b.M; g4.Ng = b.h; g4.Kg = b.f;
    g4.A = dH; g4.lda = b.f; g4.a_mn = 0;
    g4.B = W1; g4.ldb = b.f; g4.b_mn = 0;
    g4.epi = EPI_STORE_BF16; g4.out0 = dX; g4.ld0 = b.h; g4.allow_split = split_allowed(b);
    return run_gemm(g4, stream, rec);
}

zb_status backward_weight_impl(const zb_block& b, const void* X, const void* A, const void* dH,
                               const void* dY, float* dW1, float* dW2, float* db1, float* db2,
                               int accumulate, void* stream, Recorder* rec) {
    if (b.dtype == ZB_DT_F32) {
        GemmF32 g;  // dW1 (+)= X^T dY
        g.Mg = b.h; g.Ng = b.f; g.Kg = b.M;
        g.A = static_cast<const float*>(X); g.sam = 1; g.sak = b.h;
        g.B = static_cast<const float*>(dY); g.sbk = b.f; g.sbn = 1;
        g.C = dW1; g.ldc = b.f; g.accumulate = accumulate;
        return run_gemm32(g, stream, rec);
    }
    if (b.act == ZB_ACT_NONE) {
        GemmBf16 g;
        g.Mg = b.h; g.Ng = b.f; g.Kg = b.M;
        g.A = X; g.lda = b.h; g.a_mn = 1;
        g.B = dY; g.ldb = b.f; g.b_mn = 1;
        g.epi = EPI_F32; g.out0 = dW1; g.ld0 = b.f; g.accumulate = accumulate;
        zb_status s = run_gemm(g, stream, rec);
        if (s != ZB_OK || !b.has_bias) return s;
        return timed(rec, false, [&] { return colsum_bf16(dY, b.M, b.f, b.f, db1, accumulate, stream); });
    }
    GemmBf16 g5;  // dW2 (+)= A^T dY
    g5.Mg = b.f; g5.Ng = b.h; g5.Kg = b.M;
    g5.A = A; g5.lda = b.f; g5.a_mn = 1;
    g5.B = dY; g5.ldb = b.h; g5.b_mn = 1;
    g5.epi = EPI_F32; g5.out0 = dW2; g5.ld0 = b.h; g5.accumulate = accumulate;
    GemmBf16 g6;  // dW1 (+)= X^T dH
    g6.Mg = b.h; g6.Ng = b.f; g6.Kg = b.M;
    g6.A = X; g6.lda = b.h; g6.a_mn = 1;
    g6.B = dH; g6.ldb = b.f; g6.b_mn = 1;
    g6.epi = EPI_F32; g6.out0 = dW1; g6.ld0 = b.f; g6.accumulate = accumulate;
    // the two GEMMs share no output and neither reads the other's (unless
    // the caller's buffers overlap), so they may run at once
    bool independent;
    {
        const size_t hf4 = static_cast<size_t>(b.h) * b.f * 4;
        const size_t act_f = static_cast<size_t>(b.M) * b.f * 2, act_h = static_cast<size_t>(b.M) * b.h * 2;
        independent = disjoint(dW1, hf4, dW2, hf4) && disjoint(dW1, hf4, A, act_f) &&
                      disjoint(dW1, hf4, dY, act_h) && disjoint(dW2, hf4, X, act_h) &&
                      disjoint(dW2, hf4, dH, act_f);
    }
    // one grouped launch for both (one setup, one tail; the second GEMM's
    // tiles follow the first's in the same persistent kernel) when both take
    // CTA pairs; else the second launches beside the first.
    // ZB_GEMM_GROUP_W=0 in the environment keeps two launches.
    static const bool group_w = [] {
        const char* v = std::getenv("ZB_GEMM_GROUP_W");
        return !(v && v[0] == '0');
    }();
    zb_status s;
    if (group_w && !g_record && independent && gemm_bf16_cta_group(g5) == 2 && gemm_bf16_cta_group(g6) == 2) {
        g5.second = &g6;
        s = run_gemm(g5, stream, rec);
    } else {
        s = run_gemm(g5, stream, rec);
        if (s != ZB_OK) return s;
        g6.independent_of_prev = independent;
        s = run_gemm(g6, stream, rec);
    }
    if (s != ZB_OK || !b.has_bias) return s;
    s = timed(rec, false, [&] { return colsum_bf16(dH, b.M, b.f, b.f, db1, accumulate, stream); });
    if (s != ZB_OK) return s;
    return timed(rec, false, [&] { return colsum_bf16(dY, b.M, b.h, b.h, db2, accumulate, stream); });
}

}  // namespace
}  // namespace zb

using namespace zb;

extern "C" const char* zb_last_error(void) { return g_last_error.c_str(); }

extern "C" zb_status zb_persistent_plan(const zb_pipeline* pl, const zb_op* ops, size_t n_ops, int32_t pairs,
                                        zb_persistent_plan_info* info, int32_t* edges, size_t* n_edges) {
    if (!pl || !info) return fail(ZB_ERR_INVALID_ARG, "pipeline or info is NULL");
    if (pairs < 1 || pairs > 128) return fail(ZB_ERR_INVALID_ARG, "pairs must be in [1, 128]");
    zb_pipeline p = *pl;
    p.executor = ZB_EXEC_PERSISTENT;
    p.timing = 0;
    const int L = p.P * (p.chunks > 1 ? p.chunks : 1);
    if (p.P < 1 || p.m < 1 || L > 4096 || p.m > (1 << 20)) return fail(ZB_ERR_SHAPE, "P and m out of range");
    // distinct, aligned stand-in addresses for every buffer of the call (never
    // dereferenced): 2^36 bytes apart, far above the workspace's
    const uintptr_t unit = uintptr_t(1) << 36;
    uintptr_t next = uintptr_t(1) << 44;
    auto fake = [&]() { const uintptr_t a = next; next += unit; return reinterpret_cast<void*>(a); };
    std::vector<zb_stage_params> st(L);
    for (auto& sp : st) {
        sp.W1 = fake(); sp.W2 = fake(); sp.b1 = fake(); sp.b2 = fake();
        sp.dW1 = static_cast<float*>(fake()); sp.dW2 = static_cast<float*>(fake());
        sp.db1 = static_cast<float*>(fake()); sp.db2 = static_cast<float*>(fake());
        sp.grad_stats = nullptr;
    }
    std::vector<const void*> x0(p.m), dy(p.m);
    for (int j = 0; j < p.m; ++j) {
        x0[j] = fake();
        dy[j] = fake();
    }
    PlanOnly po;
    po.pairs = pairs;
    g_plan_only = &po;
    zb_status s = zb_run_stage_schedule(&p, st.data(), x0.data(), dy.data(), nullptr, nullptr, ops, n_ops,
                                        reinterpret_cast<void*>(uintptr_t(1) << 40), SIZE_MAX / 4, nullptr, nullptr);
    g_plan_only = nullptr;
    if (s != ZB_OK) return s;
    const ReplayPlan& pp = po.plan;
    info->gemms = pp.tiles.size();
    info->tiles = pp.ntiles;
    info->deps = pp.ndeps;
    info->pairs = static_cast<uint64_t>(pairs);
    info->est_makespan_kblocks = static_cast<double>(pp.makespan) / 16.0;
    info->by_chain = pp.by_level ? 1 : 0;
    info->max_tiles_per_pair = 0;
    for (const auto& l : pp.lists) info->max_tiles_per_pair = std::max<uint64_t>(info->max_tiles_per_pair, l.size());
    if (n_edges) {
        const size_t cap = *n_edges;
        size_t k = 0;
        for (size_t j = 0; j < pp.deps.size(); ++j)
            for (int d : pp.deps[j]) {
                if (edges && k < cap) {
                    edges[2 * k] = static_cast<int32_t>(j);
                    edges[2 * k + 1] = d;
                }
                ++k;
            }
        *n_edges = k;
        if (edges && k > cap) return fail(ZB_ERR_INVALID_ARG, "edges: capacity too small");
    }
    clear_error();
    return ZB_OK;
}

extern "C" const char* zb_version(void) { return "zb-gb300 0.1 sm_103a"; }

extern "C" zb_status zb_forward(const zb_block* blk, const void* X, const void* W1, const void* W2,
                                const void* b1, const void* b2, void* H_save, void* A_save, void* Y,
                                void* stream) {
    zb_status s = check_block(blk);
    if (s != ZB_OK) return s;
    const bool mlp = blk->act != ZB_ACT_NONE;
    if (!X || !W1 || !Y || (mlp && (!W2 || !H_save || !A_save)))
        return fail(ZB_ERR_INVALID_ARG, "zb_forward: required pointer is NULL");
    if (blk->has_bias && (!b1 || (mlp && !b2))) return fail(ZB_ERR_INVALID_ARG, "zb_forward: bias pointer is NULL");
    if (misaligned(X) || misaligned(W1) || misaligned(W2) || misaligned(Y) || misaligned(H_save) ||
        misaligned(A_save) || misaligned(b1) || misaligned(b2))
        return fail(ZB_ERR_ALIGN, "zb_forward: pointers must be 16-byte aligned");
    s = forward_impl(*blk, X, W1, W2, b1, b2, H_save, A_save, Y, stream, nullptr);
    if (s == ZB_OK) clear_error();
    return s;
}

extern "C" zb_status zb_backward_input(const zb_block* blk, const void* dY, const void* W1, const void* W2,
                                       const void* H_save, void* dH_out, void* dX, void* stream) {
    zb_status s = check_block(blk);
    if (s != ZB_OK) return s;
    const bool mlp = blk->act != ZB_ACT_NONE;
    if (!dY || !W1 || !dX || (mlp && (!W2 || !H_save || !dH_out)))
        return fail(ZB_ERR_INVALID_ARG, "zb_backward_input: required pointer is NULL");
    if (misaligned(dY) || misaligned(W1) || misaligned(W2) || misaligned(H_save) || misaligned(dH_out) ||
        misaligned(dX))
        return fail(ZB_ERR_ALIGN, "zb_backward_input: pointers must be 16-byte aligned");
    s = backward_input_impl(*blk, dY, W1, W2, H_save, dH_out, dX, stream, nullptr);
    if (s == ZB_OK) clear_error();
    return s;
}

extern "C" zb_status zb_backward_weight(const zb_block* blk, const void* X, const void* A_save, const void* dH,
                                        const void* dY, float* dW1, float* dW2, float* db1, float* db2,
                                        int accumulate, void* stream) {
    zb_status s = check_block(blk);
    if (s != ZB_OK) return s;
    const bool mlp = blk->act != ZB_ACT_NONE;
    if (!X || !dY || !dW1 || (mlp && (!A_save || !dH || !dW2)))
        return fail(ZB_ERR_INVALID_ARG, "zb_backward_weight: required pointer is NULL");
    if (blk->has_bias && (!db1 || (mlp && !db2)))
        return fail(ZB_ERR_INVALID_ARG, "zb_backward_weight: bias-gradient pointer is NULL");
    if (misaligned(X) || misaligned(A_save) || misaligned(dH) || misaligned(dY) || misaligned(dW1) ||
        misaligned(dW2) || misaligned(db1) || misaligned(db2))
        return fail(ZB_ERR_ALIGN, "zb_backward_weight: pointers must be 16-byte aligned");
    s = backward_weight_impl(*blk, X, A_save, dH, dY, dW1, dW2, db1, db2, accumulate ? 1 : 0, stream, nullptr);
    if (s == ZB_OK) clear_error();
    return s;
}

extern "C" zb_status zb_run_stage_schedule(const zb_pipeline* pl, const zb_stage_params* stages,
                                           const void* const* X0, const void* const* dY_last,
                                           void* const* dX0_out, void* const* Y_last_out, const zb_op* ops,
                                           size_t n_ops, void* workspace, size_t ws_bytes, zb_run_stats* stats,
                                           void* stream) {
    if (!pl || !stages || !X0 || !dY_last) return fail(ZB_ERR_INVALID_ARG, "pipeline, stages, X0 or dY_last is NULL");
    const zb_block& b = pl->blk;
    zb_status s = check_block(&b);
    if (s != ZB_OK) return s;
    const int m = pl->m;
    if (pl->P < 1 || m < 1) return fail(ZB_ERR_SHAPE, "P and m must be >= 1");
    if (pl->streams < 0) return fail(ZB_ERR_INVALID_ARG, "pipeline.streams < 0");
    // multi-chunk lists run on the chain of virtual stages; dev[i] is the
    // stage (device) of op i, which picks its stream
    std::vector<zb_op> vop;
    std::vector<int> dev;
    int P = 0;
    s = virtualize_ops(*pl, ops, n_ops, &vop, &dev, &P);
    if (s != ZB_OK) return s;
    zb_pipeline chain = *pl;
    chain.P = P;
    chain.chunks = 1;
    if (P > 1 && b.act == ZB_ACT_NONE && b.f != b.h)
        return fail(ZB_ERR_SHAPE, "a multi-stage single-linear pipeline needs f == h");
    const bool mlp = b.act != ZB_ACT_NONE;
    for (int st = 0; st < P; ++st) {
        const zb_stage_params& p = stages[st];
        if (!p.W1 || !p.dW1 || (mlp && (!p.W2 || !p.dW2)))
            return fail(ZB_ERR_INVALID_ARG, "stage " + std::to_string(st) + ": weight or gradient pointer is NULL");
        if (b.has_bias && (!p.b1 || !p.db1 || (mlp && (!p.b2 || !p.db2))))
            return fail(ZB_ERR_INVALID_ARG, "stage " + std::to_string(st) + ": bias pointer is NULL");
        if (misaligned(p.W1) || misaligned(p.W2) || misaligned(p.b1) || misaligned(p.b2) || misaligned(p.dW1) ||
            misaligned(p.dW2) || misaligned(p.db1) || misaligned(p.db2) || misaligned(p.grad_stats))
            return fail(ZB_ERR_ALIGN, "stage " + std::to_string(st) + ": pointers must be 16-byte aligned");
    }
    bool has_y = Y_last_out != nullptr, has_dx = dX0_out != nullptr;
    for (int j = 0; j < m; ++j) {
        if (!X0[j] || !dY_last[j]) return fail(ZB_ERR_INVALID_ARG, "X0 / dY_last entry is NULL");
        if (misaligned(X0[j]) || misaligned(dY_last[j])) return fail(ZB_ERR_ALIGN, "X0 / dY_last must be 16-byte aligned");
        if (has_y && !Y_last_out[j]) has_y = false;
        if (has_dx && !dX0_out[j]) has_dx = false;
        if (Y_last_out && misaligned(Y_last_out[j])) return fail(ZB_ERR_ALIGN, "Y_last_out must be 16-byte aligned");
        if (dX0_out && misaligned(dX0_out[j])) return fail(ZB_ERR_ALIGN, "dX0_out must be 16-byte aligned");
    }
    OpCheck c = validate_ops(vop.data(), n_ops, P, m);
    if (c.st != ZB_OK) return fail(c.st, c.msg);
    ArenaPlan plan;
    s = plan_arena(chain, vop.data(), n_ops, has_y, has_dx, &plan);
    if (s != ZB_OK) return s;
    if (plan.workspace_bytes > 0) {
        if (!workspace) return fail(ZB_ERR_WORKSPACE, "workspace is NULL");
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(ZB_ERR_ALIGN, "workspace must be 256-byte aligned");
        if (ws_bytes < plan.workspace_bytes)
            return fail(ZB_ERR_WORKSPACE, "workspace too small: need " + std::to_string(plan.workspace_bytes) + " bytes");
    }
    char* ws = static_cast<char*>(workspace);
    auto row_ptr = [&](int slot) -> void* { return ws + static_cast<size_t>(slot) * plan.row_bytes; };
    auto ffn_ptr = [&](int slot) -> void* {
        return ws + static_cast<size_t>(plan.row_slots) * plan.row_bytes + static_cast<size_t>(slot) * plan.ffn_bytes;
    };

    // one op's passes on `lane` (recorded instead of launched while a
    // persistent replay is being planned)
    std::vector<char> w_started(P, 0);
    auto run_op = [&](size_t i, cudaStream_t lane, Recorder* recp) -> zb_status {
        zb_status s = ZB_OK;
        const zb_op& o = vop[i];
        const int st = o.stage, j = static_cast<int>(o.micro);
        const zb_stage_params& p = stages[st];
        void* lane_v = static_cast<void*>(lane);
        const void* X = st == 0 ? X0[j] : row_ptr(plan.at(st, j, BUF_X));
        const void* dY = st == P - 1 ? dY_last[j] : row_ptr(plan.at(st, j, BUF_DY));
        void* H = mlp ? ffn_ptr(plan.at(st, j, BUF_H)) : nullptr;
        void* A = mlp ? ffn_ptr(plan.at(st, j, BUF_A)) : nullptr;
        void* dH = mlp ? ffn_ptr(plan.at(st, j, BUF_DH)) : nullptr;
        auto run_b = [&]() -> zb_status {
            void* dX;
            if (st > 0) dX = row_ptr(plan.at(st - 1, j, BUF_DY));
            else dX = has_dx ? dX0_out[j] : row_ptr(plan.tmp_slot[i]);
            return backward_input_impl(b, dY, p.W1, p.W2, H, dH, dX, lane_v, recp);
        };
        auto run_w = [&]() -> zb_status {
            const int acc = (pl->zero_grads && !w_started[st]) ? 0 : 1;
            w_started[st] = 1;
            const void* Xw = X;
            return backward_weight_impl(b, Xw, A, dH, dY, p.dW1, p.dW2, p.db1, p.db2, acc, lane_v, recp);
        };
        switch (o.kind) {
            case ZB_OP_F: {
                void* Y;
                if (st < P - 1) Y = row_ptr(plan.at(st + 1, j, BUF_X));
                else Y = has_y ? Y_last_out[j] : row_ptr(plan.tmp_slot[i]);
                s = forward_impl(b, X, p.W1, p.W2, p.b1, p.b2, H, A, Y, lane_v, recp);
                break;
            }
            case ZB_OP_B: s = run_b(); break;
            case ZB_OP_W: s = run_w(); break;
            case ZB_OP_BW:
                s = run_b();
                if (s == ZB_OK) s = run_w();
                break;
            case ZB_OP_OPT:
                if (p.grad_stats) {
                    const float* bufs[4];
                    uint64_t counts[4];
                    int nb = 0;
                    const uint64_t hf = static_cast<uint64_t>(b.h) * static_cast<uint64_t>(b.f);
                    bufs[nb] = p.dW1; counts[nb++] = hf;
                    if (mlp) { bufs[nb] = p.dW2; counts[nb++] = hf; }
                    if (b.has_bias) {
                        bufs[nb] = p.db1; counts[nb++] = static_cast<uint64_t>(b.f);
                        if (mlp) { bufs[nb] = p.db2; counts[nb++] = static_cast<uint64_t>(b.h); }
                    }
                    void* scratch = ws + plan.stats_offset + static_cast<size_t>(st) * plan.stats_bytes;
                    s = timed(recp, false, [&] {
                        return zb_grad_stats(bufs, counts, nb, p.grad_stats, scratch, plan.stats_bytes, lane_v);
                    });
                }
                break;
            default: break;
        }
        return s;
    };


    if (pl->executor == ZB_EXEC_PERSISTENT) {
        // Every GEMM of the list in one persistent kernel on `stream`
        // (replay_tc.cu), then the OPT ops' statistics in list order (an OPT
        // follows all of its stage's W, so it reads the final gradients).
        if (b.dtype != ZB_DT_BF16 || b.has_bias)
            return fail(ZB_ERR_UNSUPPORTED, "the persistent executor replays bf16 blocks without bias");
        size_t njobs = 0, ntiles = 0;
        s = replay_count(b, vop.data(), n_ops, &njobs, &ntiles);
        if (s != ZB_OK) return s;
        const size_t toff = (plan.workspace_bytes + 255) & ~static_cast<size_t>(255);
        const size_t tbytes = replay_table_bytes(njobs, ntiles);
        if (!workspace) return fail(ZB_ERR_WORKSPACE, "workspace is NULL");
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(ZB_ERR_ALIGN, "workspace must be 256-byte aligned");
        if (ws_bytes < toff + tbytes)
            return fail(ZB_ERR_WORKSPACE, "workspace too small: need " + std::to_string(toff + tbytes) + " bytes");
        cudaStream_t st0 = static_cast<cudaStream_t>(stream);
        std::vector<GemmBf16> jobs;
        g_record = &jobs;
        g_in_replay = true;
        for (size_t i = 0; i < n_ops && s == ZB_OK; ++i)
            if (vop[i].kind != ZB_OP_OPT) s = run_op(i, st0, nullptr);
        g_record = nullptr;
        g_in_replay = false;
        if (s != ZB_OK) return s;
        if (jobs.size() != njobs) return fail(ZB_ERR_UNSUPPORTED, "persistent replay: GEMM count mismatch");
        if (g_plan_only) return plan_replay(jobs, g_plan_only->pairs, &g_plan_only->plan);
        Recorder trec;  // the replay kernel (with its table upload) as one span
        trec.st = st0;
        trec.on = pl->timing != 0 && stats != nullptr;
        s = event_pool(&trec.pool);
        if (s != ZB_OK) return s;
        ReplayInfo rinfo;
        s = timed(&trec, true, [&] { return replay_persistent(jobs, ws + toff, tbytes, stream, &rinfo); });
        if (s != ZB_OK) return s;
        for (size_t i = 0; i < n_ops && s == ZB_OK; ++i)
            if (vop[i].kind == ZB_OP_OPT) s = run_op(i, st0, nullptr);
        if (s != ZB_OK) return s;
        if (stats) {
            stats->workspace_bytes = toff + tbytes;
            stats->peak_live_bytes = plan.peak_live_bytes;
            stats->n_ops = static_cast<uint32_t>(n_ops);
            // the replay kernel and the kernels that write its tables
            stats->n_gemm_launches = jobs.empty() ? 0u : static_cast<uint32_t>(1 + rinfo.upload_launches);
            stats->total_ms = 0.0;
            for (double& k : stats->kind_ms) k = 0.0;
            stats->gemm_ms = 0.0;
            if (trec.on && !trec.spans.empty()) {
                const auto& sp = trec.spans.front();
                cudaError_t e = cudaEventSynchronize((*trec.pool)[sp.b]);
                if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("timing sync: ") + cudaGetErrorString(e));
                float t = 0.f;
                cudaEventElapsedTime(&t, (*trec.pool)[sp.a], (*trec.pool)[sp.b]);
                stats->total_ms = stats->gemm_ms = static_cast<double>(t);
            }
            if (stats->op_ms)
                for (size_t i = 0; i < n_ops; ++i) stats->op_ms[i] = 0.f;
        }
        clear_error();
        return ZB_OK;
    }
    if (pl->executor != ZB_EXEC_STREAMS) return fail(ZB_ERR_INVALID_ARG, "unknown pipeline.executor");

    // Streams: ops of stage (device) d run on lanes[d % nsd]; lanes[0] is the
    // caller's stream.  With streams >= 2 P (at most 8) each stage's W and
    // OPT ops get a lane of their own (lanes[nsd + d]): a weight-gradient
    // GEMM then starts on the SMs that the stage's last F/B wave leaves idle.
    // A one-stage replay with streams >= 3 instead spreads the F/B/BW ops of
    // consecutive microbatches over streams - 1 lanes (at most 7; the
    // microbatches are independent until their W) and keeps every W / OPT on
    // the last lane, in list order: each persistent GEMM then starts on the
    // SMs that the previous one's partial last wave leaves idle.  With
    // streams >= 3 P (3 P <= 12) a stage's B and BW ops also leave its F
    // lane for a lane of their own (lanes[2 P + d]): a stage's next forward
    // then starts as soon as its producers and its arena slots allow, instead
    // of queueing behind a backward that waits for the next stage.
    const bool micro_lanes = pl->P == 1 && pl->streams >= 3;
    const bool fbw_lanes = !micro_lanes && pl->P > 1 && pl->streams >= 3 * pl->P && 3 * pl->P <= 12;
    const int nsd = micro_lanes ? std::min(pl->streams - 1, 7)
                    : fbw_lanes ? pl->P
                                : std::max(1, std::min(std::min(pl->streams, pl->P), 8));
    const bool w_lanes = micro_lanes || fbw_lanes || (pl->streams >= 2 * pl->P && 2 * pl->P <= 8);
    const int ns = nsd + (w_lanes ? (micro_lanes ? 1 : pl->P) : 0) + (fbw_lanes ? pl->P : 0);
    std::vector<int> lane_of(n_ops, 0);
    for (size_t i = 0; i < n_ops; ++i) {
        const bool wk = vop[i].kind == ZB_OP_W || vop[i].kind == ZB_OP_OPT;
        const bool bk = vop[i].kind == ZB_OP_B || vop[i].kind == ZB_OP_BW;
        if (micro_lanes)
            lane_of[i] = wk ? nsd : static_cast<int>(vop[i].micro % static_cast<uint32_t>(nsd));
        else if (fbw_lanes)
            lane_of[i] = wk ? nsd + dev[i] : bk ? 2 * nsd + dev[i] : dev[i];
        else
            lane_of[i] = (w_lanes && wk) ? nsd + dev[i] : dev[i] % nsd;
    }
    std::vector<cudaStream_t> lanes(1, static_cast<cudaStream_t>(stream));
    std::vector<cudaEvent_t>* evs = nullptr;
    if (ns > 1) {
        std::vector<cudaStream_t> extra;
        s = helper_streams(ns - 1, &extra);
        if (s != ZB_OK) return s;
        lanes.insert(lanes.end(), extra.begin(), extra.end());
        s = sync_events(n_ops + ns, &evs);
        if (s != ZB_OK) return s;
        // fork: helper lanes start after the work already on the caller's stream
        cudaEvent_t fork = (*evs)[n_ops];
        cudaError_t e = cudaEventRecord(fork, lanes[0]);
        for (int k = 1; k < ns && e == cudaSuccess; ++k) e = cudaStreamWaitEvent(lanes[k], fork, 0);
        if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("fork: ") + cudaGetErrorString(e));
    }
    // producer op of F(s,j) and of B/BW(s,j), for cross-stage waits
    std::vector<int> fwd_op(static_cast<size_t>(P) * m, -1), bwd_op(static_cast<size_t>(P) * m, -1);
    for (size_t i = 0; i < n_ops; ++i) {
        const size_t key = static_cast<size_t>(vop[i].stage) * m + vop[i].micro;
        if (vop[i].kind == ZB_OP_F) fwd_op[key] = static_cast<int>(i);
        else if (vop[i].kind == ZB_OP_B || vop[i].kind == ZB_OP_BW) bwd_op[key] = static_cast<int>(i);
    }

    Recorder rec;
    rec.st = lanes[0];
    rec.on = pl->timing != 0;
    s = event_pool(&rec.pool);
    if (s != ZB_OK) return s;
    std::vector<std::pair<size_t, size_t>> op_span(n_ops, {0, 0});  // [first span, end span)
    int gemms = 0;
    g_gemm_counter = &gemms;
    g_in_replay = true;
    g_pdl_lanes = ns == 1 || (w_lanes && !micro_lanes && nsd == 1);
    std::vector<int> last_w_op(P, -1);  // latest W / BW of each stage, for OPT

    for (size_t i = 0; i < n_ops && s == ZB_OK; ++i) {
        const zb_op& o = vop[i];  // stage = virtual stage of the chain
        const int st = o.stage, j = static_cast<int>(o.micro);
        cudaStream_t lane = lanes[lane_of[i]];
        rec.st = lane;
        if (ns > 1) {
            // wait for producers and slot releases that ran on other lanes
            std::vector<int> deps;
            if (o.kind == ZB_OP_OPT) {
                deps.push_back(last_w_op[st]);
            } else {
                deps = plan.reuse_deps[i];
                if (o.kind == ZB_OP_F && st > 0) deps.push_back(fwd_op[static_cast<size_t>(st - 1) * m + j]);
                if ((o.kind == ZB_OP_B || o.kind == ZB_OP_BW) && st < P - 1)
                    deps.push_back(bwd_op[static_cast<size_t>(st + 1) * m + j]);
                // its own forward (H, A): implied by list order on one lane,
                // an event when B runs on a lane of its own
                if (o.kind == ZB_OP_B || o.kind == ZB_OP_BW) deps.push_back(fwd_op[static_cast<size_t>(st) * m + j]);
                if (o.kind == ZB_OP_W) deps.push_back(bwd_op[static_cast<size_t>(st) * m + j]);
            }
            for (int d : deps) {
                if (d < 0 || lane_of[d] == lane_of[i]) continue;
                cudaError_t e = cudaStreamWaitEvent(lane, (*evs)[d], 0);
                if (e != cudaSuccess) {
                    s = fail(ZB_ERR_CUDA, std::string("cudaStreamWaitEvent: ") + cudaGetErrorString(e));
                    break;
                }
            }
            if (s != ZB_OK) break;
        }
        op_span[i].first = rec.spans.size();
        s = run_op(i, lane, &rec);
        op_span[i].second = rec.spans.size();
        if (o.kind == ZB_OP_W || o.kind == ZB_OP_BW) last_w_op[st] = static_cast<int>(i);
        if (ns > 1 && s == ZB_OK) {
            cudaError_t e = cudaEventRecord((*evs)[i], lane);
            if (e != cudaSuccess) s = fail(ZB_ERR_CUDA, std::string("cudaEventRecord: ") + cudaGetErrorString(e));
        }
    }
    if (ns > 1) {
        // join: the caller's stream continues after every lane's work
        for (int k = 1; k < ns; ++k) {
            cudaEvent_t ev = (*evs)[n_ops + k];
            cudaError_t e = cudaEventRecord(ev, lanes[k]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(lanes[0], ev, 0);
            if (e != cudaSuccess && s == ZB_OK)
                s = fail(ZB_ERR_CUDA, std::string("join: ") + cudaGetErrorString(e));
        }
    }
    g_gemm_counter = nullptr;
    g_in_replay = false;
    g_pdl_lanes = true;
    if (s != ZB_OK) return s;

    if (stats) {
        stats->workspace_bytes = plan.workspace_bytes;
        stats->peak_live_bytes = plan.peak_live_bytes;
        stats->n_ops = static_cast<uint32_t>(n_ops);
        stats->n_gemm_launches = static_cast<uint32_t>(gemms);
        stats->total_ms = 0.0;
        for (double& k : stats->kind_ms) k = 0.0;
        stats->gemm_ms = 0.0;
    }
    if (rec.on && stats && !rec.spans.empty()) {
        cudaError_t e = cudaStreamSynchronize(lanes[0]);  // joined: every lane is done
        if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("timing sync: ") + cudaGetErrorString(e));
        auto ms = [&](size_t a, size_t bb) {
            float t = 0.f;
            cudaEventElapsedTime(&t, (*rec.pool)[a], (*rec.pool)[bb]);
            return static_cast<double>(t);
        };
        for (const auto& sp : rec.spans) stats->total_ms = std::max(stats->total_ms, ms(rec.spans.front().a, sp.b));
        for (const auto& sp : rec.spans)
            if (sp.gemm) stats->gemm_ms += ms(sp.a, sp.b);
        for (size_t i = 0; i < n_ops; ++i) {
            double t = 0.0;
            if (op_span[i].second > op_span[i].first)
                t = ms(rec.spans[op_span[i].first].a, rec.spans[op_span[i].second - 1].b);
            if (ops[i].kind < 4) stats->kind_ms[ops[i].kind] += t;
            if (stats->op_ms) stats->op_ms[i] = static_cast<float>(t);
        }
    } else if (stats && stats->op_ms) {
        for (size_t i = 0; i < n_ops; ++i) stats->op_ms[i] = 0.f;
    }
    clear_error();
    return ZB_OK;
}
