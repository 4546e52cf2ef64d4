// optim.cu — one optimizer step of P pipeline stages with post-update
// validation, replayed on one GPU ("Zero Bubble Pipeline Parallelism",
// summary §4 "The Optimizer Synchronization Bypass" and "Why rollback is
// feasible"):
//   1. staged reduce: stage s's partial state is the sum of the local states
//      (gradient sum of squares, NaN/Inf count) of stages 0..s; the last
//      partial is the global state;
//   2. optimistic AdamW step of every stage with its partial state (clip
//      factor max_norm / ||g||_partial when that norm exceeds max_norm; no
//      update when a NaN/Inf has been seen);
//   3. validation: a stage whose clip factor or skip decision differs from
//      the global one inverts its step (AdamW is invertible given the same
//      gradient) and steps again with the global state.
// One device thread makes every decision from the device-resident states,
// so nothing waits for the host.  The tensor passes are HBM-bound: the
// optimistic step reads theta, m, v, g and writes theta, m, v and the bf16
// weight copy (30 bytes per element); validation moves the same bytes again
// for the stages that roll back and returns at once for the others.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <string>

#include "zb_internal.h"

namespace {

constexpr int MAX_STAGES = 64;
constexpr int TABLE = 64;       // tensors per launch (about 4 KB of kernel parameters)
constexpr int THREADS = 256;
constexpr int VEC = 2;                   // float4 groups per thread per chunk
constexpr int CHUNK = THREADS * 4 * VEC;  // elements per block iteration

struct StatePtrs {
    const double* p[MAX_STAGES];
};

__device__ __forceinline__ double clip_of(double sq, double max_norm) {
    if (!(max_norm > 0.0)) return 1.0;
    const double n = sqrt(sq);
    return n > max_norm ? max_norm / n : 1.0;
}

// One thread: staged (prefix) reduce, then the optimistic and global
// decisions of every stage.  Scales are compared in fp64.
__global__ void zb_post_validation_decide_kernel(StatePtrs st, int P, double max_norm,
                                                 zb_stage_decision* dec) {
    double sq = 0.0, bad = 0.0;
    double used[MAX_STAGES];
    for (int s = 0; s < P; ++s) {
        sq += st.p[s][0];
        bad += st.p[s][1];
        used[s] = clip_of(sq, max_norm);
        dec[s].norm_sq_partial = sq;
        dec[s].skip_used = (bad > 0.0 || !isfinite(sq)) ? 1 : 0;
    }
    const double g_scale = clip_of(sq, max_norm);
    const int g_skip = (bad > 0.0 || !isfinite(sq)) ? 1 : 0;
    for (int s = 0; s < P; ++s) {
        dec[s].norm_sq_global = sq;
        dec[s].scale_used = static_cast<float>(used[s]);
        dec[s].scale_global = static_cast<float>(g_scale);
        dec[s].skip_global = g_skip;
        dec[s].rolled_back = (used[s] != g_scale || dec[s].skip_used != g_skip) ? 1 : 0;
        dec[s].reserved = 0;
    }
}

// Per-call constants; every division by a constant is a multiplication by
// its reciprocal, rounded once on the host.
struct Hyper {
    float lr, lr_wd, eps;
    float b1, b2, omb1, omb2;  // beta and 1 - beta
    float inv_bc1, inv_bc2;    // 1 / (1 - beta^t)
    float inv_b1, inv_b2;      // 1 / beta
    float inv_keep;            // 1 / (1 - lr wd)
};

__device__ __forceinline__ float sqrt_approx(float x) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The step's direction mhat / (sqrt(vhat) + eps).  The forward and the
// inverse evaluate it with the same instructions on the same (m, v), so the
// inverse subtracts exactly what the forward added up to the rounding of the
// final theta.
__device__ __forceinline__ float adam_dir(float m, float v, const Hyper& h) {
    return __fdividef(m * h.inv_bc1, sqrt_approx(v * h.inv_bc2) + h.eps);
}

__device__ __forceinline__ void adamw_fwd(float& th, float& m, float& v, float g, const Hyper& h) {
    m = fmaf(h.b1, m, h.omb1 * g);
    v = fmaf(h.b2, v, h.omb2 * g * g);
    th = fmaf(-h.lr, adam_dir(m, v, h), fmaf(-h.lr_wd, th, th));
}

// Algebraic inverse of adamw_fwd for the same gradient.  v is clamped at 0:
// the subtraction can leave a rounding residue of either sign when the
// previous second moment was zero.
__device__ __forceinline__ void adamw_inv(float& th, float& m, float& v, float g, const Hyper& h) {
    th = fmaf(h.lr, adam_dir(m, v, h), th) * h.inv_keep;
    m = fmaf(-h.omb1, g, m) * h.inv_b1;
    v = fmaxf(fmaf(-h.omb2 * g, g, v) * h.inv_b2, 0.0f);
}

struct Desc {
    float* theta;
    float* m;
    float* v;
    const float* grad;
    __nv_bfloat16* wb;
    unsigned long long count;
    unsigned long long chunk_begin;  // first global chunk of this tensor
    int stage;
    int pad;
};

struct Table {
    Desc d[TABLE];
    int n;
    unsigned long long total_chunks;
};

template <int PASS>
__device__ __forceinline__ void update(float& th, float& mm, float& vv, float g, const zb_stage_decision& dec,
                                       const Hyper& h) {
    if (PASS == 0) {
        adamw_fwd(th, mm, vv, dec.scale_used * g, h);
    } else {
        if (!dec.skip_used) adamw_inv(th, mm, vv, dec.scale_used * g, h);
        if (!dec.skip_global) adamw_fwd(th, mm, vv, dec.scale_global * g, h);
    }
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* p, const float4& th) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(th.x, th.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(th.z, th.w);
    uint2 packed;
    packed.x = *reinterpret_cast<unsigned*>(&lo);
    packed.y = *reinterpret_cast<unsigned*>(&hi);
    *reinterpret_cast<uint2*>(p) = packed;
}

// PASS 0: optimistic step with the stage's partial decision (skipped stages
//         are left untouched).
// PASS 1: validation — a stage that rolled back inverts its optimistic step
//         and applies the global decision; the others return at once.
// Blocks walk the chunks of all tensors in the table with a grid stride; a
// block reloads its stage decision only when it enters a new tensor, so the
// data loads of a chunk never wait behind it.  Each thread issues the loads
// of all VEC float4 groups of a chunk before it computes.
template <int PASS>
__global__ void __launch_bounds__(THREADS)
    zb_adamw_kernel(const __grid_constant__ Table tab, Hyper h, const zb_stage_decision* __restrict__ decs) {
    int t = -1;
    bool active = false;
    zb_stage_decision dec = {};
    for (unsigned long long c = blockIdx.x; c < tab.total_chunks; c += gridDim.x) {
        int nt = t < 0 ? 0 : t;
        while (nt + 1 < tab.n && c >= tab.d[nt + 1].chunk_begin) ++nt;  // chunks ascend: scan forward
        if (nt != t) {
            t = nt;
            dec = decs[tab.d[t].stage];
            active = PASS == 0 ? !dec.skip_used : dec.rolled_back != 0;
        }
        if (!active) continue;
        const Desc& d = tab.d[t];
        const unsigned long long base = (c - d.chunk_begin) * CHUNK;
        if (base + CHUNK <= d.count) {
            float4 th[VEC], mm[VEC], vv[VEC], g[VEC];
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const unsigned long long i = base + 4ull * (threadIdx.x + k * THREADS);
                th[k] = *reinterpret_cast<const float4*>(d.theta + i);
                mm[k] = *reinterpret_cast<const float4*>(d.m + i);
                vv[k] = *reinterpret_cast<const float4*>(d.v + i);
                g[k] = *reinterpret_cast<const float4*>(d.grad + i);
            }
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const unsigned long long i = base + 4ull * (threadIdx.x + k * THREADS);
                update<PASS>(th[k].x, mm[k].x, vv[k].x, g[k].x, dec, h);
                update<PASS>(th[k].y, mm[k].y, vv[k].y, g[k].y, dec, h);
                update<PASS>(th[k].z, mm[k].z, vv[k].z, g[k].z, dec, h);
                update<PASS>(th[k].w, mm[k].w, vv[k].w, g[k].w, dec, h);
                *reinterpret_cast<float4*>(d.theta + i) = th[k];
                *reinterpret_cast<float4*>(d.m + i) = mm[k];
                *reinterpret_cast<float4*>(d.v + i) = vv[k];
                if (d.wb) store_bf16x4(d.wb + i, th[k]);
            }
        } else {
            // the tensor's last, partial chunk: element by element
            for (unsigned long long i = base + threadIdx.x; i < d.count; i += THREADS) {
                float th = d.theta[i], mm = d.m[i], vv = d.v[i];
                update<PASS>(th, mm, vv, d.grad[i], dec, h);
                d.theta[i] = th;
                d.m[i] = mm;
                d.v[i] = vv;
                if (d.wb) d.wb[i] = __float2bfloat16_rn(th);
            }
        }
    }
}

// Resident blocks of each pass's kernel on the whole GPU (grid = one full
// wave, so no block starts in a partial second wave).
template <int PASS>
unsigned resident_blocks() {
    static std::atomic<unsigned> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152u * 4;
    if (const unsigned c = cached[dev].load(std::memory_order_relaxed)) return c;
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, zb_adamw_kernel<PASS>, THREADS, 0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm < 1 || sms < 1) {
        cudaGetLastError();
        return 152u * 4;
    }
    cached[dev].store(static_cast<unsigned>(per_sm * sms), std::memory_order_relaxed);
    return static_cast<unsigned>(per_sm * sms);
}

bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

}  // namespace

extern "C" zb_status zb_post_validated_adamw(int32_t P, const double* const* stage_state,
                                             const zb_opt_tensor* tensors, int32_t n_tensors,
                                             const zb_adamw_params* hp, zb_stage_decision* decisions,
                                             void* stream) {
    if (P < 1 || P > MAX_STAGES) return zb::fail(ZB_ERR_SHAPE, "P must be in [1, 64]");
    if (n_tensors < 0) return zb::fail(ZB_ERR_SHAPE, "n_tensors must be >= 0");
    if (!stage_state || (n_tensors > 0 && !tensors) || !hp || !decisions)
        return zb::fail(ZB_ERR_INVALID_ARG, "NULL argument");
    if (misaligned(decisions, 8)) return zb::fail(ZB_ERR_ALIGN, "decisions must be 8-byte aligned");
    if (hp->step < 1 || !(hp->lr >= 0.0f) || !(hp->beta1 > 0.0f && hp->beta1 < 1.0f) ||
        !(hp->beta2 > 0.0f && hp->beta2 < 1.0f) || !(hp->eps > 0.0f) || !(hp->weight_decay >= 0.0f) ||
        !(hp->lr * hp->weight_decay < 1.0f) || !(hp->max_norm >= 0.0f) || hp->reserved != 0)
        return zb::fail(ZB_ERR_INVALID_ARG,
                        "AdamW parameters out of range (step >= 1, 0 < beta < 1, eps > 0, 0 <= lr*wd < 1)");
    StatePtrs sp = {};
    for (int s = 0; s < P; ++s) {
        if (!stage_state[s]) return zb::fail(ZB_ERR_INVALID_ARG, "stage_state entry is NULL");
        if (misaligned(stage_state[s], 8)) return zb::fail(ZB_ERR_ALIGN, "stage_state entries must be 8-byte aligned");
        sp.p[s] = stage_state[s];
    }
    for (int i = 0; i < n_tensors; ++i) {
        const zb_opt_tensor& t = tensors[i];
        const std::string which = "optimizer tensor " + std::to_string(i);
        if (t.stage < 0 || t.stage >= P) return zb::fail(ZB_ERR_INVALID_ARG, which + ": stage out of range");
        if (t.reserved != 0) return zb::fail(ZB_ERR_INVALID_ARG, which + ": reserved must be 0");
        if (t.count == 0) continue;
        if (!t.theta || !t.m || !t.v || !t.grad) return zb::fail(ZB_ERR_INVALID_ARG, which + ": NULL pointer");
        if (misaligned(t.theta, 16) || misaligned(t.m, 16) || misaligned(t.v, 16) || misaligned(t.grad, 16) ||
            misaligned(t.weight_bf16, 16))
            return zb::fail(ZB_ERR_ALIGN, which + ": pointers must be 16-byte aligned");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    zb_post_validation_decide_kernel<<<1, 1, 0, st>>>(sp, P, static_cast<double>(hp->max_norm), decisions);
    Hyper h;
    const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, t = static_cast<double>(hp->step);
    h.lr = hp->lr;
    h.lr_wd = static_cast<float>(lr * hp->weight_decay);
    h.eps = hp->eps;
    h.b1 = hp->beta1;
    h.b2 = hp->beta2;
    h.omb1 = static_cast<float>(1.0 - b1);
    h.omb2 = static_cast<float>(1.0 - b2);
    h.inv_bc1 = static_cast<float>(1.0 / (1.0 - std::pow(b1, t)));
    h.inv_bc2 = static_cast<float>(1.0 / (1.0 - std::pow(b2, t)));
    h.inv_b1 = static_cast<float>(1.0 / b1);
    h.inv_b2 = static_cast<float>(1.0 / b2);
    h.inv_keep = static_cast<float>(1.0 / (1.0 - lr * hp->weight_decay));
    // Every stage's optimistic step, then every stage's validation: the
    // validation pass needs only the decisions, which the first kernel wrote.
    for (int pass = 0; pass < 2; ++pass) {
        int i = 0;
        while (i < n_tensors) {
            Table tab = {};
            unsigned long long chunks = 0;
            for (; i < n_tensors && tab.n < TABLE; ++i) {
                const zb_opt_tensor& t = tensors[i];
                if (t.count == 0) continue;
                Desc& d = tab.d[tab.n++];
                d.theta = t.theta;
                d.m = t.m;
                d.v = t.v;
                d.grad = t.grad;
                d.wb = static_cast<__nv_bfloat16*>(t.weight_bf16);
                d.count = t.count;
                d.chunk_begin = chunks;
                d.stage = t.stage;
                chunks += (t.count + CHUNK - 1) / CHUNK;
            }
            if (chunks == 0) continue;
            tab.total_chunks = chunks;
            const unsigned long long wave = pass == 0 ? resident_blocks<0>() : resident_blocks<1>();
            const unsigned grid = static_cast<unsigned>(chunks < wave ? chunks : wave);
            if (pass == 0)
                zb_adamw_kernel<0><<<grid, THREADS, 0, st>>>(tab, h, decisions);
            else
                zb_adamw_kernel<1><<<grid, THREADS, 0, st>>>(tab, h, decisions);
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return zb::fail(ZB_ERR_CUDA, std::string("optimizer launch: ") + cudaGetErrorString(e));
    zb::clear_error();
    return ZB_OK;
}
