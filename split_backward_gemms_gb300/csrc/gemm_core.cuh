// gemm_core.cuh — the pieces of the bf16 tensor-core GEMM that its one-launch
// kernel (gemm_tc.cu) and the persistent replay kernel (replay_tc.cu)
// share: tile constants, shared-memory layout, bounded mbarrier waits, the
// GeLU / GeLU' epilogue arithmetic, staging boxes and TMA stores, the tile
// order, and on the host the tensor-map encoder and L2 priority choice.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "ptx.cuh"
#include "zb_internal.h"

namespace {


constexpr int BM = 128;  // rows per CTA
constexpr int BN = 256;  // tile columns (MMA N)
constexpr int BK = 64;   // K per stage (one 128-byte swizzle row of bf16)
constexpr uint32_t A_BYTES = BM * BK * 2;        // 16 KiB
constexpr uint32_t MN_ATOM_BYTES = 64 * BK * 2;  // 64 MN x 64 K, one TMA box
constexpr int NUM_THREADS = 64 + 32 * 8;  // producer, MMA issuer, up to 8 epilogue warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;  // 4 s
constexpr uint64_t DRAIN_LIMIT_NS = 500000000ull;  // 0.5 s
constexpr uint32_t STAGING_BYTES = 32 * 1024;  // 2 staging boxes per epilogue warp

// Epilogue shape.  The bf16-output epilogues run 8 warps, two per TMEM lane
// quadrant, each over half of the tile's 256 columns in chunks of 32 (a
// 32-row x 64-byte staging box, 64-byte swizzle): their GeLU / GeLU'
// arithmetic is latency-bound, and with one warp per scheduler the last
// tile's epilogue of a short-K GEMM (K = 1024) took longer than its K loop.
// The fp32 weight-gradient epilogue runs 4 warps over all 256 columns in
// chunks of 32 (32 x 128-byte boxes, 128-byte swizzle) and leaves warps 6-9
// idle: its reduce-adds are few and large, and spaced on purpose.
template <int EPI>
struct EpiShape {
    static constexpr int WARPS = EPI == zb::EPI_F32 ? 4 : 8;
    static constexpr int COLS = BN * 4 / WARPS;                         // columns per warp
    static constexpr uint32_t BOX = EPI == zb::EPI_F32 ? 32 * 128 : 32 * 64;  // bytes per staging box
};
static_assert(2 * 8 * 32 * 64 <= STAGING_BYTES && 2 * 4 * 32 * 128 <= STAGING_BYTES, "staging boxes");

template <int CG>
struct Cfg {
    static constexpr int B_ROWS = BN / CG;                       // B columns held per CTA
    static constexpr uint32_t B_BYTES = B_ROWS * BK * 2;         // 32 or 16 KiB
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;   // 48 or 32 KiB
    static constexpr int STAGES = CG == 1 ? 4 : 6;
    static constexpr int TILE_M = BM * CG;
    // see tile_coords; for the CTA pair, 16 M-blocks (4096 rows) per group:
    // at h=6144 every F/B GEMM is one group (the weights stream from DRAM
    // once), which measured +0.9 % on the power-capped step against 8
    static constexpr int GROUP_M = 16;
};

template <int STAGES>
struct SharedCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    uint64_t xchg;  // split K: bytes of the other CTAs' slabs received
    uint64_t hfull[4];   // hand-off epilogue: slot filled by the reader warp
    uint64_t hempty[4];  // hand-off epilogue: slot read by the math warp
};

// With the hand-off epilogue the staging area (after the ring) holds 16 KiB
// of TMA store boxes for its four math warps and four 4 KiB hand-off slots
// (one per reader / math warp pair).
constexpr uint32_t HAND_BOXES = 16 * 1024;
constexpr uint32_t HAND_SLOT = 32 * 32 * 4;  // one raw fp32 chunk: 32 rows x 32 columns
static_assert(HAND_BOXES + 4 * HAND_SLOT == STAGING_BYTES, "hand-off staging");
static_assert(4 * 2 * 32 * 64 == HAND_BOXES, "hand-off store boxes");

template <int CG>
constexpr size_t smem_bytes() {
    return 1024 + Cfg<CG>::STAGES * Cfg<CG>::STAGE_BYTES + STAGING_BYTES + sizeof(SharedCtl<Cfg<CG>::STAGES>) + 64;
}
static_assert(smem_bytes<1>() <= 232448, "shared memory budget (one CTA)");
static_assert(smem_bytes<2>() <= 232448, "shared memory budget (CTA pair)");

struct EpiArgs {
    int Mg, Ng, Kg;
    void* out0;
    long long ld0;
    void* out1;
    long long ld1;
    const __nv_bfloat16* aux;
    long long ldaux;
    const __nv_bfloat16* bias;
    int accumulate;
    int act;
    int ksplit;  // CTAs per tile along K (1 = no split; CG = 1 only)
    int late_wait;  // wait for the previous kernel in the stream at exit, not at start
    // L2 eviction priority of the A and B operand loads and of the output
    // stores (0 normal, 1 evict first, 2 evict last; see choose_l2_hints)
    int hint_a, hint_b, hint_out;
    // fp32 epilogue with CTA pairs: a second problem (the W pass's other
    // weight-gradient GEMM, same K and operand majors), its tiles after the
    // first's; A, B and output maps tmA2, tmB2, tmO1
    int groups;  // 1 or 2
    int Mg2, Ng2;
    int hint_a2, hint_b2;
    unsigned int* err;
};

// error-word bits
constexpr unsigned ERR_WAIT_PRODUCER = 1u << 0;
constexpr unsigned ERR_WAIT_MMA = 1u << 1;
constexpr unsigned ERR_WAIT_EPI = 1u << 2;

// Bounded wait on a local mbarrier phase.  CLUSTER selects acquire at
// cluster scope (arrivals that come from the other CTA of a pair).
template <bool CLUSTER>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err, unsigned code, uint64_t limit_ns,
                                         bool honour_abort) {
    auto poll = [&]() {
        return CLUSTER ? zbp::mbar_try_wait_cluster(bar, parity) : zbp::mbar_try_wait(bar, parity);
    };
    if (poll()) return true;
    const uint64_t t0 = zbp::globaltimer_ns();
    uint32_t spins = 0;
    while (true) {
        if (poll()) return true;
        if ((++spins & 63u) == 0) {
            if (honour_abort && *abort_flag) return false;
            if (zbp::globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// GeLU and its derivative without branches, so that the epilogue can
// interleave many independent elements (a per-element dependent chain with
// one warp per scheduler otherwise leaves the math latency-bound).
//
// Exact (erf) form: Phi(x) = (1 + erf(x / sqrt 2)) / 2 with erf(z), z >= 0,
// from Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26 (maximum absolute error 1.5e-7):
//     erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2),
//     t = 1 / (1 + p z),
// and erf(-z) = -erf(z).  exp(-z^2) = exp(-x^2 / 2) is also the normal
// density's exponential, so GeLU'(x) = Phi(x) + x phi(x) reuses it.
// tanh form: tanh(u) = 1 - 2 / (1 + exp(2u)).
struct AS71_26 {
    static constexpr float p = 0.3275911f;
    static constexpr float a1 = 0.254829592f;
    static constexpr float a2 = -0.284496736f;
    static constexpr float a3 = 1.421413741f;
    static constexpr float a4 = -1.453152027f;
    static constexpr float a5 = 1.061405429f;
};

// Phi(x) and exp(-x^2/2); 1 + p z lies in [1, 1 + p z_max], so the fast
// reciprocal is exact enough (relative error of a few ulp).
__device__ __forceinline__ void normal_cdf_and_exp(float x, float& Phi, float& e) {
    using C = AS71_26;
    const float z = fabsf(x) * 0.7071067811865476f;
    e = __expf(-0.5f * x * x);
    const float t = __fdividef(1.0f, fmaf(C::p, z, 1.0f));
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, C::a5, C::a4), C::a3), C::a2), C::a1);
    // q = (1 - erf(|x|/sqrt 2)) / 2 = Phi(-|x|); no cancellation for x < 0
    const float q = 0.5f * poly * e;
    Phi = x < 0.0f ? q : 1.0f - q;
}

// tanh(u) = 1 - 2 / (1 + exp(2u)); exp overflow gives 1, underflow -1.
__device__ __forceinline__ float tanh_nb(float u) {
    return 1.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * u));
}

template <bool TANH>
__device__ __forceinline__ float gelu_t(float x) {
    if (TANH) {
        const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
        return 0.5f * x * (1.0f + tanh_nb(u));
    }
    float Phi, e;
    normal_cdf_and_exp(x, Phi, e);
    return x * Phi;
}

template <bool TANH>
__device__ __forceinline__ float gelu_grad_t(float x) {
    if (TANH) {
        const float x2 = x * x;
        const float t = tanh_nb(0.7978845608028654f * (x + 0.044715f * x * x2));
        return 0.5f * (1.0f + t) +
               0.5f * x * (1.0f - t * t) * 0.7978845608028654f * (1.0f + 3.0f * 0.044715f * x2);
    }
    float Phi, e;
    normal_cdf_and_exp(x, Phi, e);
    return fmaf(x * 0.3989422804014327f, e, Phi);  // Phi(x) + x phi(x)
}

// N columns of one row: the activation form is chosen once per chunk so the
// unrolled element loops have no branches and interleave.
template <bool TANH, int N>
__device__ __forceinline__ void gelu_pack(const float (&x)[N], uint32_t (&w)[N / 2]);
template <bool TANH, int N>
__device__ __forceinline__ void gelu_grad_mul(float (&x)[N], const uint32_t (&h)[N / 2]);

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}

// ---------------------------------------------------------------------------
// Exact-erf GeLU / GeLU' on pairs of elements with the packed two-lane fp32
// instructions of sm_100-class GPUs (fma / mul / add .rn.f32x2): every
// polynomial and scaling step handles two elements per instruction, which
// halves the epilogue's arithmetic issue (the epilogue warps share their
// schedulers with the TMA-producer and MMA-issuer warps, whose loops it
// would otherwise delay).  Same formulas as normal_cdf_and_exp (A&S 7.1.26),
// with exp(v) = 2^(v / ln 2) and 1/y taken from the ex2.approx / rcp.approx
// instructions, the 1/2 of q folded into the coefficients and
// Phi(x) = 1/2 + sign(x) (1/2 - q) (q = Phi(-|x|)) instead of a select.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void up2(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float rcp_approx(float v) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Phi and exp(-x^2/2) of the pair X.
__device__ __forceinline__ void normal_cdf_and_exp2(f32x2 X, f32x2& PHI, f32x2& E) {
    using C = AS71_26;
    float x0, x1;
    up2(X, x0, x1);
    // exp(-x^2/2) = 2^(-x^2 / (2 ln 2))
    const f32x2 arg = mul2(mul2(X, X), pk2(-0.7213475204444817f, -0.7213475204444817f));
    float a0, a1;
    up2(arg, a0, a1);
    E = pk2(ex2_approx(a0), ex2_approx(a1));
    // t = 1 / (1 + p |x| / sqrt 2)
    const float pz = C::p * 0.7071067811865476f;
    const f32x2 den = fma2(pk2(fabsf(x0), fabsf(x1)), pk2(pz, pz), pk2(1.0f, 1.0f));
    float d0, d1;
    up2(den, d0, d1);
    const f32x2 T = pk2(rcp_approx(d0), rcp_approx(d1));
    // q/e = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) / 2
    f32x2 P = fma2(T, pk2(0.5f * C::a5, 0.5f * C::a5), pk2(0.5f * C::a4, 0.5f * C::a4));
    P = fma2(T, P, pk2(0.5f * C::a3, 0.5f * C::a3));
    P = fma2(T, P, pk2(0.5f * C::a2, 0.5f * C::a2));
    P = fma2(T, P, pk2(0.5f * C::a1, 0.5f * C::a1));
    P = mul2(T, P);
    const f32x2 half_minus_q = fma2(mul2(P, E), pk2(-1.0f, -1.0f), pk2(0.5f, 0.5f));
    float h0, h1;
    up2(half_minus_q, h0, h1);
    PHI = add2(pk2(copysignf(h0, x0), copysignf(h1, x1)), pk2(0.5f, 0.5f));
}

template <bool TANH, int N>
__device__ __forceinline__ void gelu_pack(const float (&x)[N], uint32_t (&w)[N / 2]) {
    if (TANH) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) w[i] = pack_bf16x2(gelu_t<true>(x[2 * i]), gelu_t<true>(x[2 * i + 1]));
    } else {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const f32x2 X = pk2(x[2 * i], x[2 * i + 1]);
            f32x2 PHI, E;
            normal_cdf_and_exp2(X, PHI, E);
            float g0, g1;
            up2(mul2(X, PHI), g0, g1);  // GeLU = x Phi(x)
            w[i] = pack_bf16x2(g0, g1);
        }
    }
}

template <bool TANH, int N>
__device__ __forceinline__ void gelu_grad_mul(float (&x)[N], const uint32_t (&h)[N / 2]) {
    if (TANH) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float2 f2 = unpack_bf16x2(h[i]);
            x[2 * i] *= gelu_grad_t<true>(f2.x);
            x[2 * i + 1] *= gelu_grad_t<true>(f2.y);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float2 f2 = unpack_bf16x2(h[i]);
            const f32x2 Hx = pk2(f2.x, f2.y);
            f32x2 PHI, E;
            normal_cdf_and_exp2(Hx, PHI, E);
            // GeLU'(h) = Phi(h) + h phi(h),  phi(h) = exp(-h^2/2) / sqrt(2 pi)
            const f32x2 G = fma2(mul2(Hx, pk2(0.3989422804014327f, 0.3989422804014327f)), E, PHI);
            up2(mul2(pk2(x[2 * i], x[2 * i + 1]), G), x[2 * i], x[2 * i + 1]);
        }
    }
}

// 32 bf16 values of row `row` from column col0 of H (GeLU' epilogue), zeros
// past the matrix edge.  Plain loads: the caller issues them ahead of use.
__device__ __forceinline__ void load_h32(const EpiArgs& args, int row, int col0, uint32_t (&hw)[16]) {
    const __nv_bfloat16* hp = args.aux + static_cast<long long>(row) * args.ldaux + col0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint4 hv = make_uint4(0u, 0u, 0u, 0u);
        if (row < args.Mg && col0 + g * 8 < args.Ng) hv = *reinterpret_cast<const uint4*>(hp + g * 8);
        hw[4 * g] = hv.x;
        hw[4 * g + 1] = hv.y;
        hw[4 * g + 2] = hv.z;
        hw[4 * g + 3] = hv.w;
    }
}

// Tile order: groups of `group` M-blocks; inside a group M is fastest, then
// N.  A wave of resident CTAs then covers about group x (clusters / group)
// tiles, so the operand panels it touches at each K step are few and shared
// from L2 (M-fastest over a tall problem would stream a new A panel per CTA).
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group, int& mb,
                                            int& nb) {
    const int per_group = group * tiles_n;
    const int g = tile / per_group;
    const int first = g * group;
    const int gsz = min(tiles_m - first, group);
    const int r = tile - g * per_group;
    mb = first + r % gsz;
    nb = r / gsz;
}

// Write one thread's 128-byte row of a 32-row staging box (TMA 128-byte
// swizzle: 16-byte chunk k of row r sits at chunk k ^ (r mod 8)).
__device__ __forceinline__ void stage_row(uint32_t stg, int lane, const uint32_t (&w)[32]) {
    const uint32_t row = stg + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = static_cast<uint32_t>((k ^ (lane & 7)) << 4);
        zbp::st_shared_v4(row + off, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}

// Write one thread's 64-byte row of a 32-row staging box (TMA 64-byte swizzle:
// 16-byte chunk k of row r sits at chunk k ^ ((r / 2) mod 4); the 8 rows a
// quarter-warp writes then hit 8 different bank groups).
__device__ __forceinline__ void stage_row64(uint32_t stg, int lane, const uint32_t (&w)[16]) {
    const uint32_t row = stg + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t off = static_cast<uint32_t>((k ^ ((lane >> 1) & 3)) << 4);
        zbp::st_shared_v4(row + off, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}

// Lane 0 makes sure the staging buffer about to be written is no longer read
// by the bulk store issued two stores ago (buffers alternate).
__device__ __forceinline__ void staging_acquire(int lane) {
    if (lane == 0) zbp::bulk_wait_read<1>();
    __syncwarp();
}

// Hand a filled staging buffer to the TMA unit.
template <bool REDUCE>
__device__ __forceinline__ void staging_release(const CUtensorMap* tm, uint32_t stg, int lane,
                                                int x, int y, uint64_t policy) {
    zbp::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (REDUCE)
            zbp::tma_reduce_add_2d_hint(tm, stg, x, y, policy);
        else
            zbp::tma_store_2d_hint(tm, stg, x, y, policy);
        zbp::bulk_commit();
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(std::string* why) {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    static std::string err;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr) {
            err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(e);
            return;
        }
        fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn && why) *why = err;
    return fn;
}

// 2-D map: inner dimension `inner` (contiguous), `outer` rows of stride ld
// elements; box of box_inner x box_outer elements, 128-byte swizzle unless
// given (the inner box extent in bytes must not exceed the swizzle span).
bool make_map(CUtensorMap* m, const void* base, bool f32, uint64_t inner, uint64_t outer,
              uint64_t ld, uint32_t box_inner, uint32_t box_outer, std::string* why,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn(why);
    if (!fn) return false;
    const uint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * es};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev].load(std::memory_order_relaxed) == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return cache[dev].load(std::memory_order_relaxed);
}

// L2 eviction priorities.  Tiles run in groups of GROUP_M M-blocks, M
// fastest inside a group (tile_coords), so every wave of resident tiles
// reads the A rows of its group again over the whole K range, and every
// group reads the whole B operand again.  An operand whose re-read part fits
// comfortably in L2 beside the streams (at most 48 MB: A's rows of one group,
// or all of B when there are several groups) is kept (evict last); a larger
// one, read once per group or too large to keep, goes first, so that it
// does not push the kept one out; an output larger than 48 MB goes first
// too (written once, read by a later kernel), a smaller one stays normal
// (the next GEMM of the pass reads it at once).  At h=6144 this keeps X and
// dY (37.7 MB) across the waves of the F1 and B1 GEMMs (DRAM reads 673 ->
// 398 MB and 934 -> 815 MB per launch) and a group's 25 MB of A in the W
// GEMMs.  ZB_GEMM_L2_HINTS=0 in the environment turns the hints off.
void choose_l2_hints(const zb::GemmBf16& g, int cg, EpiArgs* ea) {
    static const bool on = [] {
        const char* v = std::getenv("ZB_GEMM_L2_HINTS");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    ea->hint_a = ea->hint_b = ea->hint_out = 0;
    if (!on) return;
    constexpr double kKeep = 48e6;
    const long long group_rows = static_cast<long long>(Cfg<1>::GROUP_M) * BM * cg;
    const long long groups = (g.Mg + group_rows - 1) / group_rows;
    const double a_group = 2.0 * static_cast<double>(g.Mg < group_rows ? g.Mg : group_rows) * g.Kg;
    const double b_all = 2.0 * static_cast<double>(g.Ng) * g.Kg;
    const double out = (g.epi == zb::EPI_F32 ? 4.0 : 2.0) * static_cast<double>(g.Mg) * g.Ng;
    ea->hint_a = a_group <= kKeep ? 2 : 1;
    ea->hint_b = b_all > kKeep ? 1 : (groups > 1 ? 2 : 0);
    ea->hint_out = out > kKeep ? 1 : 0;
}

}  // namespace
