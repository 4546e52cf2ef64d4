// misc.cu — the true-fp32 FFMA GEMM (single-linear fp32 blocks, no TF32),
// the fixed-order column sums of the bias gradients, and the device error
// word of the bounded waits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "ptx.cuh"
#include "zb_internal.h"

namespace {

// ---------------------------------------------------------------- error word
// Bit-set by a bounded device wait that gave up (see gemm_tc.cu).  One word
// per device context; read and cleared by zb_sync_status().
__device__ unsigned int g_zb_error_word;

// ---------------------------------------------------------------- fp32 GEMM
constexpr int TM = 64, TN = 64, TK = 16;

// C[m*ldc + n] (+)= sum_k A[m*sam + k*sak] * B[k*sbk + n*sbn]; every output
// sums its products in ascending k with fmaf, so results are deterministic.
__global__ void __launch_bounds__(256)
    zb_gemm_f32_simt_kernel(zb::GemmF32 g) {
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN + 4];
    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const long long m0 = static_cast<long long>(blockIdx.y) * TM;
    const long long n0 = static_cast<long long>(blockIdx.x) * TN;
    float acc[4][4] = {};
    for (long long k0 = 0; k0 < g.Kg; k0 += TK) {
#pragma unroll
        for (int i = 0; i < (TK * TM) / 256; ++i) {
            const int idx = tid + i * 256;
            const int kk = idx / TM, mm = idx % TM;
            const long long m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < g.Mg && k < g.Kg) ? g.A[m * g.sam + k * g.sak] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < (TK * TN) / 256; ++i) {
            const int idx = tid + i * 256;
            const int kk = idx / TN, nn = idx % TN;
            const long long n = n0 + nn, k = k0 + kk;
            Bs[kk][nn] = (n < g.Ng && k < g.Kg) ? g.B[k * g.sbk + n * g.sbn] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long m = m0 + ty * 4 + i;
        if (m >= g.Mg) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const long long n = n0 + tx * 4 + j;
            if (n >= g.Ng) continue;
            float* c = g.C + m * g.ldc + n;
            *c = g.accumulate ? (*c + acc[i][j]) : acc[i][j];
        }
    }
}

// ---------------------------------------------------------------- column sums
template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Column sums db[c] (+)= sum_r X[r, c] with a fixed summation order.  A
// cluster of COLSUM_SPLIT blocks covers 32 x CPL columns: block b of the
// cluster sums the b-th contiguous range of rows; inside it each lane loads
// CPL adjacent elements of a row (8 or 16 bytes, so a warp reads 256 or 512
// contiguous bytes per row) and warp w sums rows w, w + 8, ... of the range
// in ascending order; the 8 warp partials are added in warp order, and block
// 0 adds the blocks' partials in rank order, read from their shared memory
// (distributed shared memory, no global scratch).  Every column's additions
// come in the same order whatever CPL is, so the same inputs give the same
// bits.  bf16
// matrices take CPL = 8 (16-byte loads) when that still gives two blocks per
// SM, else CPL = 4 (twice the blocks): the db1 sum of an h=6144 block (24576
// columns) is then 768 blocks, one wave (1536 with CPL = 4 was a second wave
// of 26 %), and the db2 sum (6144 columns) keeps 384 blocks.
constexpr int COLSUM_WARPS = 8;
constexpr int COLSUM_SPLIT = 8;  // blocks (row ranges) per cluster

template <typename T, int CPL>
__device__ __forceinline__ void load_cols(const T* p, float (&v)[CPL]);
template <>
__device__ __forceinline__ void load_cols<__nv_bfloat16, 4>(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xffff0000u);
}
template <>
__device__ __forceinline__ void load_cols<float, 4>(const float* p, float (&v)[4]) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
}
template <>
__device__ __forceinline__ void load_cols<__nv_bfloat16, 8>(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

int sm_count_misc() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev].load(std::memory_order_relaxed) == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev].store(n > 0 ? n : 148, std::memory_order_relaxed);
    }
    return cache[dev].load(std::memory_order_relaxed);
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

template <typename T, int CPL>
__global__ void __cluster_dims__(COLSUM_SPLIT, 1, 1) __launch_bounds__(COLSUM_WARPS * 32)
    zb_colsum_kernel(const T* __restrict__ X, long long rows, long long cols, long long ld,
                     float* __restrict__ db, int accumulate, int vec_ok) {
    constexpr int COLS = 32 * CPL;  // columns per cluster
    __shared__ float part[COLSUM_WARPS][COLS];
    __shared__ float block_sum[COLS];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t rank = zbp::cluster_ctarank();
    const long long cb = blockIdx.x / COLSUM_SPLIT;
    const long long c0 = cb * COLS + CPL * lane;
    const long long r_begin = rows * rank / COLSUM_SPLIT, r_end = rows * (rank + 1) / COLSUM_SPLIT;
    float acc[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) acc[i] = 0.0f;
    if (vec_ok && c0 + CPL <= cols) {
        // 8 rows' loads in flight per lane (128 bytes)
#pragma unroll 8
        for (long long r = r_begin + w; r < r_end; r += COLSUM_WARPS) {
            float v[CPL];
            load_cols<T, CPL>(X + r * ld + c0, v);
#pragma unroll
            for (int i = 0; i < CPL; ++i) acc[i] += v[i];
        }
    } else {
        for (long long r = r_begin + w; r < r_end; r += COLSUM_WARPS)
#pragma unroll
            for (int i = 0; i < CPL; ++i)
                if (c0 + i < cols) acc[i] += to_f<T>(X[r * ld + c0 + i]);
    }
#pragma unroll
    for (int i = 0; i < CPL; ++i) part[w][CPL * lane + i] = acc[i];
    __syncthreads();
    for (int c = threadIdx.x; c < COLS; c += COLSUM_WARPS * 32) {
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < COLSUM_WARPS; ++k) sum += part[k][c];
        block_sum[c] = sum;
    }
    zbp::cluster_sync();  // every block's partial is in its shared memory
    if (rank == 0) {
        for (int t = threadIdx.x; t < COLS; t += COLSUM_WARPS * 32) {
            const long long c = cb * COLS + t;
            if (c < cols) {
                const uint32_t local = zbp::smem_u32(&block_sum[t]);
                float sum = 0.0f;
#pragma unroll
                for (int b = 0; b < COLSUM_SPLIT; ++b) sum += ld_shared_cluster_f32(zbp::mapa_shared(local, b));
                db[c] = accumulate ? db[c] + sum : sum;
            }
        }
    }
    zbp::cluster_sync();  // no block leaves while block 0 may still read it
}

// One thread waits on an mbarrier that nothing arrives on, for at most
// limit_ns, then records the expiry in the error word (bit 31).
__global__ void zb_selftest_wait_kernel(unsigned int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = zbp::smem_u32(&bar);
    zbp::mbar_init(b, 1);
    zbp::fence_mbar_init();
    const uint64_t t0 = zbp::globaltimer_ns();
    while (!zbp::mbar_try_wait(b, 0)) {
        if (zbp::globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, 1u << 31);
            return;
        }
    }
}

// ---------------------------------------------------------------- gradient statistics
// Fixed partition (independent of the device): every buffer is cut into
// STATS_BLOCKS ranges of float4 groups; each thread sums the squares of its
// strided groups in fp32, the block combines the threads in fp64 in a fixed
// tree, and one block adds the partials in a fixed order (the final kernel).
constexpr int STATS_BLOCKS = 304;
constexpr int STATS_THREADS = 256;
constexpr int STATS_MAX_BUFS = 4;

struct StatsBufs {
    const float* p[STATS_MAX_BUFS];
    unsigned long long n[STATS_MAX_BUFS];
};

__global__ void __launch_bounds__(STATS_THREADS)
    zb_grad_stats_partial_kernel(StatsBufs b, double* part) {
    const int buf = blockIdx.y;
    const float* x = b.p[buf];
    const unsigned long long n = b.n[buf];
    const unsigned long long n4 = n / 4;
    const unsigned long long per = (n4 + STATS_BLOCKS - 1) / STATS_BLOCKS;
    const unsigned long long lo = per * blockIdx.x;
    const unsigned long long hi = min(lo + per, n4);
    // four float4 loads in flight per thread, four accumulators combined in
    // a fixed order; the tail goes to the first
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    unsigned bad = 0;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    auto add = [&](const float4& v, float& a) {
        a = fmaf(v.x, v.x, a);
        a = fmaf(v.y, v.y, a);
        a = fmaf(v.z, v.z, a);
        a = fmaf(v.w, v.w, a);
        bad += !isfinite(v.x) + !isfinite(v.y) + !isfinite(v.z) + !isfinite(v.w);
    };
    unsigned long long i = lo + threadIdx.x;
    for (; i + 3ull * STATS_THREADS < hi; i += 4ull * STATS_THREADS) {
        const float4 v0 = x4[i], v1 = x4[i + STATS_THREADS];
        const float4 v2 = x4[i + 2 * STATS_THREADS], v3 = x4[i + 3 * STATS_THREADS];
        add(v0, a0);
        add(v1, a1);
        add(v2, a2);
        add(v3, a3);
    }
    for (; i < hi; i += STATS_THREADS) add(x4[i], a0);
    float sq = (a0 + a1) + (a2 + a3);
    if (blockIdx.x == 0 && threadIdx.x < n - 4 * n4) {  // the last n mod 4 elements
        const float v = x[4 * n4 + threadIdx.x];
        sq = fmaf(v, v, sq);
        bad += !isfinite(v);
    }
    double dsq = sq, dbad = bad;
    for (int o = 16; o > 0; o >>= 1) {
        dsq += __shfl_down_sync(0xffffffffu, dsq, o);
        dbad += __shfl_down_sync(0xffffffffu, dbad, o);
    }
    __shared__ double ssq[STATS_THREADS / 32], sbad[STATS_THREADS / 32];
    if ((threadIdx.x & 31) == 0) {
        ssq[threadIdx.x >> 5] = dsq;
        sbad[threadIdx.x >> 5] = dbad;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double a = 0.0, c = 0.0;
        for (int w = 0; w < STATS_THREADS / 32; ++w) {
            a += ssq[w];
            c += sbad[w];
        }
        part[2 * (buf * STATS_BLOCKS + blockIdx.x)] = a;
        part[2 * (buf * STATS_BLOCKS + blockIdx.x) + 1] = c;
    }
}

// One block adds the partials: thread t takes partials t, t + 256, ... in
// index order, then a fixed tree (shuffles, then the warps in order).  A
// single thread walking all of them would wait on one dependent load after
// another (~0.1 ms for 1216 partials, longer than the partial kernel itself
// on a few hundred MB).
__global__ void __launch_bounds__(STATS_THREADS)
    zb_grad_stats_final_kernel(const double* part, int nbufs, double* out) {
    double a = 0.0, c = 0.0;
    for (int i = threadIdx.x; i < nbufs * STATS_BLOCKS; i += STATS_THREADS) {
        a += part[2 * i];
        c += part[2 * i + 1];
    }
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_down_sync(0xffffffffu, a, o);
        c += __shfl_down_sync(0xffffffffu, c, o);
    }
    __shared__ double sa[STATS_THREADS / 32], sc[STATS_THREADS / 32];
    if ((threadIdx.x & 31) == 0) {
        sa[threadIdx.x >> 5] = a;
        sc[threadIdx.x >> 5] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double ta = 0.0, tc = 0.0;
        for (int w = 0; w < STATS_THREADS / 32; ++w) {
            ta += sa[w];
            tc += sc[w];
        }
        out[0] = ta;
        out[1] = tc;
    }
}

}  // namespace

namespace zb {

unsigned int* device_error_word() {
    static std::mutex mu;
    static unsigned int* ptrs[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        fail(ZB_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_zb_error_word);
        if (e != cudaSuccess) {
            fail(ZB_ERR_CUDA, std::string("cudaGetSymbolAddress(error word): ") + cudaGetErrorString(e));
            return nullptr;
        }
        ptrs[dev] = static_cast<unsigned int*>(p);
    }
    return ptrs[dev];
}

zb_status gemm_f32_simt(const GemmF32& g, void* stream) {
    if (g.Mg <= 0 || g.Ng <= 0 || g.Kg <= 0) return fail(ZB_ERR_SHAPE, "fp32 GEMM extents must be >= 1");
    if (!g.A || !g.B || !g.C) return fail(ZB_ERR_INVALID_ARG, "fp32 GEMM operand is NULL");
    const long long gx = (g.Ng + TN - 1) / TN, gy = (g.Mg + TM - 1) / TM;
    if (gy > 65535) return fail(ZB_ERR_SHAPE, "fp32 GEMM M too large");
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
    zb_gemm_f32_simt_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(g);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("fp32 GEMM launch: ") + cudaGetErrorString(e));
    return ZB_OK;
}

zb_status colsum_bf16(const void* X, int64_t rows, int64_t cols, int64_t ld, float* db,
                      int accumulate, void* stream) {
    const auto* x = static_cast<const __nv_bfloat16*>(X);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long wide_blocks = (cols + 255) / 256 * COLSUM_SPLIT;
    if (wide_blocks >= 2LL * sm_count_misc()) {
        // 16-byte loads need 8-column groups that start 16-byte aligned
        const int vec_ok = (reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ld & 7) == 0;
        zb_colsum_kernel<__nv_bfloat16, 8><<<static_cast<unsigned>(wide_blocks), COLSUM_WARPS * 32, 0, st>>>(
            x, rows, cols, ld, db, accumulate, vec_ok);
    } else {
        const unsigned blocks = static_cast<unsigned>((cols + 127) / 128 * COLSUM_SPLIT);
        const int vec_ok = (reinterpret_cast<uintptr_t>(X) & 7u) == 0 && (ld & 3) == 0;
        zb_colsum_kernel<__nv_bfloat16, 4><<<blocks, COLSUM_WARPS * 32, 0, st>>>(x, rows, cols, ld, db,
                                                                                accumulate, vec_ok);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("colsum launch: ") + cudaGetErrorString(e));
    return ZB_OK;
}

zb_status colsum_f32(const float* X, int64_t rows, int64_t cols, int64_t ld, float* db,
                     int accumulate, void* stream) {
    const unsigned blocks = static_cast<unsigned>((cols + 127) / 128 * COLSUM_SPLIT);
    const int vec_ok = (reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ld & 3) == 0;
    zb_colsum_kernel<float, 4><<<blocks, COLSUM_WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        X, rows, cols, ld, db, accumulate, vec_ok);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("colsum launch: ") + cudaGetErrorString(e));
    return ZB_OK;
}

}  // namespace zb

extern "C" zb_status zb_sync_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return zb::fail(ZB_ERR_CUDA, std::string("stream: ") + cudaGetErrorString(e));
    unsigned int* w = zb::device_error_word();
    if (!w) return ZB_ERR_CUDA;
    unsigned int v = 0;
    e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return zb::fail(ZB_ERR_CUDA, std::string("read error word: ") + cudaGetErrorString(e));
    if (v != 0) {
        const unsigned int zero = 0;
        cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        return zb::fail(ZB_ERR_TIMEOUT, "a bounded device wait gave up (error word " + std::to_string(v) + ")");
    }
    zb::clear_error();
    return ZB_OK;
}

extern "C" zb_status zb_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
    unsigned int* w = zb::device_error_word();
    if (!w) return ZB_ERR_CUDA;
    if (limit_ns < 1000000ull) limit_ns = 1000000ull;
    if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;
    zb_selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(w, limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return zb::fail(ZB_ERR_CUDA, std::string("self-test launch: ") + cudaGetErrorString(e));
    zb::clear_error();
    return ZB_OK;
}

extern "C" size_t zb_grad_stats_scratch_bytes(void) {
    return static_cast<size_t>(2 * STATS_MAX_BUFS * STATS_BLOCKS) * sizeof(double);
}

extern "C" zb_status zb_grad_stats(const float* const* bufs, const uint64_t* counts, int32_t nbufs,
                                   double* out, void* scratch, size_t scratch_bytes, void* stream) {
    if (nbufs < 1 || nbufs > STATS_MAX_BUFS) return zb::fail(ZB_ERR_INVALID_ARG, "nbufs must be in [1, 4]");
    if (!bufs || !counts || !out || !scratch) return zb::fail(ZB_ERR_INVALID_ARG, "NULL argument");
    if (scratch_bytes < zb_grad_stats_scratch_bytes()) return zb::fail(ZB_ERR_WORKSPACE, "scratch too small");
    if ((reinterpret_cast<uintptr_t>(scratch) & 15u) || (reinterpret_cast<uintptr_t>(out) & 7u))
        return zb::fail(ZB_ERR_ALIGN, "scratch must be 16-byte and out 8-byte aligned");
    StatsBufs b = {};
    for (int i = 0; i < nbufs; ++i) {
        if (!bufs[i] || (reinterpret_cast<uintptr_t>(bufs[i]) & 15u))
            return zb::fail(ZB_ERR_ALIGN, "gradient buffers must be non-NULL and 16-byte aligned");
        b.p[i] = bufs[i];
        b.n[i] = counts[i];
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    double* part = static_cast<double*>(scratch);
    zb_grad_stats_partial_kernel<<<dim3(STATS_BLOCKS, nbufs), STATS_THREADS, 0, st>>>(b, part);
    zb_grad_stats_final_kernel<<<1, STATS_THREADS, 0, st>>>(part, nbufs, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return zb::fail(ZB_ERR_CUDA, std::string("grad stats launch: ") + cudaGetErrorString(e));
    zb::clear_error();
    return ZB_OK;
}
