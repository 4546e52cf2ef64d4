// gemm_tc.cu — bf16 tensor-core GEMM for sm_103a with fused epilogues.
//
// One persistent, warp-specialised kernel computes every contraction of the
// split MLP block (the three passes of "Zero Bubble Pipeline Parallelism",
// summary §3.4: F, the input gradient B and the weight gradient W):
//   warp 0      one thread issues TMA tensor copies of A/B tiles into a
//               4-stage shared-memory ring (128-byte swizzle);
//   warp 1      allocates 512 TMEM columns and one thread issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) into one of
//               two 256-column accumulators, committing each stage back to
//               the producer and each finished tile to the epilogue;
//   warps 2..5  drain the accumulator with tcgen05.ld (one TMEM lane = one
//               output row per thread) and apply the epilogue: bf16 store,
//               bias + GeLU dual store (H and A), GeLU' product with the
//               saved H (dH), or fp32 accumulation of a weight gradient.
//               Results leave through swizzled shared-memory staging boxes
//               and TMA tensor stores; the weight gradient is added in place
//               with a TMA reduce-add (one fp32 add per element, in L2).
// The two accumulators let the epilogue of tile t overlap the MMAs of t+1.
// Tiles are visited in a fixed order (tile = blockIdx.x + i * gridDim.x,
// grouped rasterisation, see tile_coords) and K is never split, so results
// are deterministic.
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel sets the
// device error word, drains its in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "ptx.cuh"
#include "zb_internal.h"

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;          // 16 KiB
constexpr uint32_t B_BYTES = BN * BK * 2;          // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t MN_ATOM_BYTES = 64 * BK * 2;    // 64 MN x 64 K, one TMA box
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;  // 4 s
constexpr uint64_t DRAIN_LIMIT_NS = 500000000ull;  // 0.5 s

constexpr uint32_t STAGING_BOX = 32 * 128;                 // 32 rows x 128 bytes
constexpr uint32_t STAGING_BYTES = 4 * 2 * STAGING_BOX;      // 2 boxes per epilogue warp

struct SharedCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + sizeof(SharedCtl) + 64;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

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
    unsigned int* err;
};

// error-word bits
constexpr unsigned ERR_WAIT_PRODUCER = 1u << 0;
constexpr unsigned ERR_WAIT_MMA = 1u << 1;
constexpr unsigned ERR_WAIT_EPI = 1u << 2;

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err, unsigned code, uint64_t limit_ns,
                                         bool honour_abort) {
    if (zbp::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = zbp::globaltimer_ns();
    uint32_t spins = 0;
    while (true) {
        if (zbp::mbar_try_wait(bar, parity)) return true;
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

__device__ __forceinline__ float gelu_f(float x, int act) {
    if (act == ZB_ACT_GELU_TANH) {
        const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
        return 0.5f * x * (1.0f + tanhf(u));
    }
    return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f));
}

__device__ __forceinline__ float gelu_grad_f(float x, int act) {
    if (act == ZB_ACT_GELU_TANH) {
        const float x2 = x * x;
        const float t = tanhf(0.7978845608028654f * (x + 0.044715f * x * x2));
        return 0.5f * (1.0f + t) +
               0.5f * x * (1.0f - t * t) * 0.7978845608028654f * (1.0f + 3.0f * 0.044715f * x2);
    }
    // Phi(x) + x phi(x)
    return 0.5f * (1.0f + erff(x * 0.7071067811865476f)) +
           x * 0.3989422804014327f * expf(-0.5f * x * x);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}

// Tile order: groups of GROUP_M M-blocks; inside a group M is fastest, then
// N.  A wave of resident CTAs then covers about GROUP_M x (grid / GROUP_M)
// tiles, so the operand panels it touches at each K step are few and shared
// from L2 (M-fastest over a tall problem would stream a new A panel per CTA).
constexpr int GROUP_M = 16;

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& mb, int& nb) {
    const int per_group = GROUP_M * tiles_n;
    const int g = tile / per_group;
    const int first = g * GROUP_M;
    const int gsz = min(tiles_m - first, GROUP_M);
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

// Lane 0 makes sure the staging buffer about to be written is no longer read
// by the bulk store issued two stores ago (buffers alternate).
__device__ __forceinline__ void staging_acquire(int lane) {
    if (lane == 0) zbp::bulk_wait_read<1>();
    __syncwarp();
}

// Hand a filled staging buffer to the TMA unit.
template <bool REDUCE>
__device__ __forceinline__ void staging_release(const CUtensorMap* tm, uint32_t stg, int lane,
                                                int x, int y) {
    zbp::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (REDUCE)
            zbp::tma_reduce_add_2d(tm, stg, x, y);
        else
            zbp::tma_store_2d(tm, stg, x, y);
        zbp::bulk_commit();
    }
}

template <int EPI, int A_MN, int B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    zb_gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmO0,
                           const __grid_constant__ CUtensorMap tmO1, const EpiArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * STAGE_BYTES;
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(staging + STAGING_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (args.Mg + BM - 1) / BM;
    const int tiles_n = (args.Ng + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = (args.Kg + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            zbp::mbar_init(zbp::smem_u32(&ctl->full[s]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            zbp::mbar_init(zbp::smem_u32(&ctl->tfull[b]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->tempty[b]), 4);
        }
        zbp::mbar_init(zbp::smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        zbp::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        zbp::tma_prefetch_desc(&tmA);
        zbp::tma_prefetch_desc(&tmB);
        zbp::tma_prefetch_desc(&tmO0);
        if (EPI == zb::EPI_GELU_DUAL) zbp::tma_prefetch_desc(&tmO1);
    }
    if (warp == 1) {
        zbp::tmem_alloc(zbp::smem_u32(&ctl->tmem_base), TMEM_COLS);
        zbp::tmem_relinquish();
    }
    zbp::tc_fence_before();
    __syncthreads();
    zbp::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, tiles_m, tiles_n, mb, nb);
                const int m0 = mb * BM;
                const int n0 = nb * BN;
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t r = it / STAGES;
                    if (!wait_bar(zbp::smem_u32(&ctl->empty[s]), (r & 1u) ^ 1u, abort_flag,
                                  args.err, ERR_WAIT_PRODUCER, WAIT_LIMIT_NS, true)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = zbp::smem_u32(&ctl->full[s]);
                    const uint32_t sa = zbp::smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const int k0 = kb * BK;
                    zbp::mbar_arrive_expect_tx(full, STAGE_BYTES);
                    if (A_MN) {
                        zbp::tma_load_2d(sa, &tmA, full, m0, k0);
                        zbp::tma_load_2d(sa + MN_ATOM_BYTES, &tmA, full, m0 + 64, k0);
                    } else {
                        zbp::tma_load_2d(sa, &tmA, full, k0, m0);
                    }
                    if (B_MN) {
#pragma unroll
                        for (int i = 0; i < BN / 64; ++i)
                            zbp::tma_load_2d(sb + i * MN_ATOM_BYTES, &tmB, full, n0 + 64 * i, k0);
                    } else {
                        zbp::tma_load_2d(sb, &tmB, full, k0, n0);
                    }
                }
            }
            if (!ok) {
                // wait for the copies that were issued but may not have landed
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t i = first; i < it; ++i) {
                    wait_bar(zbp::smem_u32(&ctl->full[i % STAGES]), (i / STAGES) & 1u, abort_flag,
                             args.err, ERR_WAIT_PRODUCER, DRAIN_LIMIT_NS, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = zbp::idesc_bf16_f32(BM, BN, A_MN, B_MN);
            uint32_t it = 0;
            uint32_t local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t buf = local & 1u;
                const uint32_t tr = local >> 1;
                if (!wait_bar(zbp::smem_u32(&ctl->tempty[buf]), (tr & 1u) ^ 1u, abort_flag,
                              args.err, ERR_WAIT_MMA, WAIT_LIMIT_NS, true)) {
                    ok = false;
                    break;
                }
                zbp::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * ACC_COLS;
                for (int kb = 0; kb < num_kb; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t r = it / STAGES;
                    if (!wait_bar(zbp::smem_u32(&ctl->full[s]), r & 1u, abort_flag, args.err,
                                  ERR_WAIT_MMA, WAIT_LIMIT_NS, true)) {
                        ok = false;
                        break;
                    }
                    zbp::tc_fence_after();
                    const uint32_t sa = zbp::smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // K-major: 16 K-elements = 32 bytes inside the 128-B swizzle row;
                        // MN-major: 16 K-rows of 128 bytes = 2048 bytes.
                        const uint64_t ad =
                            A_MN ? zbp::smem_desc_sw128(sa + kk * 2048, MN_ATOM_BYTES, 1024)
                                 : zbp::smem_desc_sw128(sa + kk * 32, 16, 1024);
                        const uint64_t bd =
                            B_MN ? zbp::smem_desc_sw128(sb + kk * 2048, MN_ATOM_BYTES, 1024)
                                 : zbp::smem_desc_sw128(sb + kk * 32, 16, 1024);
                        zbp::tc_mma_f16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    zbp::tc_commit(zbp::smem_u32(&ctl->empty[s]));
                }
                if (!ok) break;
                zbp::tc_commit(zbp::smem_u32(&ctl->tfull[buf]));
            }
            // every MMA issued here completes before TMEM is released
            zbp::tc_commit(zbp::smem_u32(&ctl->drain));
            wait_bar(zbp::smem_u32(&ctl->drain), 0, abort_flag, args.err, ERR_WAIT_MMA,
                     DRAIN_LIMIT_NS, false);
        }
    } else {
        // ---------------------------------------------------- epilogue
        // Warp w may read TMEM lanes 32*(w%4) .. +31: rows q*32 .. q*32+31 of
        // the tile, one row per thread.  Results leave through two 4-KiB
        // swizzled staging boxes per warp (32 rows x 128 bytes) and TMA
        // stores; the fp32 weight gradient is accumulated with a TMA
        // reduce-add, so the old values are never read by the SM.
        const int q = warp & 3;
        const uint32_t stg0 = zbp::smem_u32(staging + (warp - 2) * 2 * STAGING_BOX);
        uint32_t flip = 0;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const uint32_t buf = local & 1u;
            const uint32_t tr = local >> 1;
            int mb, nb;
            tile_coords(tile, tiles_m, tiles_n, mb, nb);
            const int m0 = mb * BM;
            const int n0 = nb * BN;
            const int row0 = m0 + q * 32;
            const int row = row0 + lane;
            if (EPI == zb::EPI_GELU_BWD && row < args.Mg) {
                // warm L2 with this row of H while the MMAs run
                const int ncols = min(BN, args.Ng - n0);
                zbp::prefetch_l2(args.aux + static_cast<long long>(row) * args.ldaux + n0,
                                 static_cast<uint32_t>(ncols) * 2u);
            }
            if (!wait_bar(zbp::smem_u32(&ctl->tfull[buf]), tr & 1u, abort_flag, args.err,
                          ERR_WAIT_EPI, WAIT_LIMIT_NS, true))
                break;
            zbp::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * ACC_COLS;
            const bool rows_live = row0 < args.Mg;
            if (EPI == zb::EPI_F32) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    zbp::tmem_ld_32x32b_x32(taddr + c * 32, v);
                    zbp::tmem_ld_wait();
                    const int col0 = n0 + c * 32;
                    if (!rows_live || col0 >= args.Ng) continue;
                    const uint32_t stg = stg0 + flip * STAGING_BOX;
                    flip ^= 1u;
                    staging_acquire(lane);
                    stage_row(stg, lane, v);
                    if (args.accumulate)
                        staging_release<true>(&tmO0, stg, lane, col0, row0);
                    else
                        staging_release<false>(&tmO0, stg, lane, col0, row0);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t v0[32], v1[32];
                    zbp::tmem_ld_32x32b_x32(taddr + c * 64, v0);
                    zbp::tmem_ld_32x32b_x32(taddr + c * 64 + 32, v1);
                    zbp::tmem_ld_wait();
                    const int col0 = n0 + c * 64;
                    if (!rows_live || col0 >= args.Ng) continue;
                    float x[64];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        x[i] = __uint_as_float(v0[i]);
                        x[32 + i] = __uint_as_float(v1[i]);
                    }
                    if ((EPI == zb::EPI_STORE_BF16 || EPI == zb::EPI_GELU_DUAL) && args.bias) {
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            if (col0 + g * 8 >= args.Ng) break;
                            const uint4 b = *reinterpret_cast<const uint4*>(args.bias + col0 + g * 8);
                            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f2 = unpack_bf16x2(bw[i]);
                                x[g * 8 + 2 * i] += f2.x;
                                x[g * 8 + 2 * i + 1] += f2.y;
                            }
                        }
                    }
                    if (EPI == zb::EPI_GELU_BWD && row < args.Mg) {
                        const __nv_bfloat16* hp = args.aux + static_cast<long long>(row) * args.ldaux + col0;
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            if (col0 + g * 8 >= args.Ng) break;
                            const uint4 hv = *reinterpret_cast<const uint4*>(hp + g * 8);
                            const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f2 = unpack_bf16x2(hw[i]);
                                x[g * 8 + 2 * i] *= gelu_grad_f(f2.x, args.act);
                                x[g * 8 + 2 * i + 1] *= gelu_grad_f(f2.y, args.act);
                            }
                        }
                    }
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
                    uint32_t stg = stg0 + flip * STAGING_BOX;
                    flip ^= 1u;
                    staging_acquire(lane);
                    stage_row(stg, lane, w);
                    staging_release<false>(&tmO0, stg, lane, col0, row0);
                    if (EPI == zb::EPI_GELU_DUAL) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            w[i] = pack_bf16x2(gelu_f(x[2 * i], args.act), gelu_f(x[2 * i + 1], args.act));
                        stg = stg0 + flip * STAGING_BOX;
                        flip ^= 1u;
                        staging_acquire(lane);
                        stage_row(stg, lane, w);
                        staging_release<false>(&tmO1, stg, lane, col0, row0);
                    }
                }
            }
            zbp::tc_fence_before();
            __syncwarp();
            if (lane == 0) zbp::mbar_arrive(zbp::smem_u32(&ctl->tempty[buf]));
        }
        // the staging buffers must not be released while a bulk store reads them
        if (lane == 0) zbp::bulk_wait<0>();
        __syncwarp();
    }

    __syncthreads();
    if (warp == 1) {
        zbp::tc_fence_after();
        zbp::tmem_dealloc(tmem_base, TMEM_COLS);
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
// elements; box of box_inner x box_outer elements, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, bool f32, uint64_t inner, uint64_t outer,
              uint64_t ld, uint32_t box_inner, uint32_t box_outer, std::string* why) {
    EncodeTiledFn fn = encode_fn(why);
    if (!fn) return false;
    const uint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * es};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n;
    }
    return cache[dev];
}

template <int EPI, int A_MN, int B_MN>
zb_status launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to0,
                 const CUtensorMap& to1, const EpiArgs& ea, int grid, cudaStream_t st) {
    auto kern = zb_gemm_bf16_tc_kernel<EPI, A_MN, B_MN>;
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SMEM_BYTES));
        if (e != cudaSuccess)
            return zb::fail(ZB_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
        configured[dev] = 1;
    }
    kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ta, tb, to0, to1, ea);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return zb::fail(ZB_ERR_CUDA, std::string("tensor-core GEMM launch: ") + cudaGetErrorString(e));
    return ZB_OK;
}

template <int EPI>
zb_status dispatch_major(int a_mn, int b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& to0, const CUtensorMap& to1, const EpiArgs& ea,
                         int grid, cudaStream_t st) {
    if (!a_mn && !b_mn) return launch<EPI, 0, 0>(ta, tb, to0, to1, ea, grid, st);
    if (!a_mn && b_mn) return launch<EPI, 0, 1>(ta, tb, to0, to1, ea, grid, st);
    if (a_mn && !b_mn) return launch<EPI, 1, 0>(ta, tb, to0, to1, ea, grid, st);
    return launch<EPI, 1, 1>(ta, tb, to0, to1, ea, grid, st);
}

}  // namespace

namespace zb {

zb_status gemm_bf16_tc(const GemmBf16& g, void* stream) {
    if (g.Mg <= 0 || g.Ng <= 0 || g.Kg <= 0 || g.Mg > (1LL << 30) || g.Ng > (1LL << 30) ||
        g.Kg > (1LL << 30))
        return fail(ZB_ERR_SHAPE, "GEMM extents must be in [1, 2^30]");
    if (g.Ng % 8 != 0) return fail(ZB_ERR_ALIGN, "GEMM N must be a multiple of 8");
    if ((g.lda % 8) || (g.ldb % 8) || (g.ld0 % 8) || (g.out1 && g.ld1 % 8) || (g.aux && g.ldaux % 8))
        return fail(ZB_ERR_ALIGN, "leading dimensions must be multiples of 8 elements");
    auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (mis(g.A) || mis(g.B) || mis(g.out0) || mis(g.out1) || mis(g.aux) || mis(g.bias))
        return fail(ZB_ERR_ALIGN, "GEMM pointers must be 16-byte aligned");
    if (!g.A || !g.B || !g.out0) return fail(ZB_ERR_INVALID_ARG, "GEMM operand is NULL");
    if (g.epi == EPI_GELU_DUAL && !g.out1) return fail(ZB_ERR_INVALID_ARG, "GeLU dual store needs out1");
    if (g.epi == EPI_GELU_BWD && !g.aux) return fail(ZB_ERR_INVALID_ARG, "GeLU' epilogue needs H");

    std::string why;
    CUtensorMap ta, tb, to0, to1;
    bool ok;
    if (g.a_mn)
        ok = make_map(&ta, g.A, false, g.Mg, g.Kg, g.lda, 64, BK, &why);
    else
        ok = make_map(&ta, g.A, false, g.Kg, g.Mg, g.lda, BK, BM, &why);
    if (ok) {
        if (g.b_mn)
            ok = make_map(&tb, g.B, false, g.Ng, g.Kg, g.ldb, 64, BK, &why);
        else
            ok = make_map(&tb, g.B, false, g.Kg, g.Ng, g.ldb, BK, BN, &why);
    }
    // epilogue boxes: 32 rows x 128 bytes (32 fp32 or 64 bf16 columns)
    const bool f32_out = g.epi == EPI_F32;
    const uint32_t ocols = f32_out ? 32 : 64;
    if (ok) ok = make_map(&to0, g.out0, f32_out, g.Ng, g.Mg, g.ld0, ocols, 32, &why);
    if (ok) {
        if (g.epi == EPI_GELU_DUAL)
            ok = make_map(&to1, g.out1, false, g.Ng, g.Mg, g.ld1, ocols, 32, &why);
        else
            to1 = to0;
    }
    if (!ok) return fail(ZB_ERR_CUDA, why);
    if (f32_out && (g.ld0 % 4)) return fail(ZB_ERR_ALIGN, "fp32 output leading dimension must be a multiple of 4");

    unsigned int* err = device_error_word();
    if (!err) return ZB_ERR_CUDA;

    EpiArgs ea;
    ea.Mg = static_cast<int>(g.Mg);
    ea.Ng = static_cast<int>(g.Ng);
    ea.Kg = static_cast<int>(g.Kg);
    ea.out0 = g.out0;
    ea.ld0 = g.ld0;
    ea.out1 = g.out1;
    ea.ld1 = g.ld1;
    ea.aux = static_cast<const __nv_bfloat16*>(g.aux);
    ea.ldaux = g.ldaux;
    ea.bias = static_cast<const __nv_bfloat16*>(g.bias);
    ea.accumulate = g.accumulate;
    ea.act = g.act;
    ea.err = err;

    const long long tiles = ((g.Mg + BM - 1) / BM) * ((g.Ng + BN - 1) / BN);
    const int sms = sm_count();
    if (sms <= 0) return fail(ZB_ERR_CUDA, "cannot query the SM count");
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (g.epi) {
        case EPI_STORE_BF16: return dispatch_major<EPI_STORE_BF16>(g.a_mn, g.b_mn, ta, tb, to0, to1, ea, grid, st);
        case EPI_GELU_DUAL: return dispatch_major<EPI_GELU_DUAL>(g.a_mn, g.b_mn, ta, tb, to0, to1, ea, grid, st);
        case EPI_GELU_BWD: return dispatch_major<EPI_GELU_BWD>(g.a_mn, g.b_mn, ta, tb, to0, to1, ea, grid, st);
        case EPI_F32: return dispatch_major<EPI_F32>(g.a_mn, g.b_mn, ta, tb, to0, to1, ea, grid, st);
        default: return fail(ZB_ERR_INVALID_ARG, "unknown epilogue");
    }
}

}  // namespace zb
