// gemm_tc.cu — bf16 tensor-core GEMM for sm_103a with fused epilogues.
//
// One persistent, warp-specialised kernel computes every contraction of the
// split MLP block (the three passes of "Zero Bubble Pipeline Parallelism",
// summary §3.4: F, the input gradient B and the weight gradient W):
//   warp 0      one thread issues TMA tensor copies of A/B tiles into a
//               shared-memory ring (128-byte swizzle);
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (bf16 -> fp32) into one of two 256-column accumulators,
//               committing each stage back to the producer and each
//               finished tile to the epilogue;
//   warps 2..9  drain the accumulator with tcgen05.ld (one TMEM lane = one
//               output row per thread; 8 warps for the bf16 epilogues, two
//               per lane quadrant, 4 for the fp32 one) and apply the
//               epilogue: bf16 store, bias + GeLU dual store (H and A),
//               GeLU' product with the saved H (dH), or fp32 accumulation
//               of a weight gradient.
//               Results leave through swizzled shared-memory staging boxes
//               and TMA tensor stores; the weight gradient is added in place
//               with a TMA reduce-add (one fp32 add per element, in L2).
// The two accumulators let the epilogue of tile t overlap the MMAs of t+1.
// Warp w runs on SM sub-partition w mod 4 and may read only TMEM lane
// quadrant w mod 4, so the epilogue warps of quadrants 0 and 1 share their
// schedulers with the producer and MMA-issuer warps.  For the GeLU and
// GeLU' epilogues of long-K problems (HAND, K >= 64 blocks) those four
// warps only copy raw fp32 chunks from TMEM into shared memory, and the
// warps of quadrants 2 and 3 do the arithmetic and stores of all rows.
//
// Two CTA-group shapes share the code:
//   CG = 1  one CTA per 128x256 tile (M=128, N=256 MMAs), 4 stages of 48 KB;
//   CG = 2  a cluster of two CTAs on two SMs per 256x256 tile: each CTA
//           loads its 128 rows of A and half (128 columns) of B, the even
//           CTA issues M=256, N=256 MMAs (tcgen05 cta_group::2) that write
//           each CTA's 128 rows into its own TMEM; 6 stages of 32 KB, half
//           the B traffic per SM.  Copies of both CTAs complete on the even
//           CTA's barriers; MMA completion is multicast back to both.
// Tiles are visited in a fixed order (tile = cluster + i * clusters, grouped
// rasterisation, see tile_coords), so results are deterministic for a given
// shape.
// Split K (CG = 1 only, bf16-output epilogues): when a problem has too few
// tiles to occupy the SMs, a cluster of S CTAs (S = 2 or 4) computes one
// 128x256 tile, CTA r over the r-th of S contiguous K ranges.  CTA r owns
// columns [r 256/S, (r+1) 256/S) of the tile.  Each CTA writes its fp32
// partial into its own (then idle) operand ring as S slabs, one per owner;
// after a cluster barrier (every ring idle, every partial written) each CTA
// sends slab o to CTA o with one bulk copy through distributed shared memory
// (the copy engine moves it; completion counted in bytes on CTA o's
// mbarrier).  CTA o then sums its S slabs from its own shared memory in rank
// order 0..S-1 (a fixed order, so the result is still deterministic),
// applies the epilogue and stores it.  No global workspace is involved.
// Launched as a programmatic dependent of the previous GEMM in a stream, a
// CTA runs its setup early and waits (griddepcontrol.wait) before its first
// global access; a GEMM that touches nothing the previous one writes (the W
// pass's second, when it has a launch of its own) waits only before it
// exits, and runs beside that one.  By default the W pass's two GEMMs share
// one launch instead (fp32 epilogue, CTA pairs): the second problem's tiles
// follow the first's in the same persistent grid.
// Every TMA copy carries an L2 eviction priority chosen per operand from
// the raster order's re-reads (choose_l2_hints).
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel sets the
// device error word, drains its in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ptx.cuh"
#include "zb_internal.h"

#include "gemm_core.cuh"

namespace {

// ---------------------------------------------------------------- split K
// GeLU and GeLU' of an element pair (exact-erf form), as in the tile epilogue.
__device__ __forceinline__ f32x2 gelu_pair(f32x2 X) {
    f32x2 PHI, E;
    normal_cdf_and_exp2(X, PHI, E);
    return mul2(X, PHI);
}
__device__ __forceinline__ f32x2 gelu_grad_pair(f32x2 H) {
    f32x2 PHI, E;
    normal_cdf_and_exp2(H, PHI, E);
    return fma2(mul2(H, pk2(0.3989422804014327f, 0.3989422804014327f)), E, PHI);
}

// The epilogue of one row's 4 consecutive columns (col a multiple of 4, all
// four inside the matrix), from their fp32 sums.
template <int EPI>
__device__ __forceinline__ void epilogue4(const EpiArgs& args, int row, int col, float (&x)[4]) {
    if ((EPI == zb::EPI_STORE_BF16 || EPI == zb::EPI_GELU_DUAL) && args.bias) {
        const uint2 b = *reinterpret_cast<const uint2*>(args.bias + col);
        const float2 b0 = unpack_bf16x2(b.x), b1 = unpack_bf16x2(b.y);
        x[0] += b0.x;
        x[1] += b0.y;
        x[2] += b1.x;
        x[3] += b1.y;
    }
    if (EPI == zb::EPI_GELU_BWD) {
        const uint2 hv =
            *reinterpret_cast<const uint2*>(args.aux + static_cast<long long>(row) * args.ldaux + col);
        const float2 h0 = unpack_bf16x2(hv.x), h1 = unpack_bf16x2(hv.y);
        if (args.act == ZB_ACT_GELU_TANH) {
            x[0] *= gelu_grad_t<true>(h0.x);
            x[1] *= gelu_grad_t<true>(h0.y);
            x[2] *= gelu_grad_t<true>(h1.x);
            x[3] *= gelu_grad_t<true>(h1.y);
        } else {
            up2(mul2(pk2(x[0], x[1]), gelu_grad_pair(pk2(h0.x, h0.y))), x[0], x[1]);
            up2(mul2(pk2(x[2], x[3]), gelu_grad_pair(pk2(h1.x, h1.y))), x[2], x[3]);
        }
    }
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(args.out0) + static_cast<long long>(row) * args.ld0 +
                              col) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    if (EPI == zb::EPI_GELU_DUAL) {
        float g[4];
        if (args.act == ZB_ACT_GELU_TANH) {
#pragma unroll
            for (int i = 0; i < 4; ++i) g[i] = gelu_t<true>(x[i]);
        } else {
            up2(gelu_pair(pk2(x[0], x[1])), g[0], g[1]);
            up2(gelu_pair(pk2(x[2], x[3])), g[2], g[3]);
        }
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(args.out1) +
                                  static_cast<long long>(row) * args.ld1 + col) =
            make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]));
    }
}

// Split-K layout in a CTA's shared memory (ring and staging area, 224 KiB):
// its own partial tile as ks slabs at slab o (the columns CTA o owns), then
// ks - 1 receive slots, slot(r) for the slab that CTA r sends.  A slab holds
// 128 rows of 1024/ks bytes, 16-byte chunk j of row i at chunk j ^ (i mod 8)
// (a row has at least 8 chunks, so the swizzle stays inside it; the rows
// written by the 8 lanes of a quarter-warp, or the chunks read by 8
// consecutive threads, hit 8 different bank groups).
constexpr uint32_t SPLIT_PARTIAL_BYTES = BM * 1024u;  // one fp32 128 x 256 tile
constexpr int SPLIT_MAX = 4;
__host__ __device__ constexpr uint32_t split_slab_bytes(int ks) {
    return SPLIT_PARTIAL_BYTES / static_cast<uint32_t>(ks);
}
static_assert(SPLIT_PARTIAL_BYTES + (SPLIT_MAX - 1) * split_slab_bytes(SPLIT_MAX) <=
                  Cfg<1>::STAGES * Cfg<1>::STAGE_BYTES + STAGING_BYTES,
              "split-K slabs and receive slots fit in the ring and staging area");
__device__ __forceinline__ uint32_t split_chunk_offset(int ks, int row, int j) {
    return static_cast<uint32_t>(row) * (1024u / static_cast<uint32_t>(ks)) +
           (static_cast<uint32_t>(j ^ (row & 7)) << 4);
}
// receive slot of the slab from CTA r in CTA `owner` (r != owner)
__device__ __forceinline__ uint32_t split_recv_offset(int ks, int r, int owner) {
    return SPLIT_PARTIAL_BYTES + static_cast<uint32_t>(r < owner ? r : r - 1) * split_slab_bytes(ks);
}

// CTA `kslice` of a split-K cluster: sums its 256/ks columns of the tile at
// (m0, n0) over the ks slabs in its shared memory (from `base`) in rank
// order, then applies the epilogue.  Consecutive threads take consecutive
// 16-byte chunks of a row (coalesced global stores); each thread carries
// SPLIT_ILP chunks at once (loads first), so that the loop is not one
// dependent chain of shared loads, adds and GeLU per chunk.
constexpr int SPLIT_ILP = 4;
template <int EPI>
__device__ __forceinline__ void split_reduce_store(const EpiArgs& args_in, uint32_t base, int ks,
                                                   int kslice, int m0, int n0) {
    const EpiArgs args = args_in;
    const int lg = ks == 2 ? 5 : 4;  // log2 of the chunks per owned row (ks = 2, 4)
    const int items = BM << lg;
    uint32_t src[SPLIT_MAX];
#pragma unroll
    for (int q = 0; q < SPLIT_MAX; ++q)
        src[q] = base + (q == kslice ? static_cast<uint32_t>(kslice) * split_slab_bytes(ks)
                                     : split_recv_offset(ks, q, kslice));
    const int col0 = n0 + kslice * (BN / ks);
    for (int i0 = threadIdx.x; i0 < items; i0 += SPLIT_ILP * NUM_THREADS) {
        float x[SPLIT_ILP][4];
        bool live[SPLIT_ILP];
#pragma unroll
        for (int u = 0; u < SPLIT_ILP; ++u) {
            const int i = i0 + u * NUM_THREADS;
            const int r = i >> lg;
            const int j = i & ((1 << lg) - 1);
            live[u] = i < items && m0 + r < args.Mg && col0 + 4 * j < args.Ng;
            if (live[u]) {
                const uint32_t off = static_cast<uint32_t>(r) * (16u << lg) +
                                     (static_cast<uint32_t>(j ^ (r & 7)) << 4);
                float4 p[SPLIT_MAX];
#pragma unroll
                for (int q = 0; q < SPLIT_MAX; ++q)
                    if (q < ks) p[q] = zbp::ld_shared_v4(src[q] + off);
                x[u][0] = p[0].x;
                x[u][1] = p[0].y;
                x[u][2] = p[0].z;
                x[u][3] = p[0].w;
#pragma unroll
                for (int q = 1; q < SPLIT_MAX; ++q) {
                    if (q < ks) {
                        x[u][0] += p[q].x;
                        x[u][1] += p[q].y;
                        x[u][2] += p[q].z;
                        x[u][3] += p[q].w;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < SPLIT_ILP; ++u) {
            if (live[u]) {
                const int i = i0 + u * NUM_THREADS;
                epilogue4<EPI>(args, m0 + (i >> lg), col0 + 4 * (i & ((1 << lg) - 1)), x[u]);
            }
        }
    }
}

template <int EPI, int A_MN, int B_MN, int CG, int HAND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    zb_gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmO0,
                           const __grid_constant__ CUtensorMap tmO1,
                           const __grid_constant__ CUtensorMap tmA2,
                           const __grid_constant__ CUtensorMap tmB2, const EpiArgs args) {
    using C = Cfg<CG>;
    constexpr int STAGES = C::STAGES;
    constexpr bool PAIR = CG == 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * C::STAGE_BYTES;
    SharedCtl<STAGES>* ctl = reinterpret_cast<SharedCtl<STAGES>*>(staging + STAGING_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // split K: CTAs per tile along K, and this CTA's K range (one tile per cluster)
    constexpr bool SPLITTABLE = !PAIR && EPI != zb::EPI_F32;
    const int ks = SPLITTABLE ? args.ksplit : 1;
    const uint32_t rank = PAIR ? zbp::cluster_ctarank() : 0u;
    const int kslice = ks > 1 ? static_cast<int>(zbp::cluster_ctarank()) : 0;
    const bool leader = rank == 0;
    const int cw = PAIR ? 2 : ks;  // CTAs per cluster
    const int cluster = blockIdx.x / cw;
    const int clusters = gridDim.x / cw;
    const int tiles_m = (args.Mg + C::TILE_M - 1) / C::TILE_M;
    const int tiles_n = (args.Ng + BN - 1) / BN;
    // a second problem (fp32 epilogue, CTA pairs): its tiles follow the first's
    constexpr bool GROUPABLE = EPI == zb::EPI_F32 && PAIR;
    const bool two = GROUPABLE && args.groups > 1;
    const int tiles_1 = tiles_m * tiles_n;
    const int tiles_m2 = two ? (args.Mg2 + C::TILE_M - 1) / C::TILE_M : 0;
    const int tiles_n2 = two ? (args.Ng2 + BN - 1) / BN : 0;
    const int num_tiles = tiles_1 + tiles_m2 * tiles_n2;
    // problem of a tile (0 or 1) and its M / N block inside that problem
    auto locate = [&](int tile, int& mb, int& nb) -> int {
        if (two && tile >= tiles_1) {
            tile_coords(tile - tiles_1, tiles_m2, tiles_n2, C::GROUP_M, mb, nb);
            return 1;
        }
        tile_coords(tile, tiles_m, tiles_n, C::GROUP_M, mb, nb);
        return 0;
    };
    const int num_kb_all = (args.Kg + BK - 1) / BK;
    const int kb_lo = SPLITTABLE ? static_cast<int>(static_cast<long long>(kslice) * num_kb_all / ks) : 0;
    const int kb_hi =
        SPLITTABLE ? static_cast<int>(static_cast<long long>(kslice + 1) * num_kb_all / ks) : num_kb_all;
    const int num_kb = kb_hi - kb_lo;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            zbp::mbar_init(zbp::smem_u32(&ctl->full[s]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            zbp::mbar_init(zbp::smem_u32(&ctl->tfull[b]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->tempty[b]), EpiShape<EPI>::WARPS * CG);
        }
        zbp::mbar_init(zbp::smem_u32(&ctl->drain), 1);
        if (HAND) {
            for (int pp = 0; pp < 4; ++pp) {
                zbp::mbar_init(zbp::smem_u32(&ctl->hfull[pp]), 1);
                zbp::mbar_init(zbp::smem_u32(&ctl->hempty[pp]), 1);
            }
        }
        if (SPLITTABLE) zbp::mbar_init(zbp::smem_u32(&ctl->xchg), 1);
        ctl->abort_flag = 0;
        zbp::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        zbp::tma_prefetch_desc(&tmA);
        zbp::tma_prefetch_desc(&tmB);
        zbp::tma_prefetch_desc(&tmO0);
        if (EPI == zb::EPI_GELU_DUAL || two) zbp::tma_prefetch_desc(&tmO1);
        if (two) {
            zbp::tma_prefetch_desc(&tmA2);
            zbp::tma_prefetch_desc(&tmB2);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            zbp::tmem_alloc_pair(zbp::smem_u32(&ctl->tmem_base), TMEM_COLS);
            zbp::tmem_relinquish_pair();
        } else {
            zbp::tmem_alloc(zbp::smem_u32(&ctl->tmem_base), TMEM_COLS);
            zbp::tmem_relinquish();
        }
    }
    zbp::tc_fence_before();
    __syncthreads();
    if (PAIR) zbp::cluster_sync();  // both CTAs' barriers exist before any remote use
    zbp::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;
    // split K: this CTA receives ks - 1 slabs (before any CTA can send: they
    // send after the phase-1 cluster barrier, which this thread reaches later)
    if (SPLITTABLE && ks > 1 && threadIdx.x == 0)
        zbp::mbar_arrive_expect_tx(zbp::smem_u32(&ctl->xchg), static_cast<uint32_t>(ks - 1) * split_slab_bytes(ks));
    // Launched as a programmatic dependent of the previous GEMM in its stream,
    // the setup above overlaps that GEMM's tail; nothing in global memory is
    // read or written before it has completed.  The next GEMM may then be
    // scheduled at once: its CTAs can only take SMs this grid leaves free
    // (each needs most of an SM's shared memory) and wait there.  A GEMM
    // independent of the previous kernel (late_wait) waits at its exit
    // instead: it runs beside that kernel's tail and still ends after it.
    if (!args.late_wait) zbp::grid_dependency_wait();
    zbp::allow_dependent_launch();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t it = 0;
            bool ok = true;
            const uint64_t pol_a1 = zbp::l2_policy(args.hint_a);
            const uint64_t pol_b1 = zbp::l2_policy(args.hint_b);
            const uint64_t pol_a2 = two ? zbp::l2_policy(args.hint_a2) : pol_a1;
            const uint64_t pol_b2 = two ? zbp::l2_policy(args.hint_b2) : pol_b1;
            for (int tile = cluster; tile < num_tiles && ok; tile += clusters) {
                int mb, nb;
                const int prob = locate(tile, mb, nb);
                const CUtensorMap* tma = prob ? &tmA2 : &tmA;
                const CUtensorMap* tmb = prob ? &tmB2 : &tmB;
                const uint64_t pol_a = prob ? pol_a2 : pol_a1;
                const uint64_t pol_b = prob ? pol_b2 : pol_b1;
                const int m0 = mb * C::TILE_M + static_cast<int>(rank) * BM;
                const int nb0 = nb * BN + static_cast<int>(rank) * C::B_ROWS;
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t r = it / STAGES;
                    if (!wait_bar<PAIR>(zbp::smem_u32(&ctl->empty[s]), (r & 1u) ^ 1u, abort_flag,
                                        args.err, ERR_WAIT_PRODUCER, WAIT_LIMIT_NS, true)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_local = zbp::smem_u32(&ctl->full[s]);
                    const uint32_t full = PAIR ? zbp::mapa_shared(full_local, 0) : full_local;
                    const uint32_t sa = zbp::smem_u32(smem + s * C::STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const int k0 = kb * BK;
                    if (leader) zbp::mbar_arrive_expect_tx(full_local, C::STAGE_BYTES * CG);
                    auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y, uint64_t pol) {
                        if (PAIR)
                            zbp::tma_load_2d_pair_hint(dst, tm, full, x, y, pol);
                        else
                            zbp::tma_load_2d_hint(dst, tm, full, x, y, pol);
                    };
                    if (A_MN) {
                        load(sa, tma, m0, k0, pol_a);
                        load(sa + MN_ATOM_BYTES, tma, m0 + 64, k0, pol_a);
                    } else {
                        load(sa, tma, k0, m0, pol_a);
                    }
                    if (B_MN) {
#pragma unroll
                        for (int i = 0; i < C::B_ROWS / 64; ++i)
                            load(sb + i * MN_ATOM_BYTES, tmb, nb0 + 64 * i, k0, pol_b);
                    } else {
                        load(sb, tmb, k0, nb0, pol_b);
                    }
                }
            }
            if (!ok && leader) {
                // wait for the copies that were issued but may not have landed
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t i = first; i < it; ++i) {
                    wait_bar<PAIR>(zbp::smem_u32(&ctl->full[i % STAGES]), (i / STAGES) & 1u,
                                   abort_flag, args.err, ERR_WAIT_PRODUCER, DRAIN_LIMIT_NS, false);
                }
            }
        }
        if (SPLITTABLE && ks > 1) {
            __syncwarp();
            zbp::cluster_sync();  // split K, phase 1 (see the epilogue)
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = zbp::idesc_bf16_f32(BM * CG, BN, A_MN, B_MN);
            uint32_t it = 0;
            uint32_t local = 0;
            bool ok = true;
            for (int tile = cluster; tile < num_tiles && ok; tile += clusters, ++local) {
                const uint32_t buf = local & 1u;
                const uint32_t tr = local >> 1;
                if (!wait_bar<PAIR>(zbp::smem_u32(&ctl->tempty[buf]), (tr & 1u) ^ 1u, abort_flag,
                                    args.err, ERR_WAIT_MMA, WAIT_LIMIT_NS, true)) {
                    ok = false;
                    break;
                }
                zbp::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * ACC_COLS;
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t r = it / STAGES;
                    if (!wait_bar<PAIR>(zbp::smem_u32(&ctl->full[s]), r & 1u, abort_flag, args.err,
                                        ERR_WAIT_MMA, WAIT_LIMIT_NS, true)) {
                        ok = false;
                        break;
                    }
                    zbp::tc_fence_after();
                    const uint32_t sa = zbp::smem_u32(smem + s * C::STAGE_BYTES);
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
                        const uint32_t acc = (SPLITTABLE ? (kb != kb_lo || kk != 0) : ((kb | kk) != 0)) ? 1u : 0u;
                        if (PAIR)
                            zbp::tc_mma_f16_pair(d_tmem, ad, bd, idesc, acc);
                        else
                            zbp::tc_mma_f16(d_tmem, ad, bd, idesc, acc);
                    }
                    if (PAIR)
                        zbp::tc_commit_pair_multicast(zbp::smem_u32(&ctl->empty[s]), 0x3);
                    else
                        zbp::tc_commit(zbp::smem_u32(&ctl->empty[s]));
                }
                if (!ok) break;
                if (PAIR)
                    zbp::tc_commit_pair_multicast(zbp::smem_u32(&ctl->tfull[buf]), 0x3);
                else
                    zbp::tc_commit(zbp::smem_u32(&ctl->tfull[buf]));
            }
            // every MMA issued here completes before TMEM is released
            if (PAIR)
                zbp::tc_commit_pair(zbp::smem_u32(&ctl->drain));
            else
                zbp::tc_commit(zbp::smem_u32(&ctl->drain));
            wait_bar<PAIR>(zbp::smem_u32(&ctl->drain), 0, abort_flag, args.err, ERR_WAIT_MMA,
                           DRAIN_LIMIT_NS, false);
        }
        if (SPLITTABLE && ks > 1) {
            __syncwarp();
            zbp::cluster_sync();  // split K, phase 1 (see the epilogue)
        }
    } else if (SPLITTABLE && ks > 1) {
        // ---------------------------------------------- split-K epilogue
        // One tile per cluster, in accumulator 0: its fp32 partial goes into
        // this CTA's ring (idle once its MMAs are done) as ks slabs.  Phase 1
        // (cluster barrier): every CTA's slabs are written and every ring is
        // idle, so one thread sends slab o to CTA o with a bulk copy.  The
        // owners sum after their receive barrier (after the role code).
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;  // column half (8 warps: two per lane quadrant)
        const int prow = q * 32 + lane;
        const uint32_t base = zbp::smem_u32(smem);
        const uint32_t slab = split_slab_bytes(ks);
        const bool ok = cluster < num_tiles &&
                        wait_bar<false>(zbp::smem_u32(&ctl->tfull[0]), 0, abort_flag, args.err,
                                        ERR_WAIT_EPI, WAIT_LIMIT_NS, true);
        zbp::tc_fence_after();
        if (ok) {
            const int sw = BN / ks;  // columns per owner
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = hf * 4; c < hf * 4 + 4; c += 2) {
                uint32_t v[2][32];
                zbp::tmem_ld_32x32b_x32(taddr + c * 32, v[0]);
                zbp::tmem_ld_32x32b_x32(taddr + c * 32 + 32, v[1]);
                zbp::tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int o = ((c + h) * 32) / sw;           // owner of these 32 columns
                    const int j0 = ((c + h) * 32 - o * sw) / 4;  // their first chunk in its rows
                    const uint32_t dst = base + static_cast<uint32_t>(o) * slab;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        zbp::st_shared_v4(dst + split_chunk_offset(ks, prow, j0 + k), v[h][4 * k],
                                          v[h][4 * k + 1], v[h][4 * k + 2], v[h][4 * k + 3]);
                }
            }
        }
        zbp::fence_proxy_async_smem();  // the slabs are read by the copy engine next
        __syncwarp();
        zbp::cluster_sync();
        if (ok && warp == 2 && lane == 0) {
            for (int o = 0; o < ks; ++o) {
                if (o == kslice) continue;
                const uint32_t dst = zbp::mapa_shared(base + split_recv_offset(ks, kslice, o), static_cast<uint32_t>(o));
                const uint32_t bar = zbp::mapa_shared(zbp::smem_u32(&ctl->xchg), static_cast<uint32_t>(o));
                zbp::bulk_copy_s2cluster(dst, base + static_cast<uint32_t>(o) * slab, slab, bar);
            }
        }
    } else if constexpr (HAND != 0) {
        // ---------------------------------------- hand-off epilogue (HAND)
        // Lane quadrants 0 and 1 of the accumulator can only be read by warps
        // on schedulers 0 and 1, which also host the TMA-producer and
        // MMA-issuer warps.  So here those warps (4, 5, 8, 9: "readers") only
        // copy raw fp32 chunks from TMEM into shared-memory slots, and the
        // warps on schedulers 2 and 3 (2, 3, 6, 7: "math") apply the GeLU /
        // GeLU' epilogue and store both their own chunks and their partner's
        // (pair p = 2 (q mod 2) + column half: warp 2 takes warp 4's, 3 takes
        // 5's, 6 takes 8's, 7 takes 9's).  One slot per pair: the reader
        // fills chunk c + 1 while its math warp finishes chunk c and its own
        // chunk c + 1.  Every warp arrives on the accumulator's tempty
        // barrier after its last chunk of the tile.
        using E = EpiShape<EPI>;
        constexpr int CH = E::COLS / 32;
        const int ew = warp - 2;
        if (ew < E::WARPS) {
            const int q = warp & 3;
            const int hf = ew >> 2;
            const int c_lo = hf * E::COLS;
            const int pr = (q & 1) * 2 + hf;
            const bool reader = q < 2;
            const uint32_t slot = zbp::smem_u32(staging + HAND_BOXES) + static_cast<uint32_t>(pr) * HAND_SLOT;
            const int mi = hf * 2 + (q & 1);  // math warp index 0..3 (its staging boxes)
            const uint32_t stg0 = zbp::smem_u32(staging) + static_cast<uint32_t>(mi) * 2u * E::BOX;
            const uint64_t pol_out = zbp::l2_policy(args.hint_out);
            uint32_t flip = 0;
            uint32_t local = 0;
            uint32_t k = 0;  // chunks handed off so far (the slot's phase)
            bool ok = true;
            // the GeLU / GeLU' epilogue of one 32-column chunk of row `row`
            // (x: fp32 sums; hw: H for GeLU'), stored from row0c
            auto finish = [&](float (&x)[32], const uint32_t (&hw)[16], int row0c, int col0) {
                if (EPI == zb::EPI_GELU_DUAL && args.bias) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
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
                if (EPI == zb::EPI_GELU_BWD) {
                    if (args.act == ZB_ACT_GELU_TANH)
                        gelu_grad_mul<true, 32>(x, hw);
                    else
                        gelu_grad_mul<false, 32>(x, hw);
                }
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
                uint32_t stg = stg0 + flip * E::BOX;
                flip ^= 1u;
                staging_acquire(lane);
                stage_row64(stg, lane, w);
                staging_release<false>(&tmO0, stg, lane, col0, row0c, pol_out);
                if (EPI == zb::EPI_GELU_DUAL) {
                    if (args.act == ZB_ACT_GELU_TANH)
                        gelu_pack<true, 32>(x, w);
                    else
                        gelu_pack<false, 32>(x, w);
                    stg = stg0 + flip * E::BOX;
                    flip ^= 1u;
                    staging_acquire(lane);
                    stage_row64(stg, lane, w);
                    staging_release<false>(&tmO1, stg, lane, col0, row0c, pol_out);
                }
            };
            for (int tile = cluster; tile < num_tiles && ok; tile += clusters, ++local) {
                const uint32_t buf = local & 1u;
                const uint32_t tr = local >> 1;
                int mb, nb;
                locate(tile, mb, nb);
                const int m0 = mb * C::TILE_M + static_cast<int>(rank) * BM;
                const int n0 = nb * BN;
                if (!reader && EPI == zb::EPI_GELU_BWD) {
                    // warm L2 with this warp's parts of its own and its partner's rows of H
                    const int ncols = min(E::COLS, args.Ng - n0 - c_lo);
                    const int r_own = m0 + q * 32 + lane, r_hand = m0 + (q & 1) * 32 + lane;
                    if (ncols > 0 && r_own < args.Mg)
                        zbp::prefetch_l2(args.aux + static_cast<long long>(r_own) * args.ldaux + n0 + c_lo,
                                         static_cast<uint32_t>(ncols) * 2u);
                    if (ncols > 0 && r_hand < args.Mg)
                        zbp::prefetch_l2(args.aux + static_cast<long long>(r_hand) * args.ldaux + n0 + c_lo,
                                         static_cast<uint32_t>(ncols) * 2u);
                }
                if (!wait_bar<PAIR>(zbp::smem_u32(&ctl->tfull[buf]), tr & 1u, abort_flag, args.err,
                                    ERR_WAIT_EPI, WAIT_LIMIT_NS, true))
                    break;
                zbp::tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * ACC_COLS;
                if (reader) {
#pragma unroll 1
                    for (int c = 0; c < CH; ++c, ++k) {
                        if (!wait_bar<false>(zbp::smem_u32(&ctl->hempty[pr]), (k & 1u) ^ 1u, abort_flag,
                                             args.err, ERR_WAIT_EPI, WAIT_LIMIT_NS, true)) {
                            ok = false;
                            break;
                        }
                        uint32_t v[32];
                        zbp::tmem_ld_32x32b_x32(taddr + c_lo + c * 32, v);
                        zbp::tmem_ld_wait();
                        stage_row(slot, lane, v);  // one 128-byte row per lane, 128-byte swizzle
                        __syncwarp();
                        if (lane == 0) zbp::mbar_arrive(zbp::smem_u32(&ctl->hfull[pr]));
                    }
                } else {
                    const int row0_own = m0 + q * 32, row0_hand = m0 + (q & 1) * 32;
#pragma unroll 1
                    for (int c = 0; c < CH && ok; ++c, ++k) {
                        const int col0 = n0 + c_lo + c * 32;
                        // own chunk, from TMEM
                        {
                            uint32_t hw[16];
                            if (EPI == zb::EPI_GELU_BWD) load_h32(args, row0_own + lane, col0, hw);
                            uint32_t v[32];
                            zbp::tmem_ld_32x32b_x32(taddr + c_lo + c * 32, v);
                            zbp::tmem_ld_wait();
                            float x[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
                            if (row0_own < args.Mg && col0 < args.Ng) finish(x, hw, row0_own, col0);
                        }
                        // the partner's chunk, from its slot
                        {
                            uint32_t hw[16];
                            if (EPI == zb::EPI_GELU_BWD) load_h32(args, row0_hand + lane, col0, hw);
                            if (!wait_bar<false>(zbp::smem_u32(&ctl->hfull[pr]), k & 1u, abort_flag,
                                                 args.err, ERR_WAIT_EPI, WAIT_LIMIT_NS, true)) {
                                ok = false;
                                break;
                            }
                            float x[32];
                            const uint32_t rowa = slot + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 f = zbp::ld_shared_v4(rowa + (static_cast<uint32_t>(j ^ (lane & 7)) << 4));
                                x[4 * j] = f.x;
                                x[4 * j + 1] = f.y;
                                x[4 * j + 2] = f.z;
                                x[4 * j + 3] = f.w;
                            }
                            __syncwarp();
                            if (lane == 0) zbp::mbar_arrive(zbp::smem_u32(&ctl->hempty[pr]));
                            if (row0_hand < args.Mg && col0 < args.Ng) finish(x, hw, row0_hand, col0);
                        }
                    }
                }
                if (!ok) break;
                zbp::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t te = zbp::smem_u32(&ctl->tempty[buf]);
                    if (PAIR)
                        zbp::mbar_arrive_cluster(zbp::mapa_shared(te, 0));
                    else
                        zbp::mbar_arrive(te);
                }
            }
            // the staging buffers must not be released while a bulk store reads them
            if (lane == 0) zbp::bulk_wait<0>();
            __syncwarp();
        }
    } else {
        // ---------------------------------------------------- epilogue
        // Warp w may read TMEM lanes 32*(w%4) .. +31: rows q*32 .. q*32+31 of
        // this CTA's 128 rows, one row per thread; with 8 epilogue warps the
        // two warps of a quadrant take one half of the columns each (see
        // EpiShape).  Results leave through two swizzled staging boxes per
        // warp and TMA stores; the fp32 weight gradient is accumulated with a
        // TMA reduce-add, so the old values are never read by the SM.
        using E = EpiShape<EPI>;
        const int ew = warp - 2;  // epilogue warp index
        if (ew < E::WARPS) {
            const int q = warp & 3;
            const int c_lo = (ew >> 2) * E::COLS;  // first tile column of this warp
            const uint32_t stg0 = zbp::smem_u32(staging + ew * 2 * E::BOX);
            const uint64_t pol_out = zbp::l2_policy(args.hint_out);
            uint32_t flip = 0;
            uint32_t local = 0;
            uint64_t t_prev_full = 0;  // fp32 epilogue: when the previous accumulator was ready
            for (int tile = cluster; tile < num_tiles; tile += clusters, ++local) {
                const uint32_t buf = local & 1u;
                const uint32_t tr = local >> 1;
                int mb, nb;
                const int prob = locate(tile, mb, nb);
                const int Mg_t = prob ? args.Mg2 : args.Mg;  // this tile's problem
                const int Ng_t = prob ? args.Ng2 : args.Ng;
                const CUtensorMap* tmO_t = prob ? &tmO1 : &tmO0;
                const int m0 = mb * C::TILE_M + static_cast<int>(rank) * BM;
                const int n0 = nb * BN;
                const int row0 = m0 + q * 32;
                const int row = row0 + lane;
                // GeLU': the first chunk's H values are loaded while the MMAs
                // run, each next chunk's during the current chunk's arithmetic
                uint32_t h_next[16];
                if (EPI == zb::EPI_GELU_BWD) {
                    if (row < args.Mg && n0 + c_lo < args.Ng) {
                        // warm L2 with this warp's part of the row of H
                        const int ncols = min(E::COLS, args.Ng - n0 - c_lo);
                        zbp::prefetch_l2(args.aux + static_cast<long long>(row) * args.ldaux + n0 + c_lo,
                                         static_cast<uint32_t>(ncols) * 2u);
                    }
                    load_h32(args, row, n0 + c_lo, h_next);
                }
                if (!wait_bar<PAIR>(zbp::smem_u32(&ctl->tfull[buf]), tr & 1u, abort_flag, args.err,
                                    ERR_WAIT_EPI, WAIT_LIMIT_NS, true))
                    break;
                zbp::tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * ACC_COLS;
                const bool rows_live = row0 < Mg_t;
                if (EPI == zb::EPI_F32) {
                    // The fp32 stores (TMA reduce-adds; the L2 reads the old
                    // dW from DRAM for each) share the TMA unit with the
                    // operand loads of the next tile: issued back to back they
                    // queue ahead of those loads and starve the MMAs.  So the
                    // chunks are paced over the next tile's MMAs: chunk c is
                    // issued c x spacing after this accumulator was ready, with
                    // spacing = 5/8 of the previous tile's MMA time (the time
                    // between two accumulators becoming ready) / chunks, so
                    // the reduce-adds spread over ~5/8 of a tile whatever the
                    // clock and K; the first tile assumes 20 ns per K block.
                    // Bounded: at most 20 us between chunks; no pacing on the
                    // CTA's last tile.
                    constexpr int CHUNKS = E::COLS / 32;
                    const bool last_tile = tile + clusters >= num_tiles;
                    uint64_t t_full = 0, spacing = 0;
                    if (lane == 0) {
                        t_full = zbp::globaltimer_ns();
                        spacing = t_prev_full != 0 ? (t_full - t_prev_full) * 5 / (8 * CHUNKS)
                                                   : static_cast<uint64_t>(num_kb) * 20;
                        if (spacing > 20000) spacing = 20000;
                        t_prev_full = t_full;
                    }
#pragma unroll 1
                    for (int c = 0; c < CHUNKS; ++c) {
                        if (c > 0 && !last_tile) {
                            if (lane == 0) {
                                const uint64_t target = t_full + static_cast<uint64_t>(c) * spacing;
                                while (zbp::globaltimer_ns() < target) __nanosleep(64);
                            }
                            __syncwarp();
                        }
                        uint32_t v[32];
                        zbp::tmem_ld_32x32b_x32(taddr + c_lo + c * 32, v);
                        zbp::tmem_ld_wait();
                        const int col0 = n0 + c_lo + c * 32;
                        if (!rows_live || col0 >= Ng_t) continue;
                        const uint32_t stg = stg0 + flip * E::BOX;
                        flip ^= 1u;
                        staging_acquire(lane);
                        stage_row(stg, lane, v);
                        if (args.accumulate)
                            staging_release<true>(tmO_t, stg, lane, col0, row0, pol_out);
                        else
                            staging_release<false>(tmO_t, stg, lane, col0, row0, pol_out);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < E::COLS / 32; ++c) {
                        const int col0 = n0 + c_lo + c * 32;
                        uint32_t hw[16];
                        if (EPI == zb::EPI_GELU_BWD) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) hw[i] = h_next[i];
                            if (c + 1 < E::COLS / 32) load_h32(args, row, col0 + 32, h_next);
                        }
                        uint32_t v[32];
                        zbp::tmem_ld_32x32b_x32(taddr + c_lo + c * 32, v);
                        zbp::tmem_ld_wait();
                        if (!rows_live || col0 >= args.Ng) continue;
                        float x[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
                        if ((EPI == zb::EPI_STORE_BF16 || EPI == zb::EPI_GELU_DUAL) && args.bias) {
#pragma unroll
                            for (int g = 0; g < 4; ++g) {
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
                        if (EPI == zb::EPI_GELU_BWD) {
                            if (args.act == ZB_ACT_GELU_TANH)
                                gelu_grad_mul<true, 32>(x, hw);
                            else
                                gelu_grad_mul<false, 32>(x, hw);
                        }
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
                        uint32_t stg = stg0 + flip * E::BOX;
                        flip ^= 1u;
                        staging_acquire(lane);
                        stage_row64(stg, lane, w);
                        staging_release<false>(&tmO0, stg, lane, col0, row0, pol_out);
                        if (EPI == zb::EPI_GELU_DUAL) {
                            if (args.act == ZB_ACT_GELU_TANH)
                                gelu_pack<true, 32>(x, w);
                            else
                                gelu_pack<false, 32>(x, w);
                            stg = stg0 + flip * E::BOX;
                            flip ^= 1u;
                            staging_acquire(lane);
                            stage_row64(stg, lane, w);
                            staging_release<false>(&tmO1, stg, lane, col0, row0, pol_out);
                        }
                    }
                }
                zbp::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t te = zbp::smem_u32(&ctl->tempty[buf]);
                    if (PAIR)
                        zbp::mbar_arrive_cluster(zbp::mapa_shared(te, 0));
                    else
                        zbp::mbar_arrive(te);
                }
            }
            // the staging buffers must not be released while a bulk store reads them
            if (lane == 0) zbp::bulk_wait<0>();
            __syncwarp();
        }
    }

    __syncthreads();
    if (PAIR) zbp::cluster_sync();  // no remote arrivals or copies remain
    if (SPLITTABLE && ks > 1) {
        // the other CTAs' slabs have landed here (waited for even after an
        // abort, so that no copy still writes this CTA's shared memory once it
        // exits; bounded like every wait)
        const bool got = cluster < num_tiles &&
                         wait_bar<false>(zbp::smem_u32(&ctl->xchg), 0, abort_flag, args.err, ERR_WAIT_EPI,
                                         WAIT_LIMIT_NS, false);
        if (got && !*abort_flag) {
            int mb, nb;
            tile_coords(cluster, tiles_m, tiles_n, C::GROUP_M, mb, nb);
            split_reduce_store<EPI>(args, zbp::smem_u32(smem), ks, kslice, mb * C::TILE_M, nb * BN);
        }
        zbp::cluster_sync();  // phase 2: every copy out of this CTA's slabs has landed
    }
    if (warp == 1) {
        zbp::tc_fence_after();
        if (PAIR)
            zbp::tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            zbp::tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (args.late_wait) zbp::grid_dependency_wait();
}

struct Maps {
    CUtensorMap a, b, o0, o1, a2, b2;  // a2, b2: a grouped launch's second problem
};

// Persistent grid size in CTAs for a CTA-group shape (co-resident clusters x CG).
template <int EPI, int A_MN, int B_MN, int CG, int HAND>
zb_status configure(int* max_ctas) {
    auto kern = zb_gemm_bf16_tc_kernel<EPI, A_MN, B_MN, CG, HAND>;
    // per device; a first call racing another computes the same value
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return zb::fail(ZB_ERR_CUDA, "device ordinal out of range");
    if (!cached[dev].load(std::memory_order_relaxed)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_bytes<CG>()));
        if (e != cudaSuccess)
            return zb::fail(ZB_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
        int n = sm_count();
        if (CG == 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * 256, 1, 1);
            cfg.blockDim = dim3(NUM_THREADS, 1, 1);
            cfg.dynamicSmemBytes = smem_bytes<CG>();
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 2;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (e != cudaSuccess || clusters <= 0)
                return zb::fail(ZB_ERR_UNSUPPORTED, std::string("no co-resident CTA pairs: ") +
                                                        cudaGetErrorString(e));
            n = 2 * clusters;
        }
        cached[dev].store(n, std::memory_order_relaxed);
    }
    *max_ctas = cached[dev].load(std::memory_order_relaxed);
    return ZB_OK;
}

// Co-resident clusters of `ks` one-tile CTAs (split K), per device.
template <int EPI, int A_MN, int B_MN>
int split_clusters(int ks) {
    auto kern = zb_gemm_bf16_tc_kernel<EPI, A_MN, B_MN, 1, 0>;
    static std::atomic<int> cached[64][4];
    int dev = 0;
    cudaGetDevice(&dev);
    const int slot = ks == 2 ? 1 : ks == 4 ? 2 : 3;
    if (dev < 0 || dev >= 64) return 0;
    if (!cached[dev][slot].load(std::memory_order_relaxed)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ks * 64, 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes<1>();
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = ks;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = -1;  // no clusters of this size: never split this far
        }
        cached[dev][slot].store(n, std::memory_order_relaxed);
    }
    return cached[dev][slot].load(std::memory_order_relaxed);
}

template <int EPI, int A_MN, int B_MN, int CG, int HAND>
zb_status launch(const Maps& mp, EpiArgs ea, long long tiles, cudaStream_t st, bool pdl) {
    auto kern = zb_gemm_bf16_tc_kernel<EPI, A_MN, B_MN, CG, HAND>;
    int max_ctas = 0;
    zb_status s = configure<EPI, A_MN, B_MN, CG, HAND>(&max_ctas);
    if (s != ZB_OK) return s;
    // a split pays only while every cluster of its grid is resident at once
    // (one tile each; a second wave of clusters would double the time)
    int ks = (CG == 1 && EPI != zb::EPI_F32) ? ea.ksplit : 1;
    while (ks > 1 && split_clusters<EPI, A_MN, B_MN>(ks) < tiles) ks /= 2;
    ea.ksplit = ks;
    const long long want = tiles * CG;
    const int grid = ks > 1 ? static_cast<int>(tiles * ks) : static_cast<int>(want < max_ctas ? want : max_ctas);
    const int cw = CG == 2 ? 2 : ks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<CG>();
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (cw > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cw;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mp.a, mp.b, mp.o0, mp.o1, mp.a2, mp.b2, ea);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess)
        return zb::fail(ZB_ERR_CUDA, std::string("tensor-core GEMM launch: ") + cudaGetErrorString(e));
    return ZB_OK;
}

template <int EPI, int CG, int HAND = 0>
zb_status dispatch_major(int a_mn, int b_mn, const Maps& mp, const EpiArgs& ea, long long tiles,
                         cudaStream_t st, bool pdl) {
    if (!a_mn && !b_mn) return launch<EPI, 0, 0, CG, HAND>(mp, ea, tiles, st, pdl);
    if (!a_mn && b_mn) return launch<EPI, 0, 1, CG, HAND>(mp, ea, tiles, st, pdl);
    if (a_mn && !b_mn) return launch<EPI, 1, 0, CG, HAND>(mp, ea, tiles, st, pdl);
    return launch<EPI, 1, 1, CG, HAND>(mp, ea, tiles, st, pdl);
}

// The hand-off epilogue (GeLU / GeLU' on CTA pairs): only where a tile's K
// loop outlasts the math warps' doubled epilogue share (K >= 64 blocks).
// ZB_GEMM_HANDOFF=0 in the environment turns it off.
bool use_handoff(const zb::GemmBf16& g) {
    static const bool on = [] {
        const char* v = std::getenv("ZB_GEMM_HANDOFF");
        return !(v && v[0] == '0');
    }();
    return on && (g.Kg + BK - 1) / BK >= 64;
}

template <int CG>
zb_status dispatch(const zb::GemmBf16& g, const Maps& mp, const EpiArgs& ea, long long tiles,
                   cudaStream_t st) {
    const bool pdl = g.allow_pdl != 0;
    const bool hand = CG == 2 && use_handoff(g);
    switch (g.epi) {
        case zb::EPI_STORE_BF16:
            return dispatch_major<zb::EPI_STORE_BF16, CG>(g.a_mn, g.b_mn, mp, ea, tiles, st, pdl);
        case zb::EPI_GELU_DUAL:
            if (hand) return dispatch_major<zb::EPI_GELU_DUAL, 2, 1>(g.a_mn, g.b_mn, mp, ea, tiles, st, pdl);
            return dispatch_major<zb::EPI_GELU_DUAL, CG>(g.a_mn, g.b_mn, mp, ea, tiles, st, pdl);
        case zb::EPI_GELU_BWD:
            if (hand) return dispatch_major<zb::EPI_GELU_BWD, 2, 1>(g.a_mn, g.b_mn, mp, ea, tiles, st, pdl);
            return dispatch_major<zb::EPI_GELU_BWD, CG>(g.a_mn, g.b_mn, mp, ea, tiles, st, pdl);
        case zb::EPI_F32: return dispatch_major<zb::EPI_F32, CG>(g.a_mn, g.b_mn, mp, ea, tiles, st, pdl);
        default: return zb::fail(ZB_ERR_INVALID_ARG, "unknown epilogue");
    }
}

// CTA-group choice.  A pair and two single CTAs cover the same 256 rows on
// the same two SMs, but the pair feeds each SM half of B's bytes (the MMA
// reads the other half from the peer), so the pair is chosen whenever it is
// not worse: always when its tiles fill a wave of pairs, and below that
// unless the one-CTA kernel splits K (the split exchange lives in the
// one-CTA kernel) or M fits in one 128-row block (a pair would compute
// 128 rows of padding).  Measured against choosing the pair only for a full
// wave: the P=4, h=1024 pipeline 1027 -> 1093 TF/s, 8192 x 1024 W +15 %,
// 2048 x 2048 F and B +7 %.  ZB_GEMM_CTA_GROUP=1 or =2 in the environment
// forces one shape.
int choose_cta_group(long long pair_tiles, long long Mg, int ksplit) {
    static const int forced = [] {
        const char* v = std::getenv("ZB_GEMM_CTA_GROUP");
        return (v && (std::strcmp(v, "1") == 0 || std::strcmp(v, "2") == 0)) ? std::atoi(v) : 0;
    }();
    if (forced) return forced;
    const int pairs = sm_count() / 2;
    if (pair_tiles >= pairs) return 2;
    if (ksplit > 1 || Mg <= BM) return 1;
    return 2;
}

// Split-K factor for a one-CTA-per-tile GEMM: the largest S in {2, 4}
// whose S x tiles CTAs fit on the SMs at once with at least min_kb K blocks
// (of 64) per CTA; 1 when the tiles alone fill the GPU or K is short.
// ZB_GEMM_SPLIT_K=1 or 2 in the environment caps S (1 disables it);
// ZB_GEMM_SPLIT_MIN_KB sets min_kb.
int choose_split(long long tiles, long long num_kb) {
    struct Knobs {
        int cap, min_kb;
    };
    static const Knobs knobs = [] {
        Knobs k{SPLIT_MAX, 16};
        const char* v = std::getenv("ZB_GEMM_SPLIT_K");
        const int c = v ? std::atoi(v) : SPLIT_MAX;
        k.cap = (c == 1 || c == 2) ? c : SPLIT_MAX;
        const char* w = std::getenv("ZB_GEMM_SPLIT_MIN_KB");
        if (w && std::atoi(w) > 0) k.min_kb = std::atoi(w);
        return k;
    }();
    const int sms = sm_count();
    int ks = 1;
    for (int s = 2; s <= knobs.cap && s <= SPLIT_MAX; s *= 2)
        if (tiles * s <= sms && num_kb >= static_cast<long long>(knobs.min_kb) * s) ks = s;
    return ks;
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
    if (sm_count() <= 0) return fail(ZB_ERR_CUDA, "cannot query the SM count");

    const long long pair_tiles = ((g.Mg + 2 * BM - 1) / (2 * BM)) * ((g.Ng + BN - 1) / BN);
    const long long tiles = ((g.Mg + BM - 1) / BM) * ((g.Ng + BN - 1) / BN);
    const int ksplit = (g.epi != EPI_F32 && g.allow_split) ? choose_split(tiles, (g.Kg + BK - 1) / BK) : 1;
    const int cg = choose_cta_group(pair_tiles, g.Mg, ksplit);
    const uint32_t b_rows = static_cast<uint32_t>(BN / cg);  // B columns per CTA

    std::string why;
    Maps mp;
    bool ok;
    if (g.a_mn)
        ok = make_map(&mp.a, g.A, false, g.Mg, g.Kg, g.lda, 64, BK, &why);
    else
        ok = make_map(&mp.a, g.A, false, g.Kg, g.Mg, g.lda, BK, BM, &why);
    if (ok) {
        if (g.b_mn)
            ok = make_map(&mp.b, g.B, false, g.Ng, g.Kg, g.ldb, 64, BK, &why);
        else
            ok = make_map(&mp.b, g.B, false, g.Kg, g.Ng, g.ldb, BK, b_rows, &why);
    }
    // epilogue boxes: 32 rows x 32 columns (fp32: 128 bytes, 128-byte
    // swizzle; bf16: 64 bytes, 64-byte swizzle)
    const bool f32_out = g.epi == EPI_F32;
    const CUtensorMapSwizzle osw = f32_out ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (ok) ok = make_map(&mp.o0, g.out0, f32_out, g.Ng, g.Mg, g.ld0, 32, 32, &why, osw);
    if (ok) {
        if (g.epi == EPI_GELU_DUAL)
            ok = make_map(&mp.o1, g.out1, false, g.Ng, g.Mg, g.ld1, 32, 32, &why, osw);
        else
            mp.o1 = mp.o0;
    }
    if (!ok) return fail(ZB_ERR_CUDA, why);
    if (f32_out && (g.ld0 % 4)) return fail(ZB_ERR_ALIGN, "fp32 output leading dimension must be a multiple of 4");
    mp.a2 = mp.a;
    mp.b2 = mp.b;
    const GemmBf16* g2 = g.second;
    if (g2) {
        // a grouped launch: the second problem runs in the same persistent
        // kernel, its tiles after the first's (fp32 epilogue, CTA pairs)
        if (g.epi != EPI_F32 || g2->epi != EPI_F32 || g2->Kg != g.Kg || g2->a_mn != g.a_mn ||
            g2->b_mn != g.b_mn || g2->accumulate != g.accumulate || g2->second || cg != 2)
            return fail(ZB_ERR_INVALID_ARG, "grouped GEMM: the two problems must match (fp32, K, majors)");
        if (g2->Mg <= 0 || g2->Ng <= 0 || g2->Mg > (1LL << 30) || g2->Ng > (1LL << 30))
            return fail(ZB_ERR_SHAPE, "GEMM extents must be in [1, 2^30]");
        if (g2->Ng % 8 || g2->lda % 8 || g2->ldb % 8 || g2->ld0 % 4)
            return fail(ZB_ERR_ALIGN, "grouped GEMM: second problem's extents / leading dimensions");
        if (!g2->A || !g2->B || !g2->out0) return fail(ZB_ERR_INVALID_ARG, "GEMM operand is NULL");
        if (mis(g2->A) || mis(g2->B) || mis(g2->out0)) return fail(ZB_ERR_ALIGN, "GEMM pointers must be 16-byte aligned");
        if (g2->a_mn)
            ok = make_map(&mp.a2, g2->A, false, g2->Mg, g2->Kg, g2->lda, 64, BK, &why);
        else
            ok = make_map(&mp.a2, g2->A, false, g2->Kg, g2->Mg, g2->lda, BK, BM, &why);
        if (ok) {
            if (g2->b_mn)
                ok = make_map(&mp.b2, g2->B, false, g2->Ng, g2->Kg, g2->ldb, 64, BK, &why);
            else
                ok = make_map(&mp.b2, g2->B, false, g2->Kg, g2->Ng, g2->ldb, BK, b_rows, &why);
        }
        if (ok) ok = make_map(&mp.o1, g2->out0, true, g2->Ng, g2->Mg, g2->ld0, 32, 32, &why, osw);
        if (!ok) return fail(ZB_ERR_CUDA, why);
    }

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
    ea.ksplit = 1;
    ea.late_wait = g.independent_of_prev && g.allow_pdl ? 1 : 0;
    choose_l2_hints(g, cg, &ea);
    ea.groups = 1;
    ea.Mg2 = ea.Ng2 = 0;
    ea.hint_a2 = ea.hint_b2 = 0;
    long long tiles_all = pair_tiles;
    if (g2) {
        EpiArgs e2 = ea;
        choose_l2_hints(*g2, cg, &e2);
        ea.groups = 2;
        ea.Mg2 = static_cast<int>(g2->Mg);
        ea.Ng2 = static_cast<int>(g2->Ng);
        ea.hint_a2 = e2.hint_a;
        ea.hint_b2 = e2.hint_b;
        tiles_all += ((g2->Mg + 2 * BM - 1) / (2 * BM)) * ((g2->Ng + BN - 1) / BN);
    }
    ea.err = err;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cg == 2) return dispatch<2>(g, mp, ea, tiles_all, st);
    ea.ksplit = ksplit;
    return dispatch<1>(g, mp, ea, tiles, st);
}

int gemm_bf16_cta_group(const GemmBf16& g) {
    if (sm_count() <= 0 || g.Mg <= 0 || g.Ng <= 0 || g.Kg <= 0) return 1;
    const long long pair_tiles = ((g.Mg + 2 * BM - 1) / (2 * BM)) * ((g.Ng + BN - 1) / BN);
    const long long tiles = ((g.Mg + BM - 1) / BM) * ((g.Ng + BN - 1) / BN);
    const int ksplit = (g.epi != EPI_F32 && g.allow_split) ? choose_split(tiles, (g.Kg + BK - 1) / BK) : 1;
    return choose_cta_group(pair_tiles, g.Mg, ksplit);
}

}  // namespace zb
