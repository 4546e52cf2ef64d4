// replay_tc.cu — one persistent kernel that runs every GEMM of a replayed op
// list (all pipeline stages on one GPU), with the dependencies between the
// GEMMs resolved on the device instead of by stream order.
//
// The executor records the GEMMs that the op list would launch, in list
// order ("jobs").  Job j depends on every earlier job whose byte ranges
// conflict with its own: j reads what it writes, writes what it reads, or
// writes what it writes (an fp32 reduce-add reads and writes its output).
// Any execution that keeps those edges computes what the serial replay
// computes, bit for bit: every tile is the one-launch kernel's tile (256 x
// 256 on a CTA pair, ascending K, the same epilogue arithmetic), and the
// accumulating weight-gradient GEMMs of a stage stay in list order (each
// reads the output the previous one wrote).
//
// The host orders all tiles by a list-scheduling simulation of the
// persistent grid's CTA pairs (estimated tile times; priority to the
// earliest GEMM in list order where most tiles belong to GEMMs of two or
// more waves, else to the longest chain of work after a GEMM).  On the
// device each CTA pair runs its tiles with the one-launch kernel's roles
// (TMA producer, MMA issuer, 8 epilogue warps, two TMEM accumulators), the
// producer's and MMA issuer's K loops instantiated per operand-major pair,
// plus a scheduler warp in the leader CTA.  The scheduler takes the pair's
// next tile of the order (an atomic counter) as soon as the producer has
// started on the current one, reads its entry and job record, and waits
// (bounded) until every job that job depends on has signalled all of its
// tiles: a GPU-scope acquire load of each dependency's completion counter.
// It then hands the entry to the producers, the MMA issuer and the epilogue
// warps of both CTAs through a small ring in shared memory (a cluster-scope
// release / acquire, which carries the acquire on to them), so the
// producer's first loads of a tile follow its last loads of the one before
// without a round trip to global memory in between.  Each epilogue warp
// adds 1 to its job's counter with a release once its tile's stores have
// completed.  Deadlock freedom: in the order every tile comes after every
// tile of the jobs it depends on (the host checks this before every
// launch), and tiles are taken as a prefix of the order, each pair running
// its own in the order taken, so the earliest unfinished tile has been
// taken, its dependencies and its pair's earlier tiles are finished, and it
// can always proceed.
//
// Tables (job records, dependency lists, the tile order; the tensor maps
// too when there are more than fit the launch parameters) go into the
// caller's workspace, written by small kernels that carry them as launch
// parameters, so a replay captured in a CUDA graph holds no pointer to host
// memory.  ZB_REPLAY_TRACE=1 adds per-tile timestamps (TraceRec) at the end
// of the workspace (eager replays).
#include <algorithm>
#include <cstdio>
#include <cstdint>
#include <queue>
#include <string>
#include <unordered_map>
#include <vector>

#include "gemm_core.cuh"

namespace {

constexpr unsigned ERR_WAIT_DEP = 1u << 3;
constexpr int ENTRY_JOB_SHIFT = 18;  // tile-list entry = job << 18 | tile
constexpr uint32_t ENTRY_TILE_MASK = (1u << ENTRY_JOB_SHIFT) - 1u;
constexpr size_t MAX_JOBS = size_t(1) << (32 - ENTRY_JOB_SHIFT);
constexpr int MAX_PAIRS = 128;
constexpr size_t DEPS_PER_JOB = 16;  // table room per job (after reduction)
constexpr int EPI_WARPS = 8;
constexpr uint32_t SIGNALS_PER_TILE = 2 * EPI_WARPS;  // every epilogue warp of both CTAs
// fp32 reduce-adds of a weight-gradient tile: epilogue warp w (0..7) issues
// its chunk c (0..3) (8 c + w) x (K blocks x this) ns after the accumulator
// is ready, so the CTA's 32 reduce-adds of 4 KiB are evenly spaced over about
// half of the tile's MMA time instead of leaving in bursts that queue ahead
// of the operand loads in the TMA unit
constexpr uint64_t PACE_NS_PER_KB = 7;

// One GEMM of the replay as the kernel reads it (global memory).
struct alignas(128) RJob {
    int Mg, Ng, Kg;
    int epi, a_mn, b_mn, act, accumulate;
    int hint_a, hint_b, hint_out;
    int tiles_m, tiles_n;
    int map_a, map_b, map_o0, map_o1;  // indices into the tensor-map table
    int dep0, ndeps;                   // its dependencies: deps[dep0 .. dep0 + ndeps)
    uint32_t target;                   // its counter once every tile has signalled
    long long ldaux;
    const __nv_bfloat16* aux;
    const __nv_bfloat16* bias;
};
static_assert(sizeof(RJob) == 128, "job record");

// Per-tile trace record (ZB_REPLAY_TRACE=1): written at the end of the
// caller's workspace, one per entry of the order.  entry and the simulated
// start come from the host, pair from the kernel (the pair that took the
// tile), and the times (global timer, ns) too, all in the leader CTA:
// when its scheduler took the tile and when the tile's dependencies were
// complete; when its MMA issuer had the accumulator and when it committed
// the last K block; when its first epilogue warp had the accumulator, had
// issued its last store, and signalled the tile.
struct TraceRec {
    uint32_t entry, pair;
    int64_t sim_start;
    uint64_t t_reach, t_ready, t_mma0, t_mma1, t_epi0, t_epi1, t_signal;
};
static_assert(sizeof(TraceRec) == 72, "trace record");

// Up to PARAM_MAPS distinct tensor maps travel in the launch parameters
// (the one-launch kernel's place for them); more stay in global memory.
constexpr int PARAM_MAPS = 240;

struct RParams {
    const CUtensorMap* maps;  // global copy (used when nparam == 0)
    const RJob* jobs;
    const int* deps;
    const uint32_t* entries;  // every tile, in the simulation's start order
    uint32_t* done;           // per job; done[njobs]: this launch's abort word,
                              // done[njobs + 1]: the next entry to hand out
    unsigned int* err;
    TraceRec* trace;          // or nullptr
    int njobs;
    int ntiles;
    int nparam;               // maps held in pmaps below (0: all in global memory)
    CUtensorMap pmaps[PARAM_MAPS];
};
static_assert(sizeof(RParams) <= 32000, "launch parameter size");

// A CTA pair takes its tiles one at a time from the global order (an atomic
// counter); the leader's scheduler warp hands each entry to the pair's other
// roles through a ring of RING slots in both CTAs' shared memory.
constexpr int RING = 4;
constexpr uint32_t RING_READERS = 3 + 2 * EPI_WARPS;  // both producers, MMA issuer, epilogue warps
constexpr int SCHED_WARP = 2 + EPI_WARPS;
constexpr int REPLAY_THREADS = NUM_THREADS + 32;  // the one-launch roles and the scheduler warp
// ring slot's info word: the tile's K-block count and operand majors (with
// the slot's tile coordinates, tensor maps and L2 hints, the producers and
// the MMA issuer read no global memory between tiles)
constexpr uint32_t INFO_KB_MASK = (1u << 28) - 1u;

template <int STAGES>
struct RCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t tfill[RING];  // slot k mod RING holds the pair's k-th entry (both CTAs)
    uint64_t tfree[RING];  // leader CTA: every reader has read the slot
    int tslot[RING];       // index into the order (-1: none left; -2: abort)
    uint32_t tent[RING];   // the order's entry there (job << 18 | tile)
    uint32_t tinfo[RING];  // K blocks | majors << 28
    int tm0[RING];         // the tile's first row (pair) and column
    int tn0[RING];
    uint32_t tmaps[RING];  // operand tensor maps: A | B << 16
    uint32_t thints[RING]; // L2 hints: A | B << 8
    int ptaken;            // leader CTA: entries its producer has taken
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t replay_smem_bytes() {
    return 1024 + Cfg<2>::STAGES * Cfg<2>::STAGE_BYTES + STAGING_BYTES + sizeof(RCtl<Cfg<2>::STAGES>) + 64;
}
static_assert(replay_smem_bytes() <= 232448, "replay kernel shared memory");

// Bounded wait on a local mbarrier phase (cluster-scope acquire where the
// arrivals come from the other CTA of the pair); gives up on this CTA's or
// this launch's abort, or after `limit_ns`.  The launch's abort word (global
// memory) is only read once a wait has lasted 20 us: the producer and MMA
// issuer wait on their barriers all the time, and a global load in that
// loop delays their answer to the barrier.
template <bool CLUSTER>
__device__ __forceinline__ bool rwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      volatile uint32_t* abort_all, unsigned int* err, unsigned code,
                                      uint64_t limit_ns, bool honour_abort) {
    auto poll = [&]() {
        return CLUSTER ? zbp::mbar_try_wait_cluster(bar, parity) : zbp::mbar_try_wait(bar, parity);
    };
    if (poll()) return true;
    const uint64_t t0 = zbp::globaltimer_ns();
    uint32_t spins = 0;
    while (true) {
        if (poll()) return true;
        if ((++spins & 63u) == 0) {
            const uint64_t waited = zbp::globaltimer_ns() - t0;
            if (honour_abort && (*abort_flag || (waited > 20000 && *abort_all))) {
                *abort_flag = 1;
                return false;
            }
            if (waited > limit_ns) {
                *abort_flag = 1;
                *abort_all = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// Bounded wait until every job that job `J` depends on has signalled all of
// its tiles; the calling thread's later global accesses (generic and TMA)
// then see those jobs' results.
__device__ bool wait_deps(const RParams& rp, const RJob* J, volatile int* abort_flag) {
    volatile uint32_t* abort_all = rp.done + rp.njobs;
    const int dep0 = J->dep0, ndeps = J->ndeps;
    for (int i = 0; i < ndeps; ++i) {
        const int d = rp.deps[dep0 + i];
        const uint32_t target = rp.jobs[d].target;
        if (zbp::ld_acquire_gpu(rp.done + d) >= target) continue;
        const uint64_t t0 = zbp::globaltimer_ns();
        uint32_t spins = 0;
        while (zbp::ld_acquire_gpu(rp.done + d) < target) {
            __nanosleep(32);
            if ((++spins & 15u) == 0) {
                if (*abort_flag || *abort_all) {
                    *abort_flag = 1;
                    return false;
                }
                if (zbp::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    *abort_flag = 1;
                    *abort_all = 1;
                    atomicOr(rp.err, ERR_WAIT_DEP);
                    return false;
                }
            }
        }
    }
    zbp::fence_proxy_async_global();
    return true;
}

__device__ __forceinline__ void st_shared_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// The leader's scheduler: the pair's k-th entry (e: index into the order,
// -1: none left; t when e >= 0), published to both
// CTAs' slot k mod RING once every reader has read the slot's previous use.
// What the ring carries for one tile besides its order index.
struct RingTile {
    uint32_t ent, info;  // the order's entry; K blocks | majors << 28
    int m0, n0;          // the pair's first row and column of the tile
    uint32_t maps;       // operand tensor maps: A | B << 16
    uint32_t hints;      // L2 hints of A and B: A | B << 8
};

template <int STAGES>
__device__ __forceinline__ bool ring_publish(RCtl<STAGES>* ctl, uint32_t k, int e, const RingTile& t,
                                             const RParams& rp, volatile int* abort_flag,
                                             volatile uint32_t* abort_all) {
    const uint32_t r = k % RING, use = k / RING;
    if (!rwait<true>(zbp::smem_u32(&ctl->tfree[r]), (use & 1u) ^ 1u, abort_flag, abort_all, rp.err,
                     ERR_WAIT_PRODUCER, WAIT_LIMIT_NS, true))
        return false;
    const uint32_t fill = zbp::smem_u32(&ctl->tfill[r]);
    ctl->tslot[r] = e;
    ctl->tent[r] = t.ent;
    ctl->tinfo[r] = t.info;
    ctl->tm0[r] = t.m0;
    ctl->tn0[r] = t.n0;
    ctl->tmaps[r] = t.maps;
    ctl->thints[r] = t.hints;
    auto remote = [&](const void* p, int v) { st_shared_cluster_s32(zbp::mapa_shared(zbp::smem_u32(p), 1), v); };
    remote(&ctl->tslot[r], e);
    remote(&ctl->tent[r], static_cast<int>(t.ent));
    remote(&ctl->tinfo[r], static_cast<int>(t.info));
    remote(&ctl->tm0[r], t.m0);
    remote(&ctl->tn0[r], t.n0);
    remote(&ctl->tmaps[r], static_cast<int>(t.maps));
    remote(&ctl->thints[r], static_cast<int>(t.hints));
    zbp::mbar_arrive(fill);
    zbp::mbar_arrive_cluster(zbp::mapa_shared(fill, 1));  // release: orders the remote stores
    return true;
}

// Every other role: the pair's k-th entry from slot k mod RING (its order
// index; *t with it), then the slot is released to the
// scheduler.  The wait is an acquire at cluster scope, so what the
// scheduler saw before publishing (the dependencies' results) is seen here.
template <int STAGES>
__device__ __forceinline__ int ring_take(RCtl<STAGES>* ctl, uint32_t k, const RParams& rp, volatile int* abort_flag,
                                         volatile uint32_t* abort_all, unsigned code, RingTile* t) {
    const uint32_t r = k % RING, use = k / RING;
    if (!rwait<true>(zbp::smem_u32(&ctl->tfill[r]), use & 1u, abort_flag, abort_all, rp.err, code, WAIT_LIMIT_NS,
                     true))
        return -2;
    const int e = *reinterpret_cast<volatile int*>(&ctl->tslot[r]);
    t->ent = *reinterpret_cast<volatile uint32_t*>(&ctl->tent[r]);
    t->info = *reinterpret_cast<volatile uint32_t*>(&ctl->tinfo[r]);
    t->m0 = *reinterpret_cast<volatile int*>(&ctl->tm0[r]);
    t->n0 = *reinterpret_cast<volatile int*>(&ctl->tn0[r]);
    t->maps = *reinterpret_cast<volatile uint32_t*>(&ctl->tmaps[r]);
    t->hints = *reinterpret_cast<volatile uint32_t*>(&ctl->thints[r]);
    zbp::mbar_arrive_cluster(zbp::mapa_shared(zbp::smem_u32(&ctl->tfree[r]), 0));
    return e;
}

// The scheduler: bounded wait until the leader's producer has taken `k`
// entries (the scheduler runs at most one tile ahead of it).
__device__ bool wait_taken(volatile int* ptaken, int k, volatile int* abort_flag, volatile uint32_t* abort_all,
                           unsigned int* err) {
    if (*ptaken >= k) return true;
    const uint64_t t0 = zbp::globaltimer_ns();
    uint32_t spins = 0;
    while (*ptaken < k) {
        __nanosleep(20);
        if ((++spins & 15u) == 0) {
            const uint64_t waited = zbp::globaltimer_ns() - t0;
            if (*abort_flag || (waited > 20000 && *abort_all)) {
                *abort_flag = 1;
                return false;
            }
            if (waited > WAIT_LIMIT_NS) {
                *abort_flag = 1;
                *abort_all = 1;
                atomicOr(err, ERR_WAIT_PRODUCER);
                return false;
            }
        }
    }
    return true;
}

__device__ __forceinline__ void load_h32r(const __nv_bfloat16* aux, long long ldaux, int Mg, int Ng, int row,
                                          int col0, uint32_t (&hw)[16]) {
    const __nv_bfloat16* hp = aux + static_cast<long long>(row) * ldaux + col0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint4 hv = make_uint4(0u, 0u, 0u, 0u);
        if (row < Mg && col0 + g * 8 < Ng) hv = *reinterpret_cast<const uint4*>(hp + g * 8);
        hw[4 * g] = hv.x;
        hw[4 * g + 1] = hv.y;
        hw[4 * g + 2] = hv.z;
        hw[4 * g + 3] = hv.w;
    }
}

// The K loops of one tile, with the operand majors fixed at compile time (as
// in the one-launch kernel): the MMA issuer's descriptors and instruction
// word are then built from constants.
template <int A_MN, int B_MN, int STAGES>
__device__ __forceinline__ bool load_tile(RCtl<STAGES>* ctl, uint8_t* smem, uint32_t& it, int num_kb,
                                          const CUtensorMap* tma, const CUtensorMap* tmb, int m0, int nb0,
                                          uint64_t pol_a, uint64_t pol_b, bool leader, volatile int* abort_flag,
                                          volatile uint32_t* abort_all, unsigned int* err) {
    using C = Cfg<2>;
    for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const uint32_t s = it % STAGES;
        const uint32_t r = it / STAGES;
        if (!rwait<true>(zbp::smem_u32(&ctl->empty[s]), (r & 1u) ^ 1u, abort_flag, abort_all, err,
                         ERR_WAIT_PRODUCER, WAIT_LIMIT_NS, true))
            return false;
        const uint32_t full_local = zbp::smem_u32(&ctl->full[s]);
        const uint32_t full = zbp::mapa_shared(full_local, 0);
        const uint32_t sa = zbp::smem_u32(smem + s * C::STAGE_BYTES);
        const uint32_t sb = sa + A_BYTES;
        const int k0 = kb * BK;
        if (leader) zbp::mbar_arrive_expect_tx(full_local, C::STAGE_BYTES * 2);
        if (A_MN) {
            zbp::tma_load_2d_pair_hint(sa, tma, full, m0, k0, pol_a);
            zbp::tma_load_2d_pair_hint(sa + MN_ATOM_BYTES, tma, full, m0 + 64, k0, pol_a);
        } else {
            zbp::tma_load_2d_pair_hint(sa, tma, full, k0, m0, pol_a);
        }
        if (B_MN) {
#pragma unroll
            for (int i = 0; i < C::B_ROWS / 64; ++i)
                zbp::tma_load_2d_pair_hint(sb + i * MN_ATOM_BYTES, tmb, full, nb0 + 64 * i, k0, pol_b);
        } else {
            zbp::tma_load_2d_pair_hint(sb, tmb, full, k0, nb0, pol_b);
        }
    }
    return true;
}

template <int A_MN, int B_MN, int STAGES>
__device__ __forceinline__ bool mma_tile(RCtl<STAGES>* ctl, uint8_t* smem, uint32_t& it, int num_kb, uint32_t d_tmem,
                                         volatile int* abort_flag, volatile uint32_t* abort_all, unsigned int* err) {
    using C = Cfg<2>;
    constexpr uint32_t idesc = zbp::idesc_bf16_f32(BM * 2, BN, A_MN, B_MN);
    for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const uint32_t s = it % STAGES;
        const uint32_t r = it / STAGES;
        if (!rwait<true>(zbp::smem_u32(&ctl->full[s]), r & 1u, abort_flag, abort_all, err, ERR_WAIT_MMA,
                         WAIT_LIMIT_NS, true))
            return false;
        zbp::tc_fence_after();
        const uint32_t sa = zbp::smem_u32(smem + s * C::STAGE_BYTES);
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? zbp::smem_desc_sw128(sa + kk * 2048, MN_ATOM_BYTES, 1024)
                                     : zbp::smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? zbp::smem_desc_sw128(sb + kk * 2048, MN_ATOM_BYTES, 1024)
                                     : zbp::smem_desc_sw128(sb + kk * 32, 16, 1024);
            zbp::tc_mma_f16_pair(d_tmem, ad, bd, idesc, ((kb | kk) != 0) ? 1u : 0u);
        }
        zbp::tc_commit_pair_multicast(zbp::smem_u32(&ctl->empty[s]), 0x3);
    }
    return true;
}

__global__ void __launch_bounds__(REPLAY_THREADS, 1) zb_replay_tc_kernel(const __grid_constant__ RParams rp) {
    using C = Cfg<2>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* staging = smem + STAGES * C::STAGE_BYTES;
    RCtl<STAGES>* ctl = reinterpret_cast<RCtl<STAGES>*>(staging + STAGING_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = zbp::cluster_ctarank();
    const bool leader = rank == 0;
    const uint32_t pair = blockIdx.x >> 1;
    volatile uint32_t* abort_all = rp.done + rp.njobs;
    const CUtensorMap* maps = rp.nparam > 0 ? rp.pmaps : rp.maps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            zbp::mbar_init(zbp::smem_u32(&ctl->full[s]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            zbp::mbar_init(zbp::smem_u32(&ctl->tfull[b]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->tempty[b]), SIGNALS_PER_TILE);
        }
        zbp::mbar_init(zbp::smem_u32(&ctl->drain), 1);
        for (int r = 0; r < RING; ++r) {
            zbp::mbar_init(zbp::smem_u32(&ctl->tfill[r]), 1);
            zbp::mbar_init(zbp::smem_u32(&ctl->tfree[r]), RING_READERS);
        }
        ctl->abort_flag = 0;
        ctl->ptaken = 0;
        zbp::fence_mbar_init();
    }
    if (warp == 1) {
        zbp::tmem_alloc_pair(zbp::smem_u32(&ctl->tmem_base), TMEM_COLS);
        zbp::tmem_relinquish_pair();
    }
    zbp::tc_fence_before();
    __syncthreads();
    zbp::cluster_sync();  // both CTAs' barriers exist before any remote use
    zbp::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t it = 0;
            bool ok = true;
            int cur = -1;
            for (uint32_t k = 0; ok; ++k) {
                RingTile t;
                const int e = ring_take(ctl, k, rp, abort_flag, abort_all, ERR_WAIT_PRODUCER, &t);
                if (e < 0) {
                    ok = e == -1;
                    break;
                }
                if (leader) *reinterpret_cast<volatile int*>(&ctl->ptaken) = static_cast<int>(k) + 1;
                const int job = static_cast<int>(t.ent >> ENTRY_JOB_SHIFT);
                const CUtensorMap* tma = maps + (t.maps & 0xffffu);
                const CUtensorMap* tmb = maps + (t.maps >> 16);
                if (job != cur) {
                    // the scheduler's acquire of the job's dependencies reached
                    // this thread through the ring; its TMA reads follow it
                    zbp::fence_proxy_async_global();
                    if (rp.nparam == 0) {
                        zbp::fence_tensormap_acquire(tma);
                        zbp::fence_tensormap_acquire(tmb);
                    }
                    zbp::tma_prefetch_desc(tma);
                    zbp::tma_prefetch_desc(tmb);
                    cur = job;
                }
                const int a_mn = static_cast<int>(t.info >> 29) & 1, b_mn = static_cast<int>(t.info >> 28) & 1;
                const uint64_t pol_a = zbp::l2_policy(static_cast<int>(t.hints & 0xffu));
                const uint64_t pol_b = zbp::l2_policy(static_cast<int>((t.hints >> 8) & 0xffu));
                const int m0 = t.m0 + static_cast<int>(rank) * BM;
                const int nb0 = t.n0 + static_cast<int>(rank) * C::B_ROWS;
                const int num_kb = static_cast<int>(t.info & INFO_KB_MASK);
                switch ((a_mn << 1) | b_mn) {
                    case 0: ok = load_tile<0, 0>(ctl, smem, it, num_kb, tma, tmb, m0, nb0, pol_a, pol_b, leader,
                                                 abort_flag, abort_all, rp.err); break;
                    case 1: ok = load_tile<0, 1>(ctl, smem, it, num_kb, tma, tmb, m0, nb0, pol_a, pol_b, leader,
                                                 abort_flag, abort_all, rp.err); break;
                    case 2: ok = load_tile<1, 0>(ctl, smem, it, num_kb, tma, tmb, m0, nb0, pol_a, pol_b, leader,
                                                 abort_flag, abort_all, rp.err); break;
                    default: ok = load_tile<1, 1>(ctl, smem, it, num_kb, tma, tmb, m0, nb0, pol_a, pol_b, leader,
                                                  abort_flag, abort_all, rp.err); break;
                }
            }
            if (!ok && leader) {
                // wait for the copies that were issued but may not have landed
                const uint32_t first = it > STAGES ? it - STAGES : 0;
                for (uint32_t i = first; i < it; ++i) {
                    rwait<true>(zbp::smem_u32(&ctl->full[i % STAGES]), (i / STAGES) & 1u, abort_flag, abort_all,
                                rp.err, ERR_WAIT_PRODUCER, DRAIN_LIMIT_NS, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t local = 0; ok; ++local) {
                RingTile t;
                const int e = ring_take(ctl, local, rp, abort_flag, abort_all, ERR_WAIT_MMA, &t);
                if (e < 0) break;
                const int majors = static_cast<int>(t.info >> 28) & 3;
                const int num_kb = static_cast<int>(t.info & INFO_KB_MASK);
                const uint32_t buf = local & 1u;
                const uint32_t tr = local >> 1;
                if (!rwait<true>(zbp::smem_u32(&ctl->tempty[buf]), (tr & 1u) ^ 1u, abort_flag, abort_all, rp.err,
                                 ERR_WAIT_MMA, WAIT_LIMIT_NS, true)) {
                    ok = false;
                    break;
                }
                zbp::tc_fence_after();
                if (rp.trace) rp.trace[e].t_mma0 = zbp::globaltimer_ns();
                const uint32_t d_tmem = tmem_base + buf * ACC_COLS;
                switch (majors) {
                    case 0: ok = mma_tile<0, 0>(ctl, smem, it, num_kb, d_tmem, abort_flag, abort_all, rp.err); break;
                    case 1: ok = mma_tile<0, 1>(ctl, smem, it, num_kb, d_tmem, abort_flag, abort_all, rp.err); break;
                    case 2: ok = mma_tile<1, 0>(ctl, smem, it, num_kb, d_tmem, abort_flag, abort_all, rp.err); break;
                    default: ok = mma_tile<1, 1>(ctl, smem, it, num_kb, d_tmem, abort_flag, abort_all, rp.err); break;
                }
                if (!ok) break;
                zbp::tc_commit_pair_multicast(zbp::smem_u32(&ctl->tfull[buf]), 0x3);
                if (rp.trace) rp.trace[e].t_mma1 = zbp::globaltimer_ns();
            }
            // every MMA issued here completes before TMEM is released
            zbp::tc_commit_pair(zbp::smem_u32(&ctl->drain));
            rwait<true>(zbp::smem_u32(&ctl->drain), 0, abort_flag, abort_all, rp.err, ERR_WAIT_MMA, DRAIN_LIMIT_NS,
                        false);
        }
    } else if (warp < SCHED_WARP) {
        // ---------------------------------------------------- epilogue
        // Warp w reads TMEM lanes 32 (w mod 4) .. + 31 (rows of this CTA's
        // 128), columns [128 h, 128 h + 128) of the tile with h = (w - 2) / 4,
        // in chunks of 32, through its own 4 KiB of staging: two 32 x 32 bf16
        // boxes in turn, or one 32 x 32 fp32 box.  After its last store of a
        // tile has completed it signals the tile to the tile's job counter.
        const int ew = warp - 2;
        const int q = warp & 3;
        const int c_lo = (ew >> 2) * 128;
        const uint32_t region = zbp::smem_u32(staging) + static_cast<uint32_t>(ew) * 4096u;
        uint32_t flip = 0;
        int cur = -1;
        for (uint32_t local = 0;; ++local) {
            int e = 0;
            RingTile t{};
            if (lane == 0) e = ring_take(ctl, local, rp, abort_flag, abort_all, ERR_WAIT_EPI, &t);
            e = __shfl_sync(0xffffffffu, e, 0);
            const uint32_t ent = __shfl_sync(0xffffffffu, t.ent, 0);
            const int m0 = __shfl_sync(0xffffffffu, t.m0, 0) + static_cast<int>(rank) * BM;
            const int n0 = __shfl_sync(0xffffffffu, t.n0, 0);
            __syncwarp();  // orders every lane's reads after lane 0's acquire
            if (e < 0) break;
            const int job = static_cast<int>(ent >> ENTRY_JOB_SHIFT);
            const RJob* J = rp.jobs + job;
            const int epi = J->epi, Mg = J->Mg, Ng = J->Ng;
            const CUtensorMap* tmo0 = maps + J->map_o0;
            const CUtensorMap* tmo1 = maps + J->map_o1;
            if (job != cur) {
                // the scheduler's acquire of the job's dependencies reached
                // lane 0 through the ring; its TMA stores follow it
                if (lane == 0) {
                    zbp::fence_proxy_async_global();
                    if (rp.nparam == 0) {
                        zbp::fence_tensormap_acquire(tmo0);
                        if (epi == zb::EPI_GELU_DUAL) zbp::fence_tensormap_acquire(tmo1);
                    }
                }
                cur = job;
            }
            const uint32_t buf = local & 1u;
            const uint32_t tr = local >> 1;
            const int row0 = m0 + q * 32;
            const int row = row0 + lane;
            const bool rows_live = row0 < Mg;
            const uint64_t pol_out = zbp::l2_policy(J->hint_out);
            const __nv_bfloat16* aux = J->aux;
            const long long ldaux = J->ldaux;
            uint32_t h_next[16];
            if (epi == zb::EPI_GELU_BWD) {
                if (row < Mg && n0 + c_lo < Ng) {
                    const int ncols = min(128, Ng - n0 - c_lo);
                    zbp::prefetch_l2(aux + static_cast<long long>(row) * ldaux + n0 + c_lo,
                                     static_cast<uint32_t>(ncols) * 2u);
                }
                load_h32r(aux, ldaux, Mg, Ng, row, n0 + c_lo, h_next);
            }
            if (!rwait<true>(zbp::smem_u32(&ctl->tfull[buf]), tr & 1u, abort_flag, abort_all, rp.err, ERR_WAIT_EPI,
                             WAIT_LIMIT_NS, true))
                break;
            zbp::tc_fence_after();
            const bool tr_epi = rp.trace != nullptr && leader && warp == 2 && lane == 0;
            if (tr_epi) rp.trace[e].t_epi0 = zbp::globaltimer_ns();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * ACC_COLS;
            if (epi == zb::EPI_F32) {
                const uint64_t spacing = static_cast<uint64_t>((J->Kg + BK - 1) / BK) * PACE_NS_PER_KB;
                const uint64_t t_full = zbp::globaltimer_ns();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const uint64_t slot = static_cast<uint64_t>(c * 8 + ew);
                    if (slot > 0) {
                        if (lane == 0) {
                            const uint64_t target = t_full + slot * spacing;
                            while (zbp::globaltimer_ns() < target) __nanosleep(64);
                        }
                        __syncwarp();
                    }
                    uint32_t v[32];
                    zbp::tmem_ld_32x32b_x32(taddr + c_lo + c * 32, v);
                    zbp::tmem_ld_wait();
                    const int col0 = n0 + c_lo + c * 32;
                    if (!rows_live || col0 >= Ng) continue;
                    if (lane == 0) zbp::bulk_wait_read<0>();  // one box per warp
                    __syncwarp();
                    stage_row(region, lane, v);
                    if (J->accumulate)
                        staging_release<true>(tmo0, region, lane, col0, row0, pol_out);
                    else
                        staging_release<false>(tmo0, region, lane, col0, row0, pol_out);
                }
            } else {
                const bool tanh_act = J->act == ZB_ACT_GELU_TANH;
                const __nv_bfloat16* bias = J->bias;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int col0 = n0 + c_lo + c * 32;
                    uint32_t hw[16];
                    if (epi == zb::EPI_GELU_BWD) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) hw[i] = h_next[i];
                        if (c + 1 < 4) load_h32r(aux, ldaux, Mg, Ng, row, col0 + 32, h_next);
                    }
                    uint32_t v[32];
                    zbp::tmem_ld_32x32b_x32(taddr + c_lo + c * 32, v);
                    zbp::tmem_ld_wait();
                    if (!rows_live || col0 >= Ng) continue;
                    float x[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
                    if (epi != zb::EPI_GELU_BWD && bias) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            if (col0 + g * 8 >= Ng) break;
                            const uint4 bv = *reinterpret_cast<const uint4*>(bias + col0 + g * 8);
                            const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f2 = unpack_bf16x2(bw[i]);
                                x[g * 8 + 2 * i] += f2.x;
                                x[g * 8 + 2 * i + 1] += f2.y;
                            }
                        }
                    }
                    if (epi == zb::EPI_GELU_BWD) {
                        if (tanh_act)
                            gelu_grad_mul<true, 32>(x, hw);
                        else
                            gelu_grad_mul<false, 32>(x, hw);
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
                    uint32_t stg = region + flip * 2048u;
                    flip ^= 1u;
                    staging_acquire(lane);
                    stage_row64(stg, lane, w);
                    staging_release<false>(tmo0, stg, lane, col0, row0, pol_out);
                    if (epi == zb::EPI_GELU_DUAL) {
                        if (tanh_act)
                            gelu_pack<true, 32>(x, w);
                        else
                            gelu_pack<false, 32>(x, w);
                        stg = region + flip * 2048u;
                        flip ^= 1u;
                        staging_acquire(lane);
                        stage_row64(stg, lane, w);
                        staging_release<false>(tmo1, stg, lane, col0, row0, pol_out);
                    }
                }
            }
            if (tr_epi) rp.trace[e].t_epi1 = zbp::globaltimer_ns();
            zbp::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                zbp::mbar_arrive_cluster(zbp::mapa_shared(zbp::smem_u32(&ctl->tempty[buf]), 0));
                // the tile's outputs are in global memory before it is signalled
                zbp::bulk_wait<0>();
                zbp::fence_proxy_async_global();
                zbp::red_release_gpu_add(rp.done + job, 1u);
                if (rp.trace != nullptr && leader && warp == 2) rp.trace[e].t_signal = zbp::globaltimer_ns();
            }
            __syncwarp();
        }
        // the staging boxes must not be released while a bulk store reads them
        if (lane == 0) zbp::bulk_wait<0>();
        __syncwarp();
    } else if (lane == 0 && leader) {
        // ---------------------------------------------------- scheduler
        // Takes the pair's k-th tile once the producer has taken the
        // (k-1)-th (one tile of lookahead: the pair claims no more of the
        // order than it can start on), waits for the tile's dependencies
        // when its job changes, and publishes it.
        int cur = -1;
        for (uint32_t k = 0;; ++k) {
            if (!wait_taken(&ctl->ptaken, static_cast<int>(k), abort_flag, abort_all, rp.err)) break;
            int e = static_cast<int>(atomicAdd(rp.done + rp.njobs + 1, 1u));
            RingTile t{};
            if (e >= rp.ntiles) {
                e = -1;
            } else {
                const uint32_t ent = rp.entries[e];
                const int job = static_cast<int>(ent >> ENTRY_JOB_SHIFT);
                const RJob* J = rp.jobs + job;
                if (rp.trace) {
                    rp.trace[e].pair = pair;
                    rp.trace[e].t_reach = zbp::globaltimer_ns();
                }
                if (job != cur) {
                    if (!wait_deps(rp, J, abort_flag)) break;
                    cur = job;
                }
                const uint32_t num_kb = static_cast<uint32_t>((J->Kg + BK - 1) / BK);
                int mb, nb;
                tile_coords(static_cast<int>(ent & ENTRY_TILE_MASK), J->tiles_m, J->tiles_n, Cfg<2>::GROUP_M, mb, nb);
                t.ent = ent;
                t.info = num_kb | static_cast<uint32_t>((J->a_mn << 1) | J->b_mn) << 28;
                t.m0 = mb * Cfg<2>::TILE_M;
                t.n0 = nb * BN;
                t.maps = static_cast<uint32_t>(J->map_a) | static_cast<uint32_t>(J->map_b) << 16;
                t.hints = static_cast<uint32_t>(J->hint_a) | static_cast<uint32_t>(J->hint_b) << 8;
                if (rp.trace) rp.trace[e].t_ready = zbp::globaltimer_ns();
            }
            if (!ring_publish(ctl, k, e, t, rp, abort_flag, abort_all)) break;
            if (e < 0) break;
        }
    }

    __syncthreads();
    zbp::cluster_sync();  // no remote arrivals or copies remain
    if (warp == 1) {
        zbp::tc_fence_after();
        zbp::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Copies one chunk of the tables from the launch parameters into global
// memory (16-byte aligned destination and size).
constexpr uint32_t UPLOAD_CHUNK = 31 * 1024;
struct alignas(16) UploadChunk {
    uint8_t* dst;
    uint32_t bytes;
    uint32_t pad;
    uint8_t data[UPLOAD_CHUNK];
};

__global__ void zb_replay_upload_kernel(const __grid_constant__ UploadChunk c) {
    const uint32_t stride = gridDim.x * blockDim.x * 16u;
    for (uint32_t i = (blockIdx.x * blockDim.x + threadIdx.x) * 16u; i < c.bytes; i += stride)
        *reinterpret_cast<uint4*>(c.dst + i) = *reinterpret_cast<const uint4*>(c.data + i);
}

// ---------------------------------------------------------------- host side
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ZB_REPLAY_TRACE=1 in the environment: per-tile trace records (TraceRec)
// at the end of the caller's workspace (the size query counts them).
bool trace_on() {
    static const bool on = [] {
        const char* v = std::getenv("ZB_REPLAY_TRACE");
        return v && v[0] == '1';
    }();
    return on;
}

struct Layout {
    size_t maps, jobs, deps, entries, done, total;
};

Layout table_layout(size_t nmaps, size_t njobs, size_t ndeps, size_t ntiles) {
    Layout L;
    L.maps = 0;
    L.jobs = align256(L.maps + nmaps * sizeof(CUtensorMap));
    L.deps = align256(L.jobs + njobs * sizeof(RJob));
    L.entries = align256(L.deps + ndeps * sizeof(int));
    L.done = align256(L.entries + ntiles * sizeof(uint32_t));
    L.total = align256(L.done + (njobs + 2) * sizeof(uint32_t));
    return L;
}

long long pair_tiles_of(long long Mg, long long Ng) { return ((Mg + 2 * BM - 1) / (2 * BM)) * ((Ng + BN - 1) / BN); }

// Byte range [lo, hi) of a row-major operand: `rows` rows of stride ld
// elements, `width` used elements per row.
struct Range {
    uintptr_t lo, hi;
};
Range range_of(const void* p, long long rows, long long width, long long ld, int es) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(p);
    return {b, b + static_cast<uintptr_t>(((rows - 1) * ld + width) * es)};
}
bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

int replay_pairs() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n) return n;
    auto kern = zb_replay_tc_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(replay_smem_bytes())) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256, 1, 1);
    cfg.blockDim = dim3(REPLAY_THREADS, 1, 1);
    cfg.dynamicSmemBytes = replay_smem_bytes();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        return 0;
    }
    n = std::min(clusters, MAX_PAIRS);
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Estimated time of one tile (units of 1/16 of a K block's MMA time at the
// tensor peak): its K loop at the rate tiles of the P=4, h=1024 pipeline
// were traced at (1.45 x the peak: the operand stream of a CTA pair runs
// behind the tensor pipe at these sizes), or its epilogue and completion
// signal where those are longer (the GeLU epilogues of a K = 1024 tile: ~7
// us), plus a fixed cost.
int64_t tile_cost(const zb::GemmBf16& g) {
    const int64_t kb = (g.Kg + BK - 1) / BK;
    const int64_t epi = g.epi == zb::EPI_GELU_DUAL ? 40 : g.epi == zb::EPI_GELU_BWD ? 44 : g.epi == zb::EPI_F32 ? 16 : 10;
    return std::max(kb * 23, epi * 16) + 4 * 16;
}
// Simulated time from a GEMM's last tile to its dependents' first: the
// completion signal, its detection and a cold operand pipeline, plus slack
// for tiles that run late, so that the order seldom puts a tile ahead of the
// moment a pair could start it.
// Chosen by measurement on the P=4, h=1024 pipeline, for the longest-chain
// priority (mean of ZB-H1, ZB-H2, 1F1B, ZB-2p and ZB-V, TF/s): 2 K blocks
// 1190, 20 1224, 45 1234, 70 1246, 100 1258, 150 1229.  With list order
// (GEMMs of several waves, each on every pair in turn) 2 K blocks: there a
// larger one only moves later GEMMs' tiles into the current one's waves.
constexpr int64_t READY_LATENCY_CHAIN = 100 * 16;
constexpr int64_t READY_LATENCY_LIST = 2 * 16;

}  // namespace

namespace zb {

size_t replay_table_bytes(size_t njobs, size_t ntiles) {
    return table_layout(4 * njobs, njobs, DEPS_PER_JOB * njobs, ntiles).total +
           (trace_on() ? align256(ntiles * sizeof(TraceRec)) : 0);
}

zb_status replay_count(const zb_block& b, const zb_op* ops, size_t n_ops, size_t* njobs, size_t* ntiles) {
    const bool mlp = b.act != ZB_ACT_NONE;
    const long long M = b.M, h = b.h, f = b.f;
    size_t nj = 0, nt = 0;
    auto add = [&](long long Mg, long long Ng) {
        ++nj;
        nt += static_cast<size_t>(pair_tiles_of(Mg, Ng));
    };
    for (size_t i = 0; i < n_ops; ++i) {
        const int k = ops[i].kind;
        if (k == ZB_OP_F) {
            add(M, f);
            if (mlp) add(M, h);
        }
        if (k == ZB_OP_B || k == ZB_OP_BW) {
            if (mlp) add(M, f);
            add(M, h);
        }
        if (k == ZB_OP_W || k == ZB_OP_BW) {
            if (mlp) add(f, h);
            add(h, f);
        }
    }
    *njobs = nj;
    *ntiles = nt;
    return ZB_OK;
}

// The host plan of a persistent replay: every GEMM's tiles, its
// dependencies (transitive reduction of the byte-range conflicts), the tile
// lists of the CTA pairs from the list-scheduling simulation, the global
// order of all tiles by simulated start that the kernel hands out, and the
// check that this order cannot deadlock.  No device access.
zb_status plan_replay(const std::vector<GemmBf16>& jobs, int npairs, ReplayPlan* plan) {
    const size_t nj = jobs.size();
    *plan = ReplayPlan{};
    if (nj == 0) return ZB_OK;
    if (nj > MAX_JOBS) return fail(ZB_ERR_UNSUPPORTED, "persistent replay: too many GEMMs in one op list");
    if (npairs <= 0 || npairs > MAX_PAIRS) return fail(ZB_ERR_INVALID_ARG, "persistent replay: pair count");
    auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    std::vector<long long>& tiles = plan->tiles;
    tiles.assign(nj, 0);
    std::vector<std::vector<Range>> reads(nj), writes(nj);
    size_t ntiles = 0;
    for (size_t j = 0; j < nj; ++j) {
        const GemmBf16& g = jobs[j];
        if (g.Mg <= 0 || g.Ng <= 0 || g.Kg <= 0 || g.Mg > (1LL << 30) || g.Ng > (1LL << 30) || g.Kg > (1LL << 30))
            return fail(ZB_ERR_SHAPE, "GEMM extents must be in [1, 2^30]");
        if (g.Ng % 8 != 0) return fail(ZB_ERR_ALIGN, "GEMM N must be a multiple of 8");
        if ((g.lda % 8) || (g.ldb % 8) || (g.ld0 % 8) || (g.out1 && g.ld1 % 8) || (g.aux && g.ldaux % 8))
            return fail(ZB_ERR_ALIGN, "leading dimensions must be multiples of 8 elements");
        if (mis(g.A) || mis(g.B) || mis(g.out0) || mis(g.out1) || mis(g.aux) || mis(g.bias))
            return fail(ZB_ERR_ALIGN, "GEMM pointers must be 16-byte aligned");
        if (!g.A || !g.B || !g.out0) return fail(ZB_ERR_INVALID_ARG, "GEMM operand is NULL");
        if (g.second) return fail(ZB_ERR_INVALID_ARG, "persistent replay: grouped GEMM record");
        if (g.epi == EPI_GELU_DUAL && !g.out1) return fail(ZB_ERR_INVALID_ARG, "GeLU dual store needs out1");
        if (g.epi == EPI_GELU_BWD && !g.aux) return fail(ZB_ERR_INVALID_ARG, "GeLU' epilogue needs H");
        if (g.epi == EPI_F32 && g.bias) return fail(ZB_ERR_UNSUPPORTED, "persistent replay: bias of an fp32 GEMM");
        const bool f32_out = g.epi == EPI_F32;
        if (f32_out && (g.ld0 % 4)) return fail(ZB_ERR_ALIGN, "fp32 output leading dimension must be a multiple of 4");
        tiles[j] = pair_tiles_of(g.Mg, g.Ng);
        if (tiles[j] > static_cast<long long>(ENTRY_TILE_MASK) + 1)
            return fail(ZB_ERR_UNSUPPORTED, "persistent replay: too many tiles in one GEMM");
        ntiles += static_cast<size_t>(tiles[j]);
        // byte ranges read and written
        reads[j].push_back(g.a_mn ? range_of(g.A, g.Kg, g.Mg, g.lda, 2) : range_of(g.A, g.Mg, g.Kg, g.lda, 2));
        reads[j].push_back(g.b_mn ? range_of(g.B, g.Kg, g.Ng, g.ldb, 2) : range_of(g.B, g.Ng, g.Kg, g.ldb, 2));
        if (g.epi == EPI_GELU_BWD) reads[j].push_back(range_of(g.aux, g.Mg, g.Ng, g.ldaux, 2));
        if (g.bias) reads[j].push_back(range_of(g.bias, 1, g.Ng, g.Ng, 2));
        writes[j].push_back(range_of(g.out0, g.Mg, g.Ng, g.ld0, f32_out ? 4 : 2));
        if (f32_out && g.accumulate) reads[j].push_back(writes[j].back());
        if (g.epi == EPI_GELU_DUAL) writes[j].push_back(range_of(g.out1, g.Mg, g.Ng, g.ld1, 2));
    }
    plan->ntiles = ntiles;

    // -------------------------------------------- dependencies
    // j depends on i < j when i writes what j reads or writes, or reads what
    // j writes; kept: the deps not implied by another kept dep (transitive
    // reduction over the closure bitsets)
    const size_t words = (nj + 63) / 64;
    std::vector<uint64_t> closure(nj * words, 0);
    std::vector<std::vector<int>>& deps = plan->deps;
    deps.assign(nj, {});
    size_t ndeps = 0;
    for (size_t j = 0; j < nj; ++j) {
        std::vector<uint64_t> cover(words, 0);
        uint64_t* cj = closure.data() + j * words;
        for (size_t ii = j; ii-- > 0;) {
            if (cover[ii / 64] >> (ii % 64) & 1u) continue;  // implied by a later dep
            bool hit = false;
            for (const Range& w : writes[ii]) {
                for (const Range& r : reads[j]) hit = hit || overlap(w, r);
                for (const Range& r : writes[j]) hit = hit || overlap(w, r);
            }
            for (const Range& r : reads[ii])
                for (const Range& w : writes[j]) hit = hit || overlap(r, w);
            if (!hit) continue;
            deps[j].push_back(static_cast<int>(ii));
            const uint64_t* ci = closure.data() + ii * words;
            for (size_t w = 0; w < words; ++w) cover[w] |= ci[w];
            cover[ii / 64] |= uint64_t(1) << (ii % 64);
        }
        for (size_t w = 0; w < words; ++w) cj[w] = cover[w];
        if (deps[j].size() > DEPS_PER_JOB)
            return fail(ZB_ERR_UNSUPPORTED, "persistent replay: a GEMM with more than 16 direct dependencies");
        ndeps += deps[j].size();
    }

    // -------------------------------------------- tile assignment
    std::vector<std::vector<int>> succ(nj);
    for (size_t j = 0; j < nj; ++j)
        for (int d : deps[j]) succ[d].push_back(static_cast<int>(j));
    // Which ready job a free pair takes.  Where most tiles belong to GEMMs
    // of at least two waves of tiles (the large one-stage steps): the
    // earliest in list order, so that each GEMM runs on every pair, its
    // waves walking K in step and sharing operands in L2, while the next
    // ones fill its last partial wave (h=6144: 97 ms against 107 ms for the
    // other rule).  Else (small GEMMs of many stages, which always share the
    // GPU): the one with the longest chain of work after it (the P=4, h=1024
    // pipeline: 2.97 ms against 3.24 ms).  ZB_REPLAY_PRIORITY=level or =list
    // in the environment forces one rule.
    static const int forced = [] {
        const char* v = std::getenv("ZB_REPLAY_PRIORITY");
        if (v && std::strcmp(v, "level") == 0) return 1;
        if (v && std::strcmp(v, "list") == 0) return 2;
        return 0;
    }();
    long long big_tiles = 0;
    for (size_t j = 0; j < nj; ++j)
        if (tiles[j] >= 2LL * npairs) big_tiles += tiles[j];
    const bool by_level = forced ? forced == 1 : 2 * big_tiles < static_cast<long long>(ntiles);
    const int64_t ready_latency = by_level ? READY_LATENCY_CHAIN : READY_LATENCY_LIST;
    // bottom level: the longest chain of job spans (its tiles spread over
    // all pairs) from the job to the end
    std::vector<int64_t> cost(nj), level(nj, 0);
    for (size_t j = 0; j < nj; ++j) cost[j] = tile_cost(jobs[j]);
    for (size_t j = nj; j-- > 0;) {
        int64_t tail = 0;
        for (int s : succ[j]) tail = std::max(tail, level[s] + ready_latency);
        level[j] = (tiles[j] + npairs - 1) / npairs * cost[j] + tail;
    }

    auto prio = [&](int a, int b) {
        if (by_level && level[a] != level[b]) return level[a] > level[b];
        return a < b;
    };
    std::vector<int64_t> ready_at(nj, 0), finish(nj, 0), last_start(nj, -1);
    std::vector<long long> remaining(tiles), next_tile(nj, 0);
    std::vector<int> deps_left(nj);
    std::vector<int> ready;  // jobs whose dependencies are all assigned, with tiles left
    for (size_t j = 0; j < nj; ++j) {
        deps_left[j] = static_cast<int>(deps[j].size());
        if (deps_left[j] == 0) ready.push_back(static_cast<int>(j));
    }
    using Slot = std::pair<int64_t, int>;  // (free at, pair)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
    for (int p = 0; p < npairs; ++p) free_at.push({0, p});
    std::vector<std::vector<uint32_t>>& lists = plan->lists;
    std::vector<std::vector<int64_t>>& starts = plan->starts;
    lists.assign(npairs, {});
    starts.assign(npairs, {});
    plan->order.clear();
    plan->order_start.clear();
    plan->order_pair.clear();
    plan->order.reserve(ntiles);
    plan->order_start.reserve(ntiles);
    plan->order_pair.reserve(ntiles);
    size_t assigned = 0;
    while (assigned < ntiles) {
        const Slot sl = free_at.top();
        free_at.pop();
        const int64_t t = sl.first;
        int best = -1;
        int64_t next_ready = INT64_MAX;
        for (int j : ready) {
            if (ready_at[j] > t) {
                next_ready = std::min(next_ready, ready_at[j]);
                continue;
            }
            if (best < 0 || prio(j, best)) best = j;
        }
        if (best < 0) {
            if (next_ready == INT64_MAX) return fail(ZB_ERR_UNSUPPORTED, "persistent replay: no job ready");
            free_at.push({next_ready, sl.second});
            continue;
        }
        const long long tile = next_tile[best]++;
        const uint32_t ent = (static_cast<uint32_t>(best) << ENTRY_JOB_SHIFT) | static_cast<uint32_t>(tile);
        lists[sl.second].push_back(ent);
        starts[sl.second].push_back(t);
        plan->order.push_back(ent);
        plan->order_start.push_back(t);
        plan->order_pair.push_back(static_cast<uint32_t>(sl.second));
        last_start[best] = std::max(last_start[best], t);
        finish[best] = std::max(finish[best], t + cost[best]);
        ++assigned;
        if (--remaining[best] == 0) {
            ready.erase(std::find(ready.begin(), ready.end(), best));
            for (int s : succ[best]) {
                if (--deps_left[s] == 0) {
                    int64_t r = 0;
                    for (int d : deps[s]) r = std::max(r, finish[d] + ready_latency);
                    ready_at[s] = r;
                    ready.push_back(s);
                }
            }
        }
        free_at.push({t + cost[best], sl.second});
    }
    // the order that makes the replay deadlock-free: every tile starts after
    // every tile of its dependencies, and after its pair's earlier tiles
    for (int p = 0; p < npairs; ++p) {
        for (size_t k = 0; k < lists[p].size(); ++k) {
            const int j = static_cast<int>(lists[p][k] >> ENTRY_JOB_SHIFT);
            if (k > 0 && starts[p][k] <= starts[p][k - 1])
                return fail(ZB_ERR_UNSUPPORTED, "persistent replay: a pair's tiles out of order");
            for (int d : deps[j])
                if (last_start[d] >= starts[p][k])
                    return fail(ZB_ERR_UNSUPPORTED, "persistent replay: a tile starts before its dependencies");
        }
    }
    int64_t makespan = 0;
    for (size_t j = 0; j < nj; ++j) makespan = std::max(makespan, finish[j]);
    // the order the pairs take the tiles in (each pair the next one when it
    // is free): by simulated start, then pair, so every tile comes after
    // every tile of the GEMMs it depends on (checked above).  The simulation
    // assigns tiles in that order already (its free pairs leave the heap by
    // time, then pair, and re-enter later); sorted only if that ever fails.
    bool in_order = true;
    for (size_t i = 1; i < plan->order.size() && in_order; ++i)
        in_order = plan->order_start[i - 1] < plan->order_start[i] ||
                   (plan->order_start[i - 1] == plan->order_start[i] &&
                    plan->order_pair[i - 1] < plan->order_pair[i]);
    if (!in_order) {
        std::vector<std::pair<std::pair<int64_t, int>, uint32_t>> all;
        all.reserve(ntiles);
        for (int p = 0; p < npairs; ++p)
            for (size_t k = 0; k < lists[p].size(); ++k) all.push_back({{starts[p][k], p}, lists[p][k]});
        std::sort(all.begin(), all.end());
        plan->order.resize(all.size());
        plan->order_start.resize(all.size());
        plan->order_pair.resize(all.size());
        for (size_t i = 0; i < all.size(); ++i) {
            plan->order[i] = all[i].second;
            plan->order_start[i] = all[i].first.first;
            plan->order_pair[i] = static_cast<uint32_t>(all[i].first.second);
        }
    }
    plan->ndeps = ndeps;
    plan->makespan = makespan;
    plan->by_level = by_level;
    return ZB_OK;
}

zb_status replay_persistent(const std::vector<GemmBf16>& jobs, void* table, size_t table_bytes, void* stream,
                            ReplayInfo* info) {
    const size_t nj = jobs.size();
    if (info) *info = ReplayInfo{};
    if (nj == 0) return ZB_OK;
    const int npairs = replay_pairs();
    if (npairs <= 0) return fail(ZB_ERR_UNSUPPORTED, "persistent replay: no co-resident CTA pairs");
    ReplayPlan plan;
    zb_status ps = plan_replay(jobs, npairs, &plan);
    if (ps != ZB_OK) return ps;
    const std::vector<long long>& tiles = plan.tiles;
    const std::vector<std::vector<int>>& deps = plan.deps;
    const size_t ntiles = plan.ntiles, ndeps = plan.ndeps;
    const int64_t makespan = plan.makespan;
    unsigned int* err = device_error_word();
    if (!err) return ZB_ERR_CUDA;

    // -------------------------------------------- tensor maps, job records
    std::vector<CUtensorMap> maps;
    std::unordered_map<std::string, int> map_index;
    std::string why;
    auto add_map = [&](int* idx, const void* base, bool f32, uint64_t inner, uint64_t outer, uint64_t ld,
                       uint32_t bi, uint32_t bo, CUtensorMapSwizzle sw) -> bool {
        CUtensorMap m;
        std::memset(&m, 0, sizeof(m));
        if (!make_map(&m, base, f32, inner, outer, ld, bi, bo, &why, sw)) return false;
        const std::string key(reinterpret_cast<const char*>(&m), sizeof(m));
        auto f = map_index.find(key);
        if (f != map_index.end()) {
            *idx = f->second;
            return true;
        }
        *idx = static_cast<int>(maps.size());
        maps.push_back(m);
        map_index.emplace(key, *idx);
        return true;
    };
    std::vector<RJob> rj(nj);
    size_t dep0 = 0;
    for (size_t j = 0; j < nj; ++j) {
        const GemmBf16& g = jobs[j];
        RJob& J = rj[j];
        std::memset(&J, 0, sizeof(J));
        J.Mg = static_cast<int>(g.Mg);
        J.Ng = static_cast<int>(g.Ng);
        J.Kg = static_cast<int>(g.Kg);
        J.epi = g.epi;
        J.a_mn = g.a_mn;
        J.b_mn = g.b_mn;
        J.act = g.act;
        J.accumulate = g.accumulate;
        J.tiles_m = static_cast<int>((g.Mg + 2 * BM - 1) / (2 * BM));
        J.tiles_n = static_cast<int>((g.Ng + BN - 1) / BN);
        J.dep0 = static_cast<int>(dep0);
        J.ndeps = static_cast<int>(deps[j].size());
        dep0 += deps[j].size();
        J.ldaux = g.ldaux;
        J.aux = static_cast<const __nv_bfloat16*>(g.aux);
        J.bias = static_cast<const __nv_bfloat16*>(g.bias);
        EpiArgs ea;
        choose_l2_hints(g, 2, &ea);
        J.hint_a = ea.hint_a;
        J.hint_b = ea.hint_b;
        J.hint_out = ea.hint_out;
        bool ok;
        if (g.a_mn)
            ok = add_map(&J.map_a, g.A, false, g.Mg, g.Kg, g.lda, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
        else
            ok = add_map(&J.map_a, g.A, false, g.Kg, g.Mg, g.lda, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
        if (ok) {
            if (g.b_mn)
                ok = add_map(&J.map_b, g.B, false, g.Ng, g.Kg, g.ldb, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B);
            else
                ok = add_map(&J.map_b, g.B, false, g.Kg, g.Ng, g.ldb, BK, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        const bool f32_out = g.epi == EPI_F32;
        const CUtensorMapSwizzle osw = f32_out ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        if (ok) ok = add_map(&J.map_o0, g.out0, f32_out, g.Ng, g.Mg, g.ld0, 32, 32, osw);
        J.map_o1 = J.map_o0;
        if (ok && g.epi == EPI_GELU_DUAL) ok = add_map(&J.map_o1, g.out1, false, g.Ng, g.Mg, g.ld1, 32, 32, osw);
        if (!ok) return fail(ZB_ERR_CUDA, why);
        J.target = static_cast<uint32_t>(tiles[j]) * SIGNALS_PER_TILE;
    }


    // -------------------------------------------- tables and launch
    const Layout L = table_layout(maps.size(), nj, ndeps, ntiles);
    if (!table || (reinterpret_cast<uintptr_t>(table) & 255u)) return fail(ZB_ERR_ALIGN, "persistent replay: table");
    const size_t trace_bytes = trace_on() ? align256(ntiles * sizeof(TraceRec)) : 0;
    if (table_bytes < L.total + trace_bytes)
        return fail(ZB_ERR_WORKSPACE, "persistent replay: workspace too small for its tables");
    std::vector<uint8_t> img(L.done, 0);
    std::memcpy(img.data() + L.maps, maps.data(), maps.size() * sizeof(CUtensorMap));
    std::memcpy(img.data() + L.jobs, rj.data(), nj * sizeof(RJob));
    {
        int* dp = reinterpret_cast<int*>(img.data() + L.deps);
        for (size_t j = 0; j < nj; ++j)
            for (int d : deps[j]) *dp++ = d;
        std::memcpy(img.data() + L.entries, plan.order.data(), ntiles * sizeof(uint32_t));
    }
    uint8_t* base = static_cast<uint8_t*>(table);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TraceRec* trace = nullptr;
    if (trace_bytes) {
        // the records go at the very end of the table area, host fields set
        trace = reinterpret_cast<TraceRec*>(base + table_bytes - trace_bytes);
        std::vector<TraceRec> tr(ntiles);
        for (size_t e = 0; e < ntiles; ++e)
            tr[e] = TraceRec{plan.order[e], plan.order_pair[e], plan.order_start[e], 0, 0, 0, 0, 0, 0, 0};
        cudaError_t te = cudaMemcpyAsync(trace, tr.data(), ntiles * sizeof(TraceRec), cudaMemcpyHostToDevice, st);
        if (te == cudaSuccess) te = cudaStreamSynchronize(st);
        if (te != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("trace setup: ") + cudaGetErrorString(te));
    }
    {
        std::vector<UploadChunk> chunk(1);
        UploadChunk& c = chunk[0];
        for (size_t o = 0; o < img.size(); o += UPLOAD_CHUNK) {
            const size_t n = std::min<size_t>(UPLOAD_CHUNK, img.size() - o);
            c.dst = base + o;
            c.bytes = static_cast<uint32_t>((n + 15) & ~static_cast<size_t>(15));
            std::memcpy(c.data, img.data() + o, n);
            zb_replay_upload_kernel<<<16, 128, 0, st>>>(c);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("table upload: ") + cudaGetErrorString(e));
        }
    }
    cudaError_t e = cudaMemsetAsync(base + L.done, 0, (nj + 2) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));

    std::vector<RParams> rpv(1);  // ~31 KB: not on the stack
    RParams& rp = rpv[0];
    std::memset(&rp, 0, sizeof(rp));
    rp.maps = reinterpret_cast<const CUtensorMap*>(base + L.maps);
    rp.jobs = reinterpret_cast<const RJob*>(base + L.jobs);
    rp.deps = reinterpret_cast<const int*>(base + L.deps);
    rp.entries = reinterpret_cast<const uint32_t*>(base + L.entries);
    rp.done = reinterpret_cast<uint32_t*>(base + L.done);
    rp.err = err;
    rp.trace = trace;
    rp.njobs = static_cast<int>(nj);
    rp.ntiles = static_cast<int>(ntiles);
    static const bool param_maps = [] {
        const char* v = std::getenv("ZB_REPLAY_PARAM_MAPS");
        return !(v && v[0] == '0');
    }();
    if (param_maps && maps.size() <= static_cast<size_t>(PARAM_MAPS)) {
        rp.nparam = static_cast<int>(maps.size());
        std::memcpy(rp.pmaps, maps.data(), maps.size() * sizeof(CUtensorMap));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * npairs, 1, 1);
    cfg.blockDim = dim3(REPLAY_THREADS, 1, 1);
    cfg.dynamicSmemBytes = replay_smem_bytes();
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, zb_replay_tc_kernel, rp);
    if (e != cudaSuccess) return fail(ZB_ERR_CUDA, std::string("persistent replay launch: ") + cudaGetErrorString(e));
    if (trace_on())
        std::fprintf(stderr, "persistent replay: %zu GEMMs, %zu tiles, %zu tensor maps (%d in parameters), %zu deps, %d pairs\n",
                     nj, ntiles, maps.size(), rp.nparam, ndeps, npairs);
    if (info) {
        info->jobs = nj;
        info->tiles = ntiles;
        info->maps = maps.size();
        info->deps = ndeps;
        info->pairs = static_cast<size_t>(npairs);
        info->table_bytes = L.total;
        info->upload_launches = (img.size() + UPLOAD_CHUNK - 1) / UPLOAD_CHUNK;
        info->est_makespan_kb = static_cast<double>(makespan) / 16.0;
    }
    return ZB_OK;
}

}  // namespace zb
