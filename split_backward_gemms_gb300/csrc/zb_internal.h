// zb_internal.h — declarations shared by the library's translation units.
// Not part of the public ABI (see include/zb.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/zb.h"

namespace zb {

// ---------------------------------------------------------------- errors
zb_status fail(zb_status st, const std::string& msg);  // sets zb_last_error, returns st
void clear_error();

// Device error word of the current device (bit set by a bounded wait that
// gave up).  Returns nullptr with a message on CUDA failure.
unsigned int* device_error_word();

// ---------------------------------------------------------------- GEMMs
enum Epilogue : int {
    EPI_STORE_BF16 = 0,  // out0 = bf16(acc (+ bias[col]))
    EPI_GELU_DUAL = 1,   // out0 = bf16(acc + bias) = H; out1 = bf16(GeLU(acc + bias)) = A
    EPI_GELU_BWD = 2,    // out0 = bf16(acc * GeLU'(aux))  (aux = H, bf16)
    EPI_F32 = 3          // out0 (fp32) = (accumulate ? out0 : 0) + acc
};

// D[Mg,Ng] = sum_k Aop(m,k) Bop(k,n) with bf16 operands, fp32 accumulation.
//  a_mn = 0: Aop(m,k) = A[m*lda + k]   (K-major)
//  a_mn = 1: Aop(m,k) = A[k*lda + m]   (MN-major)
//  b_mn = 0: Bop(k,n) = B[n*ldb + k]   (K-major)
//  b_mn = 1: Bop(k,n) = B[k*ldb + n]   (MN-major)
struct GemmBf16 {
    int64_t Mg = 0, Ng = 0, Kg = 0;
    const void* A = nullptr; int64_t lda = 0; int a_mn = 0;
    const void* B = nullptr; int64_t ldb = 0; int b_mn = 0;
    int epi = EPI_STORE_BF16;
    void* out0 = nullptr; int64_t ld0 = 0;
    void* out1 = nullptr; int64_t ld1 = 0;
    const void* aux = nullptr; int64_t ldaux = 0;
    const void* bias = nullptr;  // bf16 [Ng] or nullptr
    int accumulate = 0;
    int act = ZB_ACT_GELU_ERF;
    // split K over a cluster of CTAs when the tiles alone leave SMs idle
    // (bf16-output epilogues only)
    int allow_split = 0;
    // launch as a programmatic dependent of the previous kernel in the stream
    // (its setup overlaps that kernel's tail); only where no other stream's
    // kernels compete for the SMs its waiting CTAs would hold
    int allow_pdl = 0;
    // with allow_pdl: this GEMM reads and writes nothing the previous kernel
    // in the stream writes, so it starts without waiting for that kernel and
    // waits for it just before exiting instead (its own completion then still
    // implies that kernel's, for whatever follows in the stream)
    int independent_of_prev = 0;
    // a grouped launch: a second problem with the same epilogue (fp32
    // only), K and operand majors, run by the same persistent kernel after
    // this one's tiles (one launch for the W pass's two GEMMs); the two must
    // not write what the other reads or writes
    const GemmBf16* second = nullptr;
};
zb_status gemm_bf16_tc(const GemmBf16& g, void* stream);
// The CTA group gemm_bf16_tc would choose for g (1 or 2).
int gemm_bf16_cta_group(const GemmBf16& g);

// Persistent replay (replay_tc.cu): every GEMM of an op list in one
// persistent launch on CTA pairs, in the order the dependencies between the
// GEMMs' byte ranges allow (jobs in list order; no grouped records).  The
// tables go into `table` (256-byte aligned, replay_table_bytes bytes for
// the list's GEMM and tile counts).
struct ReplayInfo {
    size_t jobs = 0, tiles = 0, maps = 0, deps = 0, pairs = 0, table_bytes = 0, upload_launches = 0;
    double est_makespan_kb = 0.0;  // simulated makespan, in one K block's MMA time on a pair
};
zb_status replay_persistent(const std::vector<GemmBf16>& jobs, void* table, size_t table_bytes, void* stream,
                            ReplayInfo* info);
// The host plan of a persistent replay (no device access): tiles per GEMM,
// dependencies (reduced), the CTA pairs' tile lists (job << 18 | tile, in
// order) with their simulated starts (1/16 of a K block's MMA time), the
// simulated makespan and the priority rule used; checked deadlock-free.
struct ReplayPlan {
    std::vector<long long> tiles;
    size_t ntiles = 0, ndeps = 0;
    std::vector<std::vector<int>> deps;
    std::vector<std::vector<uint32_t>> lists;
    std::vector<std::vector<int64_t>> starts;
    // every tile in the order the pairs take them (simulated start, then
    // pair), with its simulated start and pair
    std::vector<uint32_t> order;
    std::vector<int64_t> order_start;
    std::vector<uint32_t> order_pair;
    int64_t makespan = 0;
    bool by_level = false;
};
zb_status plan_replay(const std::vector<GemmBf16>& jobs, int npairs, ReplayPlan* plan);
// GEMMs and CTA-pair tiles an op list replays (for the table size).
zb_status replay_count(const zb_block& b, const zb_op* ops, size_t n_ops, size_t* njobs, size_t* ntiles);
size_t replay_table_bytes(size_t njobs, size_t ntiles);

// fp32 FFMA GEMM (no TF32): C[m*ldc + n] (+)= sum_k A[m*sam + k*sak] * B[k*sbk + n*sbn]
struct GemmF32 {
    int64_t Mg = 0, Ng = 0, Kg = 0;
    const float* A = nullptr; int64_t sam = 0, sak = 0;
    const float* B = nullptr; int64_t sbk = 0, sbn = 0;
    float* C = nullptr; int64_t ldc = 0;
    int accumulate = 0;
};
zb_status gemm_f32_simt(const GemmF32& g, void* stream);

// db[n] (+)= sum_{r < rows} X[r*ld + n], fp32 accumulation in row order.
zb_status colsum_bf16(const void* X, int64_t rows, int64_t cols, int64_t ld, float* db,
                      int accumulate, void* stream);
zb_status colsum_f32(const float* X, int64_t rows, int64_t cols, int64_t ld, float* db,
                     int accumulate, void* stream);
// out[i] = bf16(x[i]) ... unused helpers kept out.

// ---------------------------------------------------------------- schedules
struct OpCheck {
    zb_status st = ZB_OK;
    std::string msg;
};
// Validate an op list against the replay rules.
OpCheck validate_ops(const zb_op* ops, size_t n, int P, int m);

// Map an op list of a (possibly multi-chunk) pipeline onto its chain of
// virtual stages: vops[i] has stage = the virtual stage of (stage, chunk) and
// chunk = 0; dev[i] = the op's stage (device); *L = chunks * P (P for one
// chunk).  Checks the pipeline's chunks / layout and every op's stage and
// chunk range.
zb_status virtualize_ops(const zb_pipeline& pl, const zb_op* ops, size_t n, std::vector<zb_op>* vops,
                         std::vector<int>* dev, int* L);

// Arena plan: for every op, which slots its outputs occupy and which slots
// it releases.  Two size classes: "row" buffers [M,h] and "ffn" buffers [M,f].
enum BufKind : int { BUF_X = 0, BUF_H, BUF_A, BUF_DH, BUF_DY, BUF_COUNT };
struct ArenaPlan {
    size_t row_bytes = 0, ffn_bytes = 0;  // per-slot (256-B aligned)
    int row_slots = 0, ffn_slots = 0;     // peak simultaneous slots per class
    size_t workspace_bytes = 0;
    size_t peak_live_bytes = 0;
    size_t stats_offset = 0, stats_bytes = 0;  // per-stage gradient-statistics scratch
    // slot index per (stage, micro, BufKind); -1 when the buffer is caller-owned
    std::vector<int> slot;  // index: ((s*m + j) * BUF_COUNT + kind)
    // temporary slots for Y of the last stage / dX of stage 0 when no output
    // pointer is given: one per op index (or -1)
    std::vector<int> tmp_slot;
    // per op: indices of the ops that last released a slot this op takes
    // (its next writer must follow them when ops run on several streams)
    std::vector<std::vector<int>> reuse_deps;
    int P = 0, m = 0;
    int at(int s, int j, int k) const { return slot[(static_cast<size_t>(s) * m + j) * BUF_COUNT + k]; }
};
// has_y_out / has_dx_out: whether the caller supplies the last stage's Y /
// stage 0's dX for every microbatch (else a temporary slot is used).
zb_status plan_arena(const zb_pipeline& pl, const zb_op* ops, size_t n, bool has_y_out,
                     bool has_dx_out, ArenaPlan* plan);

bool block_bytes(const zb_block& b, size_t* row_bytes, size_t* ffn_bytes);

}  // namespace zb
