// interleaved.cpp — multi-chunk pipeline orderings and the mapping of their
// op lists onto the chain of virtual stages.
//
// A stage (device) holding v model chunks makes the model a chain of
// L = v P virtual stages.  Layouts: cyclic, chunk c of stage s is c P + s
// ("Pipeline Schedules: GPipe, 1F1B and Zero Bubble", section "Interleaved
// stages"); V, chunk 0 of stage s is s and chunk 1 is 2P-1-s ("Zero Bubble
// Pipeline Parallelism", paper-graph-ui summary, §6 "ZB-V": stage i holds
// chunks i and 2p-i+1).  Dependencies are the one-chunk ones on the chain:
// F(k,j) after F(k-1,j); B(k,j) after F(k,j) and B(k+1,j); W(k,j) after
// B(k,j); T_comm between virtual stages on different devices.  A chunk pass
// lasts T/v of the stage's pass time, so the ideal per-stage time stays
// m (T_F + T_B + T_W).
//
// Orderings:
//   1F1B-I  the interleaved 1F1B the pages cite (summary §5 "1F1B-I"): fixed
//           per-stage sequences (warm-up, F / fused-BW alternation, drain);
//   ZB-V    the V layout with the handcrafted orderings' placement rules and
//           a P M_B activation cap (summary §6), on a simulated timeline.
#include <algorithm>
#include <cmath>
#include <string>
#include <utility>
#include <vector>

#include "zb_internal.h"

namespace {

struct Ev {
    int kind, dev, chunk, micro;
    double start, end;
};

struct Tm {
    double f = 1.0, b = 1.0, w = 1.0, comm = 0.0;
};

int vstage(int layout, int P, int s, int c) {
    if (layout == ZB_LAYOUT_V) return c == 0 ? s : 2 * P - 1 - s;
    return c * P + s;
}

void dev_chunk(int layout, int P, int k, int* s, int* c) {
    if (layout == ZB_LAYOUT_V) {
        *s = k < P ? k : 2 * P - 1 - k;
        *c = k < P ? 0 : 1;
    } else {
        *s = k % P;
        *c = k / P;
    }
}

double pass_len(const Tm& T, int kind, int v) {
    if (kind == ZB_OP_F) return T.f / v;
    if (kind == ZB_OP_B) return T.b / v;
    if (kind == ZB_OP_W) return T.w / v;
    return (T.b + T.w) / v;  // fused BW
}

// --------------------------------------------------------------- 1F1B-I
// (chunk, micro) of a stage's i-th chunk forward: microbatches enter in
// groups of P and every group visits the chunks in order.
std::pair<int, int> ilv_fwd(int P, int v, long long i) {
    const long long g = i / (static_cast<long long>(P) * v);
    const long long r = i % (static_cast<long long>(P) * v);
    return {static_cast<int>(r / P), static_cast<int>(g * P + i % P)};
}

struct SeqOp {
    int kind, chunk, micro;
};

std::vector<SeqOp> ilv_seq(int P, int v, int m, int s) {
    const long long total = static_cast<long long>(v) * m;
    const long long warm = std::min<long long>(2LL * (P - 1 - s) + static_cast<long long>(v - 1) * P, total);
    std::vector<SeqOp> q;
    q.reserve(static_cast<size_t>(2 * total));
    for (long long i = 0; i < warm; ++i) {
        auto f = ilv_fwd(P, v, i);
        q.push_back({ZB_OP_F, f.first, f.second});
    }
    for (long long i = 0; i < total; ++i) {
        if (warm + i < total) {
            auto f = ilv_fwd(P, v, warm + i);
            q.push_back({ZB_OP_F, f.first, f.second});
        }
        auto b = ilv_fwd(P, v, i);
        q.push_back({ZB_OP_BW, v - 1 - b.first, b.second});
    }
    return q;
}

// Each stage runs its sequence in order, every pass as soon as its producers
// have ended; the start times do not depend on the order stages are visited.
bool sim_ilv(int P, int v, int m, const Tm& T, std::vector<Ev>* out) {
    const int L = v * P;
    const int layout = ZB_LAYOUT_CYCLIC;
    std::vector<std::vector<SeqOp>> seq(P);
    for (int s = 0; s < P; ++s) seq[s] = ilv_seq(P, v, m, s);
    const size_t LM = static_cast<size_t>(L) * m;
    std::vector<double> endF(LM, -1.0), endBW(LM, -1.0);
    std::vector<size_t> pos(P, 0);
    std::vector<double> freeT(P, 0.0);
    bool progress = true;
    while (progress) {
        progress = false;
        for (int s = 0; s < P; ++s) {
            while (pos[s] < seq[s].size()) {
                const SeqOp& o = seq[s][pos[s]];
                const int k = vstage(layout, P, s, o.chunk);
                const size_t id = static_cast<size_t>(k) * m + o.micro;
                double ready = 0.0;
                bool ok = true;
                auto need = [&](double e, int kd) {
                    if (e < 0) {
                        ok = false;
                        return;
                    }
                    int ds, dc;
                    dev_chunk(layout, P, kd, &ds, &dc);
                    ready = std::max(ready, e + (ds != s ? T.comm : 0.0));
                };
                if (o.kind == ZB_OP_F) {
                    if (k > 0) need(endF[id - m], k - 1);
                } else {
                    need(endF[id], k);
                    if (ok && k < L - 1) need(endBW[id + m], k + 1);
                }
                if (!ok) break;
                const double st = std::max(ready, freeT[s]);
                const double e = st + pass_len(T, o.kind, v);
                (o.kind == ZB_OP_F ? endF : endBW)[id] = e;
                freeT[s] = e;
                out->push_back({o.kind, s, o.chunk, o.micro, st, e});
                ++pos[s];
                progress = true;
            }
        }
    }
    for (int s = 0; s < P; ++s)
        if (pos[s] < seq[s].size()) return false;
    return true;
}

// ------------------------------------------------------------------ ZB-V
// Whenever a stage is free it takes, among its passes that can start at the
// earliest moment: a W when it holds `limit` live chunk activations (only a
// W frees one), else an F before a B before a W; within a kind the oldest
// microbatch first, then the later virtual stage.  An F needs fewer than
// `limit` live activations; a chunk-0 forward fewer than limit - 1 unless a
// W of the stage is pending, so the last slot either stays free for a
// chunk-1 forward or is freed by that W next, and the oldest unfinished
// forward can always advance.  A W comes from the stage's pending ones,
// oldest first.  Stages are served in order of their pass's start.  At
// T_F = T_B = T_W this leaves no stage idle between its first and last pass.
bool sim_zbv(int P, int m, const Tm& T, std::vector<Ev>* out) {
    const int layout = ZB_LAYOUT_V, v = 2, L = 2 * P, limit = 2 * P;
    const size_t LM = static_cast<size_t>(L) * m;
    std::vector<int> nF(L, 0), nB(L, 0);
    std::vector<double> endF(LM, 0.0), endB(LM, 0.0);
    std::vector<double> freeT(P, 0.0);
    std::vector<int> live(P, 0);
    std::vector<std::vector<std::pair<int, int>>> pend(P);  // (micro, k)
    long long todo = 3LL * L * m;
    struct Cand {
        double start;
        int rank, micro, negk, kind, k;
    };
    auto better = [](const Cand& a, const Cand& b) {  // among equal starts
        if (a.rank != b.rank) return a.rank < b.rank;
        if (a.micro != b.micro) return a.micro < b.micro;
        return a.negk < b.negk;
    };
    while (todo > 0) {
        bool have = false;
        Cand best{};
        int best_s = -1;
        for (int s = 0; s < P; ++s) {
            Cand c{};
            bool any = false;
            auto offer = [&](const Cand& x) {
                if (!any || x.start < c.start || (x.start == c.start && better(x, c))) c = x;
                any = true;
            };
            for (int ci = 0; ci < 2; ++ci) {
                const int k = vstage(layout, P, s, ci);
                int j = nB[k];
                if (j < nF[k]) {
                    bool dep_done;
                    double r;
                    if (k == L - 1) {
                        dep_done = true;
                        r = endF[static_cast<size_t>(k) * m + j];
                    } else {
                        dep_done = nB[k + 1] > j;
                        r = dep_done ? endB[static_cast<size_t>(k + 1) * m + j] : 0.0;
                        int ds, dc;
                        dev_chunk(layout, P, k + 1, &ds, &dc);
                        if (ds != s) r += T.comm;
                    }
                    if (dep_done) offer({std::max(r, freeT[s]), 2, j, -k, ZB_OP_B, k});
                }
                j = nF[k];
                // a chunk-0 forward leaves the last slot to chunk 1 unless a W
                // is pending (a full stage runs that W next)
                const bool room = live[s] < limit && (k >= P || live[s] < limit - 1 || !pend[s].empty());
                if (j < m && room && (k == 0 || nF[k - 1] > j)) {
                    double r = 0.0;
                    if (k > 0) {
                        r = endF[static_cast<size_t>(k - 1) * m + j];
                        int ds, dc;
                        dev_chunk(layout, P, k - 1, &ds, &dc);
                        if (ds != s) r += T.comm;
                    }
                    offer({std::max(r, freeT[s]), 1, j, -k, ZB_OP_F, k});
                }
            }
            if (!pend[s].empty()) {
                auto it = std::min_element(pend[s].begin(), pend[s].end(), [](const auto& a, const auto& b) {
                    return a.first != b.first ? a.first < b.first : a.second > b.second;
                });
                const int j = it->first, k = it->second;
                const int wrank = live[s] >= limit ? 0 : 3;
                offer({std::max(endB[static_cast<size_t>(k) * m + j], freeT[s]), wrank, j, -k, ZB_OP_W, k});
            }
            if (!any) continue;
            if (!have || c.start < best.start) {
                best = c;
                best_s = s;
                have = true;
            }
        }
        if (!have) return false;
        const int s = best_s, k = best.k, j = best.micro;
        const double e = best.start + pass_len(T, best.kind, v);
        int ds, dc;
        dev_chunk(layout, P, k, &ds, &dc);
        out->push_back({best.kind, s, dc, j, best.start, e});
        freeT[s] = e;
        const size_t id = static_cast<size_t>(k) * m + j;
        if (best.kind == ZB_OP_F) {
            endF[id] = e;
            ++nF[k];
            ++live[s];
        } else if (best.kind == ZB_OP_B) {
            endB[id] = e;
            ++nB[k];
            pend[s].push_back({j, k});
        } else {
            for (size_t q = 0; q < pend[s].size(); ++q)
                if (pend[s][q].first == j && pend[s][q].second == k) {
                    pend[s].erase(pend[s].begin() + static_cast<long>(q));
                    break;
                }
            --live[s];
        }
        --todo;
    }
    return true;
}

// List order (start, stage); OPT(stage, chunk) right after the last op of
// each virtual stage.
size_t emit(std::vector<Ev>& ev, int P, int v, int layout, zb_op* out) {
    std::stable_sort(ev.begin(), ev.end(), [](const Ev& a, const Ev& b) {
        return a.start != b.start ? a.start < b.start : a.dev < b.dev;
    });
    const int L = v * P;
    std::vector<long long> last(L, -1);
    for (size_t i = 0; i < ev.size(); ++i) last[vstage(layout, P, ev[i].dev, ev[i].chunk)] = static_cast<long long>(i);
    size_t w = 0;
    for (size_t i = 0; i < ev.size(); ++i) {
        out[w++] = zb_op{static_cast<uint8_t>(ev[i].kind), static_cast<uint8_t>(ev[i].chunk),
                         static_cast<uint16_t>(ev[i].dev), static_cast<uint32_t>(ev[i].micro)};
        for (int k = 0; k < L; ++k)
            if (last[k] == static_cast<long long>(i)) {
                int s, c;
                dev_chunk(layout, P, k, &s, &c);
                out[w++] = zb_op{ZB_OP_OPT, static_cast<uint8_t>(c), static_cast<uint16_t>(s), 0};
            }
    }
    return w;
}

// Eq. 3 cost (max per-stage span), bubble rate, peak live chunk activations.
void fill(const std::vector<Ev>& ev, int P, int m, const Tm& T, zb_sim_result* res) {
    std::vector<Ev> sorted = ev;
    std::stable_sort(sorted.begin(), sorted.end(), [](const Ev& a, const Ev& b) { return a.start < b.start; });
    std::vector<double> first(P, -1.0), lastv(P, 0.0);
    std::vector<int> live(P, 0), peak(P, 0);
    for (const Ev& e : sorted) {
        if (first[e.dev] < 0 || e.start < first[e.dev]) first[e.dev] = e.start;
        lastv[e.dev] = std::max(lastv[e.dev], e.end);
        if (e.kind == ZB_OP_F) peak[e.dev] = std::max(peak[e.dev], ++live[e.dev]);
        else if (e.kind == ZB_OP_W || e.kind == ZB_OP_BW) --live[e.dev];
    }
    double cost = 0.0;
    int pk = 0;
    for (int s = 0; s < P; ++s) {
        cost = std::max(cost, lastv[s] - first[s]);
        pk = std::max(pk, peak[s]);
    }
    res->cost = cost;
    res->ideal = m * (T.f + T.b + T.w);
    res->bubble_rate = cost > 0 ? (cost - res->ideal) / cost : 0.0;
    res->peak_live_microbatches = static_cast<uint32_t>(pk);
    res->peak_live_stage0 = static_cast<uint32_t>(peak[0]);
}

zb_status run(int32_t kind, int32_t P, int32_t v, int32_t m, const Tm& T, zb_op* out, size_t* n_ops,
              zb_sim_result* res) {
    if (!n_ops) return zb::fail(ZB_ERR_INVALID_ARG, "n_ops is NULL");
    if (kind != ZB_SCHED_1F1B_I && kind != ZB_SCHED_ZBV)
        return zb::fail(ZB_ERR_INVALID_ARG, "kind must be ZB_SCHED_1F1B_I or ZB_SCHED_ZBV");
    if (kind == ZB_SCHED_ZBV && v != 2) return zb::fail(ZB_ERR_INVALID_ARG, "ZB-V has exactly 2 chunks per stage");
    if (kind == ZB_SCHED_1F1B_I && (v < 2 || v > 255))
        return zb::fail(ZB_ERR_INVALID_ARG, "1F1B-I needs 2 <= v <= 255 chunks per stage");
    if (P < 1 || m < 1 || static_cast<long long>(P) * v > 65535 ||
        static_cast<long long>(P) * v * m > (1LL << 20))
        return zb::fail(ZB_ERR_SHAPE, "P and m must be >= 1 (v P <= 65535, v P m <= 2^20)");
    if (kind == ZB_SCHED_1F1B_I && m % P != 0) return zb::fail(ZB_ERR_SHAPE, "1F1B-I needs m to be a multiple of P");
    const size_t L = static_cast<size_t>(P) * v;
    const size_t per = kind == ZB_SCHED_1F1B_I ? 2 : 3;
    const size_t total = L * static_cast<size_t>(m) * per + L;
    if (out && *n_ops < total) {
        *n_ops = total;
        return zb::fail(ZB_ERR_INVALID_ARG, "output capacity too small");
    }
    if (!out && !res) {
        *n_ops = total;
        zb::clear_error();
        return ZB_OK;
    }
    std::vector<Ev> ev;
    ev.reserve(total);
    const bool ok = kind == ZB_SCHED_1F1B_I ? sim_ilv(P, v, m, T, &ev) : sim_zbv(P, m, T, &ev);
    if (!ok) return zb::fail(ZB_ERR_SCHEDULE, "schedule simulation deadlocked");
    if (res) fill(ev, P, m, T, res);
    *n_ops = out ? emit(ev, P, v, kind == ZB_SCHED_ZBV ? ZB_LAYOUT_V : ZB_LAYOUT_CYCLIC, out) : total;
    zb::clear_error();
    return ZB_OK;
}

}  // namespace

namespace zb {

zb_status virtualize_ops(const zb_pipeline& pl, const zb_op* ops, size_t n, std::vector<zb_op>* vops,
                         std::vector<int>* dev, int* L) {
    const int v = pl.chunks <= 1 ? 1 : pl.chunks;
    if (pl.chunks < 0 || pl.chunks > 255) return fail(ZB_ERR_INVALID_ARG, "pipeline.chunks must be in [0, 255]");
    if (v > 1 && pl.layout != ZB_LAYOUT_CYCLIC && pl.layout != ZB_LAYOUT_V)
        return fail(ZB_ERR_INVALID_ARG, "pipeline.layout must be ZB_LAYOUT_CYCLIC or ZB_LAYOUT_V");
    if (v > 1 && pl.layout == ZB_LAYOUT_V && v != 2) return fail(ZB_ERR_INVALID_ARG, "the V layout has 2 chunks");
    if (pl.P < 1 || pl.m < 1) return fail(ZB_ERR_SHAPE, "P and m must be >= 1");
    if (static_cast<long long>(pl.P) * v > 65535) return fail(ZB_ERR_SHAPE, "chunks * P must be <= 65535");
    if (!ops && n) return fail(ZB_ERR_INVALID_ARG, "ops is NULL");
    *L = pl.P * v;
    vops->resize(n);
    dev->resize(n);
    for (size_t i = 0; i < n; ++i) {
        const zb_op& o = ops[i];
        if (o.stage >= pl.P || o.chunk >= v)
            return fail(ZB_ERR_SCHEDULE, "op " + std::to_string(i) + ": stage or chunk out of range");
        const int k = v == 1 ? o.stage : vstage(pl.layout, pl.P, o.stage, o.chunk);
        (*vops)[i] = zb_op{o.kind, 0, static_cast<uint16_t>(k), o.micro};
        (*dev)[i] = o.stage;
    }
    return ZB_OK;
}

}  // namespace zb

namespace {

zb_status read_times(const zb_sim_times* times, Tm* T) {
    T->f = times->t_f;
    T->b = times->t_b;
    T->w = times->t_w;
    T->comm = times->t_comm;
    if (!(T->f > 0) || !(T->b > 0) || !(T->w > 0) || !(T->comm >= 0) || !std::isfinite(T->f) ||
        !std::isfinite(T->b) || !std::isfinite(T->w) || !std::isfinite(T->comm))
        return zb::fail(ZB_ERR_INVALID_ARG, "pass times must be finite, T_F/T_B/T_W > 0, T_comm >= 0");
    return ZB_OK;
}

}  // namespace

extern "C" zb_status zb_make_interleaved_schedule(int32_t kind, int32_t P, int32_t v, int32_t m, zb_op* out,
                                                  size_t* n_ops) {
    return run(kind, P, v, m, Tm(), out, n_ops, nullptr);
}

extern "C" zb_status zb_simulate_interleaved_schedule(int32_t kind, int32_t P, int32_t v, int32_t m,
                                                      const zb_sim_times* times, zb_op* out, size_t* n_ops,
                                                      zb_sim_result* result) {
    if (!times || !result) return zb::fail(ZB_ERR_INVALID_ARG, "times or result is NULL");
    Tm T;
    zb_status s = read_times(times, &T);
    if (s != ZB_OK) return s;
    size_t dummy = 0;
    return run(kind, P, v, m, T, out, n_ops ? n_ops : &dummy, result);
}
