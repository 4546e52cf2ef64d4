// schedule.cpp — host-side pipeline logic: the handcrafted orderings
// (1F1B, ZB-H1, ZB-H2), op-list validation and the deferred-W arena plan.
//
// Orderings after "Zero Bubble Pipeline Parallelism" (paper-graph-ui summary
// of arXiv 2401.10241), §3.4 "Handcrafted Schedule ZB-H1 / ZB-H2", Table 2,
// the heuristic's phases "W insertion to fill bubbles" / "Memory-triggered W
// insertion" / "Cool-down", and "Pipeline Schedules: GPipe, 1F1B and Zero
// Bubble", section "1F1B: same bubble, bounded memory".  Pass times are equal
// (one time unit; the fused 1F1B backward takes two), so the simulator runs
// on integers.  Lifetimes after the summary's "The Memory Model" (F stores
// M_B, B trades M_B for M_W, W frees M_W) and "Pipeline Schedules", "Zero
// bubble": per-stage instruction sequences with gradient-buffer lifetime
// management.
#include <algorithm>
#include <cmath>
#include <limits>
#include <cstring>
#include <deque>
#include <set>
#include <string>
#include <vector>

#include "zb_internal.h"

namespace {

struct SimEvent {
    int kind, stage, micro;
    double start, end;
};

int warmup_count(int kind, int P, int m, int s) {
    int w = 0;
    if (kind == ZB_SCHED_1F1B) w = P - 1 - s;
    else if (kind == ZB_SCHED_ZBH1) w = P - s;
    else w = 2 * (P - 1 - s) + 1;
    return std::min(w, m);
}

// Fixed F/B (F/BW for 1F1B) sequence of stage s.
std::vector<std::pair<int, int>> fb_order(int kind, int P, int m, int s) {
    std::vector<std::pair<int, int>> q;
    const int w = warmup_count(kind, P, m, s);
    for (int j = 0; j < w; ++j) q.push_back({ZB_OP_F, j});
    int next_f = w;
    for (int b = 0; b < m; ++b) {
        if (kind == ZB_SCHED_1F1B) {
            if (next_f < m) q.push_back({ZB_OP_F, next_f++});
            q.push_back({ZB_OP_BW, b});
        } else {
            q.push_back({ZB_OP_B, b});
            if (next_f < m) q.push_back({ZB_OP_F, next_f++});
        }
    }
    return q;
}

struct PassTimes {
    double f = 1.0, b = 1.0, w = 1.0, comm = 0.0;
    double len(int kind) const {
        if (kind == ZB_OP_F) return f;
        if (kind == ZB_OP_B) return b;
        if (kind == ZB_OP_W) return w;
        return b + w;  // fused BW
    }
};

// List-scheduling simulation of one ordering: every stage runs its next F/B
// as soon as its producers have ended (plus T_comm across stages), else its
// oldest pending W; a W is forced before an F when the stage's live
// microbatches reach the ordering's cap.  Decisions are taken in time order,
// so each one sees every pass that ends by then.
bool simulate(int kind, int P, int m, const PassTimes& T, std::vector<SimEvent>* out) {
    const int live_cap = kind == ZB_SCHED_ZBH1 ? P : (kind == ZB_SCHED_ZBH2 ? 2 * P - 1 : 0);
    struct St {
        std::vector<std::pair<int, int>> seq;
        size_t pos = 0;
        std::deque<int> wq;
        int live = 0;
        double tfree = 0.0;
        bool parked = false;
    };
    std::vector<St> st(P);
    for (int s = 0; s < P; ++s) st[s].seq = fb_order(kind, P, m, s);
    // end times (or -1): fwd_end[s*m+j]; bwd_end = end of B or BW
    std::vector<double> fwd_end(static_cast<size_t>(P) * m, -1.0), bwd_end(static_cast<size_t>(P) * m, -1.0);
    std::vector<double> all_ends;
    auto busy = [&](int s) { return st[s].pos < st[s].seq.size() || !st[s].wq.empty(); };
    auto emit = [&](int s, int k, int j, double t0) {
        const double t1 = t0 + T.len(k);
        out->push_back({k, s, j, t0, t1});
        all_ends.push_back(t1);
        st[s].tfree = t1;
        if (k == ZB_OP_F) {
            fwd_end[static_cast<size_t>(s) * m + j] = t1;
            st[s].live++;
        } else if (k == ZB_OP_B) {
            bwd_end[static_cast<size_t>(s) * m + j] = t1;
            st[s].wq.push_back(j);
        } else if (k == ZB_OP_BW) {
            bwd_end[static_cast<size_t>(s) * m + j] = t1;
            st[s].live--;
        } else {
            st[s].live--;
        }
    };
    // earliest start of (k, s, j) given its producers, -1 if one is unscheduled
    auto ready_time = [&](int s, int k, int j) -> double {
        double t = 0.0;
        if (k == ZB_OP_F) {
            if (s > 0) {
                const double e = fwd_end[static_cast<size_t>(s - 1) * m + j];
                if (e < 0) return -1.0;
                t = e + T.comm;
            }
            return t;
        }
        const double e = fwd_end[static_cast<size_t>(s) * m + j];
        if (e < 0) return -1.0;
        t = e;
        if (s + 1 < P) {
            const double u = bwd_end[static_cast<size_t>(s + 1) * m + j];
            if (u < 0) return -1.0;
            t = std::max(t, u + T.comm);
        }
        return t;
    };
    for (;;) {
        int pick = -1;
        for (int s = 0; s < P; ++s) {
            if (!busy(s) || st[s].parked) continue;
            if (pick < 0 || st[s].tfree < st[pick].tfree) pick = s;
        }
        if (pick < 0) {
            bool any = false;
            for (int s = 0; s < P; ++s) any = any || busy(s);
            if (!any) break;
            return false;  // every stage with work is parked: cannot happen for legal orders
        }
        St& S = st[pick];
        const double now = S.tfree;
        const bool have_fb = S.pos < S.seq.size();
        double ready = -1.0;
        if (have_fb) ready = ready_time(pick, S.seq[S.pos].first, S.seq[S.pos].second);
        bool ran = true;
        if (have_fb && ready >= 0 && ready <= now) {
            const bool force_w = S.seq[S.pos].first == ZB_OP_F && live_cap > 0 &&
                                 S.live >= live_cap && !S.wq.empty();
            if (force_w) {
                const int j = S.wq.front();
                S.wq.pop_front();
                emit(pick, ZB_OP_W, j, now);
            } else {
                emit(pick, S.seq[S.pos].first, S.seq[S.pos].second, now);
                S.pos++;
            }
        } else if (!S.wq.empty()) {
            const int j = S.wq.front();
            S.wq.pop_front();
            emit(pick, ZB_OP_W, j, now);
        } else {
            ran = false;
            if (ready >= 0) {
                S.tfree = ready;
            } else {
                double nxt = -1.0;
                for (double e : all_ends)
                    if (e > now && (nxt < 0 || e < nxt)) nxt = e;
                for (int o = 0; o < P; ++o)
                    if (o != pick && busy(o) && st[o].tfree > now && (nxt < 0 || st[o].tfree < nxt))
                        nxt = st[o].tfree;
                if (nxt < 0) S.parked = true;
                else S.tfree = nxt;
            }
        }
        if (ran)
            for (auto& x : st) x.parked = false;
    }
    return true;
}

// Heuristic automatic scheduler ("Zero Bubble Pipeline Parallelism", summary
// §3 "The Heuristic Scheduling Algorithm" and "The Memory Model").  Memory in
// units of M_B: F +1, B + (r - 1), W -r with r = M_W / M_B.  Whenever a stage
// is free (decisions in time order) it runs, in this priority:
//   1. its next B if ready (critical path);
//   2. its next F if ready, within the memory limit, not more than one F
//      ahead of the next stage when h2 = 1, and - before its first B with
//      h1 = 0 - not delaying that B;
//   3. its oldest pending W if memory blocks the F, or the idle gap before
//      the next F/B is at least T_W, or idling the gap would make this
//      stage's accumulated idle time (counted from its first pass, where its
//      Eq. 3 span starts) the largest of all stages, or only W remain;
//   4. otherwise it idles until its next F/B can start.
bool auto_simulate(int P, int m, const PassTimes& T, double limit, double r, int h1, int h2,
                   std::vector<SimEvent>* out) {
    const double eps = 1e-9;
    std::vector<int> nf(P, 0), nb(P, 0);
    std::vector<std::deque<int>> wq(P);
    std::vector<double> mem(P, 0.0), idle(P, 0.0), tfree(P, 0.0);
    std::vector<char> parked(P, 0);
    std::vector<double> fend(static_cast<size_t>(P) * m, -1.0), bend(static_cast<size_t>(P) * m, -1.0);
    std::vector<double> ends;
    const double NONE = -1.0;
    auto work = [&](int s) { return nf[s] < m || nb[s] < m || !wq[s].empty(); };
    auto f_ready = [&](int s) -> double {
        const int j = nf[s];
        if (j >= m) return NONE;
        if (s == 0) return 0.0;
        const double e = fend[static_cast<size_t>(s - 1) * m + j];
        return e < 0 ? NONE : e + T.comm;
    };
    auto b_ready = [&](int s) -> double {
        const int j = nb[s];
        if (j >= m || j >= nf[s]) return NONE;
        const double e = fend[static_cast<size_t>(s) * m + j];
        if (e < 0) return NONE;
        if (s == P - 1) return e;
        const double u = bend[static_cast<size_t>(s + 1) * m + j];
        return u < 0 ? NONE : std::max(e, u + T.comm);
    };
    auto put = [&](int s, int k, int j, double t0) {
        const double t1 = t0 + T.len(k);
        out->push_back({k, s, j, t0, t1});
        ends.push_back(t1);
        tfree[s] = t1;
        if (k == ZB_OP_F) {
            fend[static_cast<size_t>(s) * m + j] = t1;
            nf[s]++;
            mem[s] += 1.0;
        } else if (k == ZB_OP_B) {
            bend[static_cast<size_t>(s) * m + j] = t1;
            nb[s]++;
            mem[s] += r - 1.0;
            wq[s].push_back(j);
        } else {
            mem[s] -= r;
        }
    };
    for (;;) {
        int s = -1;
        for (int k = 0; k < P; ++k)
            if (work(k) && !parked[k] && (s < 0 || tfree[k] < tfree[s])) s = k;
        if (s < 0) {
            for (int k = 0; k < P; ++k)
                if (work(k)) return false;
            break;
        }
        const double now = tfree[s];
        const double rb = b_ready(s), rf = f_ready(s);
        const bool fits = mem[s] + 1.0 <= limit + eps;
        bool skip = h2 && s < P - 1 && nf[s] - nf[s + 1] > 1;
        if (nb[s] == 0 && !h1 && rf >= 0 && rb >= 0 && rb < std::max(now, rf) + T.f) skip = true;
        const bool f_ok = rf >= 0 && fits && !skip;
        bool acted = true;
        if (rb >= 0 && rb <= now) {
            put(s, ZB_OP_B, nb[s], now);
        } else if (f_ok && rf <= now) {
            put(s, ZB_OP_F, nf[s], now);
        } else if (!wq[s].empty()) {
            double next = NONE;
            if (rb >= 0) next = rb;
            if (f_ok && (next < 0 || rf < next)) next = rf;
            const double gap = next >= 0 ? next - now : std::numeric_limits<double>::infinity();
            const bool mem_block = rf >= 0 && rf <= now && !fits;
            const bool tail = nf[s] == m && nb[s] == m;
            const double most_idle = *std::max_element(idle.begin(), idle.end());
            if (tail || mem_block || gap >= T.w - eps || idle[s] + gap > most_idle + eps) {
                const int j = wq[s].front();
                wq[s].pop_front();
                put(s, ZB_OP_W, j, now);
            } else {
                if (nf[s] > 0) idle[s] += gap;  // idle counts from the stage's first pass
                tfree[s] = next;
            }
        } else {
            acted = false;
            double next = NONE;
            if (rb > now) next = rb;
            if (f_ok && rf > now && (next < 0 || rf < next)) next = rf;
            if (next >= 0) {
                if (nf[s] > 0) idle[s] += next - now;
                tfree[s] = next;
            } else {
                double later = NONE;
                for (double e : ends)
                    if (e > now && (later < 0 || e < later)) later = e;
                for (int o = 0; o < P; ++o)
                    if (o != s && work(o) && tfree[o] > now && (later < 0 || tfree[o] < later)) later = tfree[o];
                if (later >= 0) {
                    if (nf[s] > 0) idle[s] += later - now;
                    tfree[s] = later;
                } else {
                    parked[s] = 1;
                }
            }
        }
        if (acted) std::fill(parked.begin(), parked.end(), 0);
    }
    return true;
}

// Ordered op list (start time, then stage; OPT after each stage's last op).
size_t emit_ops(std::vector<SimEvent>& ev, int P, zb_op* out) {
    std::stable_sort(ev.begin(), ev.end(), [](const SimEvent& a, const SimEvent& b) {
        return a.start != b.start ? a.start < b.start : a.stage < b.stage;
    });
    std::vector<size_t> last(P, 0);
    for (size_t i = 0; i < ev.size(); ++i) last[ev[i].stage] = i;
    size_t w = 0;
    for (size_t i = 0; i < ev.size(); ++i) {
        out[w++] = zb_op{static_cast<uint8_t>(ev[i].kind), 0, static_cast<uint16_t>(ev[i].stage),
                         static_cast<uint32_t>(ev[i].micro)};
        for (int s = 0; s < P; ++s)
            if (last[s] == i) out[w++] = zb_op{ZB_OP_OPT, 0, static_cast<uint16_t>(s), 0};
    }
    return w;
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace

namespace zb {

bool block_bytes(const zb_block& b, size_t* row_bytes, size_t* ffn_bytes) {
    const size_t es = b.dtype == ZB_DT_F32 ? 4 : 2;
    if (b.M <= 0 || b.h <= 0 || b.f <= 0) return false;
    // a single linear map's output is [M,f]: row slots then hold max(h, f)
    const int64_t row_w = b.act == ZB_ACT_NONE ? std::max(b.h, b.f) : b.h;
    *row_bytes = static_cast<size_t>(b.M) * static_cast<size_t>(row_w) * es;
    *ffn_bytes = static_cast<size_t>(b.M) * static_cast<size_t>(b.f) * es;
    return true;
}

OpCheck validate_ops(const zb_op* ops, size_t n, int P, int m) {
    OpCheck r;
    auto bad = [&](zb_status s, const std::string& msg) {
        r.st = s;
        r.msg = msg;
        return r;
    };
    auto name = [](const zb_op& o) {
        static const char* k[] = {"F", "B", "W", "BW", "OPT"};
        return std::string(o.kind < 5 ? k[o.kind] : "?") + "(" + std::to_string(o.stage) + "," +
               std::to_string(o.micro) + ")";
    };
    if (P <= 0 || m <= 0) return bad(ZB_ERR_SHAPE, "P and m must be >= 1");
    if (!ops && n) return bad(ZB_ERR_INVALID_ARG, "ops is NULL");
    const size_t PM = static_cast<size_t>(P) * m;
    // seen[kind][s*m+j]
    std::vector<unsigned char> seen(4 * PM, 0);
    auto has = [&](int k, int s, int j) { return seen[k * PM + static_cast<size_t>(s) * m + j] != 0; };
    std::vector<long long> last_w(P, -1);
    std::vector<char> opt_done(P, 0);
    for (size_t i = 0; i < n; ++i) {
        const zb_op& o = ops[i];
        if (o.kind > ZB_OP_OPT || o.chunk != 0) return bad(ZB_ERR_SCHEDULE, "op " + std::to_string(i) + ": bad kind or chunk");
        if (o.stage >= P) return bad(ZB_ERR_SCHEDULE, "op " + std::to_string(i) + ": stage out of range " + name(o));
        if (o.kind != ZB_OP_OPT && o.micro >= static_cast<uint32_t>(m))
            return bad(ZB_ERR_SCHEDULE, "op " + std::to_string(i) + ": micro out of range " + name(o));
        const int s = o.stage;
        if (opt_done[s]) return bad(ZB_ERR_SCHEDULE, name(o) + " after OPT of its stage");
        if (o.kind == ZB_OP_OPT) {
            opt_done[s] = 1;
            continue;
        }
        const int j = static_cast<int>(o.micro);
        if (has(o.kind, s, j)) return bad(ZB_ERR_SCHEDULE, "duplicate " + name(o));
        if (o.kind == ZB_OP_BW && (has(ZB_OP_B, s, j) || has(ZB_OP_W, s, j)))
            return bad(ZB_ERR_SCHEDULE, "BW mixed with split B/W for " + name(o));
        if ((o.kind == ZB_OP_B || o.kind == ZB_OP_W) && has(ZB_OP_BW, s, j))
            return bad(ZB_ERR_SCHEDULE, "split B/W mixed with BW for " + name(o));
        bool ok = true;
        if (o.kind == ZB_OP_F) {
            ok = s == 0 || has(ZB_OP_F, s - 1, j);
        } else if (o.kind == ZB_OP_B || o.kind == ZB_OP_BW) {
            ok = has(ZB_OP_F, s, j) && (s == P - 1 || has(ZB_OP_B, s + 1, j) || has(ZB_OP_BW, s + 1, j));
        } else {
            ok = has(ZB_OP_B, s, j);
        }
        if (!ok) return bad(ZB_ERR_SCHEDULE, name(o) + " runs before one of its producers");
        if (o.kind == ZB_OP_W || o.kind == ZB_OP_BW) {
            if (j <= last_w[s]) return bad(ZB_ERR_W_ORDER, name(o) + ": weight gradients of a stage must run in ascending micro order");
            last_w[s] = j;
        }
        seen[o.kind * PM + static_cast<size_t>(s) * m + j] = 1;
    }
    for (int s = 0; s < P; ++s)
        for (int j = 0; j < m; ++j) {
            const bool split = has(ZB_OP_B, s, j) && has(ZB_OP_W, s, j);
            if (!has(ZB_OP_F, s, j) || !(split || has(ZB_OP_BW, s, j)))
                return bad(ZB_ERR_SCHEDULE, "missing pass for stage " + std::to_string(s) + " micro " + std::to_string(j));
        }
    return r;
}

zb_status plan_arena(const zb_pipeline& pl, const zb_op* ops, size_t n, bool has_y_out,
                     bool has_dx_out, ArenaPlan* plan) {
    const int P = pl.P, m = pl.m;
    size_t rb = 0, fb = 0;
    if (!block_bytes(pl.blk, &rb, &fb)) return fail(ZB_ERR_SHAPE, "block extents must be >= 1");
    const bool mlp = pl.blk.act != ZB_ACT_NONE;
    plan->P = P;
    plan->m = m;
    plan->row_bytes = align256(rb);
    plan->ffn_bytes = align256(fb);
    plan->slot.assign(static_cast<size_t>(P) * m * BUF_COUNT, -1);
    plan->tmp_slot.assign(n, -1);
    plan->reuse_deps.assign(n, {});
    // Two pools of equal-size slots; lowest free index first (deterministic).
    std::set<int> free_row, free_ffn;
    int n_row = 0, n_ffn = 0;
    size_t live = 0, peak = 0;
    std::vector<int> row_freed_by, ffn_freed_by;  // op that last released each slot
    size_t cur = 0;                               // index of the op being planned
    // Saved activations enter the ledger; a scratch output (the last stage's Y
    // or stage 0's dX when the caller gives no buffer) takes a slot only.
    auto take = [&](bool ffn, bool saved = true) {
        std::set<int>& fr = ffn ? free_ffn : free_row;
        int& cnt = ffn ? n_ffn : n_row;
        int id;
        if (!fr.empty()) {
            id = *fr.begin();
            fr.erase(fr.begin());
            const int prev = (ffn ? ffn_freed_by : row_freed_by)[id];
            if (prev >= 0 && prev != static_cast<int>(cur)) plan->reuse_deps[cur].push_back(prev);
        } else {
            id = cnt++;
            (ffn ? ffn_freed_by : row_freed_by).push_back(-1);
        }
        if (saved) {
            live += ffn ? fb : rb;
            peak = std::max(peak, live);
        }
        return id;
    };
    auto give = [&](bool ffn, int id, bool saved = true) {
        if (id < 0) return;
        (ffn ? free_ffn : free_row).insert(id);
        (ffn ? ffn_freed_by : row_freed_by)[id] = static_cast<int>(cur);
        if (saved) live -= ffn ? fb : rb;
    };
    auto ref = [&](int s, int j, int k) -> int& {
        return plan->slot[(static_cast<size_t>(s) * m + j) * BUF_COUNT + k];
    };
    auto do_b = [&](int s, int j, size_t i) {
        if (mlp) ref(s, j, BUF_DH) = take(true);
        int tmp = -1;
        if (s > 0) ref(s - 1, j, BUF_DY) = take(false);  // dX(s) = dY(s-1)
        else if (!has_dx_out) tmp = take(false, false);
        if (mlp) give(true, ref(s, j, BUF_H));
        give(false, tmp, false);
        if (tmp >= 0) plan->tmp_slot[i] = tmp;
    };
    auto do_w = [&](int s, int j) {
        if (s > 0) give(false, ref(s, j, BUF_X));
        if (mlp) {
            give(true, ref(s, j, BUF_A));
            give(true, ref(s, j, BUF_DH));
        }
        if (s < P - 1) give(false, ref(s, j, BUF_DY));
    };
    for (size_t i = 0; i < n; ++i) {
        cur = i;
        const zb_op& o = ops[i];
        const int s = o.stage, j = static_cast<int>(o.micro);
        switch (o.kind) {
            case ZB_OP_F: {
                if (mlp) {
                    ref(s, j, BUF_H) = take(true);
                    ref(s, j, BUF_A) = take(true);
                }
                if (s < P - 1) {
                    ref(s + 1, j, BUF_X) = take(false);  // Y(s) = X(s+1)
                } else if (!has_y_out) {
                    const int tmp = take(false, false);
                    plan->tmp_slot[i] = tmp;
                    give(false, tmp, false);
                }
                break;
            }
            case ZB_OP_B: do_b(s, j, i); break;
            case ZB_OP_W: do_w(s, j); break;
            case ZB_OP_BW:
                do_b(s, j, i);
                do_w(s, j);
                break;
            default: break;
        }
    }
    plan->row_slots = n_row;
    plan->ffn_slots = n_ffn;
    plan->stats_offset = static_cast<size_t>(n_row) * plan->row_bytes + static_cast<size_t>(n_ffn) * plan->ffn_bytes;
    plan->stats_bytes = align256(zb_grad_stats_scratch_bytes());
    plan->workspace_bytes = plan->stats_offset + static_cast<size_t>(P) * plan->stats_bytes;
    plan->peak_live_bytes = peak;
    if (pl.mem_limit_bytes != 0 && peak > pl.mem_limit_bytes)
        return fail(ZB_ERR_BUDGET, "peak live activation bytes " + std::to_string(peak) + " exceed the limit " +
                                       std::to_string(pl.mem_limit_bytes));
    return ZB_OK;
}

}  // namespace zb

namespace {

// Eq. 3 cost (max per-stage span), bubble rate and peak live microbatches.
void fill_result(const std::vector<SimEvent>& ev, int P, int m, const PassTimes& T, zb_sim_result* res) {
    std::vector<double> first(P, -1.0), lastv(P, 0.0);
    std::vector<int> live(P, 0), peak(P, 0);
    std::vector<SimEvent> sorted = ev;
    std::stable_sort(sorted.begin(), sorted.end(),
                     [](const SimEvent& a, const SimEvent& b) { return a.start < b.start; });
    for (const SimEvent& e : sorted) {
        if (first[e.stage] < 0 || e.start < first[e.stage]) first[e.stage] = e.start;
        lastv[e.stage] = std::max(lastv[e.stage], e.end);
        if (e.kind == ZB_OP_F) peak[e.stage] = std::max(peak[e.stage], ++live[e.stage]);
        else if (e.kind == ZB_OP_W || e.kind == ZB_OP_BW) --live[e.stage];
    }
    double cost = 0.0;
    int pk = 0;
    for (int st = 0; st < P; ++st) {
        cost = std::max(cost, lastv[st] - first[st]);
        pk = std::max(pk, peak[st]);
    }
    res->cost = cost;
    res->ideal = m * (T.f + T.b + T.w);
    res->bubble_rate = cost > 0 ? (cost - res->ideal) / cost : 0.0;
    res->peak_live_microbatches = static_cast<uint32_t>(pk);
    res->peak_live_stage0 = static_cast<uint32_t>(peak[0]);
}

zb_status check_sched_args(int32_t kind, int32_t P, int32_t m, size_t* n_ops, size_t* total) {
    if (!n_ops) return zb::fail(ZB_ERR_INVALID_ARG, "n_ops is NULL");
    if (kind < ZB_SCHED_1F1B || kind > ZB_SCHED_ZBH2) return zb::fail(ZB_ERR_INVALID_ARG, "unknown schedule kind");
    if (P < 1 || m < 1 || P > 65535 || static_cast<long long>(P) * m > (1LL << 20))
        return zb::fail(ZB_ERR_SHAPE, "P and m must be >= 1 (P <= 65535, P*m <= 2^20)");
    const size_t per = kind == ZB_SCHED_1F1B ? 2 : 3;
    *total = static_cast<size_t>(P) * m * per + P;
    return ZB_OK;
}

zb_status run_schedule(int32_t kind, int32_t P, int32_t m, const PassTimes& T, zb_op* out, size_t* n_ops,
                       zb_sim_result* res) {
    size_t total = 0;
    zb_status s = check_sched_args(kind, P, m, n_ops, &total);
    if (s != ZB_OK) return s;
    if (out && *n_ops < total) {
        *n_ops = total;
        return zb::fail(ZB_ERR_INVALID_ARG, "output capacity too small");
    }
    if (!out && !res) {
        *n_ops = total;
        zb::clear_error();
        return ZB_OK;
    }
    std::vector<SimEvent> ev;
    ev.reserve(total);
    if (!simulate(kind, P, m, T, &ev)) return zb::fail(ZB_ERR_SCHEDULE, "schedule simulation deadlocked");
    if (res) fill_result(ev, P, m, T, res);
    if (out) {
        *n_ops = emit_ops(ev, P, out);
    } else {
        *n_ops = total;
    }
    zb::clear_error();
    return ZB_OK;
}

}  // namespace

extern "C" zb_status zb_make_schedule(int32_t kind, int32_t P, int32_t m, zb_op* out, size_t* n_ops) {
    return run_schedule(kind, P, m, PassTimes(), out, n_ops, nullptr);
}

extern "C" zb_status zb_simulate_schedule(int32_t kind, int32_t P, int32_t m, const zb_sim_times* times,
                                          zb_op* out, size_t* n_ops, zb_sim_result* result) {
    if (!times || !result) return zb::fail(ZB_ERR_INVALID_ARG, "times or result is NULL");
    PassTimes T;
    T.f = times->t_f;
    T.b = times->t_b;
    T.w = times->t_w;
    T.comm = times->t_comm;
    if (!(T.f > 0) || !(T.b > 0) || !(T.w > 0) || !(T.comm >= 0) || !std::isfinite(T.f) ||
        !std::isfinite(T.b) || !std::isfinite(T.w) || !std::isfinite(T.comm))
        return zb::fail(ZB_ERR_INVALID_ARG, "pass times must be finite, T_F/T_B/T_W > 0, T_comm >= 0");
    size_t dummy = 0;
    return run_schedule(kind, P, m, T, out, n_ops ? n_ops : &dummy, result);
}

extern "C" zb_status zb_schedule_workspace_size(const zb_pipeline* pl, const zb_op* ops, size_t n_ops,
                                                size_t* bytes, size_t* peak_live_bytes) {
    if (!pl || !bytes) return zb::fail(ZB_ERR_INVALID_ARG, "pipeline or bytes is NULL");
    if (pl->blk.flags & ~ZB_BLOCK_NO_SPLIT_K) return zb::fail(ZB_ERR_INVALID_ARG, "unknown bits in block.flags");
    std::vector<zb_op> vops;
    std::vector<int> dev;
    int L = 0;
    zb_status st = zb::virtualize_ops(*pl, ops, n_ops, &vops, &dev, &L);
    if (st != ZB_OK) return st;
    zb::OpCheck c = zb::validate_ops(vops.data(), n_ops, L, pl->m);
    if (c.st != ZB_OK) return zb::fail(c.st, c.msg);
    if (L > 1 && pl->blk.act == ZB_ACT_NONE && pl->blk.f != pl->blk.h)
        return zb::fail(ZB_ERR_SHAPE, "a multi-stage single-linear pipeline needs f == h");
    zb::ArenaPlan plan;
    zb_pipeline chain = *pl;  // the chain of virtual stages
    chain.P = L;
    chain.chunks = 1;
    // sizing assumes no caller output buffers (the largest arena)
    st = zb::plan_arena(chain, vops.data(), n_ops, false, false, &plan);
    *bytes = plan.workspace_bytes;
    if (st == ZB_OK && pl->executor == ZB_EXEC_PERSISTENT) {
        // the persistent kernel's tables follow the arena (256-byte aligned)
        size_t njobs = 0, ntiles = 0;
        st = zb::replay_count(pl->blk, vops.data(), n_ops, &njobs, &ntiles);
        *bytes = ((plan.workspace_bytes + 255) & ~static_cast<size_t>(255)) + zb::replay_table_bytes(njobs, ntiles);
    }
    if (peak_live_bytes) *peak_live_bytes = plan.peak_live_bytes;
    if (st != ZB_OK) return st;
    zb::clear_error();
    return ZB_OK;
}

extern "C" zb_status zb_auto_schedule(int32_t P, int32_t m, const zb_sim_times* times, double mem_limit,
                                      double mw_ratio, zb_op* out, size_t* n_ops, zb_sim_result* result,
                                      int32_t* hyper) {
    if (!times || !result) return zb::fail(ZB_ERR_INVALID_ARG, "times or result is NULL");
    PassTimes T;
    T.f = times->t_f;
    T.b = times->t_b;
    T.w = times->t_w;
    T.comm = times->t_comm;
    if (!(T.f > 0) || !(T.b > 0) || !(T.w > 0) || !(T.comm >= 0) || !std::isfinite(T.f) ||
        !std::isfinite(T.b) || !std::isfinite(T.w) || !std::isfinite(T.comm))
        return zb::fail(ZB_ERR_INVALID_ARG, "pass times must be finite, T_F/T_B/T_W > 0, T_comm >= 0");
    if (!(mw_ratio > 0.0 && mw_ratio <= 1.0)) return zb::fail(ZB_ERR_INVALID_ARG, "mw_ratio must be in (0, 1]");
    if (!(mem_limit >= 1.0) || !std::isfinite(mem_limit))
        return zb::fail(ZB_ERR_BUDGET, "the memory limit must allow one microbatch (>= 1 M_B)");
    size_t total = 0;
    size_t dummy = 0;
    zb_status st = check_sched_args(ZB_SCHED_ZBH1, P, m, n_ops ? n_ops : &dummy, &total);
    if (st != ZB_OK) return st;
    if (out && *n_ops < total) {
        *n_ops = total;
        return zb::fail(ZB_ERR_INVALID_ARG, "output capacity too small");
    }
    std::vector<SimEvent> best;
    double best_cost = 0.0;
    int best_h = -1;
    for (int h = 0; h < 4; ++h) {  // (h1, h2) = (0,0), (0,1), (1,0), (1,1)
        std::vector<SimEvent> ev;
        ev.reserve(total);
        if (!auto_simulate(P, m, T, mem_limit, mw_ratio, h >> 1, h & 1, &ev)) continue;
        zb_sim_result r;
        fill_result(ev, P, m, T, &r);
        if (best_h < 0 || r.cost < best_cost - 1e-12) {
            best = std::move(ev);
            best_cost = r.cost;
            best_h = h;
        }
    }
    if (best_h < 0) return zb::fail(ZB_ERR_SCHEDULE, "no hyperparameter setting produced a schedule");
    fill_result(best, P, m, T, result);
    if (hyper) {
        hyper[0] = best_h >> 1;
        hyper[1] = best_h & 1;
    }
    if (out) *n_ops = emit_ops(best, P, out);
    else if (n_ops) *n_ops = total;
    zb::clear_error();
    return ZB_OK;
}
