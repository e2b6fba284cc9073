// Host planner of libmk: op DAG -> tile tasks -> events -> static queues.
//
// Event rule: "MPK code walkthrough" (Mirage Persistent Kernel), fine-grained
// pipeline section -- every tensor edge gets event_dim[d] = gcd(producer
// cuts, consumer cuts); a producer feeding several consumers (fork) and a
// consumer fed by several producers (join) have their group sizes lcm'd so
// the edges share one event set.  Task creation walks the op linearisation
// and, per event, creates the consumer tasks inside that event's box, so an
// event's successors are contiguous (building-the-SM-level-DAG section).
// Pairing strategies whole / tile / tile_cover / tile_reduce: "MegaRTP
// megakernel article", section 4 (TaskGraph).  Queues: section 4
// (KernelPlan) and "CMU 15-779 Lecture 7 notes", sections 6.3-6.4.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <functional>
#include <numeric>
#include <queue>
#include <tuple>
#include <string>
#include <vector>

#include "mk_internal.h"
#include "planner.h"

namespace mk {

thread_local std::string g_last_error;

int set_error(int code, const std::string &msg) {
    g_last_error = msg;
    return code;
}

namespace {

constexpr int MAXD = 4;

struct OpDef {
    int opcode = MK_OP_COUNTER;
    int layer = -1;
    int grid[3] = {1, 1, 1};
    std::function<bool(const int *)> exists;      // empty: every grid point exists
    std::function<int64_t(const int *)> cost;     // bytes streamed by one task
};

struct EdgeDef {
    int prod, cons;
    int out_map[3], in_map[3];
};

struct EdgeEv {
    int ev[MAXD], pp[MAXD], cp[MAXD];
};

struct RawTask {
    int op;
    int bid[3];
    int trig = -1, dep = -1;
};

struct RawEvent {
    int ntrig, first, last;
};

void cut_counts(const int grid[3], const int map[3], int out[MAXD]) {
    for (int d = 0; d < MAXD; ++d) out[d] = 1;
    for (int a = 0; a < 3; ++a)
        if (map[a] >= 0) out[map[a]] *= grid[a];
}

int piece(const int bid[3], const int grid[3], const int map[3], int d) {
    int idx = 0;
    for (int a = 0; a < 3; ++a)
        if (map[a] == d) idx = idx * grid[a] + bid[a];
    return idx;
}

int64_t lcm64(int64_t a, int64_t b) { return a / std::gcd(a, b) * b; }

// gcd per edge, then lcm normalisation of fork groups and of join groups; a
// group whose producer (fork) or consumer (join) cuts differ, or whose lcm
// does not divide the cut, falls back to one whole event.
int derive_event_dims(const std::vector<OpDef> &ops, const std::vector<EdgeDef> &edges, std::vector<EdgeEv> &ee) {
    ee.assign(edges.size(), EdgeEv{});
    for (size_t i = 0; i < edges.size(); ++i) {
        cut_counts(ops[edges[i].prod].grid, edges[i].out_map, ee[i].pp);
        cut_counts(ops[edges[i].cons].grid, edges[i].in_map, ee[i].cp);
        for (int d = 0; d < MAXD; ++d) ee[i].ev[d] = std::gcd(ee[i].pp[d], ee[i].cp[d]);
    }
    auto normalise = [&](const std::vector<int> &idx, bool prod_side) {
        auto part = [&](int i) { return prod_side ? ee[i].pp : ee[i].cp; };
        bool same = true;
        for (int i : idx)
            for (int d = 0; d < MAXD; ++d) same &= part(i)[d] == part(idx[0])[d];
        int new_ev[MAXD];
        bool ok = same;
        for (int d = 0; ok && d < MAXD; ++d) {
            int64_t l = 1;
            for (int i : idx) l = lcm64(l, part(i)[d] / ee[i].ev[d]);
            if (part(idx[0])[d] % l != 0) ok = false;
            else new_ev[d] = (int)(part(idx[0])[d] / l);
        }
        for (int i : idx)
            for (int d = 0; d < MAXD; ++d) ee[i].ev[d] = ok ? new_ev[d] : 1;
    };
    std::vector<char> in_fork(edges.size(), 0);
    for (size_t o = 0; o < ops.size(); ++o) {
        std::vector<int> out;
        for (size_t i = 0; i < edges.size(); ++i)
            if (edges[i].prod == (int)o) out.push_back((int)i);
        if (out.size() > 1) {
            normalise(out, true);
            for (int i : out) in_fork[i] = 1;
        }
    }
    for (size_t o = 0; o < ops.size(); ++o) {
        std::vector<int> in;
        for (size_t i = 0; i < edges.size(); ++i)
            if (edges[i].cons == (int)o) in.push_back((int)i);
        if (in.size() > 1) {
            for (int i : in)
                if (in_fork[i]) return set_error(MK_ERR_UNSUPPORTED, "an edge in both a fork and a join");
            normalise(in, false);
        }
    }
    return MK_OK;
}

bool in_box(const int bid[3], const int grid[3], const int map[3], const int part[MAXD], const int ev[MAXD],
            const int coord[MAXD]) {
    for (int d = 0; d < MAXD; ++d) {
        int g = part[d] / ev[d];
        if (piece(bid, grid, map, d) / g != coord[d]) return false;
    }
    return true;
}

void unravel(int k, const int radix[MAXD], int out[MAXD]) {
    for (int d = MAXD - 1; d >= 0; --d) {
        out[d] = k % radix[d];
        k /= radix[d];
    }
}

bool exists(const OpDef &op, const int bid[3]) { return !op.exists || op.exists(bid); }

// MPK task creation (ops must be listed in a topological order).
int build_tasks(const std::vector<OpDef> &ops, const std::vector<EdgeDef> &edges, std::vector<RawTask> &tasks,
                std::vector<RawEvent> &events, int &n_first) {
    std::vector<EdgeEv> ee;
    int rc = derive_event_dims(ops, edges, ee);
    if (rc) return rc;
    std::vector<std::vector<int>> tid(ops.size());
    for (size_t o = 0; o < ops.size(); ++o)
        tid[o].assign((size_t)ops[o].grid[0] * ops[o].grid[1] * ops[o].grid[2], -1);
    auto lin = [&](int o, const int b[3]) { return ((size_t)b[0] * ops[o].grid[1] + b[1]) * ops[o].grid[2] + b[2]; };
    auto add = [&](int o, const int b[3], int dep) {
        RawTask t;
        t.op = o;
        std::memcpy(t.bid, b, sizeof(t.bid));
        t.dep = dep;
        tid[o][lin(o, b)] = (int)tasks.size();
        tasks.push_back(t);
    };
    auto for_bids = [&](int o, const std::function<void(const int *)> &f) {
        int b[3];
        for (b[0] = 0; b[0] < ops[o].grid[0]; ++b[0])
            for (b[1] = 0; b[1] < ops[o].grid[1]; ++b[1])
                for (b[2] = 0; b[2] < ops[o].grid[2]; ++b[2])
                    if (exists(ops[o], b)) f(b);
    };
    std::vector<char> done(ops.size(), 0);
    n_first = 0;
    for (int o = 0; o < (int)ops.size(); ++o) {
        if (done[o]) continue;
        std::vector<int> in;
        for (size_t i = 0; i < edges.size(); ++i)
            if (edges[i].cons == o) in.push_back((int)i);
        if (in.empty()) {
            if (!tasks.empty() && n_first != (int)tasks.size())
                return set_error(MK_ERR_UNSUPPORTED, "ops without inputs must come first");
            for_bids(o, [&](const int *b) { add(o, b, -1); });
            n_first = (int)tasks.size();
            done[o] = 1;
            continue;
        }
        if (in.size() > 1) {  // join consumer
            const EdgeEv &e0 = ee[in[0]];
            int nev = 1;
            for (int d = 0; d < MAXD; ++d) nev *= e0.ev[d];
            for (int k = 0; k < nev; ++k) {
                int c[MAXD];
                unravel(k, e0.ev, c);
                int ev_id = (int)events.size();
                RawEvent ev{0, (int)tasks.size(), 0};
                for_bids(o, [&](const int *b) {
                    if (in_box(b, ops[o].grid, edges[in[0]].in_map, e0.cp, e0.ev, c)) add(o, b, ev_id);
                });
                ev.last = (int)tasks.size();
                for (int i : in) {
                    int p = edges[i].prod;
                    for_bids(p, [&](const int *b) {
                        if (in_box(b, ops[p].grid, edges[i].out_map, ee[i].pp, e0.ev, c)) {
                            tasks[tid[p][lin(p, b)]].trig = ev_id;
                            ev.ntrig++;
                        }
                    });
                }
                events.push_back(ev);
            }
            done[o] = 1;
            continue;
        }
        const EdgeDef &e0 = edges[in[0]];
        int p = e0.prod;
        std::vector<int> bundle;
        for (size_t i = 0; i < edges.size(); ++i)
            if (edges[i].prod == p) bundle.push_back((int)i);
        for (int i : bundle) {
            int n = 0;
            for (auto &e : edges) n += e.cons == edges[i].cons;
            if (n != 1) return set_error(MK_ERR_UNSUPPORTED, "fork consumer with several in-edges");
        }
        std::sort(bundle.begin(), bundle.end(), [&](int a, int b) { return edges[a].cons < edges[b].cons; });
        const EdgeEv &eb = ee[bundle[0]];
        int nev = 1;
        for (int d = 0; d < MAXD; ++d) nev *= eb.ev[d];
        for (int k = 0; k < nev; ++k) {
            int c[MAXD];
            unravel(k, eb.ev, c);
            int ev_id = (int)events.size();
            RawEvent ev{0, (int)tasks.size(), 0};
            for (int i : bundle) {
                int co = edges[i].cons;
                for_bids(co, [&](const int *b) {
                    if (in_box(b, ops[co].grid, edges[i].in_map, ee[i].cp, eb.ev, c)) add(co, b, ev_id);
                });
            }
            ev.last = (int)tasks.size();
            for_bids(p, [&](const int *b) {
                if (in_box(b, ops[p].grid, e0.out_map, eb.pp, eb.ev, c)) {
                    tasks[tid[p][lin(p, b)]].trig = ev_id;
                    ev.ntrig++;
                }
            });
            events.push_back(ev);
        }
        for (int i : bundle) done[edges[i].cons] = 1;
    }
    return MK_OK;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// in-order queues, counters with epochs, `steps` back-to-back passes
bool simulate(const std::vector<std::vector<int>> &queues, const std::vector<TaskRec> &tasks, int n_events,
              int steps, std::string &why) {
    std::vector<int64_t> cnt(n_events, 0);
    for (int s = 0; s < steps; ++s) {
        std::vector<size_t> pos(queues.size(), 0);
        size_t remaining = 0;
        for (auto &q : queues) remaining += q.size();
        bool progress = true;
        while (remaining && progress) {
            progress = false;
            for (size_t w = 0; w < queues.size(); ++w) {
                while (pos[w] < queues[w].size()) {
                    const TaskRec &t = tasks[queues[w][pos[w]]];
                    bool ready = true;
                    for (int i = 0; i < t.nw && ready; ++i)
                        ready = cnt[t.w_ev[i]] >= (int64_t)t.w_thr[i] * (s + 1 + t.w_off[i]);
                    if (!ready) break;
                    for (int i = 0; i < t.ns; ++i) cnt[t.s_ev[i]] += t.s_inc[i];
                    pos[w]++;
                    remaining--;
                    progress = true;
                }
            }
        }
        if (remaining) {
            for (size_t w = 0; w < queues.size(); ++w)
                if (pos[w] < queues[w].size()) {
                    char buf[160];
                    std::snprintf(buf, sizeof buf, "queue simulation stuck at step %d: worker %zu task %d", s, w,
                                  queues[w][pos[w]]);
                    why = buf;
                    break;
                }
            return false;
        }
    }
    return true;
}

// Deal tasks in order to the least-loaded worker (ties: lowest index).
std::vector<std::vector<int>> greedy(const std::vector<int> &order, const std::vector<TaskRec> &tasks, int workers) {
    using Item = std::pair<int64_t, int>;
    std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
    for (int w = 0; w < workers; ++w) heap.push({0, w});
    std::vector<std::vector<int>> q(workers);
    std::vector<int64_t> pinned_load(workers, 0);
    for (int t : order) {
        if (tasks[t].opcode == MK_OP_ATTN_POOL) {  // one attention pool per worker and layer: its own worker
            const int w = tasks[t].bid[0] % workers;
            q[w].push_back(t);
            pinned_load[w] += tasks[t].cost;
            continue;
        }
        Item it = heap.top();
        heap.pop();
        it.first += pinned_load[it.second];
        pinned_load[it.second] = 0;
        q[it.second].push_back(t);
        it.first += tasks[t].cost;
        heap.push(it);
    }
    return q;
}

// List scheduling against a time model of one step.  A task is ready HOP
// after every counter it waits on (this epoch) has met its threshold, and it
// holds a worker for a fixed cost plus its bytes at the worker's share of HBM
// bandwidth.  Among the tasks whose producers are all placed, the one ready
// first (ties: earlier in `order`) goes next, to the worker on which it
// finishes first (ties: lowest index).  The placement order is thus a
// topological order and every queue a subsequence of it; it lets a consumer
// that becomes ready early (an MLP-down K chunk) run between the producer
// tiles still to come instead of behind all of them.  The model balances each
// dependency phase on its own, where the byte greedy balances whole-step
// totals.
std::vector<std::vector<int>> timed(const std::vector<int> &order, const std::vector<TaskRec> &tasks, int workers,
                                    int n_events) {
    constexpr double HOP_US = 3.0, TILE_US = 1.0, ATTN_US = 4.0, HBM_BYTES_PER_US = 6.8e6;
    const double bw = HBM_BYTES_PER_US / std::max(1, workers);
    const int n = (int)tasks.size();
    std::vector<std::vector<std::pair<double, int>>> sig(n_events);  // (finish, increment) of each placed signal
    std::vector<std::vector<int>> prod(n_events), cons(n_events);
    std::vector<int> pending(n, 0), rank(n, 0);
    for (int i = 0; i < (int)order.size(); ++i) rank[order[i]] = i;
    for (int id : order) {
        const TaskRec &t = tasks[id];
        for (int i = 0; i < t.ns; ++i) prod[t.s_ev[i]].push_back(id);
    }
    for (int id : order) {
        const TaskRec &t = tasks[id];
        for (int i = 0; i < t.nw; ++i)
            if (t.w_off[i] >= 0 && t.w_thr[i] > 0) {
                cons[t.w_ev[i]].push_back(id);
                pending[id] += (int)prod[t.w_ev[i]].size();
            }
    }
    auto time_met = [&](int e, int64_t thr) {
        auto v = sig[e];
        std::sort(v.begin(), v.end());
        int64_t acc = 0;
        double t = 0.0;
        for (auto &f : v) {
            acc += f.second;
            t = f.first;
            if (acc >= thr) break;
        }
        return t;
    };
    auto ready_time = [&](int id) {
        const TaskRec &t = tasks[id];
        double ready = 0.0;
        for (int i = 0; i < t.nw; ++i)
            if (t.w_off[i] >= 0 && t.w_thr[i] > 0) ready = std::max(ready, time_met(t.w_ev[i], t.w_thr[i]) + HOP_US);
        return ready;
    };
    using Cand = std::tuple<double, int, int>;  // ready time, rank, task
    std::priority_queue<Cand, std::vector<Cand>, std::greater<Cand>> heap;
    for (int id : order)
        if (pending[id] == 0) heap.push({ready_time(id), rank[id], id});
    std::vector<double> free_at(workers, 0.0);
    std::vector<std::vector<int>> q(workers);
    int placed = 0;
    while (!heap.empty()) {
        const auto [ready, rk, id] = heap.top();
        (void)rk;
        heap.pop();
        const TaskRec &t = tasks[id];
        const bool attn = t.opcode == MK_OP_ATTN || t.opcode == MK_OP_ATTN_POOL;
        const double dur = (attn ? ATTN_US : TILE_US) + (double)t.cost / bw;
        int best = 0;
        double best_end = 0.0;
        for (int w = 0; w < workers; ++w) {
            const double end = std::max(free_at[w], ready) + dur;
            if (w == 0 || end < best_end) {
                best = w;
                best_end = end;
            }
        }
        if (t.opcode == MK_OP_ATTN_POOL) {  // one attention pool per worker and layer: its own worker
            best = t.bid[0] % workers;
            best_end = std::max(free_at[best], ready) + dur;
        }
        free_at[best] = best_end;
        q[best].push_back(id);
        ++placed;
        for (int i = 0; i < t.ns; ++i) {
            const int e = t.s_ev[i];
            sig[e].push_back({best_end, t.s_inc[i]});
            for (int c : cons[e])
                if (--pending[c] == 0) heap.push({ready_time(c), rank[c], c});
        }
    }
    if (placed != (int)order.size()) return greedy(order, tasks, workers);  // not a DAG of this epoch: keep order
    return q;
}

}  // namespace

// ---- encode and finish a plan --------------------------------------------

void encode_task(const TaskRec &t, int task_id, int32_t *w) {
    std::memset(w, 0, W_WORDS * sizeof(int32_t));
    w[W_OPC] = t.opcode;
    w[W_ROW] = t.op_row;
    w[W_CNT] = t.nw | (t.ns << 8);
    w[W_TASK] = task_id;
    for (int i = 0; i < t.nw; ++i) {
        w[W_WAIT + 2 * i] = (int32_t)((uint32_t)t.w_ev[i] | (t.w_off[i] < 0 ? WAIT_PREV_EPOCH : 0u));
        w[W_WAIT + 2 * i + 1] = t.w_thr[i];
    }
    for (int i = 0; i < t.ns; ++i) {
        w[W_SIG + 2 * i] = t.s_ev[i];
        w[W_SIG + 2 * i + 1] = t.s_inc[i];
    }
    for (int i = 0; i < W_WORDS - W_P; ++i) w[W_P + i] = t.payload[i];
}

// Build the launch segments (one for the megakernel, one per op otherwise),
// simulate them and encode the instruction words.
int finish_queues(Plan &p, bool round_robin, bool timed_model) {
    std::vector<Segment> segs;
    std::vector<std::vector<int>> all_q;
    int n = (int)p.tasks.size();
    auto make = [&](const std::vector<int> &order, int workers) {
        std::vector<std::vector<int>> q;
        if (round_robin) {
            q.assign(workers, {});
            for (size_t i = 0; i < order.size(); ++i) q[i % workers].push_back(order[i]);
        } else if (timed_model) {
            q = timed(order, p.tasks, workers, (int)p.thresholds.size());
        } else {
            q = greedy(order, p.tasks, workers);
        }
        Segment s;
        s.workers = workers;
        s.lmax = 0;
        for (auto &r : q) s.lmax = std::max<int>(s.lmax, (int)r.size());
        s.word_offset = (int64_t)p.words.size();
        s.slot_offset = (int64_t)p.slot_task.size();
        p.words.resize(p.words.size() + (size_t)workers * s.lmax * W_WORDS, 0);
        p.slot_task.resize(p.slot_task.size() + (size_t)workers * s.lmax, -1);
        for (int w = 0; w < workers; ++w)
            for (int i = 0; i < s.lmax; ++i) {
                size_t slot = (size_t)w * s.lmax + i;
                if (i < (int)q[w].size()) {
                    int t = q[w][i];
                    encode_task(p.tasks[t], t, &p.words[s.word_offset + slot * W_WORDS]);
                    p.slot_task[s.slot_offset + slot] = t;
                }  // else NoOp: all-zero words
            }
        segs.push_back(s);
        return q;
    };
    p.words.clear();
    p.slot_task.clear();
    if (p.mode == MK_MODE_MEGAKERNEL) {
        std::vector<int> order(n);
        std::iota(order.begin(), order.end(), 0);
        auto q = make(order, p.num_workers);
        std::string why;
        if (!simulate(q, p.tasks, (int)p.thresholds.size(), 2, why)) return set_error(MK_ERR_DEADLOCK, why);
    } else {
        // per-op launches, ops in plan order; each launch only depends on earlier ones
        std::vector<std::vector<int>> by_op(p.num_ops);
        for (int t = 0; t < n; ++t) by_op[p.tasks[t].op_row].push_back(t);
        std::vector<int64_t> cnt(p.thresholds.size(), 0);
        for (int o = 0; o < p.num_ops; ++o) {
            if (by_op[o].empty()) continue;
            int workers = std::min<int>(p.num_workers, (int)by_op[o].size());
            auto q = make(by_op[o], workers);
            for (int t : by_op[o])
                for (int i = 0; i < p.tasks[t].nw; ++i)
                    if (p.tasks[t].w_off[i] == 0 && cnt[p.tasks[t].w_ev[i]] < p.tasks[t].w_thr[i])
                        return set_error(MK_ERR_DEADLOCK, "per-op launch waits on a later launch");
            for (int t : by_op[o])
                for (int i = 0; i < p.tasks[t].ns; ++i) cnt[p.tasks[t].s_ev[i]] += p.tasks[t].s_inc[i];
        }
    }
    p.segments = segs;
    p.lmax = segs.empty() ? 0 : segs[0].lmax;
    return MK_OK;
}

// ---- explicit graphs ----------------------------------------------------

int plan_graph(const mk_graph_desc *g, const mk_target_desc *tgt, int num_workers, Plan &p) {
    if (!g || g->num_ops <= 0 || !g->ops) return set_error(MK_ERR_INVALID, "empty graph");
    p = Plan{};
    p.kind = PLAN_GRAPH;
    p.mode = tgt && tgt->mode == MK_MODE_PER_OP ? MK_MODE_PER_OP : MK_MODE_MEGAKERNEL;
    p.num_workers = num_workers;
    p.num_ops = g->num_ops;
    for (int o = 0; o < g->num_ops; ++o)
        for (int a = 0; a < 3; ++a)
            if (g->ops[o].grid[a] <= 0) return set_error(MK_ERR_INVALID, "grid extents must be positive");
    if (g->num_pubs > 0) {
        // MegaRTP publications: ops in the given order, tasks in index order
        std::vector<int> base(g->num_ops + 1, 0);
        for (int o = 0; o < g->num_ops; ++o)
            base[o + 1] = base[o] + g->ops[o].grid[0] * g->ops[o].grid[1] * g->ops[o].grid[2];
        p.tasks.assign(base[g->num_ops], TaskRec{});
        for (int o = 0; o < g->num_ops; ++o)
            for (int i = base[o]; i < base[o + 1]; ++i) {
                TaskRec &t = p.tasks[i];
                t.opcode = MK_OP_COUNTER;
                t.op_row = o;
                int li = i - base[o];
                t.bid[0] = li;
                t.cost = g->ops[o].cost;
            }
        for (int k = 0; k < g->num_pubs; ++k) {
            const mk_graph_pub &pb = g->pubs[k];
            if (pb.prod < 0 || pb.prod >= g->num_ops || pb.num_pub <= 0 || pb.num_cons < 0 || pb.num_cons > 4)
                return set_error(MK_ERR_INVALID, "bad publication");
            int n_ev, thr;
            if (pb.strategy == MK_PAIR_WHOLE) { n_ev = 1; thr = pb.num_pub; }
            else if (pb.strategy == MK_PAIR_TILE) { n_ev = pb.num_pub; thr = 1; }
            else if (pb.strategy == MK_PAIR_TILE_COVER || pb.strategy == MK_PAIR_TILE_REDUCE) {
                if (pb.k <= 0 || pb.num_pub % pb.k) return set_error(MK_ERR_INVALID, "k must divide num_pub");
                n_ev = pb.num_pub / pb.k;
                thr = pb.k;
            } else return set_error(MK_ERR_INVALID, "unknown strategy");
            int first = (int)p.thresholds.size();
            for (int e = 0; e < n_ev; ++e) p.thresholds.push_back(thr);
            int per = pb.num_pub / n_ev;
            for (int j = 0; j < pb.num_pub; ++j) {
                TaskRec &t = p.tasks[base[pb.prod] + pb.first_pub + j];
                if (t.ns >= MAX_SIGS) return set_error(MK_ERR_UNSUPPORTED, "more than 2 signals on a task");
                t.s_ev[t.ns] = first + j / per;
                t.s_inc[t.ns++] = 1;
            }
            for (int c = 0; c < pb.num_cons; ++c) {
                int co = pb.cons[c];
                int nc = base[co + 1] - base[co];
                if (nc % n_ev) return set_error(MK_ERR_INVALID, "consumer tasks not divisible by events");
                for (int i = 0; i < nc; ++i) {
                    TaskRec &t = p.tasks[base[co] + i];
                    if (t.nw >= MAX_WAITS) return set_error(MK_ERR_UNSUPPORTED, "more than 3 waits on a task");
                    int ev = first + i / (nc / n_ev);
                    t.w_ev[t.nw] = ev;
                    t.w_thr[t.nw] = thr;
                    t.w_off[t.nw++] = 0;
                }
            }
        }
    } else {
        std::vector<OpDef> ops(g->num_ops);
        for (int o = 0; o < g->num_ops; ++o) {
            std::memcpy(ops[o].grid, g->ops[o].grid, sizeof(ops[o].grid));
            int c = g->ops[o].cost;
            ops[o].cost = [c](const int *) { return (int64_t)c; };
        }
        std::vector<EdgeDef> edges(g->num_edges);
        for (int i = 0; i < g->num_edges; ++i) {
            const mk_graph_edge &e = g->edges[i];
            if (e.prod < 0 || e.cons < 0 || e.prod >= g->num_ops || e.cons >= g->num_ops || e.prod >= e.cons)
                return set_error(MK_ERR_INVALID, "edges must go from an earlier op to a later one");
            edges[i] = EdgeDef{e.prod, e.cons, {e.out_map[0], e.out_map[1], e.out_map[2]},
                               {e.in_map[0], e.in_map[1], e.in_map[2]}};
            for (int a = 0; a < 3; ++a)
                if (e.out_map[a] >= MAXD || e.in_map[a] >= MAXD) return set_error(MK_ERR_INVALID, "map beyond 4 dims");
        }
        std::vector<RawTask> raw;
        std::vector<RawEvent> evs;
        int n_first;
        int rc = build_tasks(ops, edges, raw, evs, n_first);
        if (rc) return rc;
        for (auto &e : evs) p.thresholds.push_back(e.ntrig);
        p.tasks.resize(raw.size());
        for (size_t i = 0; i < raw.size(); ++i) {
            TaskRec &t = p.tasks[i];
            t.opcode = MK_OP_COUNTER;
            t.op_row = raw[i].op;
            std::memcpy(t.bid, raw[i].bid, sizeof(t.bid));
            t.cost = g->ops[raw[i].op].cost;
            if (raw[i].dep >= 0) {
                t.w_ev[0] = raw[i].dep;
                t.w_thr[0] = evs[raw[i].dep].ntrig;
                t.nw = 1;
            }
            if (raw[i].trig >= 0) {
                t.s_ev[0] = raw[i].trig;
                t.s_inc[0] = 1;
                t.ns = 1;
            }
        }
        for (auto &e : evs) p.events.push_back({e.ntrig, e.first, e.last});
    }
    p.op_kind.assign(g->num_ops, MK_OP_COUNTER);
    p.op_layer.assign(g->num_ops, -1);
    return finish_queues(p, g->round_robin != 0, false);
}

// ---- Llama-style decode step on tensor-core tiles (batch 8..16) -------------
// Per layer: NORM (attention RMSNorm, one task per sequence: bf16 high/low
// rows of x^ for the tiles; zeroes the qkv rows the K-split QKV tiles add
// into) -> QKV tiles -> attention -> O tiles (K split, added into the
// residual) -> NORM (MLP RMSNorm) -> MLP-up tiles (64 gate + 64 up rows,
// SiLU(g) u as bf16 high/low) -> MLP-down tiles per K chunk (added into the
// residual); then the final NORM and the LM-head tiles.  Every GEMV tile is
// 128 weight rows over a K range in stages of 128 columns.
// attn_pool plans: the payload of every pool instruction (its layer's task
// rows) and the attention task table -- per layer, the tasks (kv head g,
// sequence b, split) as ATTN instructions, longest first (cached rows at the
// last step of the plan; ties in (g, b, split) order).  A table instruction
// has no waits or signals: its pool slot waits for the layer's QKV and
// signals the layer's attention event; W_SIG names that event and P_ATHR its
// per-step threshold for the loader's wait on K/V rows appended by an earlier
// step of the same launch.
static void build_attn_pool(Plan &p, int Hkv, int kn_T, const std::vector<int> &nsplit, int max_steps) {
    const int L = p.model.layers, B = p.B;
    int per_layer = 0;
    for (int b = 0; b < B; ++b) per_layer += nsplit[b];
    per_layer *= Hkv;
    p.attn_table.assign((size_t)L * per_layer * W_WORDS, 0);
    std::vector<int> pool_row(L, -1), pool_ev(L, -1), pool_thr(L, 0);
    for (TaskRec &t : p.tasks) {
        if (t.opcode != MK_OP_ATTN_POOL) continue;
        t.payload[P_LAYER - W_P] = t.layer;
        t.payload[P_PT - W_P] = per_layer;
        t.payload[P_TBASE - W_P] = t.layer * per_layer;
        pool_row[t.layer] = t.op_row;
        pool_ev[t.layer] = t.ns > 0 ? t.s_ev[0] : -1;
        pool_thr[t.layer] = t.ns > 0 ? p.thresholds[t.s_ev[0]] : 0;
        t.payload[P_ATHR - W_P] = pool_thr[t.layer];
    }
    for (int l = 0; l < L; ++l) {
        struct Item { int64_t cost; int g, b, s; };
        std::vector<Item> items;
        for (int g = 0; g < Hkv; ++g)
            for (int b = 0; b < B; ++b)
                for (int sp = 0; sp < nsplit[b]; ++sp) {
                    const int last = p.seq0[b] + max_steps - 1;
                    items.push_back({std::max(0, std::min(kn_T, last - sp * kn_T)), g, b, sp});
                }
        std::stable_sort(items.begin(), items.end(), [](const Item &x, const Item &y) { return x.cost > y.cost; });
        for (int idx = 0; idx < (int)items.size(); ++idx) {
            const Item &it = items[idx];
            TaskRec a;
            a.opcode = MK_OP_ATTN;
            a.op_row = pool_row[l];
            a.layer = l;
            int32_t *pl = a.payload;
            pl[P_G - W_P] = it.g; pl[P_B - W_P] = it.b; pl[P_SPLIT - W_P] = it.s;
            pl[P_T0 - W_P] = it.s * kn_T; pl[P_T - W_P] = kn_T; pl[P_NSPLIT - W_P] = nsplit[it.b];
            pl[P_LAYER - W_P] = l; pl[P_ATHR - W_P] = pool_thr[l];
            const int row = l * per_layer + idx;
            int32_t *w = &p.attn_table[(size_t)row * W_WORDS];
            encode_task(a, row, w);
            w[W_SIG] = pool_ev[l];  // (no signal is counted: W_CNT says none)
        }
    }
}

static int plan_llama_tc(const mk_model_desc *m, const mk_step_desc *s, const mk_target_desc *tgt, int num_workers,
                         int smem_per_cta, Plan &p) {
    const int L = m->layers, H = m->hidden, Hq = m->q_heads, Hkv = m->kv_heads, D = m->head_dim, F = m->ffn,
              V = m->vocab, B = s->batch, G = Hq / Hkv;
    if (tgt->page_bytes != 0 && tgt->page_bytes != TC_STAGE_BYTES)
        return set_error(MK_ERR_UNSUPPORTED, "tensor-core plans use 32 KB pages");
    if (tgt->schedule < MK_SCHED_DEFAULT || tgt->schedule > MK_SCHED_TIMED)
        return set_error(MK_ERR_INVALID, "schedule must be one of MK_SCHED_*");
    p.schedule = tgt->schedule == MK_SCHED_BYTES ? MK_SCHED_BYTES : MK_SCHED_TIMED;
    p.tc = true;
    p.np = B <= 8 ? 8 : 16;
    p.page_bytes = TC_STAGE_BYTES;
    const int rows_group = (G + 2) * D;
    // K splits: the largest power of two up to 8 that keeps the op's tasks
    // within the workers (a split K range stays a whole number of stages)
    auto ksplit = [&](int tiles, int K, int knob) {
        if (knob > 0) return knob;
        int k = 1;
        while (k < 8 && (int64_t)tiles * k * 2 <= num_workers && (K / (k * 2)) % TC_KS == 0 && K % (k * 2) == 0) k *= 2;
        return k;
    };
    const int ks_qkv = ksplit(Hkv * rows_group / TC_M, H, 0), ks_o = ksplit(H / TC_M, Hq * D, 0);
    if (H % (ks_qkv * TC_KS) || (Hq * D) % (ks_o * TC_KS)) return set_error(MK_ERR_UNSUPPORTED, "bad K split");
    // MLP-down K chunk: the largest of 1024 .. 256 dividing ffn that still
    // gives at least half as many tasks as workers (a 2048-wide chunk makes
    // MLP-down wait on larger pieces of MLP-up: slower at batch 16)
    int kc = tgt->kchunk_down;
    if (kc <= 0) {
        kc = 0;
        for (int c : {1024, 512, 256})
            if (F % c == 0) {
                if (!kc) kc = c;
                if ((int64_t)(H / TC_M) * (F / c) * 2 >= num_workers) { kc = c; break; }
                kc = c;
            }
    }
    if (kc <= 0 || F % kc || kc % TC_KS) return set_error(MK_ERR_UNSUPPORTED, "kchunk_down must divide ffn in 128s");
    p.ksplit_qkv = ks_qkv;
    p.ksplit_o = ks_o;
    p.rows_qkv = p.rows_o = p.rows_down = p.rows_lm = TC_M;
    p.rows_up = TC_SEG;
    p.kchunk_down = kc;
    int kn_T = tgt->attn_split > 0 ? tgt->attn_split : std::max(16, std::min(256, 16384 / (2 * D)));
    if (tgt->attn_split <= 0) {
        auto attn_tasks = [&](int T) {
            int64_t n = 0;
            for (int b = 0; b < B; ++b) n += ceil_div(s->seq_len0[b] + s->max_steps, T);
            return n * Hkv;
        };
        while (2 * kn_T <= 512 && attn_tasks(kn_T) > (int64_t)num_workers) kn_T *= 2;
    }
    if (kn_T > 512 || kn_T < 1) return set_error(MK_ERR_UNSUPPORTED, "attn_split must be 1..512");
    p.attn_split = kn_T;
    // shared memory: activation ring | two attention slots | pages | op scratch | barriers | flags,
    // the ring and the pages 1024-byte aligned (swizzled TMA boxes)
    p.abuf_count = TC_XSLOTS;
    p.abuf_bytes = tc_xstage_bytes(p.np);
    const int attn_slot = (G * (D + 16) + 2 * D) * 4;
    p.act_bytes = round_up(attn_slot, 512);
    p.red_bytes = 128;
    p.aux_bytes = round_up(attn_aux_bytes(G, kn_T, D), 128) + 2 * TC_SEG * TC_MAXB * 4 + NRED * p.red_bytes;
    const int fixed = p.abuf_count * p.abuf_bytes + 2 * p.act_bytes + p.aux_bytes + MBAR_BYTES + CTRL_BYTES;
    p.num_pages = std::min(8, (smem_per_cta - fixed) / p.page_bytes);
    // an attention task holds its K pages, releases them, then waits for its V pages
    const int attn_need = attn_pages(kn_T, D, p.page_bytes);
    if (attn_need > 4 || p.num_pages < std::max(3, attn_need))
        return set_error(MK_ERR_UNSUPPORTED, "shared memory too small for the page pool");
    p.smem_bytes = fixed + p.num_pages * p.page_bytes;

    std::vector<int> nsplit(B);
    for (int b = 0; b < B; ++b) nsplit[b] = ceil_div(p.seq0[b] + s->max_steps, kn_T);
    p.nsplit_max = *std::max_element(nsplit.begin(), nsplit.end());
    const bool pool = tgt->attn_pool != 0;  // device-side attention dispatch
    if (pool && B < 2) return set_error(MK_ERR_UNSUPPORTED, "attention pools are for batches of 2 or more");
    int64_t attn_layer_bytes = 0;           // (the pools' share of it is their scheduling cost)
    for (int b = 0; b < B; ++b)
        for (int sp = 0; sp < nsplit[b]; ++sp)
            attn_layer_bytes += (int64_t)2 * D * 2 * Hkv * std::max(0, std::min(kn_T, p.seq0[b] + s->max_steps - 1 - sp * kn_T));
    std::vector<int> seq0 = p.seq0;
    const int max_steps = s->max_steps;
    std::vector<OpDef> ops;
    std::vector<EdgeDef> edges;
    std::vector<int> aux;
    auto add_op = [&](int opcode, int layer, int gx, int gy, int gz, int a = 0) {
        OpDef o;
        o.opcode = opcode;
        o.layer = layer;
        o.grid[0] = gx; o.grid[1] = gy; o.grid[2] = gz;
        ops.push_back(o);
        aux.push_back(a);
        return (int)ops.size() - 1;
    };
    const int64_t norm_cost = (int64_t)H * 2;
    int emb = add_op(MK_OP_EMBED, -1, 1, 1, 1);
    ops[emb].cost = [=](const int *) { return (int64_t)B * H * 2; };
    int prev = emb;
    const int none[3] = {-1, -1, -1};
    auto whole = [&](int a, int b) { edges.push_back({a, b, {none[0], none[1], none[2]}, {-1, -1, -1}}); };
    for (int l = 0; l < L; ++l) {
        int na = add_op(MK_OP_NORM, l, B, 1, 1, 0);
        ops[na].cost = [=](const int *) { return norm_cost; };
        int q = add_op(MK_OP_QKV, l, Hkv, rows_group / TC_M, ks_qkv);
        ops[q].cost = [=](const int *) { return (int64_t)TC_M * (H / ks_qkv) * 2; };
        int a;
        if (pool) {  // one pool per worker; its cost: the layer's attention bytes over the workers
            a = add_op(MK_OP_ATTN_POOL, l, num_workers, 1, 1);
            ops[a].cost = [=](const int *) { return attn_layer_bytes / num_workers; };
        } else {
            a = add_op(MK_OP_ATTN, l, Hkv, B, p.nsplit_max);
            ops[a].exists = [nsplit](const int *b) { return b[2] < nsplit[b[1]]; };
            ops[a].cost = [=](const int *b) {
                int last = seq0[b[1]] + max_steps - 1;
                int rows = std::max(0, std::min(kn_T, last - b[2] * kn_T));
                return (int64_t)2 * D * 2 * rows;
            };
        }
        int o = add_op(MK_OP_O, l, H / TC_M, ks_o, 1);
        ops[o].cost = [=](const int *) { return (int64_t)TC_M * (Hq * D / ks_o) * 2; };
        int nm = add_op(MK_OP_NORM, l, B, 1, 1, 1);
        ops[nm].cost = [=](const int *) { return norm_cost; };
        int u = add_op(MK_OP_UP, l, F / TC_SEG, 1, 1);
        ops[u].cost = [=](const int *) { return (int64_t)TC_M * H * 2; };
        int d = add_op(MK_OP_DOWN, l, H / TC_M, F / kc, 1);
        ops[d].cost = [=](const int *) { return (int64_t)TC_M * kc * 2; };
        whole(prev, na);                                   // residual h read whole
        whole(na, q);                                      // x^ read whole
        if (pool) {
            whole(q, a);                                   // a pool may claim any group's task
            whole(a, o);
        } else {
            edges.push_back({q, a, {1, 2, -1}, {1, 0, -1}});   // qkv [B, Hkv, rows]: group & row cuts (K split reduces)
            edges.push_back({a, o, {1, 0, -1}, {-1, -1, -1}}); // attention output read whole; the split axis reduces
        }
        whole(o, nm);                                      // h after O read whole
        whole(nm, u);                                      // x^ read whole
        edges.push_back({u, d, {1, -1, -1}, {-1, 1, -1}}); // act [B, F]: tiles vs K chunks
        prev = d;
    }
    int nf = add_op(MK_OP_NORM, -1, B, 1, 1, 2);
    ops[nf].cost = [=](const int *) { return norm_cost; };
    int lm = add_op(MK_OP_LM, -1, ceil_div(V, TC_M), 1, 1);
    ops[lm].cost = [=](const int *b) { return (int64_t)std::min(TC_M, V - b[0] * TC_M) * H * 2; };
    whole(prev, nf);
    whole(nf, lm);

    std::vector<RawTask> raw;
    std::vector<RawEvent> evs;
    int n_first;
    int rc = build_tasks(ops, edges, raw, evs, n_first);
    if (rc) return rc;
    std::vector<int64_t> cost(raw.size());
    for (size_t i = 0; i < raw.size(); ++i) cost[i] = ops[raw[i].op].cost(raw[i].bid);
    std::vector<std::pair<int, int>> ranges{{0, n_first}};
    for (auto &e : evs) ranges.push_back({e.first, e.last});
    std::sort(ranges.begin(), ranges.end());
    std::vector<int> order;
    for (auto &r : ranges) {
        std::vector<int> ids(r.second - r.first);
        std::iota(ids.begin(), ids.end(), r.first);
        std::stable_sort(ids.begin(), ids.end(), [&](int x, int y) { return cost[x] > cost[y]; });
        order.insert(order.end(), ids.begin(), ids.end());
    }
    if ((int)order.size() != (int)raw.size()) return set_error(MK_ERR_INVALID, "task ranges do not cover the graph");
    const int step_done = (int)evs.size();
    for (auto &e : evs) p.thresholds.push_back(e.ntrig);
    p.thresholds.push_back(0);
    for (auto &e : evs) p.events.push_back({e.ntrig, e.first, e.last});
    p.events.push_back({0, 0, n_first});
    p.num_ops = (int)ops.size();
    for (size_t o = 0; o < ops.size(); ++o) {
        p.op_kind.push_back(ops[o].opcode);
        p.op_layer.push_back(ops[o].layer);
        p.op_aux.push_back(aux[o]);
    }
    // QKV rows of a head group: q heads, then k, then v (kv-group-major); a
    // 64-row segment lies in one of them
    auto qkv_row = [&](int g, int lr, int &mat) {
        if (lr < G * D) { mat = 0; return g * G * D + lr; }
        if (lr < (G + 1) * D) { mat = 1; return g * D + lr - G * D; }
        mat = 2;
        return g * D + lr - (G + 1) * D;
    };
    p.tasks.reserve(order.size());
    for (int old : order) {
        const RawTask &r = raw[old];
        const OpDef &op = ops[r.op];
        TaskRec t;
        t.opcode = op.opcode;
        t.op_row = r.op;
        t.layer = op.layer;
        std::memcpy(t.bid, r.bid, sizeof(t.bid));
        t.cost = cost[old];
        if (r.dep >= 0) {
            t.w_ev[t.nw] = r.dep; t.w_thr[t.nw] = evs[r.dep].ntrig; t.w_off[t.nw++] = 0;
        }
        if (r.trig >= 0) { t.s_ev[t.ns] = r.trig; t.s_inc[t.ns++] = 1; }
        if (op.opcode == MK_OP_LM) {
            t.s_ev[t.ns] = step_done; t.s_inc[t.ns++] = 1;
            p.thresholds[step_done]++;
        }
        int32_t *pl = t.payload;
        auto tile = [&](int row0, int mat0, int row1, int mat1, int nrows, int k0, int kcn, int ktot, int out0) {
            pl[P_ROW0 - W_P] = row0; pl[P_MAT - W_P] = mat0;
            pl[P_S1_ROW0 - W_P] = row1; pl[P_S1_MAT - W_P] = mat1;
            pl[P_NROWS - W_P] = nrows; pl[P_K0 - W_P] = k0; pl[P_KC - W_P] = kcn; pl[P_KTOT - W_P] = ktot;
            pl[P_OUT0 - W_P] = out0; pl[P_NPG - W_P] = kcn / TC_KS; pl[P_RPP - W_P] = TC_M;
        };
        switch (op.opcode) {
        case MK_OP_NORM: {
            const int which = aux[r.op];
            pl[P_NB - W_P] = r.bid[0];
            pl[P_NZERO - W_P] = which == 0 && ks_qkv > 1 ? 1 : 0;
            int snap = 0;
            if (p.capture && which == 0 && op.layer > 0) snap = op.layer;  // residual after layer l - 1
            if (p.capture && which == 2) snap = L;
            pl[P_NSNAP - W_P] = snap;
            break;
        }
        case MK_OP_QKV: {
            const int g = r.bid[0], lr = r.bid[1] * TC_M, kq = H / ks_qkv;
            int m0, m1;
            const int r0 = qkv_row(g, lr, m0), r1 = qkv_row(g, lr + TC_SEG, m1);
            tile(r0, m0, r1, m1, TC_M, r.bid[2] * kq, kq, H, g * rows_group + lr);
            break;
        }
        case MK_OP_ATTN:
            pl[P_G - W_P] = r.bid[0]; pl[P_B - W_P] = r.bid[1]; pl[P_SPLIT - W_P] = r.bid[2];
            pl[P_T0 - W_P] = r.bid[2] * kn_T; pl[P_T - W_P] = kn_T; pl[P_NSPLIT - W_P] = nsplit[r.bid[1]];
            pl[P_LAYER - W_P] = op.layer;
            pl[P_ATHR - W_P] = r.trig >= 0 ? evs[r.trig].ntrig : 0;
            break;
        case MK_OP_O: {
            const int ko = Hq * D / ks_o;
            tile(r.bid[0] * TC_M, 0, r.bid[0] * TC_M + TC_SEG, 0, TC_M, r.bid[1] * ko, ko, Hq * D, r.bid[0] * TC_M);
            break;
        }
        case MK_OP_UP:
            tile(r.bid[0] * TC_SEG, 0, r.bid[0] * TC_SEG, 1, TC_SEG, 0, H, H, r.bid[0] * TC_SEG);
            break;
        case MK_OP_DOWN:
            tile(r.bid[0] * TC_M, 0, r.bid[0] * TC_M + TC_SEG, 0, TC_M, r.bid[1] * kc, kc, F, r.bid[0] * TC_M);
            break;
        case MK_OP_LM:
            tile(r.bid[0] * TC_M, 0, r.bid[0] * TC_M + TC_SEG, 0, std::min(TC_M, V - r.bid[0] * TC_M), 0, H, H,
                 r.bid[0] * TC_M);
            break;
        default:
            break;
        }
        p.tasks.push_back(t);
    }
    for (auto &t : p.tasks)
        if (t.opcode == MK_OP_EMBED) {
            t.w_ev[t.nw] = step_done; t.w_thr[t.nw] = p.thresholds[step_done]; t.w_off[t.nw++] = -1;
        }
    // algorithmic bytes at step 0: weights once, KV read, KV append, norm vectors
    int64_t weights = 0;
    for (auto &t : p.tasks)
        if (t.opcode >= MK_OP_QKV && t.opcode <= MK_OP_LM && t.opcode != MK_OP_ATTN) weights += t.cost;
    weights += (int64_t)B * H * 2;
    int64_t kv_read = 0;
    for (int b = 0; b < B; ++b) kv_read += (int64_t)2 * p.seq0[b] * Hkv * D * 2 * L;
    const int64_t kv_write = (int64_t)2 * B * Hkv * D * 2 * L;
    const int64_t norms = (int64_t)(2 * L + 1) * H * 2 + (m->qk_norm ? (int64_t)2 * L * D * 2 : 0);
    p.alg_bytes = weights + kv_read + kv_write + norms;
    if (pool) build_attn_pool(p, Hkv, kn_T, nsplit, max_steps);
    return finish_queues(p, false, p.schedule == MK_SCHED_TIMED);
}

// ---- Llama-style decode step --------------------------------------------

int plan_llama(const mk_model_desc *m, const mk_step_desc *s, const mk_target_desc *tgt, int num_workers,
               int smem_per_cta, Plan &p) {
    if (!m || !s || !tgt) return set_error(MK_ERR_INVALID, "null descriptor");
    p = Plan{};
    p.kind = PLAN_LLAMA;
    p.model = *m;
    p.mode = tgt->mode == MK_MODE_PER_OP ? MK_MODE_PER_OP : MK_MODE_MEGAKERNEL;
    p.num_workers = num_workers;
    const int L = m->layers, H = m->hidden, Hq = m->q_heads, Hkv = m->kv_heads, D = m->head_dim, F = m->ffn,
              V = m->vocab, B = s->batch;
    if (L <= 0 || H <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || F <= 0 || V <= 0 || B <= 0 || s->max_steps <= 0 ||
        !s->seq_len0 || num_workers <= 0)
        return set_error(MK_ERR_INVALID, "non-positive model or step size");
    if (Hq % Hkv) return set_error(MK_ERR_INVALID, "q_heads must be a multiple of kv_heads");
    const int G = Hq / Hkv;
    if (B > TC_MAXB) return set_error(MK_ERR_UNSUPPORTED, "batch above 16");
    if (D != 64 && D != 128) return set_error(MK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (G > 8 || 8 % G) return set_error(MK_ERR_UNSUPPORTED, "q heads per kv head must be 1, 2, 4 or 8");
    if (H % 8 || F % 8) return set_error(MK_ERR_UNSUPPORTED, "hidden and ffn must be multiples of 8");
    p.B = B;
    p.max_steps = s->max_steps;
    p.smax = s->cache_slots;
    p.capture = s->capture_hidden != 0;
    p.seq0.assign(s->seq_len0, s->seq_len0 + B);
    for (int b = 0; b < B; ++b) {
        if (p.seq0[b] < 0) return set_error(MK_ERR_INVALID, "negative sequence length");
        if ((int64_t)p.seq0[b] + s->max_steps > s->cache_slots)
            return set_error(MK_ERR_INVALID, "cache_slots smaller than seq_len0 + max_steps");
    }
    // FP8 projections: the batch-1 row-per-warp tiles over e4m3 rows of K = 2048
    const bool w8 = m->weight_fp8 != 0;
    if (w8 && (B != 1 || H != W8_K || Hq * D != W8_K || D != 64 || F % W8_K || tgt->tc_tiles > 0 ||
               (tgt->kchunk_down > 0 && tgt->kchunk_down != W8_K)))
        return set_error(MK_ERR_UNSUPPORTED, "FP8 projections need batch 1, hidden = q_heads x head_dim = 2048, "
                                             "head_dim 64, ffn a multiple of 2048 (MLP-down K chunks of 2048)");
    p.w8 = w8;
    const int wb = w8 ? 1 : 2;  // bytes per projection weight (the LM head stays bf16)
    // tensor-core tiles (128 weight rows x the batch): every K and row count a
    // multiple of 128, each head group's q/k/v rows whole 64-row segments
    const bool tc_shape = H % TC_M == 0 && (Hq * D) % TC_M == 0 && F % TC_M == 0 && ((G + 2) * D) % TC_M == 0 &&
                          D % TC_SEG == 0 && H <= 8192;
    if (tgt->tc_tiles > 0 && !tc_shape)
        return set_error(MK_ERR_UNSUPPORTED, "tensor-core tiles need hidden, q_heads*head_dim, ffn and a head "
                                             "group's q/k/v rows in multiples of 128 (hidden <= 8192)");
    if (B > 8 && (tgt->tc_tiles < 0 || !tc_shape))
        return set_error(MK_ERR_UNSUPPORTED, "batch above 8 needs tensor-core tiles");
    if (tgt->tc_tiles > 0 || (tgt->tc_tiles == 0 && B >= 8 && tc_shape))
        return plan_llama_tc(m, s, tgt, num_workers, smem_per_cta, p);
    auto clampi = [](int v, int lo, int hi) { return std::max(lo, std::min(hi, v)); };
    auto pow2_floor = [](int v) { int r = 1; while (r * 2 <= v) r *= 2; return r; };
    const int tile = 65536;
    if (tgt->page_bytes < 0 || tgt->page_bytes % 128) return set_error(MK_ERR_INVALID, "page_bytes must be a multiple of 128");
    if (tgt->schedule < MK_SCHED_DEFAULT || tgt->schedule > MK_SCHED_TIMED)
        return set_error(MK_ERR_INVALID, "schedule must be one of MK_SCHED_*");
    p.schedule = tgt->schedule == MK_SCHED_BYTES ? MK_SCHED_BYTES : MK_SCHED_TIMED;
    // batch > 1 with every K a multiple of 512: tensor-core tiles of 16 rows
    // (K slices of 64 per consumer warp); else batch > 4 keeps 8 rows x 8
    // sequences in registers
    const bool mma = H % 512 == 0 && (Hq * D) % 512 == 0 && std::min(F, 2048) % 512 == 0;
    const int rcap = B > 4 && !mma ? 8 : 16;
    // tensor-core tiles take 16 rows of any K (two pages of 8 rows at most)
    const int tile_g = mma ? 2 * tile : tile;
    int kn_qkv = tgt->rows_qkv > 0 ? tgt->rows_qkv : pow2_floor(clampi(tile_g / (2 * H), 1, rcap));
    int kn_o = tgt->rows_o > 0 ? tgt->rows_o : pow2_floor(clampi(tile_g / (2 * Hq * D), 1, rcap));
    int kn_up = tgt->rows_up > 0 ? tgt->rows_up : pow2_floor(clampi(tile_g / (4 * H), 1, rcap / 2));
    int kn_kc = tgt->kchunk_down;
    if (kn_kc <= 0) {
        kn_kc = 8;
        for (int c = 8; c <= std::min(F, 2048); c += 8)
            if (F % c == 0) kn_kc = c;
    }
    int kn_dn = tgt->rows_down > 0 ? tgt->rows_down : pow2_floor(clampi(tile_g / (2 * kn_kc), 1, rcap));
    int kn_lm = tgt->rows_lm > 0 ? tgt->rows_lm : pow2_floor(clampi(tile_g / (2 * H), 1, rcap));
    int kn_T = tgt->attn_split > 0 ? tgt->attn_split : clampi(16384 / (2 * D), 16, 256);
    if (tgt->attn_split <= 0) {
        // long caches: double the split length (up to 512 positions) while the
        // attention tasks outnumber the workers -- a second round of tasks costs
        // a whole per-task latency, a longer split only its extra positions
        auto attn_tasks = [&](int T) {
            int64_t n = 0;
            for (int b = 0; b < B; ++b) n += ceil_div(s->seq_len0[b] + s->max_steps, T);
            return n * Hkv;
        };
        while (2 * kn_T <= 512 && attn_tasks(kn_T) > (int64_t)num_workers) kn_T *= 2;
    }
    p.rows_qkv = kn_qkv; p.rows_o = kn_o; p.rows_up = kn_up; p.rows_down = kn_dn; p.kchunk_down = kn_kc;
    p.rows_lm = kn_lm; p.attn_split = kn_T;
    const int rows_group = (G + 2) * D;
    if (D % kn_qkv) return set_error(MK_ERR_UNSUPPORTED, "rows_qkv must divide head_dim");
    if (F % kn_up || F % kn_kc || kn_kc % 8) return set_error(MK_ERR_UNSUPPORTED, "rows_up / kchunk_down must divide ffn");
    if (kn_T > 512 || kn_T < 1) return set_error(MK_ERR_UNSUPPORTED, "attn_split must be 1..512");
    for (int K : {H, Hq * D, kn_kc})
        if (B * ceil_div(K, 2048) > 8 || K > 8192)
            return set_error(MK_ERR_UNSUPPORTED, "batch x K too large for register-held activations");
    // shared memory budget
    int kmax = std::max(std::max(H, Hq * D), kn_kc);
    int attn_slot = (G * (D + 16) + 2 * D) * 4;
    // GEMV activation buffer [B][K]; two small slots for per-instruction data
    // (attention q / new k / new v, the residual slice of O tiles)
    p.abuf_bytes = round_up(B * kmax * 4, 128);
    p.act_bytes = round_up(attn_slot + B * RESID_ROWS * 4, 128);
    const int maxb = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;  // kernel batch template
    // attention scratch, then the GEMV cross-warp reduction buffers
    p.red_bytes = round_up(red_bytes(maxb), 128);
    int aux = round_up(attn_aux_bytes(G, kn_T, D), 128) + NRED * p.red_bytes;
    // one activation buffer per slot when two fit in 32 KB: the activation
    // loader then stages instruction i + 1 while the consumers still read i
    p.abuf_count = 2 * p.abuf_bytes <= 32768 ? 2 : 1;
    int fixed = p.abuf_count * p.abuf_bytes + 2 * p.act_bytes + aux + MBAR_BYTES + CTRL_BYTES;
    p.aux_bytes = aux;
    // page size: a 64 KB tile per page when three of them fit (one wait and one
    // release per tile, three tiles in flight), else 32 KB, else 16 KB
    if (tgt->page_bytes > 0) {
        p.page_bytes = tgt->page_bytes;
    } else {
        p.page_bytes = 16384;
        for (int pb : {65536, 32768})
            if ((smem_per_cta - fixed) / pb >= 3) {
                p.page_bytes = pb;
                break;
            }
    }
    // tensor-core tiles want 8 rows per page: for K = 4096 that is 64 KB, which
    // three pages of need one activation buffer instead of two
    const int kmax_rows = std::max(std::max(H, Hq * D), kn_kc);
    if (tgt->page_bytes <= 0 && mma && p.page_bytes < 16 * kmax_rows && p.abuf_count == 2 && 16 * kmax_rows <= 65536 &&
        (smem_per_cta - (fixed - p.abuf_bytes)) / (16 * kmax_rows) >= 3) {
        p.abuf_count = 1;
        fixed -= p.abuf_bytes;
        p.page_bytes = 16 * kmax_rows;
    }
    for (int K : {H, Hq * D, kn_kc})
        if (2 * K > p.page_bytes) return set_error(MK_ERR_UNSUPPORTED, "a weight row does not fit one page");
    // Batch 1 with pages of exactly 16 rows (K = page_bytes / 32, a multiple of
    // 256 up to 2048): the row-per-warp path takes tiles of any number of
    // whole pages (MLP-up pages: 8 gate + 8 up rows), which spreads each
    // instruction's fixed costs over more bytes.  Defaults: QKV 32 rows (two
    // pages, a tile stays within one head), MLP-up 64 gate rows and MLP-down 64
    // rows (8 and 4 pages; each op then has 128 tiles, a multiple of the
    // down K chunks), the LM head one tile per worker; O keeps one page (its
    // residual rows are staged with the activation).
    auto multi_page = [&](int K) { return B == 1 && K % 256 == 0 && K <= 2048 && p.page_bytes == 32 * K; };
    if (multi_page(H) && tgt->rows_lm <= 0) {
        const int pages = ceil_div(V, 16);
        kn_lm = 16 * std::min(64, ceil_div(pages, num_workers));
    }
    if (multi_page(H) && tgt->rows_up <= 0 && F % 64 == 0) kn_up = 64;
    if (multi_page(kn_kc) && tgt->rows_down <= 0 && H % 64 == 0) kn_dn = 64;
    if (multi_page(H) && tgt->rows_qkv <= 0 && D % 32 == 0) kn_qkv = 32;
    p.rows_qkv = kn_qkv; p.rows_up = kn_up; p.rows_down = kn_dn; p.rows_lm = kn_lm;
    // the tensor-core tiles need whole rows in at most two pages of 8 or more
    bool mma_pages = mma;
    for (int K : {H, Hq * D, kn_kc})
        if (p.page_bytes / (2 * K) < 8 || K % 512) mma_pages = false;
    if (B > 4 && !mma_pages) {  // back to 8 rows x 8 sequences in registers
        if (tgt->rows_qkv <= 0) kn_qkv = std::min(kn_qkv, 8);
        if (tgt->rows_o <= 0) kn_o = std::min(kn_o, 8);
        if (tgt->rows_down <= 0) kn_dn = std::min(kn_dn, 8);
        if (tgt->rows_lm <= 0) kn_lm = std::min(kn_lm, 8);
        if (tgt->rows_up <= 0) kn_up = std::min(kn_up, 4);
        p.rows_qkv = kn_qkv; p.rows_o = kn_o; p.rows_up = kn_up; p.rows_down = kn_dn; p.rows_lm = kn_lm;
    }
    const int rmax = B > 4 && !mma_pages ? 8 : MAX_TILE_ROWS;
    auto rows_ok = [&](int rows, int K, bool up, bool o) {
        if (rows <= rmax) return up ? rows / 2 <= 8 || (rows / 2) % 8 == 0 : true;
        // whole 16-row pages on the batch-1 row-per-warp path, at most 64 of them
        return !o && multi_page(K) && rows <= 16 * 64 && rows % 16 == 0;
    };
    if (!rows_ok(kn_qkv, H, false, false) || !rows_ok(kn_o, Hq * D, false, true) || !rows_ok(kn_dn, kn_kc, false, false) ||
        !rows_ok(kn_lm, H, false, false) || !rows_ok(2 * kn_up, H, true, false))
        return set_error(MK_ERR_UNSUPPORTED, "tile rows above 16 (8 for batch > 4; mlp-up: half of that), except "
                                             "tiles of up to 64 whole 16-row pages at batch 1 (not O; mlp-up gate "
                                             "rows a multiple of 8)");
    if (F % kn_up) return set_error(MK_ERR_UNSUPPORTED, "rows_up must divide ffn");
    if (w8) {
        // 32 e4m3 rows per page: a tile is one page of at most 32 rows or whole
        // pages (MLP-up: pages of 16 gate + 16 up rows), and stays in one
        // 128-row block of the block scales (a power of two of rows up to 128)
        auto pow2 = [](int v) { return v > 0 && (v & (v - 1)) == 0; };
        if (kn_kc != W8_K || p.page_bytes != W8_ROWS * W8_K || !pow2(kn_qkv) || kn_qkv > 128 || !pow2(kn_dn) ||
            kn_dn > 128 || !pow2(kn_o) || kn_o > RESID_ROWS || !pow2(kn_up) || kn_up < 16 || kn_up > 64)
            return set_error(MK_ERR_UNSUPPORTED, "FP8 tiles: 64 KB pages, MLP-down K chunks of 2048, QKV / MLP-down "
                                                 "rows a power of two up to 128, O up to 16, MLP-up 16, 32 or 64 gate rows");
    }
    if (kn_T * D * 2 > p.page_bytes * 8) return set_error(MK_ERR_UNSUPPORTED, "attention split too long");
    p.num_pages = std::min(MAX_PAGES, (smem_per_cta - fixed) / p.page_bytes);
    p.smem_bytes = fixed + p.num_pages * p.page_bytes;
    // pages used by the largest instruction
    auto pages_for = [&](int rows, int row_bytes) {
        if (rows <= 0) return 0;
        int rpp = p.page_bytes / row_bytes;
        return ceil_div(rows, rpp);
    };
    // GEMV tiles release each page before waiting for the next, so any number
    // of pages streams through the ring; an attention task holds all its K
    // pages (at most 4), releases them, then waits for its V pages
    int need = pages_for(kn_T, 2 * D);
    if (need > 4 || p.num_pages < std::max(2, need))
        return set_error(MK_ERR_UNSUPPORTED, "shared memory too small for the page pool");

    // ---- op list (topological): embed, per layer qkv attn o up down, lm
    std::vector<int> nsplit(B);
    for (int b = 0; b < B; ++b) nsplit[b] = ceil_div(p.seq0[b] + s->max_steps, kn_T);
    int ns_max = *std::max_element(nsplit.begin(), nsplit.end());
    p.nsplit_max = ns_max;
    const bool pool = tgt->attn_pool != 0;  // device-side attention dispatch
    if (pool && B < 2) return set_error(MK_ERR_UNSUPPORTED, "attention pools are for batches of 2 or more");
    int64_t attn_layer_bytes = 0;           // (the pools' share of it is their scheduling cost)
    for (int b = 0; b < B; ++b)
        for (int sp = 0; sp < nsplit[b]; ++sp)
            attn_layer_bytes += (int64_t)2 * D * 2 * Hkv * std::max(0, std::min(kn_T, p.seq0[b] + s->max_steps - 1 - sp * kn_T));
    std::vector<int> seq0 = p.seq0;
    const int max_steps = s->max_steps;
    std::vector<OpDef> ops;
    std::vector<EdgeDef> edges;
    auto add_op = [&](int opcode, int layer, int gx, int gy, int gz) {
        OpDef o;
        o.opcode = opcode;
        o.layer = layer;
        o.grid[0] = gx; o.grid[1] = gy; o.grid[2] = gz;
        ops.push_back(o);
        return (int)ops.size() - 1;
    };
    auto rows_cost = [](int n_rows, int rows, int kdim, int bytes) {
        return [=](const int *b) { return (int64_t)std::min(rows, n_rows - b[0] * rows) * kdim * bytes; };
    };
    int emb = add_op(MK_OP_EMBED, -1, 1, 1, 1);
    ops[emb].cost = [=](const int *) { return (int64_t)B * H * 2; };
    int prev = emb;
    for (int l = 0; l < L; ++l) {
        int q = add_op(MK_OP_QKV, l, Hkv, rows_group / kn_qkv, 1);
        ops[q].cost = [=](const int *) { return (int64_t)kn_qkv * H * wb; };
        int a;
        if (pool) {  // one pool per worker; its cost: the layer's attention bytes over the workers
            a = add_op(MK_OP_ATTN_POOL, l, num_workers, 1, 1);
            ops[a].cost = [=](const int *) { return attn_layer_bytes / num_workers; };
        } else {
            a = add_op(MK_OP_ATTN, l, Hkv, B, ns_max);
            ops[a].exists = [nsplit](const int *b) { return b[2] < nsplit[b[1]]; };
            ops[a].cost = [=](const int *b) {
                int last = seq0[b[1]] + max_steps - 1;
                int rows = std::max(0, std::min(kn_T, last - b[2] * kn_T));
                return (int64_t)2 * D * 2 * rows;
            };
        }
        int o = add_op(MK_OP_O, l, ceil_div(H, kn_o), 1, 1);
        ops[o].cost = rows_cost(H, kn_o, Hq * D, wb);
        int u = add_op(MK_OP_UP, l, F / kn_up, 1, 1);
        ops[u].cost = [=](const int *) { return (int64_t)2 * kn_up * H * wb; };
        int d = add_op(MK_OP_DOWN, l, ceil_div(H, kn_dn), F / kn_kc, 1);
        ops[d].cost = rows_cost(H, kn_dn, kn_kc, wb);
        if (prev == emb) edges.push_back({prev, q, {-1, -1, -1}, {-1, -1, -1}});
        else edges.push_back({prev, q, {1, -1, -1}, {-1, -1, -1}});
        if (pool) {  // a pool may claim any group's task
            edges.push_back({q, a, {-1, -1, -1}, {-1, -1, -1}});
            edges.push_back({a, o, {-1, -1, -1}, {-1, -1, -1}});
        } else {
            edges.push_back({q, a, {1, 2, -1}, {1, 0, -1}});   // qkv [B, Hkv, rows]: group & row cuts vs batch & group
            edges.push_back({a, o, {1, 0, -1}, {-1, -1, -1}});  // attn_out read whole; split axis reduces
        }
        edges.push_back({o, u, {1, -1, -1}, {-1, -1, -1}}); // h read whole
        edges.push_back({u, d, {1, -1, -1}, {-1, 1, -1}});  // act [B, F]: tiles vs K chunks
        prev = d;
    }
    int lm = add_op(MK_OP_LM, -1, ceil_div(V, kn_lm), 1, 1);
    ops[lm].cost = rows_cost(V, kn_lm, H, 2);
    edges.push_back({prev, lm, {1, -1, -1}, {-1, -1, -1}});

    std::vector<RawTask> raw;
    std::vector<RawEvent> evs;
    int n_first;
    int rc = build_tasks(ops, edges, raw, evs, n_first);
    if (rc) return rc;
    // longest-first inside each successor range (stable), ranges in order
    std::vector<int64_t> cost(raw.size());
    for (size_t i = 0; i < raw.size(); ++i) cost[i] = ops[raw[i].op].cost(raw[i].bid);
    std::vector<std::pair<int, int>> ranges{{0, n_first}};
    for (auto &e : evs) ranges.push_back({e.first, e.last});
    std::sort(ranges.begin(), ranges.end());
    std::vector<int> order;
    for (auto &r : ranges) {
        std::vector<int> ids(r.second - r.first);
        std::iota(ids.begin(), ids.end(), r.first);
        std::stable_sort(ids.begin(), ids.end(), [&](int x, int y) { return cost[x] > cost[y]; });
        order.insert(order.end(), ids.begin(), ids.end());
    }
    if ((int)order.size() != (int)raw.size()) return set_error(MK_ERR_INVALID, "task ranges do not cover the graph");
    const int step_done = (int)evs.size();
    for (auto &e : evs) p.thresholds.push_back(e.ntrig);
    p.thresholds.push_back(0);
    for (auto &e : evs) p.events.push_back({e.ntrig, e.first, e.last});
    p.events.push_back({0, 0, n_first});
    // operand rows = ops
    p.num_ops = (int)ops.size();
    for (auto &o : ops) {
        p.op_kind.push_back(o.opcode);
        p.op_layer.push_back(o.layer);
    }
    std::vector<int> first_task_of_op(ops.size(), -1);
    p.tasks.reserve(order.size());
    for (int old : order) {
        const RawTask &r = raw[old];
        const OpDef &op = ops[r.op];
        TaskRec t;
        t.opcode = op.opcode;
        t.op_row = r.op;
        t.layer = op.layer;
        std::memcpy(t.bid, r.bid, sizeof(t.bid));
        t.cost = cost[old];
        if (r.dep >= 0) {
            t.w_ev[t.nw] = r.dep; t.w_thr[t.nw] = evs[r.dep].ntrig; t.w_off[t.nw++] = 0;
        }
        if (r.trig >= 0) { t.s_ev[t.ns] = r.trig; t.s_inc[t.ns++] = 1; }
        if (op.opcode == MK_OP_LM) {
            t.s_ev[t.ns] = step_done; t.s_inc[t.ns++] = 1;
            p.thresholds[step_done]++;
        }
        bool first_of_op = first_task_of_op[r.op] < 0;
        if (first_of_op) first_task_of_op[r.op] = (int)p.tasks.size();
        int32_t *pl = t.payload;
        switch (op.opcode) {
        case MK_OP_QKV: {
            int g = r.bid[0], lr = r.bid[1] * kn_qkv;
            pl[P_NROWS - W_P] = kn_qkv;
            pl[P_K0 - W_P] = 0;
            pl[P_KC - W_P] = H;
            pl[P_KTOT - W_P] = H;
            pl[P_OUT0 - W_P] = g * rows_group + lr;
            if (lr < G * D) { pl[P_MAT - W_P] = 0; pl[P_ROW0 - W_P] = g * G * D + lr; }
            else if (lr < (G + 1) * D) { pl[P_MAT - W_P] = 1; pl[P_ROW0 - W_P] = g * D + lr - G * D; }
            else { pl[P_MAT - W_P] = 2; pl[P_ROW0 - W_P] = g * D + lr - (G + 1) * D; }
            pl[P_SNAP - W_P] = (p.capture && op.layer > 0 && first_of_op) ? op.layer : 0;  // layer-1 residual
            break;
        }
        case MK_OP_ATTN:
            pl[P_G - W_P] = r.bid[0]; pl[P_B - W_P] = r.bid[1]; pl[P_SPLIT - W_P] = r.bid[2];
            pl[P_T0 - W_P] = r.bid[2] * kn_T; pl[P_T - W_P] = kn_T; pl[P_NSPLIT - W_P] = nsplit[r.bid[1]];
            pl[P_LAYER - W_P] = op.layer;
            pl[P_ATHR - W_P] = r.trig >= 0 ? evs[r.trig].ntrig : 0;
            break;
        case MK_OP_O:
            pl[P_ROW0 - W_P] = r.bid[0] * kn_o; pl[P_NROWS - W_P] = std::min(kn_o, H - r.bid[0] * kn_o);
            pl[P_K0 - W_P] = 0; pl[P_KC - W_P] = Hq * D; pl[P_KTOT - W_P] = Hq * D; pl[P_OUT0 - W_P] = r.bid[0] * kn_o;
            break;
        case MK_OP_UP:
            pl[P_ROW0 - W_P] = r.bid[0] * kn_up; pl[P_NROWS - W_P] = kn_up;
            pl[P_K0 - W_P] = 0; pl[P_KC - W_P] = H; pl[P_KTOT - W_P] = H; pl[P_OUT0 - W_P] = r.bid[0] * kn_up;
            break;
        case MK_OP_DOWN:
            pl[P_ROW0 - W_P] = r.bid[0] * kn_dn; pl[P_NROWS - W_P] = std::min(kn_dn, H - r.bid[0] * kn_dn);
            pl[P_K0 - W_P] = r.bid[1] * kn_kc; pl[P_KC - W_P] = kn_kc; pl[P_KTOT - W_P] = F;
            pl[P_OUT0 - W_P] = r.bid[0] * kn_dn;
            break;
        case MK_OP_LM:
            pl[P_ROW0 - W_P] = r.bid[0] * kn_lm; pl[P_NROWS - W_P] = std::min(kn_lm, V - r.bid[0] * kn_lm);
            pl[P_K0 - W_P] = 0; pl[P_KC - W_P] = H; pl[P_KTOT - W_P] = H; pl[P_OUT0 - W_P] = r.bid[0] * kn_lm;
            pl[P_SNAP - W_P] = (p.capture && first_of_op) ? L : 0;
            break;
        default:
            break;
        }
        if (op.opcode != MK_OP_ATTN && op.opcode != MK_OP_EMBED && op.opcode != MK_OP_ATTN_POOL) {
            // the tile's rows (MLP-up: gate rows, then up rows) packed into pages
            const bool e4m3 = w8 && op.opcode != MK_OP_LM;
            pl[P_W8 - W_P] = e4m3 ? 1 : 0;
            const int rpp = p.page_bytes / ((e4m3 ? 1 : 2) * pl[P_KC - W_P]);
            pl[P_RPP - W_P] = rpp;
            pl[P_NPG - W_P] = ceil_div((op.opcode == MK_OP_UP ? 2 : 1) * pl[P_NROWS - W_P], rpp);
        }
        p.tasks.push_back(t);
    }
    for (auto &t : p.tasks)
        if (t.opcode == MK_OP_EMBED) {
            t.w_ev[t.nw] = step_done; t.w_thr[t.nw] = p.thresholds[step_done]; t.w_off[t.nw++] = -1;
        }
    // algorithmic bytes at step 0: weights once, KV read, KV append
    int64_t weights = 0;
    for (auto &t : p.tasks)
        if (t.opcode != MK_OP_ATTN && t.opcode != MK_OP_EMBED && t.opcode != MK_OP_ATTN_POOL) weights += t.cost;
    weights += (int64_t)B * H * 2;  // embedding rows
    int64_t kv_read = 0;
    for (int b = 0; b < B; ++b) kv_read += (int64_t)2 * p.seq0[b] * Hkv * D * 2 * L;
    int64_t kv_write = (int64_t)2 * B * Hkv * D * 2 * L;
    int64_t norms = (int64_t)(2 * L + 1) * H * 2 + (m->qk_norm ? (int64_t)2 * L * D * 2 : 0);
    int64_t scales = 0;  // FP8: one fp32 per 128 x 128 block of every projection
    if (w8) {
        auto blocks = [](int n, int k) { return (int64_t)ceil_div(n, 128) * (k / 128); };
        scales = (int64_t)L * 4 *
                 (blocks(Hq * D, H) + 2 * blocks(Hkv * D, H) + blocks(H, Hq * D) + 2 * blocks(F, H) + blocks(H, F));
    }
    p.alg_bytes = weights + kv_read + kv_write + norms + scales;
    // the lean batch-1 kernel instance: every GEMV tile must take the
    // row-per-warp path (the device applies the same rule to each tile);
    // FP8 plans run their own instance
    p.lean = B == 1 && D == 64 && !w8;
    for (const TaskRec &t : p.tasks) {
        if (!p.lean) break;
        if (t.opcode < MK_OP_QKV || t.opcode > MK_OP_LM || t.opcode == MK_OP_ATTN) continue;
        const int kc = t.payload[P_KC - W_P], nrows = t.payload[P_NROWS - W_P], npg = t.payload[P_NPG - W_P];
        const bool up = t.opcode == MK_OP_UP;
        bool ok = kc % 256 == 0 && kc <= 2048;
        if (ok && npg == 1) ok = up ? nrows == 8 : nrows <= 16;
        else if (ok) ok = npg <= 64 && t.opcode != MK_OP_O && p.page_bytes == 32 * kc &&
                          (up ? nrows == 8 * npg : nrows > 16 * (npg - 1) && nrows <= 16 * npg);
        p.lean = ok;
    }
    if (pool) build_attn_pool(p, Hkv, kn_T, nsplit, s->max_steps);
    return finish_queues(p, false, p.schedule == MK_SCHED_TIMED);
}

// ---- GLM FP8 pre-attention block ------------------------------------------

int plan_glm(const mk_glm_desc *g, const mk_target_desc *tgt, int num_workers, int smem_per_cta, Plan &p) {
    if (!g || !tgt) return set_error(MK_ERR_INVALID, "null descriptor");
    p = Plan{};
    p.kind = PLAN_GLM;
    p.glm = *g;
    p.mode = MK_MODE_MEGAKERNEL;
    p.num_workers = num_workers;
    const int M = g->requests * g->tokens, H = g->hidden, QL = g->q_lora, KL = g->kv_lora, R = g->rope;
    const int NQKVA = QL + KL + R, NQ = g->q_heads * g->q_head_dim, NI = g->idx_heads * g->idx_dim;
    if (g->requests <= 0 || g->tokens <= 0 || H <= 0 || QL <= 0 || KL <= 0 || g->q_heads <= 0 ||
        g->q_head_dim <= 0 || g->gate_heads <= 0 || g->idx_heads <= 0 || g->idx_dim <= 0 || g->max_steps <= 0 ||
        g->pos0 < 0 || g->cache_slots <= 0 || !(g->eps > 0))
        return set_error(MK_ERR_INVALID, "non-positive GLM block size");
    if (g->pos0 + g->tokens > g->cache_slots) return set_error(MK_ERR_INVALID, "new tokens past the cache end");
    if (M > GLM_MAX_M || R != GLM_ROPE || H % 128 || QL % 128 || KL % 128 || H / 128 > 64 || QL / 128 > 16 ||
        g->q_head_dim % 64 || g->q_head_dim < 64 || g->idx_dim % 64 || g->idx_dim < 64 || NQKVA % 16 ||
        g->gate_heads % 16 || g->idx_dim % 16 || H > 8192 || QL > 8192 || KL > 2 * CONSUMERS ||
        g->idx_dim - R > 2 * CONSUMERS || g->gate_heads > CONSUMERS)
        return set_error(MK_ERR_UNSUPPORTED, "GLM block sizes outside the kernels' tiling");
    if (tgt->schedule < MK_SCHED_DEFAULT || tgt->schedule > MK_SCHED_TIMED)
        return set_error(MK_ERR_INVALID, "schedule must be one of MK_SCHED_*");
    p.schedule = tgt->schedule == MK_SCHED_BYTES ? MK_SCHED_BYTES : MK_SCHED_TIMED;
    p.B = 1;  // the batch-1 kernel instance; the GLM ops take M from their payload
    p.max_steps = g->max_steps;
    // tcgen05 tiles: the 16 token rows are the MMA's N side; a second-level
    // tile stages its whole K range of activation codes
    const bool tc_shape = M == GT_N && QL / 128 <= GT_MAX_STAGES;
    if (tgt->tc_tiles > 0 && !tc_shape)
        return set_error(MK_ERR_UNSUPPORTED, "tensor-core GLM tiles need M = 16 and q_lora <= 1536");
    p.tc = tgt->tc_tiles >= 0 && tc_shape;
    p.np = p.tc ? GT_N : 0;
    if (p.tc) {
        // shared memory: two activation slots (a tile's codes in 2 KB stages,
        // 1024-byte aligned for the 128-byte swizzle, then its scales), two
        // 512-byte hand-off slots (A0 / FIN), the epilogue's RoPE exchange,
        // 16 KB pages of one weight stage each
        p.abuf_bytes = round_up(GT_XSLOT_BYTES, 1024);
        p.abuf_count = GT_XSLOTS;
        p.act_bytes = 512;
        p.red_bytes = 256;
        p.aux_bytes = NRED * p.red_bytes + GT_EX_BYTES + 256;
        p.page_bytes = GT_STAGE_BYTES;
    } else {
        // shared memory: the staged A operand (M <= 16 padded rows of K bytes, then
        // the scales), a 4 KB tile reduction area per buffer, pages of whole weight rows
        const int KMAX = std::max(H, QL);
        p.abuf_bytes = round_up(GLM_MAX_M * (KMAX + 16) + GLM_MAX_M * (KMAX / 128) * 4, 128);
        p.abuf_count = 1;
        p.act_bytes = 128;
        p.red_bytes = 4096;
        p.aux_bytes = NRED * p.red_bytes + 256;
        p.page_bytes = 48 * 1024;  // 8 rows of K = 6144 or 32 rows of K = 1536
        for (int K : {H, QL})
            if (p.page_bytes % K) return set_error(MK_ERR_UNSUPPORTED, "a page must hold whole weight rows");
    }
    const int fixed = p.abuf_count * p.abuf_bytes + 2 * p.act_bytes + p.aux_bytes + MBAR_BYTES + CTRL_BYTES;
    p.num_pages = std::min(p.tc ? MAX_PAGES_TC : MAX_PAGES, (smem_per_cta - fixed) / p.page_bytes);
    if (p.num_pages < 2) return set_error(MK_ERR_UNSUPPORTED, "shared memory holds fewer than two pages");
    p.smem_bytes = fixed + p.num_pages * p.page_bytes;
    // ops (operand rows): A0, QKV-A, Head-Gate, Indexer-K, FIN, Q-B, Indexer-Q
    enum { OA0, OQKVA, OGATE, OIK, OFIN, OQB, OIQ, NOPS };
    const int kinds[NOPS] = {MK_OP_GLM_A0, MK_OP_GLM_GEMM, MK_OP_GLM_GEMM, MK_OP_GLM_GEMM, MK_OP_GLM_FIN,
                             MK_OP_GLM_GEMM, MK_OP_GLM_GEMM};
    p.num_ops = NOPS;
    for (int o = 0; o < NOPS; ++o) {
        p.op_kind.push_back(kinds[o]);
        p.op_layer.push_back(0);
    }
    // events: 0 A0 done, 1 QKV-A + Indexer-K done, 2 FIN done, 3 step done
    enum { EV_A0, EV_B, EV_FIN, EV_DONE, NEV };
    p.thresholds.assign(NEV, 0);
    auto add = [&](int op, int opcode, int64_t cost, int wait_ev, int sig_ev) -> TaskRec & {
        TaskRec t;
        t.opcode = opcode;
        t.op_row = op;
        t.layer = 0;
        t.cost = cost;
        if (wait_ev >= 0) { t.w_ev[t.nw] = wait_ev; t.w_off[t.nw++] = 0; }
        if (sig_ev >= 0) { t.s_ev[t.ns] = sig_ev; t.s_inc[t.ns++] = 1; p.thresholds[sig_ev]++; }
        t.payload[P_GL_M - W_P] = M;
        t.payload[P_GL_T - W_P] = g->tokens;
        t.payload[P_GL_POS0 - W_P] = g->pos0;
        p.tasks.push_back(t);
        return p.tasks.back();
    };
    for (int m = 0; m < M; ++m) {
        TaskRec &t = add(OA0, MK_OP_GLM_A0, (int64_t)H * 2 * 3, -1, EV_A0);
        t.bid[0] = m;
        t.payload[P_ROW0 - W_P] = m;
    }
    const int rpp_h = p.page_bytes / H, rpp_q = p.page_bytes / QL;
    auto gemm = [&](int op, int N, int K, int nr, int rpp, int wait_ev, int sig_ev, int ld, int head) {
        for (int n0 = 0; n0 < N; n0 += nr) {
            TaskRec &t = add(op, MK_OP_GLM_GEMM, (int64_t)nr * K, wait_ev, sig_ev);
            t.bid[0] = n0 / nr;
            int32_t *pl = t.payload;
            pl[P_ROW0 - W_P] = n0; pl[P_NROWS - W_P] = nr; pl[P_K0 - W_P] = 0; pl[P_KC - W_P] = K;
            pl[P_KTOT - W_P] = K; pl[P_OUT0 - W_P] = n0; pl[P_RPP - W_P] = rpp; pl[P_NPG - W_P] = ceil_div(nr, rpp);
            pl[P_GL_LD - W_P] = ld;
            pl[P_GL_ROPE - W_P] = head > 0 && n0 % head == head - GLM_ROPE ? 1 : 0;
        }
    };
    // tcgen05 tiles: 128 weight rows (the last row tile of a matrix may hold
    // fewer; the tile reads zeros past the end) over P_NPG stages of 128 K;
    // the first GEMMs split K into `ks` parts that add into fp32 sums (FIN
    // rounds them), the second GEMMs store their bf16 outputs with RoPE on
    // the 64-row halves that are a head's last 64 rows
    auto gemm_tc = [&](int op, int N, int K, int ks, bool sums, int wait_ev, int sig_ev, int ld, int head) {
        const int kc = K / ks;
        for (int n0 = 0; n0 < N; n0 += GT_M) {
            for (int part = 0; part < ks; ++part) {
                const int nr = std::min(GT_M, N - n0);
                TaskRec &t = add(op, MK_OP_GLM_GEMM, (int64_t)nr * kc, wait_ev, sig_ev);
                t.bid[0] = n0 / GT_M;
                t.bid[1] = part;
                int32_t *pl = t.payload;
                pl[P_ROW0 - W_P] = n0; pl[P_NROWS - W_P] = nr; pl[P_K0 - W_P] = part * kc; pl[P_KC - W_P] = kc;
                pl[P_KTOT - W_P] = K; pl[P_OUT0 - W_P] = n0; pl[P_RPP - W_P] = 0; pl[P_NPG - W_P] = kc / GT_KS;
                pl[P_GL_LD - W_P] = ld;
                int rope = 0;
                for (int j = 0; j < 2; ++j) {
                    const int r = n0 + GLM_ROPE * j;
                    if (head > 0 && r < N && r % head == head - GLM_ROPE) rope |= 1 << j;
                }
                pl[P_GL_ROPE - W_P] = rope;
                pl[P_GL_TCT - W_P] = 1;
                pl[P_GL_SUM - W_P] = sums ? 1 : 0;
            }
        }
    };
    if (p.tc) {
        // K parts of the first GEMMs: the largest divisor of H / 128 that
        // keeps row tiles x parts within the workers, with at most
        // GT_MAX_STAGES stages per part
        const int KB = H / GT_KS;
        const int rt = ceil_div(NQKVA, GT_M) + ceil_div(g->gate_heads, GT_M) + ceil_div(g->idx_dim, GT_M);
        int ks = 0;
        for (int d = 1; d <= KB; ++d)
            if (KB % d == 0 && KB / d <= GT_MAX_STAGES && (ks == 0 || rt * d <= num_workers)) ks = d;
        p.glm_ksplit = ks;
        // (Head-Gate's sums are rounded by FIN too, so its tiles count into FIN's event)
        gemm_tc(OQKVA, NQKVA, H, ks, true, EV_A0, EV_B, NQKVA, 0);
        gemm_tc(OIK, g->idx_dim, H, ks, true, EV_A0, EV_B, g->idx_dim, 0);
        gemm_tc(OGATE, g->gate_heads, H, ks, true, EV_A0, EV_B, g->gate_heads, 0);
    } else {
        gemm(OQKVA, NQKVA, H, 16, rpp_h, EV_A0, EV_B, NQKVA, 0);
        gemm(OIK, g->idx_dim, H, 16, rpp_h, EV_A0, EV_B, g->idx_dim, 0);
        gemm(OGATE, g->gate_heads, H, 16, rpp_h, EV_A0, EV_DONE, g->gate_heads, 0);
    }
    for (int m = 0; m < M; ++m) {
        TaskRec &t = add(OFIN, MK_OP_GLM_FIN, (int64_t)(NQKVA + g->idx_dim) * 2, EV_B, EV_FIN);
        t.bid[0] = m;
        int32_t *pl = t.payload;
        pl[P_ROW0 - W_P] = m; pl[P_GF_QLORA - W_P] = QL; pl[P_GF_KVLORA - W_P] = KL; pl[P_GF_IDX - W_P] = g->idx_dim;
        pl[P_GF_SLOTS - W_P] = g->cache_slots; pl[P_GF_QKVA_LD - W_P] = NQKVA;
        pl[P_GF_SUMS - W_P] = p.tc ? 1 : 0; pl[P_GF_GATE - W_P] = g->gate_heads;
    }
    // the last tasks of a step (Head-Gate above, FIN's cache writes, Q-B,
    // Indexer-Q) count into the step-done event
    for (auto &t : p.tasks)
        if (t.opcode == MK_OP_GLM_FIN) { t.s_ev[t.ns] = EV_DONE; t.s_inc[t.ns++] = 1; p.thresholds[EV_DONE]++; }
    if (p.tc) {
        gemm_tc(OQB, NQ, QL, 1, false, EV_FIN, EV_DONE, NQ, g->q_head_dim);
        gemm_tc(OIQ, NI, QL, 1, false, EV_FIN, EV_DONE, NI, g->idx_dim);
    } else {
        gemm(OQB, NQ, QL, 64, rpp_q, EV_FIN, EV_DONE, NQ, g->q_head_dim);
        gemm(OIQ, NI, QL, 64, rpp_q, EV_FIN, EV_DONE, NI, g->idx_dim);
    }
    if (NQ % 64 || NI % 64) return set_error(MK_ERR_UNSUPPORTED, "Q-B / Indexer-Q widths must be multiples of 64");
    for (auto &t : p.tasks) {
        for (int i = 0; i < t.nw; ++i) t.w_thr[i] = p.thresholds[t.w_ev[i]];
        if (t.opcode == MK_OP_GLM_A0) {  // the previous step's last tasks
            t.w_ev[t.nw] = EV_DONE; t.w_thr[t.nw] = p.thresholds[EV_DONE]; t.w_off[t.nw++] = -1;
        }
    }
    // RoPE table: angle (pos0 + j) * theta^(-i/32) of token j and pair i, in double
    for (int j = 0; j < g->tokens; ++j)
        for (int i = 0; i < GLM_ROPE / 2; ++i) {
            const double a = (double)(g->pos0 + j) * std::pow((double)g->rope_theta, -(double)i / (GLM_ROPE / 2));
            p.rope_tab.push_back((float)std::cos(a));
            p.rope_tab.push_back((float)std::sin(a));
        }
    p.events.assign(NEV, {0, 0, 0});
    for (int e = 0; e < NEV; ++e) p.events[e].ntrig = p.thresholds[e];
    // algorithmic bytes: FP8 weights and their scales once; the block's inputs,
    // outputs and cache rows; each intermediate written and read once
    const int64_t KBH = H / 128, KBQ = QL / 128;
    const int64_t wbytes = (int64_t)(NQKVA + g->gate_heads + g->idx_dim) * H + (int64_t)(NQ + NI) * QL;
    const int64_t sbytes = 4 * (ceil_div(NQKVA, 128) + ceil_div(g->gate_heads, 128) + ceil_div(g->idx_dim, 128)) * KBH +
                           4 * (ceil_div(NQ, 128) + ceil_div(NI, 128)) * KBQ;
    const int64_t io = (int64_t)M * H * 2 * 3 + H * 2 + (int64_t)M * (g->gate_heads + NQ + NI) * 2 +
                       (int64_t)M * (KL + R + g->idx_dim) * 2;
    const int64_t inter = (int64_t)M * (H + KBH * 4 + (NQKVA + g->idx_dim) * 2 + QL + KBQ * 4);
    p.alg_bytes = wbytes + sbytes + io + inter;
    return finish_queues(p, false, p.schedule == MK_SCHED_TIMED);
}

}  // namespace mk
