// Critical-wave split planner (host).  LiquidCP Section 5.2 and Appendix A.2.
//
// Model: K compute CTAs; with k CTAs running attention, every running task
// advances at rate 1/tau(k), tau(k) = max(rho, k/K) (Eq. 5).  A task over n_t
// tiles carries c_attn = n_t + delta_attn.  Tasks go, in queue order, to the
// first free CTA (lowest index).  A CTA that is free when no attention task is
// left releases its warps; a history reduction costs delta_red + gamma*v*s
// (Eq. 6), takes one warp in queue order and starts once the warp is free and
// every attention task of its sequence has finished.  The score is the latest
// completion.  Search: from NoSplit, try +1 per sequence below its limit and a
// joint +1 for the sequences tied at the attention tail; accept the best only
// if it lowers the score; ties go to earlier attention completion, fewer
// attention tasks, fewer splits.  Final: best of NoSplit / search / reference,
// and a split plan only if >= adopt_margin below NoSplit.
#include "planner.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <functional>
#include <thread>

namespace skv {
namespace model {

namespace {
constexpr double kEps = 1e-9;

bool feq(double a, double b) {
    return std::fabs(a - b) <= kEps * std::max({1.0, std::fabs(a), std::fabs(b)});
}

// lexicographic (score, attn_end, tasks, splits) with a tolerance on times
int cmp_result(const SimResult& a, const SimResult& b) {
    if (!feq(a.score, b.score)) return a.score < b.score ? -1 : 1;
    if (!feq(a.attn_end, b.attn_end)) return a.attn_end < b.attn_end ? -1 : 1;
    if (a.n_attn_tasks != b.n_attn_tasks) return a.n_attn_tasks < b.n_attn_tasks ? -1 : 1;
    if (a.total_splits != b.total_splits) return a.total_splits < b.total_splits ? -1 : 1;
    return 0;
}

bool decode_only(const std::vector<Seq>& seqs, const Params& p) {
    for (const Seq& s : seqs)
        if (s.q_len > p.decode_qlen_max) return false;
    return true;
}
}  // namespace

std::vector<int> split_tiles(int tiles, int n) {
    std::vector<int> out(n);
    int base = tiles / n, extra = tiles % n;
    for (int r = 0; r < n; ++r) out[r] = base + (r < extra ? 1 : 0);
    return out;
}

std::vector<QTask> attention_queue(const std::vector<Seq>& seqs, const std::vector<int>& splits,
                                   const Params& p) {
    std::vector<QTask> tasks;
    bool any_split = false;
    for (size_t b = 0; b < seqs.size(); ++b) {
        if (splits[b] > 1) any_split = true;
        std::vector<int> parts = split_tiles(seqs[b].tiles, splits[b]);
        for (int r = 0; r < splits[b]; ++r)
            for (int t = 0; t < seqs[b].tasks_per_split; ++t)
                tasks.push_back({parts[r] + p.delta_attn, (int)b, r, t});
    }
    if (decode_only(seqs, p) && any_split) {
        std::stable_sort(tasks.begin(), tasks.end(),
                         [](const QTask& x, const QTask& y) { return x.work > y.work; });
        return tasks;
    }
    std::vector<QTask> out;
    out.reserve(tasks.size());
    for (const QTask& t : tasks)
        if (seqs[t.seq].q_len > p.decode_qlen_max) out.push_back(t);
    for (const QTask& t : tasks)
        if (seqs[t.seq].q_len <= p.decode_qlen_max) out.push_back(t);
    return out;
}

int run_length(const std::vector<Seq>& seqs, const Params& p) {
    int hq = p.q_heads;
    std::vector<int> cands = {1, hq, 2 * hq, 4 * hq, std::min(8 * hq, 32)};
    std::sort(cands.begin(), cands.end(), std::greater<int>());
    cands.erase(std::unique(cands.begin(), cands.end()), cands.end());
    double need = 0.8 * p.warps_per_cta * (double)p.num_ctas;
    for (int R : cands) {
        long long n = 0;
        for (const Seq& s : seqs) n += (s.vectors + R - 1) / R;
        if ((double)n >= need) return R;
    }
    return 1;
}

namespace {

// A run of attention tasks with the same work from one sequence: the queue in group form.
// Each sequence cuts its history into `extra` parts of base+1 tiles and then parts of base
// tiles, so it contributes at most two groups; expanding the groups in order gives the
// task order of attention_queue() (a stable sort of groups by work is a stable sort of
// their tasks, since every group is a contiguous range of the unsorted queue).
struct Group {
    double work;
    int seq;
    long long count;
};

// Min-heap on (key, id) with a payload; ids are unique among the entries.  Four-ary,
// with the keys, ids and payloads in separate arrays and the smallest child picked
// without branches: the search's cost is mostly these heaps.
struct Heap {
    std::vector<double> key;
    std::vector<int> id, val;
    static bool less(double ka, int ia, double kb, int ib) { return (ka < kb) | ((ka == kb) & (ia < ib)); }
    void clear() {
        key.clear();
        id.clear();
        val.clear();
    }
    void reserve(size_t n) {
        key.reserve(n);
        id.reserve(n);
        val.reserve(n);
    }
    bool empty() const { return key.empty(); }
    size_t size() const { return key.size(); }
    double top_key() const { return key[0]; }
    int top_id() const { return id[0]; }
    int top_val() const { return val[0]; }
    void push(double k, int i, int v) {
        size_t pos = key.size();
        key.push_back(k);
        id.push_back(i);
        val.push_back(v);
        while (pos > 0) {
            size_t par = (pos - 1) / 4;
            if (!less(k, i, key[par], id[par])) break;
            key[pos] = key[par];
            id[pos] = id[par];
            val[pos] = val[par];
            pos = par;
        }
        key[pos] = k;
        id[pos] = i;
        val[pos] = v;
    }
    size_t min_child(size_t c, size_t n) const {
        if (c + 3 < n) {
            const size_t a = less(key[c + 1], id[c + 1], key[c], id[c]) ? c + 1 : c;
            const size_t b = less(key[c + 3], id[c + 3], key[c + 2], id[c + 2]) ? c + 3 : c + 2;
            return less(key[b], id[b], key[a], id[a]) ? b : a;
        }
        size_t m = c;
        for (size_t j = c + 1; j < n; ++j)
            if (less(key[j], id[j], key[m], id[m])) m = j;
        return m;
    }
    void sift_down(size_t pos, double k, int i, int v) {
        const size_t n = key.size();
        while (true) {
            const size_t c = 4 * pos + 1;
            if (c >= n) break;
            const size_t m = min_child(c, n);
            if (!less(key[m], id[m], k, i)) break;
            key[pos] = key[m];
            id[pos] = id[m];
            val[pos] = val[m];
            pos = m;
        }
        key[pos] = k;
        id[pos] = i;
        val[pos] = v;
    }
    void pop() {
        const size_t last = key.size() - 1;
        const double k = key[last];
        const int i = id[last], v = val[last];
        key.pop_back();
        id.pop_back();
        val.pop_back();
        if (last > 0) sift_down(0, k, i, v);
    }
};

// State of the attention phase between two task assignments.
struct AttnState {
    Heap running;                       // (finish clock, sequence) -> CTAs
    std::vector<double> seq_attn_end;
    long long n_running = 0, freed = 0, n_tasks = 0;
    double t = 0.0, clock = 0.0;
};

// The attention states of one plan at the start of every kSnapEvery-th queue group.  A plan that
// adds splits to some sequences keeps the groups ahead of their first group (LPT order is
// by work, and added splits only shrink a sequence's tasks; FIFO order is by sequence),
// so its simulation can start from the recorded state there.
constexpr size_t kSnapEvery = 8;
struct Trace {
    bool lpt = false;
    std::vector<AttnState> snaps;
    std::vector<int> first_group;       // per sequence: index of its first group
};

// One evaluator of the critical-wave model with its scratch memory (one per host thread).
class Simulator {
public:
    Simulator(const std::vector<Seq>& seqs, const Params& p)
        : seqs_(seqs), p_(p), R_(run_length(seqs, p)), decode_only_(decode_only(seqs, p)) {}

    // The model's times depend on which CTA or warp takes a task only through the multiset
    // of their free times: CTAs freed at one event start their next tasks at the same
    // clock, and warps with equal free times are interchangeable.  So the running set holds
    // one entry per (finish clock, sequence) with a count of CTAs, and the warp pool one
    // entry per free time with a count of warps; the times are those of the one-by-one
    // schedule (lowest CTA or warp index first), computed with the same operations.
    //
    // rec: record the attention state at the start of every queue group.  from/r: the
    // plan's first r groups are those of the recorded plan (same queue order), so the
    // attention phase resumes from the state recorded at group r.
    SimResult run(const std::vector<int>& splits, double prune_at, Trace* rec = nullptr,
                  const Trace* from = nullptr, size_t r = 0) {
        const int K = p_.num_ctas;
        const int nseq = (int)seqs_.size();
        const bool lpt = build_queue(splits);
        SimResult res;
        AttnState& s = st_;
        size_t gi = 0;
        const size_t r0 = r - r % kSnapEvery;      // last recorded group at or before r
        if (from && from->lpt == lpt && r0 > 0 && r0 < groups_.size() && r0 / kSnapEvery < from->snaps.size()) {
            s = from->snaps[r0 / kSnapEvery];
            gi = r0;
        } else {
            // All running tasks advance at the same rate, so they finish in the order of
            // (work clock at start + work): a min-heap over that "finish clock".  The work
            // clock counts tile-equivalents done by any one running task since time 0.
            s.running.clear();
            s.seq_attn_end.assign(nseq, 0.0);
            s.n_running = 0;
            s.freed = K;
            s.n_tasks = 0;
            s.t = 0.0;
            s.clock = 0.0;
        }
        if (rec) {
            rec->lpt = lpt;
            rec->snaps.resize((groups_.size() + kSnapEvery - 1) / kSnapEvery);
            rec->first_group.assign(nseq, -1);
            for (size_t g = 0; g < groups_.size(); ++g)
                if (rec->first_group[groups_[g].seq] < 0) rec->first_group[groups_[g].seq] = (int)g;
        }
        releases_.clear();
        long long left_in_group = gi < groups_.size() ? groups_[gi].count : 0;
        while (true) {
            while (s.freed > 0) {
                while (gi < groups_.size() && left_in_group == 0) {
                    ++gi;
                    left_in_group = gi < groups_.size() ? groups_[gi].count : 0;
                }
                if (gi >= groups_.size()) {
                    if (!releases_.empty() && releases_.back().first == s.t) releases_.back().second += s.freed;
                    else releases_.push_back({s.t, s.freed});
                    break;
                }
                if (rec && gi % kSnapEvery == 0 && left_in_group == groups_[gi].count)
                    rec->snaps[gi / kSnapEvery] = s;
                const long long g = std::min(s.freed, left_in_group);
                s.running.push(s.clock + groups_[gi].work, groups_[gi].seq, (int)g);
                s.n_running += g;
                left_in_group -= g;
                s.freed -= g;
                s.n_tasks += g;
            }
            s.freed = 0;
            if (s.running.empty()) break;
            const double tau = std::max(p_.rho, (double)s.n_running / (double)K);
            const double step = s.running.top_key() - s.clock;
            s.t = s.t + step * tau;
            s.clock = s.running.top_key();
            while (!s.running.empty() && s.running.top_key() - s.clock <= kEps * std::max(1.0, step)) {
                const int b = s.running.top_id();
                s.seq_attn_end[b] = std::max(s.seq_attn_end[b], s.t);
                s.freed += s.running.top_val();
                s.n_running -= s.running.top_val();
                s.running.pop();
            }
        }
        res.seq_attn_end = s.seq_attn_end;
        const long long n_tasks = s.n_tasks;
        double attn_end = 0.0;
        for (double e : res.seq_attn_end) attn_end = std::max(attn_end, e);
        res.n_attn_tasks = (int)n_tasks;
        int tot = 0;
        for (int s : splits) tot += s;
        res.total_splits = tot;
        res.attn_end = attn_end;
        // lower bound of the score without simulating the reductions: every reduction item
        // of a sequence starts no earlier than its attention end
        double lb = attn_end;
        for (int b = 0; b < nseq; ++b)
            if (seqs_[b].vectors > 0)
                lb = std::max(lb, res.seq_attn_end[b] + p_.delta_red +
                                      p_.gamma * std::min(R_, seqs_[b].vectors) * splits[b]);
        res.lower_bound = lb;
        if (prune_at < 1e300 && lb >= prune_at) {
            res.score = lb;
            res.pruned = true;
            return res;
        }
        res.score = std::max(attn_end, reductions(splits, res.seq_attn_end));
        return res;
    }

private:
    // Reductions in sequence order, each on a warp that frees first; every CTA's warps are
    // free from its release time.  Returns the latest reduction end.
    double reductions(const std::vector<int>& splits, const std::vector<double>& ready) {
        const long long W = p_.warps_per_cta;
        pool_.clear();
        for (const auto& r : releases_) pool_.push_back({r.first, r.second * W});
        size_t lo = 0;
        double red_end = 0.0;
        for (size_t b = 0; b < seqs_.size(); ++b) {
            const int vec = seqs_[b].vectors;
            if (vec <= 0) continue;
            const double a = ready[b];
            // runs of items with the same cost: vec / R full items, then the remainder
            const long long full = vec / R_;
            const int rest = vec % R_;
            for (int part = 0; part < 2; ++part) {
                long long m = part == 0 ? full : (rest > 0 ? 1 : 0);
                const int v = part == 0 ? R_ : rest;
                if (m == 0) continue;
                const double cost = p_.delta_red + p_.gamma * v * splits[b];
                if (!(cost >= 0.0)) return reductions_one_by_one(splits, ready);
                while (m > 0) {
                    const double k = pool_[lo].first;
                    const double end = std::max(k, a) + cost;
                    red_end = std::max(red_end, end);
                    if (end == k) break;          // the first free warp takes every item, unchanged
                    const long long q = std::min(m, pool_[lo].second);
                    m -= q;
                    pool_[lo].second -= q;
                    if (pool_[lo].second == 0) ++lo;
                    // end > k: the moved warps sort after the one just taken
                    auto it = std::lower_bound(pool_.begin() + lo, pool_.end(), end,
                                               [](const std::pair<double, long long>& e, double x) { return e.first < x; });
                    if (it != pool_.end() && it->first == end) {
                        it->second += q;
                    } else if (it == pool_.begin() + lo && lo > 0) {
                        pool_[--lo] = {end, q};
                    } else {
                        pool_.insert(it, {end, q});
                    }
                }
            }
        }
        return red_end;
    }

    // the same schedule item by item on a heap of warp free times (any cost sign)
    double reductions_one_by_one(const std::vector<int>& splits, const std::vector<double>& ready) {
        std::vector<double> h;
        for (const auto& r : releases_)
            for (long long i = 0; i < r.second * p_.warps_per_cta; ++i) h.push_back(r.first);
        std::make_heap(h.begin(), h.end(), std::greater<double>());
        double red_end = 0.0;
        for (size_t b = 0; b < seqs_.size(); ++b) {
            int left = seqs_[b].vectors;
            while (left > 0) {
                int v = std::min(R_, left);
                double cost = p_.delta_red + p_.gamma * v * splits[b];
                std::pop_heap(h.begin(), h.end(), std::greater<double>());
                double end = std::max(h.back(), ready[b]) + cost;
                red_end = std::max(red_end, end);
                h.back() = end;
                std::push_heap(h.begin(), h.end(), std::greater<double>());
                left -= v;
            }
        }
        return red_end;
    }

    // the model queue in group form; true when it is in LPT order
    bool build_queue(const std::vector<int>& splits) {
        groups_.clear();
        bool any_split = false;
        for (size_t b = 0; b < seqs_.size(); ++b) {
            const int s = splits[b], tiles = seqs_[b].tiles, tps = seqs_[b].tasks_per_split;
            if (s > 1) any_split = true;
            const int base = tiles / s, extra = tiles % s;
            if (extra > 0) groups_.push_back({(base + 1) + p_.delta_attn, (int)b, (long long)extra * tps});
            if (s - extra > 0) groups_.push_back({base + p_.delta_attn, (int)b, (long long)(s - extra) * tps});
        }
        if (decode_only_ && any_split) {
            std::stable_sort(groups_.begin(), groups_.end(),
                             [](const Group& x, const Group& y) { return x.work > y.work; });
            return true;
        }
        const int qmax = p_.decode_qlen_max;
        std::stable_partition(groups_.begin(), groups_.end(),
                              [&](const Group& g) { return seqs_[g.seq].q_len > qmax; });
        return false;
    }

    const std::vector<Seq>& seqs_;
    const Params& p_;
    const int R_;
    const bool decode_only_;
    std::vector<Group> groups_;
    std::vector<std::pair<double, long long>> releases_, pool_;   // (time, CTAs) / (time, warps)
    AttnState st_;
};

// Host threads for one plan: run(n, f) calls f(i, worker) for i in [0, n) across the
// workers (the calling thread is worker 0) and returns when all calls are done.  A search
// dispatches a batch every few tens of microseconds, so idle workers spin (yielding) on a
// generation counter for the pool's short life instead of sleeping on a condition.
class Pool {
public:
    explicit Pool(int workers) : n_(std::max(1, workers)) {
        for (int w = 1; w < n_; ++w) threads_.emplace_back([this]() { loop(); });
    }
    ~Pool() {
        stop_.store(true, std::memory_order_release);
        gen_.fetch_add(1, std::memory_order_acq_rel);
        for (std::thread& th : threads_) th.join();
    }
    int workers() const { return n_; }
    void run(size_t count, const std::function<void(size_t, int)>& f) {
        if (n_ == 1 || count < 2) {
            for (size_t i = 0; i < count; ++i) f(i, 0);
            return;
        }
        job_ = &f;
        count_ = count;
        next_.store(0, std::memory_order_relaxed);
        slot_.store(1, std::memory_order_relaxed);
        busy_.store(n_ - 1, std::memory_order_relaxed);
        gen_.fetch_add(1, std::memory_order_acq_rel);
        work(0);
        while (busy_.load(std::memory_order_acquire) != 0) std::this_thread::yield();
    }

private:
    void work(int w) {
        for (size_t i = next_.fetch_add(1, std::memory_order_relaxed); i < count_;
             i = next_.fetch_add(1, std::memory_order_relaxed))
            (*job_)(i, w);
    }
    void loop() {
        uint64_t seen = 0;
        while (true) {
            uint64_t g;
            while ((g = gen_.load(std::memory_order_acquire)) == seen) std::this_thread::yield();
            seen = g;
            if (stop_.load(std::memory_order_acquire)) return;
            // each batch hands every worker a distinct index for its scratch memory
            const int w = slot_.fetch_add(1, std::memory_order_relaxed);
            work(w);
            busy_.fetch_sub(1, std::memory_order_acq_rel);
        }
    }
    const int n_;
    std::vector<std::thread> threads_;
    std::atomic<uint64_t> gen_{0};
    std::atomic<bool> stop_{false};
    std::atomic<int> slot_{1}, busy_{0};
    const std::function<void(size_t, int)>* job_ = nullptr;
    size_t count_ = 0;
    std::atomic<size_t> next_{0};
};

// host threads worth starting for a search over `n` sequences
int pool_size(size_t n) {
    if (n < 8) return 1;
    const int hw = (int)std::max(1u, std::thread::hardware_concurrency());
    return std::min({hw, 16, (int)n});
}

// Evaluates candidate split vectors on the pool's threads, one Simulator per thread.
class Evaluator {
public:
    Evaluator(const std::vector<Seq>& seqs, const Params& p) : seqs_(seqs), p_(p), pool_(pool_size(seqs.size())) {
        for (int w = 0; w < pool_.workers(); ++w) sims_.emplace_back(new Simulator(seqs, p));
    }
    ~Evaluator() {
        for (Simulator* s : sims_) delete s;
    }
    SimResult one(const std::vector<int>& splits, double prune_at = 1e300, Trace* rec = nullptr) {
        return sims_[0]->run(splits, prune_at, rec);
    }
    // from/starts: candidate i resumes from the recorded state at group starts[i]
    std::vector<SimResult> many(const std::vector<std::vector<int>>& cands, double prune_at,
                                const Trace* from = nullptr, const std::vector<size_t>* starts = nullptr) {
        std::vector<SimResult> res(cands.size());
        pool_.run(cands.size(), [&](size_t i, int w) {
            res[i] = sims_[w]->run(cands[i], prune_at, nullptr, from, starts ? (*starts)[i] : 0);
        });
        return res;
    }

private:
    const std::vector<Seq>& seqs_;
    const Params& p_;
    Pool pool_;
    std::vector<Simulator*> sims_;
};

PlanResult plan_impl(Evaluator& ev, const std::vector<Seq>& seqs, const Params& p, int min_splits,
                     int max_splits) {
    const int n = (int)seqs.size();
    PlanResult out;
    std::vector<int> base(n), cap(n), ref(n), lim(n);
    long long work = 0;
    for (int b = 0; b < n; ++b) {
        base[b] = std::max(1, std::min(min_splits, seqs[b].tiles));
        cap[b] = std::max(base[b], std::min(max_splits, seqs[b].tiles));
        work += (long long)seqs[b].tiles * seqs[b].tasks_per_split;
    }
    // reference plan: work-balanced, T = ceil(work / K) tiles per task
    long long target = std::max(1LL, (work + p.num_ctas - 1) / p.num_ctas);
    for (int b = 0; b < n; ++b) {
        long long want = (seqs[b].tiles + target - 1) / target;
        ref[b] = (int)std::min<long long>(cap[b], std::max<long long>(base[b], want));
        int l = ref[b];
        if (seqs[b].q_len <= p.decode_qlen_max && seqs[b].tiles >= p.num_ctas) l = std::max(l, 4);
        lim[b] = std::max(base[b], std::min(l, cap[b]));
    }
    std::vector<int> cur = base;
    Trace trace;
    const SimResult base_r = ev.one(base, 1e300, &trace);
    SimResult cur_r = base_r;
    while (true) {
        std::vector<std::vector<int>> cands;
        std::vector<size_t> starts;      // first queue group a candidate changes
        for (int b = 0; b < n; ++b) {
            if (cur[b] < lim[b]) {
                std::vector<int> c = cur;
                c[b] += 1;
                cands.push_back(c);
                starts.push_back((size_t)trace.first_group[b]);
            }
        }
        std::vector<int> tail;
        for (int b = 0; b < n; ++b)
            if (cur[b] < lim[b] && feq(cur_r.seq_attn_end[b], cur_r.attn_end)) tail.push_back(b);
        if (tail.size() > 1) {
            std::vector<int> c = cur;
            size_t st = (size_t)-1;
            for (int b : tail) {
                c[b] += 1;
                st = std::min(st, (size_t)trace.first_group[b]);
            }
            cands.push_back(c);
            starts.push_back(st);
        }
        if (cands.empty()) break;
        // Candidates are independent simulations, evaluated on the host's cores; the best
        // is then picked in candidate order (the result of a serial loop).  Only a score
        // strictly below the current one (outside the tolerance) is accepted, so a
        // candidate whose attention phase already ends there cannot be: its reductions
        // are not simulated.
        const double prune_at = cur_r.score - kEps * std::max(1.0, std::fabs(cur_r.score));
        std::vector<SimResult> res = ev.many(cands, prune_at, &trace, &starts);
        int best = -1;
        for (size_t i = 0; i < cands.size(); ++i) {
            if (res[i].pruned) continue;
            if (best < 0 || cmp_result(res[i], res[best]) < 0) best = (int)i;
        }
        if (best < 0) break;
        if (res[best].score < cur_r.score && !feq(res[best].score, cur_r.score)) {
            cur = cands[best];
            cur_r = res[best];
            ev.one(cur, 1e300, &trace);
        } else {
            break;
        }
    }
    SimResult ref_r = ev.one(ref);
    std::vector<int> fin = base;
    SimResult fin_r = base_r;
    if (cmp_result(cur_r, fin_r) < 0) { fin = cur; fin_r = cur_r; }
    if (cmp_result(ref_r, fin_r) < 0) { fin = ref; fin_r = ref_r; }
    if (fin != base && fin_r.score > (1.0 - p.adopt_margin) * base_r.score + kEps) {
        fin = base;
        fin_r = base_r;
    }
    out.splits = fin;
    out.base = base;
    out.search = cur;
    out.reference = ref;
    out.limits = lim;
    out.score = fin_r.score;
    out.base_score = base_r.score;
    out.search_score = cur_r.score;
    out.reference_score = ref_r.score;
    return out;
}

}  // namespace

SimResult simulate(const std::vector<Seq>& seqs, const std::vector<int>& splits, const Params& p,
                   double prune_at) {
    Simulator sim(seqs, p);
    return sim.run(splits, prune_at);
}

PlanResult plan(const std::vector<Seq>& seqs, const Params& p, int min_splits, int max_splits) {
    Evaluator ev(seqs, p);
    return plan_impl(ev, seqs, p, min_splits, max_splits);
}

PlanResult plan_with_uniform(const std::vector<Seq>& seqs, const Params& p, int min_splits, int max_splits) {
    Evaluator ev(seqs, p);
    PlanResult out = plan_impl(ev, seqs, p, min_splits, max_splits);
    const int n = (int)seqs.size();
    SimResult fin_r = ev.one(out.splits);
    int max_cap = 1;
    for (int b = 0; b < n; ++b) max_cap = std::max(max_cap, std::max(1, std::min(max_splits, seqs[b].tiles)));
    std::vector<std::vector<int>> cands;
    for (int u : {2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64}) {
        if (u > max_cap) break;
        std::vector<int> c(n);
        for (int b = 0; b < n; ++b) {
            const int lo = std::max(1, std::min(min_splits, seqs[b].tiles));
            const int hi = std::max(lo, std::min(max_splits, seqs[b].tiles));
            c[b] = std::min(hi, std::max(lo, u));
        }
        if (c != out.splits) cands.push_back(c);
    }
    // evaluated together, selected in order: a candidate whose attention-phase bound is
    // not below the incumbent's score cannot win
    std::vector<SimResult> res = ev.many(cands, fin_r.score);
    for (size_t i = 0; i < cands.size(); ++i) {
        const SimResult& r = res[i];
        if (r.pruned || r.lower_bound >= fin_r.score) continue;
        // same adoption rule as the pages' selection: a split plan only if >= adopt_margin
        // below NoSplit
        // a candidate replaces the incumbent only with a strictly lower score (so the
        // attention-phase bound above prunes exactly)
        if (r.score < fin_r.score && !feq(r.score, fin_r.score) &&
            r.score <= (1.0 - p.adopt_margin) * out.base_score + kEps) {
            out.splits = cands[i];
            out.score = r.score;
            fin_r = r;
        }
    }
    return out;
}

}  // namespace model
}  // namespace skv
