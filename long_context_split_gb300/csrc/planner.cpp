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
#include <thread>
#include <functional>
#include <queue>
#include <tuple>

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

SimResult simulate(const std::vector<Seq>& seqs, const std::vector<int>& splits, const Params& p,
                   double prune_at) {
    const int K = p.num_ctas;
    std::vector<QTask> queue = attention_queue(seqs, splits, p);
    const int nseq = (int)seqs.size();
    SimResult res;
    res.seq_attn_end.assign(nseq, 0.0);
    std::vector<double> release(K, -1.0);
    // All running tasks advance at the same rate, so they finish in the order of
    // (work clock at start + work): a min-heap over that "finish clock" replaces a
    // scan of every CTA per event.  The work clock counts tile-equivalents done by
    // any one running task since time 0.
    typedef std::tuple<double, int, int> Run;   // (finish clock, cta, seq)
    std::priority_queue<Run, std::vector<Run>, std::greater<Run>> running;
    std::vector<int> free_now(K);
    for (int c = 0; c < K; ++c) free_now[c] = c;
    double t = 0.0, clock = 0.0;
    size_t nxt = 0;
    while (true) {
        std::sort(free_now.begin(), free_now.end());
        for (int c : free_now) {
            if (nxt < queue.size()) {
                running.push(Run(clock + queue[nxt].work, c, queue[nxt].seq));
                ++nxt;
            } else if (release[c] < 0.0) {
                release[c] = t;
            }
        }
        free_now.clear();
        if (running.empty()) break;
        const double tau = std::max(p.rho, (double)running.size() / (double)K);
        const double step = std::get<0>(running.top()) - clock;
        t = t + step * tau;
        clock = std::get<0>(running.top());
        while (!running.empty() && std::get<0>(running.top()) - clock <= kEps * std::max(1.0, step)) {
            const int b = std::get<2>(running.top());
            res.seq_attn_end[b] = std::max(res.seq_attn_end[b], t);
            free_now.push_back(std::get<1>(running.top()));
            running.pop();
        }
    }
    for (int c = 0; c < K; ++c)
        if (release[c] < 0.0) release[c] = t;
    double attn_end = 0.0;
    for (double e : res.seq_attn_end) attn_end = std::max(attn_end, e);
    res.n_attn_tasks = (int)queue.size();
    int tot = 0;
    for (int s : splits) tot += s;
    res.total_splits = tot;
    if (prune_at < 1e300) {
        // lower bound of the score without simulating the reductions: every reduction item
        // of a sequence starts no earlier than its attention end
        const int R0 = run_length(seqs, p);
        double lb = attn_end;
        for (int b = 0; b < nseq; ++b)
            if (seqs[b].vectors > 0)
                lb = std::max(lb, res.seq_attn_end[b] + p.delta_red +
                                      p.gamma * std::min(R0, seqs[b].vectors) * splits[b]);
        if (lb >= prune_at) {
            res.attn_end = attn_end;
            res.score = lb;
            res.pruned = true;
            return res;
        }
    }

    // reductions, in sequence order, on released warps (min-heap of (free time, cta, warp))
    const int R = run_length(seqs, p);
    typedef std::tuple<double, int, int> Warp;
    std::priority_queue<Warp, std::vector<Warp>, std::greater<Warp>> warps;
    for (int c = 0; c < K; ++c)
        for (int w = 0; w < p.warps_per_cta; ++w) warps.push(Warp(release[c], c, w));
    double red_end = 0.0;
    for (int b = 0; b < nseq; ++b) {
        int left = seqs[b].vectors;
        while (left > 0) {
            int v = std::min(R, left);
            double cost = p.delta_red + p.gamma * v * splits[b];
            Warp w = warps.top();
            warps.pop();
            double start = std::max(std::get<0>(w), res.seq_attn_end[b]);
            double end = start + cost;
            red_end = std::max(red_end, end);
            warps.push(Warp(end, std::get<1>(w), std::get<2>(w)));
            left -= v;
        }
    }
    res.attn_end = attn_end;
    res.score = std::max(attn_end, red_end);
    return res;
}

PlanResult plan(const std::vector<Seq>& seqs, const Params& p, int min_splits, int max_splits) {
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
    SimResult cur_r = simulate(seqs, cur, p);
    while (true) {
        std::vector<std::vector<int>> cands;
        for (int b = 0; b < n; ++b) {
            if (cur[b] < lim[b]) {
                std::vector<int> c = cur;
                c[b] += 1;
                cands.push_back(c);
            }
        }
        std::vector<int> tail;
        for (int b = 0; b < n; ++b)
            if (cur[b] < lim[b] && feq(cur_r.seq_attn_end[b], cur_r.attn_end)) tail.push_back(b);
        if (tail.size() > 1) {
            std::vector<int> c = cur;
            for (int b : tail) c[b] += 1;
            cands.push_back(c);
        }
        if (cands.empty()) break;
        // Candidates are independent simulations: evaluate them on the host's cores, then
        // pick the best in candidate order (same result as a serial loop).  Only a score
        // strictly below the current one (outside the tolerance) is accepted, so a
        // candidate whose attention phase already ends there cannot be: its reductions
        // are not simulated.
        const double prune_at = cur_r.score - kEps * std::max(1.0, std::fabs(cur_r.score));
        std::vector<SimResult> res(cands.size());
        const int nthreads = (int)std::min<size_t>(cands.size(), std::max(1u, std::thread::hardware_concurrency()));
        if (nthreads <= 1 || cands.size() < 4) {
            for (size_t i = 0; i < cands.size(); ++i) res[i] = simulate(seqs, cands[i], p, prune_at);
        } else {
            std::atomic<size_t> next(0);
            std::vector<std::thread> pool;
            for (int w = 0; w < nthreads; ++w)
                pool.emplace_back([&]() {
                    for (size_t i = next.fetch_add(1); i < cands.size(); i = next.fetch_add(1))
                        res[i] = simulate(seqs, cands[i], p, prune_at);
                });
            for (std::thread& th : pool) th.join();
        }
        int best = -1;
        SimResult best_r;
        for (size_t i = 0; i < cands.size(); ++i) {
            if (res[i].pruned) continue;
            if (best < 0 || cmp_result(res[i], best_r) < 0) {
                best = (int)i;
                best_r = res[i];
            }
        }
        if (best < 0) break;
        if (best_r.score < cur_r.score && !feq(best_r.score, cur_r.score)) {
            cur = cands[best];
            cur_r = best_r;
        } else {
            break;
        }
    }
    SimResult base_r = simulate(seqs, base, p);
    SimResult ref_r = simulate(seqs, ref, p);
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

PlanResult plan_with_uniform(const std::vector<Seq>& seqs, const Params& p, int min_splits, int max_splits) {
    PlanResult out = plan(seqs, p, min_splits, max_splits);
    const int n = (int)seqs.size();
    SimResult fin_r = simulate(seqs, out.splits, p);
    int max_cap = 1;
    for (int b = 0; b < n; ++b) max_cap = std::max(max_cap, std::max(1, std::min(max_splits, seqs[b].tiles)));
    for (int u : {2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64}) {
        if (u > max_cap) break;
        std::vector<int> c(n);
        for (int b = 0; b < n; ++b) {
            const int lo = std::max(1, std::min(min_splits, seqs[b].tiles));
            const int hi = std::max(lo, std::min(max_splits, seqs[b].tiles));
            c[b] = std::min(hi, std::max(lo, u));
        }
        if (c == out.splits) continue;
        SimResult r = simulate(seqs, c, p, fin_r.score);
        if (r.pruned) continue;
        // same adoption rule as the pages' selection: a split plan only if >= adopt_margin
        // below NoSplit
        if (cmp_result(r, fin_r) < 0 && r.score <= (1.0 - p.adopt_margin) * out.base_score + kEps) {
            out.splits = c;
            out.score = r.score;
            fin_r = r;
        }
    }
    return out;
}

}  // namespace model
}  // namespace skv
