// Critical-wave split planner (host).  LiquidCP Section 5.2 (Eqs. 5-6,
// "Plan selection", "Task ordering") and Appendix A.2 ("Split planning").
#pragma once

#include <cstdint>
#include <vector>

namespace skv {
namespace model {

struct Params {
    int num_ctas = 152;        // K
    int warps_per_cta = 12;
    int q_heads = 1;           // h_q of the reduction run-length rule
    int decode_qlen_max = 16;
    double rho = 0.43;
    double delta_attn = 32.0;
    double delta_red = 2.5;
    double gamma = 0.47;
    double adopt_margin = 0.10;
};

struct Seq {
    int tiles = 1;             // KV tiles of the history
    int tasks_per_split = 1;   // attention tasks per split
    int vectors = 1;           // output vectors (query token x head)
    int q_len = 1;
};

// One attention task of the model queue.
struct QTask {
    double work;               // c_attn = n_t + delta_attn
    int seq;
    int split;
    int sub;                   // index among the split's tasks_per_split tasks
};

struct SimResult {
    double score = 0.0;
    double attn_end = 0.0;
    std::vector<double> seq_attn_end;
    int n_attn_tasks = 0;
    int total_splits = 0;
    bool pruned = false;       // reductions not simulated: score is only a lower bound (attn_end)
    double lower_bound = 0.0;  // score bound from the attention phase alone (<= score)
};

struct PlanResult {
    std::vector<int> splits;
    std::vector<int> base, search, reference, limits;
    double score = 0.0, base_score = 0.0, search_score = 0.0, reference_score = 0.0;
};

// floor/remainder cut of `tiles` into n parts (first parts one larger)
std::vector<int> split_tiles(int tiles, int n);
// attention tasks in queue order: LPT for decode-only plans with a split,
// otherwise FIFO with chunk requests first
std::vector<QTask> attention_queue(const std::vector<Seq>& seqs, const std::vector<int>& splits,
                                   const Params& p);
int run_length(const std::vector<Seq>& seqs, const Params& p);
// prune_at: when the attention phase alone ends at or after it, the reductions are not
// simulated (the result is marked pruned; its score can only be higher)
SimResult simulate(const std::vector<Seq>& seqs, const std::vector<int>& splits, const Params& p,
                   double prune_at = 1e300);
// the pages' search and selection (NoSplit / search / reference)
PlanResult plan(const std::vector<Seq>& seqs, const Params& p, int min_splits, int max_splits);
// plan() whose final selection also scores uniform plans (u splits per request within
// the bounds): on plateaus of the model, where no single added split lowers the
// score, the one-split-at-a-time search stops early
PlanResult plan_with_uniform(const std::vector<Seq>& seqs, const Params& p, int min_splits, int max_splits);

}  // namespace model
}  // namespace skv
