"""Critical-wave split planner, written as the oracle for the product planner.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  Pure Python, event by
event, for small batches.  Follows LiquidCP Section 5.2 ("Critical-wave KV
Splitting": Eqs. 5 and 6, "Plan selection", "Task ordering") and Appendix A.2
("Split planning", "Release-aware ordering").

Model (LiquidCP Section 5.2):
  * One time unit is the per-CTA time to process one history KV tile with all
    K compute CTAs running attention.  With k CTAs running attention, a task
    advances at rate 1/tau(k), tau(k) = max(rho, k/K)            (Eq. 5)
  * An attention task over n_t tiles carries c_attn = n_t + delta_attn.
  * Attention tasks are dispatched in queue order, each to the first
    available compute CTA (lowest index among the CTAs free at that time).
  * A CTA releases its warps to history reduction after completing its last
    attention task, i.e. when it is free and no attention task is left.
  * A history reduction u costs c_red = delta_red + gamma * v_u * s_u
    (Eq. 6), independent of load; it uses one warp and starts, in queue
    order, when its warp and its inputs (every attention task of its
    sequence) are available.
  * The score is the latest completion over attention and reduction tasks.

Plan search (LiquidCP Section 5.2 "Plan selection", Appendix A.2):
  start from NoSplit; each iteration tries +1 split on each sequence below
  its limit and a joint +1 on the sequences whose tasks tie at the attention
  tail; the best candidate is accepted only if it lowers the score; ties
  favour earlier attention completion, then fewer attention tasks, then
  fewer total splits.  The final plan is the best of NoSplit, the search
  result and the reference plan, and a split plan is adopted only if its
  score is at least 10% below NoSplit's.  Decode requests (at most 16 query
  tokens) with at least K tiles get a limit of at least four.

Readings where the pages are silent (each listed in the design notes):
  * Reference plan: the FA3 heuristic is not on the pages, so the reference
    is work-balanced: with T = ceil(sum_b tiles_b * tasks_b / K) tiles per
    task, sequence b gets clamp(ceil(tiles_b / T), 1, limit).
  * Splits are contiguous with floor/remainder sizes (Figure 8: 176 -> 59/59/58).
  * Reduction tasks cover runs of R output vectors, R the largest of
    {1, h_q, 2h_q, 4h_q, min(8h_q, 32)} leaving at least 0.8 * warps tasks
    (Appendix A.2, stated there for unsplit sequences; used here for all).
  * Queue order: LPT (stable, decreasing c_attn) for decode-only plans with
    any split; otherwise FIFO with chunk requests (more than 16 query tokens)
    first, then the rest, each in request order.
  * A minimum split count (the million-token configuration asks for 16-64
    splits) replaces NoSplit as the search start and the adoption baseline.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

EPS = 1e-9


@dataclasses.dataclass
class ModelParams:
    num_ctas: int                 # K
    rho: float = 0.43             # per-tile time floor           (Table 2)
    delta_attn: float = 32.0      # per attention task overhead   (Table 2)
    delta_red: float = 2.5        # per reduction task overhead   (Table 2)
    gamma: float = 0.47           # cost per merged partial vector (Table 2)
    warps_per_cta: int = 12       # reduction warps per CTA (384-thread CTAs)
    adopt_margin: float = 0.10
    decode_qlen_max: int = 16


@dataclasses.dataclass
class SeqSpec:
    tiles: int                    # KV tiles of the history
    tasks_per_split: int = 1      # attention tasks per split (KV heads x query tiles)
    vectors: int = 1              # output vectors (query token x head pairs)
    q_len: int = 1                # query tokens


def split_tiles(tiles: int, n: int) -> List[int]:
    base, extra = divmod(tiles, n)
    return [base + (1 if r < extra else 0) for r in range(n)]


def _feq(a: float, b: float) -> bool:
    return abs(a - b) <= EPS * max(1.0, abs(a), abs(b))


def _cmp_key(a: Tuple, b: Tuple) -> int:
    for x, y in zip(a, b):
        if isinstance(x, float) or isinstance(y, float):
            if _feq(x, y):
                continue
        elif x == y:
            continue
        return -1 if x < y else 1
    return 0


def run_length(seqs: Sequence[SeqSpec], q_heads: int, p: ModelParams) -> int:
    """Appendix A.2: largest run in {1, h_q, 2h_q, 4h_q, min(8h_q, 32)} leaving
    at least 0.8 x (warps) reduction tasks."""
    cands = sorted({1, q_heads, 2 * q_heads, 4 * q_heads, min(8 * q_heads, 32)}, reverse=True)
    need = 0.8 * p.warps_per_cta * p.num_ctas
    for R in cands:
        ntasks = sum(-(-s.vectors // R) for s in seqs)
        if ntasks >= need:
            return R
    return 1


def is_decode_only(seqs: Sequence[SeqSpec], p: ModelParams) -> bool:
    return all(s.q_len <= p.decode_qlen_max for s in seqs)


def attention_queue(seqs: Sequence[SeqSpec], splits: Sequence[int], p: ModelParams):
    """Attention tasks (c_attn, seq) in queue order."""
    tasks = []
    for b, (s, n) in enumerate(zip(seqs, splits)):
        for nt in split_tiles(s.tiles, n):
            for _ in range(s.tasks_per_split):
                tasks.append((nt + p.delta_attn, b))
    if is_decode_only(seqs, p) and any(n > 1 for n in splits):
        # release-aware LPT without query-transfer epochs: decreasing c_attn
        order = sorted(range(len(tasks)), key=lambda t: (-tasks[t][0], t))
        return [tasks[t] for t in order]
    chunk = [t for t in tasks if seqs[t[1]].q_len > p.decode_qlen_max]
    rest = [t for t in tasks if seqs[t[1]].q_len <= p.decode_qlen_max]
    return chunk + rest


def reduction_queue(seqs: Sequence[SeqSpec], splits: Sequence[int], R: int, p: ModelParams):
    """Reduction tasks (c_red, seq) in queue order (sequence order)."""
    reds = []
    for b, (s, n) in enumerate(zip(seqs, splits)):
        left = s.vectors
        while left > 0:
            v = min(R, left)
            reds.append((p.delta_red + p.gamma * v * n, b))
            left -= v
    return reds


@dataclasses.dataclass
class SimResult:
    score: float
    attn_end: float
    seq_attn_end: List[float]
    n_attn_tasks: int
    total_splits: int

    def key(self):
        return (self.score, self.attn_end, self.n_attn_tasks, self.total_splits)


def simulate(seqs: Sequence[SeqSpec], splits: Sequence[int], p: ModelParams,
             q_heads: int = 1) -> SimResult:
    K = p.num_ctas
    queue = attention_queue(seqs, splits, p)
    nseq = len(seqs)
    seq_end = [0.0] * nseq
    release = [None] * K
    running = {}          # cta -> [remaining work, seq]
    t = 0.0
    nxt = 0
    free = list(range(K))
    while True:
        for c in sorted(free):
            if nxt < len(queue):
                running[c] = [queue[nxt][0], queue[nxt][1]]
                nxt += 1
            elif release[c] is None:
                release[c] = t
        free = []
        if not running:
            break
        k = len(running)
        tau = max(p.rho, k / K)
        step = min(r[0] for r in running.values())
        t = t + step * tau
        for c in sorted(running):
            running[c][0] -= step
        done = [c for c in sorted(running) if running[c][0] <= EPS * max(1.0, step)]
        for c in done:
            b = running[c][1]
            seq_end[b] = max(seq_end[b], t)
            del running[c]
            free.append(c)
    for c in range(K):
        if release[c] is None:
            release[c] = t
    attn_end = max(seq_end) if nseq else 0.0
    # reductions on released warps, in queue order
    R = run_length(seqs, q_heads, p)
    reds = reduction_queue(seqs, splits, R, p)
    warps = [[release[c], c, w] for c in range(K) for w in range(p.warps_per_cta)]
    red_end = 0.0
    for cost, b in reds:
        wi = min(range(len(warps)), key=lambda i: (warps[i][0], warps[i][1], warps[i][2]))
        start = max(warps[wi][0], seq_end[b])
        end = start + cost
        warps[wi][0] = end
        red_end = max(red_end, end)
    score = max(attn_end, red_end)
    return SimResult(score=score, attn_end=attn_end, seq_attn_end=seq_end,
                     n_attn_tasks=len(queue), total_splits=int(sum(splits)))


@dataclasses.dataclass
class Plan:
    splits: List[int]
    score: float
    base_splits: List[int]
    base_score: float
    search_splits: List[int]
    search_score: float
    ref_splits: List[int]
    ref_score: float
    limits: List[int]


def reference_plan(seqs: Sequence[SeqSpec], p: ModelParams, lo: List[int], hi: List[int]) -> List[int]:
    work = sum(s.tiles * s.tasks_per_split for s in seqs)
    target = max(1, -(-work // p.num_ctas))
    return [min(hi[b], max(lo[b], -(-s.tiles // target))) for b, s in enumerate(seqs)]


def plan(seqs: Sequence[SeqSpec], p: ModelParams, *, q_heads: int = 1, min_splits: int = 1,
         max_splits: int = 64) -> Plan:
    nseq = len(seqs)
    base = [max(1, min(min_splits, s.tiles)) for s in seqs]
    cap = [max(base[b], min(max_splits, s.tiles)) for b, s in enumerate(seqs)]
    ref = reference_plan(seqs, p, base, cap)
    limits = []
    for b, s in enumerate(seqs):
        lim = ref[b]
        if s.q_len <= p.decode_qlen_max and s.tiles >= p.num_ctas:
            lim = max(lim, 4)
        limits.append(max(base[b], min(lim, cap[b])))

    def ev(spl):
        return simulate(seqs, spl, p, q_heads)

    cur = list(base)
    cur_r = ev(cur)
    while True:
        cands = []
        for b in range(nseq):
            if cur[b] < limits[b]:
                c = list(cur)
                c[b] += 1
                cands.append(c)
        tail = [b for b in range(nseq)
                if cur[b] < limits[b] and _feq(cur_r.seq_attn_end[b], cur_r.attn_end)]
        if len(tail) > 1:
            c = list(cur)
            for b in tail:
                c[b] += 1
            cands.append(c)
        if not cands:
            break
        best, best_r = None, None
        for c in cands:
            r = ev(c)
            if best_r is None or _cmp_key(r.key(), best_r.key()) < 0:
                best, best_r = c, r
        if best_r.score < cur_r.score and not _feq(best_r.score, cur_r.score):
            cur, cur_r = best, best_r
        else:
            break
    base_r = ev(base)
    ref_r = ev(ref)
    final, final_r = base, base_r
    for c, r in ((cur, cur_r), (ref, ref_r)):
        if _cmp_key(r.key(), final_r.key()) < 0:
            final, final_r = c, r
    if final != base and final_r.score > (1.0 - p.adopt_margin) * base_r.score + EPS:
        final, final_r = base, base_r
    return Plan(splits=list(final), score=final_r.score, base_splits=base, base_score=base_r.score,
                search_splits=list(cur), search_score=cur_r.score, ref_splits=ref,
                ref_score=ref_r.score, limits=limits)


UNIFORM_CANDIDATES = (2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64)


def plan_with_uniform(seqs: Sequence[SeqSpec], p: ModelParams, *, q_heads: int = 1, min_splits: int = 1,
                      max_splits: int = 64) -> Plan:
    """The product planner's final selection, which has no counterpart on the
    pages: the pages' selection (``plan``), then uniform plans -- u splits per
    sequence, clamped to each sequence's bounds, for u in UNIFORM_CANDIDATES up
    to the largest bound -- scored in that order; a uniform plan replaces the
    incumbent only if its score is strictly lower and it passes the same
    adoption rule (at least adopt_margin below the baseline).  On plateaus of
    the model, where no single added split lowers the score, the pages'
    one-split-at-a-time search stops early; the uniform candidates cover them."""
    res = plan(seqs, p, q_heads=q_heads, min_splits=min_splits, max_splits=max_splits)
    lo = [max(1, min(min_splits, s.tiles)) for s in seqs]
    hi = [max(lo[b], min(max_splits, s.tiles)) for b, s in enumerate(seqs)]
    max_cap = max(1, max(max(1, min(max_splits, s.tiles)) for s in seqs))
    final, final_score = list(res.splits), res.score
    for u in UNIFORM_CANDIDATES:
        if u > max_cap:
            break
        c = [min(hi[b], max(lo[b], u)) for b in range(len(seqs))]
        if c == res.splits:
            continue
        sc = simulate(seqs, c, p, q_heads).score
        if sc < final_score and not _feq(sc, final_score) and sc <= (1.0 - p.adopt_margin) * res.base_score + EPS:
            final, final_score = c, sc
    return dataclasses.replace(res, splits=final, score=final_score)
