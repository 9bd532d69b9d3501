"""Algorithmic byte and flop counts of split-KV attention (for rooflines).

KV bytes follow Helix Parallelism's KV read-time equation (Appendix A, "The
Two Bottlenecks as DRAM Read-Time Equations"):
    Time_KV = B * 2 * ceil(K / TP_A) * Hsz * (S / KVP) * bytes / MemBW,
i.e. every cached token's K and V rows of every KV head are read once.  For
absorbed MLA the one latent row of d_c + d_r elements per token is read once
(keys and values share it; SPLASH Section 2, Eq. 1).
"""
from __future__ import annotations

import math
from typing import Sequence


def helix_kv_read_time(B: int, K: int, TP_A: int, Hsz: int, S: float, KVP: int, bytes_per_param: float,
                       mem_bw_bytes_per_s: float) -> float:
    """Helix Time_KV in seconds."""
    return B * 2 * math.ceil(K / TP_A) * Hsz * (S / KVP) * bytes_per_param / mem_bw_bytes_per_s


def kv_bytes(kind: str, seq_lens: Sequence[int], num_kv_heads: int, head_dim_qk: int, head_dim_v: int,
             elem_bytes: int) -> int:
    """Bytes of KV cache one pass must read: each token's K and V rows once."""
    tokens = int(sum(int(x) for x in seq_lens))
    if kind == "gqa":
        return tokens * num_kv_heads * (head_dim_qk + head_dim_v) * elem_bytes
    return tokens * head_dim_qk * elem_bytes   # MLA: one shared latent row per token


def io_bytes(total_q: int, num_q_heads: int, head_dim_qk: int, head_dim_v: int, elem_bytes: int,
             out_bytes: int) -> int:
    """Query read plus output and LSE write."""
    return total_q * num_q_heads * (head_dim_qk * elem_bytes + head_dim_v * out_bytes + 4)


def partial_state_bytes(num_states: int, head_dim_v: int, merged_rows: int) -> int:
    """Float32 partial states written and read back by the merge (rows that
    need merging only)."""
    return 2 * num_states * (head_dim_v + 1) * 4 if merged_rows else 0


def attention_flops(seq_lens: Sequence[int], q_lens: Sequence[int], num_q_heads: int, head_dim_qk: int,
                    head_dim_v: int) -> int:
    """2 * (D_qk + D_v) flops per (query row, visible key) pair, causal rows
    counted exactly."""
    total = 0
    for L, ql in zip(seq_lens, q_lens):
        L, ql = int(L), int(ql)
        # row i sees L - ql + i + 1 keys
        pairs = ql * (L - ql) + ql * (ql + 1) // 2
        total += pairs
    return 2 * (head_dim_qk + head_dim_v) * num_q_heads * total
