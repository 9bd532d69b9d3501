"""Pins for the oracle's merge of partial states (LiquidCP Eq. 1; Helix
Parallelism, "Attention-Phase Configuration" step 3) and its page-aligned
split bounds.

Pins: partition invariance against unsplit attention (the pages' claim that
the merge is identical to attention over the unsharded cache), a single
split returning the full result bit for bit, associativity, a hand-computed
two-state case, -inf handling, and the 59/59/58 cut of LiquidCP Figure 8.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _problem(rng, L, Hq=4, Hkv=2, D=16, P=4, q_len=1):
    npg = (L + P - 1) // P
    pt = rng.permutation(npg + 2)[:npg].astype(np.int32)[None]
    return oracle.Problem(
        kind="gqa", q=rng.standard_normal((q_len, Hq, D)).astype(np.float32),
        k=rng.standard_normal((npg + 2, Hkv, P, D)).astype(np.float32),
        v=rng.standard_normal((npg + 2, Hkv, P, D)).astype(np.float32),
        page_table=pt, seq_lens=np.array([L], np.int32), qo_indptr=np.array([0, q_len], np.int32),
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim_qk=D, head_dim_v=D, page_size=P, scale=0.3)


def _random_partition(rng, L, n):
    cuts = np.sort(rng.integers(0, L + 1, size=n - 1))
    edges = np.concatenate([[0], cuts, [L]])
    return [(int(edges[r]), int(edges[r + 1])) for r in range(n)]


@pytest.mark.parametrize("n", [2, 3, 7, 16])
def test_merge_of_any_partition_equals_unsplit(n):
    rng = np.random.default_rng(100 + n)
    L = 97
    prob = _problem(rng, L, q_len=3)
    for trial in range(4):
        parts = _random_partition(rng, L, n)
        if trial == 0:
            parts.insert(1, (parts[1][0], parts[1][0]))     # add an empty part
        for i in range(3):
            for h in range(4):
                rows = np.array([[0, i, h, a, b] for a, b in parts], dtype=np.int32)
                o_p, l_p = prob.partial_rows(rows)
                o, lse = oracle.merge(o_p, l_p)
                o_full, l_full = prob.attention_rows(np.array([[0, i, h]]))
                np.testing.assert_allclose(o, o_full[0], rtol=1e-12, atol=1e-13)
                assert lse == pytest.approx(l_full[0], abs=1e-12)


def test_single_split_is_full_result_bitwise():
    rng = np.random.default_rng(7)
    prob = _problem(rng, 45)
    o_p, l_p = prob.partial_rows(np.array([[0, 0, 2, 0, 45]]))
    o, lse = oracle.merge(o_p, l_p)
    o_full, l_full = prob.attention_rows(np.array([[0, 0, 2]]))
    np.testing.assert_array_equal(o, o_full[0])
    assert lse == l_full[0]


def test_merge_is_associative():
    rng = np.random.default_rng(8)
    o = rng.standard_normal((3, 32))
    lse = rng.standard_normal(3) * 5
    ab, lab = oracle.merge(o[:2], lse[:2])
    left, l_left = oracle.merge(np.stack([ab, o[2]]), np.array([lab, lse[2]]))
    bc, lbc = oracle.merge(o[1:], lse[1:])
    right, l_right = oracle.merge(np.stack([o[0], bc]), np.array([lse[0], lbc]))
    np.testing.assert_allclose(left, right, rtol=1e-14, atol=1e-15)
    assert l_left == pytest.approx(l_right, abs=1e-14)


def test_merge_hand_computed_two_states():
    # exp(lse) = 1 and 3: weights 1/4 and 3/4, lse = ln 4
    o_parts = np.array([[4.0, 0.0, -8.0], [0.0, 4.0, 8.0]])
    o, lse = oracle.merge(o_parts, np.array([0.0, math.log(3.0)]))
    np.testing.assert_allclose(o, [1.0, 3.0, 4.0], rtol=0, atol=1e-15)
    assert lse == pytest.approx(math.log(4.0), abs=1e-15)


def test_merge_minus_inf_terms():
    o_parts = np.array([[1.0, 2.0], [9.0, 9.0], [3.0, 4.0]])
    o, lse = oracle.merge(o_parts, np.array([0.0, -math.inf, 0.0]))
    np.testing.assert_allclose(o, [2.0, 3.0])
    assert lse == pytest.approx(math.log(2.0))
    o, lse = oracle.merge(o_parts, np.array([-math.inf] * 3))
    assert lse == -math.inf and not o.any()


def test_merge_rows_matches_single_merges():
    rng = np.random.default_rng(9)
    ind = np.array([0, 3, 3, 4, 9], dtype=np.int32)
    o_parts = rng.standard_normal((9, 8))
    lse = rng.standard_normal(9)
    o, l = oracle.merge_rows(ind, o_parts, lse)
    for x in range(4):
        oo, ll = oracle.merge(o_parts[ind[x]:ind[x + 1]], lse[ind[x]:ind[x + 1]])
        np.testing.assert_array_equal(o[x], oo)
        assert l[x] == ll or (math.isinf(l[x]) and math.isinf(ll))


def test_split_bounds_figure8_and_edges():
    g = json.load(open(os.path.join(HERE, "golden", "liquidcp_fig8.json")))
    b = oracle.split_bounds(176, 1, 3)
    assert [e - s for s, e in b] == g["split_176_three_ways"]
    # page aligned, contiguous, covering, ragged tail
    b = oracle.split_bounds(513, 16, 4)
    assert b[0][0] == 0 and b[-1][1] == 513
    assert all(b[r][1] == b[r + 1][0] for r in range(3))
    assert all(s % 16 == 0 for s, _ in b)
    assert [e - s for s, e in b] == [144, 128, 128, 113]
    # more splits than pages: trailing ranges are empty
    b = oracle.split_bounds(37, 16, 4)
    assert [e - s for s, e in b] == [16, 16, 5, 0]
