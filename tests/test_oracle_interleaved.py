"""Pins for the oracle's partial states over explicit key sets and the shards
of Helix Parallelism's staggered round-robin KV placement (Section 2.3,
step 4: blocks of the history go to the KVP ranks in turn).

Pins: a key set that is one range gives the range partial of the independent
range code; a scattered key set gives torch's float64 attention over the
gathered rows (a library routine); keys past a row's causal limit drop out;
the round-robin shards partition the history (a worked 16-token-block
example written from the definition); merging the shards' partial states
gives unsplit attention (the merge invariance the pages rely on).
"""
import numpy as np
import pytest
import torch

import oracle
from tests import test_oracle_attention as TA


def _gqa(rng, lens, q_lens, P=4, Hq=4, Hkv=2, D=16):
    arrs = TA._make_gqa(rng, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, q_lens=q_lens)
    return arrs, TA._problem("gqa", arrs, Hq, Hkv, D, D, P, 0.37)


def test_range_key_set_equals_range_partial():
    rng = np.random.default_rng(31)
    arrs, prob = _gqa(rng, [53, 20], [3, 1])
    rows5, rows3, sets = [], [], []
    for b, ql in ((0, 3), (1, 1)):
        L = int(arrs["seq_lens"][b])
        for i in range(ql):
            for h in range(4):
                for a, e in ((0, L), (5, 17), (12, 12), (L - 3, L), (40 % L, L)):
                    rows5.append((b, i, h, a, e))
                    rows3.append((b, i, h))
                    sets.append(np.arange(a, e, dtype=np.int32))
    o_r, l_r = prob.partial_rows(np.array(rows5))
    o_k, l_k = prob.partial_keysets(np.array(rows3), sets)
    np.testing.assert_allclose(o_k, o_r, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(l_k), np.isinf(l_r))
    fin = np.isfinite(l_r)
    np.testing.assert_allclose(l_k[fin], l_r[fin], rtol=0, atol=1e-12)


def test_scattered_key_set_matches_torch_attention():
    rng = np.random.default_rng(32)
    P = 4
    arrs, prob = _gqa(rng, [61], [2], P=P)
    k, v = TA._gather_gqa(arrs, 0, P)            # [Hkv, L, D]
    q = TA._as_f64(arrs["q"])                     # [q_len, Hq, D]
    L = 61
    for trial in range(5):
        keys = np.sort(rng.choice(L, size=int(rng.integers(1, L)), replace=False)).astype(np.int32)
        for i in range(2):
            pos = L - 2 + i
            vis = keys[keys <= pos]
            for h in range(4):
                o, lse = prob.partial_keysets(np.array([[0, i, h]]), [keys])
                if vis.size == 0:
                    assert lse[0] == -np.inf and not o.any()
                    continue
                kh = h // 2
                kt = torch.from_numpy(k[kh, vis])
                vt = torch.from_numpy(v[kh, vis])
                s = 0.37 * (kt @ torch.from_numpy(q[i, h]))
                ref_lse = torch.logsumexp(s, 0).item()
                ref_o = (torch.softmax(s, 0)[:, None] * vt).sum(0).numpy()
                np.testing.assert_allclose(o[0], ref_o, rtol=1e-11, atol=1e-12)
                assert lse[0] == pytest.approx(ref_lse, abs=1e-11)


def test_round_robin_shards_worked_example():
    # 100 tokens in 16-token blocks 0..6 over 3 ranks: rank 0 gets blocks 0, 3, 6;
    # rank 1 blocks 1, 4; rank 2 blocks 2, 5 (the last block holds tokens 96..99)
    sh = oracle.interleaved_split_keys(100, 16, 3)
    want = [list(range(0, 16)) + list(range(48, 64)) + list(range(96, 100)),
            list(range(16, 32)) + list(range(64, 80)),
            list(range(32, 48)) + list(range(80, 96))]
    assert [s.tolist() for s in sh] == want
    # more ranks than blocks: the extra shards are empty
    sh = oracle.interleaved_split_keys(20, 16, 4)
    assert [len(s) for s in sh] == [16, 4, 0, 0]


@pytest.mark.parametrize("L,block,n", [(1, 4, 3), (97, 4, 5), (64, 16, 4), (257, 8, 7)])
def test_round_robin_shards_partition_the_history(L, block, n):
    sh = oracle.interleaved_split_keys(L, block, n)
    allk = np.concatenate(sh)
    assert sorted(allk.tolist()) == list(range(L))          # a partition of 0 .. L-1
    nblocks = -(-L // block)
    for r, s in enumerate(sh):
        blocks = sorted(set((s // block).tolist()))
        assert blocks == list(range(r, nblocks, n))           # every n-th block from block r
        # as many blocks as the contiguous cut gives split r
        assert len(blocks) == nblocks // n + (1 if r < nblocks % n else 0)


@pytest.mark.parametrize("n", [2, 3, 5])
def test_merge_of_round_robin_partials_equals_unsplit(n):
    rng = np.random.default_rng(40 + n)
    arrs, prob = _gqa(rng, [45, 130], [3, 2])
    for b, ql in ((0, 3), (1, 2)):
        L = int(arrs["seq_lens"][b])
        shards = oracle.interleaved_split_keys(L, 4, n)
        for i in range(ql):
            for h in range(4):
                o_p, l_p = prob.partial_keysets(np.array([[b, i, h]] * n), shards)
                o, lse = oracle.merge(o_p, l_p)
                o_f, l_f = prob.attention_rows(np.array([[b, i, h]]))
                np.testing.assert_allclose(o, o_f[0], rtol=1e-12, atol=1e-13)
                assert lse == pytest.approx(l_f[0], abs=1e-12)
