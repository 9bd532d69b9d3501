"""Host-side check of the full-size parity sampler: the sampled (request, KV
head) groups always include the longest request, the request with the most
splits and every chunked-prefill request, and number at least eight."""
import numpy as np

import workloads as W
from tests.test_gpu_parity import _sample_groups


class _FakePlan:
    def __init__(self, splits):
        self._s = np.asarray(splits, dtype=np.int32)

    def splits(self):
        return self._s


def test_sample_groups_cover_the_extremes():
    spec = W.get_config("mixed_chunked_prefill")
    wl = W.build_workload(spec)
    s = np.ones(spec.batch, dtype=np.int32)
    s[5] = 9
    g = _sample_groups(wl, _FakePlan(s), 8)
    bs = [b for b, _ in g]
    assert len(set(g)) == len(g) >= 8
    assert int(np.argmax(wl.seq_lens)) in bs and 5 in bs and 48 in bs and 49 in bs
    assert all(0 <= h < spec.num_kv_heads for _, h in g)


def test_sample_groups_cover_every_request_of_a_small_batch():
    spec = W.get_config("million_token_decode")
    wl = W.build_workload(spec)
    g = _sample_groups(wl, _FakePlan(np.full(spec.batch, 32)), 8)
    assert len(set(g)) == 8 and {b for b, _ in g} == set(range(spec.batch))


def test_sample_groups_mla_distinct_requests():
    spec = W.get_config("deepseek_mla_decode")
    wl = W.build_workload(spec)
    sp = np.arange(spec.batch) % 7 + 1
    g = _sample_groups(wl, _FakePlan(sp), 8)
    assert len({b for b, _ in g}) == 8 and all(h == 0 for _, h in g)
    assert int(np.argmax(wl.seq_lens)) in [b for b, _ in g] and int(np.argmax(sp)) in [b for b, _ in g]
