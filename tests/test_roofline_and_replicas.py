"""CPU checks of the measurement helpers: the algorithmic-bytes model against
Helix Parallelism's worked KV-read example, and the replica timing path of
bench.py under a world_size-2 gloo group."""
import math
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from long_context_split_gb300 import roofline


def test_helix_kv_read_time_example():
    # Helix Parallelism, "All Results Are Normalized ...": Llama-405B, B=8, S=1M, Hsz=128, FP4
    # (0.5 B), MemBW 8000 GB/s, no KVP: 8 x 2 x 8 x 128 x 1e6 x 0.5 / 8e12 ~= 1.02 ms per layer.
    # The printed product keeps all K=8 KV heads (ceil(K/TP_A) = 8, i.e. TP_A = 1) although the
    # sentence calls it "the TP=8 case"; the arithmetic as printed is what is pinned here.
    t = roofline.helix_kv_read_time(B=8, K=8, TP_A=1, Hsz=128, S=1e6, KVP=1, bytes_per_param=0.5,
                                    mem_bw_bytes_per_s=8e12)
    assert t == pytest.approx(1.02e-3, rel=5e-3)
    # the ceil(K / TP_A) floor: from TP_A = K on, each GPU still reads one whole KV head
    t8 = roofline.helix_kv_read_time(8, 8, 8, 128, 1e6, 1, 0.5, 8e12)
    assert t8 == pytest.approx(t / 8)
    assert roofline.helix_kv_read_time(8, 8, 16, 128, 1e6, 1, 0.5, 8e12) == pytest.approx(t8)
    # KVP divides the per-GPU read volume
    assert roofline.helix_kv_read_time(8, 8, 1, 128, 1e6, 4, 0.5, 8e12) == pytest.approx(t / 4)


def test_kv_bytes_matches_helix_numerator():
    # the single-GPU bytes are Helix's numerator with TP_A = KVP = 1
    seq = [1_000_000] * 8
    b = roofline.kv_bytes("gqa", seq, num_kv_heads=8, head_dim_qk=128, head_dim_v=128, elem_bytes=2)
    t = roofline.helix_kv_read_time(8, 8, 1, 128, 1e6, 1, 2, 1.0)
    assert b == pytest.approx(t)
    assert roofline.kv_bytes("gqa", [32768] * 32, 8, 128, 128, 2) == 4 * 2 ** 30
    assert roofline.kv_bytes("mla", [10, 20], 1, 576, 512, 2) == 30 * 576 * 2


def test_attention_flops_causal_counts():
    # decode: every row sees all L keys; prefill of L rows sees L(L+1)/2 pairs
    assert roofline.attention_flops([100], [1], 2, 64, 64) == 2 * 128 * 2 * 100
    assert roofline.attention_flops([10], [10], 1, 8, 8) == 2 * 16 * 55
    assert roofline.attention_flops([30], [5], 1, 8, 8) == 2 * 16 * (5 * 25 + 15)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _replica(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    d, r, ws, local = bench._dist()
    assert (r, ws) == (rank, world)
    bench._barrier(d)
    m = bench._max_over_ranks(d, float(10 + rank))
    q.put((rank, m))
    d.destroy_process_group()


def test_bench_replica_timing_takes_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 11.0, 1: 11.0}
