"""Seeded synthetic inputs for split-KV decode attention.

This module is shared by the float64 oracle tests, the CUDA parity tests and
the benchmark.  It holds no attention arithmetic: it only draws lengths, page
tables and N(0,1)-distributed tensor values from fixed seeds, so both sides of
a parity check see the same bytes.

Values come from a counter-based generator: element n of tensor stream s
under seed S takes the value ``table[hash(S, s, n) >> 16]``, where ``table``
holds the 65,536 quantiles Phi^-1((k + 1/2) / 65536) of the standard normal
distribution.  The hash is exact 32-bit integer arithmetic, so the CPU path
(numpy) and the device path (torch int64 ops) give identical values, and any
slice of a tensor can be regenerated on the host without the rest of it.

Workload shapes follow the pages' configurations:
  * Helix Parallelism, Appendix A / Figure 1: Llama-405B attention with
    Q=128 query heads, K=8 KV heads, head size 128, 1M-token contexts.
  * SPLASH, Section 2 Eq. 1 and Appendix A: absorbed MLA with latent width
    d_c=512 plus rotary width d_r=64 shared by all 128 heads (DeepSeek-V3).
  * LiquidCP, Section 7.1: mixed batches of decode requests and chunked
    prefill of up to 4K appended tokens over cached histories.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

__all__ = [
    "WorkloadSpec", "CONFIGS", "get_config", "Workload", "build_workload",
    "normal_table", "hashed_values_np", "hashed_values_torch",
]

_M32 = 0xFFFFFFFF


# --------------------------------------------------------------------------
# counter-based hash (Wellons' "lowbias32" integer mixer)
# --------------------------------------------------------------------------
_C1 = 0x7FEB352D
_C2 = 0x846CA68B


def _lowbias32_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint32, copy=False)
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(_C1)
    x = x ^ (x >> np.uint32(15))
    x = x * np.uint32(_C2)
    x = x ^ (x >> np.uint32(16))
    return x


def _mul32_t(x: torch.Tensor, c: int) -> torch.Tensor:
    # (x * c) mod 2^32 for 0 <= x < 2^32 held in int64, without int64 overflow:
    # split c into 16-bit halves so every partial product stays below 2^48.
    c_lo, c_hi = c & 0xFFFF, c >> 16
    lo = x * c_lo
    hi = ((x * c_hi) & 0xFFFF) << 16
    return (lo + hi) & _M32


def _lowbias32_t(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32_t(x, _C1)
    x = x ^ (x >> 15)
    x = _mul32_t(x, _C2)
    x = x ^ (x >> 16)
    return x


def _stream_key(seed: int, stream: int) -> int:
    k = np.array([(seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x165667B1) & _M32],
                 dtype=np.uint32)
    return int(_lowbias32_np(k)[0])


def _index_hash_np(key: int, start: int, count: int) -> np.ndarray:
    n = np.arange(start, start + count, dtype=np.uint64)
    lo = (n & np.uint64(_M32)).astype(np.uint32)
    hi = (n >> np.uint64(32)).astype(np.uint32)
    kh = _lowbias32_np(hi ^ np.uint32(key))
    return _lowbias32_np(lo ^ kh)


def _index_hash_t(key: int, start: int, count: int, device) -> torch.Tensor:
    n = torch.arange(start, start + count, dtype=torch.int64, device=device)
    lo = n & _M32
    hi = n >> 32
    kh = _lowbias32_t(hi ^ key)
    return _lowbias32_t(lo ^ kh)


_TABLE_CACHE: Dict[str, np.ndarray] = {}


def normal_table(dtype: str) -> np.ndarray:
    """65,536 standard-normal quantiles, rounded once to ``dtype``.

    Returns float32 values for "f32" and the bf16 bit patterns (uint16) for
    "bf16".  Rounding to bf16 is round-to-nearest-even from float32.
    "e4m3/<s>" gives 8-bit E4M3 codes of quantile / s (uint8; torch's
    round-to-nearest-even conversion): an FP8 cache whose values, code * s,
    follow N(0, 1) to within the format's precision.
    """
    if dtype in _TABLE_CACHE:
        return _TABLE_CACHE[dtype]
    k = torch.arange(65536, dtype=torch.float64)
    q = torch.special.ndtri((k + 0.5) / 65536.0)
    if dtype == "f32":
        t = q.to(torch.float32).numpy()
    elif dtype == "bf16":
        t = q.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    elif dtype.startswith("e4m3/"):
        sc = float(dtype.split("/", 1)[1])
        t = (q / sc).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        raise ValueError(dtype)
    t = np.ascontiguousarray(t)
    t.setflags(write=False)
    _TABLE_CACHE[dtype] = t
    return t


def hashed_values_np(seed: int, stream: int, start: int, count: int, dtype: str) -> np.ndarray:
    """Elements [start, start+count) of stream ``stream`` as a numpy array
    (float32 for "f32", uint16 bf16 bit patterns for "bf16")."""
    key = _stream_key(seed, stream)
    idx = _index_hash_np(key, start, count) >> np.uint32(16)
    return normal_table(dtype)[idx.astype(np.int64)]


def hashed_values_torch(seed: int, stream: int, count: int, dtype: str, device,
                        out: Optional[torch.Tensor] = None,
                        chunk: int = 1 << 27, start: int = 0) -> torch.Tensor:
    """Elements [start, start+count) of a stream as a flat torch tensor on ``device``.

    The result is float32 for "f32", torch.bfloat16 for "bf16" and uint8 E4M3
    codes for "e4m3/<s>"; it is bit-identical to :func:`hashed_values_np`.  Work
    proceeds in chunks so the int64 temporaries stay small.
    """
    key = _stream_key(seed, stream)
    tdt = torch.float32 if dtype == "f32" else torch.uint8 if dtype.startswith("e4m3/") else torch.bfloat16
    table = torch.from_numpy(normal_table(dtype).view(np.int16).copy() if dtype == "bf16"
                             else normal_table(dtype).copy())
    if dtype == "bf16":
        table = table.view(torch.bfloat16)
    table = table.to(device)
    if out is None:
        out = torch.empty(count, dtype=tdt, device=device)
    for s in range(0, count, chunk):
        c = min(chunk, count - s)
        h = _index_hash_t(key, start + s, c, device) >> 16
        out[s:s + c] = table[h]
        del h
    return out


# --------------------------------------------------------------------------
# workload specifications
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    kind: str               # "gqa" or "mla"
    dtype: str              # "f32" or "bf16" (q, K, V storage type)
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    page_size: int
    scale: float
    seed: int
    lengths: str            # "fixed:<L,...>", "loguniform:<lo>:<hi>", "speculative:<lo>:<hi>:<q>", "mixed:..."
    split: str              # "uniform:<n>" or "planner:<min>:<max>"
    shuffle_pages: bool = True
    description: str = ""
    kv_fp8: bool = False    # K/V caches as E4M3 codes with one scale per tensor
    k_scale: float = 1.0
    v_scale: float = 1.0


CONFIGS: Dict[str, WorkloadSpec] = {
    "tiny_fp32_gqa": WorkloadSpec(
        name="tiny_fp32_gqa", kind="gqa", dtype="f32", batch=4, num_q_heads=8,
        num_kv_heads=1, head_dim_qk=64, head_dim_v=64, page_size=16,
        scale=1.0 / 8.0, seed=1, lengths="fixed:37,128,300,513", split="uniform:4",
        description="fp32 GQA decode, B=4, 8/1 heads, D=64, L={37,128,300,513}, P=16, 4 splits"),
    "llama405b_gqa_decode": WorkloadSpec(
        name="llama405b_gqa_decode", kind="gqa", dtype="bf16", batch=32, num_q_heads=128,
        num_kv_heads=8, head_dim_qk=128, head_dim_v=128, page_size=64,
        scale=1.0 / math.sqrt(128.0), seed=2, lengths="fixed:32768*32", split="uniform:8",
        description="Llama-405B GQA decode, B=32, 128/8 heads, D=128, L=32768, P=64, 8 splits"),
    "deepseek_mla_decode": WorkloadSpec(
        name="deepseek_mla_decode", kind="mla", dtype="bf16", batch=64, num_q_heads=128,
        num_kv_heads=1, head_dim_qk=576, head_dim_v=512, page_size=64,
        scale=1.0 / math.sqrt(192.0), seed=3, lengths="loguniform:1024:131072",
        split="planner:1:64",
        description="DeepSeek-V3 absorbed MLA decode, B=64, 128 heads, latent 512+64, "
                    "L log-uniform 1k-128k, P=64, planner splits"),
    "mixed_chunked_prefill": WorkloadSpec(
        name="mixed_chunked_prefill", kind="gqa", dtype="bf16", batch=50, num_q_heads=64,
        num_kv_heads=8, head_dim_qk=128, head_dim_v=128, page_size=64,
        scale=1.0 / math.sqrt(128.0), seed=4, lengths="mixed:48:4096:65536:2:16384:2048",
        split="planner:1:64",
        description="48 decode (L log-uniform 4k-64k) + 2 chunked prefill (2048 after 16k), "
                    "64/8 heads, D=128, P=64, planner splits"),
    "million_token_decode": WorkloadSpec(
        name="million_token_decode", kind="gqa", dtype="bf16", batch=4, num_q_heads=64,
        num_kv_heads=8, head_dim_qk=128, head_dim_v=128, page_size=128,
        scale=1.0 / math.sqrt(128.0), seed=5, lengths="fixed:1048576*4", split="planner:16:64",
        description="1M-token decode, B=4, 64/8 heads, D=128, P=128, 16-64 planner splits"),
    "llama405b_fp8_decode": WorkloadSpec(
        name="llama405b_fp8_decode", kind="gqa", dtype="bf16", batch=32, num_q_heads=128,
        num_kv_heads=8, head_dim_qk=128, head_dim_v=128, page_size=64,
        scale=1.0 / math.sqrt(128.0), seed=7, lengths="fixed:32768*32", split="uniform:8",
        kv_fp8=True, k_scale=0.0625, v_scale=0.05,
        description="Llama-405B GQA decode over an FP8 (E4M3) KV cache, one scale per tensor: "
                    "B=32, 128/8 heads, D=128, L=32768, P=64, 8 splits"),
    "deepseek_mla_fp8_decode": WorkloadSpec(
        name="deepseek_mla_fp8_decode", kind="mla", dtype="bf16", batch=64, num_q_heads=128,
        num_kv_heads=1, head_dim_qk=576, head_dim_v=512, page_size=64,
        scale=1.0 / math.sqrt(192.0), seed=8, lengths="loguniform:1024:131072",
        split="planner:1:64", kv_fp8=True, k_scale=0.0625, v_scale=0.05,
        description="DeepSeek-V3 absorbed MLA decode over an FP8 (E4M3) latent cache, one scale "
                    "per tensor (keys and values take k_scale): B=64, 128 heads, latent 512+64, "
                    "L log-uniform 1k-128k, P=64, planner splits"),
    "spec_decode_q16": WorkloadSpec(
        name="spec_decode_q16", kind="gqa", dtype="bf16", batch=48, num_q_heads=32,
        num_kv_heads=8, head_dim_qk=128, head_dim_v=128, page_size=64,
        scale=1.0 / math.sqrt(128.0), seed=6, lengths="speculative:4096:65536:16",
        split="planner:1:64",
        description="speculative decode: 48 requests x 16 query tokens (1 target + 15 drafts, "
                    "causal among them) after histories log-uniform 4k-64k, 32/8 heads, D=128, "
                    "P=64, planner splits"),
}

CONFIG_ORDER: List[str] = list(CONFIGS.keys())


def get_config(name_or_index) -> WorkloadSpec:
    if isinstance(name_or_index, int):
        return CONFIGS[CONFIG_ORDER[name_or_index]]
    return CONFIGS[name_or_index]


def _parse_lengths(spec: WorkloadSpec, rng: np.random.Generator):
    kind, _, rest = spec.lengths.partition(":")
    if kind == "fixed":
        vals: List[int] = []
        for tok in rest.split(","):
            if "*" in tok:
                v, n = tok.split("*")
                vals += [int(v)] * int(n)
            else:
                vals.append(int(tok))
        seq = np.array(vals, dtype=np.int64)
        ql = np.ones_like(seq)
    elif kind == "loguniform":
        lo, hi = (int(x) for x in rest.split(":"))
        u = rng.random(spec.batch)
        seq = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
        seq = np.clip(seq, lo, hi)
        ql = np.ones_like(seq)
    elif kind == "speculative":
        # histories log-uniform in [lo, hi], then q_len query tokens appended (their KV in the cache)
        lo, hi, qlen = (int(x) for x in rest.split(":"))
        u = rng.random(spec.batch)
        hist = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
        seq = np.clip(hist, lo, hi) + qlen
        ql = np.full(spec.batch, qlen, dtype=np.int64)
    elif kind == "mixed":
        nd, lo, hi, npf, hist, chunk = (int(x) for x in rest.split(":"))
        u = rng.random(nd)
        dec = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
        dec = np.clip(dec, lo, hi)
        seq = np.concatenate([dec, np.full(npf, hist + chunk, dtype=np.int64)])
        ql = np.concatenate([np.ones(nd, dtype=np.int64), np.full(npf, chunk, dtype=np.int64)])
    else:
        raise ValueError(spec.lengths)
    assert len(seq) == spec.batch, (spec.name, len(seq))
    return seq.astype(np.int32), ql.astype(np.int32)


# tensor stream ids (stable: changing them changes every input)
_STREAM_Q, _STREAM_K, _STREAM_V = 1, 2, 3


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    seq_lens: np.ndarray          # int32 [B], includes the appended query tokens
    q_lens: np.ndarray            # int32 [B]
    qo_indptr: np.ndarray         # int32 [B+1]
    page_table: np.ndarray        # int32 [B, max_pages_per_req], -1 = unused
    num_pages: int
    # per-tensor shapes and element counts
    q_shape: tuple
    k_shape: tuple
    v_shape: Optional[tuple]

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def max_pages_per_req(self) -> int:
        return int(self.page_table.shape[1])

    def numel(self, which: str) -> int:
        shape = {"q": self.q_shape, "k": self.k_shape, "v": self.v_shape}[which]
        return int(np.prod(shape))

    def kv_stream_ids(self):
        return _STREAM_K, _STREAM_V

    def _gen(self, which: str) -> str:
        """Generator storage type of tensor ``which`` ("q", "k", "v")."""
        if which != "q" and self.spec.kv_fp8:
            return f"e4m3/{self.spec.k_scale if which == 'k' else self.spec.v_scale!r}"
        return self.spec.dtype

    # ---- host-side (numpy) tensors: the whole thing, or slices ---------
    def q_host(self) -> np.ndarray:
        return hashed_values_np(self.spec.seed, _STREAM_Q, 0, self.numel("q"),
                                self.spec.dtype).reshape(self.q_shape)

    def k_host(self) -> np.ndarray:
        return hashed_values_np(self.spec.seed, _STREAM_K, 0, self.numel("k"),
                                self._gen("k")).reshape(self.k_shape)

    def v_host(self) -> Optional[np.ndarray]:
        if self.v_shape is None:
            return None
        return hashed_values_np(self.spec.seed, _STREAM_V, 0, self.numel("v"),
                                self._gen("v")).reshape(self.v_shape)

    def kv_pages_host(self, which: str, pages: Sequence[int], kv_head: Optional[int] = None) -> np.ndarray:
        """Host copies of selected physical pages of the K ('k') or V ('v')
        cache, regenerated from the counter-based stream.

        GQA caches are [num_pages, Hkv, P, D]; with ``kv_head`` given the
        result is [len(pages), P, D] for that head, else [len(pages), Hkv, P, D].
        MLA caches are [num_pages, P, 576] and ``kv_head`` must be None or 0.
        """
        shape = self.k_shape if which == "k" else self.v_shape
        stream = _STREAM_K if which == "k" else _STREAM_V
        per_page = int(np.prod(shape[1:]))
        if self.spec.kind == "gqa" and kv_head is not None:
            blk = int(np.prod(shape[2:]))
            parts = [hashed_values_np(self.spec.seed, stream, p * per_page + kv_head * blk, blk,
                                      self._gen(which)) for p in pages]
            return np.stack(parts).reshape((len(pages),) + tuple(shape[2:]))
        parts = [hashed_values_np(self.spec.seed, stream, p * per_page, per_page, self._gen(which))
                 for p in pages]
        return np.stack(parts).reshape((len(pages),) + tuple(shape[1:]))

    # ---- device tensors ----------------------------------------------------
    def device_tensors(self, device) -> Dict[str, torch.Tensor]:
        d = {}
        d["q"] = hashed_values_torch(self.spec.seed, _STREAM_Q, self.numel("q"), self.spec.dtype,
                                     device).view(self.q_shape)
        d["k"] = hashed_values_torch(self.spec.seed, _STREAM_K, self.numel("k"), self._gen("k"),
                                     device).view(self.k_shape)
        if self.v_shape is not None:
            d["v"] = hashed_values_torch(self.spec.seed, _STREAM_V, self.numel("v"),
                                         self._gen("v"), device).view(self.v_shape)
        else:
            d["v"] = None
        d["page_table"] = torch.from_numpy(self.page_table).to(device)
        d["seq_lens"] = torch.from_numpy(self.seq_lens).to(device)
        d["qo_indptr"] = torch.from_numpy(self.qo_indptr).to(device)
        return d


def build_workload(spec: WorkloadSpec, *, seq_lens: Optional[Sequence[int]] = None,
                   q_lens: Optional[Sequence[int]] = None, batch: Optional[int] = None,
                   extra_pages: int = 0) -> Workload:
    """Lengths and page table for ``spec`` (tensor values are generated lazily).

    ``seq_lens``/``q_lens`` override the recipe (used by edge-case tests);
    ``extra_pages`` adds unused physical pages to the pool.
    """
    rng = np.random.default_rng(spec.seed)
    if seq_lens is None:
        sl, ql = _parse_lengths(spec, rng)
    else:
        sl = np.asarray(seq_lens, dtype=np.int32)
        ql = np.ones_like(sl) if q_lens is None else np.asarray(q_lens, dtype=np.int32)
    if batch is not None and seq_lens is None:
        sl, ql = sl[:batch], ql[:batch]
    B = len(sl)
    P = spec.page_size
    npages_req = (sl.astype(np.int64) + P - 1) // P
    total = int(npages_req.sum()) + int(extra_pages)
    perm = rng.permutation(total) if spec.shuffle_pages else np.arange(total)
    maxp = max(1, int(npages_req.max()) if B else 1)
    pt = np.full((B, maxp), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(npages_req[b])
        pt[b, :n] = perm[off:off + n]
        off += n
    qo = np.zeros(B + 1, dtype=np.int32)
    qo[1:] = np.cumsum(ql)
    total_q = int(qo[-1])
    if spec.kind == "gqa":
        q_shape = (total_q, spec.num_q_heads, spec.head_dim_qk)
        k_shape = (total, spec.num_kv_heads, P, spec.head_dim_qk)
        v_shape = (total, spec.num_kv_heads, P, spec.head_dim_v)
    else:
        q_shape = (total_q, spec.num_q_heads, spec.head_dim_qk)
        k_shape = (total, P, spec.head_dim_qk)
        v_shape = None
    return Workload(spec=spec, seq_lens=sl, q_lens=ql, qo_indptr=qo, page_table=pt,
                    num_pages=total, q_shape=q_shape, k_shape=k_shape, v_shape=v_shape)


def uniform_splits(spec: WorkloadSpec) -> Optional[int]:
    kind, _, rest = spec.split.partition(":")
    return int(rest) if kind == "uniform" else None


def planner_split_range(spec: WorkloadSpec):
    kind, _, rest = spec.split.partition(":")
    if kind != "planner":
        return None
    lo, hi = (int(x) for x in rest.split(":"))
    return lo, hi
