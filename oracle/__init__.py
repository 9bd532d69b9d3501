"""Float64 CPU oracle for split-KV decode attention, the LSE-weighted merge
and the critical-wave split planner.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA path
(``long_context_split_gb300``) never imports it, and it never imports that
package: the two share no code, only the seeded inputs of ``workloads``.

Contents
  * ``splitkv_oracle.c`` (compiled here with gcc into ``liboracle.so``):
    partial attention states over key ranges and explicit key sets, full
    attention, and the merge
    of partial states (LiquidCP Section 3, Eq. 1; Helix Parallelism,
    "Attention-Phase Configuration", steps 2-3).
  * ``interleaved_split_keys``: the KV shards of Helix Parallelism's staggered
    round-robin placement (Section 2.3, step 4), for splits that are not ranges.
  * ``split_bounds``: the page-aligned uniform partition of a history into
    independent ranges (LiquidCP Section 2.1, "KV splitting divides this shard
    into independent ranges"; Figure 8 splits 176 tiles three ways as
    59/59/58).
  * ``planner``: the critical-wave model and plan search (LiquidCP Section
    5.2, Eqs. 5-6, Figure 8, Appendix A.2).

Every function is pinned in ``tests/test_oracle_*.py`` against something
other than itself (library routines, closed forms, the pages' worked
example, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "splitkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (-O2, OpenMP) when missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32), ("scale", ctypes.c_double),
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("qo_indptr", ctypes.c_void_p),
        ("kv_dtype", ctypes.c_int32), ("pad0", ctypes.c_int32),
        ("k_scale", ctypes.c_double), ("v_scale", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_partial_rows.argtypes = [P, ctypes.c_int, ip, dp, dp]
            lib.oracle_partial_rows.restype = ctypes.c_int
            lib.oracle_partial_keysets.argtypes = [P, ctypes.c_int, ip, ip, ip, dp, dp]
            lib.oracle_partial_keysets.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [P, ctypes.c_int, ip, dp, dp]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp, dp]
            lib.oracle_merge.restype = None
            lib.oracle_merge_rows.argtypes = [ctypes.c_int, ctypes.c_int, ip, dp, dp, dp, dp]
            lib.oracle_merge_rows.restype = None
            lib.oracle_e4m3_values.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint8), dp]
            lib.oracle_e4m3_values.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


class use_library:
    """Context manager that points the oracle at another build of
    ``splitkv_oracle.c`` (the mutation tests compile planted mistakes into a
    temporary library and check that the pins catch them)."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_partial_rows", "oracle_attention_rows", "oracle_merge",
                     "oracle_merge_rows", "oracle_num_threads"):
            f, g = getattr(lib, name), getattr(self.saved, name)
            f.argtypes, f.restype = g.argtypes, g.restype
        with _lock:
            _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class Problem:
    """Host description of one batch: queries, paged caches and lengths.

    ``q``: [total_q, Hq, D_qk]; ``k``: GQA [num_pages, Hkv, P, D_qk] or MLA
    [num_pages, P, D_qk]; ``v``: GQA [num_pages, Hkv, P, D_v] or None (MLA
    values are the first ``head_dim_v`` columns of ``k``).  Arrays are float32
    or uint16 bf16 bit patterns; ``k`` and ``v`` may instead be uint8 E4M3 codes,
    whose values are scaled by ``k_scale`` / ``v_scale`` (an FP8 KV cache with one
    scale per tensor; MLA latent rows take ``k_scale``).
    """

    def __init__(self, *, kind: str, q: np.ndarray, k: np.ndarray, v: Optional[np.ndarray],
                 page_table: np.ndarray, seq_lens: np.ndarray, qo_indptr: np.ndarray,
                 num_q_heads: int, num_kv_heads: int, head_dim_qk: int, head_dim_v: int,
                 page_size: int, scale: float, k_scale: float = 1.0, v_scale: float = 1.0):
        codes = {np.dtype(np.float32): 0, np.dtype(np.uint16): 1, np.dtype(np.uint8): 2}
        dt = codes[np.dtype(q.dtype)]
        self.q = np.ascontiguousarray(q)
        self.k = np.ascontiguousarray(k)
        kvdt = codes[np.dtype(self.k.dtype)]
        assert dt != 2 and (kvdt == dt or kvdt == 2), "K/V share the query's storage type or are E4M3 codes"
        self.v = None if v is None else np.ascontiguousarray(v)
        if self.v is not None:
            assert self.v.dtype == self.k.dtype
        self.k_scale = float(k_scale)
        self.v_scale = float(v_scale)
        self.page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        self.seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.qo_indptr = np.ascontiguousarray(qo_indptr, dtype=np.int32)
        self.kind = kind
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads
        self.head_dim_qk = head_dim_qk
        self.head_dim_v = head_dim_v
        self.page_size = page_size
        self.scale = scale
        self.batch = len(self.seq_lens)
        self._s = _Problem(
            kind=0 if kind == "gqa" else 1, dtype=dt, batch=self.batch,
            num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim_qk=head_dim_qk,
            head_dim_v=head_dim_v, page_size=page_size, num_pages=int(self.k.shape[0]),
            max_pages_per_req=int(self.page_table.shape[1]), scale=float(scale),
            q=self.q.ctypes.data, k_cache=self.k.ctypes.data,
            v_cache=(self.v.ctypes.data if self.v is not None else None),
            page_table=self.page_table.ctypes.data, seq_lens=self.seq_lens.ctypes.data,
            qo_indptr=self.qo_indptr.ctypes.data, kv_dtype=kvdt, pad0=0, k_scale=self.k_scale,
            v_scale=self.v_scale)

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr)

    def all_rows(self) -> np.ndarray:
        """(b, i, h) for every output row, in output order (token-major, then head)."""
        rows = []
        for b in range(self.batch):
            for i in range(int(self.q_lens[b])):
                for h in range(self.num_q_heads):
                    rows.append((b, i, h))
        return np.array(rows, dtype=np.int32).reshape(-1, 3)

    def partial_rows(self, rows5: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """Partial states for rows (b, i, h, key_begin, key_end)."""
        rows5 = np.ascontiguousarray(rows5, dtype=np.int32).reshape(-1, 5)
        n = rows5.shape[0]
        o = np.zeros((n, self.head_dim_v), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = _load().oracle_partial_rows(ctypes.byref(self._s), n, _iptr(rows5), _dptr(o), _dptr(lse))
        if rc != 0:
            raise ValueError(f"oracle_partial_rows failed with code {rc}")
        return o, lse

    def partial_keysets(self, rows3: np.ndarray, keysets: Sequence[np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
        """Partial states of rows (b, i, h), row r over the keys ``keysets[r]`` (a split that
        is not one range: Helix Parallelism Section 2.3, staggered round-robin placement)."""
        rows3 = np.ascontiguousarray(rows3, dtype=np.int32).reshape(-1, 3)
        n = rows3.shape[0]
        if len(keysets) != n:
            raise ValueError("one key set per row")
        ind = np.zeros(n + 1, dtype=np.int32)
        ind[1:] = np.cumsum([len(k) for k in keysets])
        keys = (np.concatenate([np.asarray(k, dtype=np.int32) for k in keysets]) if n
                else np.zeros(0, dtype=np.int32))
        keys = np.ascontiguousarray(keys if keys.size else np.zeros(1, dtype=np.int32), dtype=np.int32)
        o = np.zeros((n, self.head_dim_v), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = _load().oracle_partial_keysets(ctypes.byref(self._s), n, _iptr(rows3), _iptr(ind), _iptr(keys),
                                            _dptr(o), _dptr(lse))
        if rc != 0:
            raise ValueError(f"oracle_partial_keysets failed with code {rc}")
        return o, lse

    def attention_rows(self, rows3: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
        """Unsplit attention for rows (b, i, h) (default: every row)."""
        if rows3 is None:
            rows3 = self.all_rows()
        rows3 = np.ascontiguousarray(rows3, dtype=np.int32).reshape(-1, 3)
        n = rows3.shape[0]
        o = np.zeros((n, self.head_dim_v), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        rc = _load().oracle_attention_rows(ctypes.byref(self._s), n, _iptr(rows3), _dptr(o), _dptr(lse))
        if rc != 0:
            raise ValueError(f"oracle_attention_rows failed with code {rc}")
        return o, lse


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """Float64 value of each 8-bit E4M3 code (the decoder the attention uses)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    out = np.zeros(codes.size, dtype=np.float64)
    _load().oracle_e4m3_values(codes.size, codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), _dptr(out))
    return out


def merge(o_parts: np.ndarray, lse_parts: np.ndarray) -> Tuple[np.ndarray, float]:
    """LiquidCP Eq. (1) over n partial states: o_parts [n, d], lse_parts [n]."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _load().oracle_merge(n, d, _dptr(o_parts), _dptr(lse_parts), _dptr(o), _dptr(lse))
    return o, float(lse[0])


def merge_rows(state_indptr: np.ndarray, o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge rows x over partial states state_indptr[x] .. state_indptr[x+1]-1."""
    ind = np.ascontiguousarray(state_indptr, dtype=np.int32)
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    nrows = len(ind) - 1
    d = o_parts.shape[1]
    o = np.zeros((nrows, d), dtype=np.float64)
    lse = np.zeros(nrows, dtype=np.float64)
    _load().oracle_merge_rows(nrows, d, _iptr(ind), _dptr(o_parts), _dptr(lse_parts), _dptr(o),
                              _dptr(lse))
    return o, lse


def split_bounds(seq_len: int, page_size: int, n_splits: int) -> List[Tuple[int, int]]:
    """Key ranges of a history cut into ``n_splits`` page-aligned, contiguous
    ranges: with N pages, range r gets floor(N/n) pages plus one more for the
    first N mod n ranges (the 59/59/58 cut of LiquidCP Figure 8).  Ranges past
    the history are empty."""
    n_pages = -(-seq_len // page_size)
    base, extra = divmod(n_pages, n_splits)
    out = []
    page = 0
    for r in range(n_splits):
        cnt = base + (1 if r < extra else 0)
        kb = page * page_size
        ke = min((page + cnt) * page_size, seq_len)
        out.append((kb, max(kb, ke)))
        page += cnt
    return out


def interleaved_split_keys(seq_len: int, block: int, n_splits: int) -> List[np.ndarray]:
    """Keys of each KV shard under Helix Parallelism's staggered round-robin
    placement (Section 2.3, step 4): the history is cut into blocks of ``block``
    tokens, block m goes to shard m mod n_splits.  Returns n_splits ascending key
    arrays; shards that receive no block are empty."""
    out = []
    for r in range(n_splits):
        keys = [j for m in range(r, -(-seq_len // block), n_splits)
                for j in range(m * block, min((m + 1) * block, seq_len))]
        out.append(np.array(keys, dtype=np.int32))
    return out


def problem_from_workload(wl, *, with_v: bool = True) -> Problem:
    """Oracle problem holding the whole of a (small) workload on the host."""
    s = wl.spec
    return Problem(kind=s.kind, q=wl.q_host(), k=wl.k_host(), v=wl.v_host() if with_v else None,
                   page_table=wl.page_table, seq_lens=wl.seq_lens, qo_indptr=wl.qo_indptr,
                   num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads,
                   head_dim_qk=s.head_dim_qk, head_dim_v=s.head_dim_v, page_size=s.page_size,
                   scale=s.scale, k_scale=getattr(s, "k_scale", 1.0), v_scale=getattr(s, "v_scale", 1.0))


def subproblem_for_group(wl, b: int, kv_head: int) -> Problem:
    """Oracle problem for one request and one KV head of a large workload.

    Only the pages of request ``b`` (and, for GQA, KV head ``kv_head``) are
    regenerated on the host; the sub-problem has batch 1, one KV head, the
    group's query heads and an identity page table.  Output row (i, h_local)
    of the sub-problem is row (i, kv_head*g + h_local) of the full problem.
    """
    s = wl.spec
    L = int(wl.seq_lens[b])
    n_pages = -(-L // s.page_size)
    pages = [int(p) for p in wl.page_table[b, :n_pages]]
    q_all = wl.q_host()
    qs, qe = int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1])
    if s.kind == "gqa":
        g = s.num_q_heads // s.num_kv_heads
        k = wl.kv_pages_host("k", pages, kv_head)[:, None]
        v = wl.kv_pages_host("v", pages, kv_head)[:, None]
        q = q_all[qs:qe, kv_head * g:(kv_head + 1) * g]
        hq = g
    else:
        k = wl.kv_pages_host("k", pages)
        v = None
        q = q_all[qs:qe]
        hq = s.num_q_heads
    return Problem(kind=s.kind, q=q, k=k, v=v, page_table=np.arange(n_pages, dtype=np.int32)[None],
                   seq_lens=np.array([L], dtype=np.int32),
                   qo_indptr=np.array([0, qe - qs], dtype=np.int32), num_q_heads=hq,
                   num_kv_heads=1, head_dim_qk=s.head_dim_qk, head_dim_v=s.head_dim_v,
                   page_size=s.page_size, scale=s.scale, k_scale=getattr(s, "k_scale", 1.0),
                   v_scale=getattr(s, "v_scale", 1.0))
