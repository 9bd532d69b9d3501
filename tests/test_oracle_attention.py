"""Pins for the float64 oracle's attention (partial states over key subsets).

Each test checks the oracle against something other than itself:
  * library routines: torch's scaled_dot_product_attention (float64, math
    backend) for GQA decode, MLA decode (D_qk != D_v) and causal prefill;
    torch.logsumexp for the LSE;
  * closed forms (one key, zero query, identical keys, one dominant key);
  * invariants (page permutation, key shift, chunk rows = prefill rows).
A plausible slip -- a dropped scale, a wrong KV-head map, a transposed
operand, a causal off-by-one, a wrong page index or LSE offset -- fails one.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _make_gqa(rng, *, B, Hq, Hkv, D, P, lens, q_lens=None, dtype="f32", shuffle=True, extra_pages=3):
    lens = np.asarray(lens, dtype=np.int32)
    q_lens = np.ones_like(lens) if q_lens is None else np.asarray(q_lens, dtype=np.int32)
    npg = (lens + P - 1) // P
    total = int(npg.sum()) + extra_pages
    perm = rng.permutation(total) if shuffle else np.arange(total)
    pt = np.full((B, int(npg.max())), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        pt[b, :npg[b]] = perm[off:off + npg[b]]
        off += npg[b]
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = rng.standard_normal((int(qo[-1]), Hq, D)).astype(np.float32)
    k = rng.standard_normal((total, Hkv, P, D)).astype(np.float32)
    v = rng.standard_normal((total, Hkv, P, D)).astype(np.float32)
    if dtype == "bf16":
        q, k, v = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    return dict(q=q, k=k, v=v, page_table=pt, seq_lens=lens, qo_indptr=qo)


def _problem(kind, arrs, Hq, Hkv, Dqk, Dv, P, scale):
    return oracle.Problem(kind=kind, q=arrs["q"], k=arrs["k"], v=arrs.get("v"),
                          page_table=arrs["page_table"], seq_lens=arrs["seq_lens"],
                          qo_indptr=arrs["qo_indptr"], num_q_heads=Hq, num_kv_heads=Hkv,
                          head_dim_qk=Dqk, head_dim_v=Dv, page_size=P, scale=scale)


def _as_f64(a):
    return _bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def _gather_gqa(arrs, b, P):
    """Contiguous [Hkv, L, D] K and V of request b (plain numpy indexing)."""
    L = int(arrs["seq_lens"][b])
    pages = arrs["page_table"][b, :(L + P - 1) // P]
    k = _as_f64(arrs["k"])[pages]            # [np, Hkv, P, D]
    v = _as_f64(arrs["v"])[pages]
    k = np.concatenate(list(k), axis=1)[:, :L]   # [Hkv, L, D]
    v = np.concatenate(list(v), axis=1)[:, :L]
    return k, v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gqa_decode_matches_sdpa(dtype):
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, P = 4, 8, 2, 16, 4
    lens = [1, 7, 33, 64]
    arrs = _make_gqa(rng, B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dtype=dtype)
    scale = 0.37
    prob = _problem("gqa", arrs, Hq, Hkv, D, D, P, scale)
    o, lse = prob.attention_rows()
    o = o.reshape(B, Hq, D)
    lse = lse.reshape(B, Hq)
    q = _as_f64(arrs["q"])
    for b in range(B):
        k, v = _gather_gqa(arrs, b, P)
        qt = torch.from_numpy(q[b])[None, :, None, :]            # [1, Hq, 1, D]
        kt = torch.from_numpy(k)[None]                            # [1, Hkv, L, D]
        vt = torch.from_numpy(v)[None]
        ref = F.scaled_dot_product_attention(qt, kt, vt, scale=scale, enable_gqa=True)[0, :, 0]
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=1e-12, atol=1e-12)
        kt_rep = kt.repeat_interleave(Hq // Hkv, dim=1)
        ref_lse = torch.logsumexp(scale * (qt @ kt_rep.transpose(-1, -2)), dim=-1)[0, :, 0]
        np.testing.assert_allclose(lse[b], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_mla_matches_sdpa_with_shared_latent():
    """Absorbed MLA: keys are the whole latent row, values its first D_v columns."""
    rng = np.random.default_rng(12)
    B, Hq, Dqk, Dv, P = 3, 4, 24, 16, 4
    lens = np.array([5, 17, 40], dtype=np.int32)
    npg = (lens + P - 1) // P
    total = int(npg.sum()) + 2
    perm = rng.permutation(total)
    pt = np.full((B, int(npg.max())), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        pt[b, :npg[b]] = perm[off:off + npg[b]]
        off += npg[b]
    q = rng.standard_normal((B, Hq, Dqk)).astype(np.float32)
    ckv = rng.standard_normal((total, P, Dqk)).astype(np.float32)
    arrs = dict(q=q, k=ckv, v=None, page_table=pt, seq_lens=lens,
                qo_indptr=np.arange(B + 1, dtype=np.int32))
    scale = 1.0 / math.sqrt(12.0)
    prob = _problem("mla", arrs, Hq, 1, Dqk, Dv, P, scale)
    o, lse = prob.attention_rows()
    o = o.reshape(B, Hq, Dv)
    for b in range(B):
        rows = ckv.astype(np.float64)[pt[b, :npg[b]]].reshape(-1, Dqk)[:lens[b]]
        kt = torch.from_numpy(rows)[None, None]           # [1, 1, L, 24]
        vt = torch.from_numpy(rows[:, :Dv])[None, None]   # [1, 1, L, 16]
        qt = torch.from_numpy(q[b].astype(np.float64))[None, :, None, :]
        ref = F.scaled_dot_product_attention(qt, kt, vt, scale=scale, enable_gqa=True)[0, :, 0]
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_causal_prefill_matches_sdpa_and_chunk_rows_match_prefill_rows():
    """q_len = L is causal prefill (SDPA is_causal); a chunk of the last q rows
    appended after a history sees exactly what those prefill rows see."""
    rng = np.random.default_rng(13)
    Hq, Hkv, D, P, L, C = 4, 2, 8, 4, 29, 9
    full = _make_gqa(rng, B=1, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=[L], q_lens=[L])
    scale = 0.5
    prob_full = _problem("gqa", full, Hq, Hkv, D, D, P, scale)
    o_full, lse_full = prob_full.attention_rows()
    o_full = o_full.reshape(L, Hq, D)
    k, v = _gather_gqa(full, 0, P)
    qt = torch.from_numpy(full["q"].astype(np.float64)).permute(1, 0, 2)[None]   # [1, Hq, L, D]
    ref = F.scaled_dot_product_attention(qt, torch.from_numpy(k)[None], torch.from_numpy(v)[None],
                                         scale=scale, is_causal=True, enable_gqa=True)[0]
    np.testing.assert_allclose(o_full, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)

    chunk = dict(full)
    chunk["q"] = full["q"][L - C:]
    chunk["qo_indptr"] = np.array([0, C], dtype=np.int32)
    prob_chunk = _problem("gqa", chunk, Hq, Hkv, D, D, P, scale)
    o_c, lse_c = prob_chunk.attention_rows()
    np.testing.assert_array_equal(o_c.reshape(C, Hq, D), o_full[L - C:])
    np.testing.assert_array_equal(lse_c.reshape(C, Hq), lse_full.reshape(L, Hq)[L - C:])


def test_page_permutation_invariance_is_bitwise():
    rng = np.random.default_rng(14)
    B, Hq, Hkv, D, P = 2, 4, 2, 8, 4
    arrs = _make_gqa(rng, B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=[13, 30], shuffle=False)
    prob = _problem("gqa", arrs, Hq, Hkv, D, D, P, 0.3)
    o1, l1 = prob.attention_rows()
    total = arrs["k"].shape[0]
    perm = rng.permutation(total)             # new physical slot of each old page
    k2 = np.empty_like(arrs["k"])
    v2 = np.empty_like(arrs["v"])
    k2[perm] = arrs["k"]
    v2[perm] = arrs["v"]
    pt2 = np.where(arrs["page_table"] >= 0, perm[np.maximum(arrs["page_table"], 0)], -1).astype(np.int32)
    arrs2 = dict(arrs, k=k2, v=v2, page_table=pt2)
    o2, l2 = _problem("gqa", arrs2, Hq, Hkv, D, D, P, 0.3).attention_rows()
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_closed_forms():
    rng = np.random.default_rng(15)
    Hq, Hkv, D, P = 2, 1, 8, 4
    # one key: out = v_0, lse = s_0
    a = _make_gqa(rng, B=1, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=[1])
    o, lse = _problem("gqa", a, Hq, Hkv, D, D, P, 0.25).attention_rows()
    k0 = a["k"][a["page_table"][0, 0], 0, 0].astype(np.float64)
    v0 = a["v"][a["page_table"][0, 0], 0, 0].astype(np.float64)
    for h in range(Hq):
        np.testing.assert_array_equal(o[h], v0)
        assert lse[h] == pytest.approx(0.25 * float(a["q"][0, h].astype(np.float64) @ k0), abs=1e-14)
    # zero query: uniform weights, out = mean(V), lse = ln L
    L = 37
    a = _make_gqa(rng, B=1, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=[L])
    a["q"][:] = 0
    o, lse = _problem("gqa", a, Hq, Hkv, D, D, P, 0.25).attention_rows()
    _, v = _gather_gqa(a, 0, P)
    np.testing.assert_allclose(o[0], v[0].mean(axis=0), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(L), rtol=0, atol=1e-13)
    # identical keys: lse = s + ln L, out = mean(V)
    a = _make_gqa(rng, B=1, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=[L])
    a["k"][:] = a["k"][0, 0, 0]
    o, lse = _problem("gqa", a, Hq, Hkv, D, D, P, 0.25).attention_rows()
    s = 0.25 * a["q"][0].astype(np.float64) @ a["k"][0, 0, 0].astype(np.float64)
    np.testing.assert_allclose(lse, s + math.log(L), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[1], _gather_gqa(a, 0, P)[1][0].mean(axis=0), rtol=1e-13, atol=1e-14)
    # one dominant key: out ~= v_j*
    a = _make_gqa(rng, B=1, Hq=1, Hkv=1, D=D, P=P, lens=[L])
    jstar = 22
    kk, vv = _gather_gqa(a, 0, P)
    a["q"][0, 0] = (60.0 * kk[0, jstar] / np.linalg.norm(kk[0, jstar])).astype(np.float32)
    a["k"][:] *= 0.01
    page = a["page_table"][0, jstar // P]
    a["k"][page, 0, jstar % P] = kk[0, jstar].astype(np.float32)
    o, _ = _problem("gqa", a, 1, 1, D, D, P, 1.0).attention_rows()
    np.testing.assert_allclose(o[0], _gather_gqa(a, 0, P)[1][0, jstar], rtol=0, atol=1e-9)


def test_key_shift_moves_lse_only():
    """k_j -> k_j + delta for every j adds scale*<q,delta> to every score:
    lse moves by that amount and the output does not change."""
    rng = np.random.default_rng(16)
    Hq, Hkv, D, P = 2, 1, 8, 4
    a = _make_gqa(rng, B=1, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=[21])
    a["q"] = np.round(a["q"] * 4) / 4
    a["k"] = np.round(a["k"] * 4) / 4
    delta = np.array([0.5, -1, 0, 0.25, 1, 0, -0.5, 2], dtype=np.float32)
    o1, l1 = _problem("gqa", a, Hq, Hkv, D, D, P, 0.5).attention_rows()
    a2 = dict(a, k=(a["k"] + delta).astype(np.float32))
    o2, l2 = _problem("gqa", a2, Hq, Hkv, D, D, P, 0.5).attention_rows()
    shift = 0.5 * a["q"][0].astype(np.float64) @ delta.astype(np.float64)
    np.testing.assert_allclose(l2 - l1, shift, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)


def test_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(17)
    a = _make_gqa(rng, B=2, Hq=4, Hkv=2, D=8, P=4, lens=[9, 14], dtype="bf16")
    o1, l1 = _problem("gqa", a, 4, 2, 8, 8, 4, 0.3).attention_rows()
    f = {k: (_bits_to_f64(v).astype(np.float32) if isinstance(v, np.ndarray) and v.dtype == np.uint16 else v)
         for k, v in a.items()}
    o2, l2 = _problem("gqa", f, 4, 2, 8, 8, 4, 0.3).attention_rows()
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_partial_key_ranges_and_empty_subset():
    rng = np.random.default_rng(18)
    a = _make_gqa(rng, B=1, Hq=2, Hkv=1, D=8, P=4, lens=[19])
    prob = _problem("gqa", a, 2, 1, 8, 8, 4, 0.4)
    # keys [5, 12) equal attention over a problem holding only those keys
    o, lse = prob.partial_rows(np.array([[0, 0, 1, 5, 12], [0, 0, 1, 19, 40]]))
    assert lse[1] == -math.inf and not o[1].any()
    k, v = _gather_gqa(a, 0, 4)
    qt = torch.from_numpy(a["q"][0, 1].astype(np.float64))[None, None, None]
    ref = F.scaled_dot_product_attention(qt, torch.from_numpy(k[:, 5:12])[None],
                                         torch.from_numpy(v[:, 5:12])[None], scale=0.4)
    np.testing.assert_allclose(o[0], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_invalid_rows_and_pages_raise():
    rng = np.random.default_rng(19)
    a = _make_gqa(rng, B=1, Hq=2, Hkv=1, D=8, P=4, lens=[9])
    prob = _problem("gqa", a, 2, 1, 8, 8, 4, 0.4)
    with pytest.raises(ValueError):
        prob.attention_rows(np.array([[1, 0, 0]]))
    a["page_table"][0, 1] = 10_000
    with pytest.raises(ValueError):
        _problem("gqa", a, 2, 1, 8, 8, 4, 0.4).attention_rows()
