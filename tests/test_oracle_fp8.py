"""Pins for the oracle's FP8 KV cache (8-bit E4M3 codes, one scale per
tensor: the FP8 KV cache of SPLASH Appendix C.1).

Pins: the decoder against torch's float8_e4m3fn on all 256 codes (a library
routine), attention over E4M3 keys and values against torch's float64
scaled-dot-product attention over the dequantized tensors (dequantized by
torch), and the scales' closed-form effects (k_scale multiplies the scores,
v_scale the outputs, the LSE moving accordingly).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests import test_oracle_attention as TA


def test_e4m3_decoder_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_values(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.tolist() == np.isnan(ours).tolist() and nan.sum() == 2       # S.1111.111
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _fp8_codes(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * 3.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _deq(codes, s):
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64) * s


def _fp8_problem(rng, lens, q_lens, Hq=8, Hkv=2, D=16, P=4, ks=0.37, vs=0.61, scale=0.25):
    arrs = TA._make_gqa(rng, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, q_lens=q_lens, dtype="bf16")
    arrs["k"] = _fp8_codes(rng, arrs["k"].shape)
    arrs["v"] = _fp8_codes(rng, arrs["v"].shape)
    prob = oracle.Problem(kind="gqa", q=arrs["q"], k=arrs["k"], v=arrs["v"], page_table=arrs["page_table"],
                          seq_lens=arrs["seq_lens"], qo_indptr=arrs["qo_indptr"], num_q_heads=Hq,
                          num_kv_heads=Hkv, head_dim_qk=D, head_dim_v=D, page_size=P, scale=scale,
                          k_scale=ks, v_scale=vs)
    return arrs, prob


def test_fp8_attention_matches_sdpa_on_dequantized_cache():
    rng = np.random.default_rng(51)
    P, Hq, Hkv, D = 4, 8, 2, 16
    lens, q_lens = [37, 9], [3, 1]
    arrs, prob = _fp8_problem(rng, lens, q_lens)
    o, lse = prob.attention_rows()
    o = o.reshape(-1, Hq, D)
    lse = lse.reshape(-1, Hq)
    q_all = TA._as_f64(arrs["q"])
    row = 0
    for b, (L, ql) in enumerate(zip(lens, q_lens)):
        pages = arrs["page_table"][b, :(L + P - 1) // P]
        k = torch.cat(list(_deq(arrs["k"], 0.37)[pages]), dim=1)[:, :L]      # [Hkv, L, D]
        v = torch.cat(list(_deq(arrs["v"], 0.61)[pages]), dim=1)[:, :L]
        q = torch.from_numpy(q_all[row:row + ql]).permute(1, 0, 2)            # [Hq, ql, D]
        kk = k.repeat_interleave(Hq // Hkv, dim=0)
        vv = v.repeat_interleave(Hq // Hkv, dim=0)
        # row i sits at position L - ql + i: it sees keys 0 .. L - ql + i
        mask = torch.arange(L)[None, :] <= (L - ql + torch.arange(ql))[:, None]
        ref = F.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=0.25)
        s = 0.25 * q @ kk.transpose(1, 2)
        ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
        np.testing.assert_allclose(o[row:row + ql], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(lse[row:row + ql], ref_lse.permute(1, 0).numpy(), rtol=0, atol=1e-10)
        row += ql


def test_fp8_scales_closed_forms():
    rng = np.random.default_rng(52)
    arrs, p1 = _fp8_problem(rng, [30], [1], ks=1.0, vs=1.0, scale=0.2)
    mk = lambda **kw: oracle.Problem(kind="gqa", q=arrs["q"], k=arrs["k"], v=arrs["v"],
                                     page_table=arrs["page_table"], seq_lens=arrs["seq_lens"],
                                     qo_indptr=arrs["qo_indptr"], num_q_heads=8, num_kv_heads=2,
                                     head_dim_qk=16, head_dim_v=16, page_size=4, **kw)
    o1, l1 = p1.attention_rows()
    # k_scale 2 with score scale 0.1 is the same softmax as k_scale 1 with 0.2
    o2, l2 = mk(scale=0.1, k_scale=2.0, v_scale=1.0).attention_rows()
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    # v_scale multiplies the output and leaves the LSE
    o3, l3 = mk(scale=0.2, k_scale=1.0, v_scale=-2.5).attention_rows()
    np.testing.assert_allclose(o3, -2.5 * o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(l3, l1)


def test_fp8_mla_attention_matches_sdpa_on_dequantized_latent():
    """Absorbed MLA over an E4M3 latent cache: each latent row is both the key (all 576
    columns) and, through its first 512 columns, the value, so both roles take k_scale
    (v_scale must not enter).  Against torch's float64 SDPA over the dequantized latent."""
    rng = np.random.default_rng(53)
    P, Hq, Dqk, Dv = 4, 4, 24, 16
    lens, q_lens = [19, 6], [2, 1]
    B = len(lens)
    npg = [(L + P - 1) // P for L in lens]
    total = sum(npg) + 2
    perm = rng.permutation(total)
    pt = np.full((B, max(npg)), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        pt[b, :npg[b]] = perm[off:off + npg[b]]
        off += npg[b]
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = TA._bf16_bits(rng.standard_normal((int(qo[-1]), Hq, Dqk)).astype(np.float32))
    lat = _fp8_codes(rng, (total, P, Dqk))
    ks, scale = 0.29, 0.3
    prob = oracle.Problem(kind="mla", q=q, k=lat, v=None, page_table=pt, seq_lens=np.asarray(lens, np.int32),
                          qo_indptr=qo, num_q_heads=Hq, num_kv_heads=1, head_dim_qk=Dqk, head_dim_v=Dv,
                          page_size=P, scale=scale, k_scale=ks, v_scale=123.0)
    o, lse = prob.attention_rows()
    o = o.reshape(-1, Hq, Dv)
    lse = lse.reshape(-1, Hq)
    q_all = TA._as_f64(q)
    row = 0
    for b, (L, ql) in enumerate(zip(lens, q_lens)):
        k = torch.cat(list(_deq(lat, ks)[pt[b, :npg[b]]]), dim=0)[:L]            # [L, Dqk]
        v = k[:, :Dv]
        qq = torch.from_numpy(q_all[row:row + ql]).permute(1, 0, 2)               # [Hq, ql, Dqk]
        mask = torch.arange(L)[None, :] <= (L - ql + torch.arange(ql))[:, None]
        ref = F.scaled_dot_product_attention(qq, k[None].expand(Hq, L, Dqk), v[None].expand(Hq, L, Dv),
                                             attn_mask=mask, scale=scale)
        s = scale * qq @ k.T[None]
        ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
        np.testing.assert_allclose(o[row:row + ql], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(lse[row:row + ql], ref_lse.permute(1, 0).numpy(), rtol=0, atol=1e-10)
        row += ql
