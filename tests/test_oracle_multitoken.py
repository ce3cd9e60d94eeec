"""Pins for the oracle's multi-token decode attention (CPU only).

Several new query tokens per request (verifying speculative drafts): the
pages say nothing about it; the reading taken is that the n new tokens are
the request's last n positions, already in the cache, and that query token i
attends causally to positions 0 .. L - n + i.  Pins: dense fp64 softmax
attention with a causal mask built from torch primitives over the gathered
dequantised tensors (library); n = 1 against the single-token oracle; each
query against the single-token oracle over its visible prefix; closed forms
(a query that sees one position returns that position's value; one that sees
none returns zeros); invariance under a random re-placement of pages.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from test_oracle_attention import bf16_torch, dequant_torch, populate, small_ragged


def causal_dense_reference(q_bits, k_cache, v_cache, ks, vs, block_table, seq_lens, sigma):
    """softmax(sigma q K^T + causal mask) V from torch primitives; q [B][n][Hq][D]."""
    B, n, Hq, D = q_bits.shape
    Hkv, ps = k_cache.shape[1], k_cache.shape[2]
    g = Hq // Hkv
    if k_cache.dtype == np.uint16:
        K, V = bf16_torch(k_cache), bf16_torch(v_cache)
    else:
        K, V = dequant_torch(k_cache, ks), dequant_torch(v_cache, vs)
    q = bf16_torch(q_bits)
    out = torch.zeros(B, n, Hq, D, dtype=torch.float64)
    for r in range(B):
        L = int(seq_lens[r])
        pages = torch.from_numpy(block_table[r, :(L + ps - 1) // ps].astype(np.int64))
        Kr = K[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L].repeat_interleave(g, dim=0)
        Vr = V[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L].repeat_interleave(g, dim=0)
        s = torch.einsum("ihd,hld->ihl", q[r], Kr) * float(np.float32(sigma))   # [n][Hq][L]
        pos = torch.arange(L).view(1, 1, L)
        last = (L - n + torch.arange(n)).view(n, 1, 1)                          # last visible position
        s = s.masked_fill(pos > last, float("-inf"))
        seen = (last >= 0).view(n, 1, 1).to(torch.float64)
        p = torch.softmax(s, dim=-1).nan_to_num(0.0) * seen
        out[r] = torch.einsum("ihl,hld->ihd", p, Vr)
    return out.numpy()


def multi_case(n, g=4, ps=16, lens=(1, 3, 15, 16, 17, 100, 257), seed=7, bf16=False):
    w, hv = small_ragged(seed=seed, g=g, ps=ps, lens=lens)
    kc, vc = populate(w, hv, bf16=bf16)
    rng = np.random.default_rng(seed + 1)
    q = W.normal_bf16(rng, (w.batch, n, w.num_q_heads, w.head_dim))
    return w, hv, kc, vc, q


@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("bf16", [False, True])
def test_multi_matches_dense_causal_attention(n, bf16):
    w, hv, kc, vc, q = multi_case(n, bf16=bf16)
    got = oracle.decode_attn_multi(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                                   w.softmax_scale)
    ref = causal_dense_reference(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                                 w.softmax_scale)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_one_query_token_is_the_single_token_oracle():
    w, hv, kc, vc, q = multi_case(1, g=8)
    got = oracle.decode_attn_multi(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                                   w.softmax_scale)
    ref = oracle.decode_attn(q[:, 0], kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                             w.softmax_scale)
    assert np.array_equal(got[:, 0], ref)


def test_each_query_is_a_single_token_decode_over_its_prefix():
    n = 4
    w, hv, kc, vc, q = multi_case(n, g=2)
    got = oracle.decode_attn_multi(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                                   w.softmax_scale)
    for i in range(n):
        seen = np.maximum(w.seq_lens - n + 1 + i, 0).astype(np.int32)
        ref = oracle.decode_attn(q[:, i], kc, vc, hv.k_scale, hv.v_scale, w.block_table, seen,
                                 w.softmax_scale)
        assert np.array_equal(got[:, i], ref), i


def test_short_requests_closed_forms():
    """A request of L = 2 with n = 4: queries 0, 1 see nothing (zeros), query 2
    sees position 0 only (its value), query 3 sees positions 0 and 1."""
    n = 4
    w, hv, kc, vc, q = multi_case(n, g=2, lens=(2, 40))
    got = oracle.decode_attn_multi(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                                   w.softmax_scale)
    assert np.all(got[0, 0] == 0.0) and np.all(got[0, 1] == 0.0)
    ps = w.page_size
    page0 = w.block_table[0, 0]
    v0 = oracle.e4m3_decode(vc[page0, :, 0, :]) * hv.v_scale[:, None]     # [Hkv][D]
    assert np.array_equal(got[0, 2], np.repeat(v0, w.group, axis=0))
    assert np.all(got[0, 3] != 0.0)
    assert ps > 2


def test_zeroed_requests_and_page_placement():
    n = 3
    w, hv, kc, vc, q = multi_case(n, g=4)
    abort = np.zeros(w.batch, np.uint8)
    abort[2] = 1
    bt = w.block_table.copy()
    bt[4, 1] = w.num_pages                  # a page id out of range
    got = oracle.decode_attn_multi(q, kc, vc, hv.k_scale, hv.v_scale, bt, w.seq_lens,
                                   w.softmax_scale, abort)
    assert np.all(got[2] == 0.0) and np.all(got[4] == 0.0)
    assert np.any(got[5] != 0.0)
    # the same pages moved to other physical places: bit-identical
    perm = np.random.default_rng(3).permutation(w.num_pages)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    a = oracle.decode_attn_multi(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table, w.seq_lens,
                                 w.softmax_scale)
    b = oracle.decode_attn_multi(q, kc2, vc2, hv.k_scale, hv.v_scale, bt2, w.seq_lens,
                                 w.softmax_scale)
    assert np.array_equal(a, b)
