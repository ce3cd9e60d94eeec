"""Pins for the oracle's append, paged decode attention and tag check (CPU only).

Passages followed:
  * FP8 e4m3 KV cache, converted on read by the attention kernel -- blog post
    "Smaller, faster, safer", section on quantising the KV cache (page 1);
    page 3 section "FP8 省的不仅是显存".
  * paged attention over physical pages shared by many requests; each page
    carries a tag bumped on reallocation; a separate batched check before
    decode reads aborts a request on any mismatch -- page 2 section "KV Cache
    完整性检查", page 3 section "一个不能出错的共享缓存".

Pins used: torch's float8_e4m3fn conversion (library), dense fp64 softmax
attention built from torch primitives over the gathered tensors (library),
closed forms (one token, identical keys), invariance under a random
re-placement of physical pages, and brute-force loops for the tag check.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def dequant_torch(codes: np.ndarray, scale_per_head: np.ndarray) -> torch.Tensor:
    """[..., Hkv, ps, D] codes -> fp64 through torch's float8 dtype."""
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)
    s = torch.from_numpy(scale_per_head.astype(np.float64)).view(1, -1, 1, 1)
    return v * s


def bf16_torch(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def dense_reference(q_bits, k_cache, v_cache, ks, vs, block_table, seq_lens, sigma):
    """softmax(sigma * q K^T) V per request/head, from torch primitives."""
    B, Hq, D = q_bits.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    ps = k_cache.shape[2]
    if k_cache.dtype == np.uint16:
        K = bf16_torch(k_cache)
        V = bf16_torch(v_cache)
    else:
        K = dequant_torch(k_cache, ks)
        V = dequant_torch(v_cache, vs)
    q = bf16_torch(q_bits)
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for r in range(B):
        L = int(seq_lens[r])
        pages = torch.from_numpy(block_table[r, :(L + ps - 1) // ps].astype(np.int64))
        Kr = K[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L]   # [Hkv][L][D]
        Vr = V[pages].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L]
        Kr = Kr.repeat_interleave(g, dim=0)
        Vr = Vr.repeat_interleave(g, dim=0)
        s = torch.einsum("hd,hld->hl", q[r], Kr) * float(np.float32(sigma))
        out[r] = torch.einsum("hl,hld->hd", torch.softmax(s, dim=-1), Vr)
    return out.numpy()


def populate(w: W.Workload, hv: W.HostValues, bf16: bool = False):
    dt = np.uint16 if bf16 else np.uint8
    rng = np.random.default_rng(99)
    kc = rng.integers(0, 0x7F, size=w.cache_shape(), dtype=np.uint8).astype(dt)   # finite junk
    vc = rng.integers(0, 0x7F, size=w.cache_shape(), dtype=np.uint8).astype(dt)
    oracle.append(kc, vc, hv.k_prefill, hv.v_prefill, w.prefill_slot_mapping(),
                  hv.k_scale, hv.v_scale, page_size=w.page_size)
    oracle.append(kc, vc, hv.k_new, hv.v_new, w.append_slot_mapping(),
                  hv.k_scale, hv.v_scale, page_size=w.page_size)
    return kc, vc


def small_ragged(seed=5, g=4, ps=16, lens=(1, 15, 16, 17, 100, 257)):
    rng = np.random.default_rng(seed)
    Hkv, D = 2, 128
    seq = np.array(lens, np.int32)
    pages = [(int(L) + ps - 1) // ps for L in seq]
    N = int(sum(pages) * 1.5) + 3
    perm = rng.permutation(N).astype(np.int32)
    bt = np.full((len(seq), max(pages)), -1, np.int32)
    at = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[at:at + p]
        at += p
    tags = rng.integers(0, 2**32, N, dtype=np.uint64).astype(np.uint32)
    exp = np.zeros_like(bt, dtype=np.uint32)
    exp[bt >= 0] = tags[bt[bt >= 0]]
    w = W.Workload("small", len(seq), Hkv * g, Hkv, D, ps, N, seq, bt, tags, exp,
                   1.0 / math.sqrt(D), seed, outlier_frac=0.01)
    return w, W.host_values(w)


# ------------------------------------------------------------------ append

def test_append_codes_match_torch_float8_and_touch_only_their_slots():
    w, hv = small_ragged()
    canary = np.uint8(0xA5)
    kc = np.full(w.cache_shape(), canary, np.uint8)
    vc = np.full(w.cache_shape(), canary, np.uint8)
    slots = w.prefill_slot_mapping()
    oracle.append(kc, vc, hv.k_prefill, hv.v_prefill, slots, hv.k_scale, hv.v_scale,
                  page_size=w.page_size)
    # library quantisation of the same fp32 quotients
    for cache, src, sc in ((kc, hv.k_prefill, hv.k_scale), (vc, hv.v_prefill, hv.v_scale)):
        quot = (W.bf16_bits_to_f32(src) / sc[None, :, None]).astype(np.float32)
        lib = torch.from_numpy(np.clip(quot, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        page, off = slots // w.page_size, slots % w.page_size
        got = cache[page, :, off, :]                       # [T][Hkv][D]
        assert np.array_equal(got, lib)
        mask = np.ones(w.cache_shape(), bool)
        mask[page, :, off, :] = False
        assert np.all(cache[mask] == canary)


def test_append_saturates_outliers():
    w, hv = small_ragged()
    big = np.full_like(hv.k_new, W.f32_to_bf16_bits(np.array([1e6], np.float32))[0])
    kc = np.zeros(w.cache_shape(), np.uint8)
    vc = np.zeros(w.cache_shape(), np.uint8)
    oracle.append(kc, vc, big, big ^ np.uint16(0x8000),                # +1e6 and -1e6
                  w.append_slot_mapping(), hv.k_scale, hv.v_scale, page_size=w.page_size)
    slots = w.append_slot_mapping()
    assert np.all(kc[slots // w.page_size, :, slots % w.page_size, :] == 0x7E)
    assert np.all(vc[slots // w.page_size, :, slots % w.page_size, :] == 0xFE)


def test_append_skips_negative_out_of_range_and_aborted():
    w, hv = small_ragged()
    kc = np.zeros(w.cache_shape(), np.uint8)
    vc = np.zeros(w.cache_shape(), np.uint8)
    slots = w.append_slot_mapping().copy()
    slots[0] = -1
    slots[1] = w.num_pages * w.page_size          # one past the end
    abort = np.zeros(w.batch, np.uint8)
    abort[2] = 1
    oracle.append(kc, vc, hv.k_new, hv.v_new, slots, hv.k_scale, hv.v_scale, abort,
                  page_size=w.page_size)
    written = np.zeros(w.batch, bool)
    for r in range(w.batch):
        s = w.append_slot_mapping()[r]
        written[r] = np.any(kc[s // w.page_size, :, s % w.page_size, :] != 0)
    assert not written[0] and not written[1] and not written[2]
    assert written[3:].all()


def test_append_bf16_cache_is_a_copy():
    w, hv = small_ragged()
    kc = np.zeros(w.cache_shape(), np.uint16)
    vc = np.zeros(w.cache_shape(), np.uint16)
    slots = w.prefill_slot_mapping()
    oracle.append(kc, vc, hv.k_prefill, hv.v_prefill, slots, None, None, page_size=w.page_size)
    assert np.array_equal(kc[slots // w.page_size, :, slots % w.page_size, :], hv.k_prefill)
    assert np.array_equal(vc[slots // w.page_size, :, slots % w.page_size, :], hv.v_prefill)


# --------------------------------------------------------------- attention

@pytest.mark.parametrize("g,ps", [(1, 16), (2, 64), (4, 16), (8, 32)])
@pytest.mark.parametrize("bf16", [False, True])
def test_attention_matches_dense_torch_softmax(g, ps, bf16):
    w, hv = small_ragged(g=g, ps=ps)
    kc, vc = populate(w, hv, bf16)
    ours = oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                              w.seq_lens, w.softmax_scale)
    ref = dense_reference(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                          w.seq_lens, w.softmax_scale)
    assert np.allclose(ours, ref, rtol=1e-11, atol=1e-12)


def test_attention_tiny_workload_matches_dense():
    w = W.make("tiny")
    hv = W.host_values(w)
    kc, vc = populate(w, hv)
    ours = oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                              w.seq_lens, w.softmax_scale)
    ref = dense_reference(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                          w.seq_lens, w.softmax_scale)
    assert np.allclose(ours, ref, rtol=1e-11, atol=1e-12)


def test_attention_invariant_under_physical_page_permutation():
    w, hv = small_ragged(g=2)
    kc, vc = populate(w, hv)
    base = oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                              w.seq_lens, w.softmax_scale)
    perm = np.random.default_rng(3).permutation(w.num_pages)      # new slot of old page p
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    moved = oracle.decode_attn(hv.q, kc2, vc2, hv.k_scale, hv.v_scale, bt2,
                               w.seq_lens, w.softmax_scale)
    assert np.array_equal(base, moved)                   # bit-identical


def test_attention_single_token_returns_its_value():
    w, hv = small_ragged(lens=(1, 1, 1))
    kc, vc = populate(w, hv)
    out = oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                             w.seq_lens, w.softmax_scale)
    V = dequant_torch(vc, hv.v_scale).numpy()
    for r in range(w.batch):
        p = w.block_table[r, 0]
        for h in range(w.num_q_heads):
            assert np.array_equal(out[r, h], V[p, h // w.group, 0])


def test_attention_equal_keys_average_the_values():
    w, hv = small_ragged(lens=(37, 64))
    kc, vc = populate(w, hv)
    kc[:] = 0x38                                           # every key element = 1.0 * scale
    out = oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                             w.seq_lens, w.softmax_scale)
    V = dequant_torch(vc, hv.v_scale).numpy()
    for r in range(w.batch):
        L = int(w.seq_lens[r])
        rows = np.stack([V[w.block_table[r, j // w.page_size], :, j % w.page_size] for j in range(L)])
        mean = rows.mean(axis=0)                           # [Hkv][D]
        for h in range(w.num_q_heads):
            assert np.allclose(out[r, h], mean[h // w.group], rtol=1e-12, atol=1e-14)


def test_attention_zero_for_aborted_empty_and_invalid_requests():
    w, hv = small_ragged()
    kc, vc = populate(w, hv)
    abort = np.zeros(w.batch, np.uint8)
    abort[1] = 1
    seq = w.seq_lens.copy()
    seq[2] = 0
    bt = w.block_table.copy()
    bt[3, 0] = w.num_pages                                 # out of range
    seq[4] = bt.shape[1] * w.page_size + 1                 # longer than its table row
    out = oracle.decode_attn(hv.q, kc, vc, hv.k_scale, hv.v_scale, bt, seq,
                             w.softmax_scale, abort)
    for r in (1, 2, 3, 4):
        assert np.all(out[r] == 0.0)
    assert np.all(np.any(out[0] != 0, axis=-1))
    assert np.all(np.any(out[5] != 0, axis=-1))


def test_gqa_head_mapping_is_contiguous_groups():
    """Query heads h*g .. h*g+g-1 share KV head h: identical queries inside a
    group give identical outputs, and differ across groups."""
    w, hv = small_ragged(g=4, lens=(33,))
    kc, vc = populate(w, hv)
    q = hv.q.copy()
    for kvh in range(w.num_kv_heads):
        q[:, kvh * 4:(kvh + 1) * 4] = q[:, kvh * 4:kvh * 4 + 1]
    out = oracle.decode_attn(q, kc, vc, hv.k_scale, hv.v_scale, w.block_table,
                             w.seq_lens, w.softmax_scale)
    for kvh in range(w.num_kv_heads):
        for j in range(4):
            assert np.array_equal(out[0, kvh * 4 + j], out[0, kvh * 4])
    assert not np.array_equal(out[0, 0], out[0, 4])


# --------------------------------------------------------------- tag check

def brute_tag_check(bt, exp, seq, tags, ps):
    out = []
    for r in range(bt.shape[0]):
        L = max(int(seq[r]), 0)
        n = -(-L // ps)
        bad = n > bt.shape[1]
        for i in range(min(n, bt.shape[1])):
            p = int(bt[r, i])
            if not (0 <= p < len(tags)) or int(tags[p]) != int(exp[r, i]):
                bad = True
        out.append(int(bad))
    return np.array(out, np.uint8)


def test_tag_check_flags_exactly_the_seeded_stale_requests():
    rng = np.random.default_rng(11)
    for ps in (16, 64):
        w = W.make("ragged64", seed=int(rng.integers(1000)), scale_down=8)
        exp = w.expected_tags.copy()
        tags = w.page_tags.copy()
        stale = set()
        for r in rng.choice(w.batch, size=9, replace=False):
            n = -(-int(w.seq_lens[r]) // w.page_size)
            i = int(rng.integers(n))
            if rng.random() < 0.5:
                tags[w.block_table[r, i]] += np.uint32(1)      # page reallocated: tag bumped
            else:
                exp[r, i] ^= np.uint32(1 << int(rng.integers(32)))
            stale.add(int(r))
        # a page past a request's used length must not matter
        exp[0, -1] ^= np.uint32(7) if (-(-int(w.seq_lens[0]) // w.page_size)) < exp.shape[1] else 0
        flags = oracle.tag_check(w.block_table, exp, w.seq_lens, tags, page_size=w.page_size)
        # a bumped page may be shared by no other request (pages are distinct)
        assert set(np.nonzero(flags)[0].tolist()) == stale
        assert np.array_equal(flags, brute_tag_check(w.block_table, exp, w.seq_lens, tags, w.page_size))


def test_tag_check_edge_cases():
    tags = np.array([5, 6, 7, 8], np.uint32)
    bt = np.array([[0, 1, -1], [2, 9, 3], [3, 2, 1], [0, 0, 0], [1, 2, 3]], np.int32)
    exp = np.array([[5, 6, 0], [7, 0, 8], [8, 7, 6], [5, 5, 5], [6, 7, 8]], np.uint32)
    seq = np.array([32, 16, 48, 0, 49], np.int32)      # ps 16
    flags = oracle.tag_check(bt, exp, seq, tags, page_size=16)
    # r0: 2 pages fine; r1: 1 page fine (page 9 unused); r2: 3 pages fine;
    # r3: empty; r4: needs 4 entries but the row has 3
    assert flags.tolist() == [0, 0, 0, 0, 1]
    seq2 = np.array([33, 17, 48, 0, 48], np.int32)
    flags2 = oracle.tag_check(bt, exp, seq2, tags, page_size=16)
    assert flags2.tolist() == [1, 1, 0, 0, 0]
    assert np.array_equal(flags2, brute_tag_check(bt, exp, seq2, tags, 16))
