"""GPU parity of each kernel against the CPU oracle, through the C ABI.

Bit-exact: e4m3 cache codes written by kvq_append and the abort flags of
kvq_tag_check.  Within tolerance (|gpu - oracle| <= 1e-2 + 1e-2 |oracle| for
bf16 output, 2e-4 + 2e-4 |oracle| for fp32 output): kvq_decode_attn.
"""
import math

import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
import workloads as W
from kvq_harness import DeviceWorkload
from gpu_util import (assert_close, oracle_attention, oracle_caches, out_to_np, to_np_bits)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _no_device_errors():
    kvq.kvq_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert kvq.kvq_device_error() == 0


# ------------------------------------------------------------------ append

def _append_case(values_bits: np.ndarray, scales_k, scales_v, page_size=16, num_pages=None,
                 slots=None, abort=None, bf16=False):
    T, Hkv, D = values_bits.shape
    num_pages = num_pages or (T + page_size - 1) // page_size + 3
    slots = np.arange(T, dtype=np.int64) if slots is None else slots
    dt = np.uint16 if bf16 else np.uint8
    canary = 0xA5A5 if bf16 else 0xA5
    kc = np.full((num_pages, Hkv, page_size, D), canary, dt)
    vc = kc.copy()
    vbits = values_bits ^ np.uint16(0x8000)                       # V = -K
    oracle.append(kc, vc, values_bits, vbits, slots, scales_k, scales_v, abort, page_size=page_size)
    desc = kvq.CacheDesc(num_pages, page_size, Hkv, D,
                         kvq.KVQ_CACHE_BF16 if bf16 else kvq.KVQ_CACHE_FP8_E4M3)
    if bf16:
        gk = torch.full(kc.shape, -0x5A5B, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    else:
        gk = torch.full(kc.shape, canary, dtype=torch.uint8, device=DEV)
    gv = gk.clone()
    as_bf16 = lambda b: torch.from_numpy(b.view(np.int16)).to(DEV).view(torch.bfloat16)
    kvq.kvq_append(desc, as_bf16(values_bits), as_bf16(vbits), torch.from_numpy(slots).to(DEV),
                   torch.from_numpy(np.asarray(scales_k, np.float32)).to(DEV),
                   torch.from_numpy(np.asarray(scales_v, np.float32)).to(DEV),
                   None if abort is None else torch.from_numpy(abort).to(DEV), gk, gv)
    torch.cuda.synchronize()
    return kc, vc, to_np_bits(gk), to_np_bits(gv)


def _split_nan(values_f32, codes_gpu, codes_ref):
    """NaN inputs may map to either NaN code; everything else must match bit for bit."""
    nan = np.isnan(values_f32)
    assert np.array_equal(codes_gpu[~nan], codes_ref[~nan])
    assert np.all((codes_gpu[nan] & 0x7F) == 0x7F)


def test_append_every_bf16_value_scale_one_bit_exact():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(64, 8, 128)
    ones = np.ones(8, np.float32)
    kc, vc, gk, gv = _append_case(bits, ones, ones)
    slots = np.arange(64)
    ref = kc[slots // 16, :, slots % 16, :]
    got = gk[slots // 16, :, slots % 16, :]
    _split_nan(W.bf16_bits_to_f32(bits), got, ref)
    refv = vc[slots // 16, :, slots % 16, :]
    gotv = gv[slots // 16, :, slots % 16, :]
    _split_nan(W.bf16_bits_to_f32(bits), gotv, refv)
    untouched = np.ones(kc.shape, bool)
    untouched[slots // 16, :, slots % 16, :] = False
    assert np.all(gk[untouched] == 0xA5) and np.all(gv[untouched] == 0xA5)


@pytest.mark.parametrize("scales", [
    [1.0, 0.37, 3.1e-3, 17.5, 1e-30, 1e30, 2.0 ** -20, 448.0 / 3.0],
    [0.011, 0.0123, 0.2, 0.75, 1.0 / 448.0, 5.0 / 448.0, 100.0 / 448.0, 7.77],
])
def test_append_every_bf16_value_with_scales_bit_exact(scales):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(64, 8, 128)
    sk = np.array(scales, np.float32)
    sv = sk[::-1].copy()
    kc, vc, gk, gv = _append_case(bits, sk, sv, page_size=64)
    slots = np.arange(64)
    for ref_c, got_c, sc in ((kc, gk, sk), (vc, gv, sv)):
        ref = ref_c[slots // 64, :, slots % 64, :]
        got = got_c[slots // 64, :, slots % 64, :]
        vals = W.bf16_bits_to_f32(bits if ref_c is kc else bits ^ np.uint16(0x8000))
        _split_nan(vals / sc[None, :, None], got, ref)


def test_append_slots_skips_and_bf16_cache():
    rng = np.random.default_rng(7)
    T = 200
    bits = W.normal_bf16(rng, (T, 4, 128), 0.01)
    scales = np.array([0.01, 0.02, 0.03, 0.05], np.float32)
    num_pages = 40
    slots = rng.permutation(num_pages * 16)[:T].astype(np.int64)
    slots[3] = -1
    slots[5] = num_pages * 16
    slots[7] = 1 << 40
    abort = (rng.random(T) < 0.1).astype(np.uint8)
    for ps in (16, 32, 128):
        npg = num_pages * 16 // ps
        kc, vc, gk, gv = _append_case(bits, scales, scales, page_size=ps, num_pages=npg,
                                      slots=slots, abort=abort)
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    kc, vc, gk, gv = _append_case(bits, scales, scales, page_size=16, num_pages=num_pages,
                                  slots=slots, abort=abort, bf16=True)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)


# --------------------------------------------------------------- tag check

def _tag_gpu(bt, exp, seq, tags, ps):
    out = torch.full((bt.shape[0],), 7, dtype=torch.uint8, device=DEV)
    kvq.kvq_tag_check(torch.from_numpy(bt).to(DEV), torch.from_numpy(exp.view(np.int32)).to(DEV),
                      torch.from_numpy(seq).to(DEV), ps,
                      torch.from_numpy(tags.view(np.int32)).to(DEV), out)
    return out.cpu().numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tag_check_bit_exact_with_stale_invalid_and_long_entries(seed):
    rng = np.random.default_rng(seed)
    for name, down in (("ragged64", 4), ("churn", 8), ("long4", 64)):
        w = W.make(name, seed=seed, scale_down=down)
        bt, exp, tags, seq = (w.block_table.copy(), w.expected_tags.copy(), w.page_tags.copy(),
                              w.seq_lens.copy())
        B = w.batch
        # 0.5 % of used entries pointed at stale-tag pages, plus a few other faults
        used = [(r, i) for r in range(B) for i in range(-(-int(seq[r]) // w.page_size))]
        for k in rng.choice(len(used), size=max(1, len(used) // 200), replace=False):
            r, i = used[k]
            exp[r, i] = tags[bt[r, i]] - np.uint32(1)
        r = int(rng.integers(B))
        bt[r, 0] = w.num_pages + 5
        r = int(rng.integers(B))
        bt[r, 0] = -3
        r = int(rng.integers(B))
        seq[r] = bt.shape[1] * w.page_size + 1
        r = int(rng.integers(B))
        seq[r] = 0
        ref = oracle.tag_check(bt, exp, seq, tags, page_size=w.page_size)
        got = _tag_gpu(bt, exp, seq, tags, w.page_size)
        assert np.array_equal(got, ref), name
        assert ref.any() and not ref.all()


def test_tag_check_single_and_many_requests():
    for B in (1, 7, 8, 9, 513):
        rng = np.random.default_rng(B)
        w = W.make_custom(rng.integers(1, 300, size=B), group=1, page_size=16, seed=B)
        exp = w.expected_tags.copy()
        if B > 3:
            exp[3, 0] ^= np.uint32(1)
        ref = oracle.tag_check(w.block_table, exp, w.seq_lens, w.page_tags, page_size=16)
        assert np.array_equal(_tag_gpu(w.block_table, exp, w.seq_lens, w.page_tags, 16), ref)


# --------------------------------------------------------------- attention

LENS = (1, 15, 16, 17, 31, 32, 33, 100, 257, 1000, 2049)


def _decode_case(w, cache_dtype, out_fp32, num_splits, abort=None):
    dw = DeviceWorkload(w, cache_dtype)
    dw.append()
    ws = dw.workspace(num_splits)
    out = dw.out(out_fp32)
    ab = None if abort is None else torch.from_numpy(abort).to(DEV)
    dw.attend(out, ws, ab, num_splits)
    torch.cuda.synchronize()
    kc, vc = oracle_caches(dw)
    assert np.array_equal(to_np_bits(dw.k_cache), kc) and np.array_equal(to_np_bits(dw.v_cache), vc)
    ref = oracle_attention(dw, kc, vc, abort)
    return dw, out_to_np(out), ref


@pytest.mark.parametrize("g,ps", [(1, 16), (2, 64), (4, 16), (8, 16), (8, 32), (4, 128), (3, 64)])
@pytest.mark.parametrize("cache", ["fp8", "bf16"])
@pytest.mark.parametrize("out_kind", ["bf16", "fp32"])
def test_decode_attention_matches_oracle(g, ps, cache, out_kind):
    w = W.make_custom(LENS, group=g, page_size=ps, seed=g * 100 + ps, outlier_frac=0.01)
    cd = kvq.KVQ_CACHE_FP8_E4M3 if cache == "fp8" else kvq.KVQ_CACHE_BF16
    # 5 splits: small batches merge them through distributed shared memory
    # (one cluster per request and KV head); 12 (> 8, the cluster limit):
    # through the workspace
    for splits in (0, 1, 5, 12):
        _, got, ref = _decode_case(w, cd, out_kind == "fp32", splits)
        assert_close(got, ref, out_kind, f"g{g} ps{ps} {cache} splits{splits}")


def test_decode_edge_requests_zeroed():
    lens = [40, 0, 77, 300, 5, 64]
    w = W.make_custom(lens, group=4, page_size=16, seed=3)
    w.block_table[2, 1] = w.num_pages + 1          # out-of-range page id
    w.block_table[3, 15] = -7                      # bad id late in a long request (other split)
    w.seq_lens[4] = w.block_table.shape[1] * 16 + 3  # longer than its table row
    abort = np.zeros(len(lens), np.uint8)
    abort[5] = 1
    rng = np.random.default_rng(4)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    for splits in (1, 0, 4, 12):
        dw = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3, populate=False)
        dw.k_cache.copy_(torch.from_numpy(rng.choice(finite, size=w.cache_shape()).astype(np.uint8)))
        dw.v_cache.copy_(torch.from_numpy(rng.choice(finite, size=w.cache_shape()).astype(np.uint8)))
        dw.q.normal_()
        out = dw.out(True)
        out.fill_(123.0)
        dw.attend(out, dw.workspace(splits), torch.from_numpy(abort).to(DEV), splits)
        got = out_to_np(out)
        for r in (1, 2, 3, 4, 5):
            assert np.all(got[r] == 0.0), (splits, r)
        assert np.all(np.isfinite(got[0])) and np.any(got[0] != 0)


def test_cluster_and_workspace_combine_agree():
    """The two forms of the split combine give the same attention."""
    w = W.make_custom([3000, 1, 700, 2049, 64], group=8, page_size=16, seed=21)
    dw = DeviceWorkload(w)
    dw.append()
    counters = (w.batch * w.num_kv_heads * 4 + 255) // 256 * 256
    _, n6, ws6 = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads, w.max_pages_per_seq, 6)
    _, n12, ws12 = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads, w.max_pages_per_seq, 12)
    assert n6 == 6 and ws6 == counters                      # 10 clusters of 6 CTAs: resident
    assert n12 == 12 and ws12 > counters                    # partials go through the workspace
    outs = []
    for splits in (6, 12):
        out = dw.out(True)
        dw.attend(out, dw.workspace(splits), None, splits)
        outs.append(out_to_np(out))
    kc, vc = oracle_caches(dw)
    ref = oracle_attention(dw, kc, vc)
    for got in outs:
        assert_close(got, ref, "fp32", "combine forms")
    assert np.all(np.abs(outs[0] - outs[1]) <= 4e-4 + 4e-4 * np.abs(outs[1]))


def test_decode_invariant_to_physical_page_placement():
    w = W.make_custom([700, 1500, 33], group=8, page_size=16, seed=11, pool_factor=3.0)
    dw = DeviceWorkload(w)
    dw.append()
    out1 = dw.out(True)
    dw.attend(out1, dw.workspace(0))
    perm = torch.from_numpy(np.random.default_rng(1).permutation(w.num_pages)).to(DEV)
    k2 = torch.empty_like(dw.k_cache)
    v2 = torch.empty_like(dw.v_cache)
    k2[perm] = dw.k_cache
    v2[perm] = dw.v_cache
    bt2 = torch.where(dw.block_table >= 0, perm[dw.block_table.clamp(min=0).long()].int(),
                      dw.block_table)
    out2 = dw.out(True)
    kvq.kvq_decode_attn(dw.desc, dw.q, k2, v2, dw.k_scale, dw.v_scale, bt2.contiguous(),
                        dw.seq_lens, w.softmax_scale, None, out2, dw.workspace(0))
    assert torch.equal(out1, out2)                  # bit-identical: order depends on logical positions


def test_decode_every_e4m3_code_decodes_exactly():
    """Caches filled with every finite code (an input written by the test)."""
    rng = np.random.default_rng(5)
    w = W.make_custom([1, 1, 37, 64, 500], group=8, page_size=16, seed=5)
    dw = DeviceWorkload(w, populate=False)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    kc = rng.choice(finite, size=w.cache_shape()).astype(np.uint8)
    vc = rng.choice(finite, size=w.cache_shape()).astype(np.uint8)
    vc[w.block_table[0, 0], 0, 0, :] = finite[:128]
    vc[w.block_table[1, 0], 0, 0, :] = finite[126:]
    dw.k_cache.copy_(torch.from_numpy(kc))
    dw.v_cache.copy_(torch.from_numpy(vc))
    dw.k_scale_host = np.full(w.num_kv_heads, 1.0 / 64, np.float32)
    dw.v_scale_host = np.full(w.num_kv_heads, 0.5, np.float32)
    dw.k_scale.copy_(torch.from_numpy(dw.k_scale_host))
    dw.v_scale.copy_(torch.from_numpy(dw.v_scale_host))
    for fp32 in (True, False):
        out = dw.out(fp32)
        dw.attend(out, dw.workspace(0))
        ref = oracle_attention(dw, kc, vc)
        assert_close(out_to_np(out), ref, "fp32" if fp32 else "bf16", "all codes")
    # single-token requests return exactly their decoded V row (head 0 group)
    out = dw.out(True)
    dw.attend(out, dw.workspace(0))
    dec = oracle.e4m3_decode(finite) * 0.5
    got = out_to_np(out)
    assert np.array_equal(got[0, 0], dec[:128])
    assert np.array_equal(got[1, 0], dec[126:])


def _bf16_bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("cache", ["fp8", "bf16"])
def test_decode_q_rows_far_outside_the_f16_range(cache):
    """Any finite bf16 q is valid input.  The FP8 path multiplies each q row by
    an exact power of two before its f16 product, so rows at 1e6 or 1e30 do
    not overflow and rows at 1e-6, 1e-30 or bf16 subnormals keep their bits;
    the outputs match the oracle, which takes q as given."""
    w = W.make_custom([37, 500, 1000, 2049], group=8, page_size=16, seed=31, outlier_frac=0.01)
    cd = kvq.KVQ_CACHE_FP8_E4M3 if cache == "fp8" else kvq.KVQ_CACHE_BF16
    dw = DeviceWorkload(w, cd)
    dw.append()
    rng = np.random.default_rng(32)
    base = rng.standard_normal((w.batch, w.num_q_heads, w.head_dim)).astype(np.float32)
    mult = np.ones((w.batch, w.num_q_heads, 1), np.float32)
    mult[0] = 1e6                                  # every head of request 0 far above 65504
    mult[1] = 1e-6                                 # every head of request 1 far below 2^-14
    row_mults = [1e6, 1e-6, 1e30, 1e-30, 0.0, 1e-39, 1.0, 3e4]   # one per head of a group
    for kvh in range(w.num_kv_heads):
        mult[2, kvh * 8:(kvh + 1) * 8, 0] = row_mults
    q = base * mult
    q[2, 6, :4] = 2e5                              # a row of N(0,1) with four elements at 2e5
    q[3, 1, 5] = -7e4                              # one element just beyond f16 in a normal row
    q_bits = _bf16_bits(q)
    dw.q.copy_(torch.from_numpy(q_bits.view(np.int16)).to(DEV).view(torch.bfloat16))
    kc, vc = oracle_caches(dw)
    ref = oracle_attention(dw, kc, vc, q=q_bits)
    assert np.all(np.isfinite(ref))
    for splits in (0, 1, 12):
        for fp32 in (True, False):
            out = dw.out(fp32)
            dw.attend(out, dw.workspace(splits), None, splits)
            torch.cuda.synchronize()
            assert_close(out_to_np(out), ref, "fp32" if fp32 else "bf16",
                         f"{cache} q rows far from 1, splits {splits}")


# ------------------------------------------------- fused tag check + append

@pytest.mark.parametrize("bf16", [False, True])
def test_tag_check_append_matches_the_two_oracle_passes(bf16):
    rng = np.random.default_rng(8)
    w = W.make_custom(rng.integers(1, 900, size=37), group=4, page_size=16, num_kv_heads=8, seed=8)
    cd = kvq.KVQ_CACHE_BF16 if bf16 else kvq.KVQ_CACHE_FP8_E4M3
    dw = DeviceWorkload(w, cd)
    exp = w.expected_tags.copy()
    exp[3, 0] ^= np.uint32(5)                       # stale: request 3 must be flagged and not written
    exp[11, -1 + (-(-int(w.seq_lens[11]) // 16))] ^= np.uint32(1)
    dw.expected_tags.copy_(torch.from_numpy(exp.view(np.int32)))
    slots = w.append_slot_mapping().copy()
    slots[5] = -1                                  # skipped token
    dw.append_slots.copy_(torch.from_numpy(slots))
    kc_ref, vc_ref = to_np_bits(dw.k_cache), to_np_bits(dw.v_cache)
    dw.abort.fill_(9)
    dw.tag_check_append()
    torch.cuda.synchronize()
    flags = oracle.tag_check(w.block_table, exp, w.seq_lens, w.page_tags, page_size=16)
    assert np.array_equal(dw.abort.cpu().numpy(), flags)
    assert flags[3] == 1 and flags[11] == 1 and flags.sum() == 2
    oracle.append(kc_ref, vc_ref, to_np_bits(dw.k_new), to_np_bits(dw.v_new), slots,
                  dw.k_scale_host, dw.v_scale_host, flags, page_size=16)
    assert np.array_equal(to_np_bits(dw.k_cache), kc_ref)
    assert np.array_equal(to_np_bits(dw.v_cache), vc_ref)


# ------------------------------------------------- fused append + attention

def _fused_vs_separate(w, cd, fp32, splits, abort=None, fill=None):
    """Run the separate (append, then decode) and the fused call on two copies
    of the same workload.  fill: cache bytes to start from instead of the
    populated prefill (same for both)."""
    sep = DeviceWorkload(w, cd, populate=fill is None)
    fus = DeviceWorkload(w, cd, populate=fill is None)
    if fill is not None:
        for dw in (sep, fus):
            dw.k_cache.copy_(torch.from_numpy(fill[0]))
            dw.v_cache.copy_(torch.from_numpy(fill[1]))
    ab = None if abort is None else torch.from_numpy(abort).to(DEV)
    out_s, out_f = sep.out(fp32), fus.out(fp32)
    sep.append(ab)
    sep.attend(out_s, sep.workspace(splits), ab, splits)
    kvq.kvq_decode_attn_append(fus.desc, fus.q, fus.k_cache, fus.v_cache, fus.k_scale, fus.v_scale,
                               fus.block_table, fus.seq_lens, w.softmax_scale, ab, fus.k_new,
                               fus.v_new, out_f, fus.workspace(splits), splits)
    torch.cuda.synchronize()
    return sep, fus, out_s, out_f


@pytest.mark.parametrize("cache", ["fp8", "bf16"])
@pytest.mark.parametrize("ps", [16, 64])
@pytest.mark.parametrize("splits", [0, 1, 5, 12])
def test_decode_attn_append_equals_append_then_decode(cache, ps, splits):
    """kvq_decode_attn_append == kvq_append (token r at position L_r - 1) then
    kvq_decode_attn: caches and outputs bit for bit, both forms of the
    combine; and the output matches the oracle."""
    cd = kvq.KVQ_CACHE_FP8_E4M3 if cache == "fp8" else kvq.KVQ_CACHE_BF16
    w = W.make_custom(LENS, group=4, page_size=ps, seed=40 + ps + splits, outlier_frac=0.01)
    abort = np.zeros(w.batch, np.uint8)
    abort[3] = 1
    for fp32 in (False, True):
        sep, fus, out_s, out_f = _fused_vs_separate(w, cd, fp32, splits, abort)
        assert torch.equal(fus.k_cache, sep.k_cache) and torch.equal(fus.v_cache, sep.v_cache)
        assert torch.equal(out_f.view(torch.int32 if fp32 else torch.int16),
                           out_s.view(torch.int32 if fp32 else torch.int16))
    kc, vc = oracle_caches(fus, [r for r in range(w.batch) if not abort[r]])
    # the aborted request's new token is not written: the oracle caches hold
    # its prefill only
    r = 3
    L = int(w.seq_lens[r])
    k, v, _ = fus.host_request(r)
    oracle.append(kc, vc, k[:L - 1], v[:L - 1], w.slots_of(r, np.arange(L - 1)),
                  fus.k_scale_host, fus.v_scale_host, page_size=w.page_size)
    assert np.array_equal(to_np_bits(fus.k_cache), kc) and np.array_equal(to_np_bits(fus.v_cache), vc)
    ref = oracle_attention(fus, kc, vc, abort)
    assert_close(out_to_np(out_f), ref, "fp32", f"fused {cache} ps{ps} splits{splits}")


def test_decode_attn_append_edge_requests():
    """Empty, too-long and bad-page requests: zeros, and the cache is written
    exactly where kvq_append would write it."""
    lens = [40, 0, 77, 300, 5, 64]
    w = W.make_custom(lens, group=4, page_size=16, seed=3)
    w.block_table[2, 1] = w.num_pages + 1            # bad id in another page than the last
    w.block_table[3, 18] = -7                         # bad id: the request's last page
    w.seq_lens[4] = w.block_table.shape[1] * 16 + 3   # longer than its table row
    rng = np.random.default_rng(8)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    fill = (rng.choice(finite, size=w.cache_shape()).astype(np.uint8),
            rng.choice(finite, size=w.cache_shape()).astype(np.uint8))
    for splits in (1, 0, 4, 12):
        sep, fus, out_s, out_f = _fused_vs_separate(w, kvq.KVQ_CACHE_FP8_E4M3, True, splits,
                                                    fill=fill)
        assert torch.equal(fus.k_cache, sep.k_cache) and torch.equal(fus.v_cache, sep.v_cache)
        got = out_to_np(out_f)
        for r in (1, 2, 3, 4):
            assert np.all(got[r] == 0.0), (splits, r)
        assert torch.equal(out_f.view(torch.int32), out_s.view(torch.int32))


def test_read_probe_reads_every_word_once():
    """The calibration probe XORs every 32-bit word: compare with numpy, for a
    size that leaves a ragged tail of the grid-stride loop."""
    rng = np.random.default_rng(3)
    for n_words in (4, 4 * 1000 + 8, (1 << 22) + 36):
        host = rng.integers(0, 2**32, size=n_words, dtype=np.uint64).astype(np.uint32)
        src = torch.from_numpy(host.view(np.int32)).to(DEV)
        sink = torch.zeros(1, dtype=torch.int32, device=DEV)
        kvq.kvq_read_probe(src, sink)
        torch.cuda.synchronize()
        want = np.bitwise_xor.reduce(host)
        assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want), n_words
