"""kvq_decode_step (tag check + append + attention in one launch) against the
separate calls on copies of the same inputs: abort flags, cache bytes and
outputs bit for bit; flags against the oracle's tag check; outputs of the
requests that pass against the oracle's attention."""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
import workloads as W
from kvq_harness import DeviceWorkload
from gpu_util import assert_close, oracle_attention, oracle_caches, out_to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = (1, 15, 16, 17, 31, 32, 33, 100, 257, 1000, 2049)


@pytest.fixture(autouse=True)
def _no_device_errors():
    kvq.kvq_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert kvq.kvq_device_error() == 0


def _stale(w, r, page_index):
    """Request r's expected tag for one of its pages no longer matches."""
    w.expected_tags[r, page_index] ^= np.uint32(0x5A5A5A5A)


def _one_vs_separate(w, cd, fp32, splits, fill=None):
    """kvq_decode_step on one copy; kvq_tag_check then kvq_decode_attn_append
    on another."""
    sep = DeviceWorkload(w, cd, populate=fill is None)
    one = DeviceWorkload(w, cd, populate=fill is None)
    if fill is not None:
        for dw in (sep, one):
            dw.k_cache.copy_(torch.from_numpy(fill[0]))
            dw.v_cache.copy_(torch.from_numpy(fill[1]))
    out_s, out_o = sep.out(fp32), one.out(fp32)
    sep.tag_check()
    kvq.kvq_decode_attn_append(sep.desc, sep.q, sep.k_cache, sep.v_cache, sep.k_scale, sep.v_scale,
                               sep.block_table, sep.seq_lens, w.softmax_scale, sep.abort, sep.k_new,
                               sep.v_new, out_s, sep.workspace(splits), splits)
    one.abort.fill_(0xCC)                                # every flag must be written
    one.decode_step(out_o, one.workspace(splits), splits)
    torch.cuda.synchronize()
    return sep, one, out_s, out_o


def _assert_same(sep, one, out_s, out_o, fp32):
    assert torch.equal(one.abort, sep.abort)
    assert torch.equal(one.k_cache, sep.k_cache) and torch.equal(one.v_cache, sep.v_cache)
    iv = torch.int32 if fp32 else torch.int16
    assert torch.equal(out_o.view(iv), out_s.view(iv))


@pytest.mark.parametrize("cache", ["fp8", "bf16"])
@pytest.mark.parametrize("splits", [0, 1, 5, 12])
def test_decode_step_equals_check_then_fused(cache, splits):
    cd = kvq.KVQ_CACHE_FP8_E4M3 if cache == "fp8" else kvq.KVQ_CACHE_BF16
    w = W.make_custom(LENS, group=4, page_size=16, seed=70 + splits, outlier_frac=0.01)
    _stale(w, 3, 0)                                      # first page
    _stale(w, 9, 62)                                     # the last page of a 1,000-token request
    flags = oracle.tag_check(w.block_table, w.expected_tags, w.seq_lens, w.page_tags,
                             page_size=w.page_size)
    assert flags[3] == 1 and flags[9] == 1 and flags.sum() == 2
    for fp32 in (False, True):
        sep, one, out_s, out_o = _one_vs_separate(w, cd, fp32, splits)
        _assert_same(sep, one, out_s, out_o, fp32)
        assert np.array_equal(one.abort.cpu().numpy(), flags)
    alive = [r for r in range(w.batch) if not flags[r]]
    kc, vc = oracle_caches(one, alive)
    ref = oracle_attention(one, kc, vc, flags)
    got = out_to_np(out_o)
    assert_close(got[alive], ref[alive], "fp32", f"decode_step {cache} splits{splits}")
    assert np.all(got[[3, 9]] == 0.0)


def test_decode_step_edge_requests():
    """Empty, too-long and bad-page requests, and a stale tag: the flags of
    the separate tag check, zeros, and the cache written only where the
    separate calls write it."""
    lens = [40, 0, 77, 300, 5, 64, 33]
    w = W.make_custom(lens, group=4, page_size=16, seed=5)
    w.block_table[2, 1] = w.num_pages + 1            # bad id in another page than the last
    w.block_table[3, 18] = -7                         # bad id: the request's last page
    w.seq_lens[4] = w.block_table.shape[1] * 16 + 3   # longer than its table row
    _stale(w, 6, 2)                                   # stale tag on the page holding token 32
    flags = oracle.tag_check(w.block_table, w.expected_tags, w.seq_lens, w.page_tags,
                             page_size=w.page_size)
    assert list(flags) == [0, 0, 1, 1, 1, 0, 1]
    rng = np.random.default_rng(9)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    fill = (rng.choice(finite, size=w.cache_shape()).astype(np.uint8),
            rng.choice(finite, size=w.cache_shape()).astype(np.uint8))
    for splits in (1, 0, 4, 12):
        sep, one, out_s, out_o = _one_vs_separate(w, kvq.KVQ_CACHE_FP8_E4M3, True, splits, fill=fill)
        _assert_same(sep, one, out_s, out_o, True)
        assert np.array_equal(one.abort.cpu().numpy(), flags)
        got = out_to_np(out_o)
        for r in (1, 2, 3, 4, 6):
            assert np.all(got[r] == 0.0), (splits, r)


def test_decode_step_uniform8_full_size():
    """The uniform8 step (8 x 8,193 tokens) with one request made stale, in the
    configuration the bench times: the same flags, cache and output bytes as
    kvq_tag_check_append followed by kvq_decode_attn."""
    w = W.make("uniform8", seed=0)
    _stale(w, 5, 300)
    a = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3)
    b = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3)
    out_a, out_b = a.out(False), b.out(False)
    a.step(out_a, a.workspace(0), fused=True)
    b.abort.fill_(0xCC)
    b.decode_step(out_b, b.workspace(0))
    torch.cuda.synchronize()
    flags = b.abort.cpu().numpy()
    assert list(flags) == [0, 0, 0, 0, 0, 1, 0, 0]
    assert torch.equal(a.abort, b.abort)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert np.all(out_to_np(out_b)[5] == 0.0)


def test_decode_step_argument_checks():
    w = W.make_custom([40, 17], group=4, page_size=16, seed=2)
    dw = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3)
    out = dw.out(False)
    ws = dw.workspace(0)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    lib = kvq.load()
    import ctypes
    st = lib.kvq_decode_step(ctypes.byref(dw.desc.c()), kvq._ptr(dw.q), w.batch, w.num_q_heads,
                             kvq._ptr(dw.k_cache), kvq._ptr(dw.v_cache), kvq._ptr(dw.k_scale),
                             kvq._ptr(dw.v_scale), kvq._ptr(dw.block_table), w.block_table.shape[1],
                             kvq._ptr(dw.seq_lens), None, kvq._ptr(dw.page_tags), kvq._ptr(dw.abort),
                             ctypes.c_float(w.softmax_scale), kvq._ptr(dw.k_new), kvq._ptr(dw.v_new),
                             kvq._ptr(out), 0, kvq._ptr(ws), ws_bytes, 0, None)
    assert st == 1                                       # no expected tags: invalid argument


@pytest.mark.parametrize("splits", [0, 3])
def test_decode_step_consecutive_steps(splits):
    """Four steps in a row, each appending one more token that the next step
    reads back from the cache; a page handed to another owner between steps
    (its live tag bumped) aborts its request from then on.  Flags, caches and
    outputs equal the separate calls after every step."""
    steps = 4
    final = np.array([40, 129, 300, 17, 1000, 64], np.int64)
    w = W.make_custom(final, group=4, page_size=16, seed=90 + splits)
    w.seq_lens = (final - (steps - 1)).astype(np.int32)          # the prefill ends steps - 1 earlier
    sep = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3)
    one = DeviceWorkload(w, kvq.KVQ_CACHE_FP8_E4M3)
    assert torch.equal(sep.k_cache, one.k_cache)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    for s in range(steps):
        if s:
            for dw in (sep, one):
                dw.seq_lens += 1
        if s == 2:                                                # request 4's page 10 is reallocated
            page = int(w.block_table[4, 10])
            for dw in (sep, one):
                dw.page_tags[page] += 1
        kn = W.normal_bf16_torch(tuple(sep.k_new.shape), gen, DEV, 0.0)
        vn = W.normal_bf16_torch(tuple(sep.v_new.shape), gen, DEV, 0.0)
        for dw in (sep, one):
            dw.k_new.copy_(kn)
            dw.v_new.copy_(vn)
        out_s, out_o = sep.out(False), one.out(False)
        sep.tag_check()
        kvq.kvq_decode_attn_append(sep.desc, sep.q, sep.k_cache, sep.v_cache, sep.k_scale, sep.v_scale,
                                   sep.block_table, sep.seq_lens, w.softmax_scale, sep.abort, sep.k_new,
                                   sep.v_new, out_s, sep.workspace(splits), splits)
        one.abort.fill_(0xCC)
        one.decode_step(out_o, one.workspace(splits), splits)
        torch.cuda.synchronize()
        _assert_same(sep, one, out_s, out_o, False)
        assert int(one.abort[4]) == (1 if s >= 2 else 0)
        assert int(one.abort.sum()) == (1 if s >= 2 else 0)
