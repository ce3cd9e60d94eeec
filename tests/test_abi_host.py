"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/kvq.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import fp8_quantised_paged_kv_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]*?\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared()
    for n in ("kvq_append", "kvq_tag_check", "kvq_decode_attn", "kvq_decode_plan",
              "kvq_status_string"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    lib = kvq.load()
    for name in declared():
        assert hasattr(lib, name), name
    assert set(declared()) <= set(kvq.EXPORTED)


def test_status_strings():
    assert kvq.kvq_status_string(0) == "ok"
    assert kvq.kvq_status_string(3) == "workspace too small"


def _plan(ps=16, hkv=8, B=8, hq=64, maxp=513, splits=0, dtype=0, head_dim=128):
    desc = kvq.CacheDesc(4104, ps, hkv, head_dim, dtype)
    return kvq.kvq_decode_plan(desc, B, hq, maxp, splits)


def test_plan_splits_cover_the_context():
    for ps in (16, 32, 64, 128):
        for maxp in (1, 2, 33, 513, 4096):
            for splits in (0, 1, 3, 64):
                st, ms, ws = _plan(ps=ps, maxp=maxp, splits=splits)
                ctx = maxp * ps
                assert st % 32 == 0 and st % min(ps, 32) == 0 and st % ps == 0 and st <= 8192
                assert ms == -(-ctx // st)
                assert (ws == 256) == (ms == 1)      # the arrival counters (8 x 8 x 4 B, padded) are always there
                if splits:
                    assert ms <= max(splits, -(-ctx // 8192))


def test_plan_rejects_unsupported_shapes():
    with pytest.raises(kvq.KvqError) as e:
        _plan(head_dim=64)
    assert e.value.status == 2
    with pytest.raises(kvq.KvqError) as e:
        _plan(ps=8)
    assert e.value.status == 2
    with pytest.raises(kvq.KvqError) as e:
        _plan(hq=16 * 8)          # g = 16
    assert e.value.status == 2
    with pytest.raises(kvq.KvqError) as e:
        _plan(hq=63)              # not a multiple of Hkv
    assert e.value.status == 1


def test_calls_with_null_pointers_fail_on_the_host():
    lib = kvq.load()
    desc = kvq.CacheDesc(64, 16, 8).c()
    st = lib.kvq_append(ctypes.byref(desc), None, None, None, 4, None, None, None, None, None, None)
    assert st == 1
    st = lib.kvq_tag_check(None, None, None, 4, 8, 16, None, 64, None, None)
    assert st == 1
    st = lib.kvq_decode_attn(ctypes.byref(desc), None, 2, 8, None, None, None, None, None, 8,
                             None, ctypes.c_float(0.1), None, None, 0, None, 0, 0, None)
    assert st == 1
    # zero-sized work is a no-op
    assert lib.kvq_append(ctypes.byref(desc), None, None, None, 0, None, None, None, None, None,
                          None) == 0
    assert lib.kvq_tag_check(None, None, None, 0, 8, 16, None, 64, None, None) == 0


def test_decode_step_argument_checks_on_the_host():
    """kvq_decode_step: null tensors, a missing tag array or output flags, and
    a short workspace are reported before anything reaches a GPU."""
    lib = kvq.load()
    desc = kvq.CacheDesc(4104, 16, 8).c()
    p = ctypes.c_void_p(0x10000)
    f = ctypes.c_float(0.1)
    st = lib.kvq_decode_step(ctypes.byref(desc), None, 2, 16, None, None, None, None, None, 8, None,
                             None, None, None, f, None, None, None, 0, None, 0, 0, None)
    assert st == 1
    big = 1 << 30
    for missing in range(3):                     # expected tags, live tags, flags
        tags = [p, p, p]
        tags[missing] = None
        st = lib.kvq_decode_step(ctypes.byref(desc), p, 8, 64, p, p, p, p, p, 513, p, *tags, f, p, p, p,
                                 0, p, big, 0, None)
        assert st == 1
    st = lib.kvq_decode_step(ctypes.byref(desc), p, 8, 64, p, p, p, p, p, 513, p, p, p, p, f, None, p, p,
                             0, p, big, 0, None)
    assert st == 1                               # no new token
    st = lib.kvq_decode_step(ctypes.byref(desc), p, 8, 64, p, p, p, p, p, 513, p, p, p, p, f, p, p, p,
                             0, p, 16, 0, None)
    assert st == 3                               # workspace too small
    assert lib.kvq_decode_step(ctypes.byref(desc), p, 0, 64, p, p, p, p, p, 513, p, p, p, p, f, p, p, p,
                               0, p, big, 0, None) == 0    # empty batch: nothing to do


def test_misaligned_pointer_rejected():
    lib = kvq.load()
    desc = kvq.CacheDesc(64, 16, 8).c()
    p = ctypes.c_void_p(0x1000 + 8)
    st = lib.kvq_append(ctypes.byref(desc), p, p, p, 4, p, p, None, p, p, None)
    assert st == 1


def test_workspace_too_small_is_reported():
    lib = kvq.load()
    desc = kvq.CacheDesc(4104, 16, 8).c()
    p = ctypes.c_void_p(0x10000)
    st = lib.kvq_decode_attn(ctypes.byref(desc), p, 8, 64, p, p, p, p, p, 513, p,
                             ctypes.c_float(0.1), None, p, 0, p, 16, 0, None)
    assert st == 3
    st = lib.kvq_decode_attn(ctypes.byref(desc), p, 8, 64, p, p, p, p, p, 513, p,
                             ctypes.c_float(0.1), None, p, 0, None, 1 << 30, 0, None)
    assert st == 3                      # the arrival counters are always needed


def test_auto_split_fills_the_resident_slots():
    # 8 requests x 8 KV heads at 8,208 tokens: 7 splits fill 448 of the 456
    # resident CTA slots of a 152-SM part in one wave (a GB300 itself takes 6,
    # the most that fit as resident clusters; a host without a GPU has none)
    st, ms, _ = _plan(ps=16, hkv=8, B=8, hq=64, maxp=513)
    assert ms in (6, 7)
    st, ms, _ = _plan(ps=64, hkv=8, B=4, hq=16, maxp=16384)     # long contexts
    assert st == 8192 and ms == 128


def test_batch_limit():
    with pytest.raises(kvq.KvqError) as e:
        _plan(B=65536)
    assert e.value.status == 2


def test_w4a16_plan_and_argument_checks():
    import ctypes
    lib = kvq.load()
    assert kvq.kvq_w4a16_plan(1, 12288, 5120) in range(1, 9)
    assert kvq.kvq_w4a16_plan(16, 64, 256, 1) == 1
    for m, n, k, ns in [(1, 64, 200, 0), (1, 60, 256, 0), (1, 64, 256, 2), (1, 64, 65536 + 256, 0)]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_w4a16_plan(m, n, k, ns)
        assert e.value.status == 2                       # unsupported shape / split count
    st = lib.kvq_w4a16_gemm(None, None, None, 1, 64, 256, None, 0, 0, None)
    assert st == 1                                        # null pointers: invalid argument
    st = lib.kvq_w4a16_gemm(None, None, None, 0, 64, 256, None, 0, 0, None)
    assert st == 0                                        # empty batch: nothing to do


@pytest.mark.parametrize("B,hq,ps,maxp,want", [
    (8, 64, 16, 513, (1184, 7)),       # uniform8: seven splits fill one wave of 456 slots
    (64, 32, 64, 511, (4096, 8)),      # ragged64: 4-8 waves at the longest context -> halved splits
    (4, 16, 64, 16384, (8192, 128)),   # long4: >= 8 waves -> 8,192-token splits
    (32, 32, 16, 257, (4128, 1)),      # 32 x 4,097: one split beats a workspace combine
    (64, 32, 16, 129, (1056, 2)),      # 64 x 2,049: no one-wave plan -> wave-filling rule
])
def test_planner_choices_on_a_host_without_a_gpu(B, hq, ps, maxp, want):
    """The planner's automatic choices with the host fallback (a 152-SM GB300,
    no clusters): the wave rules for long jobs and the one-wave estimate."""
    st, ms, _ = _plan(ps=ps, hkv=8, B=B, hq=hq, maxp=maxp)
    assert (st, ms) == want


def test_multi_token_plan_and_argument_checks():
    """kvq_decode_plan_mt / kvq_decode_attn_mt on the host: one query token
    plans exactly as kvq_decode_plan; n tokens need their rows' partials in
    the workspace, with an arrival counter per 16-row block (mma.sync build),
    or per (request, KV head) when an FP8 call has 64 or more rows per KV
    head (the tensor-memory kernel, splits of whole 64-token tiles); n
    outside 1..16 is refused before anything reaches a GPU."""
    desc = kvq.CacheDesc(4104, 16, 8)
    for splits in (0, 1, 12):
        assert kvq.kvq_decode_plan_mt(desc, 8, 1, 64, 513, splits) == \
            kvq.kvq_decode_plan(desc, 8, 64, 513, splits)
    rows = 8 * 4 * 64
    lse = (rows * 12 * 4 + 255) // 256 * 256
    # 4 tokens x 8 heads = 32 rows per KV head: the mma.sync build, counters
    # of 8 x 8 x ceil(32 / 16) blocks, for either cache type
    for d in (desc, kvq.CacheDesc(4104, 16, 8, cache_dtype=kvq.KVQ_CACHE_BF16)):
        _, ms, ws = kvq.kvq_decode_plan_mt(d, 8, 4, 64, 513, 12)
        assert ms == 12
        assert ws == (8 * 8 * 2 * 4 + 255) // 256 * 256 + lse + rows * 12 * 128 * 4
    # 8 tokens x 8 heads = 64 rows over FP8: the tensor-memory kernel, one
    # CTA (and counter) per (request, KV head), splits of whole 64-token tiles
    rows8 = 8 * 8 * 64
    lse8 = (rows8 * 12 * 4 + 255) // 256 * 256
    st, ms, ws = kvq.kvq_decode_plan_mt(desc, 8, 8, 64, 513, 12)
    assert ms == 12 and st % 64 == 0
    assert ws == (8 * 8 * 4 + 255) // 256 * 256 + lse8 + rows8 * 12 * 128 * 4
    # its automatic plan (host fallback: 152 SMs, one CTA each): uniform8's
    # shape takes 2 splits of 65 tiles, one wave of 128 CTAs
    st, ms, _ = kvq.kvq_decode_plan_mt(desc, 8, 8, 64, 513, 0)
    assert (st, ms) == (4160, 2)
    for n, status in ((0, 1), (17, 2)):
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_decode_plan_mt(desc, 8, n, 64, 513, 0)
        assert e.value.status == status
    lib = kvq.load()
    p = ctypes.c_void_p(0x10000)
    st = lib.kvq_decode_attn_mt(ctypes.byref(desc.c()), None, 8, 4, 64, p, p, p, p, p, 513, p,
                                ctypes.c_float(0.1), None, p, 0, p, 1 << 30, 0, None)
    assert st == 1                                  # null q
    st = lib.kvq_decode_attn_mt(ctypes.byref(desc.c()), p, 8, 4, 64, p, p, p, p, p, 513, p,
                                ctypes.c_float(0.1), None, p, 0, p, 16, 12, None)
    assert st == 3                                  # workspace too small
    # a request of a multi-token call takes at most 512 splits
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_plan_mt(kvq.CacheDesc(1 << 20, 64, 8), 1, 2, 16, 16384, 1024)
    assert e.value.status == 2
