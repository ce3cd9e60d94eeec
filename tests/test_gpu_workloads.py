"""GPU parity on the named workloads at their full sizes, through the C ABI.

Each test runs the decode step the benchmark times (tag check -> FP8 append
of the new token -> split-K paged attention + LSE combine) on the full-size
workload, then checks sampled requests against the CPU oracle: the cache
bytes of every page the request owns bit for bit, its abort flag, and its
attention output within tolerance.  The oracle is fed the same seeded bf16
inputs, regenerated from the seed.
"""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
import workloads as W
from kvq_harness import DeviceWorkload
from gpu_util import (assert_close, compact_request, gpu_request_pages, oracle_attention,
                      oracle_caches, out_to_np, to_np_bits)

pytestmark = pytest.mark.gpu
FP8, BF16 = kvq.KVQ_CACHE_FP8_E4M3, kvq.KVQ_CACHE_BF16


@pytest.fixture(autouse=True)
def _fresh():
    kvq.kvq_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert kvq.kvq_device_error() == 0
    torch.cuda.empty_cache()


def _step(name, cache=FP8, fp32=False, num_splits=0):
    w = W.make(name)
    dw = DeviceWorkload(w, cache)
    out = dw.out(fp32)
    dw.step(out, dw.workspace(num_splits), num_splits)
    torch.cuda.synchronize()
    assert int(dw.abort.sum().item()) == 0
    return dw, out


def _check_request(dw, out, r, kind):
    kc, vc, q, bt, seq = compact_request(dw, r)
    gk, gv = gpu_request_pages(dw, r)
    assert np.array_equal(gk, kc), f"K cache bytes of request {r}"
    assert np.array_equal(gv, vc), f"V cache bytes of request {r}"
    ref = oracle.decode_attn(q, kc, vc, dw.k_scale_host, dw.v_scale_host, bt, seq,
                             dw.w.softmax_scale)
    return assert_close(out_to_np(out)[r:r + 1], ref, kind, f"{dw.w.name} request {r}")


@pytest.mark.parametrize("cache", [FP8, BF16])
@pytest.mark.parametrize("fp32", [False, True])
def test_tiny_whole_workload(cache, fp32):
    dw, out = _step("tiny", cache, fp32)
    kc, vc = oracle_caches(dw)
    assert np.array_equal(to_np_bits(dw.k_cache), kc) and np.array_equal(to_np_bits(dw.v_cache), vc)
    ref = oracle_attention(dw, kc, vc)
    assert_close(out_to_np(out), ref, "fp32" if fp32 else "bf16", "tiny")


@pytest.mark.parametrize("cache", [FP8, BF16])
def test_uniform8_sampled(cache):
    dw, out = _step("uniform8", cache)
    for r in (0, 7):
        _check_request(dw, out, r, "bf16")
    # same requests in fp32 output
    out32 = dw.out(True)
    dw.attend(out32, dw.workspace(0))
    for r in (3,):
        _check_request(dw, out32, r, "fp32")


def test_uniform8_fp8_bytes_are_half_of_bf16():
    w = W.make("uniform8")
    a = DeviceWorkload(w, FP8, populate=False)
    b = DeviceWorkload(w, BF16, populate=False)
    nbytes = lambda t: t.numel() * t.element_size()
    assert 2 * (nbytes(a.k_cache) + nbytes(a.v_cache)) == nbytes(b.k_cache) + nbytes(b.v_cache)
    assert w.kv_bytes(1) // w.kv_tokens() == 2048 and w.kv_bytes(2) // w.kv_tokens() == 4096


def test_ragged64_sampled():
    dw, out = _step("ragged64")
    L = dw.w.seq_lens
    for r in sorted({int(np.argmin(L)), int(np.argmax(L)), 17}):
        _check_request(dw, out, r, "bf16")


def test_long4_sampled_error_vs_length():
    dw, out = _step("long4")
    errs = {}
    for r in (0, 3):
        errs[int(dw.w.seq_lens[r])] = _check_request(dw, out, r, "bf16")
    print("long4 max |gpu - oracle| by context length:", errs)


def test_long4_at_256_splits_of_4096_tokens():
    """The long-context workload with its contexts cut into 4,096-token
    splits: 32, 64, 128 and 256 splits per request, merged by their
    log-sum-exp weights through the workspace; the shortest and the longest
    request against the oracle."""
    w = W.make("long4")
    dw = DeviceWorkload(w)
    split_tokens, max_splits, _ = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads,
                                                      w.max_pages_per_seq, 256)
    assert (split_tokens, max_splits) == (4096, 256)
    assert [-(-int(L) // split_tokens) for L in w.seq_lens] == [32, 64, 128, 256]
    out = dw.out(False)
    dw.step(out, dw.workspace(256), 256)
    torch.cuda.synchronize()
    assert int(dw.abort.sum().item()) == 0
    for r in (0, 3):
        _check_request(dw, out, r, "bf16")


def test_split_counts_agree_at_full_size():
    dw, out = _step("ragged64", fp32=True)
    for splits in (1, 7):
        o2 = dw.out(True)
        dw.attend(o2, dw.workspace(splits), None, splits)
        torch.cuda.synchronize()
        a, b = out_to_np(out), out_to_np(o2)
        assert np.all(np.abs(a - b) <= 4e-4 + 4e-4 * np.abs(a))


def test_packed_step_inputs_give_the_same_step():
    """The host-fed step keeps its inputs in one packed buffer (one copy per
    step); running the step on those views changes nothing."""
    w = W.make("uniform8", scale_down=8)
    dw = DeviceWorkload(w)
    out1 = dw.out(False)
    dw.step(out1, dw.workspace(0))
    host, dev = dw.pack_step_inputs()
    assert host.numel() == dev.numel() and host.numel() % 256 == 0
    dev.zero_()
    dev.copy_(host.to(dev.device))
    out2 = dw.out(False)
    dw.step(out2, dw.workspace(0))
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("lens,group", [([8193] * 16, 8), ([4097] * 32, 4), ([2049] * 64, 4)])
def test_mid_size_plans_sampled(lens, group):
    """Mid-size batches (268 MB each) with the plans the planner picks for them
    (a one-wave cluster of 3 splits, one split, a multi-wave workspace plan),
    through the one-launch step; sampled requests against the oracle."""
    w = W.make_custom(lens, group=group, page_size=16, num_kv_heads=8, seed=3, pool_factor=1.2)
    dw = DeviceWorkload(w, FP8)
    out = dw.out(False)
    print("plan", kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads, w.max_pages_per_seq, 0))
    dw.abort.fill_(1)
    dw.decode_step(out, dw.workspace(0))
    torch.cuda.synchronize()
    assert int(dw.abort.sum().item()) == 0
    for r in (0, len(lens) // 2, len(lens) - 1):
        _check_request(dw, out, r, "bf16")
