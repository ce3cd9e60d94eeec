"""GPU parity of multi-token decode attention (kvq_decode_attn_mt) against
the oracle's multi-token attention: n new query tokens per request, query
token i attending causally to positions 0 .. L - n + i.  Through the C ABI;
tolerances as for single-token decode (1e-2 + 1e-2 |o| for bf16 output,
2e-4 + 2e-4 |o| for fp32)."""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
import workloads as W
from gpu_util import assert_close, compact_request, oracle_caches, out_to_np, to_np_bits
from kvq_harness import DeviceWorkload

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8, BF16 = kvq.KVQ_CACHE_FP8_E4M3, kvq.KVQ_CACHE_BF16
LENS = (1, 2, 3, 5, 16, 17, 33, 100, 257, 1000, 2049)


@pytest.fixture(autouse=True)
def _no_device_errors():
    kvq.kvq_device_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert kvq.kvq_device_error() == 0


def _q(w, n, seed):
    bits = W.normal_bf16(np.random.default_rng(seed), (w.batch, n, w.num_q_heads, w.head_dim))
    return bits, torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)


def _run(dw, q, n, fp32, splits, abort=None):
    w = dw.w
    out = torch.full((w.batch, n, w.num_q_heads, w.head_dim), 7.0,
                     dtype=torch.float32 if fp32 else torch.bfloat16, device=DEV)
    ws = kvq.workspace_for_mt(dw.desc, w.batch, n, w.num_q_heads, w.max_pages_per_seq, splits, DEV)
    kvq.kvq_decode_attn_mt(dw.desc, q, dw.k_cache, dw.v_cache, dw.k_scale, dw.v_scale,
                           dw.block_table, dw.seq_lens, w.softmax_scale, abort, out, ws, splits)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("g,ps", [(1, 16), (2, 64), (4, 16), (8, 16), (3, 32)])
@pytest.mark.parametrize("cache", ["fp8", "bf16"])
def test_multi_token_matches_oracle(n, g, ps, cache):
    w = W.make_custom(LENS, group=g, page_size=ps, seed=n * 10 + g, outlier_frac=0.01)
    dw = DeviceWorkload(w, FP8 if cache == "fp8" else BF16)
    dw.append()
    q_bits, q = _q(w, n, 7 + n)
    kc, vc = oracle_caches(dw)
    ref = oracle.decode_attn_multi(q_bits, kc, vc, dw.k_scale_host, dw.v_scale_host, w.block_table,
                                   w.seq_lens, w.softmax_scale)
    # 0: the planner; 1: one split; 5: a cluster of 5 splits; 12: through the workspace
    for splits in (0, 1, 5, 12):
        for fp32 in (True, False):
            got = out_to_np(_run(dw, q, n, fp32, splits))
            assert_close(got, ref, "fp32" if fp32 else "bf16", f"n{n} g{g} ps{ps} {cache} splits{splits}")


@pytest.mark.parametrize("n,g,ps", [(8, 8, 16), (16, 4, 32), (16, 8, 16), (11, 6, 64), (13, 5, 128)])
def test_tensor_memory_kernel_matches_oracle(n, g, ps):
    """64 or more query rows per KV head over an FP8 cache take the
    tensor-memory kernel: one CTA per (split, request, KV head) for every row,
    rows copied across the 128 M slots (66 and 65 rows: not a power of two,
    so part of the slots are padding), splits of whole 64-token tiles."""
    w = W.make_custom(LENS, group=g, page_size=ps, seed=n * 100 + g, outlier_frac=0.01)
    dw = DeviceWorkload(w)
    dw.append()
    q_bits, q = _q(w, n, 31 + n)
    kc, vc = oracle_caches(dw)
    ref = oracle.decode_attn_multi(q_bits, kc, vc, dw.k_scale_host, dw.v_scale_host, w.block_table,
                                   w.seq_lens, w.softmax_scale)
    for splits in (0, 1, 5, 12):
        for fp32 in (True, False):
            got = out_to_np(_run(dw, q, n, fp32, splits))
            assert_close(got, ref, "fp32" if fp32 else "bf16", f"n{n} g{g} ps{ps} splits{splits}")


def test_tensor_memory_kernel_zeroed_requests():
    """The tensor-memory kernel's zero paths: an empty request, a page id out
    of range, a request longer than its table row and an aborted one get
    zeros for every row; the others finite output."""
    n = 16
    w = W.make_custom([300, 0, 77, 500, 40], group=4, page_size=16, seed=19)
    w.block_table[2, 1] = w.num_pages + 3
    w.seq_lens[3] = w.block_table.shape[1] * 16 + 1
    abort = np.zeros(w.batch, np.uint8)
    abort[4] = 1
    dw = DeviceWorkload(w, populate=False)
    rng = np.random.default_rng(12)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    dw.k_cache.copy_(torch.from_numpy(rng.choice(finite, size=w.cache_shape()).astype(np.uint8)))
    dw.v_cache.copy_(torch.from_numpy(rng.choice(finite, size=w.cache_shape()).astype(np.uint8)))
    _, q = _q(w, n, 15)
    for splits in (1, 0, 4, 12):
        got = out_to_np(_run(dw, q, n, True, splits, torch.from_numpy(abort).to(DEV)))
        for r in (1, 2, 3, 4):
            assert np.all(got[r] == 0.0), (splits, r)
        assert np.all(np.isfinite(got[0])) and np.any(got[0] != 0)


def test_tensor_memory_kernel_many_splits():
    """A 70,000-token request with 16 query tokens x 8 heads (128 rows per KV
    head) in 122 splits: more (row, split) weights than the combine keeps in
    shared memory, so it computes them from the workspace as it goes.  Against
    the oracle, and against the same call in 8 splits (weights in the table)."""
    n = 16
    w = W.make_custom([70000, 3000], group=8, page_size=16, seed=61)
    dw = DeviceWorkload(w)
    dw.append()
    q_bits, q = _q(w, n, 62)
    got_many = out_to_np(_run(dw, q, n, True, 128))
    got_few = out_to_np(_run(dw, q, n, True, 8))
    plan = kvq.kvq_decode_plan_mt(dw.desc, w.batch, n, w.num_q_heads, w.max_pages_per_seq, 128)
    assert plan[1] * n * w.group > 8192
    assert_close(got_many, got_few, "fp32", "122 splits against 8")
    kc, vc, _, bt, seq = compact_request(dw, 0)
    ref = oracle.decode_attn_multi(q_bits[0:1], kc, vc, dw.k_scale_host, dw.v_scale_host, bt, seq,
                                   w.softmax_scale)
    assert_close(got_many[0:1], ref, "fp32", "70,000 tokens, 122 splits")


def test_one_query_token_is_kvq_decode_attn():
    w = W.make_custom(LENS, group=8, page_size=16, seed=3)
    dw = DeviceWorkload(w)
    dw.append()
    for splits in (0, 1, 12):
        out1 = dw.out(True)
        dw.attend(out1, dw.workspace(splits), None, splits)
        got = _run(dw, dw.q.view(w.batch, 1, w.num_q_heads, w.head_dim), 1, True, splits)
        assert torch.equal(got[:, 0], out1)


def test_multi_token_zeroed_requests():
    n = 4
    w = W.make_custom([300, 0, 77, 500, 40], group=4, page_size=16, seed=9)
    w.block_table[2, 1] = w.num_pages + 3                 # a page id out of range
    w.seq_lens[3] = w.block_table.shape[1] * 16 + 1       # longer than its table row
    abort = np.zeros(w.batch, np.uint8)
    abort[4] = 1
    dw = DeviceWorkload(w, populate=False)
    rng = np.random.default_rng(2)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    dw.k_cache.copy_(torch.from_numpy(rng.choice(finite, size=w.cache_shape()).astype(np.uint8)))
    dw.v_cache.copy_(torch.from_numpy(rng.choice(finite, size=w.cache_shape()).astype(np.uint8)))
    _, q = _q(w, n, 5)
    for splits in (1, 0, 4, 12):
        got = out_to_np(_run(dw, q, n, True, splits, torch.from_numpy(abort).to(DEV)))
        for r in (1, 2, 3, 4):
            assert np.all(got[r] == 0.0), (splits, r)
        assert np.all(np.isfinite(got[0])) and np.any(got[0] != 0)


@pytest.mark.parametrize("n", [2, 4, 8, 16])
def test_uniform8_multi_token_sampled(n):
    """The uniform8 workload (8 x 8,193 tokens, GQA 64/8) with n new query
    tokens per request: n * 8 query rows per KV head (the mma.sync build below
    64 rows, the tensor-memory kernel from 64); sampled requests against the
    oracle."""
    w = W.make("uniform8")
    dw = DeviceWorkload(w)
    dw.append()                                           # the last position too
    q_bits, q = _q(w, n, 11)
    out = _run(dw, q, n, False, 0)
    got = out_to_np(out)
    for r in (0, 7):
        kc, vc, _, bt, seq = compact_request(dw, r)
        ref = oracle.decode_attn_multi(q_bits[r:r + 1], kc, vc, dw.k_scale_host, dw.v_scale_host, bt,
                                       seq, w.softmax_scale)
        assert_close(got[r:r + 1], ref, "bf16", f"uniform8 n{n} request {r}")
