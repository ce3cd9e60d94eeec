"""The decode kernel's copy-timeout path, run on purpose and safely.

Every wait of a warp on one of its bulk copies has a time limit (about one
second).  A warp that gives up sets bit 0 of the device error word, waits
for the copies it still has in flight (with the full limit: they are
ordinary copies of valid pages, so they land), and its CTA publishes an
invalid partial, so the (request, KV head) it served gets zeros.  Here the
test hook kvq_diag_set_copy_wait_ns(0) gives every wait a zero time limit, so
each warp gives up at its first wait while its first copies are still in
flight; nothing is stalled and nothing faults.  The test checks the error
bit, that every (request, KV head) with tokens comes out as zeros, that no
copy was left in flight (bit 1 clear), and that the next call with the
normal limit matches the oracle everywhere."""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import workloads as W
from gpu_util import assert_close, oracle_attention, oracle_caches, out_to_np
from kvq_harness import DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_splits", [1, 4, 12])
def test_copy_wait_timeout_zeroes_what_it_served_and_recovers(num_splits):
    # 4 requests of 8,192 tokens: 64 chunks per warp with one split, so a
    # warp meets copies still in flight; two short ones for the edges
    w = W.make_custom([8192, 8192, 8192, 8192, 300, 33], group=8, page_size=16, seed=41)
    dw = DeviceWorkload(w)
    dw.append()
    kc, vc = oracle_caches(dw)
    ref = oracle_attention(dw, kc, vc)
    torch.cuda.synchronize()
    kvq.kvq_device_error(clear=True)
    out = dw.out(True)
    out.fill_(7.0)
    try:
        kvq.kvq_diag_set_copy_wait_ns(0)
        dw.attend(out, dw.workspace(num_splits), None, num_splits)
        torch.cuda.synchronize()
    finally:
        kvq.kvq_diag_set_copy_wait_ns(-1)
    bits = kvq.kvq_device_error(clear=True)
    assert bits & 1, "no warp gave up on a copy"
    assert not bits & 2, "a copy was left in flight"
    got = out_to_np(out)
    assert np.all(got == 0.0), "a (request, KV head) served by a failed CTA kept a result"
    # the normal limit again: every output matches
    out2 = dw.out(True)
    dw.attend(out2, dw.workspace(num_splits), None, num_splits)
    torch.cuda.synchronize()
    assert kvq.kvq_device_error() == 0
    assert_close(out_to_np(out2), ref, "fp32", "after the limit is restored")


@pytest.mark.parametrize("n,num_splits", [(4, 1), (4, 4), (16, 1), (16, 4)])
def test_copy_wait_timeout_in_the_multi_token_build(n, num_splits):
    """The same failure path in the multi-token builds: the mma.sync build
    (4 tokens x 4 heads = 16 rows per KV head) and the tensor-memory kernel
    (16 x 4 = 64 rows), whose converter warps give up at their first wait,
    raise the CTA's abort flag so that every other warp's wait gives up too,
    and whose producer lane drains the copies in flight before the tensor
    memory is freed.  Every query row of every (request, KV head) gets
    zeros, no copy is left in flight, and the next call matches the
    oracle."""
    import oracle
    w = W.make_custom([4096, 4096, 300, 33], group=4, page_size=16, seed=43)
    dw = DeviceWorkload(w)
    dw.append()
    kc, vc = oracle_caches(dw)
    q_bits = W.normal_bf16(np.random.default_rng(44), (w.batch, n, w.num_q_heads, w.head_dim))
    q = torch.from_numpy(q_bits.view(np.int16)).to("cuda").view(torch.bfloat16)
    ref = oracle.decode_attn_multi(q_bits, kc, vc, dw.k_scale_host, dw.v_scale_host, w.block_table,
                                   w.seq_lens, w.softmax_scale)
    ws = kvq.workspace_for_mt(dw.desc, w.batch, n, w.num_q_heads, w.max_pages_per_seq, num_splits)
    out = torch.full(q.shape, 7.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    kvq.kvq_device_error(clear=True)
    try:
        kvq.kvq_diag_set_copy_wait_ns(0)
        kvq.kvq_decode_attn_mt(dw.desc, q, dw.k_cache, dw.v_cache, dw.k_scale, dw.v_scale,
                               dw.block_table, dw.seq_lens, w.softmax_scale, None, out, ws, num_splits)
        torch.cuda.synchronize()
    finally:
        kvq.kvq_diag_set_copy_wait_ns(-1)
    bits = kvq.kvq_device_error(clear=True)
    assert bits & 1 and not bits & 2
    assert np.all(out_to_np(out) == 0.0)
    out2 = torch.empty_like(out)
    kvq.kvq_decode_attn_mt(dw.desc, q, dw.k_cache, dw.v_cache, dw.k_scale, dw.v_scale,
                           dw.block_table, dw.seq_lens, w.softmax_scale, None, out2, ws, num_splits)
    torch.cuda.synchronize()
    assert kvq.kvq_device_error() == 0
    assert_close(out_to_np(out2), ref, "fp32", "multi-token, after the limit is restored")
