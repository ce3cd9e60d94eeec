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
