"""kvq_decode_attn_static_ws: decode attention for callers that cannot
allocate device memory while decoding (an engine whose device memory is all
in its own pool, or C code without an allocator).  The entry point uses the
library's built-in scratch array instead of a caller workspace; this file
checks it through the C ABI against kvq_decode_attn with a workspace, on two
calls in a row, and checks that it refuses plans larger than the array.
It is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import workloads as W
from gpu_util import assert_close, oracle_attention, oracle_caches, out_to_np
from kvq_harness import DeviceWorkload

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_call(dw, out, num_splits, abort=None):
    w = dw.w
    return kvq.load().kvq_decode_attn_static_ws(
        ctypes.byref(dw.desc.c()), _p(dw.q), w.batch, w.num_q_heads, _p(dw.k_cache), _p(dw.v_cache),
        _p(dw.k_scale), _p(dw.v_scale), _p(dw.block_table), w.max_pages_per_seq, _p(dw.seq_lens),
        ctypes.c_float(w.softmax_scale), _p(abort), _p(out),
        kvq.KVQ_OUT_FP32 if out.dtype == torch.float32 else kvq.KVQ_OUT_BF16, num_splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# 0: the planner's choice; 4: a cluster of 4 splits (partials in shared
# memory); 12: more splits than a cluster holds, so the partials go through
# the built-in scratch and the last split to finish merges them
@pytest.mark.parametrize("num_splits", [0, 4, 12])
def test_static_scratch_matches_the_workspace_entry_point_twice(num_splits):
    w = W.make_custom([3000, 700, 4100, 1, 2500, 0], group=8, page_size=16, seed=21,
                      outlier_frac=0.01)
    dw = DeviceWorkload(w)
    dw.append()
    if num_splits == 12:
        need = kvq.kvq_decode_plan(dw.desc, w.batch, w.num_q_heads, w.max_pages_per_seq, 12)[2]
        assert (w.batch * w.num_kv_heads * 4 + 255) // 256 * 256 < need <= (16 << 20)
    abort_np = np.zeros(w.batch, np.uint8)
    abort_np[2] = 1
    abort = torch.from_numpy(abort_np).to("cuda")
    ref = dw.out()
    dw.attend(ref, dw.workspace(num_splits), abort, num_splits)
    torch.cuda.synchronize()
    kc, vc = oracle_caches(dw)
    oracle_out = oracle_attention(dw, kc, vc, abort_np)
    for call in range(2):
        out = dw.out()
        out.fill_(7.0)
        assert _static_call(dw, out, num_splits, abort) == 0
        torch.cuda.synchronize()
        assert_close(out_to_np(out), out_to_np(ref), "bf16", f"static scratch, call {call + 1}")
        assert_close(out_to_np(out), oracle_out, "bf16", f"static scratch vs oracle, call {call + 1}")
    assert kvq.kvq_device_error() == 0


def test_static_scratch_refuses_plans_beyond_its_size():
    B, hq, hkv, ps, maxp = 64, 64, 8, 16, 4096
    desc = kvq.CacheDesc(16, ps, hkv)
    need = kvq.kvq_decode_plan(desc, B, hq, maxp, 256)[2]
    assert need > (16 << 20)
    dev = "cuda"
    q = torch.zeros((B, hq, 128), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((16, hkv, ps, 128), dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    sc = torch.ones(hkv, dtype=torch.float32, device=dev)
    bt = torch.full((B, maxp), -1, dtype=torch.int32, device=dev)
    seq = torch.zeros(B, dtype=torch.int32, device=dev)          # even a launch would read no page
    out = torch.empty((B, hq, 128), dtype=torch.bfloat16, device=dev)
    st = kvq.load().kvq_decode_attn_static_ws(
        ctypes.byref(desc.c()), _p(q), B, hq, _p(kc), _p(vc), _p(sc), _p(sc), _p(bt), maxp, _p(seq),
        ctypes.c_float(0.1), None, _p(out), kvq.KVQ_OUT_BF16, 256,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3                                              # KVQ_ERR_WORKSPACE
