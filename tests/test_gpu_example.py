"""examples/decode_step.py runs as written; its step equals the separate
calls (kvq_tag_check, kvq_append, kvq_decode_attn) on the same inputs, and a
request's output matches the oracle fed the example's own bf16 inputs."""
import os
import runpy

import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
from gpu_util import assert_close, out_to_np, to_np_bits

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_example_runs_and_matches_separate_calls_and_oracle():
    torch.manual_seed(0)
    env = runpy.run_path(os.path.join(ROOT, "examples", "decode_step.py"), run_name="example")
    torch.cuda.synchronize()
    assert int(env["abort"].sum()) == 0
    desc, B, Hq, D, L, ps = env["desc"], env["B"], env["Hq"], env["D"], env["L"], env["ps"]
    # the same step as separate calls, on a copy of the cache the step left (the
    # new token is the only thing it wrote, so the append writes it again)
    k2, v2 = env["k_cache"].clone(), env["v_cache"].clone()
    out2 = torch.empty_like(env["out"])
    ab2 = torch.empty_like(env["abort"])
    kvq.kvq_tag_check(env["block_table"], env["expected"], env["seq_lens"], ps, env["page_tags"], ab2)
    kvq.kvq_append(desc, env["k_new"], env["v_new"], env["new_slots"], env["k_scale"], env["v_scale"],
                   ab2, k2, v2)
    kvq.kvq_decode_attn(desc, env["q"], k2, v2, env["k_scale"], env["v_scale"], env["block_table"],
                        env["seq_lens"], 1 / np.sqrt(D), ab2, out2,
                        kvq.workspace_for(desc, B, Hq, env["maxp"]))
    torch.cuda.synchronize()
    assert torch.equal(ab2, env["abort"])
    assert torch.equal(k2, env["k_cache"]) and torch.equal(v2, env["v_cache"])
    assert torch.equal(out2.view(torch.int16), env["out"].view(torch.int16))
    # request 0 against the oracle, from the example's bf16 inputs (prefill
    # rows 0 .. L-2 of the K = V tensor, then the new token)
    kp = to_np_bits(env["kp"][:L - 1])
    k = np.concatenate([kp, to_np_bits(env["k_new"][:1])])
    v = np.concatenate([kp, to_np_bits(env["v_new"][:1])])
    n_pages = -(-L // ps)
    shape = (n_pages, env["Hkv"], ps, D)
    kc, vc = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    ks = env["k_scale"].cpu().numpy()
    vs = env["v_scale"].cpu().numpy()
    oracle.append(kc, vc, k, v, np.arange(L, dtype=np.int64), ks, vs, page_size=ps)
    ref = oracle.decode_attn(to_np_bits(env["q"][:1]), kc, vc, ks, vs,
                             np.arange(n_pages, dtype=np.int32).reshape(1, -1),
                             np.array([L], np.int32), float(np.float32(1 / np.sqrt(D))))
    assert_close(out_to_np(env["out"][:1]), ref, "bf16", "example request 0")
