"""One layer of a paged FP8 KV cache and one decode step through the Python
binding of libkvq (GB300, sm_103a).

The step follows the order the integrity check asks for: the batched tag
check runs first, as its own pass, and writes one abort flag per request;
then each surviving request's new token is quantised into its slot (fused
into the check's launch here, kvq_tag_check_append), and only then does the
paged attention read the cache (kvq_decode_attn), skipping flagged requests.

Run:  python examples/decode_step.py
"""
import math
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import fp8_quantised_paged_kv_gb300 as kvq  # noqa: E402

B, Hq, Hkv, D, ps, L = 8, 64, 8, 128, 16, 8193        # requests, heads, head_dim, page size, tokens
maxp = -(-L // ps)                                    # pages per request
N = B * maxp                                          # pages in the pool
dev = "cuda"
desc = kvq.CacheDesc(N, ps, Hkv, D, kvq.KVQ_CACHE_FP8_E4M3)
k_cache = torch.zeros((N, Hkv, ps, D), dtype=torch.uint8, device=dev)      # e4m3 codes
v_cache = torch.zeros_like(k_cache)
k_scale = torch.full((Hkv,), 4.0 / 448, device=dev)                          # per KV head (amax / 448)
v_scale = torch.full((Hkv,), 4.0 / 448, device=dev)
block_table = torch.randperm(N, device=dev).int().view(B, maxp)            # page ids per request
page_tags = torch.randint(0, 2**31, (N,), dtype=torch.int32, device=dev)  # live tag per page
expected = page_tags[block_table.long()]                                   # the tags each request holds
seq_lens = torch.full((B,), L, dtype=torch.int32, device=dev)              # includes the new token

# prefill: write tokens 0 .. L-2 of every request (slot = page * ps + offset)
pos = torch.arange(L - 1, device=dev)
slots = (block_table[:, pos // ps].long() * ps + pos % ps).reshape(-1)
kp = torch.randn((B * (L - 1), Hkv, D), device=dev).bfloat16()
kvq.kvq_append(desc, kp, kp, slots, k_scale, v_scale, None, k_cache, v_cache)

# one decode step: tag check + append of token L-1 (one launch), then attention
q = torch.randn((B, Hq, D), device=dev).bfloat16()
k_new = torch.randn((B, Hkv, D), device=dev).bfloat16()
v_new = torch.randn((B, Hkv, D), device=dev).bfloat16()
new_slots = block_table[:, (L - 1) // ps].long() * ps + (L - 1) % ps     # where token L-1 goes
ws = kvq.workspace_for(desc, B, Hq, maxp)              # zeroed scratch the plan asks for
abort = torch.empty(B, dtype=torch.uint8, device=dev)  # written: 1 = a page changed owner
out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
kvq.kvq_tag_check_append(desc, block_table, expected, seq_lens, page_tags, k_new, v_new, new_slots,
                         k_scale, v_scale, k_cache, v_cache, abort)
kvq.kvq_decode_attn(desc, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                    1 / math.sqrt(D), abort, out, ws)
torch.cuda.synchronize()
assert kvq.kvq_device_error() == 0

if __name__ == "__main__":
    print(f"decode step done: {int(abort.sum())} of {B} requests aborted, "
          f"out[0, 0, :4] = {out[0, 0, :4].float().tolist()}")
