"""Host-side checks of the seeded workloads and of the pages' KV-size facts."""
import json
import os

import numpy as np
import pytest

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_kv_capacity.json")


def kv_formula(requests_tokens, layers, kv_heads, head_dim, bytes_per_elem):
    # page 4: requests x tokens x layers x KV heads x head_dim x 2 x bytes
    return requests_tokens * layers * kv_heads * head_dim * 2 * bytes_per_elem


def test_fp8_halves_kv_bytes_like_the_pages_capacity_figures():
    g = json.load(open(GOLDEN))
    ratio = g["fp8_tokens_in_memory"] / g["bf16_tokens_in_memory"]
    assert abs(ratio - 2.0) < 0.01          # the pages' own rounding (1.37 M / 686 K)
    w = W.make("uniform8")
    assert w.kv_bytes(1) * 2 == w.kv_bytes(2)
    per_token_fp8 = kv_formula(1, 1, w.num_kv_heads, w.head_dim, g["bytes_per_element"]["fp8_e4m3"])
    per_token_bf16 = kv_formula(1, 1, w.num_kv_heads, w.head_dim, g["bytes_per_element"]["bf16"])
    assert (per_token_fp8, per_token_bf16) == (2048, 4096)


@pytest.mark.parametrize("name,tokens", [
    ("tiny", 512), ("uniform8", 8 * 8193), ("long4", 131072 + 262144 + 524288 + 1048576)])
def test_workload_sizes(name, tokens):
    w = W.make(name)
    assert w.kv_tokens() == tokens
    assert w.kv_bytes(1) == kv_formula(tokens, 1, w.num_kv_heads, w.head_dim, 1)


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_tables_are_distinct_in_range_and_tagged(name):
    w = W.make(name)
    used = []
    for r in range(w.batch):
        n = -(-int(w.seq_lens[r]) // w.page_size)
        row = w.block_table[r]
        assert np.all(row[:n] >= 0) and np.all(row[:n] < w.num_pages)
        assert np.all(row[n:] == -1)
        assert np.array_equal(w.expected_tags[r, :n], w.page_tags[row[:n]])
        used.extend(row[:n].tolist())
    assert len(used) == len(set(used))


def test_workload_recipes():
    t = W.make("tiny")
    assert (t.batch, t.num_q_heads, t.num_kv_heads, t.page_size, t.num_pages) == (1, 8, 8, 16, 64)
    assert t.block_table.shape == (1, 32)
    r = W.make("ragged64")
    assert r.seq_lens.min() >= 1024 and r.seq_lens.max() <= 32768
    demand = sum(-(-int(L) // 64) for L in r.seq_lens)
    assert r.num_pages == int(np.ceil(1.2 * demand))
    c = W.make("churn")
    assert c.num_layers == 32 and c.page_size == 16 and c.seq_lens.min() >= 2048


def test_bf16_rounding_helper_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5e-3, 3.0e38], np.float32)
    b = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(b)
    import torch
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(back, lib)


def test_host_values_are_seeded():
    w = W.make("tiny")
    a, b = W.host_values(w), W.host_values(w)
    assert np.array_equal(a.k_prefill, b.k_prefill) and np.array_equal(a.q, b.q)
    assert a.k_scale.dtype == np.float32 and np.all(a.k_scale > 0)
