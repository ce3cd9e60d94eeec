"""Pins for the oracle's prefill -> decode handoff functions (CPU only).

Prefill keeps a BF16 cache and decode an FP8 one (blog post "Smaller,
faster, safer", section on quantising the KV cache: prefill is compute-bound,
so its cache stays BF16; the decode pool uses FP8), so pages handed to the
decode pool are quantised with per-KV-head scales.  Pinned against numpy's
max (library) and torch's float8_e4m3fn conversion (library)."""
import numpy as np
import torch

import oracle
import workloads as W


def _bf16_cache(rng, N=12, H=4, ps=16, D=128, scale=1.0):
    x = (rng.standard_normal((N, H, ps, D)) * scale).astype(np.float32)
    return W.f32_to_bf16_bits(x)


def test_amax_scales_match_numpy_max():
    rng = np.random.default_rng(1)
    kc, vc = _bf16_cache(rng), _bf16_cache(rng, scale=7.0)
    pages = np.array([3, 0, 7, 11], np.int32)
    ks, vs = oracle.amax_scales(kc, vc, pages)
    for cache, got in ((kc, ks), (vc, vs)):
        vals = np.abs(W.bf16_bits_to_f32(cache[pages]))            # [n][H][ps][D]
        amax = vals.max(axis=(0, 2, 3)).astype(np.float32)
        assert np.array_equal(got, (amax / np.float32(448)).astype(np.float32))


def test_amax_scales_of_zero_pages_are_one():
    kc = np.zeros((4, 2, 16, 128), np.uint16)
    ks, vs = oracle.amax_scales(kc, kc.copy(), np.array([1, 2], np.int32))
    assert np.all(ks == 1.0) and np.all(vs == 1.0)


def test_quantize_pages_match_torch_float8_and_touch_only_listed_pages():
    rng = np.random.default_rng(2)
    ksrc, vsrc = _bf16_cache(rng), _bf16_cache(rng, scale=30.0)
    src = np.array([5, 1, 9], np.int32)
    dst = np.array([0, 6, 2], np.int32)
    ks, vs = oracle.amax_scales(ksrc, vsrc, src)
    ks = (ks * np.float32(0.75)).astype(np.float32)                # some values saturate
    kd = np.full((8, 4, 16, 128), 0xA5, np.uint8)
    vd = kd.copy()
    oracle.quantize_pages(ksrc, vsrc, src, kd, vd, dst, ks, vs)
    for s_cache, d_cache, sc in ((ksrc, kd, ks), (vsrc, vd, vs)):
        quot = (W.bf16_bits_to_f32(s_cache[src]) / sc[None, :, None, None]).astype(np.float32)
        lib = torch.from_numpy(np.clip(quot, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(d_cache[dst], lib)
        rest = np.ones(8, bool)
        rest[dst] = False
        assert np.all(d_cache[rest] == 0xA5)
