"""Prefill -> decode handoff on the GPU (bf16 pages -> e4m3 pages), through the
C ABI: per-KV-head scales and page codes bit-exact against the oracle, and
attention over the handed-over pages within tolerance."""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
import workloads as W
from gpu_util import assert_close, out_to_np, to_np_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16_cache(N, H, ps, seed, scale=1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (torch.randn((N, H, ps, 128), generator=g, device=DEV) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("ps", [16, 64])
def test_amax_scales_and_quantize_pages_bit_exact(ps):
    N, H = 40, 8
    ksrc, vsrc = _bf16_cache(N, H, ps, 1), _bf16_cache(N, H, ps, 2, scale=25.0)
    src = np.array([3, 17, 0, 39, 22, 8], np.int32)
    dst = np.array([5, 0, 11, 2, 9, 7], np.int32)
    src_desc = kvq.CacheDesc(N, ps, H, 128, kvq.KVQ_CACHE_BF16)
    dst_desc = kvq.CacheDesc(12, ps, H, 128, kvq.KVQ_CACHE_FP8_E4M3)
    ks = torch.empty(H, dtype=torch.float32, device=DEV)
    vs = torch.empty(H, dtype=torch.float32, device=DEV)
    src_d = torch.from_numpy(src).to(DEV)
    kvq.kvq_amax_scales(src_desc, ksrc, vsrc, src_d, ks, vs)
    ref_ks, ref_vs = oracle.amax_scales(to_np_bits(ksrc), to_np_bits(vsrc), src)
    assert np.array_equal(ks.cpu().numpy(), ref_ks) and np.array_equal(vs.cpu().numpy(), ref_vs)

    kd = torch.full((12, H, ps, 128), 0xA5, dtype=torch.uint8, device=DEV)
    vd = kd.clone()
    dst_l = dst.copy()
    src_l = src.copy()
    src_l[4] = N + 3                                  # out-of-range pair: skipped
    kvq.kvq_quantize_pages(src_desc, ksrc, vsrc, torch.from_numpy(src_l).to(DEV), dst_desc, kd, vd,
                           torch.from_numpy(dst_l).to(DEV), ks, vs)
    kref = np.full((12, H, ps, 128), 0xA5, np.uint8)
    vref = kref.copy()
    keep = np.arange(len(src)) != 4
    oracle.quantize_pages(to_np_bits(ksrc), to_np_bits(vsrc), src[keep], kref, vref, dst[keep],
                          ref_ks, ref_vs)
    assert np.array_equal(to_np_bits(kd), kref) and np.array_equal(to_np_bits(vd), vref)


def _split_nan(values_f32, codes_gpu, codes_ref):
    """NaN inputs may map to either NaN code; everything else must match bit for bit."""
    nan = np.isnan(values_f32)
    assert np.array_equal(codes_gpu[~nan], codes_ref[~nan])
    assert np.all((codes_gpu[nan] & 0x7F) == 0x7F)


@pytest.mark.parametrize("scales", [
    [1.0, 0.37, 3.1e-3, 17.5, 1e-30, 1e30, 2.0 ** -20, 3e38],
    [0.011, 0.0123, 0.2, 0.75, 1.0 / 448.0, 5.0 / 448.0, 100.0 / 448.0, 7.77],
])
def test_quantize_pages_every_bf16_value_bit_exact(scales):
    """Every bf16 bit pattern in every head, under given scales: the same codes
    as one IEEE division per element (scale 1 puts inputs on e4m3 ties; 3e38 has
    a subnormal reciprocal; 1e-30 overflows the quotient)."""
    ps, H, N = 16, 8, 32
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(N, 1, ps, 128)
    kbits = np.ascontiguousarray(np.broadcast_to(bits, (N, H, ps, 128)))
    vbits = kbits ^ np.uint16(0x8000)
    ksrc = torch.from_numpy(kbits.view(np.int16)).view(torch.bfloat16).to(DEV)
    vsrc = torch.from_numpy(vbits.view(np.int16)).view(torch.bfloat16).to(DEV)
    sk = np.array(scales, np.float32)
    sv = sk[::-1].copy()
    src = np.arange(N, dtype=np.int32)
    dst = np.random.default_rng(5).permutation(N).astype(np.int32)
    src_desc = kvq.CacheDesc(N, ps, H, 128, kvq.KVQ_CACHE_BF16)
    dst_desc = kvq.CacheDesc(N, ps, H, 128, kvq.KVQ_CACHE_FP8_E4M3)
    kd = torch.full((N, H, ps, 128), 0xA5, dtype=torch.uint8, device=DEV)
    vd = kd.clone()
    kvq.kvq_quantize_pages(src_desc, ksrc, vsrc, torch.from_numpy(src).to(DEV), dst_desc, kd, vd,
                           torch.from_numpy(dst).to(DEV), torch.from_numpy(sk).to(DEV),
                           torch.from_numpy(sv).to(DEV))
    kref = np.zeros((N, H, ps, 128), np.uint8)
    vref = np.zeros_like(kref)
    oracle.quantize_pages(kbits, vbits, src, kref, vref, dst, sk, sv)
    for ref, got, b, sc in ((kref, to_np_bits(kd), kbits, sk), (vref, to_np_bits(vd), vbits, sv)):
        vals = W.bf16_bits_to_f32(b[src]) / sc[None, :, None, None]
        _split_nan(vals, got[dst], ref[dst])


def test_decode_over_handed_over_pages():
    """A request prefilled in a bf16 cache, handed to an e4m3 cache, then decoded."""
    ps, H, g, L = 16, 8, 8, 1500
    n = -(-L // ps)
    ksrc, vsrc = _bf16_cache(n + 5, H, ps, 3), _bf16_cache(n + 5, H, ps, 4)
    src = np.random.default_rng(0).permutation(n + 5)[:n].astype(np.int32)
    dst = np.random.default_rng(1).permutation(2 * n)[:n].astype(np.int32)
    src_desc = kvq.CacheDesc(n + 5, ps, H, 128, kvq.KVQ_CACHE_BF16)
    dst_desc = kvq.CacheDesc(2 * n, ps, H, 128, kvq.KVQ_CACHE_FP8_E4M3)
    ks = torch.empty(H, dtype=torch.float32, device=DEV)
    vs = torch.empty(H, dtype=torch.float32, device=DEV)
    kvq.kvq_amax_scales(src_desc, ksrc, vsrc, torch.from_numpy(src).to(DEV), ks, vs)
    kd = torch.zeros((2 * n, H, ps, 128), dtype=torch.uint8, device=DEV)
    vd = torch.zeros_like(kd)
    kvq.kvq_quantize_pages(src_desc, ksrc, vsrc, torch.from_numpy(src).to(DEV), dst_desc, kd, vd,
                           torch.from_numpy(dst).to(DEV), ks, vs)
    gq = torch.Generator(device=DEV)
    gq.manual_seed(9)
    q = torch.randn((1, H * g, 128), generator=gq, device=DEV).to(torch.bfloat16)
    bt = torch.from_numpy(dst.reshape(1, -1)).to(DEV)
    seq = torch.tensor([L], dtype=torch.int32, device=DEV)
    out = torch.empty((1, H * g, 128), dtype=torch.float32, device=DEV)
    ws = kvq.workspace_for(dst_desc, 1, H * g, n, 0, DEV)
    kvq.kvq_decode_attn(dst_desc, q, kd, vd, ks, vs, bt, seq, 1 / np.sqrt(128), None, out, ws)
    torch.cuda.synchronize()
    # oracle: its own scales and codes from the same bf16 pages
    ref_ks, ref_vs = oracle.amax_scales(to_np_bits(ksrc), to_np_bits(vsrc), src)
    kref = np.zeros((2 * n, H, ps, 128), np.uint8)
    vref = kref.copy()
    oracle.quantize_pages(to_np_bits(ksrc), to_np_bits(vsrc), src, kref, vref, dst, ref_ks, ref_vs)
    ref = oracle.decode_attn(to_np_bits(q), kref, vref, ref_ks, ref_vs, dst.reshape(1, -1),
                             np.array([L], np.int32), float(np.float32(1 / np.sqrt(128))))
    assert_close(out_to_np(out), ref, "fp32", "handoff then decode")


def test_handoff_full_size_sampled_pages():
    """uniform8-sized prefill (4,104 bf16 pages of 8 heads x 16 tokens): scales
    bit-exact over all pages; sampled destination pages bit-exact."""
    ps, H, N = 16, 8, 8 * 513
    ksrc, vsrc = _bf16_cache(N, H, ps, 21), _bf16_cache(N, H, ps, 22, scale=7.0)
    rng = np.random.default_rng(2)
    src = rng.permutation(N).astype(np.int32)
    dst = rng.permutation(N).astype(np.int32)
    src_desc = kvq.CacheDesc(N, ps, H, 128, kvq.KVQ_CACHE_BF16)
    dst_desc = kvq.CacheDesc(N, ps, H, 128, kvq.KVQ_CACHE_FP8_E4M3)
    ks = torch.empty(H, dtype=torch.float32, device=DEV)
    vs = torch.empty(H, dtype=torch.float32, device=DEV)
    kvq.kvq_amax_scales(src_desc, ksrc, vsrc, torch.from_numpy(src).to(DEV), ks, vs)
    kd = torch.empty((N, H, ps, 128), dtype=torch.uint8, device=DEV)
    vd = torch.empty_like(kd)
    kvq.kvq_quantize_pages(src_desc, ksrc, vsrc, torch.from_numpy(src).to(DEV), dst_desc, kd, vd,
                           torch.from_numpy(dst).to(DEV), ks, vs)
    torch.cuda.synchronize()
    kbits, vbits = to_np_bits(ksrc), to_np_bits(vsrc)
    ref_ks, ref_vs = oracle.amax_scales(kbits, vbits, src)
    assert np.array_equal(ks.cpu().numpy(), ref_ks) and np.array_equal(vs.cpu().numpy(), ref_vs)
    pick = rng.choice(N, size=24, replace=False)
    kref = np.zeros((N, H, ps, 128), np.uint8)
    vref = np.zeros_like(kref)
    oracle.quantize_pages(kbits, vbits, src[pick], kref, vref, dst[pick], ref_ks, ref_vs)
    got_k, got_v = to_np_bits(kd), to_np_bits(vd)
    assert np.array_equal(got_k[dst[pick]], kref[dst[pick]])
    assert np.array_equal(got_v[dst[pick]], vref[dst[pick]])
