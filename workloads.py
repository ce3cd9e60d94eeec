"""Seeded synthetic inputs for the FP8 paged-KV decode path.

This module is shared by the tests, the smoke check and the benchmark.  It
holds no arithmetic of the method itself (no quantisation, no attention, no
tag comparison): only random values, page placements, block tables, slot
positions and tags, plus the per-head scale recipe the workloads prescribe
(scale = amax / 448 over the prefill values of that head, computed in fp32
from the bf16 inputs -- an input to the quantiser, never checked).

The five workloads (sizes follow the page-4 KV-size formula: requests x
tokens x layers x KV heads x head_dim x {K, V} x bytes per element):

  tiny        1 request, MHA 8/8 heads, D 128, 512 tokens, page 16,
              32 pages at a seeded permutation of 64 physical pages
  uniform8    8 requests, GQA 64/8, 8,192 tokens + 1 appended, page 16,
              N(0,1) with 1 % of K/V elements x20 (outliers)
  ragged64    64 requests, GQA 32/8, lengths U{1,024..32,768}, page 64,
              pool 1.2 x demand, shuffled
  long4       4 requests, GQA 16/8, lengths 128K/256K/512K/1M, page 64
  churn       32 layers x 64 requests, GQA 32/8, lengths U{2,048..65,536},
              page 16, uint32 tags, 20 % of requests replaced per step,
              0.5 % of table entries pointed at stale-tag pages

A request's ``seq_len`` is the number of tokens attention reads after the
step's append: tokens 0 .. L-2 are the prefill context and token L-1 is the
one the step appends (uniform8 therefore attends over 8,193 tokens).
"""
from __future__ import annotations

import dataclasses
import math
import numpy as np

E4M3_MAX = 448.0


# ------------------------------------------------------------------ values

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even), as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, outlier_frac: float = 0.0,
                outlier_mult: float = 20.0) -> np.ndarray:
    """N(0,1) values (a seeded fraction multiplied by ``outlier_mult``) as bf16 bits."""
    x = rng.standard_normal(shape, dtype=np.float32)
    if outlier_frac > 0:
        mask = rng.random(shape, dtype=np.float32) < outlier_frac
        x = np.where(mask, x * np.float32(outlier_mult), x).astype(np.float32)
    return f32_to_bf16_bits(x)


def normal_bf16_torch(shape, generator, device, outlier_frac: float = 0.0,
                      outlier_mult: float = 20.0):
    """Device-side twin of :func:`normal_bf16` for the large workloads (torch bf16)."""
    import torch
    x = torch.randn(shape, generator=generator, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        mask = torch.rand(shape, generator=generator, device=device) < outlier_frac
        x = torch.where(mask, x * outlier_mult, x)
    return x.to(torch.bfloat16)


def scales_from_amax(amax_per_head: np.ndarray) -> np.ndarray:
    """Per-head scale recipe of the workloads: amax / 448 in fp32 (1 if amax is 0)."""
    a = np.asarray(amax_per_head, dtype=np.float32)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(a > 0, s, np.float32(1.0)).astype(np.float32)


def amax_per_head_bf16(values_bits: np.ndarray) -> np.ndarray:
    """max |x| per KV head of bf16 bits shaped [..., Hkv, D] (exact)."""
    v = np.abs(bf16_bits_to_f32(values_bits))
    hkv = v.shape[-2]
    return v.reshape(-1, hkv, v.shape[-1]).max(axis=(0, 2)).astype(np.float32)


# ---------------------------------------------------------------- structure

@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    seq_lens: np.ndarray          # int32 [B], tokens attended after the append
    block_table: np.ndarray       # int32 [B][max_pages]; -1 past each request's pages
    page_tags: np.ndarray         # uint32 [N] live tags
    expected_tags: np.ndarray     # uint32 [B][max_pages]; 0 past each request's pages
    softmax_scale: float
    seed: int
    outlier_frac: float = 0.0
    num_layers: int = 1

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def slots_of(self, r: int, positions) -> np.ndarray:
        """Cache slot (page * page_size + offset) of request r's token positions."""
        pos = np.asarray(positions, dtype=np.int64)
        pages = self.block_table[r][pos // self.page_size].astype(np.int64)
        return pages * self.page_size + pos % self.page_size

    def prefill_slot_mapping(self) -> np.ndarray:
        """Slots of tokens 0 .. L-2 of every request, requests in order."""
        return np.concatenate([self.slots_of(r, np.arange(int(L) - 1))
                               for r, L in enumerate(self.seq_lens)]).astype(np.int64)

    def append_slot_mapping(self) -> np.ndarray:
        """Slot of each request's appended token (position L-1); -1 (skip) if the
        request is empty or longer than its block-table row."""
        cap = self.block_table.shape[1] * self.page_size
        return np.array([self.slots_of(r, [int(L) - 1])[0] if 0 < L <= cap else -1
                         for r, L in enumerate(self.seq_lens)], dtype=np.int64)

    def kv_tokens(self) -> int:
        return int(np.sum(self.seq_lens))

    def kv_bytes(self, bytes_per_elem: int) -> int:
        """Algorithmic KV bytes one attention pass reads (K and V, every KV head)."""
        return self.kv_tokens() * self.num_kv_heads * self.head_dim * 2 * bytes_per_elem

    def cache_shape(self):
        return (self.num_pages, self.num_kv_heads, self.page_size, self.head_dim)


def _tables(rng, seq_lens, page_size, num_pages):
    """Place each request's pages at distinct shuffled physical pages."""
    pages_per_req = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    total = sum(pages_per_req)
    assert total <= num_pages
    perm = rng.permutation(num_pages)[:total].astype(np.int32)
    maxp = max(pages_per_req)
    bt = np.full((len(seq_lens), maxp), -1, dtype=np.int32)
    at = 0
    for r, p in enumerate(pages_per_req):
        bt[r, :p] = perm[at:at + p]
        at += p
    return bt


def _tags(rng, num_pages, bt):
    page_tags = rng.integers(0, 2**32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    expected = np.zeros(bt.shape, dtype=np.uint32)
    valid = bt >= 0
    expected[valid] = page_tags[bt[valid]]
    return page_tags, expected


def make(name: str, seed: int = 0, *, scale_down: int = 1) -> Workload:
    """Structure of a named workload.  ``scale_down`` > 1 shrinks the context
    lengths by that factor (ragged tails kept) for oracle-sized test cases."""
    rng = np.random.default_rng(seed)
    D = 128
    if name == "tiny":
        B, Hq, Hkv, ps, N = 1, 8, 8, 16, 64
        seq = np.array([512], np.int32)
        perm = rng.permutation(N).astype(np.int32)
        bt = perm[:32].reshape(1, 32).copy()
        page_tags, expected = _tags(rng, N, bt)
        return Workload(name, B, Hq, Hkv, D, ps, N, seq, bt, page_tags, expected,
                        1.0 / math.sqrt(D), seed)
    if name == "uniform8":
        B, Hq, Hkv, ps = 8, 64, 8, 16
        seq = np.full(B, max(8192 // scale_down, 1) + 1, np.int32)
        N = int(sum((int(L) + ps - 1) // ps for L in seq))
        outl = 0.01
    elif name == "ragged64":
        B, Hq, Hkv, ps = 64, 32, 8, 64
        lo, hi = 1024 // scale_down, 32768 // scale_down
        seq = rng.integers(lo, hi + 1, size=B).astype(np.int32)
        N = int(math.ceil(1.2 * sum((int(L) + ps - 1) // ps for L in seq)))
        outl = 0.0
    elif name == "long4":
        B, Hq, Hkv, ps = 4, 16, 8, 64
        seq = np.array([131072, 262144, 524288, 1048576], np.int32) // scale_down
        N = int(sum((int(L) + ps - 1) // ps for L in seq))
        outl = 0.0
    elif name == "churn":
        B, Hq, Hkv, ps = 64, 32, 8, 16
        lo, hi = 2048 // scale_down, 65536 // scale_down
        seq = rng.integers(lo, hi + 1, size=B).astype(np.int32)
        N = int(math.ceil(1.2 * sum((int(L) + ps - 1 + CHURN_STEPS) // ps for L in seq)))
        outl = 0.0
    else:
        raise KeyError(name)
    bt = _tables(rng, seq, ps, N)
    page_tags, expected = _tags(rng, N, bt)
    return Workload(name, B, Hq, Hkv, D, ps, N, seq, bt, page_tags, expected,
                    1.0 / math.sqrt(D), seed, outlier_frac=outl,
                    num_layers=32 if name == "churn" else 1)


def make_custom(lens, *, group: int, page_size: int, num_kv_heads: int = 2, seed: int = 0,
                pool_factor: float = 1.5, outlier_frac: float = 0.0, name: str = "custom") -> Workload:
    """A small workload with the given per-request lengths (test cases)."""
    rng = np.random.default_rng(seed)
    seq = np.asarray(lens, dtype=np.int32)
    demand = sum(max(-(-int(L) // page_size), 1) for L in seq)
    N = int(math.ceil(pool_factor * demand)) + 1
    bt = _tables(rng, np.maximum(seq, 1), page_size, N)
    page_tags, expected = _tags(rng, N, bt)
    D = 128
    return Workload(name, len(seq), num_kv_heads * group, num_kv_heads, D, page_size, N, seq, bt,
                    page_tags, expected, 1.0 / math.sqrt(D), seed, outlier_frac=outlier_frac)


CHURN_STEPS = 100
WORKLOADS = ("tiny", "uniform8", "ragged64", "long4", "churn")


# ----------------------------------------------------------- host values

@dataclasses.dataclass
class HostValues:
    """bf16 bits of one layer's inputs for a workload (numpy, host)."""
    q: np.ndarray            # [B][Hq][D]
    k_prefill: np.ndarray    # [T_prefill][Hkv][D]
    v_prefill: np.ndarray
    k_new: np.ndarray        # [B][Hkv][D]  (the step's appended token)
    v_new: np.ndarray
    k_scale: np.ndarray      # fp32 [Hkv]
    v_scale: np.ndarray


def host_values(w: Workload, seed: int | None = None, layer: int = 0) -> HostValues:
    """Seeded host-side values (small workloads; the oracle reads these)."""
    rng = np.random.default_rng([w.seed if seed is None else seed, 1 + layer])
    T = int(np.sum(w.seq_lens)) - w.batch
    q = normal_bf16(rng, (w.batch, w.num_q_heads, w.head_dim))
    kp = normal_bf16(rng, (T, w.num_kv_heads, w.head_dim), w.outlier_frac)
    vp = normal_bf16(rng, (T, w.num_kv_heads, w.head_dim), w.outlier_frac)
    kn = normal_bf16(rng, (w.batch, w.num_kv_heads, w.head_dim), w.outlier_frac)
    vn = normal_bf16(rng, (w.batch, w.num_kv_heads, w.head_dim), w.outlier_frac)
    src_k = kp if T > 0 else kn
    src_v = vp if T > 0 else vn
    ks = scales_from_amax(amax_per_head_bf16(src_k))
    vs = scales_from_amax(amax_per_head_bf16(src_v))
    return HostValues(q, kp, vp, kn, vn, ks, vs)
