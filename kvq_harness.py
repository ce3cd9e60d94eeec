"""Device-resident workloads driven through the public binding (tests, smoke, bench).

Builds one layer of a named workload on the GPU: seeded bf16 K/V/Q generated
on the device (``workloads.normal_bf16_torch``), block tables and tags from
``workloads.make``, caches populated with ``kvq_append`` (the product path),
and the decode step tag-check -> append -> attention.  Every value a check
needs can be regenerated from the seed, so an oracle can be fed the same bf16
inputs without reading anything the CUDA path produced.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import workloads as W


def _gen(device, *key):
    g = torch.Generator(device=device)
    h = 0
    for k in key:
        h = (h * 1_000_003 + int(k) + 1) % (2**62)
    g.manual_seed(h)
    return g


class DeviceWorkload:
    """One layer of workload ``w`` resident in HBM."""

    def __init__(self, w: W.Workload, cache_dtype: int = kvq.KVQ_CACHE_FP8_E4M3,
                 device: str = "cuda", layer: int = 0, populate: bool = True):
        self.w = w
        self.device = device
        self.layer = layer
        self.cache_dtype = cache_dtype
        self.desc = kvq.CacheDesc(w.num_pages, w.page_size, w.num_kv_heads, w.head_dim, cache_dtype)
        dt = torch.uint8 if cache_dtype == kvq.KVQ_CACHE_FP8_E4M3 else torch.bfloat16
        self.k_cache = torch.zeros(w.cache_shape(), dtype=dt, device=device)
        self.v_cache = torch.zeros(w.cache_shape(), dtype=dt, device=device)
        self.block_table = torch.from_numpy(w.block_table).to(device)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(device)
        self.page_tags = torch.from_numpy(w.page_tags.view(np.int32)).to(device)
        self.expected_tags = torch.from_numpy(w.expected_tags.view(np.int32)).to(device)
        self.abort = torch.zeros(w.batch, dtype=torch.uint8, device=device)
        self.q = W.normal_bf16_torch((w.batch, w.num_q_heads, w.head_dim),
                                     _gen(device, w.seed, layer, 1 << 20), device)
        self.k_new, self.v_new = self.new_token_values()
        self.append_slots = torch.from_numpy(w.append_slot_mapping()).to(device)
        self.k_scale = torch.ones(w.num_kv_heads, dtype=torch.float32, device=device)
        self.v_scale = torch.ones(w.num_kv_heads, dtype=torch.float32, device=device)
        self.k_scale_host = np.ones(w.num_kv_heads, np.float32)
        self.v_scale_host = np.ones(w.num_kv_heads, np.float32)
        if populate:
            self.populate()

    # ---------------------------------------------------------------- values
    def prefill_values(self, r: int):
        """bf16 K, V of request r's prefill tokens 0 .. L-2, [L-1][Hkv][D] (device)."""
        w = self.w
        n = int(w.seq_lens[r]) - 1
        g = _gen(self.device, w.seed, self.layer, r)
        shape = (max(n, 0), w.num_kv_heads, w.head_dim)
        k = W.normal_bf16_torch(shape, g, self.device, w.outlier_frac)
        v = W.normal_bf16_torch(shape, g, self.device, w.outlier_frac)
        return k, v

    def new_token_values(self):
        w = self.w
        g = _gen(self.device, w.seed, self.layer, 1 << 21)
        shape = (w.batch, w.num_kv_heads, w.head_dim)
        return (W.normal_bf16_torch(shape, g, self.device, w.outlier_frac),
                W.normal_bf16_torch(shape, g, self.device, w.outlier_frac))

    def populate(self):
        """Scales from the prefill amax (recipe amax / 448), then append every prefill token."""
        w = self.w
        kmax = torch.zeros(w.num_kv_heads, dtype=torch.float32, device=self.device)
        vmax = torch.zeros_like(kmax)
        for r in range(w.batch):
            k, v = self.prefill_values(r)
            if k.shape[0]:
                kmax = torch.maximum(kmax, k.abs().float().amax(dim=(0, 2)))
                vmax = torch.maximum(vmax, v.abs().float().amax(dim=(0, 2)))
        if self.cache_dtype == kvq.KVQ_CACHE_FP8_E4M3:
            self.k_scale_host = W.scales_from_amax(kmax.cpu().numpy())
            self.v_scale_host = W.scales_from_amax(vmax.cpu().numpy())
            self.k_scale = torch.from_numpy(self.k_scale_host).to(self.device)
            self.v_scale = torch.from_numpy(self.v_scale_host).to(self.device)
        for r in range(w.batch):
            k, v = self.prefill_values(r)
            n = k.shape[0]
            if n == 0:
                continue
            slots = torch.from_numpy(w.slots_of(r, np.arange(n))).to(self.device)
            kvq.kvq_append(self.desc, k, v, slots, self.k_scale, self.v_scale, None,
                           self.k_cache, self.v_cache)

    # ------------------------------------------------------------------ step
    def workspace(self, num_splits: int = 0):
        return kvq.workspace_for(self.desc, self.w.batch, self.w.num_q_heads,
                                 self.w.max_pages_per_seq, num_splits, self.device)

    def out(self, fp32: bool = False):
        return torch.empty((self.w.batch, self.w.num_q_heads, self.w.head_dim),
                           dtype=torch.float32 if fp32 else torch.bfloat16, device=self.device)

    def tag_check(self, stream=None):
        kvq.kvq_tag_check(self.block_table, self.expected_tags, self.seq_lens, self.w.page_size,
                          self.page_tags, self.abort, stream)

    def append(self, abort=None, stream=None):
        kvq.kvq_append(self.desc, self.k_new, self.v_new, self.append_slots, self.k_scale,
                       self.v_scale, abort, self.k_cache, self.v_cache, stream)

    def attend(self, out, workspace, abort=None, num_splits=0, stream=None):
        return kvq.kvq_decode_attn(self.desc, self.q, self.k_cache, self.v_cache, self.k_scale,
                                   self.v_scale, self.block_table, self.seq_lens,
                                   self.w.softmax_scale, abort, out, workspace, num_splits, stream)

    def attend_append(self, out, workspace, num_splits=0, stream=None):
        """Attention with the append of each passing request's new token fused
        in (kvq_decode_attn_append), reading the flags the check wrote."""
        return kvq.kvq_decode_attn_append(self.desc, self.q, self.k_cache, self.v_cache,
                                          self.k_scale, self.v_scale, self.block_table,
                                          self.seq_lens, self.w.softmax_scale, self.abort,
                                          self.k_new, self.v_new, out, workspace, num_splits, stream)

    def tag_check_append(self, stream=None):
        kvq.kvq_tag_check_append(self.desc, self.block_table, self.expected_tags, self.seq_lens,
                                 self.page_tags, self.k_new, self.v_new, self.append_slots,
                                 self.k_scale, self.v_scale, self.k_cache, self.v_cache,
                                 self.abort, stream)

    def decode_step(self, out, workspace, num_splits=0, stream=None):
        """The whole step in one launch (kvq_decode_step): tag check, append
        of each passing request's token at seq_lens[r] - 1, attention."""
        kvq.kvq_decode_step(self.desc, self.q, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                            self.block_table, self.seq_lens, self.expected_tags, self.page_tags,
                            self.abort, self.w.softmax_scale, self.k_new, self.v_new, out, workspace,
                            num_splits, stream)
        return out

    def step(self, out, workspace, num_splits=0, stream=None, fused=True):
        """tag check -> append (skips aborted) -> attention (zeros for aborted).
        fused: the first two as one launch (kvq_tag_check_append)."""
        if fused:
            self.tag_check_append(stream)
        else:
            self.tag_check(stream)
            self.append(self.abort, stream)
        return self.attend(out, workspace, self.abort, num_splits, stream)

    # ---------------------------------------------------------- oracle feed
    STEP_INPUTS = ("q", "k_new", "v_new", "append_slots", "block_table", "seq_lens", "expected_tags")

    def pack_step_inputs(self):
        """Move the step's inputs into one device buffer (256-byte aligned
        segments) and return it with a pinned host copy, so that a host-fed
        step is a single host-to-device copy.  The workload's tensors become
        views of the device buffer."""
        import torch
        offs, total = [], 0
        for n in self.STEP_INPUTS:
            t = getattr(self, n)
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        dev = torch.zeros(total, dtype=torch.uint8, device=self.device)
        host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for n, o in zip(self.STEP_INPUTS, offs):
            t = getattr(self, n)
            nb = t.numel() * t.element_size()
            view = dev[o:o + nb].view(t.dtype).view(t.shape)
            view.copy_(t)
            host[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
            setattr(self, n, view)
        return host, dev

    def host_request(self, r: int):
        """bf16 bits (numpy uint16) of request r: K and V of all L tokens in
        logical order [L][Hkv][D], and q [Hq][D] -- regenerated from the seed."""
        k, v = self.prefill_values(r)
        k = torch.cat([k, self.k_new[r:r + 1]], 0)
        v = torch.cat([v, self.v_new[r:r + 1]], 0)
        to_np = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return to_np(k), to_np(v), to_np(self.q[r])


def compact_oracle_inputs(dw: DeviceWorkload, r: int, heads=None):
    """Inputs for the oracle restricted to request r: its tokens re-placed in
    a private pool of ceil(L / ps) pages (identity table).  The oracle's
    attention is invariant to where pages sit (pinned by the oracle tests)."""
    w = dw.w
    L = int(w.seq_lens[r])
    k, v, q = dw.host_request(r)
    ps = w.page_size
    n_pages = -(-L // ps)
    bt = np.arange(n_pages, dtype=np.int32).reshape(1, -1)
    slots = np.arange(L, dtype=np.int64)
    return dict(k=k, v=v, q=q[None], bt=bt, seq=np.array([L], np.int32), slots=slots,
                n_pages=n_pages)


def softmax_scale(head_dim: int = 128) -> float:
    return 1.0 / math.sqrt(head_dim)
