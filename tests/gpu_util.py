"""Helpers shared by the GPU parity tests: feed the oracle the same seeded
bf16 inputs the device used (regenerated, never read back from the CUDA
path's outputs) and compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# |gpu - oracle| <= ATOL + RTOL * |oracle| per element
TOL = {"bf16": (1e-2, 1e-2), "fp32": (2e-4, 2e-4)}


def to_np_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bits of a device tensor as numpy (uint8 / uint16)."""
    t = t.contiguous()
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def out_to_np(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(gpu: np.ndarray, ref: np.ndarray, kind: str, what: str = ""):
    atol, rtol = TOL[kind]
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements beyond {kind} tolerance; "
            f"max err {err.max():.3e}; first {idx.tolist()} gpu {gpu[bad][:5]} ref {ref[bad][:5]}")
    return float(err.max()) if err.size else 0.0


def oracle_caches(dw, requests=None):
    """Host caches (zero-initialised like the device ones) filled by the
    oracle's own append from the regenerated bf16 inputs of every request."""
    w = dw.w
    dt = np.uint8 if dw.k_cache.dtype == torch.uint8 else np.uint16
    kc = np.zeros(w.cache_shape(), dt)
    vc = np.zeros(w.cache_shape(), dt)
    for r in (range(w.batch) if requests is None else requests):
        L = int(w.seq_lens[r])
        if L <= 0:
            continue
        k, v, _ = dw.host_request(r)
        slots = w.slots_of(r, np.arange(L))
        oracle.append(kc, vc, k, v, slots, dw.k_scale_host, dw.v_scale_host, page_size=w.page_size)
    return kc, vc


def oracle_attention(dw, kc, vc, abort=None, block_table=None, seq_lens=None, q=None):
    w = dw.w
    q = to_np_bits(dw.q) if q is None else q
    return oracle.decode_attn(q, kc, vc, dw.k_scale_host, dw.v_scale_host,
                              w.block_table if block_table is None else block_table,
                              w.seq_lens if seq_lens is None else seq_lens,
                              w.softmax_scale, abort)


def compact_request(dw, r):
    """Oracle inputs of request r alone in a private pool (identity table)."""
    w = dw.w
    L = int(w.seq_lens[r])
    k, v, q = dw.host_request(r)
    n_pages = -(-L // w.page_size)
    dt = np.uint8 if dw.k_cache.dtype == torch.uint8 else np.uint16
    shape = (n_pages, w.num_kv_heads, w.page_size, w.head_dim)
    kc = np.zeros(shape, dt)
    vc = np.zeros(shape, dt)
    oracle.append(kc, vc, k, v, np.arange(L, dtype=np.int64), dw.k_scale_host, dw.v_scale_host,
                  page_size=w.page_size)
    bt = np.arange(n_pages, dtype=np.int32).reshape(1, -1)
    return kc, vc, q[None], bt, np.array([L], np.int32)


def gpu_request_pages(dw, r):
    """The device cache bytes of request r's pages, in logical page order."""
    w = dw.w
    n_pages = -(-int(w.seq_lens[r]) // w.page_size)
    idx = torch.from_numpy(w.block_table[r, :n_pages].astype(np.int64)).to(dw.k_cache.device)
    return to_np_bits(dw.k_cache.index_select(0, idx)), to_np_bits(dw.v_cache.index_select(0, idx))
