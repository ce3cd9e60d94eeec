"""Python binding of the FP8 paged-KV decode path (libkvq.so, sm_103a).

Argument marshalling only: every step runs in the CUDA kernels behind the C
ABI declared in ``include/kvq.h``.  Functions carry the C names and take
torch CUDA tensors (device memory, PyTorch's streams); nothing here computes
on the host, and there is no CPU fallback -- if the library or a GPU is
missing the calls raise.

    kvq_tag_check(...)      separate batched per-page tag check -> abort flags
    kvq_append(...)         quantise-on-append of new K/V into paged slots
    kvq_decode_attn(...)    split-K paged decode attention + LSE combine
    kvq_decode_plan(...)    split / workspace sizes for kvq_decode_attn
    kvq_decode_attn_mt(...), kvq_decode_plan_mt(...)   several new query tokens per request
    kvq_decode_attn_append(...), kvq_tag_check_append(...)   fused forms
    kvq_decode_step(...)    tag check + append + attention of a decode step, one launch
    kvq_amax_scales(...), kvq_quantize_pages(...)            prefill -> decode handoff
    kvq_w4a16_gemm(...)     INT4 weight-only product for decode
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

from .build import LIB, build

KVQ_CACHE_FP8_E4M3 = 0
KVQ_CACHE_BF16 = 1
KVQ_OUT_BF16 = 0
KVQ_OUT_FP32 = 1

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace too small",
           4: "CUDA error"}


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class _Desc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32)]


@dataclasses.dataclass(frozen=True)
class CacheDesc:
    """Shape of one layer's K (and V) cache: [num_pages][num_kv_heads][page_size][head_dim]."""
    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim: int = 128
    cache_dtype: int = KVQ_CACHE_FP8_E4M3

    def c(self) -> _Desc:
        return _Desc(self.num_pages, self.page_size, self.num_kv_heads, self.head_dim,
                     self.cache_dtype)


_lib = None
_SIGS = {
    "kvq_append": ["desc", "p", "p", "p", "i32", "p", "p", "p", "p", "p", "p"],
    "kvq_tag_check": ["p", "p", "p", "i32", "i32", "i32", "p", "i32", "p", "p"],
    "kvq_decode_plan": ["desc", "i32", "i32", "i32", "i32", "p", "p", "p"],
    "kvq_decode_attn": ["desc", "p", "i32", "i32", "p", "p", "p", "p", "p", "i32", "p", "f32",
                        "p", "p", "i32", "p", "size", "i32", "p"],
    "kvq_decode_attn_append": ["desc", "p", "i32", "i32", "p", "p", "p", "p", "p", "i32", "p", "f32",
                               "p", "p", "p", "p", "i32", "p", "size", "i32", "p"],
    "kvq_decode_step": ["desc", "p", "i32", "i32", "p", "p", "p", "p", "p", "i32", "p", "p", "p", "p",
                        "f32", "p", "p", "p", "i32", "p", "size", "i32", "p"],
    "kvq_w4a16_plan": ["i32", "i32", "i32", "i32", "p"],
    "kvq_read_probe": ["p", "size", "p", "p"],
    "kvq_w4a16_gemm": ["p", "p", "p", "i32", "i32", "i32", "p", "i32", "i32", "p"],
    "kvq_device_error": ["p", "i32"],
    "kvq_diag_set_copy_wait_ns": ["i64"],
    "kvq_decode_plan_mt": ["desc", "i32", "i32", "i32", "i32", "i32", "p", "p", "p"],
    "kvq_decode_attn_mt": ["desc", "p", "i32", "i32", "i32", "p", "p", "p", "p", "p", "i32", "p", "f32",
                           "p", "p", "i32", "p", "size", "i32", "p"],
    "kvq_amax_scales": ["desc", "p", "p", "p", "i32", "p", "p", "p"],
    "kvq_quantize_pages": ["desc", "p", "p", "p", "desc", "p", "p", "p", "i32", "p", "p", "p"],
    "kvq_tag_check_append": ["desc", "p", "p", "p", "i32", "i32", "p", "p", "p", "p", "p", "p",
                             "p", "p", "p", "p"],
    "kvq_decode_attn_static_ws": ["desc", "p", "i32", "i32", "p", "p", "p", "p", "p", "i32", "p",
                                  "f32", "p", "p", "i32", "i32", "p"],
}
EXPORTED = tuple(_SIGS) + ("kvq_status_string",)


def load(path: str | None = None):
    """Load libkvq.so (building it first if absent); raises if that fails."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        build()
    lib = ctypes.CDLL(path)
    T = {"p": ctypes.c_void_p, "i32": ctypes.c_int32, "f32": ctypes.c_float,
         "size": ctypes.c_size_t, "desc": ctypes.POINTER(_Desc), "i64": ctypes.c_int64}
    for name, sig in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = [T[s] for s in sig]
        fn.restype = ctypes.c_int
    lib.kvq_status_string.argtypes = [ctypes.c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise KvqError(fn, status)


def _ptr(t):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _expect(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def kvq_append(desc: CacheDesc, k_new, v_new, slot_mapping, k_scale, v_scale, abort_flags,
               k_cache, v_cache, stream=None):
    """Quantise-on-append (FP8) or copy (BF16) of T new tokens into their slots."""
    import torch
    T = k_new.shape[0]
    _expect(k_new, torch.bfloat16, (T, desc.num_kv_heads, desc.head_dim), "k_new")
    _expect(v_new, torch.bfloat16, (T, desc.num_kv_heads, desc.head_dim), "v_new")
    _expect(slot_mapping, torch.int64, (T,), "slot_mapping")
    if abort_flags is not None:
        _expect(abort_flags, torch.uint8, (T,), "abort_flags")
    st = load().kvq_append(ctypes.byref(desc.c()), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T,
                           _ptr(k_scale), _ptr(v_scale), _ptr(abort_flags), _ptr(k_cache),
                           _ptr(v_cache), _stream(stream))
    _check("kvq_append", st)


def kvq_tag_check(block_table, expected_tags, seq_lens, page_size: int, page_tags, abort_flags,
                  stream=None):
    """Per-request abort flags (written into ``abort_flags``, uint8 [B])."""
    import torch
    B, maxp = block_table.shape
    _expect(block_table, torch.int32, None, "block_table")
    if expected_tags.element_size() != 4 or tuple(expected_tags.shape) != (B, maxp):
        raise ValueError("expected_tags: expected 32-bit tags [B][max_pages]")
    if page_tags.element_size() != 4 or page_tags.dim() != 1:
        raise ValueError("page_tags: expected 32-bit tags [num_pages]")
    _expect(seq_lens, torch.int32, (B,), "seq_lens")
    _expect(abort_flags, torch.uint8, (B,), "abort_flags")
    st = load().kvq_tag_check(_ptr(block_table), _ptr(expected_tags), _ptr(seq_lens), B, maxp,
                              page_size, _ptr(page_tags), page_tags.shape[0], _ptr(abort_flags),
                              _stream(stream))
    _check("kvq_tag_check", st)


def kvq_tag_check_append(desc: CacheDesc, block_table, expected_tags, seq_lens, page_tags,
                         k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache,
                         abort_flags, stream=None):
    """Tag check of every request, then the append of token r for request r
    unless it was aborted -- kvq_tag_check + kvq_append in one launch."""
    import torch
    B, maxp = block_table.shape
    _expect(block_table, torch.int32, None, "block_table")
    if expected_tags.element_size() != 4 or tuple(expected_tags.shape) != (B, maxp):
        raise ValueError("expected_tags: expected 32-bit tags [B][max_pages]")
    if page_tags.element_size() != 4 or page_tags.dim() != 1:
        raise ValueError("page_tags: expected 32-bit tags [num_pages]")
    _expect(seq_lens, torch.int32, (B,), "seq_lens")
    _expect(abort_flags, torch.uint8, (B,), "abort_flags")
    _expect(k_new, torch.bfloat16, (B, desc.num_kv_heads, desc.head_dim), "k_new")
    _expect(v_new, torch.bfloat16, (B, desc.num_kv_heads, desc.head_dim), "v_new")
    _expect(slot_mapping, torch.int64, (B,), "slot_mapping")
    st = load().kvq_tag_check_append(
        ctypes.byref(desc.c()), _ptr(block_table), _ptr(expected_tags), _ptr(seq_lens), B, maxp,
        _ptr(page_tags), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_scale),
        _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), _ptr(abort_flags), _stream(stream))
    _check("kvq_tag_check_append", st)


def kvq_amax_scales(desc: CacheDesc, k_cache, v_cache, pages, k_scale, v_scale, stream=None):
    """Per-KV-head scales amax / 448 of the listed pages of bf16 caches (written into k_scale, v_scale)."""
    import torch
    _expect(pages, torch.int32, None, "pages")
    _expect(k_scale, torch.float32, (desc.num_kv_heads,), "k_scale")
    _expect(v_scale, torch.float32, (desc.num_kv_heads,), "v_scale")
    st = load().kvq_amax_scales(ctypes.byref(desc.c()), _ptr(k_cache), _ptr(v_cache), _ptr(pages),
                                pages.numel(), _ptr(k_scale), _ptr(v_scale), _stream(stream))
    _check("kvq_amax_scales", st)


def kvq_quantize_pages(src_desc: CacheDesc, k_src, v_src, src_pages, dst_desc: CacheDesc, k_dst,
                       v_dst, dst_pages, k_scale, v_scale, stream=None):
    """bf16 pages src_pages[i] -> e4m3 pages dst_pages[i], per-KV-head scales."""
    import torch
    _expect(src_pages, torch.int32, None, "src_pages")
    _expect(dst_pages, torch.int32, (src_pages.numel(),), "dst_pages")
    st = load().kvq_quantize_pages(ctypes.byref(src_desc.c()), _ptr(k_src), _ptr(v_src),
                                   _ptr(src_pages), ctypes.byref(dst_desc.c()), _ptr(k_dst),
                                   _ptr(v_dst), _ptr(dst_pages), src_pages.numel(), _ptr(k_scale),
                                   _ptr(v_scale), _stream(stream))
    _check("kvq_quantize_pages", st)


def kvq_decode_plan(desc: CacheDesc, batch: int, num_q_heads: int, max_pages_per_seq: int,
                    num_splits: int = 0):
    """(split_tokens, max_splits, workspace_bytes) that kvq_decode_attn will use."""
    a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    st = load().kvq_decode_plan(ctypes.byref(desc.c()), batch, num_q_heads, max_pages_per_seq,
                                num_splits, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    _check("kvq_decode_plan", st)
    return a.value, b.value, c.value


def kvq_decode_plan_mt(desc: CacheDesc, batch: int, num_query_tokens: int, num_q_heads: int,
                       max_pages_per_seq: int, num_splits: int = 0):
    """(split_tokens, max_splits, workspace_bytes) that kvq_decode_attn_mt will use."""
    a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_size_t()
    st = load().kvq_decode_plan_mt(ctypes.byref(desc.c()), batch, num_query_tokens, num_q_heads,
                                   max_pages_per_seq, num_splits, ctypes.byref(a), ctypes.byref(b),
                                   ctypes.byref(c))
    _check("kvq_decode_plan_mt", st)
    return a.value, b.value, c.value


def workspace_for_mt(desc: CacheDesc, batch, num_query_tokens, num_q_heads, max_pages_per_seq,
                     num_splits=0, device="cuda"):
    """Allocate (with torch) the zero-filled workspace of a multi-token decode call."""
    import torch
    nbytes = kvq_decode_plan_mt(desc, batch, num_query_tokens, num_q_heads, max_pages_per_seq,
                                num_splits)[2]
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def workspace_for(desc: CacheDesc, batch, num_q_heads, max_pages_per_seq, num_splits=0, device="cuda"):
    """Allocate (with torch) the zero-filled decode workspace the plan asks for."""
    import torch
    nbytes = kvq_decode_plan(desc, batch, num_q_heads, max_pages_per_seq, num_splits)[2]
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def _decode(fn_name, desc: CacheDesc, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
            softmax_scale, abort_flags, out, workspace, num_splits, stream):
    import torch
    B, Hq, D = q.shape
    _expect(q, torch.bfloat16, (B, Hq, desc.head_dim), "q")
    _expect(block_table, torch.int32, None, "block_table")
    _expect(seq_lens, torch.int32, (B,), "seq_lens")
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("out: expected bf16 or fp32 [B][Hq][D]")
    out_dtype = KVQ_OUT_FP32 if out.dtype == torch.float32 else KVQ_OUT_BF16
    if abort_flags is not None:
        _expect(abort_flags, torch.uint8, (B,), "abort_flags")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = getattr(load(), fn_name)(
        ctypes.byref(desc.c()), _ptr(q), B, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        ctypes.c_float(softmax_scale), _ptr(abort_flags), _ptr(out), out_dtype, _ptr(workspace),
        ws_bytes, num_splits, _stream(stream))
    _check(fn_name, st)
    return out


def kvq_decode_attn(desc, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                    softmax_scale, abort_flags, out, workspace, num_splits=0, stream=None):
    """Paged decode attention into ``out`` (bf16 or fp32 [B][Hq][D])."""
    return _decode("kvq_decode_attn", desc, q, k_cache, v_cache, k_scale, v_scale, block_table,
                   seq_lens, softmax_scale, abort_flags, out, workspace, num_splits, stream)


def kvq_decode_attn_mt(desc, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                       softmax_scale, abort_flags, out, workspace, num_splits=0, stream=None):
    """Decode attention for n new query tokens per request, causal among them:
    q bf16 [B][n][Hq][D] into ``out`` (bf16 or fp32 [B][n][Hq][D])."""
    import torch
    B, n, Hq, D = q.shape
    _expect(q, torch.bfloat16, (B, n, Hq, desc.head_dim), "q")
    _expect(block_table, torch.int32, None, "block_table")
    _expect(seq_lens, torch.int32, (B,), "seq_lens")
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, n, Hq, D):
        raise ValueError("out: expected bf16 or fp32 [B][n][Hq][D]")
    out_dtype = KVQ_OUT_FP32 if out.dtype == torch.float32 else KVQ_OUT_BF16
    if abort_flags is not None:
        _expect(abort_flags, torch.uint8, (B,), "abort_flags")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().kvq_decode_attn_mt(
        ctypes.byref(desc.c()), _ptr(q), B, n, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        ctypes.c_float(softmax_scale), _ptr(abort_flags), _ptr(out), out_dtype, _ptr(workspace),
        ws_bytes, num_splits, _stream(stream))
    _check("kvq_decode_attn_mt", st)


def kvq_decode_attn_append(desc, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                           softmax_scale, abort_flags, k_new, v_new, out, workspace, num_splits=0,
                           stream=None):
    """Append request r's new token (row r of k_new/v_new, bf16 [B][Hkv][D]) at
    its position seq_lens[r] - 1, then paged decode attention into ``out``:
    one launch, the same results as kvq_append followed by kvq_decode_attn."""
    import torch
    B, Hq, D = q.shape
    _expect(q, torch.bfloat16, (B, Hq, desc.head_dim), "q")
    _expect(block_table, torch.int32, None, "block_table")
    _expect(seq_lens, torch.int32, (B,), "seq_lens")
    _expect(k_new, torch.bfloat16, (B, desc.num_kv_heads, desc.head_dim), "k_new")
    _expect(v_new, torch.bfloat16, (B, desc.num_kv_heads, desc.head_dim), "v_new")
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("out: expected bf16 or fp32 [B][Hq][D]")
    out_dtype = KVQ_OUT_FP32 if out.dtype == torch.float32 else KVQ_OUT_BF16
    if abort_flags is not None:
        _expect(abort_flags, torch.uint8, (B,), "abort_flags")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().kvq_decode_attn_append(
        ctypes.byref(desc.c()), _ptr(q), B, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        ctypes.c_float(softmax_scale), _ptr(abort_flags), _ptr(k_new), _ptr(v_new), _ptr(out),
        out_dtype, _ptr(workspace), ws_bytes, num_splits, _stream(stream))
    _check("kvq_decode_attn_append", st)
    return out


def kvq_decode_step(desc, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, expected_tags,
                    page_tags, abort_flags, softmax_scale, k_new, v_new, out, workspace, num_splits=0,
                    stream=None):
    """A whole decode step in one launch: the tag check of every request
    (flags written into ``abort_flags``, uint8 [B]), then, for each request
    that passed, the append of its new token at seq_lens[r] - 1 and paged
    decode attention into ``out``.  The same results as kvq_tag_check
    followed by kvq_decode_attn_append."""
    import torch
    B, Hq, D = q.shape
    maxp = block_table.shape[1]
    _expect(q, torch.bfloat16, (B, Hq, desc.head_dim), "q")
    _expect(block_table, torch.int32, None, "block_table")
    _expect(seq_lens, torch.int32, (B,), "seq_lens")
    if expected_tags.element_size() != 4 or tuple(expected_tags.shape) != (B, maxp):
        raise ValueError("expected_tags: expected 32-bit tags [B][max_pages]")
    if page_tags.element_size() != 4 or tuple(page_tags.shape) != (desc.num_pages,):
        raise ValueError("page_tags: expected 32-bit tags [num_pages]")
    _expect(abort_flags, torch.uint8, (B,), "abort_flags")
    _expect(k_new, torch.bfloat16, (B, desc.num_kv_heads, desc.head_dim), "k_new")
    _expect(v_new, torch.bfloat16, (B, desc.num_kv_heads, desc.head_dim), "v_new")
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("out: expected bf16 or fp32 [B][Hq][D]")
    out_dtype = KVQ_OUT_FP32 if out.dtype == torch.float32 else KVQ_OUT_BF16
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().kvq_decode_step(
        ctypes.byref(desc.c()), _ptr(q), B, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), maxp, _ptr(seq_lens), _ptr(expected_tags), _ptr(page_tags),
        _ptr(abort_flags), ctypes.c_float(softmax_scale), _ptr(k_new), _ptr(v_new), _ptr(out),
        out_dtype, _ptr(workspace), ws_bytes, num_splits, _stream(stream))
    _check("kvq_decode_step", st)
    return out


def kvq_read_probe(src, sink, stream=None):
    """Calibration: read every byte of the CUDA tensor ``src`` once with a
    plain streaming kernel, XOR-ing its 32-bit words into ``sink`` (a
    zeroed 1-element int32/uint32 CUDA tensor)."""
    nbytes = src.numel() * src.element_size()
    if sink.element_size() != 4 or sink.numel() < 1:
        raise ValueError("sink: expected a 32-bit CUDA tensor")
    _check("kvq_read_probe", load().kvq_read_probe(_ptr(src), nbytes, _ptr(sink), _stream(stream)))


def kvq_w4a16_plan(m: int, n: int, k: int, num_splits: int = 0) -> int:
    """Split count of K that kvq_w4a16_gemm uses for these shapes."""
    s = ctypes.c_int32()
    _check("kvq_w4a16_plan", load().kvq_w4a16_plan(m, n, k, num_splits, ctypes.byref(s)))
    return s.value


def kvq_w4a16_gemm(x, w, scales, y, num_splits: int = 0, stream=None):
    """y = x W^T with INT4 weights: x bf16 [M][K], w uint8 [N][K/2] (signed
    nibbles, low nibble = even k), scales bf16 [N][K/128]; y bf16 or fp32 [M][N]."""
    import torch
    M, K = x.shape
    N = w.shape[0]
    _expect(x, torch.bfloat16, (M, K), "x")
    _expect(w, torch.uint8, (N, K // 2), "w")
    _expect(scales, torch.bfloat16, (N, K // 128), "scales")
    if y.dtype not in (torch.bfloat16, torch.float32) or tuple(y.shape) != (M, N):
        raise ValueError("y: expected bf16 or fp32 [M][N]")
    st = load().kvq_w4a16_gemm(_ptr(x), _ptr(w), _ptr(scales), M, N, K, _ptr(y),
                               KVQ_OUT_FP32 if y.dtype == torch.float32 else KVQ_OUT_BF16,
                               num_splits, _stream(stream))
    _check("kvq_w4a16_gemm", st)
    return y


def kvq_diag_set_copy_wait_ns(ns: int) -> None:
    """Test hook: the decode kernel's limit on each wait for a bulk copy, for
    later launches (0 = give up at once; negative = the default of about 1 s)."""
    _check("kvq_diag_set_copy_wait_ns", load().kvq_diag_set_copy_wait_ns(int(ns)))


def kvq_device_error(clear: bool = False) -> int:
    """Sticky device error bits of the current device (synchronous)."""
    v = ctypes.c_uint32()
    _check("kvq_device_error", load().kvq_device_error(ctypes.byref(v), int(clear)))
    return v.value


def kvq_status_string(status: int) -> str:
    return load().kvq_status_string(status).decode()
