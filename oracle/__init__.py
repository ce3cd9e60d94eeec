"""CPU fp64 oracle for the FP8 paged-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library: the arithmetic lives in ``kvq_oracle.c`` (plain C, fp64), compiled
with gcc by :func:`build` and driven here through ctypes over numpy arrays.

Source passages (blog post "Smaller, faster, safer: running Kimi and GLM at
scale" and its mirrors):
  * FP8 e4m3 KV cache instead of BF16, converted on read -- page 1, section
    "量化KV缓存" (quantised KV cache); page 3, section "FP8 省的不仅是显存".
  * per-page tags, expected (page, tag) per request, separate batched check
    before decode reads, abort on mismatch -- page 2, section "KV Cache
    完整性检查"; page 3, section "一个不能出错的共享缓存".
  * KV size = requests x tokens x layers x KV heads x head_dim x 2 x bytes
    -- page 4, section "显存为什么会成为长上下文推理的瓶颈".

Every function is pinned by ``tests/test_oracle_*.py`` against things other
than itself: torch's float8_e4m3fn conversion, a brute-force nearest-code
search, dense fp64 softmax attention from torch, closed forms and
invariances.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkvq_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c with gcc (OpenMP when the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode_n.argtypes = [P, P, ctypes.c_int64]
    lib.oracle_e4m3_encode_n.restype = None
    lib.oracle_e4m3_decode_n.argtypes = [P, P, ctypes.c_int64]
    lib.oracle_e4m3_decode_n.restype = None
    lib.oracle_append.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
    lib.oracle_append.restype = None
    lib.oracle_tag_check.argtypes = [P, P, P, i32, i32, i32, P, i32, P]
    lib.oracle_tag_check.restype = None
    lib.oracle_decode_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, P, P, P,
                                       P, i32, P, ctypes.c_float, P, P]
    lib.oracle_decode_attn.restype = None
    lib.oracle_decode_attn_multi.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                             P, P, P, i32, P, ctypes.c_float, P, P]
    lib.oracle_decode_attn_multi.restype = None
    lib.oracle_amax_scales.argtypes = [i32, i32, i32, P, P, P, i32, P, P]
    lib.oracle_amax_scales.restype = None
    lib.oracle_quantize_pages.argtypes = [i32, i32, i32, P, P, P, P, P, P, i32, P, P]
    lib.oracle_quantize_pages.restype = None
    lib.oracle_w4a16_gemm.argtypes = [i32, i32, i32, P, P, P, P]
    lib.oracle_w4a16_gemm.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous array of exactly ``dtype`` (no value conversion for views)."""
    a = np.asarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def e4m3_decode(codes) -> np.ndarray:
    """Real value (fp64) of each e4m3 code; NaN for S.1111.111."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, np.float64)
    lib.oracle_e4m3_decode_n(_ptr(codes), _ptr(out), codes.size)
    return out


def e4m3_encode(values_f32) -> np.ndarray:
    """e4m3 code of each fp32 value: nearest, ties to even, saturate at +-448."""
    lib = _load()
    v = np.ascontiguousarray(values_f32, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib.oracle_e4m3_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def append(k_cache, v_cache, k_new, v_new, slot_mapping, k_scale, v_scale,
           abort_flags=None, *, page_size: int):
    """In-place quantise-on-append into ``k_cache``/``v_cache`` (numpy).

    Caches are uint8 [N][Hkv][ps][D] (e4m3 codes) or uint16 (bf16 bits);
    ``k_new``/``v_new`` are uint16 bf16 bits [T][Hkv][D].
    """
    lib = _load()
    is_bf16 = k_cache.dtype == np.uint16
    N, Hkv, ps, D = k_cache.shape
    assert ps == page_size and v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    T = k_new.shape[0]
    assert k_new.shape == (T, Hkv, D) and v_new.shape == (T, Hkv, D)
    slot_mapping = _c(slot_mapping, np.int64)
    ks = _c(k_scale, np.float32) if k_scale is not None else np.ones(Hkv, np.float32)
    vs = _c(v_scale, np.float32) if v_scale is not None else np.ones(Hkv, np.float32)
    ab = None if abort_flags is None else _c(abort_flags, np.uint8)
    lib.oracle_append(T, Hkv, D, ps, N, int(is_bf16), _ptr(k_new), _ptr(v_new),
                      _ptr(slot_mapping), _ptr(ks), _ptr(vs), _ptr(ab),
                      _ptr(k_cache), _ptr(v_cache))


def tag_check(block_table, expected_tags, seq_lens, page_tags, *, page_size: int) -> np.ndarray:
    """Per-request abort flags (uint8 0/1)."""
    lib = _load()
    bt = _c(block_table, np.int32)
    et = _c(expected_tags, np.uint32)
    sl = _c(seq_lens, np.int32)
    pt = _c(page_tags, np.uint32)
    B, maxp = bt.shape
    assert et.shape == bt.shape and sl.shape == (B,)
    out = np.empty(B, np.uint8)
    lib.oracle_tag_check(_ptr(bt), _ptr(et), _ptr(sl), B, maxp, page_size,
                         _ptr(pt), pt.shape[0], _ptr(out))
    return out


def decode_attn(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                softmax_scale: float, abort_flags=None, *, num_q_heads: int | None = None) -> np.ndarray:
    """fp64 decode attention; returns float64 [B][Hq][D].

    ``q`` is uint16 bf16 bits [B][Hq][D]; caches as in :func:`append`.
    """
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    is_bf16 = k_cache.dtype == np.uint16
    N, Hkv, ps, D2 = k_cache.shape
    assert D2 == D and Hq % Hkv == 0
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ks = _c(k_scale, np.float32) if k_scale is not None else np.ones(Hkv, np.float32)
    vs = _c(v_scale, np.float32) if v_scale is not None else np.ones(Hkv, np.float32)
    ab = None if abort_flags is None else _c(abort_flags, np.uint8)
    out = np.empty((B, Hq, D), np.float64)
    lib.oracle_decode_attn(B, Hq, Hkv, D, ps, N, int(is_bf16), _ptr(q), _ptr(k_cache),
                           _ptr(v_cache), _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1],
                           _ptr(sl), ctypes.c_float(softmax_scale), _ptr(ab), _ptr(out))
    return out


def decode_attn_multi(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                      softmax_scale: float, abort_flags=None) -> np.ndarray:
    """fp64 multi-token decode attention; returns float64 [B][n][Hq][D].

    ``q`` is uint16 bf16 bits [B][n][Hq][D]: n new query tokens per request,
    the request's last n positions (seq_lens count them).  Query token i of
    request r attends causally to positions 0 .. seq_lens[r] - n + i; a query
    with no position to attend to, and every query of a request the
    single-token attention zeroes, gives zeros.
    """
    lib = _load()
    q = _c(q, np.uint16)
    B, n, Hq, D = q.shape
    is_bf16 = k_cache.dtype == np.uint16
    N, Hkv, ps, D2 = k_cache.shape
    assert D2 == D and Hq % Hkv == 0
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ks = _c(k_scale, np.float32) if k_scale is not None else np.ones(Hkv, np.float32)
    vs = _c(v_scale, np.float32) if v_scale is not None else np.ones(Hkv, np.float32)
    ab = None if abort_flags is None else _c(abort_flags, np.uint8)
    out = np.empty((B, n, Hq, D), np.float64)
    lib.oracle_decode_attn_multi(B, n, Hq, Hkv, D, ps, N, int(is_bf16), _ptr(q), _ptr(k_cache),
                                 _ptr(v_cache), _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1],
                                 _ptr(sl), ctypes.c_float(softmax_scale), _ptr(ab), _ptr(out))
    return out


def amax_scales(k_cache, v_cache, pages):
    """Per-KV-head (k_scale, v_scale): amax / 448 over the listed bf16 pages (1 if amax is 0)."""
    lib = _load()
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    assert kc.dtype == np.uint16 and vc.dtype == np.uint16
    N, Hkv, ps, D = kc.shape
    pg = _c(pages, np.int32)
    ks = np.empty(Hkv, np.float32)
    vs = np.empty(Hkv, np.float32)
    lib.oracle_amax_scales(Hkv, D, ps, _ptr(kc), _ptr(vc), _ptr(pg), pg.size, _ptr(ks), _ptr(vs))
    return ks, vs


def quantize_pages(k_src, v_src, src_pages, k_dst, v_dst, dst_pages, k_scale, v_scale):
    """In-place: bf16 pages src_pages[i] -> e4m3 pages dst_pages[i] of k_dst/v_dst."""
    lib = _load()
    ks_ = np.ascontiguousarray(k_src)
    vs_ = np.ascontiguousarray(v_src)
    N, Hkv, ps, D = ks_.shape
    assert k_dst.dtype == np.uint8 and k_dst.flags.c_contiguous and v_dst.flags.c_contiguous
    sp = _c(src_pages, np.int32)
    dp = _c(dst_pages, np.int32)
    assert sp.size == dp.size
    lib.oracle_quantize_pages(Hkv, D, ps, _ptr(ks_), _ptr(vs_), _ptr(sp), _ptr(k_dst), _ptr(v_dst),
                              _ptr(dp), sp.size, _ptr(_c(k_scale, np.float32)),
                              _ptr(_c(v_scale, np.float32)))


def w4a16_gemm(x_bits, w_packed, scale_bits):
    """y[m][n] = sum_k x[m][k] * q[n][k] * s[n][k / 128] in fp64.

    x_bits: uint16 bf16 bits [M][K]; w_packed: uint8 [N][K / 2] (low nibble =
    even k, two's complement); scale_bits: uint16 bf16 bits [N][K / 128]."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    w = _c(w_packed, np.uint8)
    sc = _c(scale_bits, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    assert K % 128 == 0 and w.shape == (N, K // 2) and sc.shape == (N, K // 128)
    y = np.empty((M, N), np.float64)
    lib.oracle_w4a16_gemm(M, N, K, _ptr(x), _ptr(w), _ptr(sc), _ptr(y))
    return y
