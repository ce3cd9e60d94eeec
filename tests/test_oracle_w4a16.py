"""Pins of the oracle's INT4 weight-only product (y = x W^T with W = q * s,
symmetric 4-bit q, one bf16 scale per output column and 128-wide group of
k).  The pages fix no packing; the oracle's reading is pinned here against
(a) hand-built bytes whose values are known, and (b) an independent numpy
unpacking multiplied with numpy's matmul (library)."""
import numpy as np
import pytest

import oracle
import workloads as W


def _bf16(a):
    return W.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_nibble_order_sign_and_group_scales_by_one_hot_inputs():
    K, N = 256, 2
    w = np.zeros((N, K // 2), np.uint8)
    w[0, 0] = 0x7F        # k=0: 0xF -> -1, k=1: 0x7 -> 7
    w[0, 63] = 0x80       # k=126: 0 , k=127: 0x8 -> -8
    w[0, 64] = 0x19       # k=128: 9 -> -7, k=129: 1
    w[1, 5] = 0xE2        # k=10: 2, k=11: 0xE -> -2
    scales = np.zeros((N, 2), np.uint16)
    scales[0] = _bf16([0.5, 4.0])
    scales[1] = _bf16([-3.0, 1.0])
    expect = {(0, 0): -0.5, (0, 1): 3.5, (0, 126): 0.0, (0, 127): -4.0, (0, 128): -28.0,
              (0, 129): 4.0, (1, 10): -6.0, (1, 11): 6.0, (1, 3): 0.0}
    for (n, k), val in expect.items():
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y = oracle.w4a16_gemm(_bf16(x), w, scales)
        assert y[0, n] == val, (n, k)


def _numpy_reference(x_bits, w, scale_bits):
    lo = (w & 0x0F).astype(np.int16)
    hi = (w >> 4).astype(np.int16)
    q = np.empty((w.shape[0], w.shape[1] * 2), np.int16)
    q[:, 0::2], q[:, 1::2] = lo, hi
    q = np.where(q >= 8, q - 16, q).astype(np.float64)
    s = W.bf16_bits_to_f32(scale_bits).astype(np.float64)
    wt = q * np.repeat(s, 128, axis=1)
    return W.bf16_bits_to_f32(x_bits).astype(np.float64) @ wt.T


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (3, 40, 512), (16, 64, 1024), (17, 24, 384)])
def test_matches_numpy_unpack_and_matmul(M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K)
    x = _bf16(rng.standard_normal((M, K)))
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = _bf16(rng.uniform(-0.05, 0.05, size=(N, K // 128)))
    got = oracle.w4a16_gemm(x, w, s)
    ref = _numpy_reference(x, w, s)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_all_256_bytes_in_both_nibble_positions():
    """Every byte value: y for x = ones over a 2-wide window equals q_lo + q_hi."""
    K = 512
    w = np.zeros((256, K // 2), np.uint8)
    w[:, 0] = np.arange(256, dtype=np.uint8)
    s = np.tile(_bf16([1.0, 1.0, 1.0, 1.0]), (256, 1))
    x = np.zeros((2, K), np.float32)
    x[0, 0] = 1.0                # low nibble
    x[1, 1] = 1.0                # high nibble
    y = oracle.w4a16_gemm(_bf16(x), w, s)
    b = np.arange(256)
    signed = lambda v: np.where(v >= 8, v - 16, v)
    assert np.array_equal(y[0], signed(b & 15)) and np.array_equal(y[1], signed(b >> 4))
