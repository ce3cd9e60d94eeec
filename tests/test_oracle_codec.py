"""Pins for the oracle's e4m3 codec (CPU only).

The pages fix only that the cache is stored as FP8 e4m3 instead of BF16
(blog post "Smaller, faster, safer", section on the quantised KV cache); the
bit format is the OCP E4M3 definition.  The oracle's codec is checked here
against things other than itself:
  * torch's float8_e4m3fn dtype (a library implementation of the format),
  * a brute-force nearest-code search over every finite code in exact fp64,
  * structural facts of the format (NaN codes, extremes, monotonicity).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f32

ALL_CODES = np.arange(256, dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_force_encode(y: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 code by exhaustive search; ties go to the code with
    an even mantissa; |y| beyond the largest code saturates; NaN -> S.1111.111."""
    y = np.asarray(y, dtype=np.float32)
    mags = torch_decode(np.arange(0x7F, dtype=np.uint8))      # 127 non-negative finite magnitudes
    with np.errstate(invalid="ignore"):
        a = np.abs(y.astype(np.float64))
    out = np.empty(y.shape, np.uint8)
    chunk = 1 << 16
    flat_a = a.ravel()
    flat_o = out.ravel()
    for s in range(0, flat_a.size, chunk):
        aa = flat_a[s:s + chunk]
        finite = np.isfinite(aa)
        dist = np.abs(np.where(finite, aa, 0.0)[:, None] - mags[None, :])
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        # among equally near codes prefer the even one (mantissa LSB 0)
        even = cand & ((np.arange(127) % 2) == 0)[None, :]
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        # beyond the largest finite code everything saturates (fp64 distances
        # to far-away inputs would otherwise round to spurious ties)
        pick = np.where(finite & (aa < mags[-1]), pick, 0x7E)
        flat_o[s:s + chunk] = pick.astype(np.uint8)
    sign = (np.signbit(y)).astype(np.uint8) << 7
    out = out | sign
    out[np.isnan(y)] = (0x7F | sign[np.isnan(y)])
    return out


def test_decode_matches_torch_float8_for_all_256_codes():
    ours = oracle.e4m3_decode(ALL_CODES)
    lib = torch_decode(ALL_CODES)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    fin = ~np.isnan(ours)
    assert np.array_equal(ours[fin], lib[fin])
    # signed zeros too
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(lib[fin]))


def test_decode_format_facts():
    v = oracle.e4m3_decode(ALL_CODES)
    nan_codes = set(np.nonzero(np.isnan(v))[0].tolist())
    assert nan_codes == {0x7F, 0xFF}
    assert np.isfinite(v).sum() == 254
    assert v[0x7E] == 448.0 and np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    assert v[0x01] == 2.0 ** -9            # smallest subnormal
    assert v[0x08] == 2.0 ** -6            # smallest normal
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)         # strictly increasing magnitudes
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])
    # eight codes per binade, constant spacing inside a binade
    for e in range(1, 16):
        b = pos[8 * e: 8 * e + 8] if e < 15 else pos[120:127]
        assert len(set(np.diff(b).tolist())) <= 1


def test_encode_all_bf16_matches_brute_force():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = bf16_bits_to_f32(bits)
    ours = oracle.e4m3_encode(y)
    ref = brute_force_encode(y)
    assert np.array_equal(ours, ref)


def test_encode_matches_torch_in_range():
    # torch's conversion is non-saturating (overflow -> NaN), so compare on
    # clamped inputs, which the saturating rule maps identically.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = bf16_bits_to_f32(bits)
    y = y[~np.isnan(y)]
    clamped = np.clip(y, -448.0, 448.0).astype(np.float32)
    lib = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(y), lib)


def test_encode_random_fp32_patterns_match_brute_force():
    rng = np.random.default_rng(1234)
    raw = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # bias toward the e4m3 range: also take exponents in [2^-12, 2^10]
    exps = rng.integers(127 - 12, 127 + 10, size=200_000).astype(np.uint32)
    near = (raw & np.uint32(0x807FFFFF)) | (exps << np.uint32(23))
    y = np.concatenate([raw.view(np.float32), near.view(np.float32)])
    assert np.array_equal(oracle.e4m3_encode(y), brute_force_encode(y))


def test_round_trip_and_ties():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    # exact midpoints between neighbouring positive codes go to the even code
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)   # exact in fp32
    got = oracle.e4m3_encode(mids)
    lo = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, expect)


def test_one_ulp_either_side_of_every_midpoint():
    """fp32 values one ulp above / below each midpoint between neighbouring
    positive codes round up / down (bits far below bf16 precision decide),
    with either sign."""
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    lo = np.arange(0x7E, dtype=np.uint8)
    above = np.nextafter(mids, np.float32(np.inf))
    below = np.nextafter(mids, np.float32(0))
    assert np.array_equal(oracle.e4m3_encode(above), lo + 1)
    assert np.array_equal(oracle.e4m3_encode(below), lo)
    assert np.array_equal(oracle.e4m3_encode(-above), (lo + 1) | 0x80)
    assert np.array_equal(oracle.e4m3_encode(-below), lo | 0x80)
    assert np.array_equal(oracle.e4m3_encode(above), brute_force_encode(above))


@pytest.mark.parametrize("y,code", [
    (448.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E),
    (-np.inf, 0xFE), (-500.0, 0xFE), (0.0, 0x00), (-0.0, 0x80),
    (2.0 ** -10, 0x00), (-(2.0 ** -10), 0x80), (3 * 2.0 ** -10, 0x02),
    (2.0 ** -10 * 1.0001, 0x01),
])
def test_encode_special_values(y, code):
    assert int(oracle.e4m3_encode(np.array([y], np.float32))[0]) == code


def test_encode_nan_keeps_sign():
    y = np.array([np.nan, -np.nan], np.float32)
    y[1] = -np.abs(y[1])
    out = oracle.e4m3_encode(y)
    assert out[0] == 0x7F and out[1] == 0xFF
