"""INT4 weight-only product on the GPU through the C ABI, against the fp64
oracle fed the same bytes: every output for small shapes (all split counts
that apply, bf16 and fp32 output, batches that are not a multiple of 16),
sampled columns for a large one."""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
import workloads as W
from gpu_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(M, N, K, seed, scale=0.02):
    rng = np.random.default_rng(seed)
    x = W.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    s = W.f32_to_bf16_bits(rng.uniform(-scale, scale, size=(N, K // 128)).astype(np.float32))
    return x, w, s


def _dev(x, w, s):
    return (torch.from_numpy(x.view(np.int16)).to(DEV).view(torch.bfloat16),
            torch.from_numpy(w).to(DEV),
            torch.from_numpy(s.view(np.int16)).to(DEV).view(torch.bfloat16))


@pytest.mark.parametrize("M,N,K", [(1, 64, 256), (3, 128, 512), (8, 192, 1024), (16, 256, 2048),
                                   (17, 64, 768), (40, 128, 256)])
def test_matches_oracle(M, N, K):
    kvq.kvq_device_error(clear=True)
    x, w, s = _case(M, N, K, M * 7 + N + K)
    ref = oracle.w4a16_gemm(x, w, s)
    xd, wd, sd = _dev(x, w, s)
    splits = [0] + [p for p in range(1, 9) if K % (p * 256) == 0]
    for ns in splits:
        for fp32 in (False, True):
            y = torch.empty((M, N), dtype=torch.float32 if fp32 else torch.bfloat16, device=DEV)
            kvq.kvq_w4a16_gemm(xd, wd, sd, y, ns)
            torch.cuda.synchronize()
            assert_close(y.float().cpu().numpy().astype(np.float64), ref, "fp32" if fp32 else "bf16",
                         f"w4a16 M{M} N{N} K{K} splits{ns}")
    assert kvq.kvq_device_error() == 0


def test_extreme_nibbles_and_scales():
    """All-(-8) and all-7 weights with one-hot-free inputs of mixed sign."""
    M, N, K = 4, 64, 512
    x, _, s = _case(M, N, K, 3, scale=1.0)
    w = np.full((N, K // 2), 0x88, np.uint8)        # q = -8 everywhere
    w[N // 2:] = 0x77                                # q = 7
    ref = oracle.w4a16_gemm(x, w, s)
    xd, wd, sd = _dev(x, w, s)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    kvq.kvq_w4a16_gemm(xd, wd, sd, y)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy().astype(np.float64), ref, "fp32", "extreme nibbles")


def test_large_shape_sampled_columns():
    M, N, K = 16, 12288, 5120
    x, w, s = _case(M, N, K, 11)
    xd, wd, sd = _dev(x, w, s)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    kvq.kvq_w4a16_gemm(xd, wd, sd, y)
    torch.cuda.synchronize()
    cols = np.random.default_rng(1).choice(N, size=96, replace=False)
    ref = oracle.w4a16_gemm(x, w[cols], s[cols])
    assert_close(y.cpu().numpy().astype(np.float64)[:, cols], ref, "fp32", "w4a16 large")
    assert kvq.kvq_device_error() == 0


@pytest.mark.parametrize("M", [1, 4, 16])
def test_bench_shape_sampled_columns(M):
    """The shape and launch bench.py times (K 8,192, N 24,576, automatic
    splits, bf16 out), checked on sampled columns."""
    N, K = 24576, 8192
    x, w, s = _case(M, N, K, 100 + M)
    xd, wd, sd = _dev(x, w, s)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    kvq.kvq_w4a16_gemm(xd, wd, sd, y)
    torch.cuda.synchronize()
    cols = np.random.default_rng(M).choice(N, size=64, replace=False)
    cols = np.concatenate([cols, [0, 63, N - 64, N - 1]])
    ref = oracle.w4a16_gemm(x, w[cols], s[cols])
    assert_close(y.float().cpu().numpy().astype(np.float64)[:, cols], ref, "bf16", f"w4a16 bench shape M{M}")
    assert kvq.kvq_device_error() == 0


def test_longest_k_eight_split_cluster():
    """K = 65,536, the longest K: eight splits of 8,192 k, one cluster of 8."""
    M, N, K = 2, 128, 65536
    assert kvq.kvq_w4a16_plan(M, N, K) == 8
    x, w, s = _case(M, N, K, 21)
    ref = oracle.w4a16_gemm(x, w, s)
    xd, wd, sd = _dev(x, w, s)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    kvq.kvq_w4a16_gemm(xd, wd, sd, y)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy().astype(np.float64), ref, "fp32", "w4a16 K 65536")
    assert kvq.kvq_device_error() == 0


def test_empty_batch_writes_nothing():
    N, K = 64, 256
    _, w, s = _case(1, N, K, 5)
    _, wd, sd = _dev(np.zeros((1, K), np.uint16), w, s)
    x = torch.empty((0, K), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((0, N), dtype=torch.float32, device=DEV)
    kvq.kvq_w4a16_gemm(x, wd, sd, y)
    torch.cuda.synchronize()
