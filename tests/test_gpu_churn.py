"""The churn workload with integrity tags on the GPU: 100 steps x 32 layers.

Every step: the abort flags of kvq_tag_check must equal the seeded stale set
and the oracle's flags (bit-exact); the e4m3 codes kvq_append wrote for every
live request's new token in the checked layers must equal the oracle's codes
for the same bf16 rows (bit-exact); aborted requests get zeros.  At steps 0,
50 and 99 the attention output of two live requests in layers 0 and 31 is
checked against the oracle run on page contents rebuilt from the seed and the
append log.
"""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
import oracle
from gpu_util import assert_close, out_to_np, to_np_bits
from kvq_churn import ChurnDevice, ChurnState

pytestmark = pytest.mark.gpu

LAYERS = 32
SAMPLED_STEPS = (0, 50, 99)
SAMPLED_LAYERS = (0, LAYERS - 1)
CODE_LAYERS = (0, 1, 17, LAYERS - 1)


def _oracle_codes(kn_bits, vn_bits, ks, vs, ps=16):
    """Codes the oracle's append writes for B rows (into a scratch cache)."""
    B, H, D = kn_bits.shape
    kc = np.zeros(((B + ps - 1) // ps, H, ps, D), np.uint8)
    vc = np.zeros_like(kc)
    slots = np.arange(B, dtype=np.int64)
    oracle.append(kc, vc, kn_bits, vn_bits, slots, ks, vs, page_size=ps)
    return kc[slots // ps, :, slots % ps, :], vc[slots // ps, :, slots % ps, :]


def test_churn_100_steps_32_layers():
    kvq.kvq_device_error(clear=True)
    st = ChurnState(seed=0)
    dev = ChurnDevice(st, layers=LAYERS, log_layers=SAMPLED_LAYERS)
    rng = np.random.default_rng(123)
    flagged = 0
    for step in range(st.steps):
        bt, exp, seq, stale, slots, abort, kept = dev.run_step(keep_layers=CODE_LAYERS)
        torch.cuda.synchronize()
        assert set(np.nonzero(abort)[0].tolist()) == stale, f"step {step}"
        assert np.array_equal(abort, oracle.tag_check(bt, exp, seq, st.pool.tags, page_size=st.ps))
        flagged += len(stale)

        live = np.nonzero((slots >= 0) & (abort == 0))[0]
        sl = torch.from_numpy(slots[live]).to(dev.device)
        pages, offs = sl // st.ps, sl % st.ps
        for layer, (out, q, kn, vn) in kept.items():
            ref_k, ref_v = _oracle_codes(to_np_bits(kn)[live], to_np_bits(vn)[live],
                                         dev.k_scale_host[layer], dev.v_scale_host[layer])
            assert np.array_equal(to_np_bits(dev.k[layer][pages, :, offs, :]), ref_k), \
                f"step {step} layer {layer} K codes"
            assert np.array_equal(to_np_bits(dev.v[layer][pages, :, offs, :]), ref_v), \
                f"step {step} layer {layer} V codes"
            assert np.all(to_np_bits(out)[abort.astype(bool)] == 0)        # aborted -> zeros

        if step in SAMPLED_STEPS:
            for r in rng.choice(live, size=2, replace=False):
                r = int(r)
                for layer in SAMPLED_LAYERS:
                    L = int(seq[r])
                    k, v = dev.request_bf16(layer, bt[r], L)
                    n_pages = -(-L // st.ps)
                    kc = np.zeros((n_pages, dev.hkv, st.ps, dev.D), np.uint8)
                    vc = np.zeros_like(kc)
                    oracle.append(kc, vc, k, v, np.arange(L, dtype=np.int64),
                                  dev.k_scale_host[layer], dev.v_scale_host[layer], page_size=st.ps)
                    q = to_np_bits(kept[layer][1])[r:r + 1]
                    ref = oracle.decode_attn(q, kc, vc, dev.k_scale_host[layer],
                                             dev.v_scale_host[layer],
                                             np.arange(n_pages, dtype=np.int32).reshape(1, -1),
                                             np.array([L], np.int32), dev.sigma)
                    got = out_to_np(kept[layer][0])[r:r + 1]
                    assert_close(got, ref, "bf16", f"churn step {step} layer {layer} request {r}")
        st.advance(stale)
    assert flagged > 0
    assert kvq.kvq_device_error() == 0
