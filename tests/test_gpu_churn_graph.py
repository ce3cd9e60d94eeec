"""The churn step captured once as a CUDA graph and replayed gives, bit for
bit, the abort flags, cache codes and attention outputs of the same step
launched eagerly (appends are idempotent: the same rows go to the same
slots)."""
import numpy as np
import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq
from kvq_churn import ChurnDevice, ChurnGraphStep, ChurnState

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused_append", [False, True])
def test_graph_replay_matches_eager_launches(fused_append):
    kvq.kvq_device_error(clear=True)
    st = ChurnState(seed=3, batch=16, lo=300, hi=3000, steps=4)
    dev = ChurnDevice(st, layers=3, log_layers=())
    gs = ChurnGraphStep(dev, fused_append=fused_append)
    gs.load()
    gs.capture()
    flagged = 0
    for _ in range(4):
        _, _, _, stale, _ = gs.load()
        gs.launch()
        torch.cuda.synchronize()
        eager_out = [o.clone() for o in gs.out]
        eager_abort = dev.abort.clone()
        eager_k = [k.clone() for k in dev.k]
        for o in gs.out:
            o.fill_(float("nan"))
        dev.abort.fill_(7)
        gs.replay()
        torch.cuda.synchronize()
        assert torch.equal(dev.abort, eager_abort)
        assert set(np.nonzero(dev.abort.cpu().numpy())[0].tolist()) == stale
        for a, b in zip(gs.out, eager_out):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        for a, b in zip(dev.k, eager_k):
            assert torch.equal(a, b)
        flagged += len(stale)
        st.advance(stale)
    assert flagged > 0
    assert kvq.kvq_device_error() == 0


def test_fused_append_churn_step_equals_separate_launches():
    """tag check + per-layer kvq_decode_attn_append gives the flags, caches and
    outputs of tag check + per-layer kvq_append and kvq_decode_attn."""
    kvq.kvq_device_error(clear=True)
    states = [ChurnState(seed=5, batch=16, lo=300, hi=3000, steps=3) for _ in range(2)]
    devs = [ChurnDevice(s, layers=2, log_layers=()) for s in states]
    steps = [ChurnGraphStep(d, fused_append=f) for d, f in zip(devs, (False, True))]
    for _ in range(3):
        stale = [g.load()[3] for g in steps]
        assert stale[0] == stale[1]
        for g in steps:
            g.launch()
        torch.cuda.synchronize()
        assert torch.equal(devs[0].abort, devs[1].abort)
        for l in range(2):
            assert torch.equal(devs[0].k[l], devs[1].k[l]) and torch.equal(devs[0].v[l], devs[1].v[l])
            assert torch.equal(steps[0].out[l].view(torch.int16), steps[1].out[l].view(torch.int16))
        for s, st in zip(stale, states):
            st.advance(s)
    assert kvq.kvq_device_error() == 0
