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


def test_graph_replay_matches_eager_launches():
    kvq.kvq_device_error(clear=True)
    st = ChurnState(seed=3, batch=16, lo=300, hi=3000, steps=4)
    dev = ChurnDevice(st, layers=3, log_layers=())
    gs = ChurnGraphStep(dev)
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
