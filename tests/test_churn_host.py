"""Host bookkeeping of the churn workload (CPU): the allocator keeps the live
requests' pages distinct, bumps a page's tag whenever it changes owner, and
the seeded stale set is exactly what the oracle's tag check flags."""
import math

import numpy as np

import oracle
from kvq_churn import ChurnState


def test_churn_bookkeeping_100_steps():
    s = ChurnState(seed=0)
    assert s.num_pages == math.ceil(1.2 * sum(math.ceil((r.length - 1 + s.steps) / s.ps)
                                              for r in s.slots))
    owner_tag = {}
    flagged_total = 0
    for step in range(s.steps):
        bt, exp, seq, stale = s.tables()
        n_used = np.array([math.ceil(int(L) / s.ps) for L in seq])
        mask = np.arange(bt.shape[1])[None, :] < n_used[:, None]
        pages = bt[mask]
        assert len(pages) == len(set(pages.tolist()))               # no page shared
        assert np.all((pages >= 0) & (pages < s.num_pages))
        n_stale = int(np.sum((exp != s.pool.tags[np.maximum(bt, 0)]) & mask))
        assert n_stale == int(round(0.005 * mask.sum()))
        flags = oracle.tag_check(bt, exp, seq, s.pool.tags, page_size=s.ps)
        assert set(np.nonzero(flags)[0].tolist()) == stale
        assert 0 < len(stale) < s.batch // 4                        # most requests stay live
        flagged_total += len(stale)
        for r in s.slots:                                           # a new owner sees a new tag
            for p, t in zip(r.pages, r.expected):
                if p in owner_tag and owner_tag[p][0] != r.rid:
                    assert t != owner_tag[p][1]
                owner_tag[p] = (r.rid, t)
        s.advance(stale)
        assert all(r is not None for r in s.slots)
    assert flagged_total > 0
