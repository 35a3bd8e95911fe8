"""Failure paths on the host, driven by the pool's injected allocation failure
(rc_pool_inject_alloc_failure): the failing call changes nothing, and a plan that fails after its
match leaves no lock behind, so the same request can be planned again. CPU only."""
import numpy as np
import pytest

import prefix_cached_paged_gb300 as rc
from prefix_cached_paged_gb300 import runtime
import synth


def test_injected_alloc_failure_changes_nothing_and_fires_once():
    order = synth.permutation(7, 12)
    p, ref = rc.Pool(12, order), rc.Pool(12, order)
    p.inject_alloc_failure(1)
    assert p.alloc(3).tolist() == ref.alloc(3).tolist()      # one more success first
    with pytest.raises(rc.RcError) as e:
        p.alloc(2)
    assert e.value.code == rc.RC_ERR_OOM and "injected" in str(e.value)
    assert p.available() == ref.available() == 9              # nothing taken
    assert p.alloc(2).tolist() == ref.alloc(2).tolist()      # disarmed; free-list order intact
    p.inject_alloc_failure(0)
    p.inject_alloc_failure(-1)                                 # disarm before it fires
    assert p.alloc(1).tolist() == ref.alloc(1).tolist()
    with pytest.raises(rc.RcError) as e:
        p.inject_alloc_failure(-2)
    assert e.value.code == rc.RC_ERR_INVALID
    # a real shortage is not one of the successful calls the injection counts down
    p.inject_alloc_failure(1)
    with pytest.raises(rc.RcError) as e:
        p.alloc(100)
    assert "injected" not in str(e.value)
    assert p.alloc(1).tolist() == ref.alloc(1).tolist()
    with pytest.raises(rc.RcError) as e:
        p.alloc(1)
    assert "injected" in str(e.value)


def _cache(hc, seqs):
    for s in seqs:
        plan = hc.plan([s], match_all=True)
        hc.finish(plan)


@pytest.mark.parametrize("evict", [False, True])
def test_failed_plan_releases_its_locks(evict):
    """A batch matches cached prefixes (locking them), may evict, then its allocation fails: the
    locks are released, the evictions stand, and planning the batch again succeeds with the same
    matches."""
    pre = synth.tokens(11, 1, 300)
    seqs = [np.concatenate([pre, synth.tokens(11, 10 + i, 40)]).astype(np.int32)
            for i in range(3)]
    others = [synth.tokens(11, 50 + i, 200) for i in range(4)]
    num_slots = 300 + 4 * 200 + (120 if not evict else 60)
    hc = runtime.HostCache(num_slots, 512)
    _cache(hc, [pre] + others)
    before = hc.tree.stats()
    assert before["protected_tokens"] == 0
    hc.pool.inject_alloc_failure(0)
    with pytest.raises(rc.RcError) as e:
        hc.plan(seqs)
    assert e.value.code == rc.RC_ERR_OOM
    after = hc.tree.stats()
    assert after["protected_tokens"] == 0                     # no lock left behind
    if evict:
        # 120 new tokens, 60 free: unlocked leaves were evicted before the allocation failed
        assert after["evicted_tokens"] > before["evicted_tokens"]
        assert after["cached_tokens"] < before["cached_tokens"]
        assert hc.pool.available() >= 120
    else:
        assert after["cached_tokens"] == before["cached_tokens"]
        assert hc.pool.available() == 120
    plan = hc.plan(seqs)                                      # the retry succeeds
    assert plan.prefix_len.tolist() == [300, 300, 300]
    assert hc.tree.stats()["protected_tokens"] > 0            # now locked by the running batch
    hc.finish(plan)
    assert hc.tree.stats()["protected_tokens"] == 0
