"""Pins for the oracle's host tier (CPU only).

The SGLang blog (Sec. 6.1, HiCache) describes GPU memory as the first tier of the KV cache and
host memory as the second: KV that no longer fits on the GPU is kept in host memory and reused
from there instead of being recomputed. These tests check the oracle's tier against:
  * a hand-worked scenario (spill of the least recently used leaf, load back on a match, drop of
    the least recently used host leaf when the host tier is full), with the exact copies;
  * the content invariant, on random request streams: simulated device and host memories
    updated only by the copies the tree hands out (spills before loads) and by the computed
    tokens' own KV always hold, in every slot of every node, the KV of exactly that node's token
    prefix -- so reloaded KV equals recomputed KV (paper digest App. A.1: KV depends only on the
    prefix);
  * reuse: with a host tier large enough, the computed-token count equals that of a device pool
    so large that nothing is ever evicted.
"""
import random

import numpy as np
import pytest

import oracle


def _seq(*t):
    return np.array(t, dtype=np.int32)


def test_host_tier_hand_scenario():
    sim = oracle.CacheSim(6, host_slots=4)
    sim.cache([_seq(1, 2, 3)])                 # A: device slots 0 1 2
    sim.cache([_seq(4, 5, 6)])                 # B: device slots 3 4 5; the pool is empty
    assert sim.pool.available() == 0
    # [7 8] needs 2 slots: the least recently used leaf A moves to host slots 0 1 2, its device
    # slots go to the pool tail, [7 8] takes device slots 0 1
    res = sim.extend_prepare([_seq(7, 8)], match_all=True)
    sd, sh, lh, ld = res.copies
    assert (sd.tolist(), sh.tolist(), lh.tolist(), ld.tolist()) == ([0, 1, 2], [0, 1, 2], [], [])
    assert res.rows[0].tolist() == [0, 1]
    sim.extend_finish([_seq(7, 8)], res)
    st = sim.tree.stats()
    assert (st["host_tokens"], st["spilled_tokens"], st["cached_tokens"]) == (3, 3, 5)
    assert sim.tree.match_tiered(_seq(1, 2, 3))[:2] == (0, 3)
    # [1 2 3 9] matches A in the host tier (3 tokens to load back) and computes [9]: 4 device
    # slots, 1 free. Eviction takes B, the least recently used device leaf (3 tokens); the host
    # tier has 1 free slot and no leaf it may drop (A is locked by the match), so B is freed.
    # A loads into the pool's next slots 2 3 4, [9] takes 5.
    res = sim.extend_prepare([_seq(1, 2, 3, 9)])
    assert res.host_len == [3] and res.prefix_len == [3]
    sd, sh, lh, ld = res.copies
    assert (sd.tolist(), sh.tolist(), lh.tolist(), ld.tolist()) == ([], [], [0, 1, 2], [2, 3, 4])
    assert res.rows[0].tolist() == [2, 3, 4, 5]
    st = sim.tree.stats()
    assert (st["dropped_tokens"], st["loaded_tokens"], st["host_tokens"]) == (3, 3, 0)
    sim.extend_finish([_seq(1, 2, 3, 9)], res)
    n, slots, _ = sim.tree.match(_seq(1, 2, 3, 9))
    assert n == 4 and slots.tolist() == [2, 3, 4, 5]
    assert sim.host_pool.available() == 4      # the loaded host slots came back at the drain
    assert sim.tree.match(_seq(7, 8))[0] == 2  # [7 8] was never touched


def test_host_tier_drops_least_recently_used_host_leaf():
    sim = oracle.CacheSim(4, host_slots=4)
    sim.cache([_seq(1, 2)])                    # A, oldest
    sim.cache([_seq(3, 4)])                    # B
    res, _ = sim.cache([_seq(5, 6)])           # A spills to host slots 0 1
    assert res.copies[1].tolist() == [0, 1]
    res, _ = sim.cache([_seq(7, 8)])           # B spills to host slots 2 3: the host is full
    assert res.copies[1].tolist() == [2, 3]
    # [9 9]: the next device victim [5 6] needs 2 host slots; the older host leaf A is dropped
    # and [5 6] takes its host slots
    res, _ = sim.cache([_seq(9, 9)])
    assert res.copies[1].tolist() == [0, 1]
    assert sim.tree.match_tiered(_seq(1, 2))[:2] == (0, 0)     # gone from both tiers
    assert sim.tree.match_tiered(_seq(3, 4))[:2] == (0, 2)     # still in the host tier
    assert sim.tree.match_tiered(_seq(5, 6))[:2] == (0, 2)
    assert sim.tree.stats()["dropped_tokens"] == 2


def _check_contents(sim, dev_mem, host_mem):
    """Every slot of every node holds the KV (here: the token prefix) of exactly its token."""
    nodes = sim.tree.nodes()
    tiers = dict(zip(sim.tree.tiers()[0::2].tolist(), sim.tree.tiers()[1::2].tolist()))
    path = {0: ()}
    for n in nodes:                            # dump order: parents before children
        p = path[n["parent"]]
        mem = host_mem if tiers[n["id"]] else dev_mem
        for t, s in zip(n["key"].tolist(), n["slots"].tolist()):
            p = p + (t,)
            assert mem.get(s) == p, (n["id"], s)
        path[n["id"]] = p


@pytest.mark.parametrize("seed", range(8))
def test_host_tier_keeps_every_node_s_kv_exact(seed):
    rng = random.Random(300 + seed)
    sim = oracle.CacheSim(rng.choice([60, 90]), host_slots=rng.choice([30, 80, 200]))
    dev_mem, host_mem = {}, {}
    progs = [[rng.randrange(4) for _ in range(rng.randint(3, 20))] for _ in range(6)]
    moved = 0
    for step in range(60):
        batch = []
        for _ in range(rng.randint(1, 3)):
            base = rng.choice(progs)[:rng.randint(1, 20)]
            batch.append(_seq(*(base + [rng.randrange(4) for _ in range(rng.randint(1, 6))])))
        need = sum(len(s) for s in batch)
        if need > sim.pool.num_slots // 2:
            continue
        try:
            res = sim.extend_prepare(batch)
        except oracle.OutOfSlots:
            pytest.fail("a batch of at most half the pool must always fit")
        sd, sh, lh, ld = res.copies
        moved += len(sd) + len(lh)
        for d, h in zip(sd, sh):               # spills first ...
            host_mem[int(h)] = dev_mem.get(int(d))
        for h, d in zip(lh, ld):               # ... then loads
            dev_mem[int(d)] = host_mem.get(int(h))
        for s, p, row in zip(batch, res.prefix_len, res.rows):
            for i in range(p, len(s)):         # the computed tokens' own KV
                dev_mem[int(row[i])] = tuple(s[:i + 1].tolist())
            for i in range(p):                 # reused KV is the prefix's own
                assert dev_mem.get(int(row[i])) == tuple(s[:i + 1].tolist())
        sim.extend_finish(batch, res)
        _check_contents(sim, dev_mem, host_mem)
    assert moved > 0


@pytest.mark.parametrize("seed", range(4))
def test_host_tier_reuses_like_an_unbounded_pool(seed):
    rng = random.Random(700 + seed)
    progs = [[100 * p + rng.randrange(50) for _ in range(30)] for p in range(5)]
    seqs = [_seq(*(rng.choice(progs) + [rng.randrange(1000, 2000)])) for _ in range(40)]

    def computed(sim):
        c = 0
        for s in seqs:
            res = sim.extend_prepare([s])
            c += len(s) - res.prefix_len[0]
            sim.extend_finish([s], res)
        return c

    big = computed(oracle.CacheSim(10_000))
    small = computed(oracle.CacheSim(64))
    tiered = oracle.CacheSim(64, host_slots=10_000)
    assert computed(tiered) == big < small
    assert tiered.tree.stats()["loaded_tokens"] > 0
