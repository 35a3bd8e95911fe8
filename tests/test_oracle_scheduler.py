"""Pins for the oracle's cache-aware scheduler (CPU only).

The paper digest's Sec. 3 ("cache-aware scheduling") and App. A.2/A.3 fix:
  * the order: waiting requests sorted by their matched prefix length, longest first;
  * Theorem 3.1: for a batch of requests and a cache at least as large as the longest request,
    running the requests in the depth-first order of the radix tree built from them computes
    every edge of that tree exactly once, so C = the tree's total edge length, the minimum any
    order can reach; longest-shared-prefix-first is that order;
  * the hit rate: 1 - C / (sum of the requests' prefill tokens).
These tests check the oracle against a hand-worked admission example and, on tiny random
request sets, against brute force over every order.
"""
import itertools
import random

import numpy as np
import pytest

import oracle


def _seq(*t):
    return np.array(t, dtype=np.int32)


def test_lspf_hand_example():
    # cached: [1 2 3 4 5] and [1 2 9] -> 6 slots used of 10, every node unreferenced
    sim = oracle.CacheSim(10)
    sim.cache([_seq(1, 2, 3, 4, 5), _seq(1, 2, 9)])
    assert sim.pool.available() == 4
    waiting = [_seq(7, 7, 7), _seq(1, 2, 3, 4, 8), _seq(1, 2, 9, 9), _seq(1, 2, 6)]
    order, match, adm = oracle.schedule_batch(sim.tree, waiting)
    assert match == [0, 4, 3, 2]
    assert order == [1, 2, 3, 0]
    # room 4 free + 6 evictable = 10: [1 2 3 4 8] computes 1 and locks 4 cached tokens (5),
    # [1 2 9 9] computes 1 and locks 9 (7), [1 2 6] computes 1 (8), [7 7 7] computes 3 (11 > 10)
    assert adm == 3
    assert oracle.schedule_batch(sim.tree, waiting, max_new_tokens=2)[2] == 2
    assert oracle.schedule_batch(sim.tree, waiting, max_batch=1)[2] == 1
    assert oracle.schedule_batch(sim.tree, waiting, reserve=3)[2] == 2
    assert oracle.schedule_batch(sim.tree, waiting, max_batch=0)[2] == 0
    # a locked cached path is not room: with [5 5 5] cached too (1 free + 9 evictable = 10)
    # the same three fit; locked, its 3 tokens leave the room (7) and only two fit
    sim3 = oracle.CacheSim(10)
    for s in (_seq(1, 2, 3, 4, 5), _seq(1, 2, 9), _seq(5, 5, 5)):
        sim3.cache([s])
    assert sim3.pool.available() == 1
    assert oracle.schedule_batch(sim3.tree, waiting)[2] == 3
    _, _, node = sim3.tree.match(_seq(5, 5, 5))
    sim3.tree.lock(node)
    assert oracle.schedule_batch(sim3.tree, waiting)[2] == 2
    # a lock on the batch's own path costs nothing more: [1 2 9] locked leaves room 7, and the
    # admitted requests then lock only [3 4] anew (1 + 2, 1, 1 -> 5; [7 7 7] would make 8)
    _, _, node = sim.tree.match(_seq(1, 2, 9))
    sim.tree.lock(node)
    assert oracle.schedule_batch(sim.tree, waiting)[2] == 3
    assert oracle.schedule_batch(sim.tree, waiting, reserve=3)[2] == 2
    sim.tree.unlock(node)
    # the admission is exact: the admitted batch fits, one more request does not
    batch = [waiting[w] for w in order[:adm]]
    res = sim.extend_prepare(batch, match_all=True)
    assert res.prefix_len == [4, 3, 2]
    sim.extend_finish(batch, res)
    sim2 = oracle.CacheSim(10)
    sim2.cache([_seq(1, 2, 3, 4, 5), _seq(1, 2, 9)])
    with pytest.raises(oracle.OutOfSlots):
        sim2.extend_prepare([waiting[w] for w in order[:adm + 1]], match_all=True)


def _requests(rng, n):
    """n distinct requests over a 3-token alphabet, each ending in its own terminal token, so
    that none is a prefix of another."""
    out = []
    for i in range(n):
        body = [rng.randrange(3) for _ in range(rng.randint(0, 6))]
        out.append(np.array(body + [100 + i], dtype=np.int32))
    return out


def _tree_edge_total(reqs):
    """Total edge length of the radix tree of the requests = the number of distinct non-empty
    prefixes."""
    return len({tuple(r[:k].tolist()) for r in reqs for k in range(1, len(r) + 1)})


def _dfs_order(reqs, rng=None):
    """A depth-first order of the requests' trie (children in token order, or shuffled)."""
    def visit(prefix, idx):
        here = [i for i in idx if len(reqs[i]) == len(prefix)]
        kids = {}
        for i in idx:
            if len(reqs[i]) > len(prefix):
                kids.setdefault(int(reqs[i][len(prefix)]), []).append(i)
        keys = sorted(kids)
        if rng is not None:
            rng.shuffle(keys)
        out = list(here)
        for k in keys:
            out += visit(prefix + (k,), kids[k])
        return out
    return visit((), list(range(len(reqs))))


def _run(reqs, order, capacity):
    """One request per batch through the oracle's loop; returns tokens computed (C)."""
    sim = oracle.CacheSim(capacity)
    computed = 0
    for i in order:
        res = sim.extend_prepare([reqs[i]])
        computed += len(reqs[i]) - res.prefix_len[0]
        sim.extend_finish([reqs[i]], res)
    return computed


def _run_lspf(reqs, capacity):
    """One request per batch, each picked by the oracle's scheduler from all that still wait."""
    sim = oracle.CacheSim(capacity)
    waiting = list(range(len(reqs)))
    computed = 0
    while waiting:
        seqs = [reqs[i] for i in waiting]
        order, match, adm = oracle.schedule_batch(sim.tree, seqs,
                                                 match_lens=[len(s) - 1 for s in seqs],
                                                 max_batch=1)
        assert adm == 1
        i = waiting.pop(order[0])
        res = sim.extend_prepare([reqs[i]])
        assert res.prefix_len[0] == match[order[0]]
        computed += len(reqs[i]) - res.prefix_len[0]
        sim.extend_finish([reqs[i]], res)
    return computed


@pytest.mark.parametrize("seed", range(6))
def test_theorem_3_1_dfs_order_is_optimal(seed):
    rng = random.Random(seed)
    beaten = 0
    for case in range(12):
        reqs = _requests(rng, rng.randint(2, 5))
        cap = max(len(r) for r in reqs)          # the cache holds the longest request
        c_min = _tree_edge_total(reqs)
        assert _run(reqs, _dfs_order(reqs), cap) == c_min
        assert _run(reqs, _dfs_order(reqs, rng), cap) == c_min
        costs = [_run(reqs, p, cap) for p in itertools.permutations(range(len(reqs)))]
        assert min(costs) == c_min                # no order computes less
        beaten += max(costs) > c_min
        assert _run_lspf(reqs, cap) == c_min      # longest shared prefix first reaches it
        total = sum(len(r) for r in reqs)
        hit = 1 - c_min / total                   # App. A.3 hit rate at the optimum
        assert 0 <= hit < 1
    assert beaten > 0    # the instances are not trivial: some orders recompute


def test_lspf_beats_fifo_on_interleaved_programs():
    """Programs with a long shared prefix arriving interleaved: FIFO with a cache that holds
    one program at a time recomputes every prefix, LSPF computes each once."""
    rng = random.Random(7)
    prefixes = [[p] + [rng.randrange(50) for _ in range(19)] for p in range(3)]
    reqs = []
    for q in range(4):
        for p in range(3):
            reqs.append(np.array(prefixes[p] + [1000 + 10 * q + p], dtype=np.int32))
    cap = 22
    c_min = _tree_edge_total(reqs)
    assert c_min == 3 * 20 + 12
    assert _run_lspf(reqs, cap) == c_min
    fifo = _run(reqs, range(len(reqs)), cap)
    assert fifo == sum(len(r) for r in reqs)      # nothing reused
    # the scheduler's first-come-first-served order is the queue order
    sim = oracle.CacheSim(cap)
    sim.cache([reqs[0]])
    order, match, adm = oracle.schedule_batch(sim.tree, reqs, fcfs=True, max_batch=4)
    assert order == list(range(len(reqs))) and match[0] == 21 and match[3] == 20 and adm == 1
