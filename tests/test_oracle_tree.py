"""Pins for the oracle's pool and radix tree (CPU only).

The oracle is checked against things the pages fix, not against itself:
  * a brute-force uncompressed per-token trie on tiny random inputs: match length = longest
    present prefix, slots follow their tokens, insert reports what was present, node boundaries
    sit only at sequence ends, branch points or match ends, the tree holds exactly the prefixes
    of what was inserted and not evicted;
  * a scripted scenario in the manner of the paper's Fig. 3 (nine time points: insert, reuse,
    split for a second chat, LRU eviction of the first chat's leaf, a new branch for few-shot
    queries, split for a batch of them, eviction of the second chat's nodes, eviction of the
    few-shot leaves for self-consistency samples) with hand-derived expected evictions;
  * the SGLang blog's worked count (Sec. 2.5): 3 requests of 2000 + 50 tokens compute 2150
    tokens instead of 6150.
"""
import json
import os
import random

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _present_paths(tree):
    """All token prefixes held by the oracle tree, with the slot of each prefix's last token."""
    nodes = tree.nodes()
    by_id = {n["id"]: n for n in nodes}
    path_of = {0: ()}
    slot_of = {}

    def path(nid):
        if nid in path_of:
            return path_of[nid]
        n = by_id[nid]
        p = path(n["parent"])
        for t, s in zip(n["key"].tolist(), n["slots"].tolist()):
            p = p + (t,)
            slot_of[p] = s
        path_of[nid] = p
        return p

    for n in nodes:
        path(n["id"])
    return slot_of, {n["id"]: path_of[n["id"]] for n in nodes}


class BruteTrie:
    def __init__(self):
        self.slot = {}          # prefix tuple -> slot of its last token

    def longest(self, toks):
        n = 0
        while n < len(toks) and tuple(toks[: n + 1]) in self.slot:
            n += 1
        return n

    def insert(self, toks, slots):
        ex = self.longest(toks)
        for i in range(ex, len(toks)):
            self.slot[tuple(toks[: i + 1])] = slots[i]
        return ex

    def branch_points(self):
        kids = {}
        for p in self.slot:
            kids.setdefault(p[:-1], set()).add(p[-1])
        return {p for p, k in kids.items() if len(k) >= 2 and p}


@pytest.mark.parametrize("seed", range(40))
def test_tree_matches_brute_force_trie(seed):
    rnd = random.Random(seed)
    alpha = rnd.choice([2, 3, 4])
    pool = oracle.Pool(400)
    tree = oracle.Tree(pool)
    brute = BruteTrie()
    seq_ends, match_ends = set(), set()
    ever = set()  # every reason a boundary was ever owed (nodes never merge back)
    locked = []
    for _ in range(120):
        op = rnd.random()
        toks = [rnd.randrange(alpha) for _ in range(rnd.randint(1, 12))]
        if op < 0.35:
            n, slots, node = tree.match(toks)
            assert n == brute.longest(toks)
            assert slots.tolist() == [brute.slot[tuple(toks[: i + 1])] for i in range(n)]
            if n:
                match_ends.add(tuple(toks[:n]))
                # a match that ends inside an edge splits it: its end is a node boundary
                assert tuple(toks[:n]) in set(_present_paths(tree)[1].values())
            if rnd.random() < 0.3:
                tree.lock(node)
                locked.append((node, tuple(toks[:n])))
        elif op < 0.75:
            slots = pool.alloc(len(toks))
            if slots is None:
                continue
            ex_b = brute.longest(toks)
            ex, node = tree.insert(toks, slots)
            assert ex == ex_b
            brute.insert(toks, slots.tolist())
            if ex > 0:
                pool.free(slots[:ex])    # the caller's duplicates of present tokens
            seq_ends.add(tuple(toks))
        elif op < 0.85 and locked:
            node, _ = locked.pop(rnd.randrange(len(locked)))
            tree.unlock(node)
        else:
            want = rnd.randint(1, 20)
            before = pool.available()
            ok, freed, ids = tree.evict(want)
            assert pool.available() == before + freed
            assert ok == (freed >= want)
            # remove from brute force whatever the tree no longer holds
            held, _ = _present_paths(tree)
            gone = [p for p in brute.slot if p not in held]
            for p in gone:
                del brute.slot[p]
            # a boundary that eviction removed is no longer owed
            seq_ends = {e for e in seq_ends if e in held}
            match_ends = {e for e in match_ends if e in held}
            # locked paths survive eviction
            for _, p in locked:
                for i in range(1, len(p) + 1):
                    assert p[:i] in held
        held, node_paths = _present_paths(tree)
        # the tree holds exactly the brute-force prefix set, slots included
        assert held == brute.slot
        # prefix-closed (an ancestor never disappears before its descendants)
        for p in held:
            assert p[:-1] in held or len(p) == 1
        # node boundaries: only at sequence ends, branch points or match ends; and every branch
        # point and every present sequence end is a boundary
        ends = set(node_paths.values())
        bps = brute.branch_points()
        ever |= seq_ends | match_ends | bps
        for e in ends:
            assert e in ever, e
        for b in bps:
            assert b in ends
        for s in seq_ends:
            if s in held:
                assert s in ends
        # no slot is in two places and slots + free list partition the pool
        slots_used = list(held.values())
        assert len(set(slots_used)) == len(slots_used)
        assert len(slots_used) + pool.available() == 400


def _serve(tree, pool, seq, evict_before_alloc=0):
    """One request through the loop: match all but the last token, lock, optional forced
    eviction (memory pressure), allocate the rest, insert, free duplicates, unlock."""
    n, slots, node = tree.match(seq[:-1])
    tree.lock(node)
    evicted = []
    if evict_before_alloc:
        ok, freed, evicted = tree.evict(evict_before_alloc)
        assert ok
    new = pool.alloc(len(seq) - n)
    ex, end = tree.insert(seq, np.concatenate([slots, new]))
    if ex > n:
        pool.free(new[: ex - n])
    tree.unlock(node)
    return n, evicted


def test_fig3_style_lru_scenario():
    pool = oracle.Pool(1000)
    tree = oracle.Tree(pool)
    SYS = [1, 2, 3, 4]
    chat1_t1 = SYS + [10, 11, 12, 13]
    chat1_t2 = chat1_t1 + [14, 15, 16, 17]
    chat2_t1 = SYS + [20, 21, 22, 23]
    chat2_t2 = chat2_t1 + [24, 25, 26, 27]
    EX = [40, 41, 42, 43, 44, 45]
    # (2) first chat turn: one edge from the root
    assert _serve(tree, pool, chat1_t1)[0] == 0
    keys = {tuple(n["key"].tolist()): n for n in tree.nodes()}
    assert list(keys) == [tuple(chat1_t1)]
    # (3) second turn reuses the whole first turn and appends a node
    assert _serve(tree, pool, chat1_t2)[0] == 8
    # (4) a second chat shares only the system prompt: the first edge splits after it
    n, _ = _serve(tree, pool, chat2_t1)
    assert n == 4
    nodes = tree.nodes()
    keys = {tuple(x["key"].tolist()): x for x in nodes}
    assert set(keys) == {tuple(SYS), (10, 11, 12, 13), (14, 15, 16, 17), (20, 21, 22, 23)}
    # the split-off upper part is new (id 3); the lower part kept the old id 1
    assert keys[tuple(SYS)]["id"] == 3 and keys[(10, 11, 12, 13)]["id"] == 1
    # (5) second chat continues under memory pressure: the first chat's newest turn is the LRU
    #     leaf and goes; the second chat's nodes are locked by the running request
    n, ev = _serve(tree, pool, chat2_t2, evict_before_alloc=4)
    assert n == 8
    assert ev == [2]  # node (14..17)
    # (6) an unrelated few-shot query opens a new branch at the root
    assert _serve(tree, pool, EX + [50, 51, 90])[0] == 0
    # (7) a batch of few-shot queries sharing the examples: the few-shot edge splits after EX
    seqs = [EX + [52, 53, 91], EX + [54, 55, 92]]
    res = []
    for s in seqs:
        res.append(tree.match(s[:-1]))
        tree.lock(res[-1][2])
    assert [r[0] for r in res] == [6, 6]
    for s, (n, slots, node) in zip(seqs, res):
        new = pool.alloc(len(s) - n)
        tree.insert(s, np.concatenate([slots, new]))
        tree.unlock(node)
    keys = {tuple(x["key"].tolist()): x for x in tree.nodes()}
    assert tuple(EX) in keys and (50, 51, 90) in keys
    # (8) a new message of the first chat: the second chat's nodes are least recently used and
    #     go leaf first (its second turn, then its first turn once that became a leaf)
    chat1_t3 = chat1_t1 + [18, 19]
    n, ev = _serve(tree, pool, chat1_t3, evict_before_alloc=8)
    assert n == 8
    ids = {tuple(x["key"].tolist()): x["id"] for x in nodes}
    assert ev == [5, 4]  # (24..27) then (20..23)
    keys = {tuple(x["key"].tolist()) for x in tree.nodes()}
    assert (20, 21, 22, 23) not in keys and (24, 25, 26, 27) not in keys
    # (9) self-consistency samples of a new few-shot question: the fork hint caches the shared
    #     question first; making room evicts the older few-shot query leaves, and the shared
    #     examples (locked by the running request) stay
    q = EX + [56, 57]
    n, slots, node = tree.match(q)
    tree.lock(node)
    ok, freed, ev = tree.evict(9)
    assert ok and freed == 9
    assert ev == [6, 8, 9]  # (50,51,90), (52,53,91), (54,55,92) in LRU order
    tree.unlock(node)
    keys = {tuple(x["key"].tolist()) for x in tree.nodes()}
    assert tuple(EX) in keys and tuple(SYS) in keys


def test_refcount_protects_older_leaf():
    pool = oracle.Pool(100)
    tree = oracle.Tree(pool)
    old = [1, 2, 3]
    new = [7, 8, 9]
    for s in (old, new):
        slots = pool.alloc(3)
        tree.insert(s, slots)
    n, _, node = tree.match(old)
    # touch `new` afterwards so that `old` is the least recently used again
    tree.match(new)
    tree.lock(node)
    ok, freed, ids = tree.evict(1)
    assert ok and freed == 3
    keys = {tuple(x["key"].tolist()) for x in tree.nodes()}
    assert keys == {tuple(old)}
    # nothing unreferenced is left: eviction reports the shortfall
    ok, freed, _ = tree.evict(1)
    assert not ok and freed == 0
    tree.unlock(node)
    with pytest.raises(KeyError):
        tree.unlock(node)  # reference count never goes negative


def test_pool_all_or_nothing_and_order():
    pool = oracle.Pool(5, order=[4, 2, 0, 1, 3])
    assert pool.alloc(2).tolist() == [4, 2]
    assert pool.alloc(4) is None and pool.available() == 3
    pool.free([9, 8])
    assert pool.alloc(5).tolist() == [0, 1, 3, 9, 8]


def test_worked_few_shot_count():
    g = json.load(open(os.path.join(GOLDEN, "worked_count.json")))
    rnd = np.random.default_rng(0)
    prefix = rnd.integers(0, 32000, g["shared_prefix_tokens"]).astype(np.int32)
    seqs = [np.concatenate([prefix, rnd.integers(0, 32000, g["query_tokens"]).astype(np.int32)])
            for _ in range(g["requests"])]
    computed = 0
    sim = oracle.CacheSim(10_000)
    for s in seqs:  # requests arrive one after another
        r = sim.extend_prepare([s])
        computed += len(s) - r.prefix_len[0]
        sim.extend_finish([s], r)
    assert computed == g["computed_with_radix_cache"]
    no_cache = sum(len(s) for s in seqs)
    assert no_cache == g["computed_without_cache"]
    assert round(100 * (1 - computed / no_cache)) == g["saving_percent"]


def test_tiny_extend_skips_192_of_320():
    from synth import workloads as W
    w = W.tiny_extend()
    sim = oracle.CacheSim(w.pool_slots, w.pool_order)
    skipped = total = 0
    for ph in w.phases:
        r = sim.extend_prepare(ph.seqs)
        skipped += sum(r.prefix_len)
        total += sum(len(s) for s in ph.seqs)
        sim.extend_finish(ph.seqs, r)
    assert (skipped, total) == (192, 320)


def test_duplicate_insert_in_one_batch_frees_the_later_copy():
    sim = oracle.CacheSim(50)
    a = np.array([5, 6, 7, 8, 9], dtype=np.int32)
    b = np.array([5, 6, 7, 8, 1], dtype=np.int32)
    r = sim.extend_prepare([a, b])
    assert r.prefix_len == [0, 0]  # no reuse inside one batch
    sim.extend_finish([a, b], r)
    assert r.existing == [0, 4] and r.freed_dups == 4
    # the tree keeps the first request's slots for the shared four tokens
    n, slots, _ = sim.tree.match(b)
    assert n == 5 and slots[:4].tolist() == r.rows[0][:4].tolist()
    assert sim.pool.available() == 50 - 6


def test_lock_protects_exactly_the_matched_prefix():
    """Reference counts protect what a running request uses (paper digest Sec. 3: only nodes
    with count 0 are freed). A match that ends inside an edge locks exactly the matched tokens:
    the rest of that edge is unreferenced and can go."""
    pool = oracle.Pool(100)
    tree = oracle.Tree(pool)
    seq = [3, 1, 4, 1, 5, 9, 2, 6]
    tree.insert(seq, pool.alloc(len(seq)))
    n, slots, node = tree.match([3, 1, 4, 7])
    assert n == 3
    tree.lock(node)
    ok, freed, _ = tree.evict(100)
    assert not ok and freed == 5
    held, _ = _present_paths(tree)
    assert set(held) == {(3,), (3, 1), (3, 1, 4)}
    tree.unlock(node)
    ok, freed, _ = tree.evict(3)
    assert ok and freed == 3 and pool.available() == 100


def _cache_one(sim, seq):
    r = sim.extend_prepare([seq], match_all=True)
    sim.extend_finish([seq], r)
    return r.rows[0].tolist()


def test_decode_prepare_locks_evicts_then_allocates():
    """Decode entry under memory pressure, expected slots worked out by hand (paper digest
    App. A.1: a decode step appends one token per request over its cached KV; Sec. 3 and
    Fig. 3: running requests hold references, eviction takes the least recently used
    unreferenced leaves, whole nodes, and freed slots go to the tail of the free list).
    Pool of 12 slots in identity order; A, B, C cached in that order (A oldest):
      A = [1 2 3 4] -> slots 0-3, B = [5 6 7] -> 4-6, C = [8 9 10 11] -> 7-10; free [11].
    Decoding A and C: both matched whole and locked (the matches make them newer than B); two
    new slots are needed, one is free, so eviction frees the shortfall: B, the LRU unreferenced
    leaf (3 tokens, slots 4 5 6 to the tail: free [11 4 5 6]); then the new tokens get 11 and 4
    in request order."""
    sim = oracle.CacheSim(12)
    A, B, C = [1, 2, 3, 4], [5, 6, 7], [8, 9, 10, 11]
    assert [_cache_one(sim, s) for s in (A, B, C)] == [[0, 1, 2, 3], [4, 5, 6], [7, 8, 9, 10]]
    r = sim.decode_prepare([A, C])
    assert r.prefix_len == [4, 4]
    assert [x.tolist() for x in r.rows] == [[0, 1, 2, 3], [7, 8, 9, 10]]
    assert (r.evict_request, r.evicted) == (1, 3)
    assert r.extra_slots.tolist() == [11, 4]
    assert sim.pool.available() == 2
    assert sim.pool.alloc(2).tolist() == [5, 6]   # the rest of B's slots, in token order
    keys = {tuple(n["key"].tolist()) for n in sim.tree.nodes()}
    assert keys == {tuple(A), tuple(C)}
    # the running contexts stay protected: nothing else is unreferenced
    ok, freed, _ = sim.tree.evict(1)
    assert not ok and freed == 0


def test_decode_prepare_cannot_evict_a_running_context():
    """Three decoding requests lock every cached node (A, B, C as above); three new slots are
    needed with one free, so there is nothing to evict: the step must fail rather than take a
    context that a running request reads (Sec. 3: only nodes with reference count 0 go)."""
    sim = oracle.CacheSim(12)
    for s in ([1, 2, 3, 4], [5, 6, 7], [8, 9, 10, 11]):
        _cache_one(sim, s)
    with pytest.raises(oracle.OutOfSlots):
        sim.decode_prepare([[1, 2, 3, 4], [8, 9, 10, 11], [5, 6, 7]])
    assert sim.pool.available() == 1
    assert len(sim.tree.nodes()) == 3


def test_mixed_step_allocates_extend_suffixes_before_decode_tokens():
    """A mixed step (extend batch plus `extra` decode tokens), expected slots by hand.
    Pool of 10 slots in identity order; X = [1 2 3 4 5] -> 0-4, Y = [6 7 8] -> 5-7 and
    Z = [20 21] -> 8 9 cached in that order; nothing is free. Extending X + [9 10] matches and
    locks X (5 tokens, the match makes X the newest) and needs 2 suffix slots + 2 decode slots:
    eviction frees the shortfall of 4 leaf by leaf in LRU order, Y (3) then Z (2), giving free
    [5 6 7 8 9]; the suffix takes 5 6 (request order first), the decode tokens 7 8."""
    sim = oracle.CacheSim(10)
    for s in ([1, 2, 3, 4, 5], [6, 7, 8], [20, 21]):
        _cache_one(sim, s)
    seq = [1, 2, 3, 4, 5, 9, 10]
    r = sim.extend_prepare([seq], extra=2)
    assert r.prefix_len == [5]
    assert (r.evict_request, r.evicted) == (4, 5)
    assert r.rows[0].tolist() == [0, 1, 2, 3, 4, 5, 6]
    assert r.extra_slots.tolist() == [7, 8]
    assert sim.pool.available() == 1
    # without pressure: two requests, suffixes in request order, then the decode slots
    sim = oracle.CacheSim(16)
    for s in ([1, 2, 3, 4, 5], [6, 7, 8]):
        _cache_one(sim, s)
    r = sim.extend_prepare([[1, 2, 3, 4, 5, 9, 10], [6, 7, 8, 11]], extra=2)
    assert r.prefix_len == [5, 3] and (r.evict_request, r.evicted) == (0, 0)
    assert [x.tolist() for x in r.rows] == [[0, 1, 2, 3, 4, 8, 9], [5, 6, 7, 10]]
    assert r.extra_slots.tolist() == [11, 12]
