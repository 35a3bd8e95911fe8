"""librc's host side against the oracle (CPU only): bit-exact slots, match lengths, evictions and
whole-tree dumps, plus the C-ABI exports."""
import os
import random
import re

import numpy as np
import pytest

import oracle
import prefix_cached_paged_gb300 as rc
from tests import planner_ref
from prefix_cached_paged_gb300 import runtime
from prefix_cached_paged_gb300._lib import SIGNATURES, lib
from synth import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "rc.h")).read()
    declared = set(re.findall(r"^\s*(?:[\w\*]+\s+)+\**(rc_\w+)\s*\(", header, re.M))
    assert declared, "no declarations parsed"
    L = lib()
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert declared == set(SIGNATURES), declared ^ set(SIGNATURES)


def test_pool_semantics():
    p = rc.Pool(5, [4, 2, 0, 1, 3])
    assert p.alloc(2).tolist() == [4, 2]
    with pytest.raises(rc.RcError) as e:
        p.alloc(4)
    assert e.value.code == rc.RC_ERR_OOM and p.available() == 3
    with pytest.raises(rc.RcError):
        p.free([4, 4])          # repeated
    with pytest.raises(rc.RcError):
        p.free([0])             # already free
    with pytest.raises(rc.RcError):
        p.free([7])             # out of range
    assert p.available() == 3
    p.free([2, 4])
    assert p.alloc(5).tolist() == [0, 1, 3, 2, 4]
    with pytest.raises(rc.RcError):
        rc.Pool(3, [0, 0, 1])


@pytest.mark.parametrize("seed", range(30))
def test_random_ops_match_oracle_bit_exact(seed):
    rnd = random.Random(1000 + seed)
    alpha = rnd.choice([2, 3, 5])
    N = 300
    order = np.array(rnd.sample(range(N), N), dtype=np.int32)
    op_, ot = oracle.Pool(N, order), None
    ot = oracle.Tree(op_)
    pp = rc.Pool(N, order)
    pt = rc.RadixTree(pp)
    locked = []  # (oracle id, product handle)
    for step in range(150):
        r = rnd.random()
        toks = [rnd.randrange(alpha) for _ in range(rnd.randint(0, 14))]
        if r < 0.35:
            n1, s1, id1 = ot.match(toks)
            n2, s2, h2 = pt.match_prefix(toks)
            assert (n1, s1.tolist()) == (n2, s2.tolist())
            if rnd.random() < 0.4:
                ot.lock(id1)
                pt.lock(h2)
                locked.append((id1, h2))
        elif r < 0.7:
            a1 = op_.alloc(len(toks))
            if a1 is None:
                with pytest.raises(rc.RcError):
                    pp.alloc(len(toks))
                continue
            a2 = pp.alloc(len(toks))
            assert a1.tolist() == a2.tolist()
            e1, _ = ot.insert(toks, a1)
            e2, _ = pt.insert(toks, a2)
            assert e1 == e2
            op_.free(a1[:e1])
            pp.free(a2[:e2])
        elif r < 0.8 and locked:
            i1, h2 = locked.pop(rnd.randrange(len(locked)))
            ot.unlock(i1)
            pt.unlock(h2)
        else:
            want = rnd.randint(0, 30)
            ok1, f1, _ = ot.evict(want)
            st, f2 = pt.evict_lru(want)
            assert f1 == f2 and ok1 == (st == rc.RC_OK)
        assert op_.available() == pp.available()
        np.testing.assert_array_equal(ot.dump(), pt.dump())
    s1, s2 = ot.stats(), pt.stats()
    for k in ("splits", "evicted_nodes", "evicted_tokens", "nodes", "cached_tokens",
              "protected_tokens"):
        assert s1[k] == s2[k], k
    # the free lists agree in order
    n = op_.available()
    assert op_.alloc(n).tolist() == pp.alloc(n).tolist()


def _waiting_list(rnd, cached, alpha):
    """Waiting sequences: extensions of cached sequences (cut at random points) and fresh ones."""
    out = []
    for _ in range(rnd.randint(0, 12)):
        if cached and rnd.random() < 0.7:
            base = rnd.choice(cached)
            base = base[:rnd.randint(0, len(base))]
        else:
            base = []
        out.append(base + [rnd.randrange(alpha) for _ in range(rnd.randint(0, 8))])
    return out


@pytest.mark.parametrize("seed", range(20))
def test_schedule_batch_matches_oracle_bit_exact(seed):
    """rc_schedule_batch against the oracle's scheduler on random tree states (locks, partial
    edges, a short pool), both policies: same order, matches and admitted count, and the tree
    unchanged."""
    rnd = random.Random(5000 + seed)
    alpha = rnd.choice([2, 3, 6])
    N = 200
    order = np.array(rnd.sample(range(N), N), dtype=np.int32)
    op_ = oracle.Pool(N, order)
    ot = oracle.Tree(op_)
    pp = rc.Pool(N, order)
    pt = rc.RadixTree(pp)
    locked, cached = [], []
    compared = admitted_some = 0
    for step in range(120):
        r = rnd.random()
        toks = [rnd.randrange(alpha) for _ in range(rnd.randint(1, 14))]
        if r < 0.25 and cached:
            toks = rnd.choice(cached)[:rnd.randint(0, 14)]
            _, _, id1 = ot.match(toks)
            _, _, h2 = pt.match_prefix(toks)
            if rnd.random() < 0.6:
                ot.lock(id1)
                pt.lock(h2)
                locked.append((id1, h2))
        elif r < 0.6:
            a1 = op_.alloc(len(toks))
            if a1 is None:
                continue
            a2 = pp.alloc(len(toks))
            e1, _ = ot.insert(toks, a1)
            e2, _ = pt.insert(toks, a2)
            op_.free(a1[:e1])
            pp.free(a2[:e2])
            cached.append(toks)
        elif r < 0.7 and locked:
            i1, h2 = locked.pop(rnd.randrange(len(locked)))
            ot.unlock(i1)
            pt.unlock(h2)
        elif r < 0.8:
            want = rnd.randint(0, 30)
            ot.evict(want)
            pt.evict_lru(want)
        else:
            waiting = _waiting_list(rnd, cached, alpha)
            mlen = None
            if waiting and rnd.random() < 0.5:
                mlen = [max(len(w) - 1, 0) for w in waiting]
            kw = dict(max_batch=rnd.choice([0, 1, 3, 1 << 30]),
                      max_new_tokens=rnd.choice([-1, 0, 5, 20]),
                      reserve=rnd.choice([0, 0, 10, 150]))
            fcfs = rnd.random() < 0.3
            o1, m1, a1 = oracle.schedule_batch(ot, waiting, mlen, fcfs, **kw)
            lens = np.array([len(w) for w in waiting], dtype=np.int64)
            indptr = np.zeros(len(waiting) + 1, dtype=np.int64)
            np.cumsum(lens, out=indptr[1:])
            flat = (np.concatenate([np.array(w, np.int32) for w in waiting]) if waiting
                    else np.zeros(0, np.int32))
            o2, m2, a2 = pt.schedule_batch(flat, indptr, mlen,
                                           rc.RC_SCHED_FCFS if fcfs else rc.RC_SCHED_LSPF,
                                           kw["max_batch"], kw["max_new_tokens"], kw["reserve"])
            assert (list(o1), list(m1), a1) == (o2.tolist(), m2.tolist(), a2)
            # the same sequences as ranges of one buffer, shuffled and with gaps between them
            r2 = random.Random(7919 * seed + compared)
            buf, starts = [], np.zeros(len(waiting), np.int64)
            for wi in r2.sample(range(len(waiting)), len(waiting)):
                buf += [r2.randrange(alpha) for _ in range(r2.randint(0, 3))]
                starts[wi] = len(buf)
                buf += list(waiting[wi])
            o3, m3, a3 = pt.schedule_batch_ranges(np.array(buf, np.int32), starts, lens, mlen,
                                                  rc.RC_SCHED_FCFS if fcfs else rc.RC_SCHED_LSPF,
                                                  kw["max_batch"], kw["max_new_tokens"],
                                                  kw["reserve"])
            assert (o3.tolist(), m3.tolist(), a3) == (o2.tolist(), m2.tolist(), a2)
            compared += 1
            admitted_some += a2 > 0
        np.testing.assert_array_equal(ot.dump(), pt.dump())
    assert compared >= 10 and admitted_some > 0


def test_schedule_admission_is_feasible_and_tight():
    """Planning the admitted batch through the engine's host path never runs out of slots;
    when admission stopped for room, adding the next request does."""
    rnd = random.Random(99)
    stops = 0
    for trial in range(40):
        N = rnd.choice([60, 120, 250])
        hc = runtime.HostCache(N, 64)
        hc2 = runtime.HostCache(N, 64)
        cached = []
        for _ in range(rnd.randint(1, 10)):
            s = [rnd.randrange(4) for _ in range(rnd.randint(2, 30))]
            for h in (hc, hc2):
                try:
                    h.finish(h.plan([s], match_all=True))
                except rc.RcError:
                    break
            else:
                cached.append(s)
        waiting = [w for w in _waiting_list(rnd, cached, 4) if w]
        if not waiting:
            continue
        lens = np.array([len(w) for w in waiting], dtype=np.int64)
        indptr = np.zeros(len(waiting) + 1, dtype=np.int64)
        np.cumsum(lens, out=indptr[1:])
        flat = np.concatenate([np.array(w, np.int32) for w in waiting])
        mlen = np.maximum(lens - 1, 0).astype(np.int32)
        policy = rc.RC_SCHED_FCFS if trial % 3 == 0 else rc.RC_SCHED_LSPF
        order, match, adm = hc.tree.schedule_batch(flat, indptr, mlen, policy)
        batch = [waiting[w] for w in order[:adm]]
        if batch:
            p = hc.plan(batch)
            assert p.prefix_len.tolist() == [match[w] for w in order[:adm]]
            hc.finish(p)
        if adm < len(waiting):
            stops += 1
            with pytest.raises(rc.RcError):
                hc2.plan([waiting[w] for w in order[:adm + 1]])
    assert stops > 0


def test_stale_handles_and_unlock_underflow():
    pool = rc.Pool(20)
    t = rc.RadixTree(pool)
    t.insert([1, 2, 3], pool.alloc(3))
    n, _, h = t.match_prefix([1, 2, 3])
    st, freed = t.evict_lru(3)
    assert st == rc.RC_OK and freed == 3
    with pytest.raises(rc.RcError) as e:
        t.lock(h)
    assert e.value.code == rc.RC_ERR_INVALID
    t.insert([4, 5], pool.alloc(2))
    _, _, h2 = t.match_prefix([4, 5])
    with pytest.raises(rc.RcError):
        t.unlock(h2)


def _run_phases_both(w, steps=None):
    """Run a workload's host steps through the product runtime and the oracle's loop; compare."""
    pc = runtime.HostCache(w.pool_slots, w.max_ctx, w.pool_order)
    oc = oracle.CacheSim(w.pool_slots, w.pool_order)
    for ph in w.phases:
        if ph.kind == "decode":
            ctx = [s[:-1] for s in ph.seqs]
            pp = pc.plan(ctx, extra=len(ctx), match_all=True)
            op = oc.decode_prepare(ctx)
            assert pp.prefix_len.tolist() == op.prefix_len
            assert pp.extra.tolist() == op.extra_slots.tolist()
            continue
        match_all = ph.kind == "cache"
        # a cache phase inserts its sequences one at a time (requests that finished earlier)
        batches = [[s] for s in ph.seqs] if match_all else [ph.seqs]
        for seqs in batches:
            pp = pc.plan(seqs, match_all=match_all)
            op = oc.extend_prepare(seqs, match_all=match_all)
            assert pp.prefix_len.tolist() == op.prefix_len
            for b, s in enumerate(seqs):
                assert pp.rows[b, :len(s)].tolist() == op.rows[b].tolist()
            assert (pp.evict_request, pp.evicted) == (op.evict_request, op.evicted)
            _, dups = pc.finish(pp, keep_locked=ph.keep_locked)
            oc.extend_finish(seqs, op, keep_locked=ph.keep_locked)
            assert dups == op.freed_dups
        np.testing.assert_array_equal(oc.tree.dump(), pc.tree.dump())
    return pc, oc


@pytest.mark.parametrize("name", ["tiny_extend", "few_shot_extend", "two_level_extend"])
def test_extend_workloads_match_oracle(name):
    w = W.CONFIGS[name]()
    pc, oc = _run_phases_both(w)
    assert pc.pool.available() == oc.pool.available()


@pytest.mark.slow
def test_multi_turn_decode_host_matches_oracle():
    w = W.multi_turn_decode()
    _run_phases_both(w)


@pytest.mark.slow
def test_fork_mixed_steps_host_match_oracle():
    fm = W.fork_mixed_step()
    w = fm.workload
    pc, oc = _run_phases_both(w)
    assert pc.pool.available() == 4096
    for step in range(3):
        ext = fm.extend_seqs(step)
        pp = pc.plan(ext, extra=len(fm.decode_seqs))
        op = oc.extend_prepare(ext, extra=len(fm.decode_seqs))
        assert pp.prefix_len.tolist() == op.prefix_len == [1500] * 80
        assert pp.evicted == op.evicted and pp.evicted >= 12032
        assert pp.extra.tolist() == op.extra_slots.tolist()
        pc.finish(pp)
        oc.extend_finish(ext, op)
        np.testing.assert_array_equal(oc.tree.dump(), pc.tree.dump())


# ---------------------------------------------------------------- decode grouping (host)
def _lcp(a, b, n):
    d = np.flatnonzero(a[:n] != b[:n])
    return int(d[0]) if d.size else n


@pytest.mark.parametrize("seed", range(12))
def test_shared_context_groups_are_valid(seed):
    """Every group: disjoint members, 2..cap of them, rows identical over the shared length, the
    shared length is the smallest common prefix with the leader and at least min_shared, and
    no longer than any member's context."""
    from prefix_cached_paged_gb300 import shared_context_groups
    rng = np.random.default_rng(seed)
    B, W_ = 40, 300
    rows = rng.integers(0, 10_000, (B, W_)).astype(np.int32)
    lengths = rng.integers(1, W_ + 1, B)
    # families: copy a leader's prefix of random length into some requests
    for b in range(B):
        if rng.random() < 0.7:
            src = int(rng.integers(0, B))
            n = int(rng.integers(0, W_))
            rows[b, :n] = rows[src, :n]
    cap = int(rng.choice([2, 4, 8]))
    min_shared = int(rng.choice([1, 16, 64]))
    indptr, members, shared = shared_context_groups(rows, lengths, cap, min_shared)
    assert indptr[0] == 0 and len(indptr) == len(shared) + 1
    assert len(set(members.tolist())) == len(members)            # each request at most once
    for g in range(len(shared)):
        mem = members[indptr[g]:indptr[g + 1]]
        assert 2 <= len(mem) <= cap
        sh = int(shared[g])
        assert sh >= min_shared
        lead = mem[0]
        assert sh == min(_lcp(rows[lead], rows[x], int(min(lengths[lead], lengths[x])))
                         for x in mem[1:])
        for x in mem:
            assert sh <= lengths[x]
            np.testing.assert_array_equal(rows[x, :sh], rows[lead, :sh])


def test_shared_context_groups_find_families():
    """Four families of three requests over long shared prefixes and four loners: each family
    becomes one group whose shared length is its prefix."""
    from prefix_cached_paged_gb300 import shared_context_groups
    rng = np.random.default_rng(7)
    rows = rng.integers(0, 1 << 30, (16, 900)).astype(np.int32)
    lengths = np.full(16, 900)
    for f in range(4):
        for i in (1, 2):
            rows[3 * f + i, :500 + 100 * f] = rows[3 * f, :500 + 100 * f]
    indptr, members, shared = shared_context_groups(rows, lengths, 8, 64)
    got = sorted((tuple(sorted(members[indptr[g]:indptr[g + 1]].tolist())), int(shared[g]))
                 for g in range(len(shared)))
    assert got == [((0, 1, 2), 500), ((3, 4, 5), 600), ((6, 7, 8), 700), ((9, 10, 11), 800)]


# ---------------------------------------------------------------- extend stacking groups (host)
@pytest.mark.parametrize("seed", range(12))
def test_prefix_stacking_groups_are_valid(seed):
    """Ranges ascending and disjoint, at least two requests each, rows identical over the shared
    length, which is at least min_shared, within every member's prefix, and the smallest
    agreement with the run's first request; max_group_rows bounds each group's new tokens."""
    from tests.planner_ref import prefix_stacking_groups
    rng = np.random.default_rng(100 + seed)
    B, W_ = 30, 400
    rows = rng.integers(0, 10_000, (B, W_)).astype(np.int32)
    P = rng.integers(0, W_, B)
    S = rng.integers(0, 50, B)
    for b in range(1, B):
        if rng.random() < 0.6:
            n = int(rng.integers(0, W_))
            rows[b, :n] = rows[b - 1, :n]
    min_shared = int(rng.choice([1, 32, 128]))
    ranges, shared, max_rows = prefix_stacking_groups(rows, P, S, min_shared)
    assert len(ranges) == 2 * len(shared)
    prev_end = 0
    for g in range(len(shared)):
        b0, b1 = int(ranges[2 * g]), int(ranges[2 * g + 1])
        assert prev_end <= b0 and b1 - b0 >= 2
        prev_end = b1
        sh = int(shared[g])
        assert sh >= min_shared
        assert int(S[b0:b1].sum()) <= max_rows
        agree = []
        for b in range(b0, b1):
            assert sh <= P[b]
            np.testing.assert_array_equal(rows[b, :sh], rows[b0, :sh])
            if b > b0:
                n = int(min(P[b0], P[b]))
                d = np.flatnonzero(rows[b0, :n] != rows[b, :n])
                agree.append(int(d[0]) if d.size else n)
        assert sh == min(agree + [int(P[b0])])


def test_stacking_policy_on_the_measured_workloads():
    """The calibrated cost model makes the choices the kernel replays measured best on GB300:
    it stacks the few-shot batch (50-token suffixes over 2000 shared tokens, MHA; folded 586 vs
    368 TFLOP/s unstacked) and leaves each program of the fork step (5 x 200-token suffixes over
    1500 shared tokens; unstacked 813 vs 709 folded) and the two-level GQA batch (unstacked 636
    vs 603 folded) alone."""
    from tests.planner_ref import stacking_pays
    assert stacking_pays([2000] * 64, [50] * 64, 2000, 1)
    assert not stacking_pays([1500] * 5, [200] * 5, 1500, 1)
    v = np.random.default_rng(0).integers(1, 99, 64)
    assert not stacking_pays(1000 + v, (100 - v) + 20, 1000, 8)


def _serve_queue_product(pq, policy):
    """Serve the whole queue batch by batch through the product's host path."""
    w = pq.workload
    hc = runtime.HostCache(w.pool_slots, w.max_ctx, w.pool_order)
    waiting = list(range(len(pq.seqs)))
    steps = []
    while waiting:
        idx = hc.schedule([pq.seqs[i] for i in waiting], pq.max_batch, pq.max_new_tokens,
                          policy=policy)
        assert idx, "no progress"
        ids = [waiting[i] for i in idx]
        p = hc.plan([pq.seqs[i] for i in ids])
        steps.append((ids, p.prefix_len.tolist(), int(p.evicted)))
        hc.finish(p)
        for i in sorted(idx, reverse=True):
            waiting.pop(i)
    return steps


def _serve_queue_oracle(pq, fcfs):
    w = pq.workload
    sim = oracle.CacheSim(w.pool_slots, w.pool_order)
    waiting = list(range(len(pq.seqs)))
    steps = []
    while waiting:
        seqs = [pq.seqs[i] for i in waiting]
        order, _, adm = oracle.schedule_batch(sim.tree, seqs, [len(s) - 1 for s in seqs], fcfs,
                                              pq.max_batch, pq.max_new_tokens)
        assert adm > 0, "no progress"
        ids = [waiting[i] for i in order[:adm]]
        batch = [pq.seqs[i] for i in ids]
        res = sim.extend_prepare(batch)
        steps.append((ids, list(res.prefix_len), int(res.evicted)))
        sim.extend_finish(batch, res)
        for i in sorted(order[:adm], reverse=True):
            waiting.pop(i)
    return steps


@pytest.mark.parametrize("size", ["small", "full"])
def test_program_queue_schedules_match_oracle(size):
    """The program queue served under both policies: the same batches, matches and evictions
    as the oracle's loop, and longest-shared-prefix-first computes far fewer tokens."""
    if size == "small":
        pq = W.program_queue(n_programs=6, prefix_len=200, n_questions=4, question_len=20,
                             pool_slots=700, max_batch=8, max_new_tokens=1200)
    else:
        pq = W.program_queue()
    computed = {}
    for policy, fcfs in ((rc.RC_SCHED_LSPF, False), (rc.RC_SCHED_FCFS, True)):
        a = _serve_queue_product(pq, policy)
        b = _serve_queue_oracle(pq, fcfs)
        assert a == b
        served = sorted(i for ids, _, _ in a for i in ids)
        assert served == list(range(len(pq.seqs)))
        computed[fcfs] = sum(len(pq.seqs[i]) - p for ids, pl, _ in a for i, p in zip(ids, pl))
    assert computed[False] < 0.5 * computed[True]


@pytest.mark.parametrize("seed", range(24))
def test_host_tier_random_ops_match_oracle_bit_exact(seed):
    """A tree with a host tier against the oracle's: random matches (device-only and through
    both tiers, with loads), inserts, locks, evictions that spill and drop, and drains; the
    same dumps, tiers, pool contents, owed copies and counters after every step."""
    rnd = random.Random(9000 + seed)
    alpha = rnd.choice([2, 3, 5])
    N, NH = rnd.choice([(120, 60), (200, 150), (80, 400), (100, 25)])
    order = np.array(rnd.sample(range(N), N), dtype=np.int32)
    horder = np.array(rnd.sample(range(NH), NH), dtype=np.int32)
    op_, oh = oracle.Pool(N, order), oracle.Pool(NH, horder)
    ot = oracle.Tree(op_)
    ot.attach_host(oh)
    pp, ph = rc.Pool(N, order), rc.Pool(NH, horder)
    pt = rc.RadixTree(pp)
    pt.attach_host_tier(ph)
    locked, cached = [], []
    seen = {"spill": 0, "load": 0, "drop": 0, "refused": 0}
    for step in range(160):
        r = rnd.random()
        toks = [rnd.randrange(alpha) for _ in range(rnd.randint(1, 14))]
        if cached and rnd.random() < 0.5:
            toks = rnd.choice(cached)[:rnd.randint(1, 14)] + toks[:rnd.randint(0, 3)]
        if r < 0.2:
            n1, s1, id1 = ot.match(toks)
            n2, s2, h2 = pt.match_prefix(toks)
            assert (n1, s1.tolist()) == (n2, s2.tolist())
            if rnd.random() < 0.4:
                ot.lock(id1)
                pt.lock(h2)
                locked.append((id1, h2))
        elif r < 0.4:
            # through both tiers, then load the host part if the device pool has room
            d1, h1, s1, id1 = ot.match_tiered(toks)
            ot.lock(id1)
            t = np.array(toks, np.int32)
            ip = np.array([0, len(t)], np.int64)
            rows = np.zeros((1, 32), np.int32)
            pl, nodes, hl = pt.match_batch_tiered(t, ip, None, rows)
            assert (d1, h1, s1.tolist()) == (int(pl[0]), int(hl[0]), rows[0, :d1].tolist())
            locked.append((id1, int(nodes[0])))
            if h1 and op_.available() >= h1:
                row1 = ot.load(t[:d1 + h1])
                pt.load_batch(t, ip, rows, pl, hl)
                assert row1.tolist() == rows[0, :d1 + h1].tolist() and pl[0] == d1 + h1
                seen["load"] += 1
        elif r < 0.6:
            a1 = op_.alloc(len(toks))
            if a1 is None:
                continue
            a2 = pp.alloc(len(toks))
            assert a1.tolist() == a2.tolist()
            e1, _ = ot.insert(toks, a1)
            e2, _ = pt.insert(toks, a2)
            assert e1 == e2
            op_.free(a1[:e1])
            pp.free(a2[:e2])
            cached.append(toks)
        elif r < 0.7 and locked:
            i1, h2 = locked.pop(rnd.randrange(len(locked)))
            ot.unlock(i1)
            pt.unlock(h2)
        elif r < 0.84:
            want = rnd.randint(0, 40)
            ok1, f1, _ = ot.evict(want)
            try:
                st, f2 = pt.evict_lru(want)
            except rc.RcError as e:      # loads still owed: both refuse and change nothing
                assert e.code == rc.RC_ERR_INVALID and not ok1 and f1 == 0
                seen["refused"] += 1
                continue
            assert f1 == f2 and ok1 == (st == rc.RC_OK)
        else:
            c1 = ot.drain()
            c2 = pt.drain_copies()
            for a, b in zip(c1, c2):
                assert a.tolist() == b.tolist()
            seen["spill"] += len(c1[0])
        np.testing.assert_array_equal(ot.dump(), pt.dump())
        np.testing.assert_array_equal(ot.tiers(), pt.tiers())
        assert (op_.available(), oh.available()) == (pp.available(), ph.available())
        s1, s2 = ot.stats(), pt.stats()
        for k in ("evicted_nodes", "evicted_tokens", "nodes", "cached_tokens",
                  "protected_tokens", "host_tokens", "spilled_tokens", "loaded_tokens",
                  "dropped_tokens"):
            assert s1[k] == s2[k], k
        seen["drop"] = s2["dropped_tokens"]
    c1, c2 = ot.drain(), pt.drain_copies()
    for a, b in zip(c1, c2):
        assert a.tolist() == b.tolist()
    # both free lists agree in order
    assert op_.alloc(op_.available()).tolist() == pp.alloc(pp.available()).tolist()
    assert oh.alloc(oh.available()).tolist() == ph.alloc(ph.available()).tolist()
    assert pt.stats()["spilled_tokens"] > 0


def _serve_tiered(pq, fcfs, host_slots, product):
    """Serve the queue with a host tier: per batch (ids, prefix_len, host_len, copies)."""
    w = pq.workload
    if product:
        hc = runtime.HostCache(w.pool_slots, w.max_ctx, w.pool_order, host_slots=host_slots)
    else:
        sim = oracle.CacheSim(w.pool_slots, w.pool_order, host_slots=host_slots)
    waiting = list(range(len(pq.seqs)))
    steps = []
    while waiting:
        seqs = [pq.seqs[i] for i in waiting]
        if product:
            idx = hc.schedule(seqs, pq.max_batch, pq.max_new_tokens,
                              policy=rc.RC_SCHED_FCFS if fcfs else rc.RC_SCHED_LSPF)
            p = hc.plan([pq.seqs[waiting[i]] for i in idx])
            step = (p.prefix_len.tolist(), p.host_len.tolist(), [c.tolist() for c in p.copies])
            hc.finish(p)
        else:
            order, _, adm = oracle.schedule_batch(sim.tree, seqs, [len(s) - 1 for s in seqs],
                                                  fcfs, pq.max_batch, pq.max_new_tokens)
            idx = order[:adm]
            batch = [pq.seqs[waiting[i]] for i in idx]
            res = sim.extend_prepare(batch)
            step = (list(res.prefix_len), list(res.host_len), [c.tolist() for c in res.copies])
            sim.extend_finish(batch, res)
        assert idx, "no progress"
        steps.append(([waiting[i] for i in idx],) + step)
        for i in sorted(idx, reverse=True):
            waiting.pop(i)
    return steps


@pytest.mark.parametrize("fcfs", [False, True])
@pytest.mark.parametrize("size", ["small", "full"])
def test_program_queue_with_host_tier_matches_oracle(fcfs, size):
    """The program queue with a host tier behind a small device pool: the same batches, matches,
    loads and owed copies as the oracle's loop; the tier turns recomputation into loads."""
    if size == "small":
        kw = dict(n_programs=6, prefix_len=200, n_questions=4, question_len=20, pool_slots=700,
                  max_batch=8, max_new_tokens=1200)
        host = 2000
    else:
        kw = dict(pool_slots=8_000)
        host = 60_000
    pq = W.program_queue(**kw)
    a = _serve_tiered(pq, fcfs, host, product=True)
    b = _serve_tiered(pq, fcfs, host, product=False)
    assert a == b
    loaded = sum(sum(h) for _, _, h, _ in a)
    computed = sum(len(pq.seqs[i]) - p for ids, pl, _, _ in a for i, p in zip(ids, pl))
    without = sum(len(pq.seqs[i]) - p for ids, pl, _ in
                  _serve_queue_product(pq, rc.RC_SCHED_FCFS if fcfs else rc.RC_SCHED_LSPF)
                  for i, p in zip(ids, pl))
    if fcfs:
        # interleaved arrival evicts every prefix before its next question: the tier loads
        # them back instead of recomputing
        assert loaded > 0 and computed < without
    else:
        # longest shared prefix first finishes a program before leaving it: little to reload
        assert computed <= without


@pytest.mark.parametrize("seed", range(10))
def test_prefix_stacking_levels_are_valid(seed):
    """Nested stacking groups: within a level ranges ascend and are disjoint; each deeper group
    lies inside a group of the level above and starts at that group's shared length; members
    agree with the group's first over [0, shared), shared >= start + min_shared."""
    rnd = random.Random(400 + seed)
    B, width, min_shared = rnd.randint(2, 24), 120, 8
    rows = np.zeros((B, width), np.int32)
    base = [rnd.randrange(1000) for _ in range(width)]
    for b in range(B):
        # nested agreement: a random cut sequence along the sorted requests
        cut = rnd.choice([10, 30, 60, 90, 119]) if b % rnd.randint(1, 4) else rnd.randint(0, 40)
        rows[b] = base
        rows[b, cut:] = [rnd.randrange(1000, 2000) for _ in range(width - cut)]
    P = np.full(B, width, np.int64)
    S = np.array([rnd.randint(0, 30) for _ in range(B)], np.int64)
    ranges, shared, start, lvl, max_rows = planner_ref.prefix_stacking_levels(rows, P, S,
                                                                              min_shared)
    assert lvl[0] == 0 and lvl[-1] == len(shared) and np.all(np.diff(lvl) > 0)
    spans = {}
    for l in range(len(lvl) - 1):
        prev_end = 0
        for g in range(lvl[l], lvl[l + 1]):
            b0, b1, sh, st = int(ranges[2 * g]), int(ranges[2 * g + 1]), int(shared[g]), int(start[g])
            assert prev_end <= b0 < b1 and b1 - b0 >= 2
            prev_end = b1
            assert sh >= st + min_shared
            for b in range(b0, b1):
                assert np.array_equal(rows[b, :sh], rows[b0, :sh])
            if l == 0:
                assert st == 0
            else:
                parents = [(p0, p1, psh) for (p0, p1, psh) in spans[l - 1] if p0 <= b0 and b1 <= p1]
                assert len(parents) == 1 and parents[0][2] == st
            spans.setdefault(l, []).append((b0, b1, sh))
    assert max_rows == max([int(S[int(ranges[2 * g]):int(ranges[2 * g + 1])].sum())
                            for g in range(len(shared))], default=0)


def test_new_entry_points_reject_bad_arguments():
    """Argument checks of the scheduler, the host tier and the KV copy (host side; nothing here
    reaches a device)."""
    import ctypes
    from prefix_cached_paged_gb300._lib import RcKvCopyArgs
    pool, hpool = rc.Pool(50), rc.Pool(20)
    t = rc.RadixTree(pool)
    # the scheduler: unknown policy, match longer than the sequence
    tok = np.arange(6, dtype=np.int32)
    ip = np.array([0, 6], np.int64)
    with pytest.raises(rc.RcError) as e:
        t.schedule_batch(tok, ip, None, policy=7)
    assert e.value.code == rc.RC_ERR_INVALID
    with pytest.raises(rc.RcError):
        t.schedule_batch(tok, ip, np.array([7], np.int32))
    # loads need a host tier; a tier is attached once and is not the device pool
    rows = np.zeros((1, 8), np.int32)
    with pytest.raises(rc.RcError):
        t.load_batch(tok, ip, rows, np.zeros(1, np.int32), np.zeros(1, np.int32))
    with pytest.raises(rc.RcError):
        t.attach_host_tier(pool)
    t.attach_host_tier(hpool)
    with pytest.raises(rc.RcError):
        t.attach_host_tier(rc.Pool(5))
    # a load asks for more device slots than are free: RC_ERR_OOM, nothing moved
    t.insert(list(range(6)), pool.alloc(6))
    assert t.evict_lru(6) == (rc.RC_OK, 6)           # spilled to the host tier
    assert t.drain_copies()[0].size == 6
    pl, nodes, hl = t.match_batch_tiered(tok, ip, None, rows)
    assert (int(pl[0]), int(hl[0])) == (0, 6)
    pool.alloc(pool.available() - 3)
    with pytest.raises(rc.RcError) as e:
        t.load_batch(tok, ip, rows, pl, hl)
    assert e.value.code == rc.RC_ERR_OOM and pl[0] == 0
    # the KV copy: rows not a multiple of 16 bytes, NULL planes, misaligned planes
    def kv(**kw):
        a = dict(n=1, layers=1, row_bytes=256, src_slots=16, dst_slots=16, src_k=256, src_v=512,
                 src_num_slots=4, dst_k=768, dst_v=1024, dst_num_slots=4)
        a.update(kw)
        return lib().rc_kv_copy(ctypes.byref(RcKvCopyArgs(**a)), None)
    assert kv(row_bytes=100) == rc.RC_ERR_INVALID
    assert kv(src_k=0) == rc.RC_ERR_INVALID
    assert kv(dst_v=1032) == rc.RC_ERR_INVALID
    assert kv(layers=0) == rc.RC_ERR_INVALID


@pytest.mark.parametrize("seed", range(8))
def test_fold_groups_follow_their_rule(seed):
    """fold_groups marks exactly the groups that no deeper group lies inside and whose folded
    pass the cost model puts at no more than the stacked pass plus the members' own passes
    (every innermost group with force); all_folded is whether every request is in such a
    group."""
    rnd = random.Random(600 + seed)
    B, width = rnd.randint(2, 20), 400
    rows = np.zeros((B, width), np.int32)
    base = [rnd.randrange(1000) for _ in range(width)]
    for b in range(B):
        cut = rnd.choice([50, 120, 260, 300, 399]) if b % rnd.randint(1, 3) else rnd.randint(0, 60)
        rows[b] = base
        rows[b, cut:] = [rnd.randrange(1000, 2000) for _ in range(width - cut)]
    P = np.array([rnd.randint(260, width) for _ in range(B)], np.int64)
    S = np.array([rnd.randint(1, 150) for _ in range(B)], np.int64)
    grp = rnd.choice([1, 4, 8])
    ranges, shared, start, lvl, _ = planner_ref.prefix_stacking_levels(rows, P, S, 8)
    for force in (False, True):
        fold, all_folded = planner_ref.fold_groups(ranges, shared, lvl, P, S, grp, start,
                                                   force=force)
        G = len(shared)
        level = np.repeat(np.arange(len(lvl) - 1), np.diff(lvl))
        covered = np.zeros(B, bool)
        for g in range(G):
            b0, b1 = int(ranges[2 * g]), int(ranges[2 * g + 1])
            leaf = not any(level[h] > level[g] and b0 <= ranges[2 * h] and ranges[2 * h + 1] <= b1
                           for h in range(G))
            _, unfolded, folded = planner_ref._stacking_costs(P[b0:b1], S[b0:b1], int(shared[g]),
                                                              grp, int(start[g]))
            fits = planner_ref._folded_cost_us(P[b0:b1], S[b0:b1], int(shared[g]),
                                               int(start[g]), max(128 // grp, 1), limits=True)
            assert bool(fold[g]) == (leaf and fits and (force or folded <= unfolded)), g
            if fold[g]:
                covered[b0:b1] = True
        assert all_folded == bool(covered.all())


@pytest.mark.parametrize("shared", [True, False])
def test_waiting_queue_schedules_like_the_list(shared):
    """Serving a program queue through a WaitingQueue (ranges of one buffer, rc_schedule_batch_
    ranges) forms the same batches as passing the waiting sequences as lists, and leaves the same
    tree."""
    from synth import workloads as W
    pq = W.program_queue(layers=1, shared=shared, n_programs=6)
    w = pq.workload
    runs = []
    for use_queue in (False, True):
        hc = runtime.HostCache(w.pool_slots, w.max_ctx, w.pool_order)
        wq = runtime.WaitingQueue(pq.seqs)
        waiting = list(range(len(pq.seqs)))
        batches = []
        while waiting:
            arg = wq if use_queue else [pq.seqs[i] for i in waiting]
            idx = hc.schedule(arg, pq.max_batch, pq.max_new_tokens, policy=rc.RC_SCHED_LSPF)
            assert idx
            ids = [waiting[i] for i in idx]
            if use_queue:
                assert [wq.ids[i] for i in idx] == ids
                assert all(np.array_equal(wq.seq(q), pq.seqs[q]) for q in ids)
            p = hc.plan([pq.seqs[i] for i in ids])
            batches.append((ids, p.prefix_len.tolist()))
            hc.finish(p)
            for i in sorted(idx, reverse=True):
                waiting.pop(i)
            wq.remove(idx)
        runs.append((batches, hc.tree.dump()))
    assert runs[0][0] == runs[1][0]
    np.testing.assert_array_equal(runs[0][1], runs[1][1])


def test_schedule_ranges_rejects_bad_arguments():
    t = rc.RadixTree(rc.Pool(20))
    tok = np.arange(6, dtype=np.int32)
    for starts, lengths, ml in (([-1], [3], None), ([0], [-2], None), ([0], [3], [4])):
        with pytest.raises(rc.RcError) as e:
            t.schedule_batch_ranges(tok, np.array(starts), np.array(lengths),
                                    None if ml is None else np.array(ml, np.int32))
        assert e.value.code == rc.RC_ERR_INVALID
    with pytest.raises(rc.RcError):
        t.schedule_batch_ranges(tok, np.array([0]), np.array([3]), None, policy=9)
    order, match, adm = t.schedule_batch_ranges(tok, np.zeros(0), np.zeros(0))
    assert (len(order), adm) == (0, 0)


def _random_stacking_case(rnd):
    """Families of consecutive requests sharing slot prefixes of random lengths (some nested),
    random private parts and new-token counts."""
    B, width = rnd.randint(2, 24), 700
    rows = np.zeros((B, width), np.int32)
    P = np.zeros(B, np.int64)
    S = np.zeros(B, np.int64)
    b = 0
    fresh = iter(range(10_000, 10_000_000))
    while b < B:
        n = min(rnd.randint(1, 7), B - b)
        base = [next(fresh) for _ in range(width)]
        sub = rnd.choice([0, 0, rnd.randint(1, 600)])
        for i in range(n):
            row = list(base)
            cut = rnd.choice([rnd.randint(0, 80), rnd.randint(200, 690)])
            if sub and i % 2:
                cut = max(cut, sub)
            for c in range(cut, width):
                row[c] = next(fresh)
            rows[b + i] = row
            P[b + i] = rnd.randint(min(cut + 1, width - 1) if rnd.random() < 0.5 else 0, width - 1)
            S[b + i] = rnd.choice([0, 1, rnd.randint(1, 60), rnd.randint(60, 400)])
        b += n
    return rows, P, S


@pytest.mark.parametrize("seed", range(40))
def test_stacking_planner_matches_reference(seed):
    """rc_plan_extend_stacking makes exactly the reference planner's decisions (groups, levels,
    shared lengths, key starts, folds, max rows, all folded) on random batches, for every policy,
    fold mode, group size and depth."""
    rnd = random.Random(900 + seed)
    rows, P, S = _random_stacking_case(rnd)
    for grp in (1, 8):
        for policy in ("cost", "all"):
            for fold in (False, True, "always"):
                levels = rnd.randint(1, 4)
                got = rc.plan_extend_stacking(rows, P, S, 256, grp, levels, policy, fold)
                pays = None if policy == "all" else (
                    lambda b0, b1, sh, st: planner_ref.stacking_pays(P[b0:b1], S[b0:b1], sh, grp,
                                                                     st))
                ranges, shared, start, lvl, max_rows = planner_ref.prefix_stacking_levels(
                    rows, P, S, 256, pays, levels)
                if len(shared) and fold:
                    fo, allf = planner_ref.fold_groups(ranges, shared, lvl, P, S, grp, start,
                                                       force=fold == "always")
                else:
                    fo, allf = np.zeros(len(shared), np.int32), False
                assert got[0].tolist() == ranges.tolist()
                assert got[1].tolist() == shared.tolist()
                assert got[2].tolist() == start.tolist()
                assert got[3].tolist() == lvl.tolist()
                assert got[4] == max_rows
                assert got[5].tolist() == fo.tolist()
                assert got[6] == (bool(allf) and len(shared) > 0)


@pytest.mark.parametrize("name", ["few_shot_extend", "two_level_extend", "fork_extend"])
def test_stacking_planner_on_the_target_batches(name):
    """The C planner and the reference agree on the target workloads' extend batches (host
    plans built through the product's tree): few-shot, two-level tree, and one step of the fork
    mixed step."""
    from synth import workloads as W
    if name == "fork_extend":
        fm = W.fork_mixed_step(layers=1)
        w = fm.workload
        cache, ext = fm.programs, fm.extend_seqs(0)
    else:
        w = W.CONFIGS[name]()
        cache = [s for ph in w.phases[:-1] for s in ph.seqs]
        ext = w.phases[-1].seqs
    hc = runtime.HostCache(w.pool_slots, w.max_ctx, w.pool_order)
    for s in cache:
        p = hc.plan([s], match_all=True)
        hc.finish(p)
    plan = hc.plan(ext)
    S = plan.lengths - plan.prefix_len
    G = w.model.n_q_heads // w.model.n_kv_heads
    got = rc.plan_extend_stacking(plan.rows, plan.prefix_len, S, 256, G, 4, "cost", True)
    pays = lambda b0, b1, sh, st: planner_ref.stacking_pays(plan.prefix_len[b0:b1], S[b0:b1], sh,
                                                            G, st)
    ranges, shared, start, lvl, max_rows = planner_ref.prefix_stacking_levels(
        plan.rows, plan.prefix_len, S, 256, pays, 4)
    assert got[0].tolist() == ranges.tolist() and got[1].tolist() == shared.tolist()
    assert got[2].tolist() == start.tolist() and got[3].tolist() == lvl.tolist()
    assert got[4] == max_rows
    if len(shared):
        fo, allf = planner_ref.fold_groups(ranges, shared, lvl, plan.prefix_len, S, G, start)
        assert got[5].tolist() == fo.tolist() and got[6] == allf


@pytest.mark.parametrize("seed", range(30))
def test_decode_planner_matches_reference(seed):
    """rc_plan_decode_groups forms exactly the reference's shared-context groups on random slot
    rows (buckets by first slot, ties, caps, short contexts)."""
    rnd = random.Random(1300 + seed)
    B, width = rnd.randint(0, 40), 300
    rows = np.zeros((B, width), np.int32)
    lengths = np.zeros(B, np.int64)
    bases = [[rnd.randrange(5) * 1000 + c for c in range(width)] for _ in range(4)]
    for b in range(B):
        rows[b] = bases[rnd.randrange(4)]
        cut = rnd.choice([0, rnd.randint(1, 100), rnd.randint(100, 299)])
        rows[b, cut:] = [rnd.randrange(10**6, 10**7) for _ in range(width - cut)]
        lengths[b] = rnd.randint(0, width)
    for cap in (1, 2, 4, 8):
        for min_shared in (1, 32, 128):
            got = rc.shared_context_groups(rows, lengths, cap, min_shared)
            ref = planner_ref.shared_context_groups(rows, lengths, cap, min_shared)
            for x, y in zip(got, ref):
                assert x.tolist() == y.tolist(), (cap, min_shared)


def test_decode_planner_on_the_target_batches():
    """Both decode planners agree on the multi-turn decode contexts and the fork step's decode
    requests."""
    from synth import workloads as W
    for w, ctx in ((W.multi_turn_decode(), None), (W.fork_mixed_step(layers=1).workload, "fork")):
        hc = runtime.HostCache(w.pool_slots, w.max_ctx, w.pool_order)
        for ph in w.phases[:-1] if ctx is None else w.phases:
            for s in ph.seqs:
                p = hc.plan([s], match_all=True)
                hc.finish(p)
        if ctx is None:
            seqs = [s[:-1] for s in w.phases[-1].seqs]
        else:
            seqs = [s[:-1] for s in W.fork_mixed_step(layers=1).decode_seqs]
        plan = hc.plan(seqs, match_all=True)
        G = w.model.n_q_heads // w.model.n_kv_heads
        got = rc.shared_context_groups(plan.rows, plan.lengths, 8 // G, 512)
        ref = planner_ref.shared_context_groups(plan.rows, plan.lengths, 8 // G, 512)
        assert got[1].size > 0
        for x, y in zip(got, ref):
            assert x.tolist() == y.tolist()
