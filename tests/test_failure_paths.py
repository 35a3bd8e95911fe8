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


def _fake(i):
    # a 16-byte aligned address that is never dereferenced: every call below is rejected (or
    # returns) before anything reaches a device
    return 0x10000 + 256 * i


def test_extend_rejects_bad_arguments_before_any_device_work():
    import ctypes
    from prefix_cached_paged_gb300._lib import RcExtendArgs, lib
    ptrs = ["q", "k_new", "v_new", "out_loc", "qo_indptr", "prefix_len", "req_idx",
            "req_to_token", "k_pool", "v_pool", "o"]

    def call(**kw):
        a = dict(dtype=rc.RC_DTYPE_BF16, num_reqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                 max_reqs=4, max_ctx=64, max_q_len=8, max_prefix_len=8, num_tokens=16,
                 num_slots=100, sm_scale=0.088)
        a.update({n: _fake(i) for i, n in enumerate(ptrs)})
        a.update(kw)
        return lib().rc_extend_attention(ctypes.byref(RcExtendArgs(**a)), None)

    bad = [dict(dtype=7), dict(num_kv_heads=3), dict(num_q_heads=0), dict(head_dim=96),
           dict(head_dim=64),                        # 64 only for fp32
           dict(max_ctx=62), dict(max_reqs=0), dict(num_slots=0), dict(num_tokens=-1),
           dict(q=0), dict(req_to_token=0), dict(k_pool=_fake(3) + 8), dict(num_groups=-1),
           dict(num_groups=1),                       # no group arrays
           dict(num_groups=1, group_range=_fake(20), group_shared=_fake(21), max_group_rows=8,
                workspace=_fake(22), workspace_bytes=16)]    # workspace too small
    for kw in bad:
        assert call(**kw) == rc.RC_ERR_INVALID, kw
    # levels: at most RC_MAX_STACK_LEVELS; level_indptr (host) from 0 to num_groups, no empty level
    stack = dict(num_groups=3, group_range=_fake(20), group_shared=_fake(21), max_group_rows=8,
                 workspace=_fake(22), workspace_bytes=1 << 20)
    assert call(num_levels=rc.MAX_STACK_LEVELS + 1, **stack) == rc.RC_ERR_INVALID
    for lv in ([0, 0, 3], [1, 2, 3], [0, 2, 2], [0, 1, 4]):
        li = np.array(lv, np.int32)
        assert call(num_levels=2, level_indptr=li.ctypes.data, **stack) == rc.RC_ERR_INVALID, lv
    # nothing to do is not an error, and touches no device
    assert call(num_reqs=0) == rc.RC_OK and call(max_q_len=0) == rc.RC_OK


def test_decode_rejects_bad_arguments_before_any_device_work():
    import ctypes
    from prefix_cached_paged_gb300._lib import RcDecodeArgs, lib
    ptrs = ["q", "k_new", "v_new", "out_loc", "seq_len", "req_idx", "req_to_token", "k_pool",
            "v_pool", "o"]

    def args(**kw):
        a = dict(dtype=rc.RC_DTYPE_BF16, num_reqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                 max_reqs=4, max_ctx=64, kv_chunk=0, max_total_tokens=128, num_slots=100,
                 sm_scale=0.088)
        a.update({n: _fake(i) for i, n in enumerate(ptrs)})
        a.update(kw)
        return RcDecodeArgs(**a)

    need = ctypes.c_size_t()
    assert lib().rc_decode_workspace_bytes(ctypes.byref(args()), ctypes.byref(need)) == rc.RC_OK
    ws = _fake(30)

    def call(ws=ws, ws_bytes=need.value, **kw):
        return lib().rc_decode_attention(ctypes.byref(args(**kw)), ws, ws_bytes, None)

    bad = [dict(dtype=7), dict(num_q_heads=6),      # group size 3
           dict(num_q_heads=32),                     # group size 16
           dict(head_dim=96), dict(kv_chunk=100), dict(kv_chunk=-64), dict(max_ctx=0),
           dict(num_slots=0), dict(max_total_tokens=-1), dict(num_groups=-1), dict(num_groups=1),
           dict(q=0), dict(k_pool=_fake(7) + 8)]
    for kw in bad:
        assert call(**kw) == rc.RC_ERR_INVALID, kw
    assert call(ws=None) == rc.RC_ERR_INVALID                     # no workspace
    assert call(ws=ws + 8) == rc.RC_ERR_INVALID                   # misaligned workspace
    assert call(ws_bytes=need.value - 1) == rc.RC_ERR_INVALID     # workspace too small
    assert call(num_reqs=0) == rc.RC_OK
    # the allocation-free variant rejects work beyond its fixed scratch area
    big = args(kv_chunk=64, max_total_tokens=10**9)
    assert lib().rc_decode_attention_noalloc(ctypes.byref(big), None) == rc.RC_ERR_INVALID
    assert "scratch" in lib().rc_last_error().decode()


def test_engine_checks_slot_table_rows_before_planning():
    """With too few free slot-table rows, extend_begin and decode_begin fail before planning,
    so no slot is allocated and no prefix stays locked (the engine's device side is not needed
    to reach the check)."""
    from prefix_cached_paged_gb300.serving import Engine
    hc = runtime.HostCache(1000, 64)
    pre = synth.tokens(3, 1, 40)
    _cache(hc, [pre])
    eng = Engine.__new__(Engine)           # host side only: no device tensors
    eng.host = hc
    eng._free_rows = [1, 0]
    seqs = [np.concatenate([pre, synth.tokens(3, 10 + i, 5)]).astype(np.int32) for i in range(3)]
    avail = hc.pool.available()
    with pytest.raises(RuntimeError, match="free rows"):
        eng.extend_begin(seqs)
    with pytest.raises(RuntimeError, match="free rows"):
        eng.decode_begin([pre, pre, pre])
    assert hc.pool.available() == avail
    assert hc.tree.stats()["protected_tokens"] == 0


class _HostOnlyDevice:
    """Stands in for the engine's device side in host-bookkeeping tests: slot-table writes and
    metadata uploads are accepted and dropped."""

    def write_rows(self, row_ids, rows, ends, cols=None):
        pass

    def upload_i32(self, arrays):
        return [None for _ in arrays]


def _host_engine(hc, rows=8, max_ctx=64):
    from prefix_cached_paged_gb300.serving import Engine
    eng = Engine.__new__(Engine)
    eng.host, eng.dev = hc, _HostOnlyDevice()
    eng._free_rows = list(range(rows - 1, -1, -1))
    eng.share_decode, eng.kv_chunk, eng.max_ctx = False, 0, max_ctx
    eng.stack_extend = False
    return eng


@pytest.mark.parametrize("insert", [False, True])
def test_decode_end_returns_or_caches_the_generated_tokens(insert):
    """Every decode step takes a slot per request; when the requests end, their generated
    tokens' slots go back to the pool, or the finished sequences are inserted into the tree (the
    pages' insert after a request finishes) and their generated tokens become reusable."""
    hc = runtime.HostCache(1000, 64)
    ctx = [synth.tokens(5, 1 + i, 20 + 3 * i) for i in range(3)]
    _cache(hc, ctx)
    eng = _host_engine(hc)
    avail0 = hc.pool.available()
    db = eng.decode_begin(ctx)
    steps = 4
    for _ in range(steps):
        eng.decode_step(db)
    assert hc.pool.available() == avail0 - 3 * steps
    gen = [synth.tokens(6, 40 + i, steps) for i in range(3)]
    full = [np.concatenate([c, g]).astype(np.int32) for c, g in zip(ctx, gen)]
    with pytest.raises(ValueError):
        eng.decode_end(db, [c for c in ctx])                  # missing the generated tokens
    eng.decode_end(db, full if insert else None)
    st = hc.tree.stats()
    assert st["protected_tokens"] == 0 and len(eng._free_rows) == 8
    if insert:
        assert hc.pool.available() == avail0 - 3 * steps        # the generated KV stays cached
        plan = hc.plan(full, match_all=True)
        assert plan.prefix_len.tolist() == [len(s) for s in full] and plan.num_tokens == 0
        hc.finish(plan)
    else:
        assert hc.pool.available() == avail0                    # every generated slot returned
        assert st["cached_tokens"] == sum(len(c) for c in ctx)


@pytest.mark.parametrize("host_slots", [0, 150])
@pytest.mark.parametrize("seed", range(6))
def test_engine_bookkeeping_conserves_slots(seed, host_slots):
    """Random extend and decode batches through the engine's host side, with duplicates in a
    batch, eviction under a small pool (spilling to a host tier and loading back, when there is
    one) and injected allocation failures: after every call, each device slot is either free or
    holds a cached token, each host-tier slot likewise, and nothing stays locked."""
    import random
    rnd = random.Random(900 + seed)
    N = 400
    hc = runtime.HostCache(N, 128, synth.permutation(seed, N), host_slots=host_slots)
    eng = _host_engine(hc, rows=8, max_ctx=128)
    eng._tier_copies = lambda copies: None     # the KV copies themselves are device work
    stems = [synth.tokens(seed, 10 + i, rnd.randint(5, 30)) for i in range(4)]

    def new_seq():
        s = rnd.choice(stems)[:rnd.randint(0, 30)]
        tail = np.array([rnd.randrange(3) for _ in range(rnd.randint(1, 25))], np.int32)
        return np.concatenate([s, tail]).astype(np.int32)

    def check():
        st = hc.tree.stats()
        assert st["protected_tokens"] == 0
        assert hc.pool.available() + st["cached_tokens"] == N
        if host_slots:
            # a plan that failed after loading host-tier nodes back leaves their copies owed
            # (handed out by the next plan or allocation): their host slots are held until then
            import ctypes
            from prefix_cached_paged_gb300._lib import lib
            ns, nl = ctypes.c_int64(), ctypes.c_int64()
            assert lib().rc_radix_pending_copies(hc.tree.h, ctypes.byref(ns),
                                                 ctypes.byref(nl)) == rc.RC_OK
            assert hc.host_pool.available() + st["host_tokens"] + nl.value == host_slots
        assert len(eng._free_rows) == 8

    cached = []
    for step in range(150):
        if rnd.random() < 0.15:
            hc.pool.inject_alloc_failure(rnd.randint(0, 1))
        try:
            if rnd.random() < 0.6 or not cached:
                seqs = [new_seq() for _ in range(rnd.randint(1, 4))]
                b = eng.extend_begin(seqs)
                eng.extend_end(b)
                cached += seqs
            else:
                ctx = [rnd.choice(cached) for _ in range(rnd.randint(1, 3))]
                db = eng.decode_begin(ctx)
                n = rnd.randint(1, 4)
                try:
                    for _ in range(n):
                        eng.decode_step(db)
                except rc.RcError:
                    eng.decode_end(db)          # leave decoding: free what was generated
                    raise
                if rnd.random() < 0.5:
                    done = len(db.gen_slots)
                    full = [np.concatenate([c, np.array([rnd.randrange(3) for _ in range(done)],
                                                        np.int32)]).astype(np.int32)
                            for c in ctx]
                    eng.decode_end(db, full)
                    cached += full
                else:
                    eng.decode_end(db)
        except rc.RcError as e:
            assert e.code in (rc.RC_ERR_OOM, rc.RC_ERR_INSUFFICIENT), e
        except ValueError:
            pass        # a decode context evicted before it was matched: not cached any more
        hc.pool.inject_alloc_failure(-1)
        check()
    if host_slots:
        st = hc.tree.stats()
        assert st["spilled_tokens"] > 0 and st["loaded_tokens"] > 0


def test_failed_tiered_plan_hands_its_copies_to_the_next_call():
    """A plan that loaded host-tier nodes back and then failed to allocate leaves copies owed.
    Left in the tree they made every later eviction fail ("loads are pending"); now they come
    out of take_owed (spills and loads, for the caller to run first) and the next plan that needs
    eviction succeeds."""
    hc = runtime.HostCache(100, 128, host_slots=200)
    a = synth.tokens(8, 1, 60)
    b = synth.tokens(8, 2, 60)
    _cache(hc, [a])
    _cache(hc, [b])                       # evicts a to the host tier (100 slots)
    assert hc.take_owed() == [] and hc.tree.stats()["host_tokens"] == 60
    # a + 10 new tokens: loads a back (evicting b to the host tier), then the allocation fails
    seq = np.concatenate([a, synth.tokens(8, 3, 10)]).astype(np.int32)
    hc.pool.inject_alloc_failure(0)
    with pytest.raises(rc.RcError) as e:
        hc.plan([seq])
    assert e.value.code == rc.RC_ERR_OOM
    owed = hc.take_owed()
    assert len(owed) == 1 and len(owed[0][0]) > 0 and len(owed[0][2]) == 60
    assert hc.take_owed() == []
    # the same request again: needs eviction, and works
    plan = hc.plan([seq])
    assert plan.prefix_len.tolist() == [60]
    hc.finish(plan)
    assert hc.tree.stats()["protected_tokens"] == 0


@pytest.mark.parametrize("host_slots", [0, 120])
@pytest.mark.parametrize("seed", range(4))
def test_fork_style_steps_conserve_slots(seed, host_slots):
    """The mixed step's interleaving on the host side: a decode batch lives across steps and takes
    its new tokens' slots from each extend plan's extra allocation, under a nearly full pool and
    injected failures. While it lives, free + cached + its generated slots = the pool; after
    decode_end (inserting or freeing), free + cached = the pool and nothing is locked."""
    import random
    rnd = random.Random(seed)
    N = 500
    hc = runtime.HostCache(N, 256, synth.permutation(seed, N), host_slots=host_slots)
    eng = _host_engine(hc, rows=16, max_ctx=256)
    eng._tier_copies = lambda copies: None
    ctx = [synth.tokens(seed, 100 + i, rnd.randint(10, 40)) for i in range(3)]
    _cache(hc, ctx)
    db = eng.decode_begin(ctx)
    progs = [synth.tokens(seed, 200 + i, rnd.randint(10, 30)) for i in range(2)]
    _cache(hc, progs)
    gen_tok = [[] for _ in ctx]
    failed = 0
    for step in range(40):
        if rnd.random() < 0.15:
            hc.pool.inject_alloc_failure(rnd.randint(0, 1))
        seqs = [np.concatenate([rnd.choice(progs),
                                synth.tokens(seed, 1000 + 10 * step + f, rnd.randint(1, 20))])
                .astype(np.int32) for f in range(rnd.randint(1, 3))]
        try:
            eb = eng.extend_begin(seqs, extra=len(ctx))
        except rc.RcError:
            failed += 1
            hc.pool.inject_alloc_failure(-1)
            continue
        eng.decode_step(db, new_slots=eb.plan.extra)
        for g in gen_tok:
            g.append(rnd.randrange(5))
        eng.extend_end(eb)
        hc.pool.inject_alloc_failure(-1)
        st = hc.tree.stats()
        assert hc.pool.available() + st["cached_tokens"] + len(db.gen_slots) * len(ctx) == N
    assert failed > 0
    full = [np.concatenate([c, np.array(g, np.int32)]).astype(np.int32)
            for c, g in zip(ctx, gen_tok)]
    eng.decode_end(db, full if seed % 2 else None)
    st = hc.tree.stats()
    assert st["protected_tokens"] == 0 and hc.pool.available() + st["cached_tokens"] == N
    if host_slots:
        assert hc.host_pool.available() + st["host_tokens"] == host_slots
