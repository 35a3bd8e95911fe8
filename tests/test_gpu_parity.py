"""GPU path (librc through its C ABI) against the oracle, on seeded synthetic workloads.

Bit-exact: match lengths / prefill tokens skipped, slot rows in the device slot table, and the
pool rows the kernels scatter (compared with the generator's values). Within tolerance (bf16:
max-abs 1e-2 and rel-L2 5e-3 against fp64; fp32: 1e-4 and 1e-5): attention outputs and LSE.
Small cases compare every (request, layer, KV head) unit; the full-size workloads compare a
seeded sample of units in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _libs():
    import torch
    import prefix_cached_paged_gb300 as rc
    from synth import device as sdev
    rc.lib()
    sdev.build()
    rc.device_status()  # clear
    yield
    torch.cuda.synchronize()


def _status_clear():
    import prefix_cached_paged_gb300 as rc
    assert rc.device_status() == 0


def _check_extend(w, batch, outs, seqs, units, lse_check=True):
    m = w.model
    qo = batch.plan.qo_indptr
    P = batch.plan.prefix_len
    worst = (0.0, 0.0)
    for (b, layer, kvh) in units:
        o_ref, lse_ref = H.oracle_unit(m, seqs[b], int(P[b]), layer, kvh)
        o, l = outs[layer]
        got = o[qo[b]:qo[b + 1], kvh * m.group:(kvh + 1) * m.group].float().cpu().numpy()
        ok, ma, rl = H.compare(got, o_ref, m.dtype)
        worst = (max(worst[0], ma), max(worst[1], rl))
        assert ok, f"unit {(b, layer, kvh)} P={P[b]} S={qo[b+1]-qo[b]}: max-abs {ma} rel {rl}"
        if lse_check and l is not None:
            gl = l[qo[b]:qo[b + 1], kvh * m.group:(kvh + 1) * m.group].cpu().numpy()
            assert np.max(np.abs(gl - lse_ref)) < (2e-3 if m.dtype == "bf16" else 1e-5)
    return worst


def _check_slot_rows(engine, batch):
    rows = engine.dev.req_to_token.cpu().numpy()
    for i, r in enumerate(batch.row_ids):
        L = int(batch.plan.lengths[i])
        np.testing.assert_array_equal(rows[r, :L], batch.plan.rows[i, :L])


def _check_scatter(engine, w, seqs, batch, sample=None):
    """Pool rows at the computed tokens' slots equal the generator's K/V values, bit for bit."""
    m = w.model
    hs = H.new_token_hashes(m, seqs, batch.plan.prefix_len)
    slots = batch.plan.out_loc
    idx = np.arange(len(slots)) if sample is None else sample
    for layer in range(m.layers):
        kk = engine.dev.k[layer][slots[idx]].cpu()
        vv = engine.dev.v[layer][slots[idx]].cpu()
        ek = synth.values_bits(hs[idx], synth.TENSOR_K, layer, range(m.n_kv_heads), m.head_dim,
                               m.dtype)
        ev = synth.values_bits(hs[idx], synth.TENSOR_V, layer, range(m.n_kv_heads), m.head_dim,
                               m.dtype)
        if m.dtype == "bf16":
            kk = kk.view(dtype=__import__("torch").int16).numpy().view(np.uint16)
            vv = vv.view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        else:
            kk, vv = kk.numpy(), vv.numpy()
        np.testing.assert_array_equal(kk, ek)
        np.testing.assert_array_equal(vv, ev)


def test_device_fill_matches_generator():
    import torch
    from synth import device as sdev
    h = synth.prefix_hashes(3, synth.tokens(3, 9, 300))
    hd = sdev.hashes_to_device(h)
    for dt, tdt in (("bf16", torch.bfloat16), ("f32", torch.float32)):
        out = torch.empty((300, 4, 128), dtype=tdt, device="cuda")
        sdev.fill_rows(hd, synth.TENSOR_V, 5, out, head0=2)
        exp = synth.values(h, synth.TENSOR_V, 5, range(2, 6), 128, dt)
        np.testing.assert_array_equal(out.float().cpu().numpy(), exp)


def test_tiny_extend_fp32_all_units():
    w = W.tiny_extend()
    eng = H.make_engine(w)
    skipped = 0
    for ph in w.phases:
        b, outs = H.run_extend_phase(eng, w.model, ph.seqs, lse=True)
        skipped += int(b.plan.prefix_len.sum())
        units = [(i, 0, h) for i in range(len(ph.seqs)) for h in range(w.model.n_kv_heads)]
        _check_extend(w, b, outs, ph.seqs, units)
        _check_slot_rows(eng, b)
        _check_scatter(eng, w, ph.seqs, b)
    assert skipped == 192
    _status_clear()


def _custom_extend(Hq, Hkv, pairs, seed=11, dtype="bf16"):
    """Requests with given (cached prefix P, new tokens S): phase 1 caches the prefixes, phase 2
    extends all requests in one batch."""
    m = W.Model(1, Hq, Hkv, 128, dtype, seed)
    pre, seqs = [], []
    for i, (P, S) in enumerate(pairs):
        p = synth.tokens(seed, 500 + i, P)
        s = synth.tokens(seed, 900 + i, S)
        if P:
            pre.append(p)
        seqs.append(np.concatenate([p, s]).astype(np.int32))
    L = max(len(s) for s in seqs)
    w = W.Workload("custom", m, 40_000, synth.permutation(seed, 40_000), max_ctx=(L + 15) // 16 * 16)
    w.phases = [W.Phase("cache", pre), W.Phase("extend", seqs)]
    return w


PAIRS = [(0, 1), (0, 130), (1, 1), (37, 64), (130, 129), (300, 7), (513, 200), (2, 257),
         (128, 128), (255, 1)]


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 2), (16, 4)])
def test_extend_bf16_ragged_all_units(Hq, Hkv):
    w = _custom_extend(Hq, Hkv, PAIRS)
    eng = H.make_engine(w)
    H.run_cache_phase(eng, w.model, w.phases[0].seqs)
    seqs = w.phases[1].seqs
    b, outs = H.run_extend_phase(eng, w.model, seqs, lse=True)
    assert b.plan.prefix_len.tolist() == [min(p, p + s - 1) for p, s in PAIRS]
    units = [(i, 0, h) for i in range(len(seqs)) for h in range(Hkv)]
    _check_extend(w, b, outs, seqs, units)
    _check_slot_rows(eng, b)
    _check_scatter(eng, w, seqs, b)
    _status_clear()


PAIRS_WIDE = [(0, 1), (37, 64), (130, 129), (2, 257), (255, 1)]


@pytest.mark.parametrize("Hq,Hkv", [(6, 2), (32, 2), (64, 2), (128, 2)])
def test_extend_bf16_group_sizes(Hq, Hkv):
    """Query tiles of 128 / G positions x G heads for G = 3 (42 positions, 126 rows; no lane
    shift, as 3 does not divide 32), 16 and 32 (ragged tiles start 2 and 1 positions early, at
    TMEM lane 32) and 64 (two positions per tile; no lane shift): every unit within tolerance."""
    w = _custom_extend(Hq, Hkv, PAIRS_WIDE, seed=13)
    eng = H.make_engine(w)
    H.run_cache_phase(eng, w.model, w.phases[0].seqs)
    seqs = w.phases[1].seqs
    b, outs = H.run_extend_phase(eng, w.model, seqs, lse=True)
    assert b.plan.prefix_len.tolist() == [min(p, p + s - 1) for p, s in PAIRS_WIDE]
    units = [(i, 0, h) for i in range(len(seqs)) for h in range(Hkv)]
    _check_extend(w, b, outs, seqs, units)
    _check_scatter(eng, w, seqs, b)
    _status_clear()


def _sample_units(rng, n_req, layers, n_kv, k):
    """k distinct (request, layer, KV head) units (all of them if there are fewer)."""
    k = min(k, n_req * layers * n_kv)
    units = set()
    while len(units) < k:
        units.add((int(rng.integers(n_req)), int(rng.integers(layers)), int(rng.integers(n_kv))))
    return sorted(units)


def test_few_shot_extend_full_size_sampled():
    w = W.few_shot_extend()
    eng = H.make_engine(w)
    H.run_extend_phase(eng, w.model, w.phases[0].seqs)   # warm: the prefix alone
    seqs = w.phases[1].seqs
    b, outs = H.run_extend_phase(eng, w.model, seqs, lse=True)
    assert int(b.plan.prefix_len.sum()) == 128_000 and b.num_tokens == 3200
    rng = np.random.default_rng(0)
    units = _sample_units(rng, 64, 1, 32, 96)
    assert len(units) >= 64
    _check_extend(w, b, outs, seqs, units)
    _check_slot_rows(eng, b)
    _check_scatter(eng, w, seqs, b)
    _status_clear()


def test_two_level_extend_full_size_sampled():
    w = W.two_level_extend()
    eng = H.make_engine(w)
    H.run_extend_phase(eng, w.model, w.phases[0].seqs)
    H.run_extend_phase(eng, w.model, w.phases[1].seqs)
    seqs = w.phases[2].seqs
    b, outs = H.run_extend_phase(eng, w.model, seqs, lse=True)
    v = w.notes["v"]
    assert b.plan.prefix_len.tolist() == [1000 + v[i // 4] for i in range(64)]
    rng = np.random.default_rng(1)
    units = _sample_units(rng, 64, 1, 8, 96)
    assert len(units) >= 64
    _check_extend(w, b, outs, seqs, units)
    _check_slot_rows(eng, b)
    _check_scatter(eng, w, seqs, b)
    _status_clear()


def _check_decode(w, db, outs, seqs, units):
    m = w.model
    for (b, layer, kvh) in units:
        s = seqs[b]
        o_ref, lse_ref = H.oracle_unit(m, s, len(s) - 1, layer, kvh)
        o, l = outs[layer]
        got = o[b, kvh * m.group:(kvh + 1) * m.group].float().cpu().numpy()[None]
        ok, ma, rl = H.compare(got, o_ref, m.dtype)
        assert ok, f"decode unit {(b, layer, kvh)} L={len(s)}: max-abs {ma} rel {rl}"
        if l is not None:
            gl = l[b, kvh * m.group:(kvh + 1) * m.group].cpu().numpy()
            assert np.max(np.abs(gl - lse_ref[0])) < (2e-3 if m.dtype == "bf16" else 1e-5)


def _decode_scatter(eng, w, seqs, db):
    m = w.model
    h = np.array([synth.prefix_hashes(m.seed, s)[-1] for s in seqs], dtype=np.uint64)
    for layer in range(m.layers):
        for plane, tensor in ((eng.dev.k, synth.TENSOR_K), (eng.dev.v, synth.TENSOR_V)):
            got = plane[layer][db.new_slots].float().cpu().numpy()
            np.testing.assert_array_equal(
                got, synth.values(h, tensor, layer, range(m.n_kv_heads), m.head_dim, m.dtype))


@pytest.mark.parametrize("chunk", [0, 64, 192, 4096])
def test_decode_small_all_units(chunk):
    L = [1, 2, 63, 64, 65, 191, 192, 193, 700, 1500, 3000, 129]
    m = W.Model(1, 32, 8, 128, "bf16", 5)
    seqs = [synth.tokens(5, 40 + i, n) for i, n in enumerate(L)]
    w = W.Workload("dec_small", m, 20_000, synth.permutation(5, 20_000), max_ctx=3008)
    eng = H.make_engine(w, max_reqs=32, kv_chunk=chunk)
    H.run_cache_phase(eng, m, [s[:-1] for s in seqs if len(s) > 1])
    db, outs = H.run_decode(eng, m, seqs, lse=True)
    _check_decode(w, db, outs, seqs, [(i, 0, h) for i in range(len(L)) for h in range(8)])
    _decode_scatter(eng, w, seqs, db)
    _status_clear()


@pytest.mark.parametrize("Hq,Hkv,dtype,d", [(8, 8, "bf16", 128), (16, 2, "bf16", 128),
                                            (8, 1, "bf16", 64), (4, 4, "f32", 128),
                                            (4, 2, "f32", 64)])
def test_decode_group_and_dtype_variants(Hq, Hkv, dtype, d):
    L = [5, 300, 1030]
    m = W.Model(2, Hq, Hkv, d, dtype, 6)
    seqs = [synth.tokens(6, 60 + i, n) for i, n in enumerate(L)]
    w = W.Workload("dec_var", m, 4000, None, max_ctx=1040)
    eng = H.make_engine(w, max_reqs=8, kv_chunk=256)
    H.run_cache_phase(eng, m, [s[:-1] for s in seqs])
    db, outs = H.run_decode(eng, m, seqs, lse=True)
    _check_decode(w, db, outs, seqs, [(i, l, h) for i in range(3) for l in range(2)
                                      for h in range(Hkv)])
    _status_clear()


def test_multi_turn_decode_full_size_sampled():
    w = W.multi_turn_decode()
    eng = H.make_engine(w, max_reqs=264)
    H.run_cache_phase(eng, w.model, w.phases[0].seqs)
    seqs = w.phases[1].seqs
    db, outs = H.run_decode(eng, w.model, seqs, lse=True)
    rng = np.random.default_rng(2)
    units = _sample_units(rng, 256, 1, 8, 80)
    # always include the longest and the shortest request
    Ls = np.array([len(s) for s in seqs])
    units += [(int(Ls.argmax()), 0, 3), (int(Ls.argmin()), 0, 5)]
    _check_decode(w, db, outs, seqs, units)
    _decode_scatter(eng, w, seqs, db)
    _status_clear()


def test_multi_turn_decode_unshared_twin_sampled():
    w0 = W.multi_turn_decode()
    w = W.multi_turn_decode(shared=False, lengths=w0.notes["lengths"])
    eng = H.make_engine(w, max_reqs=264)
    H.run_cache_phase(eng, w.model, w.phases[0].seqs)
    seqs = w.phases[1].seqs
    db, outs = H.run_decode(eng, w.model, seqs)
    rng = np.random.default_rng(3)
    _check_decode(w, db, outs, seqs, _sample_units(rng, 256, 1, 8, 72))
    _status_clear()


# ---------------------------------------------------------------- decode over shared contexts
def _families(seed, spec):
    """Requests in families: family f has a shared prefix of spec[f][0] tokens and one member per
    entry of spec[f][1], whose own tokens follow (the decode token is the last one)."""
    seqs = []
    for f, (ls, owns) in enumerate(spec):
        shared = synth.tokens(seed, 500 + f, ls)
        for i, lo in enumerate(owns):
            own = synth.tokens(seed, 900 + 37 * f + i, lo)
            seqs.append(np.concatenate([shared, own]).astype(np.int32))
    return seqs


_FAMILY_SPEC = [(700, [1, 5, 300]), (1300, [2, 2, 2, 2, 2, 2, 2, 2, 9]), (64, [3, 40]),
                (2100, [1, 700]), (40, [30]), (1030, [1])]


@pytest.mark.parametrize("Hq,Hkv,d,chunk,dtype", [(8, 8, 128, 0, "bf16"), (8, 8, 128, 64, "bf16"),
                                                  (16, 8, 64, 256, "bf16"),
                                                  (16, 4, 128, 192, "bf16"),
                                                  (16, 2, 128, 0, "bf16"), (4, 4, 128, 64, "f32")])
def test_decode_shared_context_groups(Hq, Hkv, d, chunk, dtype):
    """Groups of requests over a shared prefix: the stacked kernel matches the oracle, and it is
    bit-identical to decoding every request on its own (stacking changes no arithmetic)."""
    import torch
    m = W.Model(1, Hq, Hkv, d, dtype, 8)
    seqs = _families(8, _FAMILY_SPEC)
    w = W.Workload("dec_shared", m, 20_000, synth.permutation(8, 20_000), max_ctx=2816)
    runs = {}
    for share in (True, False):
        eng = H.make_engine(w, max_reqs=32, kv_chunk=chunk, share_decode=share)
        H.run_cache_phase(eng, m, [s[:-1] for s in seqs])
        db, o = H.run_decode(eng, m, seqs, lse=True)
        runs[share] = (eng, db, o)
        _status_clear()
    eng, db, o = runs[True]
    # groups form wherever a KV head's query heads leave room for two requests in a tile
    assert (db.num_groups > 0) == (8 // (Hq // Hkv) >= 2)
    _check_decode(w, db, o, seqs, [(i, 0, h) for i in range(len(seqs)) for h in range(Hkv)])
    _decode_scatter(eng, w, seqs, db)
    (og, lg), (ou, lu) = o[0], runs[False][2][0]
    assert torch.equal(og, ou) and torch.equal(lg, lu)


def test_decode_group_contract_breaches_are_reported():
    """A request in two groups, or a shared length past a member's context, is reported through
    the device status word; every access stays in range."""
    import prefix_cached_paged_gb300 as rc
    m = W.Model(1, 8, 8, 128, "bf16", 9)
    seqs = _families(9, [(600, [3, 4, 5])])
    w = W.Workload("dec_breach", m, 4000, None, max_ctx=640)
    eng = H.make_engine(w, max_reqs=8, kv_chunk=64, share_decode=False)
    H.run_cache_phase(eng, m, [s[:-1] for s in seqs])
    db, _ = H.run_decode(eng, m, seqs)
    _status_clear()
    from synth import device as sdev
    import torch
    h = np.array([synth.prefix_hashes(m.seed, s)[-1] for s in seqs], dtype=np.uint64)
    q, k, v = H.dense_qkv(m, sdev.hashes_to_device(h), 0, len(seqs))
    o = torch.empty_like(q)
    mt = int(db.seq_len.sum())
    ws = eng.workspace(q, k, mt)
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    bad = [((dev([0, 2, 4]), dev([0, 1, 1, 2]), dev([512, 512]))),     # request 1 twice
           ((dev([0, 3]), dev([0, 1, 2]), dev([int(db.seq_len.max())])))]  # shared past a context
    for groups in bad:
        rc.decode_attention(q, k, v, db.dev_out_loc, db.dev_seq_len, db.dev_req_idx,
                            eng.dev.req_to_token, eng.dev.k[0], eng.dev.v[0], o, ws,
                            sm_scale=eng.sm_scale, max_total_tokens=mt, kv_chunk=64,
                            groups=groups)
        torch.cuda.synchronize()
        assert rc.device_status() != 0


# ---------------------------------------------------------------- extend: prefix stacking (E3b)
def _stack_families(seed, spec):
    """Consecutive requests per family: family f shares spec[f][0] cached tokens; member i adds
    spec[f][1][i] = (private cached tokens, new tokens). Returns (cache seqs, extend seqs)."""
    cache, ext = [], []
    for f, (ls, mem) in enumerate(spec):
        shared = synth.tokens(seed, 700 + f, ls)
        cache.append(shared)
        for i, (priv, new) in enumerate(mem):
            own = synth.tokens(seed, 1200 + 31 * f + i, priv + new)
            full = np.concatenate([shared, own]).astype(np.int32)
            if priv:
                cache.append(full[:ls + priv])
            ext.append(full)
    return cache, ext


_STACK_SPEC = [(700, [(0, 40), (0, 1), (30, 200), (0, 130)]),   # private parts, long and 1-row
               (300, [(0, 5), (0, 7)]),                          # stacked tile in split mode
               (2000, [(0, 50)] * 6),                            # few-shot like
               (100, [(0, 20), (0, 20)]),                        # shared below the threshold
               (900, [(5, 60)])]                                 # alone


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 2), (16, 8)])
def test_extend_prefix_stacking(Hq, Hkv):
    """Stacked prefix pass + per-request pass with merge: every unit within tolerance of the
    oracle, and the engine without stacking too."""
    m = W.Model(1, Hq, Hkv, 128, "bf16", 11)
    cache, ext = _stack_families(11, _STACK_SPEC)
    w = W.Workload("ext_stack", m, 40_000, synth.permutation(11, 40_000), max_ctx=3008)
    for stack in (True, False):
        eng = H.make_engine(w, max_reqs=64, stack_extend="always" if stack else False)
        for c in cache:
            H.run_cache_phase(eng, m, [c])
        b, outs = H.run_extend_phase(eng, m, ext, lse=True)
        if stack:
            assert b.stack is not None and int(b.stack[1].numel()) == 3   # three stacked groups
        _status_clear()
        units = [(i, 0, h) for i in range(len(ext)) for h in range(Hkv)]
        _check_extend(w, b, outs, ext, units)


def test_extend_stacking_contract_breach_is_reported():
    """A shared length past a member's matched prefix is reported through the status word."""
    import torch
    import prefix_cached_paged_gb300 as rc
    from synth import device as sdev
    m = W.Model(1, 8, 8, 128, "bf16", 12)
    cache, ext = _stack_families(12, [(600, [(0, 30), (0, 40)])])
    w = W.Workload("ext_breach", m, 4000, None, max_ctx=704)
    eng = H.make_engine(w, max_reqs=8, stack_extend=False)
    for c in cache:
        H.run_cache_phase(eng, m, [c])
    b = eng.extend_begin(ext)
    h = H.new_token_hashes(m, ext, b.plan.prefix_len)
    q, k, v = H.dense_qkv(m, sdev.hashes_to_device(h), 0, b.num_tokens)
    o = torch.empty_like(q)
    ws = torch.empty(rc.extend_workspace_bytes(b.num_tokens, m.n_q_heads), dtype=torch.uint8,
                     device="cuda")
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    stack = (dev([0, 2]), dev([650]), 70)      # 650 > the matched prefix of 600
    rc.extend_attention(q, k, v, b.out_loc, b.qo_indptr, b.prefix_len, b.req_idx,
                        eng.dev.req_to_token, eng.dev.k[0], eng.dev.v[0], o,
                        sm_scale=eng.sm_scale, max_q_len=b.max_q_len,
                        max_prefix_len=b.max_prefix_len, stack=stack, workspace=ws)
    torch.cuda.synchronize()
    assert rc.device_status() != 0
    eng.extend_end(b)


@pytest.mark.parametrize("policy", ["lspf", "fcfs"])
def test_program_queue_served_by_the_scheduler(policy):
    """The program queue (small) served batch by batch: rc_schedule_batch picks each batch, the
    extend kernel computes it over slots that eviction keeps recycling; every batch's sampled
    outputs match the oracle, its slot rows and scattered K/V are exact."""
    import torch
    import prefix_cached_paged_gb300 as rc
    from synth import device as sdev
    pq = W.program_queue(n_programs=6, prefix_len=200, n_questions=4, question_len=20,
                         pool_slots=700, max_batch=8, max_new_tokens=1200)
    w = pq.workload
    eng = H.make_engine(w, max_reqs=pq.max_batch + 8)
    pol = rc.RC_SCHED_LSPF if policy == "lspf" else rc.RC_SCHED_FCFS
    waiting = list(range(len(pq.seqs)))
    rng = np.random.default_rng(3)
    batches = evicted = 0
    while waiting:
        idx = eng.host.schedule([pq.seqs[i] for i in waiting], pq.max_batch, pq.max_new_tokens,
                                policy=pol)
        assert idx
        seqs = [pq.seqs[waiting[i]] for i in idx]
        b = eng.extend_begin(seqs)
        evicted += int(b.plan.evicted)
        h = H.new_token_hashes(w.model, seqs, b.plan.prefix_len)
        q, k, v = H.dense_qkv(w.model, sdev.hashes_to_device(h), 0, b.num_tokens)
        o = torch.empty_like(q)
        eng.extend_layer(b, 0, q, k, v, o)
        _check_extend(w, b, {0: (o, None)}, seqs, _sample_units(rng, len(seqs), 1, 32, 6))
        _check_slot_rows(eng, b)
        _check_scatter(eng, w, seqs, b, sample=rng.choice(b.num_tokens, 32, replace=False))
        eng.extend_end(b)
        for i in sorted(idx, reverse=True):
            waiting.pop(i)
        batches += 1
    assert evicted > 0 and batches > 2
    _status_clear()


@pytest.mark.parametrize("dtype,Hkv,d,layers", [("bf16", 4, 128, 3), ("f32", 2, 64, 2)])
def test_kv_copy_round_trip_through_pinned_host(dtype, Hkv, d, layers):
    """rc_kv_copy device -> pinned host -> device at scattered slots: every row bit-exact, rows
    not named untouched; an out-of-range slot is reported, not written."""
    import torch
    import prefix_cached_paged_gb300 as rc
    dt = H.torch_dtype(dtype)
    g = torch.Generator(device="cuda").manual_seed(5)
    N, NH, n = 3000, 2000, 777
    dk = torch.randn((layers, N, Hkv, d), device="cuda", generator=g).to(dt)
    dv = torch.randn((layers, N, Hkv, d), device="cuda", generator=g).to(dt)
    hk = torch.zeros((layers, NH, Hkv, d), dtype=dt).pin_memory()
    hv = torch.zeros((layers, NH, Hkv, d), dtype=dt).pin_memory()
    rng = np.random.default_rng(2)
    src = rng.choice(N, n, replace=False).astype(np.int32)
    hst = rng.choice(NH, n, replace=False).astype(np.int32)
    dst = rng.choice(N, n, replace=False).astype(np.int32)
    S, Hs, D = (torch.from_numpy(a).cuda() for a in (src, hst, dst))
    rc.kv_copy(dk, dv, S, hk, hv, Hs)
    ek, ev = dk.clone(), dv.clone()
    out_k = torch.zeros_like(dk)
    out_v = torch.zeros_like(dv)
    rc.kv_copy(hk, hv, Hs, out_k, out_v, D)
    torch.cuda.synchronize()
    assert torch.equal(hk[:, torch.from_numpy(hst).long()], ek[:, torch.from_numpy(src).long()].cpu())
    assert torch.equal(out_k[:, D.long()], ek[:, S.long()])
    assert torch.equal(out_v[:, D.long()], ev[:, S.long()])
    untouched = np.setdiff1d(np.arange(N), dst)
    assert int(out_k[:, torch.from_numpy(untouched).cuda().long()].abs().sum()) == 0
    _status_clear()
    bad = torch.tensor([0, N], dtype=torch.int32, device="cuda")
    ok = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    rc.kv_copy(dk, dv, bad, hk, hv, ok)
    assert rc.device_status() == 1      # slot out of range, reported and skipped


@pytest.mark.parametrize("policy", ["fcfs", "lspf"])
def test_program_queue_with_host_tier(policy):
    """The small program queue behind a 700-slot device pool and a host tier: each batch's
    matches, loads and copies equal the oracle's; reloaded slots hold the generator's K/V bit for
    bit; sampled outputs match the oracle."""
    import torch
    import prefix_cached_paged_gb300 as rc
    from synth import device as sdev
    pq = W.program_queue(n_programs=6, prefix_len=200, n_questions=4, question_len=20,
                         pool_slots=700, max_batch=8, max_new_tokens=1200, layers=2)
    w = pq.workload
    eng = H.make_engine(w, max_reqs=pq.max_batch + 8, host_tier_slots=2000)
    sim = oracle.CacheSim(w.pool_slots, w.pool_order, host_slots=2000)
    fcfs = policy == "fcfs"
    waiting = list(range(len(pq.seqs)))
    rng = np.random.default_rng(4)
    loaded = 0
    while waiting:
        seqs_w = [pq.seqs[i] for i in waiting]
        idx = eng.host.schedule(seqs_w, pq.max_batch, pq.max_new_tokens,
                                policy=rc.RC_SCHED_FCFS if fcfs else rc.RC_SCHED_LSPF)
        order, _, adm = oracle.schedule_batch(sim.tree, seqs_w, [len(s) - 1 for s in seqs_w],
                                              fcfs, pq.max_batch, pq.max_new_tokens)
        assert idx == order[:adm]
        seqs = [pq.seqs[waiting[i]] for i in idx]
        res = sim.extend_prepare(seqs)
        b = eng.extend_begin(seqs)
        assert b.plan.prefix_len.tolist() == res.prefix_len
        assert b.plan.host_len.tolist() == res.host_len
        for x, y in zip(b.plan.copies, res.copies):
            assert x.tolist() == y.tolist()
        loaded += int(b.plan.host_len.sum())
        h = H.new_token_hashes(w.model, seqs, b.plan.prefix_len)
        hd = sdev.hashes_to_device(h)
        outs = {}
        for layer in range(w.model.layers):
            q, k, v = H.dense_qkv(w.model, hd, layer, b.num_tokens)
            o = torch.empty_like(q)
            eng.extend_layer(b, layer, q, k, v, o)
            outs[layer] = (o, None)
        _check_extend(w, b, outs, seqs, _sample_units(rng, len(seqs), w.model.layers, 32, 6))
        _check_slot_rows(eng, b)
        # the slots just loaded back hold each token's own K/V in every layer
        for i, s in enumerate(seqs):
            hl = int(b.plan.host_len[i])
            if hl:
                p = int(b.plan.prefix_len[i])
                slots = b.plan.rows[i, p - hl:p]
                hs = synth.prefix_hashes(w.model.seed, s)[p - hl:p]
                for layer in range(w.model.layers):
                    got = eng.dev.k[layer][torch.from_numpy(slots).long().cuda()].cpu()
                    want = synth.values_bits(hs, synth.TENSOR_K, layer, range(w.model.n_kv_heads),
                                             w.model.head_dim, w.model.dtype)
                    np.testing.assert_array_equal(
                        got.view(torch.int16).numpy().view(np.uint16), want)
        eng.extend_end(b)
        sim.extend_finish(seqs, res)
        for i in sorted(idx, reverse=True):
            waiting.pop(i)
    if fcfs:
        assert loaded > 0
    _status_clear()


def _tree_families(seed, root, branches, leaves, news):
    """A three-level family: `root` tokens shared by all requests; `branches` branches add their
    own cached tokens; each branch holds `leaves` leaf groups adding more; each leaf group has
    one request per entry of `news` (its new tokens). Returns (cache seqs, extend seqs)."""
    r = synth.tokens(seed, 900, root)
    cache, ext = [r], []
    for bi, bl in enumerate(branches):
        b = np.concatenate([r, synth.tokens(seed, 910 + bi, bl)])
        cache.append(b)
        for li, ll in enumerate(leaves):
            lf = np.concatenate([b, synth.tokens(seed, 950 + 10 * bi + li, ll)])
            cache.append(lf)
            for k, n in enumerate(news):
                own = synth.tokens(seed, 2000 + 100 * bi + 10 * li + k, n)
                ext.append(np.concatenate([lf, own]).astype(np.int32))
    return cache, ext


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
def test_extend_prefix_stacking_cascade(Hq, Hkv):
    """Stacking over three tree levels (root shared by all, branches, leaf groups): each deeper
    level's stacked pass covers only its own keys and merges into the partial above; every unit
    within tolerance of the oracle."""
    m = W.Model(1, Hq, Hkv, 128, "bf16", 12)
    cache, ext = _tree_families(12, 600, [300, 280], [260, 300], [1, 17, 40])
    w = W.Workload("ext_cascade", m, 40_000, synth.permutation(12, 40_000), max_ctx=2048)
    eng = H.make_engine(w, max_reqs=64, stack_extend="always")
    for c in cache:
        H.run_cache_phase(eng, m, [c])
    b, outs = H.run_extend_phase(eng, m, ext, lse=True)
    assert b.stack is not None
    shared, start, level_indptr, fold, all_folded = (b.stack[1], b.stack[3], b.stack[4],
                                                     b.stack[5], b.stack[6])
    assert level_indptr.tolist() == [0, 1, 3, 7]          # 1 root, 2 branch, 4 leaf groups
    assert start.cpu().tolist() == [0, 600, 600, 900, 900, 880, 880]
    # the leaf groups take their members' remainders; no per-request pass is left
    assert fold.cpu().tolist() == [0, 0, 0, 1, 1, 1, 1] and all_folded
    _status_clear()
    units = [(i, 0, h) for i in range(len(ext)) for h in range(Hkv)]
    _check_extend(w, b, outs, ext, units)


@pytest.mark.parametrize("groups", [False, True])
def test_decode_plan_reuse_across_layers(groups):
    """The layers of a decode step reuse the first layer's plan (job list; the main kernel leaves
    its item counter reset): every layer's output and LSE are bit-identical to a call that plans
    afresh, and within tolerance of the oracle."""
    import torch
    import prefix_cached_paged_gb300 as rc
    L = [70, 600, 1500, 1501, 2900, 3000, 513, 64]
    m = W.Model(3, 16, 4, 128, "bf16", 6)
    base = synth.tokens(6, 77, 2000)
    seqs = [np.concatenate([base[:min(n, 1700)], synth.tokens(6, 80 + i, max(n - 1700, 0))])
            .astype(np.int32)[:n] for i, n in enumerate(L)]
    w = W.Workload("dec_reuse", m, 30_000, synth.permutation(6, 30_000), max_ctx=3008)
    eng = H.make_engine(w, max_reqs=32, kv_chunk=256, share_decode=groups)
    H.run_cache_phase(eng, m, [s[:-1] for s in seqs])
    db, outs = H.run_decode(eng, m, seqs, lse=True)
    assert (db.num_groups > 0) == groups
    h = np.array([synth.prefix_hashes(m.seed, s)[-1] for s in seqs], dtype=np.uint64)
    from synth import device as sdev
    hd = sdev.hashes_to_device(h)
    mt = int(db.seq_len.sum())
    for layer in range(m.layers):
        q, k, v = H.dense_qkv(m, hd, layer, len(seqs))
        o = torch.empty_like(q)
        lse = torch.empty((len(seqs), m.n_q_heads), dtype=torch.float32, device="cuda")
        ws = torch.empty(rc.decode_workspace_bytes(q, k, eng.dev.req_to_token, eng.dev.k[0],
                                                   max_total_tokens=mt, kv_chunk=256),
                         dtype=torch.uint8, device="cuda")
        rc.decode_attention(q, k, v, db.dev_out_loc, db.dev_seq_len, db.dev_req_idx,
                            eng.dev.req_to_token, eng.dev.k[layer], eng.dev.v[layer], o, ws,
                            sm_scale=eng.sm_scale, max_total_tokens=mt, kv_chunk=256, lse=lse,
                            groups=db.groups)
        assert torch.equal(o, outs[layer][0]), layer
        assert torch.equal(lse, outs[layer][1]), layer
    _check_decode(w, db, outs, seqs, [(i, l, hh) for i in range(len(L)) for l in range(3)
                                      for hh in range(4)])
    _status_clear()


_FOLD_SPEC = [(600, [(20, 30), (50, 60), (0, 128), (100, 1)]),   # private cached keys, a full tile
              (300, [(0, 5)] * 7),                                # few-shot like
              (900, [(10, 100), (0, 200)]),                       # remainders of 1 and 2 tiles
              (400, [(0, 200)] * 5),                              # forks: 1000 stacked rows
              (260, [(140, 190), (3, 260)])]                      # 3 remainder tiles


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 2), (16, 8)])
def test_extend_fold(Hq, Hkv):
    """Folded stacked passes (each member's remainder -- its own cached tokens past the shared
    prefix, then its new tokens, in as many key tiles as it takes -- in the group's pass, final
    outputs written there): all groups folded, the cost model's choice (folded and unfolded
    groups side by side), and none folded; every unit within tolerance of the oracle, the new
    K/V scattered bit-exactly."""
    m = W.Model(1, Hq, Hkv, 128, "bf16", 13)
    cache, ext = _stack_families(13, _FOLD_SPEC)
    w = W.Workload("ext_fold", m, 40_000, synth.permutation(13, 40_000), max_ctx=1216)
    for fold in ("always", True, False):
        eng = H.make_engine(w, max_reqs=64, stack_extend="always", fold_extend=fold)
        for c in cache:
            H.run_cache_phase(eng, m, [c])
        b, outs = H.run_extend_phase(eng, m, ext, lse=True)
        assert b.stack is not None
        flags = b.stack[5].cpu().tolist()
        if fold == "always":
            assert flags == [1] * len(_FOLD_SPEC) and b.stack[6]
        elif not fold:
            assert flags == [0] * len(_FOLD_SPEC) and not b.stack[6]
        _status_clear()
        units = [(i, 0, h) for i in range(len(ext)) for h in range(Hkv)]
        _check_extend(w, b, outs, ext, units)
        _check_slot_rows(eng, b)
        _check_scatter(eng, w, ext, b)



def test_fork_mixed_step_full_size_sampled():
    """The fork / self-consistency mixed step at full size (300k-slot pool kept full so that LRU
    eviction runs, 80 extend sequences of 1500 cached + 200 new tokens, 128 decode requests over
    512..8192-token contexts in fork groups) in the benchmark's launch configuration, on two of
    its 32 layers (every layer launches the same kernels): two consecutive steps, each checking
    a seeded sample of extend and decode units against the oracle, the slot rows and the
    scattered K/V (extend and decode). Decode inputs at step s come from each request's real s-th
    generated token."""
    import torch
    from synth import device as sdev
    fm = W.fork_mixed_step(layers=2)
    w = fm.workload
    m = w.model
    Bd = len(fm.decode_seqs)
    eng = H.make_engine(w, max_reqs=Bd + 80 + 8)
    for ph in w.phases:
        H.run_cache_phase(eng, m, ph.seqs, keep_locked=False)
    db = eng.decode_begin([s[:-1] for s in fm.decode_seqs])
    assert eng.host.pool.available() == 4096
    mt = int(db.seq_len.sum()) + Bd * 3
    rng = np.random.default_rng(11)
    for step in range(2):
        seqs = fm.extend_seqs(step)
        eb = eng.extend_begin(seqs, extra=Bd)
        eng.decode_step(db, new_slots=eb.plan.extra)
        assert eb.plan.prefix_len.tolist() == [1500] * 80 and eb.num_tokens == 16_000
        # the pool is full: LRU eviction makes room every step (4096 slots free at the first)
        assert eb.plan.evicted >= (16_000 + Bd - 4096 if step == 0 else 1)
        h_ext = sdev.hashes_to_device(H.new_token_hashes(m, seqs, eb.plan.prefix_len))
        dseqs = fm.decode_step_seqs(step)
        h_dec = sdev.hashes_to_device(
            np.array([synth.prefix_hashes(m.seed, s)[-1] for s in dseqs], np.uint64))
        ext_outs, dec_outs = {}, {}
        for layer in range(m.layers):
            q, k, v = H.dense_qkv(m, h_ext, layer, eb.num_tokens)
            o = torch.empty_like(q)
            l = torch.empty((eb.num_tokens, m.n_q_heads), dtype=torch.float32, device="cuda")
            eng.extend_layer(eb, layer, q, k, v, o, lse=l)
            ext_outs[layer] = (o, l)
            dq, dk, dv = H.dense_qkv(m, h_dec, layer, Bd)
            do = torch.empty_like(dq)
            dl = torch.empty((Bd, m.n_q_heads), dtype=torch.float32, device="cuda")
            eng.decode_layer(db, layer, dq, dk, dv, do, lse=dl, max_total_tokens=mt)
            dec_outs[layer] = (do, dl)
        torch.cuda.synchronize()
        # at least 64 sampled (request, layer, head) units per kernel and step
        _check_extend(w, eb, ext_outs, seqs, _sample_units(rng, 80, 2, 32, 64))
        _check_decode(w, db, dec_outs, dseqs, _sample_units(rng, Bd, 2, 32, 64) +
                      [(int(np.argmax([len(s) for s in dseqs])), 1, 7)])
        _check_slot_rows(eng, eb)
        _check_scatter(eng, w, seqs, eb, sample=rng.choice(eb.num_tokens, 256, replace=False))
        _decode_scatter(eng, w, dseqs, db)
        eng.extend_end(eb)
    _status_clear()
