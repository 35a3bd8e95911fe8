"""Pins for the oracle's fp64 attention and state merge (CPU only).

Each check is fixed by mathematics or the pages, not by re-typing the oracle's formula:
  * a hand-derived two-key example (golden fixture);
  * q = 0 makes every score equal, so each output is the plain mean of the values at positions
    <= the query's (catches causal off-by-one and dropped terms);
  * GQA head grouping: query head h reads kv head h // (Hq / Hkv) (values constant per kv head);
  * a dominant key makes the output that key's value;
  * key order does not matter for the last query (a joint permutation of K and V rows);
  * merging partial states over any partition of the keys equals the unsplit result;
  * the reuse invariant (paper digest App. A.1): attention computed with the prefix KV fetched
    from the slots a radix-tree match returns equals a from-scratch full causal prefill.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_two_key_golden():
    g = json.load(open(os.path.join(GOLDEN, "attention_two_keys.json")))
    q = np.array(g["q"]).reshape(1, 1, 2)
    k = np.array(g["k"]).reshape(2, 1, 2)
    v = np.array(g["v"]).reshape(2, 1, 2)
    o, lse = oracle.attention(q, k, v, P=1, scale=1.0, n_q_heads=1, n_kv_heads=1)
    np.testing.assert_allclose(o[0, 0], g["expected_o"], rtol=0, atol=1e-14)
    assert abs(lse[0, 0] - g["expected_lse"]) < 1e-14


@pytest.mark.parametrize("P,S", [(0, 1), (0, 7), (5, 3), (11, 1)])
def test_zero_query_is_causal_mean(P, S):
    rng = np.random.default_rng(P * 10 + S)
    Hq, Hkv, d = 4, 2, 8
    q = np.zeros((S, Hq, d))
    k = rng.standard_normal((P + S, Hkv, d))
    v = rng.standard_normal((P + S, Hkv, d))
    o, lse = oracle.attention(q, k, v, P, 0.3, Hq, Hkv)
    for i in range(S):
        for h in range(Hq):
            np.testing.assert_allclose(o[i, h], v[: P + i + 1, h // 2].mean(axis=0), atol=1e-13)
            assert abs(lse[i, h] - np.log(P + i + 1)) < 1e-13


def test_gqa_grouping_is_contiguous():
    Hq, Hkv, d, L = 8, 2, 4, 6
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, Hq, d))
    k = rng.standard_normal((L, Hkv, d))
    v = np.zeros((L, Hkv, d))
    v[:, 1, :] = 1.0
    o, _ = oracle.attention(q, k, v, L - 1, 0.5, Hq, Hkv)
    np.testing.assert_allclose(o[0, :4], 0.0, atol=1e-15)
    np.testing.assert_allclose(o[0, 4:], 1.0, atol=1e-13)


def test_dominant_key_selects_its_value():
    d, L = 4, 9
    rng = np.random.default_rng(2)
    k = rng.standard_normal((L, 1, d)) * 0.01
    k[3, 0] = [1.0, 0, 0, 0]
    q = np.array([[[60.0, 0, 0, 0]]])
    v = rng.standard_normal((L, 1, d))
    o, _ = oracle.attention(q, k, v, L - 1, 1.0, 1, 1)
    np.testing.assert_allclose(o[0, 0], v[3, 0], atol=1e-20 + 1e-12)


def test_key_permutation_invariance_for_last_query():
    rng = np.random.default_rng(3)
    L, Hq, Hkv, d = 13, 2, 1, 8
    q = rng.standard_normal((1, Hq, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    perm = rng.permutation(L)
    o1, l1 = oracle.attention(q, k, v, L - 1, 0.4, Hq, Hkv)
    o2, l2 = oracle.attention(q, k[perm], v[perm], L - 1, 0.4, Hq, Hkv)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("cuts", [[20], [1, 2], [3, 8, 15], [5, 6, 7, 19]])
def test_merge_of_any_partition_equals_unsplit(cuts):
    rng = np.random.default_rng(len(cuts))
    L, d = 21, 16
    q = rng.standard_normal((1, 1, d)) * 2
    k = rng.standard_normal((L, 1, d))
    v = rng.standard_normal((L, 1, d))
    full, lfull = oracle.attention(q, k, v, L - 1, 0.7, 1, 1)
    bounds = [0] + cuts + [L]
    parts, lses = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, l = oracle.attention(q, k[a:b], v[a:b], b - a - 1, 0.7, 1, 1)
        parts.append(o[0, 0])
        lses.append(l[0, 0])
    mo, ml = oracle.merge(np.array(parts), np.array(lses))
    np.testing.assert_allclose(mo, full[0, 0], atol=1e-13)
    assert abs(ml - lfull[0, 0]) < 1e-13
    # one part: merge is the identity
    mo1, ml1 = oracle.merge(full[0], lfull[0])
    np.testing.assert_allclose(mo1, full[0, 0], atol=0)


def _qkv(model, seq, layer=0):
    h = synth.prefix_hashes(model.seed, seq)
    hq = range(model.n_q_heads)
    hk = range(model.n_kv_heads)
    d = model.head_dim
    return (synth.values(h, synth.TENSOR_Q, layer, hq, d, model.dtype),
            synth.values(h, synth.TENSOR_K, layer, hk, d, model.dtype),
            synth.values(h, synth.TENSOR_V, layer, hk, d, model.dtype))


def test_reused_prefix_equals_from_scratch_prefill():
    """tiny_extend: request 1 prefills 80 tokens and writes its KV to its slots; requests 2-4
    fetch their 64-token prefix KV from the slots a match returns and compute only the suffix.
    Their outputs equal a full causal prefill of each whole sequence to fp64 round-off."""
    w = W.tiny_extend()
    m = w.model
    sim = oracle.CacheSim(w.pool_slots, w.pool_order)
    store_k = np.full((w.pool_slots, m.n_kv_heads, m.head_dim), np.nan)
    store_v = np.full_like(store_k, np.nan)
    for ph in w.phases:
        res = sim.extend_prepare(ph.seqs)
        for seq, P, row in zip(ph.seqs, res.prefix_len, res.rows):
            q, k, v = _qkv(m, seq)
            # reuse: prefix KV comes from the pool slots the tree handed back
            k_use = np.concatenate([store_k[row[:P]], k[P:]])
            v_use = np.concatenate([store_v[row[:P]], v[P:]])
            assert not np.isnan(k_use).any()
            o, lse = oracle.attention(q[P:], k_use, v_use, P, m.sm_scale, m.n_q_heads,
                                      m.n_kv_heads)
            full, lfull = oracle.attention(q, k, v, 0, m.sm_scale, m.n_q_heads, m.n_kv_heads)
            assert np.max(np.abs(o - full[P:])) <= 1e-12
            assert np.max(np.abs(lse - lfull[P:])) <= 1e-12
            # write the computed suffix KV to the request's own new slots
            store_k[row[P:]] = k[P:]
            store_v[row[P:]] = v[P:]
        sim.extend_finish(ph.seqs, res)
    assert res.prefix_len == [64, 64, 64]
