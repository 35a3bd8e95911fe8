"""Runs the seeded workloads through the product path (librc via serving.Engine) and computes the
oracle's results for the same requests. Shared by the GPU tests, the smoke check and bench.py.

Inputs: every Q/K/V value is the synthetic model's value of its token (synth), written on the
device by synth.device; cached tokens' KV is written straight into the pool at the slots the
product's tree assigned ('cache' phases), computed tokens' K/V reach the pool only through the
kernels' scatter. The oracle never sees the pool: it regenerates K/V from token identity.
"""
from __future__ import annotations

import numpy as np

import synth
from synth import device as sdev
from synth import workloads as W


def torch_dtype(name):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_engine(w, max_reqs=None, kv_chunk=0, share_decode=True, stack_extend=True,
                host_tier_slots=0, host_planes=None, stack_levels=4, fold_extend=True):
    from prefix_cached_paged_gb300.serving import Engine
    m = w.model
    n_reqs = max_reqs or max(max((len(p.seqs) for p in w.phases), default=0) + 8, 64)
    return Engine(m.layers, m.n_q_heads, m.n_kv_heads, m.head_dim, torch_dtype(m.dtype),
                  w.pool_slots, n_reqs, w.max_ctx, w.pool_order, kv_chunk=kv_chunk,
                  share_decode=share_decode, stack_extend=stack_extend,
                  host_tier_slots=host_tier_slots, host_planes=host_planes,
                  stack_levels=stack_levels, fold_extend=fold_extend)


def new_token_hashes(model, seqs, prefix_len):
    """Prefix hashes of the computed tokens of a batch, in batch order (uint64 [T])."""
    hs = synth.prefix_hashes_batch(model.seed, seqs)
    parts = [h[int(p):] for h, p in zip(hs, prefix_len)]
    return np.concatenate(parts) if parts else np.zeros(0, np.uint64)


def fill_pool(engine, model, hashes, slots):
    """Write the synthetic K and V of tokens (given by prefix hash) into the pool at `slots`,
    every layer."""
    import torch
    if len(slots) == 0:
        return
    hd = sdev.hashes_to_device(hashes)
    sd = torch.from_numpy(np.ascontiguousarray(slots, dtype=np.int32)).cuda()
    for layer in range(model.layers):
        sdev.fill_rows(hd, synth.TENSOR_K, layer, engine.dev.k[layer], slots_dev=sd)
        sdev.fill_rows(hd, synth.TENSOR_V, layer, engine.dev.v[layer], slots_dev=sd)


def dense_qkv(model, hashes_dev, layer, n):
    """q [n, Hq, d], k_new / v_new [n, Hkv, d] on the device for tokens given by prefix hash."""
    import torch
    dt = torch_dtype(model.dtype)
    q = torch.empty((n, model.n_q_heads, model.head_dim), dtype=dt, device="cuda")
    k = torch.empty((n, model.n_kv_heads, model.head_dim), dtype=dt, device="cuda")
    v = torch.empty_like(k)
    sdev.fill_rows(hashes_dev, synth.TENSOR_Q, layer, q)
    sdev.fill_rows(hashes_dev, synth.TENSOR_K, layer, k)
    sdev.fill_rows(hashes_dev, synth.TENSOR_V, layer, v)
    return q, k, v


def run_cache_phase(engine, model, seqs, keep_locked=False):
    """Insert sequences one at a time as already computed; their KV goes straight to the pool."""
    for s in seqs:
        b = engine.extend_begin([s], match_all=True)
        h = new_token_hashes(model, [s], b.plan.prefix_len)
        fill_pool(engine, model, h, b.plan.out_loc)
        engine.extend_end(b, keep_locked=keep_locked)


def run_extend_phase(engine, model, seqs, keep_outputs=True, lse=False, layers=None):
    """One extend batch through the product path. Returns (batch, {layer: (o, lse)})."""
    import torch
    b = engine.extend_begin(seqs)
    T = b.num_tokens
    h = new_token_hashes(model, seqs, b.plan.prefix_len)
    hd = sdev.hashes_to_device(h)
    outs = {}
    for layer in (range(model.layers) if layers is None else layers):
        q, k, v = dense_qkv(model, hd, layer, T)
        o = torch.empty_like(q)
        l = torch.empty((T, model.n_q_heads), dtype=torch.float32, device="cuda") if lse else None
        engine.extend_layer(b, layer, q, k, v, o, lse=l)
        if keep_outputs:
            outs[layer] = (o, l)
    engine.extend_end(b)
    return b, outs


def run_decode(engine, model, seqs, lse=False, layers=None):
    """Decode phase: contexts (all but the last token) must be cached; each request decodes its
    last token. Returns (decode batch, {layer: (o, lse)}); the batch is left locked."""
    import torch
    ctx = [s[:-1] for s in seqs]
    db = engine.decode_begin(ctx)
    engine.decode_step(db)
    h = np.array([synth.prefix_hashes(model.seed, s)[-1] for s in seqs], dtype=np.uint64)
    hd = sdev.hashes_to_device(h)
    outs = {}
    for layer in (range(model.layers) if layers is None else layers):
        q, k, v = dense_qkv(model, hd, layer, len(seqs))
        o = torch.empty_like(q)
        l = torch.empty((len(seqs), model.n_q_heads), dtype=torch.float32,
                        device="cuda") if lse else None
        engine.decode_layer(db, layer, q, k, v, o, lse=l)
        outs[layer] = (o, l)
    return db, outs


# ---------------------------------------------------------------- oracle side
def oracle_unit(model, seq, P, layer, kv_head):
    """The oracle's output for one (request, layer, KV head): queries of positions P..L-1, the
    query heads of that KV head. Returns (o [S, g, d], lse [S, g]) in fp64."""
    import oracle
    g = model.group
    h = synth.prefix_hashes(model.seed, seq)
    qh = range(kv_head * g, kv_head * g + g)
    q = synth.values(h[P:], synth.TENSOR_Q, layer, qh, model.head_dim, model.dtype)
    k = synth.values(h, synth.TENSOR_K, layer, [kv_head], model.head_dim, model.dtype)
    v = synth.values(h, synth.TENSOR_V, layer, [kv_head], model.head_dim, model.dtype)
    return oracle.attention(q, k, v, P, model.sm_scale, g, 1)


def tolerance(dtype):
    """(max-abs, rel-L2) accepted between the kernel and the fp64 oracle."""
    return (1e-2, 5e-3) if dtype == "bf16" else (1e-4, 1e-5)


def compare(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    ma, rl = tolerance(dtype)
    return max_abs <= ma and rel <= rl, max_abs, rel
