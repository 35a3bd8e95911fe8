"""Oracle for prefix-cached paged attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may import this
package. The product library never imports or links it, and the two share no code.

It wraps `oracle.cpp` (a plain C++ radix tree, token pool and fp64 attention; see that file's
header for what it restates and the readings it takes) and adds `CacheSim`, the pages' per-request
loop -- traverse, reuse, compute, insert, plus LRU eviction when the pool runs short -- written
out plainly on the oracle's own tree (SGLang blog Sec. 2.3 four-step loop and LRU eviction;
paper digest Sec. 3 and App. A.2 batch formation).

Pins that tie it to the pages and to mathematics live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.cpp with the host C++ compiler into _build/liboracle.so."""
    src = os.path.join(_HERE, "oracle.cpp")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", src,
                           "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.or_pool_create.restype = _P
        L.or_pool_create.argtypes = [_I64, _P]
        L.or_pool_destroy.argtypes = [_P]
        L.or_pool_available.restype = _I64
        L.or_pool_available.argtypes = [_P]
        L.or_pool_alloc.restype = ctypes.c_int
        L.or_pool_alloc.argtypes = [_P, _I64, _P]
        L.or_pool_free.argtypes = [_P, _P, _I64]
        L.or_tree_create.restype = _P
        L.or_tree_create.argtypes = [_P]
        L.or_tree_destroy.argtypes = [_P]
        L.or_match.argtypes = [_P, _P, _I64, _P, _P, _P]
        L.or_insert.argtypes = [_P, _P, _P, _I64, _P, _P]
        L.or_lock.restype = ctypes.c_int
        L.or_lock.argtypes = [_P, _I64]
        L.or_unlock.restype = ctypes.c_int
        L.or_unlock.argtypes = [_P, _I64]
        L.or_evict.restype = ctypes.c_int
        L.or_evict.argtypes = [_P, _I64, _P, _P, _I64, _P]
        L.or_dump.restype = _I64
        L.or_dump.argtypes = [_P, _P, _I64]
        L.or_stats.argtypes = [_P, _P]
        L.or_attention.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
                                   _P, _P]
        L.or_attention_units.argtypes = [_I64, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                         ctypes.c_double, _P, _I64]
        L.or_merge.argtypes = [_P, _P, _I64, _I64, _P, _P]
        L.or_attach_host.argtypes = [_P, _P]
        L.or_match_tiered.argtypes = [_P, _P, _I64, _P, _P, _P, _P]
        L.or_load.restype = ctypes.c_int
        L.or_load.argtypes = [_P, _P, _I64, _P]
        L.or_pending.argtypes = [_P, _P, _P]
        L.or_drain.argtypes = [_P, _P, _P, _P, _P]
        L.or_tiers.restype = _I64
        L.or_tiers.argtypes = [_P, _P, _I64]
        _lib = L
    return _lib


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Pool:
    """Token pool: a free list of slot indices (one slot = one token's KV in every layer)."""

    def __init__(self, num_slots: int, order=None):
        self.num_slots = int(num_slots)
        self._order = None if order is None else _i32(order)
        self.h = lib().or_pool_create(self.num_slots,
                                      None if self._order is None else _ptr(self._order))

    def __del__(self):
        if getattr(self, "h", None):
            lib().or_pool_destroy(self.h)
            self.h = None

    def available(self) -> int:
        return int(lib().or_pool_available(self.h))

    def alloc(self, n: int):
        out = np.empty(max(n, 0), dtype=np.int32)
        if lib().or_pool_alloc(self.h, int(n), _ptr(out)) != 0:
            return None
        return out

    def free(self, slots) -> None:
        s = _i32(slots)
        lib().or_pool_free(self.h, _ptr(s), len(s))


class Tree:
    """Radix tree over token sequences; nodes are addressed by their id (root = 0)."""

    def __init__(self, pool: Pool):
        self.pool = pool
        self.h = lib().or_tree_create(pool.h)

    def __del__(self):
        if getattr(self, "h", None):
            lib().or_tree_destroy(self.h)
            self.h = None

    def match(self, tokens):
        t = _i32(tokens)
        slots = np.empty(len(t), dtype=np.int32)
        n = ctypes.c_int64()
        node = ctypes.c_int64()
        lib().or_match(self.h, _ptr(t), len(t), _ptr(slots), ctypes.byref(n), ctypes.byref(node))
        return int(n.value), slots[: n.value].copy(), int(node.value)

    def insert(self, tokens, slots):
        t = _i32(tokens)
        s = _i32(slots)
        assert len(t) == len(s)
        ex = ctypes.c_int64()
        node = ctypes.c_int64()
        lib().or_insert(self.h, _ptr(t), _ptr(s), len(t), ctypes.byref(ex), ctypes.byref(node))
        return int(ex.value), int(node.value)

    def lock(self, node: int) -> None:
        if lib().or_lock(self.h, int(node)) != 0:
            raise KeyError(node)

    def unlock(self, node: int) -> None:
        rc = lib().or_unlock(self.h, int(node))
        if rc != 0:
            raise KeyError((node, rc))

    def attach_host(self, host_pool: Pool) -> None:
        """Evicted device leaves move to the host tier's slots instead of being freed."""
        self.host_pool = host_pool
        lib().or_attach_host(self.h, host_pool.h)

    def match_tiered(self, tokens):
        """Match through both tiers: (device-resident length, host-resident length after it,
        device slots, node id)."""
        t = _i32(tokens)
        slots = np.empty(len(t), dtype=np.int32)
        dev, host, node = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        lib().or_match_tiered(self.h, _ptr(t), len(t), _ptr(slots), ctypes.byref(dev),
                              ctypes.byref(host), ctypes.byref(node))
        return int(dev.value), int(host.value), slots[: dev.value].copy(), int(node.value)

    def load(self, tokens):
        """Move the host-resident nodes on the path of `tokens` to the device; returns the
        path's slots, or None if the device pool is short."""
        t = _i32(tokens)
        row = np.empty(len(t), dtype=np.int32)
        if lib().or_load(self.h, _ptr(t), len(t), _ptr(row)) != 0:
            return None
        return row

    def drain(self):
        """Owed copies since the last drain: (spill_dev, spill_host, load_host, load_dev)."""
        ns, nl = ctypes.c_int64(), ctypes.c_int64()
        lib().or_pending(self.h, ctypes.byref(ns), ctypes.byref(nl))
        out = [np.empty(ns.value, np.int32), np.empty(ns.value, np.int32),
               np.empty(nl.value, np.int32), np.empty(nl.value, np.int32)]
        lib().or_drain(self.h, *(_ptr(a) for a in out))
        return tuple(out)

    def tiers(self) -> np.ndarray:
        cap = 1 << 16
        while True:
            buf = np.empty(cap, dtype=np.int64)
            n = lib().or_tiers(self.h, _ptr(buf), cap)
            if n >= 0:
                return buf[:n].copy()
            cap = -n

    def evict(self, n: int):
        """Evict LRU unreferenced leaves until >= n tokens are freed. Returns (ok, freed, ids)."""
        freed = ctypes.c_int64()
        nids = ctypes.c_int64()
        cap = 1 << 16
        ids = np.empty(cap, dtype=np.int64)
        rc = lib().or_evict(self.h, int(n), ctypes.byref(freed), _ptr(ids), cap,
                            ctypes.byref(nids))
        return rc == 0, int(freed.value), ids[: min(nids.value, cap)].tolist()

    def dump(self) -> np.ndarray:
        cap = 1 << 16
        while True:
            buf = np.empty(cap, dtype=np.int64)
            n = lib().or_dump(self.h, _ptr(buf), cap)
            if n >= 0:
                return buf[:n].copy()
            cap = -n

    def nodes(self):
        """Parsed dump: list of dicts with id, parent, ref, stamp, key, slots (DFS order)."""
        d = self.dump()
        out, i = [], 0
        while i < len(d):
            nid, par, ref, stamp, ln = (int(x) for x in d[i:i + 5])
            key = d[i + 5:i + 5 + ln].astype(np.int32)
            slots = d[i + 5 + ln:i + 5 + 2 * ln].astype(np.int32)
            out.append(dict(id=nid, parent=par, ref=ref, stamp=stamp, key=key, slots=slots))
            i += 5 + 2 * ln
        return out

    def stats(self) -> dict:
        s = np.zeros(10, dtype=np.int64)
        lib().or_stats(self.h, _ptr(s))
        keys = ["splits", "evicted_nodes", "evicted_tokens", "nodes", "cached_tokens",
                "protected_tokens", "host_tokens", "spilled_tokens", "loaded_tokens",
                "dropped_tokens"]
        return {k: int(v) for k, v in zip(keys, s)}


def attention(q, k, v, P: int, scale: float, n_q_heads: int, n_kv_heads: int):
    """fp64 attention of one request: q [S, Hq, d] at positions P..P+S-1 over k, v [P+S, Hkv, d].

    Returns (out [S, Hq, d], lse [S, Hq]) as float64.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    S, Hq, d = q.shape
    assert Hq == n_q_heads and k.shape == (P + S, n_kv_heads, d) and v.shape == k.shape
    out = np.empty((S, Hq, d), dtype=np.float64)
    lse = np.empty((S, Hq), dtype=np.float64)
    lib().or_attention(_ptr(q), _ptr(k), _ptr(v), P, S, Hq, n_kv_heads, d, float(scale),
                       _ptr(out), _ptr(lse))
    return out, lse


def attention_units(units, scale: float, n_q_heads: int, n_kv_heads: int, threads: int):
    """Many independent attention() calls on `threads` host threads (CPU-baseline timing).

    units: list of (q, k, v, P) fp64 arrays. Returns the list of outputs.
    """
    n = len(units)
    qs = [np.ascontiguousarray(u[0], dtype=np.float64) for u in units]
    ks = [np.ascontiguousarray(u[1], dtype=np.float64) for u in units]
    vs = [np.ascontiguousarray(u[2], dtype=np.float64) for u in units]
    Ps = np.array([u[3] for u in units], dtype=np.int64)
    Ss = np.array([q.shape[0] for q in qs], dtype=np.int64)
    outs = [np.empty_like(q) for q in qs]
    d = qs[0].shape[2]
    arr = lambda xs: (ctypes.c_void_p * n)(*[x.ctypes.data for x in xs])
    lib().or_attention_units(n, arr(qs), arr(ks), arr(vs), _ptr(Ps), _ptr(Ss), n_q_heads,
                             n_kv_heads, d, float(scale), arr(outs), int(threads))
    return outs


def merge(o_parts, lse_parts):
    """Combine partial states (o_i [n, d], lse_i [n]) over disjoint key sets -> (o [d], lse)."""
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    l = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o.shape
    out = np.empty(d, dtype=np.float64)
    lse = ctypes.c_double()
    lib().or_merge(_ptr(o), _ptr(l), n, d, _ptr(out), ctypes.byref(lse))
    return out, float(lse.value)


def peek_match(children, seq):
    """Longest cached prefix of `seq` by walking the tree from the root, changing nothing.

    `children` maps (parent id, first token of the edge) to a dumped node. Returns the matched
    length and the path as [(node id, tokens of its edge matched)], root excluded.
    """
    cur, pos, path = 0, 0, []
    while pos < len(seq):
        c = children.get((cur, int(seq[pos])))
        if c is None:
            break
        key = c["key"]
        k = 0
        while k < len(key) and pos + k < len(seq) and key[k] == seq[pos + k]:
            k += 1
        path.append((c["id"], k))
        pos += k
        if k < len(key):
            break
        cur = c["id"]
    return pos, path


def schedule_batch(tree: Tree, seqs, match_lens=None, fcfs: bool = False,
                   max_batch: int = 1 << 30, max_new_tokens: int = -1, reserve: int = 0):
    """Cache-aware batch formation, longest shared prefix first (paper digest Sec. 3
    "cache-aware scheduling" and App. A.2: match every waiting request, sort by match length,
    admit into the batch while memory allows); `fcfs` keeps queue order instead, the
    first-come-first-served order the digest contrasts it with.

    Readings: with a host tier, matches and room count device-resident tokens only; ties keep
    queue order; admission stops at the first request that does not fit;
    a request fits while the batch holds at most `max_batch` requests and `max_new_tokens`
    computed tokens (len - match; negative = no limit), and while free slots plus the cached
    tokens of unreferenced nodes, less `reserve`, cover the computed tokens plus the set of
    unreferenced cached tokens the admitted matches lock. Returns (order, match, admitted).
    """
    nodes = tree.nodes()
    if getattr(tree, "host_pool", None) is not None:
        # with a host tier, scheduling sees the device-resident part of the tree only
        t = tree.tiers()
        host = {int(i) for i, h in zip(t[0::2], t[1::2]) if h}
        nodes = [n for n in nodes if n["id"] not in host]
    children = {(n["parent"], int(n["key"][0])): n for n in nodes}
    ref = {n["id"]: n["ref"] for n in nodes}
    match, paths = [], []
    for w, s in enumerate(seqs):
        s = _i32(s)
        lim = len(s) if match_lens is None else int(match_lens[w])
        m, path = peek_match(children, s[:lim])
        match.append(m)
        paths.append(path)
    order = list(range(len(seqs)))
    if not fcfs:
        order.sort(key=lambda w: -match[w])     # stable: ties in queue order
    room = (tree.pool.available() + sum(len(n["key"]) for n in nodes if n["ref"] == 0)
            - reserve)
    locked = set()     # (node id, offset in its edge) of unreferenced cached tokens locked
    computed = admitted = 0
    for w in order:
        if admitted == max_batch:
            break
        fresh = len(seqs[w]) - match[w]
        if max_new_tokens >= 0 and computed + fresh > max_new_tokens:
            break
        mine = {(nid, j) for nid, k in paths[w] if ref[nid] == 0 for j in range(k)}
        if computed + fresh + len(locked | mine) > room:
            break
        locked |= mine
        computed += fresh
        admitted += 1
    return order, match, admitted


@dataclass
class BatchResult:
    prefix_len: list = field(default_factory=list)   # matched (reused) tokens per request
    rows: list = field(default_factory=list)         # full slot row per request (len L_r)
    nodes: list = field(default_factory=list)        # node id locked by the match
    evict_request: int = 0                           # tokens asked of eviction (0 = none)
    evicted: int = 0                                 # tokens eviction freed
    existing: list = field(default_factory=list)     # insert: leading tokens already present
    freed_dups: int = 0                              # duplicate slots returned after insert
    extra_slots: np.ndarray = None                   # slots allocated for decode tokens
    host_len: list = field(default_factory=list)     # host-tier tokens loaded per request
    copies: tuple = None                             # (spill_dev, spill_host, load_host, load_dev)


class OutOfSlots(RuntimeError):
    pass


class CacheSim:
    """The pages' loop on the oracle's own tree and pool, written out plainly.

    extend batch: for each request in order, match its tokens except the last (at least one
    token is always computed) and lock the matched node; if the pool has fewer free slots than
    the batch needs, evict LRU leaves for the shortfall; allocate each request's unmatched
    suffix, in request order; (attention runs here); insert each full sequence with its slots,
    free the request's own slots for tokens that an earlier request of the batch already
    inserted, and unlock the matched node.
    """

    def __init__(self, num_slots: int, order=None, host_slots: int = 0, host_order=None):
        self.pool = Pool(num_slots, order)
        self.tree = Tree(self.pool)
        self.host_pool = None
        if host_slots:
            # host tier (SGLang blog Sec. 6.1): evicted leaves move to host slots; a later match
            # that reaches them loads them back instead of recomputing
            self.host_pool = Pool(host_slots, host_order)
            self.tree.attach_host(self.host_pool)

    def _make_room(self, need: int, res: BatchResult):
        avail = self.pool.available()
        if avail < need:
            res.evict_request = need - avail
            ok, freed, _ = self.tree.evict(need - avail)
            res.evicted = freed
            if not ok:
                raise OutOfSlots(f"need {need}, available {avail}, evicted {freed}")

    def extend_prepare(self, seqs, extra: int = 0, match_all: bool = False) -> BatchResult:
        """match + lock, make room, allocate. `extra` more slots are allocated after the batch's
        own (decode tokens of a mixed step). `match_all` matches every token (cache fill)."""
        res = BatchResult()
        for s in seqs:
            s = _i32(s)
            lim = len(s) if match_all else len(s) - 1
            if self.host_pool is None:
                n, slots, node = self.tree.match(s[:max(lim, 0)])
                h = 0
            else:
                n, h, slots, node = self.tree.match_tiered(s[:max(lim, 0)])
            self.tree.lock(node)
            res.prefix_len.append(n)
            res.host_len.append(h)
            res.rows.append(slots)
            res.nodes.append(node)
        # device slots for the computed suffixes and for the host-tier tokens to load back
        need = sum(len(s) - p for s, p in zip(seqs, res.prefix_len)) + extra
        self._make_room(need, res)
        for i, s in enumerate(seqs):
            if res.host_len[i]:
                p = res.prefix_len[i] + res.host_len[i]
                row = self.tree.load(_i32(s)[:p])
                assert row is not None
                res.rows[i] = row
                res.prefix_len[i] = p
        for i, s in enumerate(seqs):
            new = self.pool.alloc(len(s) - res.prefix_len[i])
            assert new is not None
            res.rows[i] = np.concatenate([res.rows[i], new]).astype(np.int32)
        if extra:
            res.extra_slots = self.pool.alloc(extra)
            assert res.extra_slots is not None
        if self.host_pool is not None:
            res.copies = self.tree.drain()
        return res

    def extend_finish(self, seqs, res: BatchResult, keep_locked: bool = False) -> list:
        """insert, free duplicates, unlock. Returns the end node of each inserted sequence."""
        ends = []
        for i, s in enumerate(seqs):
            ex, node = self.tree.insert(s, res.rows[i])
            res.existing.append(ex)
            p = res.prefix_len[i]
            if ex > p:
                self.pool.free(res.rows[i][p:ex])
                res.freed_dups += ex - p
            if keep_locked:
                self.tree.lock(node)
            self.tree.unlock(res.nodes[i])
            ends.append(node)
        return ends

    def cache(self, seqs, keep_locked: bool = False):
        """Insert sequences as if already computed (their KV is written directly)."""
        res = self.extend_prepare(seqs, match_all=True)
        ends = self.extend_finish(seqs, res, keep_locked)
        return res, ends

    def decode_prepare(self, contexts) -> BatchResult:
        """Decode entry: match + lock each cached context, make room, allocate one slot per
        request for its new token. rows[r] = context slots (the new slot is extra_slots[r])."""
        res = BatchResult()
        for c in contexts:
            n, slots, node = self.tree.match(_i32(c))
            self.tree.lock(node)
            res.prefix_len.append(n)
            res.rows.append(slots)
            res.nodes.append(node)
        self._make_room(len(contexts), res)
        res.extra_slots = self.pool.alloc(len(contexts))
        if self.host_pool is not None:
            res.copies = self.tree.drain()
        return res
