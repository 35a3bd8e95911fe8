"""Scheduler-step composition of librc's host calls, plus device-side state for a model.

`HostCache` runs one batch through the pages' loop with librc's batched calls (SGLang blog
Sec. 2.3: traverse, reuse, compute, insert; LRU eviction when the pool runs short; paper digest
App. A.2 batch formation):

  schedule: pick the next batch from a waiting queue, longest cached prefix first, as much as
          the pool can take (rc_schedule_batch; paper digest Sec. 3 cache-aware scheduling);
  plan:   match every sequence (all but its last token; all of it for a cache fill) and lock the
          matched node (rc_radix_match_batch); if fewer slots are free than the batch needs,
          evict LRU leaves for the shortfall (rc_radix_evict_lru); allocate the unmatched
          suffixes in request order, then any extra slots (rc_kv_pool_alloc);
  finish: insert every sequence with its slot row, free duplicate slots, unlock
          (rc_radix_insert_batch).

`DeviceKV` holds a model's KV planes and slot table on the GPU and uploads a plan's metadata.
"""
from __future__ import annotations

import time
from dataclasses import dataclass

import numpy as np

from . import RC_OK, RC_SCHED_LSPF, Pool, RadixTree, RcError


@dataclass
class Plan:
    tokens: np.ndarray        # concatenated sequences, int32
    indptr: np.ndarray        # int64 [B+1]
    lengths: np.ndarray       # int64 [B]
    prefix_len: np.ndarray    # int32 [B], matched (reused) tokens
    nodes: np.ndarray         # uint64 [B], locked by the match
    rows: np.ndarray          # int32 [B, row_stride], full slot rows
    qo_indptr: np.ndarray     # int32 [B+1], offsets of the computed tokens
    out_loc: np.ndarray       # int32 [T], slots of the computed tokens
    extra: np.ndarray         # int32 [extra], slots allocated after the batch's own
    evict_request: int = 0
    evicted: int = 0
    host_len: np.ndarray = None   # int32 [B], tokens loaded back from the host tier
    copies: tuple = None          # host-tier copies owed: (spill_dev, spill_host, load_host,
                                  # load_dev), spills before loads

    @property
    def num_tokens(self) -> int:
        return int(self.qo_indptr[-1])


class WaitingQueue:
    """Waiting sequences kept in one token buffer. HostCache.schedule passes the entries still
    waiting as ranges of that buffer (rc_schedule_batch_ranges), so a queue is packed once, not
    for every scheduling call. `ids` are the queue positions still waiting, in queue order."""

    def __init__(self, seqs):
        seqs = [np.asarray(s, dtype=np.int32) for s in seqs]
        self.lengths = np.array([len(s) for s in seqs], dtype=np.int64)
        self.starts = np.zeros(len(seqs), dtype=np.int64)
        if len(seqs) > 1:
            np.cumsum(self.lengths[:-1], out=self.starts[1:])
        self.tokens = np.concatenate(seqs) if seqs else np.zeros(0, np.int32)
        self.ids = list(range(len(seqs)))

    def __len__(self) -> int:
        return len(self.ids)

    def seq(self, qid: int) -> np.ndarray:
        """The tokens of queue entry qid (a view of the buffer)."""
        s = int(self.starts[qid])
        return self.tokens[s:s + int(self.lengths[qid])]

    def remove(self, positions) -> None:
        """Drop the waiting entries at these positions of `ids`."""
        for i in sorted(positions, reverse=True):
            self.ids.pop(i)


class HostCache:
    def __init__(self, num_slots: int, row_stride: int, initial_order=None, host_slots: int = 0,
                 host_order=None):
        self.pool = Pool(num_slots, initial_order)
        self.tree = RadixTree(self.pool)
        self.row_stride = int(row_stride)
        self.host_pool = None
        if host_slots:
            self.host_pool = Pool(host_slots, host_order)
            self.tree.attach_host_tier(self.host_pool)
        # host-tier copies that a failed call left owed, oldest first; the caller performs them
        # (take_owed) before its next device work
        self._owed = []

    def _stash_copies(self) -> None:
        """After a failed call: take the copies its evictions and loads already owe out of the
        tree (the tree refuses to evict while loads are pending) and keep them for take_owed."""
        if self.host_pool is None:
            return
        c = self.tree.drain_copies()
        if len(c[0]) or len(c[2]):
            self._owed.append(c)

    def take_owed(self) -> list:
        """Copies (spill_dev, spill_host, load_host, load_dev) that failed calls left owed, oldest
        first: perform them, each spills before loads, before any later device work."""
        out, self._owed = self._owed, []
        return out

    def _release_on_error(self, nodes, fn, *args):
        """fn(*args); if it fails, the nodes this plan's match locked are unlocked first, so a
        failed plan leaves the tree as it found it apart from evictions (which are complete)."""
        try:
            return fn(*args)
        except RcError:
            for n in nodes:
                self.tree.unlock(int(n))
            self._stash_copies()
            raise

    def _make_room(self, need: int, plan: Plan, nodes) -> None:
        avail = self.pool.available()
        if avail < need:
            plan.evict_request = need - avail
            rc, freed = self.tree.evict_lru(need - avail)
            plan.evicted = freed
            if rc != RC_OK:
                for n in nodes:
                    self.tree.unlock(int(n))
                self._stash_copies()
                raise RcError(rc, f"make room for {need} slots ({avail} free, {freed} evicted)")

    host_seconds = 0.0   # accumulated time spent in the tree / pool calls of plan and finish

    def plan(self, seqs, extra: int = 0, match_all: bool = False) -> Plan:
        t0 = time.perf_counter()
        try:
            return self._plan(seqs, extra, match_all)
        finally:
            self.host_seconds += time.perf_counter() - t0

    def _plan(self, seqs, extra: int = 0, match_all: bool = False) -> Plan:
        seqs = [np.asarray(s, dtype=np.int32) for s in seqs]
        B = len(seqs)
        lengths = np.array([len(s) for s in seqs], dtype=np.int64)
        indptr = np.zeros(B + 1, dtype=np.int64)
        np.cumsum(lengths, out=indptr[1:])
        tokens = np.concatenate(seqs) if B else np.zeros(0, np.int32)
        match_len = lengths if match_all else np.maximum(lengths - 1, 0)
        rows = np.zeros((B, self.row_stride), dtype=np.int32)
        host_len = None
        pre = Plan(*(np.zeros(0),) * 9)     # eviction done before a load, if any
        if self.host_pool is None:
            prefix_len, nodes = self.tree.match_batch(tokens, indptr,
                                                      match_len.astype(np.int32), rows)
        else:
            prefix_len, nodes, host_len = self.tree.match_batch_tiered(
                tokens, indptr, match_len.astype(np.int32), rows)
            if host_len.any():
                # device room for the suffixes and the host-tier tokens, then load those back
                self._make_room(int((lengths - prefix_len).sum()) + int(extra), pre, nodes)
                self._release_on_error(nodes, self.tree.load_batch, tokens, indptr, rows,
                                       prefix_len, host_len)
        S = lengths - prefix_len
        qo = np.zeros(B + 1, dtype=np.int32)
        np.cumsum(S, out=qo[1:])
        plan = Plan(tokens, indptr, lengths, prefix_len, nodes, rows, qo,
                    np.zeros(0, np.int32), np.zeros(0, np.int32))
        need = int(qo[-1]) + int(extra)
        self._make_room(need, plan, nodes)
        if pre.evict_request:
            plan.evict_request, plan.evicted = pre.evict_request, pre.evicted
        new = self._release_on_error(nodes, self.pool.alloc, need)
        for b in range(B):
            rows[b, prefix_len[b]:lengths[b]] = new[qo[b]:qo[b + 1]]
        plan.out_loc = new[: qo[-1]]
        plan.extra = new[qo[-1]:]
        if self.host_pool is not None:
            plan.host_len = host_len
            plan.copies = self.tree.drain_copies()
        return plan

    def schedule(self, waiting, max_batch: int = 1 << 30, max_new_tokens: int = -1,
                 reserve: int = 0, policy: int = RC_SCHED_LSPF):
        """Batch formation (rc_schedule_batch; longest shared prefix first by default) over the
        waiting sequences, matched like `plan` matches them (all but the last token). Returns
        the queue positions of the admitted batch, in the order to plan them. `waiting` is a
        list of token arrays, or a WaitingQueue (its entries still waiting; no repacking)."""
        t0 = time.perf_counter()
        try:
            if isinstance(waiting, WaitingQueue):
                ids = np.asarray(waiting.ids, dtype=np.int64)
                lengths = waiting.lengths[ids]
                order, _, admitted = self.tree.schedule_batch_ranges(
                    waiting.tokens, waiting.starts[ids], lengths,
                    np.maximum(lengths - 1, 0).astype(np.int32), policy, max_batch,
                    max_new_tokens, reserve)
                return order[:admitted].tolist()
            seqs = [np.asarray(s, dtype=np.int32) for s in waiting]
            lengths = np.array([len(s) for s in seqs], dtype=np.int64)
            indptr = np.zeros(len(seqs) + 1, dtype=np.int64)
            np.cumsum(lengths, out=indptr[1:])
            tokens = np.concatenate(seqs) if seqs else np.zeros(0, np.int32)
            order, _, admitted = self.tree.schedule_batch(
                tokens, indptr, np.maximum(lengths - 1, 0).astype(np.int32), policy, max_batch,
                max_new_tokens, reserve)
            return order[:admitted].tolist()
        finally:
            self.host_seconds += time.perf_counter() - t0

    def finish(self, plan: Plan, keep_locked: bool = False):
        """Insert, free duplicates, unlock. Returns (end nodes, duplicates freed)."""
        t0 = time.perf_counter()
        try:
            return self.tree.insert_batch(plan.tokens, plan.indptr, plan.rows, plan.prefix_len,
                                          plan.nodes, keep_locked)
        finally:
            self.host_seconds += time.perf_counter() - t0

    def alloc(self, n: int) -> np.ndarray:
        """n slots for decode tokens, evicting LRU leaves if the pool is short."""
        p = Plan(*(np.zeros(0),) * 9)
        self._make_room(n, p, [])
        out = self._release_on_error([], self.pool.alloc, n)
        self.last_alloc_evicted = p.evicted
        self.last_alloc_copies = (self.tree.drain_copies() if self.host_pool is not None
                                  else None)
        return out


class DeviceKV:
    """KV planes [layers, num_slots, Hkv, d] for K and V and the slot table on one GPU."""

    def __init__(self, layers, num_slots, n_kv_heads, head_dim, dtype, max_reqs, max_ctx,
                 device="cuda"):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        self.k = torch.empty((layers, num_slots, n_kv_heads, head_dim), dtype=dtype,
                             device=self.device)
        self.v = torch.empty_like(self.k)
        self.req_to_token = torch.zeros((max_reqs, max_ctx), dtype=torch.int32,
                                        device=self.device)
        self._ring = [None] * 8      # pinned staging buffers, reused round-robin
        self._ring_ev = [None] * 8
        self._ring_i = 0

    def upload_i32(self, arrays):
        """Copy int32 host arrays to the device in one transfer through a pinned staging buffer;
        returns device views in order."""
        torch = self.torch
        arrays = [np.ascontiguousarray(a, dtype=np.int32).ravel() for a in arrays]
        sizes = [len(a) for a in arrays]
        total = max(sum(sizes), 1)
        i = self._ring_i
        self._ring_i = (i + 1) % len(self._ring)
        if self._ring_ev[i] is not None:
            self._ring_ev[i].synchronize()   # the copy that last used this buffer is done
        if self._ring[i] is None or self._ring[i].numel() < total:
            self._ring[i] = torch.empty(max(total, 1 << 16), dtype=torch.int32, pin_memory=True)
        stage = self._ring[i]
        host = stage.numpy()
        off = 0
        for a in arrays:
            host[off:off + len(a)] = a
            off += len(a)
        dev = stage[:total].to(self.device, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record()
        self._ring_ev[i] = ev
        out, off = [], 0
        for n in sizes:
            out.append(dev[off:off + n])
            off += n
        return out

    def write_rows(self, row_ids, rows, ends, cols=None):
        """req_to_token[row_ids[b], cols[b]:ends[b]] = rows[b, cols[b]:ends[b]] (cols default 0),
        one upload and one slot-table kernel for the whole batch."""
        from . import slot_table_write
        B = len(row_ids)
        cols = np.zeros(B, np.int64) if cols is None else np.asarray(cols, dtype=np.int64)
        seg_len = np.asarray(ends, dtype=np.int64) - cols
        vals = [rows[b, cols[b]:cols[b] + seg_len[b]] for b in range(B)]
        indptr = np.zeros(B + 1, dtype=np.int64)
        np.cumsum(seg_len, out=indptr[1:])
        values = np.concatenate(vals) if B else np.zeros(0, np.int32)
        r, c, ip, v = self.upload_i32([row_ids, cols, indptr, values])
        slot_table_write(self.req_to_token, r, c, ip, v)
