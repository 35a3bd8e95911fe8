"""One model's prefix-cached paged attention state and its per-step calls.

`Engine` ties the host pool and radix tree (HostCache) to the device KV planes and slot table
(DeviceKV) and exposes the steps a scheduler runs, each a composition of librc calls:

  extend_begin   plan a batch (match + lock, evict if short, allocate), write each request's slot
                 row into the device slot table and upload the kernel metadata;
  extend_layer   extend attention of one layer (scatters the new K/V into the pool);
  extend_end     insert the sequences, free duplicate slots, unlock, release slot-table rows;
  decode_begin   requests enter decoding: match their cached context, lock it, take a row;
  decode_step    allocate one slot per request for its new token and write it to the row;
  decode_layer   split-K decode attention of one layer;
  decode_end     insert the finished sequences (context + generated tokens) or free the generated
                 tokens' slots, unlock, release rows.

The model's projections (q, k_new, v_new per layer) are the caller's: this module never
computes them.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import (DEFAULT_KV_CHUNK, decode_attention, decode_workspace_bytes, extend_attention,
               extend_workspace_bytes, kv_copy, plan_extend_stacking, shared_context_groups,
               MAX_STACK_LEVELS)
from .runtime import DeviceKV, HostCache, Plan


@dataclass
class ExtendBatch:
    plan: Plan
    row_ids: np.ndarray
    qo_indptr: object      # device int32 [B+1]
    prefix_len: object     # device int32 [B]
    req_idx: object        # device int32 [B]
    out_loc: object        # device int32 [T]
    max_q_len: int
    max_prefix_len: int
    stack: object = None       # (device ranges, device shared, max_group_rows) or None
    workspace: object = None   # device scratch of the stacked pass

    @property
    def num_tokens(self) -> int:
        return self.plan.num_tokens


@dataclass
class DecodeBatch:
    row_ids: np.ndarray
    nodes: np.ndarray      # locked context nodes
    seq_len: np.ndarray    # host int32 [B], including the current new token
    new_slots: np.ndarray  # host int32 [B], slots of the current new tokens
    dev_seq_len: object = None
    dev_req_idx: object = None
    dev_out_loc: object = None
    groups: object = None   # device (indptr, members, shared) of shared-context groups, or None
    num_groups: int = 0
    step_id: object = None  # identity of the current step's lengths (a fresh object per step)
    context_rows: object = None  # host int32 [B, max_ctx]: each context's slots (decode_begin)
    context_len: object = None   # host int64 [B]
    gen_slots: list = None       # host int32 [B] per decode_step: the generated tokens' slots


# shortest shared prefix worth a stacked pass: two key tiles
STACK_MIN_SHARED = 256


class Engine:
    def __init__(self, layers, n_q_heads, n_kv_heads, head_dim, dtype, num_slots, max_reqs,
                 max_ctx, initial_order=None, device="cuda", kv_chunk=0, share_decode=True,
                 stack_extend=True, host_tier_slots=0, host_planes=None,
                 stack_levels=MAX_STACK_LEVELS, fold_extend=True):
        self.layers = layers
        self.n_q_heads, self.n_kv_heads, self.head_dim = n_q_heads, n_kv_heads, head_dim
        self.sm_scale = 1.0 / float(np.sqrt(head_dim))
        self.host = HostCache(num_slots, max_ctx, initial_order, host_slots=host_tier_slots)
        self.dev = DeviceKV(layers, num_slots, n_kv_heads, head_dim, dtype, max_reqs, max_ctx,
                            device)
        self.host_k = self.host_v = None
        if host_tier_slots:
            # the host tier's KV planes: pinned host memory the kernels address directly
            # (host_planes: a caller's (k, v) pair of that shape, reused across engines)
            torch = self.dev.torch
            shape = (layers, host_tier_slots, n_kv_heads, head_dim)
            if host_planes is not None:
                self.host_k, self.host_v = host_planes
                if tuple(self.host_k.shape) != shape or not self.host_k.is_pinned():
                    raise ValueError(f"host_planes must be pinned tensors of shape {shape}")
            else:
                self.host_k = torch.empty(shape, dtype=dtype, pin_memory=True)
                self.host_v = torch.empty(shape, dtype=dtype, pin_memory=True)
        self.max_ctx = max_ctx
        self.kv_chunk = kv_chunk
        # decode reads a context prefix that several requests share once for all of them
        self.share_decode = share_decode
        # extend stacks the new tokens of consecutive requests over a prefix they share, where
        # that is estimated to pay (True), for every group found ("always"), or never (False)
        self.stack_extend = stack_extend
        self.stack_levels = stack_levels   # tree levels stacked (1: the shallowest group only)
        # an innermost stacked group takes its members' remainders in its own pass where that is
        # estimated to pay (True), always ("always"), or never (False)
        self.fold_extend = fold_extend
        self._ext_ws = None
        self._free_rows = list(range(max_reqs - 1, -1, -1))
        self._ws = None
        self._ws_plan = None   # (step id, workspace address, token bound) of the plan in _ws

    def _tier_copies(self, copies):
        """Perform the host tier's owed copies on the stream: spills (device -> host) before
        loads (host -> device), both before any later kernel that writes a recycled slot."""
        if copies is None:
            return
        sd, sh, lh, ld = copies
        if len(sd) == 0 and len(lh) == 0:
            return
        d_sd, d_sh, d_lh, d_ld = self.dev.upload_i32([sd, sh, lh, ld])
        if len(sd):
            kv_copy(self.dev.k, self.dev.v, d_sd, self.host_k, self.host_v, d_sh)
        if len(lh):
            kv_copy(self.host_k, self.host_v, d_lh, self.dev.k, self.dev.v, d_ld)

    # ---------------------------------------------------------------- rows
    def _check_rows(self, n):
        if n > len(self._free_rows):
            raise RuntimeError(f"slot table has {len(self._free_rows)} free rows, {n} needed")

    def _take_rows(self, n):
        self._check_rows(n)
        return np.array([self._free_rows.pop() for _ in range(n)], dtype=np.int32)

    def _release_rows(self, rows):
        self._free_rows.extend(int(r) for r in rows[::-1])

    # ---------------------------------------------------------------- extend
    def _owed_copies(self):
        """Host-tier copies a failed plan or allocation left owed: on the stream first."""
        for c in self.host.take_owed():
            self._tier_copies(c)

    def extend_begin(self, seqs, extra: int = 0, match_all: bool = False) -> ExtendBatch:
        # rows first: a plan allocates slots and locks prefixes, which a late failure would leak
        self._check_rows(len(seqs))
        self._owed_copies()
        plan = self.host.plan(seqs, extra=extra, match_all=match_all)
        self._tier_copies(plan.copies)
        B = len(seqs)
        row_ids = self._take_rows(B)
        self.dev.write_rows(row_ids, plan.rows, plan.lengths)
        qo, pl, ri, ol = self.dev.upload_i32([plan.qo_indptr, plan.prefix_len, row_ids,
                                              plan.out_loc])
        S = plan.lengths - plan.prefix_len
        batch = ExtendBatch(plan, row_ids, qo, pl, ri, ol, int(S.max()) if B else 0,
                            int(plan.prefix_len.max()) if B else 0)
        if self.stack_extend and B > 1:
            # stacking groups over the levels of the tree, each kept where it is estimated to pay
            G = self.n_q_heads // self.n_kv_heads
            ranges, shared, start, level_indptr, max_rows, fold, all_folded = plan_extend_stacking(
                plan.rows, plan.prefix_len, S, STACK_MIN_SHARED, G, self.stack_levels,
                policy="all" if self.stack_extend == "always" else "cost",
                fold=self.fold_extend)
            if len(shared):
                r, sh, st, fo = self.dev.upload_i32([ranges, shared, start, fold])
                batch.stack = (r, sh, max_rows, st, level_indptr, fo, all_folded)
                need = extend_workspace_bytes(plan.num_tokens, self.n_q_heads)
                if self._ext_ws is None or self._ext_ws.numel() < need:
                    self._ext_ws = self.dev.torch.empty(need, dtype=self.dev.torch.uint8,
                                                        device=self.dev.device)
                batch.workspace = self._ext_ws
        return batch

    def extend_layer(self, batch: ExtendBatch, layer: int, q, k_new, v_new, o, lse=None):
        extend_attention(q, k_new, v_new, batch.out_loc, batch.qo_indptr, batch.prefix_len,
                         batch.req_idx, self.dev.req_to_token, self.dev.k[layer],
                         self.dev.v[layer], o, sm_scale=self.sm_scale,
                         max_q_len=batch.max_q_len, max_prefix_len=batch.max_prefix_len, lse=lse,
                         stack=batch.stack, workspace=batch.workspace)

    def extend_end(self, batch: ExtendBatch, keep_locked: bool = False):
        ends, dups = self.host.finish(batch.plan, keep_locked=keep_locked)
        self._release_rows(batch.row_ids)
        return ends, dups

    # ---------------------------------------------------------------- decode
    def decode_begin(self, contexts) -> DecodeBatch:
        """Requests enter decoding: each context must be cached; it is matched and locked, its
        slots written to a fresh slot-table row. The first decode_step allocates the new tokens."""
        self._check_rows(len(contexts))
        self._owed_copies()
        plan = self.host.plan(contexts, match_all=True)
        self._tier_copies(plan.copies)
        if plan.num_tokens:
            self.host.pool.free(plan.out_loc)
            for n in plan.nodes:
                self.host.tree.unlock(int(n))
            raise ValueError("decode_begin: every context must already be cached")
        row_ids = self._take_rows(len(contexts))
        self.dev.write_rows(row_ids, plan.rows, plan.lengths)
        self._decode_plan = plan
        batch = DecodeBatch(row_ids, plan.nodes, plan.lengths.astype(np.int32),
                            np.zeros(len(contexts), np.int32), context_rows=plan.rows,
                            context_len=plan.lengths.astype(np.int64), gen_slots=[])
        if self.share_decode:
            # the contexts' slots never change while they decode (new tokens get new slots), so
            # the groups hold for the whole batch
            G = self.n_q_heads // self.n_kv_heads
            indptr, members, shared = shared_context_groups(
                plan.rows, plan.lengths, 8 // G, self.kv_chunk or DEFAULT_KV_CHUNK)
            if len(shared):
                batch.groups = tuple(self.dev.upload_i32([indptr, members, shared]))
                batch.num_groups = len(shared)
        return batch

    def decode_step(self, batch: DecodeBatch, new_slots=None) -> DecodeBatch:
        """Append one token per request: allocate its slot (evicting if needed) unless given,
        write it to the request's row at position seq_len, and upload the step's metadata."""
        B = len(batch.row_ids)
        self._owed_copies()
        if new_slots is None:
            new_slots = self.host.alloc(B)
            self._tier_copies(self.host.last_alloc_copies)
        cols = batch.seq_len.astype(np.int64)
        rows = np.zeros((B, self.max_ctx), dtype=np.int32)
        rows[np.arange(B), cols] = new_slots
        self.dev.write_rows(batch.row_ids, rows, cols + 1, cols=cols)
        batch.seq_len = batch.seq_len + 1
        batch.new_slots = np.asarray(new_slots, dtype=np.int32)
        if batch.gen_slots is not None:
            batch.gen_slots.append(batch.new_slots.copy())
        batch.step_id = object()   # the lengths changed: the next layer plans again
        batch.dev_seq_len, batch.dev_req_idx, batch.dev_out_loc = self.dev.upload_i32(
            [batch.seq_len, batch.row_ids, batch.new_slots])
        return batch

    def workspace(self, q, k_new, max_total_tokens):
        need = decode_workspace_bytes(q, k_new, self.dev.req_to_token, self.dev.k[0],
                                      max_total_tokens=max_total_tokens, kv_chunk=self.kv_chunk)
        if self._ws is None or self._ws.numel() < need:
            self._ws = self.dev.torch.empty(need, dtype=self.dev.torch.uint8,
                                            device=self.dev.device)
        return self._ws

    def decode_layer(self, batch: DecodeBatch, layer: int, q, k_new, v_new, o, lse=None,
                     max_total_tokens=None):
        mt = int(batch.seq_len.sum()) if max_total_tokens is None else max_total_tokens
        ws = self.workspace(q, k_new, mt)
        # every layer of a step has the same requests and lengths: the first plans, the others
        # reuse its job list (same workspace, same bound)
        key = (batch.step_id, ws.data_ptr(), mt)
        reuse = batch.step_id is not None and self._ws_plan is not None and \
            self._ws_plan[0] is key[0] and self._ws_plan[1:] == key[1:]
        decode_attention(q, k_new, v_new, batch.dev_out_loc, batch.dev_seq_len,
                         batch.dev_req_idx, self.dev.req_to_token, self.dev.k[layer],
                         self.dev.v[layer], o, ws, sm_scale=self.sm_scale, max_total_tokens=mt,
                         kv_chunk=self.kv_chunk, lse=lse, groups=batch.groups,
                         reuse_plan=reuse)
        self._ws_plan = key     # the workspace now holds this step's plan

    def decode_end(self, batch: DecodeBatch, seqs=None):
        """The requests leave decoding. With `seqs` (each request's context followed by the
        tokens its decode steps fed in, one per step), the sequences are inserted into the tree
        like a finished extend (the generated tokens' KV stays cached; slots of tokens the tree
        already holds are freed); without, the generated tokens' slots return to the pool. Then
        the contexts are unlocked and the slot-table rows released."""
        B = len(batch.row_ids)
        gen = (np.stack(batch.gen_slots, axis=1) if batch.gen_slots
               else np.zeros((B, 0), dtype=np.int32))
        if seqs is not None:
            seqs = [np.asarray(s, dtype=np.int32) for s in seqs]
            want = batch.context_len + gen.shape[1]
            if len(seqs) != B or any(len(s) != int(n) for s, n in zip(seqs, want)):
                raise ValueError("decode_end: each sequence must be its context plus one token "
                                 f"per decode step ({gen.shape[1]})")
            lengths = want.astype(np.int64)
            indptr = np.zeros(B + 1, dtype=np.int64)
            np.cumsum(lengths, out=indptr[1:])
            rows = np.array(batch.context_rows, dtype=np.int32, copy=True)
            for b in range(B):
                rows[b, batch.context_len[b]:lengths[b]] = gen[b]
            empty = np.zeros(0, dtype=np.int32)
            self.host.finish(Plan(np.concatenate(seqs) if B else empty, indptr, lengths,
                                  batch.context_len.astype(np.int32), batch.nodes, rows,
                                  empty, empty, empty))
        else:
            if gen.size:
                self.host.pool.free(gen.reshape(-1))
            for n in batch.nodes:
                self.host.tree.unlock(int(n))
        self._release_rows(batch.row_ids)
