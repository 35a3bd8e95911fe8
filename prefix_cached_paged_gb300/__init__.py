"""prefix_cached_paged_gb300 -- RadixAttention's data path on one GB300 (sm_103a).

A thin binding of librc (include/rc.h): a token-granular KV pool, a radix tree that finds each
request's longest cached prefix and evicts unreferenced leaves in LRU order (host C++), and the
extend / decode attention kernels that run on a paged KV pool through a slot table (CUDA).
The binding only marshals arguments: every step runs in librc, and there is no fallback path --
without the compiled library every call raises.

Names follow the C ABI without the `rc_` prefix. Device functions take torch CUDA tensors (used
for device memory and streams only) and launch on the current torch stream.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import (RC_DTYPE_BF16, RC_DTYPE_F32, RC_ERR_CUDA, RC_ERR_DEVICE, RC_ERR_INSUFFICIENT,
                   RC_ERR_INVALID, RC_ERR_OOM, RC_OK, RC_SCHED_FCFS, RC_SCHED_LSPF, RcDecodeArgs,
                   RcError, RcExtendArgs, RcKvCopyArgs, RcSlotWriteArgs, RcStackPlan,
                   RcStackPlanArgs, RcStats, check, lib)

__all__ = [
    "Pool", "RadixTree", "RcError", "slot_table_write", "extend_attention", "decode_attention",
    "decode_workspace_bytes", "decode_attention_noalloc", "device_status", "launch_count", "RC_OK", "RC_ERR_INVALID",
    "RC_ERR_OOM", "RC_ERR_INSUFFICIENT", "RC_ERR_CUDA", "RC_ERR_DEVICE", "RC_SCHED_LSPF",
    "RC_SCHED_FCFS",
]


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def launch_count() -> int:
    return int(lib().rc_launch_count())


def set_wait_limit_ns(ns: int) -> None:
    """Test hook (rc_debug_set_wait_limit_ns): bound of the extend kernel's waits for later
    launches; 0 restores the default."""
    check(lib().rc_debug_set_wait_limit_ns(int(ns)), "rc_debug_set_wait_limit_ns")


class Pool:
    """The token pool (free list of KV slots). rc_pool_* / rc_kv_pool_*."""

    def __init__(self, num_slots: int, initial_order=None):
        self._order = None if initial_order is None else _i32(initial_order)
        h = ctypes.c_void_p()
        check(lib().rc_pool_create(int(num_slots), None if self._order is None else
                                   _p(self._order), ctypes.byref(h)), "rc_pool_create")
        self.h = h
        self.num_slots = int(num_slots)

    def __del__(self):
        if getattr(self, "h", None) is not None and self.h.value:
            lib().rc_pool_destroy(self.h)
            self.h = None

    def alloc(self, n: int, out: np.ndarray | None = None) -> np.ndarray:
        out = np.empty(int(n), dtype=np.int32) if out is None else out
        check(lib().rc_kv_pool_alloc(self.h, int(n), _p(out)), "rc_kv_pool_alloc")
        return out

    def free(self, slots) -> None:
        s = _i32(slots)
        check(lib().rc_kv_pool_free(self.h, _p(s), len(s)), "rc_kv_pool_free")

    def available(self) -> int:
        v = ctypes.c_int64()
        check(lib().rc_kv_pool_available(self.h, ctypes.byref(v)), "rc_kv_pool_available")
        return int(v.value)

    def inject_alloc_failure(self, after_calls: int) -> None:
        """Test hook: the alloc() after `after_calls` more successful ones fails with
        RC_ERR_OOM and changes nothing (one shot; -1 disarms)."""
        check(lib().rc_pool_inject_alloc_failure(self.h, int(after_calls)),
              "rc_pool_inject_alloc_failure")


class RadixTree:
    """The radix tree over token sequences. rc_radix_*."""

    def __init__(self, pool: Pool):
        self.pool = pool
        h = ctypes.c_void_p()
        check(lib().rc_radix_create(pool.h, ctypes.byref(h)), "rc_radix_create")
        self.h = h

    def __del__(self):
        if getattr(self, "h", None) is not None and self.h.value:
            lib().rc_radix_destroy(self.h)
            self.h = None

    def match_prefix(self, tokens):
        t = _i32(tokens)
        out = np.empty(len(t), dtype=np.int32)
        n = ctypes.c_int64()
        node = ctypes.c_uint64()
        check(lib().rc_radix_match_prefix(self.h, _p(t), len(t), _p(out), ctypes.byref(n),
                                          ctypes.byref(node)), "rc_radix_match_prefix")
        return int(n.value), out[: n.value].copy(), int(node.value)

    def insert(self, tokens, slots):
        t, s = _i32(tokens), _i32(slots)
        ex = ctypes.c_int64()
        node = ctypes.c_uint64()
        check(lib().rc_radix_insert(self.h, _p(t), _p(s), len(t), ctypes.byref(ex),
                                    ctypes.byref(node)), "rc_radix_insert")
        return int(ex.value), int(node.value)

    def lock(self, node: int) -> None:
        check(lib().rc_radix_lock(self.h, int(node)), "rc_radix_lock")

    def unlock(self, node: int) -> None:
        check(lib().rc_radix_unlock(self.h, int(node)), "rc_radix_unlock")

    def evict_lru(self, n_tokens: int):
        """Returns (status, freed): status RC_OK or RC_ERR_INSUFFICIENT."""
        f = ctypes.c_int64()
        rc = lib().rc_radix_evict_lru(self.h, int(n_tokens), ctypes.byref(f))
        if rc not in (RC_OK, RC_ERR_INSUFFICIENT):
            check(rc, "rc_radix_evict_lru")
        return rc, int(f.value)

    def stats(self) -> dict:
        s = RcStats()
        check(lib().rc_radix_stats(self.h, ctypes.byref(s)), "rc_radix_stats")
        return {k: int(getattr(s, k)) for k, _ in RcStats._fields_}

    def dump(self) -> np.ndarray:
        n = lib().rc_radix_dump(self.h, None, 0)
        need = -n if n < 0 else n
        buf = np.empty(max(need, 1), dtype=np.int64)
        w = lib().rc_radix_dump(self.h, _p(buf), need)
        assert w >= 0
        return buf[:w].copy()

    def match_batch(self, tokens: np.ndarray, indptr: np.ndarray, match_len, rows: np.ndarray):
        """Match + lock B sequences in order. rows: [B, row_stride] int32 (written in place).
        Returns (prefix_len int32[B], nodes uint64[B])."""
        B = len(indptr) - 1
        pl = np.empty(B, dtype=np.int32)
        nodes = np.empty(B, dtype=np.uint64)
        ml = None if match_len is None else _i32(match_len)
        check(lib().rc_radix_match_batch(self.h, _p(tokens), _p(indptr), B,
                                         None if ml is None else _p(ml), _p(rows),
                                         rows.shape[1], _p(pl), _p(nodes)),
              "rc_radix_match_batch")
        return pl, nodes

    def attach_host_tier(self, host_pool: "Pool") -> None:
        """Evicted device leaves move to host_pool's slots instead of being freed."""
        check(lib().rc_radix_attach_host_tier(self.h, host_pool.h), "rc_radix_attach_host_tier")
        self.host_pool = host_pool

    def match_batch_tiered(self, tokens, indptr, match_len, rows):
        """Match + lock B sequences through both tiers. Returns (prefix_len int32[B] = the
        device-resident part, nodes uint64[B], host_len int32[B])."""
        B = len(indptr) - 1
        pl = np.empty(B, dtype=np.int32)
        nodes = np.empty(B, dtype=np.uint64)
        hl = np.empty(B, dtype=np.int32)
        ml = None if match_len is None else _i32(match_len)
        check(lib().rc_radix_match_batch_tiered(self.h, _p(tokens), _p(indptr), B,
                                                None if ml is None else _p(ml), _p(rows),
                                                rows.shape[1], _p(pl), _p(nodes), _p(hl)),
              "rc_radix_match_batch_tiered")
        return pl, nodes, hl

    def load_batch(self, tokens, indptr, rows, prefix_len, host_len) -> None:
        """Move the matched host-resident tokens back to the device; prefix_len (int32, in
        place) grows by host_len and rows receive the new device slots."""
        assert prefix_len.dtype == np.int32 and prefix_len.flags.c_contiguous
        hl = _i32(host_len)
        check(lib().rc_radix_load_batch(self.h, _p(tokens), _p(indptr), len(indptr) - 1,
                                        _p(rows), rows.shape[1], _p(prefix_len), _p(hl)),
              "rc_radix_load_batch")

    def drain_copies(self):
        """The copies owed since the last drain: (spill_dev, spill_host, load_host, load_dev),
        spills to run before loads."""
        ns, nl = ctypes.c_int64(), ctypes.c_int64()
        check(lib().rc_radix_pending_copies(self.h, ctypes.byref(ns), ctypes.byref(nl)),
              "rc_radix_pending_copies")
        sd = np.empty(ns.value, np.int32)
        sh = np.empty(ns.value, np.int32)
        lh = np.empty(nl.value, np.int32)
        ld = np.empty(nl.value, np.int32)
        check(lib().rc_radix_drain_copies(self.h, _p(sd), _p(sh), _p(lh), _p(ld)),
              "rc_radix_drain_copies")
        return sd, sh, lh, ld

    def tiers(self) -> np.ndarray:
        """(node id, 1 if host-resident) per node, in the dump's order."""
        n = lib().rc_radix_tiers(self.h, None, 0)
        need = -n if n < 0 else n
        buf = np.empty(max(need, 1), dtype=np.int64)
        w = lib().rc_radix_tiers(self.h, _p(buf), need)
        assert w >= 0
        return buf[:w]

    def schedule_batch(self, tokens: np.ndarray, indptr: np.ndarray, match_len=None,
                       policy: int = 0, max_batch: int = 1 << 30, max_new_tokens: int = -1,
                       reserve_slots: int = 0):
        """Batch formation over W waiting sequences (the tree is not changed); policy
        RC_SCHED_LSPF (longest shared prefix first) or RC_SCHED_FCFS (queue order). Returns
        (order int32[W], match int32[W], admitted): the batch is order[:admitted]."""
        W = len(indptr) - 1
        order = np.empty(W, dtype=np.int32)
        match = np.empty(W, dtype=np.int32)
        adm = ctypes.c_int32()
        ml = None if match_len is None else _i32(match_len)
        tok = _i32(tokens)
        ip = np.ascontiguousarray(indptr, np.int64)
        check(lib().rc_schedule_batch(self.h, _p(tok), _p(ip), W,
                                      None if ml is None else _p(ml), int(policy),
                                      int(max_batch), int(max_new_tokens), int(reserve_slots),
                                      _p(order), _p(match), ctypes.byref(adm)),
              "rc_schedule_batch")
        return order, match, int(adm.value)

    def schedule_batch_ranges(self, tokens: np.ndarray, starts: np.ndarray, lengths: np.ndarray,
                              match_len=None, policy: int = 0, max_batch: int = 1 << 30,
                              max_new_tokens: int = -1, reserve_slots: int = 0):
        """schedule_batch over W sequences given as ranges of one buffer: sequence w is
        tokens[starts[w] : starts[w] + lengths[w]]. Same outputs as schedule_batch."""
        W = len(starts)
        order = np.empty(W, dtype=np.int32)
        match = np.empty(W, dtype=np.int32)
        adm = ctypes.c_int32()
        ml = None if match_len is None else _i32(match_len)
        tok = _i32(tokens)
        st = np.ascontiguousarray(starts, np.int64)
        ln = np.ascontiguousarray(lengths, np.int64)
        check(lib().rc_schedule_batch_ranges(self.h, _p(tok), _p(st), _p(ln), W,
                                             None if ml is None else _p(ml), int(policy),
                                             int(max_batch), int(max_new_tokens),
                                             int(reserve_slots), _p(order), _p(match),
                                             ctypes.byref(adm)),
              "rc_schedule_batch_ranges")
        return order, match, int(adm.value)

    def insert_batch(self, tokens, indptr, rows, prefix_len, unlock_nodes, keep_locked=False):
        """Insert B sequences with their slot rows, free duplicates, optionally lock the ends,
        unlock the matched nodes. Returns (end_nodes uint64[B], duplicates freed)."""
        B = len(indptr) - 1
        ends = np.empty(B, dtype=np.uint64)
        freed = ctypes.c_int64()
        un = None if unlock_nodes is None else np.ascontiguousarray(unlock_nodes, np.uint64)
        check(lib().rc_radix_insert_batch(self.h, _p(tokens), _p(indptr), B, _p(rows),
                                          rows.shape[1], _p(_i32(prefix_len)),
                                          None if un is None else _p(un), int(keep_locked),
                                          _p(ends), ctypes.byref(freed)),
              "rc_radix_insert_batch")
        return ends, int(freed.value)


# ------------------------------------------------------------------ device entry points
def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return RC_DTYPE_BF16
    if t.dtype == torch.float32:
        return RC_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def slot_table_write(req_to_token, seg_row, seg_col, seg_indptr, values, stream=None):
    """req_to_token[seg_row[i], seg_col[i] + j] = values[seg_indptr[i] + j] (device int32)."""
    a = RcSlotWriteArgs(num_segments=seg_row.numel(), max_reqs=req_to_token.shape[0],
                        max_ctx=req_to_token.shape[1], total_values=values.numel(),
                        seg_row=seg_row.data_ptr(), seg_col=seg_col.data_ptr(),
                        seg_indptr=seg_indptr.data_ptr(), values=values.data_ptr(),
                        req_to_token=req_to_token.data_ptr())
    check(lib().rc_slot_table_write(ctypes.byref(a), _stream(stream)), "rc_slot_table_write")


def kv_copy(src_k, src_v, src_slots, dst_k, dst_v, dst_slots, stream=None):
    """For every i and layer: K and V rows of src_slots[i] -> dst_slots[i]. Planes are
    [layers, num_slots, Hkv, d] tensors on the device or in pinned host memory (the host tier);
    slot arrays are device int32."""
    for t in (src_k, src_v, dst_k, dst_v):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("kv_copy: planes must be device tensors or pinned host tensors")
        if not t.is_contiguous():
            raise ValueError("kv_copy: planes must be contiguous")
    if src_k.shape[0] != dst_k.shape[0] or src_k.shape[2:] != dst_k.shape[2:] or \
            src_k.dtype != dst_k.dtype or src_k.shape != src_v.shape or dst_k.shape != dst_v.shape:
        raise ValueError("kv_copy: plane shapes or dtypes differ")
    if src_slots.numel() != dst_slots.numel():
        raise ValueError("kv_copy: slot arrays differ in length")
    row = src_k.shape[2] * src_k.shape[3] * src_k.element_size()
    a = RcKvCopyArgs(n=src_slots.numel(), layers=src_k.shape[0], row_bytes=row,
                     src_slots=src_slots.data_ptr(), dst_slots=dst_slots.data_ptr(),
                     src_k=src_k.data_ptr(), src_v=src_v.data_ptr(),
                     src_num_slots=src_k.shape[1], dst_k=dst_k.data_ptr(),
                     dst_v=dst_v.data_ptr(), dst_num_slots=dst_k.shape[1])
    check(lib().rc_kv_copy(ctypes.byref(a), _stream(stream)), "rc_kv_copy")


def _extend_args(q, k_new, v_new, out_loc, qo_indptr, prefix_len, req_idx, req_to_token,
                 k_pool, v_pool, o, lse, sm_scale, max_q_len, max_prefix_len, stack=None,
                 workspace=None):
    T, Hq, d = q.shape
    Hkv = k_new.shape[1]
    g = {}
    if stack is not None:
        # (ranges, shared, max_rows) or, for a cascade over tree levels, (ranges, shared,
        # max_rows, start, level_indptr) -- level_indptr a host int32 numpy array
        ranges, shared, max_rows = stack[:3]
        g = dict(num_groups=int(shared.numel()), max_group_rows=int(max_rows),
                 group_range=ranges.data_ptr(), group_shared=shared.data_ptr(),
                 workspace=0 if workspace is None else workspace.data_ptr(),
                 workspace_bytes=0 if workspace is None else
                 workspace.numel() * workspace.element_size())
        if len(stack) >= 5:
            start, level_indptr = stack[3], stack[4]
            assert level_indptr.dtype == np.int32 and level_indptr.flags.c_contiguous
            g.update(num_levels=len(level_indptr) - 1, level_indptr=level_indptr.ctypes.data,
                     group_start=start.data_ptr())
        if len(stack) >= 7 and stack[5] is not None:
            # (..., group_fold device int32 [G], every request folded)
            g.update(group_fold=stack[5].data_ptr(), skip_request_pass=int(bool(stack[6])))
    return RcExtendArgs(**g,
        dtype=_dtype_code(q), num_reqs=prefix_len.numel(), num_q_heads=Hq, num_kv_heads=Hkv,
        head_dim=d, max_reqs=req_to_token.shape[0], max_ctx=req_to_token.shape[1], max_q_len=int(max_q_len),
        max_prefix_len=int(max_prefix_len), num_tokens=T, num_slots=k_pool.shape[0],
        sm_scale=float(sm_scale), q=q.data_ptr(), k_new=k_new.data_ptr(),
        v_new=v_new.data_ptr(), out_loc=out_loc.data_ptr(), qo_indptr=qo_indptr.data_ptr(),
        prefix_len=prefix_len.data_ptr(), req_idx=req_idx.data_ptr(),
        req_to_token=req_to_token.data_ptr(), k_pool=k_pool.data_ptr(),
        v_pool=v_pool.data_ptr(), o=o.data_ptr(), lse=0 if lse is None else lse.data_ptr())


def extend_workspace_bytes(num_tokens: int, num_q_heads: int) -> int:
    """Workspace of the stacked prefix pass (rc_extend_workspace_bytes)."""
    a = RcExtendArgs(num_tokens=int(num_tokens), num_q_heads=int(num_q_heads))
    n = ctypes.c_size_t()
    check(lib().rc_extend_workspace_bytes(ctypes.byref(a), ctypes.byref(n)),
          "rc_extend_workspace_bytes")
    return int(n.value)


def extend_attention(q, k_new, v_new, out_loc, qo_indptr, prefix_len, req_idx, req_to_token,
                     k_pool, v_pool, o, *, sm_scale, max_q_len, max_prefix_len, lse=None,
                     stack=None, workspace=None, stream=None):
    """Extend attention of one layer (see rc_extend_attention). k_pool / v_pool are this layer's
    planes [num_slots, Hkv, d]. stack: optional prefix-stacking groups (ranges, shared,
    max_group_rows) -- int32 CUDA tensors and an int, as built by prefix_stacking_groups() --
    with a uint8 CUDA workspace of extend_workspace_bytes(T, Hq) bytes."""
    a = _extend_args(q, k_new, v_new, out_loc, qo_indptr, prefix_len, req_idx, req_to_token,
                     k_pool, v_pool, o, lse, sm_scale, max_q_len, max_prefix_len, stack,
                     workspace)
    check(lib().rc_extend_attention(ctypes.byref(a), _stream(stream)), "rc_extend_attention")


def _decode_args(q, k_new, v_new, out_loc, seq_len, req_idx, req_to_token, k_pool, v_pool, o,
                 lse, sm_scale, max_total_tokens, kv_chunk, groups=None):
    B, Hq, d = q.shape
    g = dict(num_groups=0, group_indptr=0, group_members=0, group_shared=0)
    if groups is not None:
        indptr, members, shared = groups
        g = dict(num_groups=int(shared.numel()), group_indptr=indptr.data_ptr(),
                 group_members=members.data_ptr(), group_shared=shared.data_ptr())
    return RcDecodeArgs(**g,
        dtype=_dtype_code(q), num_reqs=B, num_q_heads=Hq, num_kv_heads=k_new.shape[1],
        head_dim=d, max_reqs=req_to_token.shape[0], max_ctx=req_to_token.shape[1], kv_chunk=int(kv_chunk),
        max_total_tokens=int(max_total_tokens), num_slots=k_pool.shape[0],
        sm_scale=float(sm_scale), q=q.data_ptr(), k_new=k_new.data_ptr(),
        v_new=v_new.data_ptr(), out_loc=out_loc.data_ptr(), seq_len=seq_len.data_ptr(),
        req_idx=req_idx.data_ptr(), req_to_token=req_to_token.data_ptr(),
        k_pool=k_pool.data_ptr(), v_pool=v_pool.data_ptr(), o=o.data_ptr(),
        lse=0 if lse is None else lse.data_ptr())


def decode_workspace_bytes(q, k_new, req_to_token, k_pool, *, max_total_tokens, kv_chunk=0) -> int:
    B, Hq, d = q.shape
    a = RcDecodeArgs(dtype=_dtype_code(q), num_reqs=B, num_q_heads=Hq,
                     num_kv_heads=k_new.shape[1], head_dim=d, max_reqs=req_to_token.shape[0],
                     max_ctx=req_to_token.shape[1],
                     kv_chunk=int(kv_chunk), max_total_tokens=int(max_total_tokens),
                     num_slots=k_pool.shape[0])
    n = ctypes.c_size_t()
    check(lib().rc_decode_workspace_bytes(ctypes.byref(a), ctypes.byref(n)),
          "rc_decode_workspace_bytes")
    return int(n.value)


def decode_attention(q, k_new, v_new, out_loc, seq_len, req_idx, req_to_token, k_pool, v_pool,
                     o, workspace, *, sm_scale, max_total_tokens, kv_chunk=0, lse=None,
                     groups=None, stream=None, reuse_plan=False):
    """Split-K decode attention of one layer (see rc_decode_attention). workspace: a uint8 CUDA
    tensor of at least decode_workspace_bytes(...) bytes. groups: optional shared-context groups
    (indptr, members, shared), int32 CUDA tensors, as built by shared_context_groups().
    reuse_plan: the previous call on this workspace had the same requests and sizes (the other
    layers of a decode step) -- its job list is reused."""
    a = _decode_args(q, k_new, v_new, out_loc, seq_len, req_idx, req_to_token, k_pool, v_pool,
                     o, lse, sm_scale, max_total_tokens, kv_chunk, groups)
    a.reuse_plan = 1 if reuse_plan else 0
    check(lib().rc_decode_attention(ctypes.byref(a), ctypes.c_void_p(workspace.data_ptr()),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "rc_decode_attention")


DEFAULT_KV_CHUNK = 512   # tokens per split-K chunk when kv_chunk = 0 (rc.h)


MAX_STACK_LEVELS = 4   # RC_MAX_STACK_LEVELS
_FOLD_MODES = {False: 0, True: 1, "always": 2}   # RC_FOLD_NONE / RC_FOLD_COST / RC_FOLD_ALL


def plan_extend_stacking(rows, prefix_len, new_len, min_shared: int, group: int,
                         max_levels: int = MAX_STACK_LEVELS, policy="cost", fold=True):
    """rc_plan_extend_stacking: the extend batch's stacking groups over the levels of the tree.
    rows: int32 [B, stride] host slot rows; policy "cost" (groups estimated to pay) or "all";
    fold True (where estimated to pay), "always" or False. Returns (ranges [2 G], shared [G],
    start [G], level_indptr [L + 1], max_group_rows, fold [G], all_folded) as int32 numpy arrays
    (and an int and a bool); G = 0 when there is none."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    B = rows.shape[0]
    P, S = _i32(prefix_len), _i32(new_len)
    a = RcStackPlanArgs(num_reqs=B, rows=_p(rows), row_stride=rows.shape[1] if rows.ndim == 2 else 0,
                        prefix_len=_p(P), new_len=_p(S), min_shared=int(min_shared),
                        group_size=int(group), max_levels=int(max_levels),
                        policy={"cost": 0, "all": 1}[policy], fold=_FOLD_MODES[fold])
    cap = max(B * int(max_levels), 1)
    rng, sh, st, fo = (np.zeros(2 * cap, np.int32), np.zeros(cap, np.int32),
                       np.zeros(cap, np.int32), np.zeros(cap, np.int32))
    out = RcStackPlan(capacity=cap, group_range=_p(rng), group_shared=_p(sh), group_start=_p(st),
                      group_fold=_p(fo))
    check(lib().rc_plan_extend_stacking(ctypes.byref(a), ctypes.byref(out)),
          "rc_plan_extend_stacking")
    G, L = out.num_groups, out.num_levels
    return (rng[:2 * G].copy(), sh[:G].copy(), st[:G].copy(),
            np.asarray(out.level_indptr[:L + 1], np.int32), int(out.max_group_rows),
            fo[:G].copy(), bool(out.all_folded))


def shared_context_groups(rows, lengths, group_size: int, min_shared: int):
    """rc_plan_decode_groups: decode requests whose slot rows start with the same slots share
    that prefix's KV. rows: int32 [B, >= max(lengths)] host slot rows, lengths: context tokens
    per request. Returns (indptr, members, shared) int32 numpy arrays (no groups: [0] and two
    empty arrays)."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    L = np.ascontiguousarray(lengths, dtype=np.int64)
    B = len(L)
    indptr = np.zeros(B + 1, np.int32)
    members = np.zeros(max(B, 1), np.int32)
    shared = np.zeros(max(B, 1), np.int32)
    ng = ctypes.c_int32()
    check(lib().rc_plan_decode_groups(_p(rows), rows.shape[1] if rows.ndim == 2 else 0, _p(L),
                                      B, int(group_size), int(min_shared), _p(indptr),
                                      _p(members), _p(shared), ctypes.byref(ng)),
          "rc_plan_decode_groups")
    G = ng.value
    return indptr[:G + 1].copy(), members[:indptr[G]].copy(), shared[:G].copy()


STATIC_SCRATCH_BYTES = 32 << 20


def decode_attention_noalloc(q, k_new, v_new, out_loc, seq_len, req_idx, req_to_token, k_pool,
                             v_pool, o, *, sm_scale, max_total_tokens, kv_chunk=0, lse=None,
                             stream=None):
    """decode_attention without a workspace, for callers that cannot allocate device memory
    (see rc_decode_attention_noalloc): its scratch is a fixed STATIC_SCRATCH_BYTES area inside
    librc shared by every call on the device, so calls that overlap on the GPU race."""
    a = _decode_args(q, k_new, v_new, out_loc, seq_len, req_idx, req_to_token, k_pool, v_pool,
                     o, lse, sm_scale, max_total_tokens, kv_chunk)
    check(lib().rc_decode_attention_noalloc(ctypes.byref(a), _stream(stream)),
          "rc_decode_attention_noalloc")


def device_status(stream=None) -> int:
    """Read and clear the device status word (0 = no kernel reported bad data)."""
    v = ctypes.c_int32()
    check(lib().rc_device_status(ctypes.byref(v), _stream(stream)), "rc_device_status")
    return int(v.value)
