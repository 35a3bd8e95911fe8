"""ctypes declarations of librc's C ABI (include/rc.h). Argument marshalling only."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

RC_OK = 0
RC_ERR_INVALID = -1
RC_ERR_OOM = -2
RC_ERR_INSUFFICIENT = -3
RC_ERR_CUDA = -4
RC_ERR_DEVICE = -5
RC_DTYPE_BF16 = 0
RC_DTYPE_F32 = 1
RC_SCHED_LSPF = 0
RC_SCHED_FCFS = 1
RC_STACK_COST = 0
RC_STACK_ALL = 1
RC_FOLD_NONE = 0
RC_FOLD_COST = 1
RC_FOLD_ALL = 2
RC_MAX_STACK_LEVELS = 4

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64

# every function the header declares, with (restype, argtypes)
SIGNATURES = {
    "rc_last_error": (ctypes.c_char_p, []),
    "rc_launch_count": (_U64, []),
    "rc_pool_create": (ctypes.c_int, [_I64, _P, ctypes.POINTER(_P)]),
    "rc_pool_destroy": (None, [_P]),
    "rc_kv_pool_alloc": (ctypes.c_int, [_P, _I64, _P]),
    "rc_kv_pool_free": (ctypes.c_int, [_P, _P, _I64]),
    "rc_kv_pool_available": (ctypes.c_int, [_P, ctypes.POINTER(_I64)]),
    "rc_pool_inject_alloc_failure": (ctypes.c_int, [_P, _I64]),
    "rc_radix_create": (ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    "rc_radix_destroy": (None, [_P]),
    "rc_radix_match_prefix": (ctypes.c_int, [_P, _P, _I64, _P, ctypes.POINTER(_I64),
                                             ctypes.POINTER(_U64)]),
    "rc_radix_insert": (ctypes.c_int, [_P, _P, _P, _I64, ctypes.POINTER(_I64),
                                       ctypes.POINTER(_U64)]),
    "rc_radix_lock": (ctypes.c_int, [_P, _U64]),
    "rc_radix_unlock": (ctypes.c_int, [_P, _U64]),
    "rc_radix_evict_lru": (ctypes.c_int, [_P, _I64, ctypes.POINTER(_I64)]),
    "rc_radix_stats": (ctypes.c_int, [_P, _P]),
    "rc_radix_dump": (_I64, [_P, _P, _I64]),
    "rc_radix_match_batch": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I64, _P, _P]),
    "rc_radix_insert_batch": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I64, _P, _P, _I32, _P, _P]),
    "rc_radix_match_batch_tiered": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _I64, _P, _P, _P]),
    "rc_radix_attach_host_tier": (ctypes.c_int, [_P, _P]),
    "rc_radix_load_batch": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I64, _P, _P]),
    "rc_radix_pending_copies": (ctypes.c_int, [_P, _P, _P]),
    "rc_radix_drain_copies": (ctypes.c_int, [_P, _P, _P, _P, _P]),
    "rc_radix_tiers": (_I64, [_P, _P, _I64]),
    "rc_schedule_batch": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _I32, _I64, _I64, _P, _P,
                                         _P]),
    "rc_schedule_batch_ranges": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I64, _I64,
                                                _P, _P, _P]),
    "rc_slot_table_write": (ctypes.c_int, [_P, _P]),
    "rc_kv_copy": (ctypes.c_int, [_P, _P]),
    "rc_extend_workspace_bytes": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t)]),
    "rc_extend_attention": (ctypes.c_int, [_P, _P]),
    "rc_decode_workspace_bytes": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t)]),
    "rc_decode_attention": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P]),
    "rc_decode_attention_noalloc": (ctypes.c_int, [_P, _P]),
    "rc_device_status": (ctypes.c_int, [ctypes.POINTER(_I32), _P]),
    "rc_debug_set_wait_limit_ns": (ctypes.c_int, [_U64]),
    "rc_plan_extend_stacking": (ctypes.c_int, [_P, _P]),
    "rc_plan_decode_groups": (ctypes.c_int, [_P, _I64, _P, _I32, _I32, _I64, _P, _P, _P,
                                             ctypes.POINTER(_I32)]),
}


class RcStats(ctypes.Structure):
    _fields_ = [(n, _I64) for n in ("nodes", "cached_tokens", "evictable_tokens",
                                    "protected_tokens", "splits", "evicted_nodes",
                                    "evicted_tokens", "matched_tokens", "match_queries",
                                    "host_tokens", "spilled_tokens", "loaded_tokens",
                                    "dropped_tokens")]


class RcKvCopyArgs(ctypes.Structure):
    _fields_ = [("n", _I64), ("layers", _I32), ("row_bytes", _I64), ("src_slots", _P),
                ("dst_slots", _P), ("src_k", _P), ("src_v", _P), ("src_num_slots", _I64),
                ("dst_k", _P), ("dst_v", _P), ("dst_num_slots", _I64)]


class RcSlotWriteArgs(ctypes.Structure):
    _fields_ = [("num_segments", _I32), ("max_reqs", _I32), ("max_ctx", _I32),
                ("total_values", _I64), ("seg_row", _P), ("seg_col", _P), ("seg_indptr", _P),
                ("values", _P), ("req_to_token", _P)]


class RcStackPlanArgs(ctypes.Structure):
    _fields_ = [("num_reqs", _I32), ("rows", _P), ("row_stride", _I64), ("prefix_len", _P),
                ("new_len", _P), ("min_shared", _I32), ("group_size", _I32),
                ("max_levels", _I32), ("policy", _I32), ("fold", _I32)]


class RcStackPlan(ctypes.Structure):
    _fields_ = [("capacity", _I32), ("group_range", _P), ("group_shared", _P),
                ("group_start", _P), ("group_fold", _P),
                ("level_indptr", _I32 * (RC_MAX_STACK_LEVELS + 1)), ("num_groups", _I32),
                ("num_levels", _I32), ("max_group_rows", _I32), ("all_folded", _I32)]


class RcExtendArgs(ctypes.Structure):
    _fields_ = [("dtype", _I32), ("num_reqs", _I32), ("num_q_heads", _I32),
                ("num_kv_heads", _I32), ("head_dim", _I32), ("max_reqs", _I32),
                ("max_ctx", _I32), ("max_q_len", _I32), ("max_prefix_len", _I32), ("num_tokens", _I64),
                ("num_slots", _I64), ("sm_scale", ctypes.c_float), ("q", _P), ("k_new", _P),
                ("v_new", _P), ("out_loc", _P), ("qo_indptr", _P), ("prefix_len", _P),
                ("req_idx", _P), ("req_to_token", _P), ("k_pool", _P), ("v_pool", _P),
                ("o", _P), ("lse", _P), ("num_groups", _I32), ("max_group_rows", _I32),
                ("group_range", _P), ("group_shared", _P), ("workspace", _P),
                ("workspace_bytes", ctypes.c_size_t), ("num_levels", _I32),
                ("level_indptr", _P), ("group_start", _P), ("group_fold", _P),
                ("skip_request_pass", _I32)]


class RcDecodeArgs(ctypes.Structure):
    _fields_ = [("dtype", _I32), ("num_reqs", _I32), ("num_q_heads", _I32),
                ("num_kv_heads", _I32), ("head_dim", _I32), ("max_reqs", _I32),
                ("max_ctx", _I32), ("kv_chunk", _I32), ("max_total_tokens", _I64), ("num_slots", _I64),
                ("sm_scale", ctypes.c_float), ("q", _P), ("k_new", _P), ("v_new", _P),
                ("out_loc", _P), ("seq_len", _P), ("req_idx", _P), ("req_to_token", _P),
                ("k_pool", _P), ("v_pool", _P), ("o", _P), ("lse", _P),
                ("num_groups", _I32), ("group_indptr", _P), ("group_members", _P),
                ("group_shared", _P), ("reuse_plan", _I32)]


_lib = None


def lib(build_if_missing: bool = True):
    """The loaded librc. Builds it in-tree when missing (nvcc is needed); there is no fallback:
    without the library every call fails loudly."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"librc is not built ({path}); run prefix_cached_paged_gb300.build")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class RcError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().rc_last_error().decode(errors="replace")
        super().__init__(f"{where}: status {code}: {msg}")
        self.code = code


def check(code: int, where: str) -> int:
    if code != RC_OK:
        raise RcError(code, where)
    return code
