"""ctypes declarations of libpkv.so (include/pkv.h).  Argument marshalling only.

Importing this module loads the in-tree library and fails loudly when it is missing: there
is no fallback implementation of any entry point.
"""

from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

PKV_OK = 0
PKV_BF16 = 0
PKV_FP8_E4M3 = 1

ERRORS = {
    0: "ok", -1: "invalid argument", -2: "unsupported shape or dtype", -3: "workspace or buffer too small",
    -4: "CUDA error", -5: "no free KV slots", -6: "unknown tree node", -7: "device-side check failed",
    -8: "plan does not match the call",
}


class PkvPool(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("num_slots", C.c_int64), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("dtype", C.c_int32), ("k_scale", C.c_float), ("v_scale", C.c_float),
                ("slot_stride", C.c_int64)]


class PkvBatch(C.Structure):
    _fields_ = [("req_to_token", C.c_void_p), ("stride", C.c_int64), ("num_rows", C.c_int32),
                ("req_pool_indices", C.c_void_p), ("seq_lens", C.c_void_p), ("batch", C.c_int32),
                ("page_size", C.c_int32)]


class PkvCascade(C.Structure):
    _fields_ = [("num_spans", C.c_int32), ("span_req", C.c_void_p), ("span_start", C.c_void_p),
                ("span_len", C.c_void_p), ("grp_indptr", C.c_void_p), ("grp_req", C.c_void_p)]


class PkvPlanOpts(C.Structure):
    _fields_ = [("chunk_keys", C.c_int32), ("span_chunk", C.c_int32), ("num_sms", C.c_int32),
                ("dynamic_tail", C.c_int32), ("span_sms", C.c_int32), ("fuse_store", C.c_int32)]


class PkvPlanInfo(C.Structure):
    _fields_ = [("op", C.c_int32), ("batch", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("num_items", C.c_int32), ("num_span_items", C.c_int32),
                ("num_records", C.c_int32), ("num_merge", C.c_int32), ("total_q", C.c_int32),
                ("plan_bytes", C.c_size_t), ("workspace_bytes", C.c_size_t), ("offsets", C.c_int64 * 24)]


_P = C.c_void_p
_I32 = C.c_int32
_I64 = C.c_int64
_SZ = C.c_size_t
_F = C.c_float
_PI64 = C.POINTER(C.c_int64)
_PI32 = C.POINTER(C.c_int32)

SIGNATURES = {
    "pkv_strerror": (C.c_char_p, [C.c_int]),
    "pkv_version": (C.c_int, []),
    "pkv_kv_store": (C.c_int, [C.POINTER(PkvPool), _P, _P, _P, _I64, _P, _P]),
    "pkv_check_out_cache_loc": (C.c_int, [_P, _I64, _I64, _PI64]),
    "pkv_plan_decode": (C.c_int, [_I32, _P, _I32, _I32, _I32, C.POINTER(PkvCascade), C.POINTER(PkvPlanOpts), _P, _SZ,
                                  C.POINTER(PkvPlanInfo)]),
    "pkv_plan_extend": (C.c_int, [_I32, _P, _P, _P, _I32, _I32, _I32, C.POINTER(PkvCascade),
                                  C.POINTER(PkvPlanOpts), _P, _SZ, C.POINTER(PkvPlanInfo)]),
    "pkv_plan_extend_ctx": (C.c_int, [_I32, _P, _P, _P, _P, _I64, _I32, _I32, _I32, C.POINTER(PkvPlanOpts), _P, _SZ,
                                      C.POINTER(PkvPlanInfo)]),
    "pkv_attn_extend_store": (C.c_int, [C.POINTER(PkvPool), C.POINTER(PkvBatch), _P, _P, _F, _P, _P, _P,
                                        C.POINTER(PkvPlanInfo), _P, _P, _SZ, _P]),
    "pkv_attn_extend_ctx": (C.c_int, [C.POINTER(PkvPool), _P, _P, _F, _P, _P, _P, _P, _P, _I64,
                                      C.POINTER(PkvPlanInfo), _P, _P, _SZ, _P]),
    "pkv_attn_decode": (C.c_int, [C.POINTER(PkvPool), C.POINTER(PkvBatch), _P, _P, _F, C.POINTER(PkvPlanInfo), _P,
                                  _P, _SZ, _P]),
    "pkv_attn_extend": (C.c_int, [C.POINTER(PkvPool), C.POINTER(PkvBatch), _P, _P, _F, C.POINTER(PkvPlanInfo), _P,
                                  _P, _SZ, _P]),
    "pkv_get_device_error": (C.c_int, [_P, _P, _PI32]),
    "pkv_set_kernel_events": (C.c_int, [_P, _P]),
    "pkv_set_wait_limit_ns": (C.c_int, [C.c_uint64]),
    "pkv_get_wait_limit_ns": (C.c_uint64, []),
    "pkv_attn_decode_noalloc": (C.c_int, [C.POINTER(PkvPool), C.POINTER(PkvBatch), _P, _P, _F,
                                          C.POINTER(PkvPlanInfo), _P, _P]),
    "pkv_get_noalloc_device_error": (C.c_int, [_P, _PI32]),
    "pkv_tree_new": (_P, []),
    "pkv_tree_free": (None, [_P]),
    "pkv_tree_match_prefix": (C.c_int, [_P, _P, _I64, _P, _I64, _PI64, _PI64]),
    "pkv_tree_insert": (C.c_int, [_P, _P, _P, _I64, _PI64]),
    "pkv_tree_insert_priority": (C.c_int, [_P, _P, _P, _I64, _I64, _PI64]),
    "pkv_tree_set_policy": (C.c_int, [_P, C.c_int]),
    "pkv_tree_set_page_size": (C.c_int, [_P, _I32]),
    "pkv_tree_match_len": (C.c_int, [_P, _P, _I64, _PI64]),
    "pkv_schedule": (C.c_int, [_P, _P, _P, _I32, C.c_int, _P, _P]),
    "pkv_tree_evict": (C.c_int, [_P, _I64, _P, _I64, _PI64]),
    "pkv_tree_inc_lock_ref": (C.c_int, [_P, _I64, _PI64]),
    "pkv_tree_match_lock_batch": (C.c_int, [_P, _P, _P, _I32, _P, _P, _P]),
    "pkv_fill_batch_table": (C.c_int, [_P, _P, _P, _P, _I32, _P, _I64]),
    "pkv_tree_dec_lock_ref": (C.c_int, [_P, _I64, _PI64]),
    "pkv_tree_sizes": (C.c_int, [_P, _PI64, _PI64, _PI64, _PI64]),
    "pkv_tree_dump": (C.c_int, [_P, _P, _I64, _PI64]),
    "pkv_tree_cascade": (C.c_int, [_P, _P, _I32, _I32, _P, _P, _P, _P, _P, _I32, _I32, _PI32, _PI32]),
    "pkv_allocator_new": (_P, [_P, _I64]),
    "pkv_allocator_free_all": (None, [_P]),
    "pkv_allocator_alloc": (C.c_int, [_P, _I64, _P]),
    "pkv_allocator_release": (C.c_int, [_P, _P, _I64]),
    "pkv_allocator_available": (C.c_int64, [_P]),
}


class PkvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {ERRORS.get(code, 'error')} ({code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python prefix_shared_kv_token_gb300/build.py, or "
            "__graft_entry__.build()); there is no fallback implementation")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def check(fn: str, code: int) -> None:
    if code != PKV_OK:
        raise PkvError(fn, code)
