"""Prefix-shared, token-indexed KV attention for GB300 (sm_103a).

Thin Python binding of ``libpkv.so`` (C ABI in ``include/pkv.h``): every call below only
marshals arguments -- torch tensors supply device memory and streams, numpy arrays host
memory -- and forwards to the library.  Names follow the C entry points without the
``pkv_`` prefix:

    kv_store      scatter new K/V rows into pool slots (bf16 copy or fp8 quantisation)
    check_out_cache_loc  host check that a store's slots are in range and distinct
    plan_decode   host work decomposition of a decode call (split-KV, shared-prefix cascade)
    plan_extend   host work decomposition of an extend call
    attn_decode   one query token per request over its whole context (widely shared spans on
                  the tensor cores, the rest by a persistent bulk-copy kernel with mma.sync)
    attn_extend   causal extend of the uncached suffix (key gather, then tcgen05 / TMEM / TMA)
    attn_extend_store  kv_store + attn_extend in one call: the new rows are stored into the pool
                  and straight into the gathered rows (the gather reads cached positions only)
    plan_extend_ctx / attn_extend_ctx  chunked prefill over a caller-kept context buffer: each
                  chunk is stored into the pool and its context rows in one pass, nothing gathered
    RadixTree     host radix tree: match_prefix (with split), insert, LRU evict, lock_ref,
                  cascade extraction
    Allocator     token-slot free list

There is no CPU or eager fallback: importing the package loads the library or raises.
"""

from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from ._lib import (PKV_BF16, PKV_FP8_E4M3, PkvBatch, PkvCascade, PkvError, PkvPlanInfo, PkvPlanOpts, PkvPool,
                   check, lib)

__all__ = ["Pool", "Batch", "Plan", "Cascade", "kv_store", "check_out_cache_loc", "plan_decode", "plan_extend",
           "plan_extend_ctx", "attn_decode", "attn_extend", "attn_extend_store", "attn_extend_ctx", "get_device_error", "get_noalloc_device_error", "set_kernel_events",
           "set_wait_limit_ns", "get_wait_limit_ns", "fill_batch_table",
           "RadixTree", "Allocator", "PkvError", "version"]


def version() -> int:
    return lib.pkv_version()


def _ptr(t) -> int:
    """Device pointer of a torch tensor or host pointer of a numpy array (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ----------------------------------------------------------------------------------------
# pool, batch, plan


@dataclass
class Pool:
    """Device KV pool: k, v are torch tensors [num_slots, num_kv_heads, head_dim] of bfloat16
    (dtype 'bf16') or uint8 holding e4m3 codes (dtype 'fp8_e4m3') -- two dense arrays, or
    (layout 'interleaved') the K and V halves of one [num_slots, 2, num_kv_heads, head_dim]
    array, so a slot's K and V rows are one contiguous run."""
    k: object
    v: object
    dtype: str = "bf16"
    k_scale: float = 1.0
    v_scale: float = 1.0

    @classmethod
    def allocate(cls, num_slots, num_kv_heads, head_dim, dtype="bf16", k_scale=1.0, v_scale=1.0, device="cuda",
                 layout="separate"):
        import torch
        tdt = torch.bfloat16 if dtype == "bf16" else torch.uint8
        if layout == "interleaved":
            kv = torch.zeros((num_slots, 2, num_kv_heads, head_dim), dtype=tdt, device=device)
            k, v = kv[:, 0], kv[:, 1]
        elif layout == "separate":
            k = torch.zeros((num_slots, num_kv_heads, head_dim), dtype=tdt, device=device)
            v = torch.zeros_like(k)
        else:
            raise ValueError(f"unknown pool layout {layout!r}")
        return cls(k, v, dtype, float(k_scale), float(v_scale))

    @property
    def num_slots(self):
        return self.k.shape[0]

    @property
    def layout(self) -> str:
        return "separate" if self.k.stride(0) == self.k.shape[1] * self.k.shape[2] else "interleaved"

    def c(self) -> PkvPool:
        assert self.k.stride(0) == self.v.stride(0) and self.k.stride(1) == self.k.shape[2] and self.k.stride(2) == 1
        return PkvPool(_ptr(self.k), _ptr(self.v), self.k.shape[0], self.k.shape[1], self.k.shape[2],
                       PKV_BF16 if self.dtype == "bf16" else PKV_FP8_E4M3, self.k_scale, self.v_scale,
                       int(self.k.stride(0)))


@dataclass
class Batch:
    """Device batch tables: req_to_token [rows, stride] int32, req_pool_indices [B] int32,
    seq_lens [B] int32 (torch tensors on the GPU).  With page_size P > 1, req_to_token holds
    the page of each P-token block of a row (see pkv_batch)."""
    req_to_token: object
    req_pool_indices: object
    seq_lens: object
    page_size: int = 1

    def c(self) -> PkvBatch:
        rt = self.req_to_token
        return PkvBatch(_ptr(rt), rt.shape[1], rt.shape[0], _ptr(self.req_pool_indices), _ptr(self.seq_lens),
                        self.req_pool_indices.shape[0], int(self.page_size))


@dataclass
class Cascade:
    """Host description of the shared spans of a batch (see pkv_cascade in pkv.h)."""
    span_req: np.ndarray
    span_start: np.ndarray
    span_len: np.ndarray
    grp_indptr: np.ndarray
    grp_req: np.ndarray

    @property
    def num_spans(self):
        return int(self.span_req.shape[0])

    def c(self) -> PkvCascade:
        return PkvCascade(self.num_spans, _ptr(self.span_req), _ptr(self.span_start), _ptr(self.span_len),
                          _ptr(self.grp_indptr), _ptr(self.grp_req))


@dataclass
class Plan:
    info: PkvPlanInfo
    blob: np.ndarray  # uint8 host copy of the plan


def _opts(opts):
    if opts is None:
        return None
    o = PkvPlanOpts()
    for k, v in opts.items():
        setattr(o, k, int(v))
    return C.byref(o)


def _cascade_ref(cascade):
    if cascade is None:
        return None, None
    c = cascade.c()
    return C.byref(c), c


def plan_decode(seq_lens, num_q_heads, num_kv_heads, head_dim, cascade=None, opts=None) -> Plan:
    seq = _i32(seq_lens)
    info = PkvPlanInfo()
    cref, _keep = _cascade_ref(cascade)
    o = _opts(opts)
    args = (len(seq), _ptr(seq), num_q_heads, num_kv_heads, head_dim, cref, o)
    check("pkv_plan_decode", lib.pkv_plan_decode(*args, None, 0, C.byref(info)))
    blob = np.zeros(info.plan_bytes, dtype=np.uint8)
    check("pkv_plan_decode", lib.pkv_plan_decode(*args, _ptr(blob), blob.nbytes, C.byref(info)))
    return Plan(info, blob)


def plan_extend(seq_lens, extend_lens, qo_indptr, num_q_heads, num_kv_heads, head_dim, cascade=None,
                opts=None) -> Plan:
    seq, ext, qo = _i32(seq_lens), _i32(extend_lens), _i32(qo_indptr)
    info = PkvPlanInfo()
    cref, _keep = _cascade_ref(cascade)
    o = _opts(opts)
    args = (len(seq), _ptr(seq), _ptr(ext), _ptr(qo), num_q_heads, num_kv_heads, head_dim, cref, o)
    check("pkv_plan_extend", lib.pkv_plan_extend(*args, None, 0, C.byref(info)))
    blob = np.zeros(info.plan_bytes, dtype=np.uint8)
    check("pkv_plan_extend", lib.pkv_plan_extend(*args, _ptr(blob), blob.nbytes, C.byref(info)))
    return Plan(info, blob)


def plan_extend_ctx(seq_lens, extend_lens, qo_indptr, ctx_row0, ctx_rows, num_q_heads, num_kv_heads, head_dim,
                    opts=None) -> Plan:
    """Extend plan over a caller-kept context buffer (chunked prefill): request r's context
    position t is row ctx_row0[r] + t of the context arrays (see pkv_plan_extend_ctx)."""
    seq, ext, qo, row0 = _i32(seq_lens), _i32(extend_lens), _i32(qo_indptr), _i32(ctx_row0)
    info = PkvPlanInfo()
    o = _opts(opts)
    args = (len(seq), _ptr(seq), _ptr(ext), _ptr(qo), _ptr(row0), int(ctx_rows), num_q_heads, num_kv_heads,
            head_dim, o)
    check("pkv_plan_extend_ctx", lib.pkv_plan_extend_ctx(*args, None, 0, C.byref(info)))
    blob = np.zeros(info.plan_bytes, dtype=np.uint8)
    check("pkv_plan_extend_ctx", lib.pkv_plan_extend_ctx(*args, _ptr(blob), blob.nbytes, C.byref(info)))
    return Plan(info, blob)


# ----------------------------------------------------------------------------------------
# device calls


def kv_store(pool: Pool, k_new, v_new, out_cache_loc, workspace=None, stream=None) -> None:
    p = pool.c()
    check("pkv_kv_store", lib.pkv_kv_store(C.byref(p), _ptr(k_new), _ptr(v_new), _ptr(out_cache_loc),
                                           int(out_cache_loc.shape[0]), _ptr(workspace), _stream(stream)))


def fill_batch_table(cached, cached_len, fresh, fresh_len, table) -> None:
    """Row i of ``table`` (numpy int32 [n][stride], C-contiguous) = request i's cached slots,
    then its new slots (flat arrays with per-row lengths); the rest of each row is untouched."""
    assert table.dtype == np.int32 and table.flags["C_CONTIGUOUS"] and table.ndim == 2
    c, f = _i32(cached) if len(cached) else np.zeros(1, np.int32), _i32(fresh) if len(fresh) else np.zeros(1, np.int32)
    cl = np.ascontiguousarray(np.asarray(cached_len, dtype=np.int64))
    fl = np.ascontiguousarray(np.asarray(fresh_len, dtype=np.int64))
    assert len(cl) == len(fl) <= table.shape[0]
    check("pkv_fill_batch_table", lib.pkv_fill_batch_table(_ptr(c), _ptr(cl), _ptr(f), _ptr(fl), len(cl), _ptr(table),
                                                           table.shape[1]))


def check_out_cache_loc(out_cache_loc, num_slots) -> int:
    """Host check of kv_store's slot list (numpy int32 [n]): -1 when every slot is in range
    and distinct, else the index of the first entry that is out of range or repeats a slot."""
    loc = _i32(out_cache_loc)
    bad = C.c_int64(-1)
    rc = lib.pkv_check_out_cache_loc(_ptr(loc), len(loc), int(num_slots), C.byref(bad))
    if rc not in (0, -1) or (rc == -1 and bad.value < 0):
        check("pkv_check_out_cache_loc", rc)
    return bad.value


def attn_decode(pool: Pool, batch: Batch, q, o, sm_scale, plan: Plan, plan_dev, workspace, stream=None) -> None:
    p, b = pool.c(), batch.c()
    check("pkv_attn_decode", lib.pkv_attn_decode(C.byref(p), C.byref(b), _ptr(q), _ptr(o), float(sm_scale),
                                                 C.byref(plan.info), _ptr(plan_dev), _ptr(workspace),
                                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def attn_extend(pool: Pool, batch: Batch, q, o, sm_scale, plan: Plan, plan_dev, workspace, stream=None) -> None:
    p, b = pool.c(), batch.c()
    check("pkv_attn_extend", lib.pkv_attn_extend(C.byref(p), C.byref(b), _ptr(q), _ptr(o), float(sm_scale),
                                                 C.byref(plan.info), _ptr(plan_dev), _ptr(workspace),
                                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def attn_extend_store(pool: Pool, batch: Batch, q, o, sm_scale, k_new, v_new, out_cache_loc, plan: Plan, plan_dev,
                      workspace, stream=None) -> None:
    """kv_store of the call's new tokens and attn_extend in one call (a plan made with
    opts={"fuse_store": 1}): the new rows go to the pool and straight to their gathered rows."""
    p, b = pool.c(), batch.c()
    check("pkv_attn_extend_store", lib.pkv_attn_extend_store(
        C.byref(p), C.byref(b), _ptr(q), _ptr(o), float(sm_scale), _ptr(k_new), _ptr(v_new), _ptr(out_cache_loc),
        C.byref(plan.info), _ptr(plan_dev), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def attn_extend_ctx(pool: Pool, q, o, sm_scale, k_new, v_new, out_cache_loc, ctx_k, ctx_v, plan: Plan, plan_dev,
                    workspace, stream=None) -> None:
    """Store one chunk's new tokens (pool and context rows) and attend over the context arrays
    ctx_k / ctx_v (torch bf16 [ctx_rows, Hkv, d])."""
    p = pool.c()
    check("pkv_attn_extend_ctx", lib.pkv_attn_extend_ctx(
        C.byref(p), _ptr(q), _ptr(o), float(sm_scale), _ptr(k_new), _ptr(v_new), _ptr(out_cache_loc), _ptr(ctx_k),
        _ptr(ctx_v), int(ctx_k.shape[0]), C.byref(plan.info), _ptr(plan_dev), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def get_device_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns the raw error word (0 = no error)."""
    raw = C.c_int32(0)
    rc = lib.pkv_get_device_error(_ptr(workspace), _stream(stream), C.byref(raw))
    if rc not in (0, -7):
        check("pkv_get_device_error", rc)
    return raw.value


def get_noalloc_device_error(stream=None) -> int:
    """Synchronises the stream and returns the raw error word of attn_decode_noalloc's fixed
    array on the current device (0 = no error)."""
    raw = C.c_int32(0)
    rc = lib.pkv_get_noalloc_device_error(_stream(stream), C.byref(raw))
    if rc not in (0, -7):
        check("pkv_get_noalloc_device_error", rc)
    return raw.value


def set_wait_limit_ns(ns: int = 0) -> None:
    """Limit of every wait inside the attention kernels launched after this call (0 = the
    default, 2 s).  A tiny limit makes the kernels give up and report PKV_DERR_TIMEOUT."""
    check("pkv_set_wait_limit_ns", lib.pkv_set_wait_limit_ns(int(ns)))


def get_wait_limit_ns() -> int:
    return int(lib.pkv_get_wait_limit_ns())


def set_kernel_events(start=None, stop=None) -> None:
    """Times the attention kernel of the next attn_extend call alone: ``start`` / ``stop``
    (torch.cuda.Event with timing enabled) are recorded right before and after it."""
    def handle(ev):
        if ev is None:
            return None
        if not ev.cuda_event:       # torch creates the CUDA event on its first record
            ev.record()
        return C.c_void_p(ev.cuda_event)
    check("pkv_set_kernel_events", lib.pkv_set_kernel_events(handle(start), handle(stop)))


# ----------------------------------------------------------------------------------------
# host radix tree and allocator


class RadixTree:
    POLICIES = ("lru", "lfu", "slru", "fifo", "mru", "filo", "priority")   # = PKV_EVICT_* order

    def __init__(self, policy: str = "lru", page_size: int = 1):
        self._h = lib.pkv_tree_new()
        if not self._h:
            raise MemoryError("pkv_tree_new")
        self.page_size = int(page_size)
        if self.page_size != 1:
            check("pkv_tree_set_page_size", lib.pkv_tree_set_page_size(self._h, self.page_size))
        if policy != "lru":
            self.set_policy(policy)

    def set_policy(self, policy: str) -> None:
        check("pkv_tree_set_policy", lib.pkv_tree_set_policy(self._h, self.POLICIES.index(policy)))

    def __del__(self):
        if getattr(self, "_h", None):
            lib.pkv_tree_free(self._h)
            self._h = None

    def match_prefix(self, key):
        key = _i32(key)
        out = np.zeros(len(key), dtype=np.int32)
        matched, last = C.c_int64(0), C.c_int64(0)
        check("pkv_tree_match_prefix", lib.pkv_tree_match_prefix(self._h, _ptr(key), len(key), _ptr(out), len(out),
                                                                 C.byref(matched), C.byref(last)))
        return out[:matched.value], last.value

    def insert(self, key, value, priority: int = 0) -> int:
        key, value = _i32(key), _i32(value)
        assert len(key) == len(value)
        n = C.c_int64(0)
        check("pkv_tree_insert_priority", lib.pkv_tree_insert_priority(self._h, _ptr(key), _ptr(value), len(key),
                                                                       int(priority), C.byref(n)))
        return n.value

    def match_len(self, key) -> int:
        """Cached prefix length of ``key``; the tree is not changed."""
        key = _i32(key)
        n = C.c_int64(0)
        check("pkv_tree_match_len", lib.pkv_tree_match_len(self._h, _ptr(key), len(key), C.byref(n)))
        return n.value

    def schedule(self, queue, policy: str = "lpm"):
        """Admission order of ``queue`` (token lists): "lpm" longest cached prefix first (ties
        in queue order) or "fcfs"; returns (order, cached prefix lengths)."""
        offs = np.zeros(len(queue) + 1, dtype=np.int64)
        for i, q in enumerate(queue):
            offs[i + 1] = offs[i] + len(q)
        toks = _i32(np.concatenate([np.asarray(q, dtype=np.int32) for q in queue]) if queue else [])
        order = np.zeros(max(len(queue), 1), dtype=np.int32)
        lens = np.zeros(max(len(queue), 1), dtype=np.int64)
        check("pkv_schedule", lib.pkv_schedule(self._h, _ptr(toks), _ptr(offs), len(queue),
                                               {"lpm": 0, "fcfs": 1}[policy], _ptr(order), _ptr(lens)))
        return order[:len(queue)].tolist(), lens[:len(queue)].tolist()

    def sizes(self):
        e, p, t, n = C.c_int64(0), C.c_int64(0), C.c_int64(0), C.c_int64(0)
        check("pkv_tree_sizes", lib.pkv_tree_sizes(self._h, C.byref(e), C.byref(p), C.byref(t), C.byref(n)))
        return {"evictable": e.value, "protected": p.value, "total": t.value, "nodes": n.value}

    def evict(self, num_tokens: int) -> np.ndarray:
        cap = self.sizes()["evictable"]
        out = np.zeros(max(cap, 1), dtype=np.int32)
        n = C.c_int64(0)
        check("pkv_tree_evict", lib.pkv_tree_evict(self._h, int(num_tokens), _ptr(out), len(out), C.byref(n)))
        return out[:n.value].copy()

    def match_lock_batch(self, keys, flat: bool = False):
        """match_prefix then inc_lock_ref of the last node, for every key in order, in one native
        call.  Returns (list of matched value arrays, int64 array of last nodes), or with
        ``flat`` (all matched values back to back, int64 matched lengths, last nodes)."""
        n = len(keys)
        off = np.zeros(n + 1, dtype=np.int64)
        if n:
            np.cumsum([len(k) for k in keys], out=off[1:])
        key_flat = _i32(np.concatenate([np.asarray(k, dtype=np.int32) for k in keys])) if n and off[-1] else \
            np.zeros(1, dtype=np.int32)
        values = np.zeros(max(int(off[-1]), 1), dtype=np.int32)
        matched = np.zeros(max(n, 1), dtype=np.int64)
        last = np.zeros(max(n, 1), dtype=np.int64)
        check("pkv_tree_match_lock_batch", lib.pkv_tree_match_lock_batch(self._h, _ptr(key_flat), _ptr(off), n, _ptr(values),
                                                                         _ptr(matched), _ptr(last)))
        if flat:
            return values[:int(matched[:n].sum())], matched[:n], last[:n]
        ends = np.cumsum(matched[:n])
        return [values[e - m:e] for e, m in zip(ends, matched[:n])], last[:n]

    def inc_lock_ref(self, node: int) -> int:
        d = C.c_int64(0)
        check("pkv_tree_inc_lock_ref", lib.pkv_tree_inc_lock_ref(self._h, int(node), C.byref(d)))
        return d.value

    def dec_lock_ref(self, node: int) -> int:
        d = C.c_int64(0)
        check("pkv_tree_dec_lock_ref", lib.pkv_tree_dec_lock_ref(self._h, int(node), C.byref(d)))
        return d.value

    def dump(self):
        """[(id, parent, lock_ref, time, key tuple, value tuple, num_children, hit_count, priority)]
        in id order."""
        used = C.c_int64(0)
        check("pkv_tree_dump", lib.pkv_tree_dump(self._h, None, 0, C.byref(used)))
        buf = np.zeros(max(used.value, 1), dtype=np.int64)
        check("pkv_tree_dump", lib.pkv_tree_dump(self._h, _ptr(buf), len(buf), C.byref(used)))
        rows, i = [], 0
        while i < used.value:
            nid, par, lock, t, n, nch, hits, prio = (int(x) for x in buf[i:i + 8])
            key = tuple(int(x) for x in buf[i + 8:i + 8 + n])
            val = tuple(int(x) for x in buf[i + 8 + n:i + 8 + 2 * n])
            rows.append((nid, par, lock, t, key, val, nch, hits, prio))
            i += 8 + 2 * n
        return rows

    def cascade(self, last_nodes, min_group: int = 2) -> Cascade:
        last = np.ascontiguousarray(np.asarray(last_nodes, dtype=np.int64))
        ns, nm = C.c_int32(0), C.c_int32(0)
        check("pkv_tree_cascade", lib.pkv_tree_cascade(self._h, _ptr(last), len(last), min_group, None, None, None,
                                                       None, None, 0, 0, C.byref(ns), C.byref(nm)))
        s, m = ns.value, nm.value
        sr, ss, sl = (np.zeros(s, np.int32) for _ in range(3))
        ip, gr = np.zeros(s + 1, np.int32), np.zeros(max(m, 1), np.int32)
        check("pkv_tree_cascade", lib.pkv_tree_cascade(self._h, _ptr(last), len(last), min_group, _ptr(sr), _ptr(ss),
                                                       _ptr(sl), _ptr(ip), _ptr(gr), s, m, C.byref(ns),
                                                       C.byref(nm)))
        return Cascade(sr, ss, sl, ip, gr[:m])


class Allocator:
    """FIFO free list of pool slots."""

    def __init__(self, free_slots):
        fs = _i32(free_slots)
        self._h = lib.pkv_allocator_new(_ptr(fs), len(fs))
        if not self._h:
            raise MemoryError("pkv_allocator_new")

    def __del__(self):
        if getattr(self, "_h", None):
            lib.pkv_allocator_free_all(self._h)
            self._h = None

    def alloc(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 1), dtype=np.int32)
        check("pkv_allocator_alloc", lib.pkv_allocator_alloc(self._h, int(n), _ptr(out)))
        return out[:n]

    def release(self, slots) -> None:
        s = _i32(slots)
        check("pkv_allocator_release", lib.pkv_allocator_release(self._h, _ptr(s), len(s)))

    @property
    def available(self) -> int:
        return int(lib.pkv_allocator_available(self._h))
