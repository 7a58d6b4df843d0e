"""Host side of one serving step: prefix-cache population, batch tables, cascade, plans and
device buffers for the kv_store + attention calls.

A *workload* (see ``workloads/``) describes token segments with their K/V rows and a batch
of requests whose contexts are paths of segments; the last ``n_new`` tokens of each context
are new in the step.  :class:`PrefixCache` owns the device pool, the radix tree and the
slot allocator; :meth:`PrefixCache.populate` caches every request's already-cached part the
way a server would have after earlier steps (match, allocate the unmatched rest, store its
K/V, insert), and :meth:`PrefixCache.prepare` builds one attention call (extend or decode):
match the cached part (it must hit completely), lock the path, allocate slots for the new
tokens (``out_cache_loc``), write ``req_to_token`` rows, extract the shared-prefix cascade
from the tree and plan the kernels.  Everything runs through ``libpkv`` (tree, allocator,
planner, kernels); this module only moves arrays around.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import (Allocator, Batch, Pool, RadixTree, attn_decode, attn_extend, attn_extend_ctx, attn_extend_store,
               check_out_cache_loc, fill_batch_table, kv_store, plan_decode, plan_extend, plan_extend_ctx)


def _ctx_tokens(w, req):
    return np.concatenate([w.segments[s].tokens for s in req.path])


def _ctx_kv(w, req, lo, hi):
    """bf16 bits of context rows [lo, hi) of K and V, as [n, Hkv, d] uint16 arrays."""
    ks, vs, pos = [], [], 0
    for s in req.path:
        seg = w.segments[s]
        n = len(seg.tokens)
        a, b = max(lo, pos), min(hi, pos + n)
        if a < b:
            ks.append(seg.k[a - pos:b - pos])
            vs.append(seg.v[a - pos:b - pos])
        pos += n
    if not ks:
        shape = (0, w.num_kv_heads, w.head_dim)
        return np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    return np.concatenate(ks), np.concatenate(vs)


def _bf16_dev(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


@dataclass
class Call:
    """One attention call of a step with all its device inputs."""
    kind: str
    pool: Pool
    batch: Batch
    plan: object
    plan_dev: torch.Tensor
    workspace: torch.Tensor
    q: torch.Tensor
    o: torch.Tensor
    out_cache_loc: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    sm_scale: float
    last_nodes: list
    host: dict = field(default_factory=dict)
    cascade: object = None
    contexts: list = field(default_factory=list)   # per request: (tokens, req_to_token row, cached length)
    requests: list = field(default_factory=list)
    graph: object = None                           # captured attention launches (capture_attend)
    ctx: tuple = None                              # (ctx_k, ctx_v): a chunk over a context buffer
    fused: bool = False                            # extend: the attention call stores the new rows

    @property
    def num_queries(self) -> int:
        return int(self.q.shape[0])

    def layer(self, pool: Pool, w, ctx=None) -> "Call":
        """The same call for another layer of the model: that layer's pool, and its queries and
        new K/V rows from ``w`` (a workload of the same structure whose requests match this
        call's one for one).  Tables, plan and slots are shared by all layers; a chunk over a
        context buffer takes that layer's context arrays ``ctx`` = (ctx_k, ctx_v)."""
        if (self.ctx is None) != (ctx is None):
            raise ValueError("a context-buffer call needs the layer's context arrays (and only it does)")
        reqs = [w.requests[r.rid] for r in self.requests]
        kn, vn = [], []
        for r, (_, row, cached) in zip(reqs, self.contexts):
            kb, vb = _ctx_kv(w, r, cached, len(row))
            kn.append(kb)
            vn.append(vb)
        dev = self.q.device
        q = _bf16_dev(np.concatenate([r.q for r in reqs]), dev)
        return Call(self.kind, pool, self.batch, self.plan, self.plan_dev, torch.zeros_like(self.workspace), q,
                    torch.empty_like(q), self.out_cache_loc, _bf16_dev(np.concatenate(kn), dev),
                    _bf16_dev(np.concatenate(vn), dev), w.sm_scale, self.last_nodes, cascade=self.cascade,
                    contexts=self.contexts, requests=reqs, ctx=ctx, fused=self.fused)

    def store(self, stream=None):
        if self.ctx is not None or self.fused:
            return  # stored inside the attention call
        kv_store(self.pool, self.k_new, self.v_new, self.out_cache_loc, self.workspace, stream)

    def attend(self, stream=None):
        if self.fused:
            attn_extend_store(self.pool, self.batch, self.q, self.o, self.sm_scale, self.k_new, self.v_new,
                              self.out_cache_loc, self.plan, self.plan_dev, self.workspace, stream)
            return
        if self.ctx is not None:
            attn_extend_ctx(self.pool, self.q, self.o, self.sm_scale, self.k_new, self.v_new, self.out_cache_loc,
                            self.ctx[0], self.ctx[1], self.plan, self.plan_dev, self.workspace, stream)
            return
        f = attn_extend if self.kind == "extend" else attn_decode
        f(self.pool, self.batch, self.q, self.o, self.sm_scale, self.plan, self.plan_dev, self.workspace, stream)

    def run(self, stream=None):
        self.store(stream)
        self.attend(stream)

    def capture_attend(self):
        """Record this call's attention launches once into a CUDA graph; :meth:`replay_attend`
        then re-issues them with one launch (same plan, tables, buffers and workspace, as in
        a decode loop whose plan is reused).  The library is called on a side stream while
        capturing, exactly as :meth:`attend` calls it."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.attend()          # resolve lazy set-up outside the capture
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            self.attend()
        self.graph = g

    def replay_attend(self):
        self.graph.replay()

    def launches(self) -> int:
        """Kernels one run() launches: the store, then the attention call's kernels."""
        info = self.plan.info
        n = 1 if self.out_cache_loc.numel() > 0 else 0
        if self.ctx is not None:                                 # store (with the context rows),
            n = 1 if self.out_cache_loc.numel() > 0 else 0       # then the extend kernel(s)
            nprec = int(info.offsets[10])
            n += (1 if info.num_items - nprec > 0 else 0) + (1 if nprec > 0 else 0)
        elif self.kind == "extend":                              # (a fused call's store is its own
            nprec = int(info.offsets[10])                        # launch, counted above)
            n += (1 if info.offsets[5] > 0 else 0)               # key gather
            n += (1 if info.num_items - nprec > 0 else 0) + (1 if nprec > 0 else 0)  # extend kernel(s)
        else:
            nx, nprec = int(info.offsets[8]), int(info.offsets[18])
            if nx > 0:                                           # tensor-core pass: one gather, then
                n += 1 + (1 if nx - nprec > 0 else 0) + (1 if nprec > 0 else 0)  # span / short items
            n += 1 if info.num_items > 0 else 0                  # decode kernel
        return n + (1 if info.num_merge > 0 else 0)

    # ---- end-to-end variant: inputs from pinned host buffers, output back to the host
    def pin_host(self):
        h = self.host
        for name in ("q", "k_new", "v_new", "out_cache_loc"):
            t = getattr(self, name)
            h[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        for name in ("req_to_token", "req_pool_indices", "seq_lens"):
            t = getattr(self.batch, name)
            h[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        h["plan"] = torch.from_numpy(self.plan.blob).pin_memory()
        h["o"] = torch.empty(self.o.shape, dtype=self.o.dtype, pin_memory=True)

    def h2d_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for k, v in self.host.items() if k != "o")

    def d2h_bytes(self) -> int:
        return self.o.numel() * self.o.element_size()

    def copy_in(self):
        """Host -> device copies of the call's inputs (on the current stream)."""
        h = self.host
        for name in ("q", "k_new", "v_new", "out_cache_loc"):
            getattr(self, name).copy_(h[name], non_blocking=True)
        for name in ("req_to_token", "req_pool_indices", "seq_lens"):
            getattr(self.batch, name).copy_(h[name], non_blocking=True)
        self.plan_dev.copy_(h["plan"], non_blocking=True)

    def copy_out(self, host_o=None):
        """Device -> host copy of the call's output (on the current stream)."""
        (self.host["o"] if host_o is None else host_o).copy_(self.o, non_blocking=True)

    def run_e2e(self, stream=None):
        self.copy_in()
        self.run(stream)
        self.copy_out()

    def e2e_sets(self, n: int = 2) -> list:
        """``n`` copies of this call with their own device inputs and output (the first is
        this call itself), sharing the pool, plan, workspace and host buffers: the buffers a
        pipelined end-to-end loop fills and drains while another copy computes."""
        out = [self]
        for _ in range(n - 1):
            b = self.batch
            batch = Batch(torch.empty_like(b.req_to_token), torch.empty_like(b.req_pool_indices),
                          torch.empty_like(b.seq_lens), b.page_size)
            c = Call(self.kind, self.pool, batch, self.plan, torch.empty_like(self.plan_dev), self.workspace,
                     torch.empty_like(self.q), torch.empty_like(self.o), torch.empty_like(self.out_cache_loc),
                     torch.empty_like(self.k_new), torch.empty_like(self.v_new), self.sm_scale, self.last_nodes,
                     host=self.host, cascade=self.cascade, contexts=self.contexts, requests=self.requests,
                     ctx=self.ctx, fused=self.fused)
            out.append(c)
        return out


def run_e2e_pipelined(sets, steps: int, flush=None):
    """End-to-end steps with the copies overlapped: step k's inputs go host -> device on one
    copy stream while step k-1 computes, and step k-1's output goes device -> host on another
    while step k computes.  ``sets`` holds, per call of a step, the buffer copies from
    :meth:`Call.e2e_sets` (step k uses copy k mod n).  Every step's own copies happen inside
    the returned span.  ``flush`` (a device tensor) is zeroed on the compute stream before each
    step's kernels, inside the span.  Returns the elapsed milliseconds (CUDA events)."""
    n = len(sets[0])
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    loaded = [torch.cuda.Event() for _ in range(n)]
    done = [torch.cuda.Event() for _ in range(n)]
    free = [torch.cuda.Event() for _ in range(n)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    cin.wait_event(start)
    cout.wait_event(start)
    for k in range(steps):
        b = k % n
        with torch.cuda.stream(cin):
            if k >= n:
                cin.wait_event(free[b])       # copy b's previous step has been read back
            for calls in sets:
                calls[b].copy_in()
            loaded[b].record(cin)
        comp.wait_event(loaded[b])
        if flush is not None:
            flush.zero_()
        for calls in sets:
            calls[b].run()
        done[b].record(comp)
        with torch.cuda.stream(cout):
            cout.wait_event(done[b])
            for calls in sets:
                calls[b].copy_out()
            free[b].record(cout)
    comp.wait_stream(cout)
    end.record(comp)
    end.synchronize()
    return start.elapsed_time(end)


class PrefixCache:
    """Device pool + host radix tree + slot allocator for one workload's shapes.

    ``page_size`` P > 1 makes a paged pool: the allocator hands out pages of P slots, the
    tree caches whole P-token blocks only, every block of a request's context lives in one
    page (slot = page * P + position % P), and the batch tables are page tables.  A
    request's trailing partial block is its own (``private``): it is not in the tree, and
    the request's next tokens fill the rest of that page before new pages are taken.

    ``check_slots`` runs the host check of every call's ``out_cache_loc`` (slots in range and
    distinct, kv_store's precondition) before anything is copied to the device.
    ``kv_layout``: "interleaved" (a slot's K and V rows adjacent: decode reads both with one
    copy) or "separate" (two dense arrays).  ``fuse_store``: extend calls store their new
    rows themselves (pool and gathered rows in one pass) instead of a separate kv_store."""

    def __init__(self, w, device="cuda", page_size=1, check_slots=True, kv_layout="interleaved", fuse_store=True):
        self.w = w
        self.check_slots = bool(check_slots)
        self.fuse_store = bool(fuse_store)
        self.device = device
        self.page = int(page_size)
        self.pool = Pool.allocate(w.num_slots, w.num_kv_heads, w.head_dim, w.dtype, w.k_scale, w.v_scale, device,
                                  layout=kv_layout)
        self.tree = RadixTree(page_size=self.page)
        self.alloc = Allocator(w.slot_perm if self.page == 1 else w.page_perm(self.page))
        self.private = {}   # paged pool: request id -> slots of its trailing partial block
        self._tokens = {}   # request id -> its context tokens (the workload's, fixed)
        self.err = torch.zeros(64, dtype=torch.int32, device=device)

    # ---- slots of positions
    def _extend_slots(self, slots, n):
        """Slots for the next ``n`` positions of a context whose first len(slots) positions
        use ``slots``: fresh slots, or in a paged pool the rest of the last page, then new pages."""
        if self.page == 1:
            return self.alloc.alloc(n)
        P, L0 = self.page, len(slots)
        out = []
        if L0 % P and n > 0:
            page = int(slots[-1]) // P
            take = min(n, P - L0 % P)
            out.append(page * P + np.arange(L0 % P, L0 % P + take, dtype=np.int32))
            n -= take
        if n > 0:
            pages = self.alloc.alloc((n + P - 1) // P)
            out.append((pages[:, None].astype(np.int64) * P + np.arange(P)).reshape(-1)[:n].astype(np.int32))
        return np.concatenate(out) if out else np.zeros(0, np.int32)

    def _release_blocks(self, row, lo, hi):
        """Give back the slots of positions [lo, hi) of ``row`` (whole blocks in a paged pool)."""
        if hi <= lo:
            return
        if self.page == 1:
            self.alloc.release(row[lo:hi])
        else:
            self.alloc.release(np.asarray(row[lo:hi:self.page]) // self.page)

    def _table(self, rows, seq):
        """Batch table of the rows: slots per position, or pages per block."""
        B, P = len(rows), self.page
        if P == 1:
            stride = max(16, ((max(seq) if len(seq) else 1) + 15) // 16 * 16)
            rt = np.zeros((max(B, 1), stride), dtype=np.int32)
            for i, row in enumerate(rows):
                rt[i, :len(row)] = row
            return rt
        nb = max(1, max(((len(r) + P - 1) // P for r in rows), default=1))
        rt = np.zeros((max(B, 1), (nb + 3) // 4 * 4), dtype=np.int32)
        for i, row in enumerate(rows):
            pages = np.asarray(row[::P], dtype=np.int64) // P
            # every block must sit in one page, in position order
            want = (pages.repeat(P)[:len(row)] * P + np.arange(len(row)) % P).astype(np.int32)
            if not np.array_equal(want, row):
                raise RuntimeError("a context block is not one page of the pool")
            rt[i, :len(pages)] = pages
        return rt

    # ---- cache population (setup, not part of a step)
    def populate(self, max_batch_tokens=1 << 18):
        w = self.w
        ks, vs, locs, pending = [], [], [], 0
        for r in w.requests:
            toks = _ctx_tokens(w, r)
            c = len(toks) - r.n_new
            vals, _ = self.tree.match_prefix(toks[:c])
            m = len(vals)
            if m == c:
                continue
            new = self._extend_slots(vals, c - m)
            kb, vb = _ctx_kv(w, r, m, c)
            ks.append(kb)
            vs.append(vb)
            locs.append(new)
            pending += c - m
            row = np.concatenate([vals, new]).astype(np.int32)
            pre = self.tree.insert(toks[:c], row)
            assert pre == m, (pre, m)
            if self.page > 1:   # the trailing partial block stays with the request
                self.private[r.rid] = row[c // self.page * self.page:c]
            if pending >= max_batch_tokens:
                self._store(ks, vs, locs)
                ks, vs, locs, pending = [], [], [], 0
        if ks:
            self._store(ks, vs, locs)
        torch.cuda.synchronize()

    def _store(self, ks, vs, locs):
        k = _bf16_dev(np.concatenate(ks), self.device)
        v = _bf16_dev(np.concatenate(vs), self.device)
        loc = torch.from_numpy(np.concatenate(locs).astype(np.int32)).to(self.device)
        kv_store(self.pool, k, v, loc, self.err)

    # ---- one attention call of a step
    def _plan_host(self, kind, cascade, opts, min_group, requests, ctx_base=None):
        """The host half of one call: match every request's cached part in the tree (it must hit
        completely) and lock its path, allocate slots for the new tokens, build the batch table,
        extract the cascade and plan the kernels.  Returns a dict of host arrays."""
        w = self.w
        reqs = [r for r in (w.requests if requests is None else requests) if r.kind == kind]
        rows, last_nodes, seq, ext, new_all = [], [], [], [], []
        toks_all = []
        for r in reqs:
            t = self._tokens.get(r.rid)
            if t is None:
                t = self._tokens[r.rid] = _ctx_tokens(w, r)
            toks_all.append(t)
        rt = None
        if self.page == 1:
            # one native call matches and locks every request's cached part, in order; the new
            # tokens' slots come from one FIFO allocation, split in request order (the same
            # slots as one allocation per request); one more fills the batch table, and each
            # request's slot row is a view of its table row
            cached = np.fromiter((len(t) - r.n_new for t, r in zip(toks_all, reqs)), dtype=np.int64,
                                 count=len(reqs))
            vals_flat, matched, last_all = self.tree.match_lock_batch(
                [t[:c] for t, c in zip(toks_all, cached.tolist())], flat=True)
            if not np.array_equal(matched, cached):
                i = int(np.nonzero(matched != cached)[0][0])
                for n in last_all:
                    self.tree.dec_lock_ref(int(n))
                raise RuntimeError(f"request {reqs[i].rid}: cached part not fully in the tree "
                                   f"({int(matched[i])} of {int(cached[i])})")
            n_new = np.fromiter((r.n_new for r in reqs), dtype=np.int64, count=len(reqs))
            new_flat = self.alloc.alloc(int(n_new.sum()))
            seq = (cached + n_new).tolist()
            stride = max(16, ((max(seq) if seq else 1) + 15) // 16 * 16)
            rt = np.zeros((max(len(reqs), 1), stride), dtype=np.int32)
            fill_batch_table(vals_flat, matched, new_flat, n_new, rt)
            ends = np.cumsum(n_new)
            rows = [rt[i, :L] for i, L in enumerate(seq)]
            new_all = [new_flat[e - n:e] for e, n in zip(ends.tolist(), n_new.tolist())]
            last_nodes = [int(n) for n in last_all]
            ext = n_new.tolist()
        else:
            for r, toks in zip(reqs, toks_all):
                L, c = len(toks), len(toks) - r.n_new
                vals, last = self.tree.match_prefix(toks[:c])
                # whole blocks from the tree, the partial one from the request
                vals = np.concatenate([vals, self.private.get(r.rid, np.zeros(0, np.int32))]).astype(np.int32)
                if len(vals) != c:
                    raise RuntimeError(f"request {r.rid}: cached part not fully in the tree ({len(vals)} of {c})")
                self.tree.inc_lock_ref(last)
                new = self._extend_slots(vals, r.n_new)
                rows.append(np.concatenate([vals, new]).astype(np.int32))
                last_nodes.append(last)
                seq.append(L)
                ext.append(r.n_new)
                new_all.append(new)
        B = len(reqs)
        if rt is None:
            rt = self._table(rows, seq)
        seq = np.asarray(seq, dtype=np.int32)
        ext = np.asarray(ext, dtype=np.int32)
        casc = self.tree.cascade(last_nodes, min_group) if (cascade and B > 1) else None
        if casc is not None and casc.num_spans == 0:
            casc = None
        hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
        if ctx_base is not None:   # chunks over a context buffer: rows by prompt, no cascade
            casc = None
            qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
            row0 = [ctx_base["row0"][r.path[0]] for r in reqs]
            plan = plan_extend_ctx(seq, ext, qo, row0, ctx_base["rows"], hq, hkv, d, opts)
        elif kind == "extend":
            qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
            if self.fuse_store:
                opts = dict(opts or {}, fuse_store=1)
            plan = plan_extend(seq, ext, qo, hq, hkv, d, casc, opts)
        else:
            plan = plan_decode(seq, hq, hkv, d, casc, opts)
        loc_host = np.concatenate(new_all).astype(np.int32) if new_all else np.zeros(0, np.int32)
        if self.page == 1:
            loc_host = np.ascontiguousarray(new_flat, dtype=np.int32)
        if self.check_slots:
            bad = check_out_cache_loc(loc_host, self.pool.num_slots)
            if bad >= 0:
                raise RuntimeError(f"out_cache_loc[{bad}] = {loc_host[bad]} is out of range or repeats a slot")
        return {"reqs": reqs, "rows": rows, "last_nodes": last_nodes, "seq": seq, "ext": ext, "new": new_all,
                "rt": rt, "cascade": casc, "plan": plan, "loc": loc_host}

    def host_step_ms(self, kind, reps=5, cascade=True, opts=None, min_group=2, requests=None) -> float:
        """Host time of planning one call like :meth:`prepare` (tree match and lock, slot
        allocation, batch table, cascade, plan, slot check), in ms, the mean of ``reps`` runs:
        what a server pays on the host for every new batch before its kernels can start.  Each
        run's slots and locks are given back, so the cache holds the same nodes, tokens and
        free slots afterwards (access times and hit counts move, as any match moves them).
        Token pools only (a paged pool's partial pages are not given back)."""
        import time
        if self.page != 1:
            raise ValueError("host_step_ms: token pools only")
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            h = self._plan_host(kind, cascade, opts, min_group, requests)
            ts.append(time.perf_counter() - t0)
            for new in h["new"]:
                if len(new):
                    self.alloc.release(new)
            for n in h["last_nodes"]:
                self.tree.dec_lock_ref(n)
        return 1e3 * float(np.mean(ts))

    def prepare(self, kind, cascade=True, opts=None, min_group=2, requests=None, ctx=None) -> Call:
        """One attention call over the workload's requests of ``kind`` (or the given subset).
        ``ctx`` (from :meth:`context_buffer`): an extend chunk over that context buffer."""
        w = self.w
        h = self._plan_host(kind, cascade, opts, min_group, requests, ctx_base=ctx)
        reqs, rows, plan = h["reqs"], h["rows"], h["plan"]
        kn, vn = [], []
        for r, row in zip(reqs, rows):
            kb, vb = _ctx_kv(w, r, len(row) - r.n_new, len(row))
            kn.append(kb)
            vn.append(vb)
        B = len(reqs)
        dev = self.device
        batch = Batch(torch.from_numpy(h["rt"]).to(dev), torch.arange(B, dtype=torch.int32, device=dev),
                      torch.from_numpy(h["seq"]).to(dev), self.page)
        plan_dev = torch.from_numpy(plan.blob).to(dev)
        ws = torch.zeros((plan.info.workspace_bytes + 3) // 4, dtype=torch.int32, device=dev)
        q = _bf16_dev(np.concatenate([r.q for r in reqs]), dev)
        o = torch.empty_like(q)
        loc = torch.from_numpy(h["loc"]).to(dev)
        k_new = _bf16_dev(np.concatenate(kn), dev)
        v_new = _bf16_dev(np.concatenate(vn), dev)
        call = Call(kind, self.pool, batch, plan, plan_dev, ws, q, o, loc, k_new, v_new, w.sm_scale,
                    h["last_nodes"], cascade=h["cascade"],
                    ctx=None if ctx is None else (ctx["k"], ctx["v"]),
                    fused=kind == "extend" and ctx is None and self.fuse_store)
        call.contexts = [(_ctx_tokens(w, r), row, len(row) - r.n_new) for r, row in zip(reqs, rows)]
        call.requests = reqs
        return call

    def release(self, call: Call):
        for n in call.last_nodes:
            self.tree.dec_lock_ref(n)

    def context_buffer(self):
        """Context arrays for chunked prefill: one run of rows per prompt (the requests under one
        root segment), as long as its longest context; bf16 [rows, Hkv, d] for K and for V."""
        w = self.w
        length = {}
        for r in w.requests:
            length[r.path[0]] = max(length.get(r.path[0], 0), w.context_len(r))
        row0, rows = {}, 0
        for root in sorted(length):
            row0[root] = rows
            rows += length[root]
        k = torch.zeros((max(rows, 1), w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device=self.device)
        return {"k": k, "v": torch.zeros_like(k), "row0": row0, "rows": max(rows, 1)}

    def prepare_chunked(self, opts=None, fused=True) -> list:
        """Chunked prefill of a workload whose ``meta["chunk"]`` numbers each extend request's
        step: one call per step, planned over the chunks the earlier steps cached.  The tree
        learns each step's tokens when the step is planned (host only), so all the calls can be
        planned ahead; run them in order.  ``fused``: every call stores its chunk into the pool
        and into a context buffer shared by the calls, and attends over that buffer (nothing
        is gathered); else each call's store is separate and its attention gathers the whole
        context from the pool."""
        steps = self.w.meta["chunk"]
        ctx = self.context_buffer() if fused else None
        self.ctx = ctx
        calls = []
        for c in sorted(set(steps)):
            reqs = [r for r, k in zip(self.w.requests, steps) if k == c]
            call = self.prepare("extend", opts=opts, requests=reqs, ctx=ctx)
            self.commit(call)
            calls.append(call)
        return calls

    def commit(self, call: Call):
        """After the call ran: cache every request's whole context (its new tokens join the
        tree with the slots they were stored in) and unlock its path, as a server does when a
        prefill chunk or a request finishes."""
        P = self.page
        for (toks, row, cached), n, r in zip(call.contexts, call.last_nodes, call.requests):
            pre = self.tree.insert(toks, row)
            lo = cached // P * P   # the tree held the request's blocks up to here
            if pre > lo:           # another request of the call inserted the same new tokens first
                self._release_blocks(row, lo, pre)
            if P > 1:
                L = len(row)
                self.private[r.rid] = row[L // P * P:L]
            self.tree.dec_lock_ref(n)
