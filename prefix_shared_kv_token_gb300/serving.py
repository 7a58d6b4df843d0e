"""Multi-step serving over the prefix cache: cache-aware admission, LRU eviction under memory
pressure, prefill (extend) and decode steps, and a decode plan reused across steps.

The loop follows the pages' account of the runtime: requests whose prefix is longest in the
radix tree are admitted first ("Efficiently Programming Large Language Models using SGLang"
summary, §Cache-Aware Scheduling); only the uncached remainder of a prompt is prefilled
(§RadixAttention); when the pool is short of slots, unlocked leaves are evicted least
recently used first and the paths of running requests are locked ("[SGLang] RadixAttention
...", "Eviction 전략", "참조 카운트: lock_ref"); a finished request's whole sequence is
inserted into the tree, where later requests can hit it.

Every step the host (C++ tree, scheduler and planner through ``libpkv``) decides the batch
and the device runs attn_extend_store for the admitted prompts (their new rows stored by the
extend call itself) and kv_store + attn_decode for one new token of every running request.  The decode plan is made with
``dynamic_tail`` (each request's last item reads its end from the device ``seq_lens``), so it
stays valid while the running set is unchanged and is only re-planned when a request joins
or leaves.  Synthetic inputs come from the seeded generators in ``workloads``: the K/V of a
context entry depends only on (token, position), so shared prefixes share K/V exactly.

With ``page_size`` P > 1 the pool is paged: slots come in pages of P, the tree caches whole
P-token blocks only (a cached length is a multiple of P; a fully cached prompt recomputes its
whole last block), every block of a request lives in one page, and the batch table is a
page table written once at admission.  A request's trailing partial block is its own and is
freed when it finishes.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import (Allocator, Batch, Pool, RadixTree, attn_decode, attn_extend_store, kv_store, plan_decode,
               plan_extend)


def _bf16(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


@dataclass
class _Running:
    req: object                  # the stream request
    row: int                     # its req_to_token row
    slots: np.ndarray            # pool slots of prompt + outputs (outputs reserved at admission)
    last_node: int               # locked end of its cached path
    tokens: list = field(default_factory=list)   # prompt, then generated tokens
    gen: int = 0


@dataclass
class StepRecord:
    """One attention call of a step, for checking: the requests, the query positions of each,
    their context tokens, and the outputs (bf16, [queries, Hq, d])."""
    kind: str
    rids: list
    positions: list
    contexts: list
    o: torch.Tensor


class ServingSim:
    def __init__(self, stream, capacity: int, policy: str = "lpm", max_running: int = 64,
                 prefill_budget: int = 16384, device: str = "cuda", record: bool = False,
                 eviction: str = "lru", chunk_keys: int = 0, page_size: int = 1):
        self.s = stream
        self.policy = policy
        self.max_running = max_running
        self.prefill_budget = prefill_budget
        self.device = device
        self.record = record
        self.opts = {"dynamic_tail": 1, **({"chunk_keys": chunk_keys} if chunk_keys else {})}
        s = stream
        self.pool = Pool.allocate(capacity, s.num_kv_heads, s.head_dim, "bf16", device=device, layout="interleaved")
        self.page = P = int(page_size)
        self.tree = RadixTree(eviction, page_size=P)
        self.alloc = Allocator(np.arange(capacity // P, dtype=np.int32))   # slots, or pages
        longest = max(len(r.prompt) + r.out_len for r in s.requests)
        self.stride = (longest + 15) // 16 * 16
        self.rt = torch.zeros((max_running, self.stride if P == 1 else (longest + P - 1) // P), dtype=torch.int32,
                              device=device)
        self.seq = torch.zeros(max_running, dtype=torch.int32, device=device)
        self.free_rows = list(range(max_running - 1, -1, -1))
        self.pending = sorted(s.requests, key=lambda r: (r.arrival, r.rid))
        self.waiting, self.running, self.records = [], [], []
        self.step_no = 0
        self.stats = {"prompt_tokens": 0, "cached_tokens": 0, "prefill_tokens": 0, "decode_tokens": 0,
                      "finished": 0, "evicted_tokens": 0, "plans": 0, "device_ms": 0.0, "steps": 0}
        self._decode = None          # (running rids, plan, plan_dev, workspace, batch)
        self._ev = []
        self._err_words = []      # the header words of every call's workspace, checked after the run
        self._plans = []

    # ---- slots ---------------------------------------------------------------------
    def _ensure(self, n: int) -> bool:
        """Room for n more positions (n fresh slots, or ceil(n / P) fresh pages)."""
        P = self.page
        short = (n + P - 1) // P - self.alloc.available
        if short > 0:
            freed = self.tree.evict(short * P)
            if len(freed):
                self._free(freed)
                self.stats["evicted_tokens"] += len(freed)
        return self.alloc.available * P >= n

    def _take(self, n: int) -> np.ndarray:
        """Slots of n positions that start a block: fresh slots, or whole fresh pages."""
        P = self.page
        if P == 1:
            return self.alloc.alloc(n)
        pages = self.alloc.alloc((n + P - 1) // P).astype(np.int64)
        return (pages[:, None] * P + np.arange(P)).reshape(-1)[:n].astype(np.int32)

    def _free(self, slots) -> None:
        """Give back slots that cover whole blocks (whole pages in a paged pool)."""
        slots = np.asarray(slots)
        self.alloc.release(slots if self.page == 1 else slots[::self.page] // self.page)

    def _write_row(self, run) -> None:
        """A paged pool's table row: the page of every block of prompt + outputs."""
        P = self.page
        pages = np.asarray(run.slots[::P], np.int64) // P
        self.rt[run.row, :len(pages)] = torch.from_numpy(pages.astype(np.int32)).to(self.device)

    # ---- one step ------------------------------------------------------------------
    def done(self) -> bool:
        return not (self.pending or self.waiting or self.running)

    def step(self):
        while self.pending and self.pending[0].arrival <= self.step_no:
            self.waiting.append(self.pending.pop(0))
        admitted = self._admit()
        if admitted:
            self._prefill(admitted)
        if self.running:
            self._decode_step()
        self._finish()
        self.step_no += 1
        self.stats["steps"] += 1

    def run(self, max_steps: int = 100000):
        while not self.done() and self.step_no < max_steps:
            self.step()
        torch.cuda.synchronize()
        self.stats["device_ms"] = sum(a.elapsed_time(b) for a, b in self._ev)
        # every call's error word (kernels only set it): a range or timeout flag fails the run
        if self._err_words:
            words = torch.stack(self._err_words).cpu()
            bad = (words[:, 0] != 0).nonzero()
            if len(bad):
                k = int(bad[0, 0])
                info = self._plans[k].info
                code, w1, w2, w3 = (int(x) for x in words[k, :4])
                if code & 0x200:    # a pipeline wait gave up (low byte: which wait)
                    where = f"wait site {code & 0xFF}"
                elif code & 0x400 and info.op == 2:   # the fused store: token and context row
                    where = f"token {w1} / context row {w2}, or a work item outside its row"
                else:
                    where = f"header words {[w1, w2, w3]}"
                raise RuntimeError(f"a kernel of the serving run set its error word: {code:#x} (call {k}, op "
                                   f"{info.op}, {where}; plan: {info.num_items} items, "
                                   f"{int(info.offsets[10])} of them in the second list)")
        return self.stats

    # ---- admission: scheduler order, lock the cached path, reserve slots ----------------
    def _admit(self):
        if not self.waiting or len(self.running) >= self.max_running:
            return []
        order, _ = self.tree.schedule([r.prompt for r in self.waiting], self.policy)
        admitted, taken, budget = [], set(), self.prefill_budget
        for i in order:
            if len(self.running) + len(admitted) >= self.max_running:
                break
            r = self.waiting[i]
            vals, node = self.tree.match_prefix(r.prompt)
            # a fully cached prompt still recomputes its last token (the step's first query);
            # in a paged pool its whole last block, so the new positions start a block
            cached = min(len(vals), len(r.prompt) - 1) if self.page == 1 else \
                (len(vals) if len(vals) < len(r.prompt) else len(vals) - self.page)
            new = len(r.prompt) - cached
            if new > budget and admitted:   # an oversized prompt goes alone, first in line
                continue
            self.tree.inc_lock_ref(node)
            if not self._ensure(new + r.out_len):
                self.tree.dec_lock_ref(node)
                continue
            slots = np.concatenate([vals[:cached], self._take(new + r.out_len)]).astype(np.int32)
            admitted.append((_Running(r, self.free_rows.pop(), slots, node, list(r.prompt)), cached))
            taken.add(i)
            budget -= new
            self.stats["prompt_tokens"] += len(r.prompt)
            self.stats["cached_tokens"] += cached
        self.waiting = [r for i, r in enumerate(self.waiting) if i not in taken]
        return admitted

    # ---- prefill of the admitted prompts' uncached parts --------------------------------
    def _prefill(self, admitted):
        import workloads as W
        s, dev = self.s, self.device
        seq, ext, rows, locs, ks, vs, qs, nodes = [], [], [], [], [], [], [], []
        for run, cached in admitted:
            L = len(run.req.prompt)
            if self.page == 1:
                self.rt[run.row, :L] = torch.from_numpy(run.slots[:L]).to(dev)
            else:
                self._write_row(run)
            seq.append(L)
            ext.append(L - cached)
            rows.append(run.row)
            locs.append(run.slots[cached:L])
            k, v = W.token_kv(s.seed, run.req.prompt[cached:], range(cached, L), s.num_kv_heads, s.head_dim)
            ks.append(k)
            vs.append(v)
            qs.append(np.stack([W.stream_query(s.seed, run.req.rid, p, s.num_q_heads, s.head_dim)
                                for p in range(cached, L)]))
            nodes.append(run.last_node)
        seq = np.asarray(seq, np.int32)
        ext = np.asarray(ext, np.int32)
        qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
        casc = self.tree.cascade(nodes, 2) if len(nodes) > 1 else None
        if casc is not None and casc.num_spans == 0:
            casc = None
        plan = plan_extend(seq, ext, qo, s.num_q_heads, s.num_kv_heads, s.head_dim, casc, {"fuse_store": 1})
        self.seq[rows] = torch.from_numpy(seq).to(dev)
        batch = Batch(self.rt, torch.tensor(rows, dtype=torch.int32, device=dev), self.seq[rows].contiguous(),
                      self.page)
        q = _bf16(np.concatenate(qs), dev)
        o = torch.empty_like(q)
        ws = torch.zeros((plan.info.workspace_bytes + 3) // 4, dtype=torch.int32, device=dev)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record()
        # the prompts' new rows are stored by the attention call itself (pool and gathered rows)
        attn_extend_store(self.pool, batch, q, o, s.sm_scale, _bf16(np.concatenate(ks), dev),
                          _bf16(np.concatenate(vs), dev), torch.from_numpy(np.concatenate(locs)).to(dev), plan,
                          torch.from_numpy(plan.blob).to(dev), ws)
        ev[1].record()
        self._ev.append(ev)
        self._err_words.append(ws[:4].clone())
        self._plans.append(plan)
        self.stats["prefill_tokens"] += int(ext.sum())
        if self.record:
            self.records.append(StepRecord("extend", [run.req.rid for run, _ in admitted],
                                           [list(range(c, len(run.req.prompt))) for run, c in admitted],
                                           [run.req.prompt for run, _ in admitted], o))
        # the prompts join the tree; each request locks its whole prompt path instead
        for run, cached in admitted:
            L = len(run.req.prompt)
            pre = self.tree.insert(run.req.prompt, run.slots[:L])
            vals, node = self.tree.match_prefix(run.req.prompt)
            if pre > cached:   # another admitted prompt inserted the same tokens first: use its slots
                mine = run.slots[cached:pre].copy()
                run.slots[:len(vals)] = vals
                if self.page == 1:
                    self.rt[run.row, :L] = torch.from_numpy(run.slots[:L]).to(dev)
                else:
                    self._write_row(run)
                torch.cuda.current_stream().synchronize()   # our copies of those rows are still being read
                self._free(mine)
            self.tree.inc_lock_ref(node)
            self.tree.dec_lock_ref(run.last_node)
            run.last_node = node
            self.running.append(run)
        self._decode = None   # the running set changed

    # ---- one decode token for every running request ---------------------------------
    def _decode_step(self):
        import workloads as W
        s, dev = self.s, self.device
        runs = self.running
        if self._decode is None:
            seq = np.array([len(r.tokens) + 1 for r in runs], np.int32)
            casc = self.tree.cascade([r.last_node for r in runs], 2) if len(runs) > 1 else None
            if casc is not None and casc.num_spans == 0:
                casc = None
            plan = plan_decode(seq, s.num_q_heads, s.num_kv_heads, s.head_dim, casc, self.opts)
            rows = torch.tensor([r.row for r in runs], dtype=torch.int32, device=dev)
            ws = torch.zeros((plan.info.workspace_bytes + 3) // 4, dtype=torch.int32, device=dev)
            self._decode = (plan, torch.from_numpy(plan.blob).to(dev), ws, rows)
            self.stats["plans"] += 1
        plan, plan_dev, ws, rows = self._decode
        toks, pos, locs, ks, vs, qs = [], [], [], [], [], []
        for r in runs:
            p = len(r.tokens)
            t = W.generated_token(s.seed, r.req.rid, r.gen)
            toks.append(t)
            pos.append(p)
            locs.append(r.slots[p])
            k, v = W.token_kv(s.seed, [t], [p], s.num_kv_heads, s.head_dim)
            ks.append(k)
            vs.append(v)
            qs.append(W.stream_query(s.seed, r.req.rid, p, s.num_q_heads, s.head_dim)[None])
        locs_t = torch.tensor(locs, dtype=torch.int32, device=dev)
        if self.page == 1:   # a page table already names every reserved position's page
            self.rt[rows.long(), torch.tensor(pos, device=dev)] = locs_t
        seq_now = torch.tensor([p + 1 for p in pos], dtype=torch.int32, device=dev)
        self.seq[rows.long()] = seq_now
        batch = Batch(self.rt, rows, seq_now, self.page)
        q = _bf16(np.concatenate(qs), dev)
        o = torch.empty_like(q)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record()
        kv_store(self.pool, _bf16(np.concatenate(ks), dev), _bf16(np.concatenate(vs), dev), locs_t, ws)
        attn_decode(self.pool, batch, q, o, s.sm_scale, plan, plan_dev, ws)
        ev[1].record()
        self._ev.append(ev)
        self._err_words.append(ws[:4].clone())
        self._plans.append(plan)
        self.stats["decode_tokens"] += len(runs)
        if self.record:
            self.records.append(StepRecord("decode", [r.req.rid for r in runs], [[p] for p in pos],
                                           [r.tokens + [t] for r, t in zip(runs, toks)], o))
        for r, t in zip(runs, toks):
            r.tokens.append(t)
            r.gen += 1

    # ---- finished requests: cache the whole sequence, unlock, free the table row ---------
    def _finish(self):
        keep = []
        for r in self.running:
            if r.gen < r.req.out_len:
                keep.append(r)
                continue
            n, P = len(r.tokens), self.page
            pre = self.tree.insert(np.asarray(r.tokens, np.int32), r.slots[:n])
            lo = len(r.req.prompt) // P * P   # the tree held the request's blocks up to here
            if pre > lo:   # generated tokens already cached by another request
                torch.cuda.current_stream().synchronize()
                self._free(r.slots[lo:pre])
            if n % P:      # the trailing partial block is not in the tree: its page is free now
                torch.cuda.current_stream().synchronize()
                self._free(r.slots[n // P * P:n // P * P + 1])
            self.tree.dec_lock_ref(r.last_node)
            self.free_rows.append(r.row)
            self.stats["finished"] += 1
        if len(keep) != len(self.running):
            self._decode = None
        self.running = keep

    def summary(self) -> dict:
        st = dict(self.stats)
        st["hit_rate"] = st["cached_tokens"] / max(st["prompt_tokens"], 1)
        st["tokens"] = st["prefill_tokens"] + st["decode_tokens"]
        st["tokens_per_s_device"] = st["tokens"] / max(st["device_ms"], 1e-9) * 1e3
        return st
