"""Seeded generators for the five synthetic workloads and for small variants of them.

A workload is a forest of token *segments* (each with its own K/V values, one
row per token) and a batch of *requests*.  A request's context is the
concatenation of the segments on its path from a root-level segment down to
its leaf segment; the last ``n_new`` tokens of that context are new in this
step (their K/V are written to the pool by ``kv_store``), everything before is
already cached.  Extend requests query every new token, decode requests query
their single new token (the last token of the context).

Identical prefixes carry identical K/V because they are the same segments,
which is what a causal model produces for an identical token prefix.  Sibling
segments always start with different tokens, so a radix tree built over the
contexts has exactly the branching written down here.

Values: Q, K and V are N(0, 1) drawn in float32 and rounded to bf16 (round to
nearest even); arrays hold the raw bf16 bit patterns as ``uint16``.  Token ids
are uniform in [0, 32000).  Slot numbers handed out by an allocator come from
``Workload.slot_perm``, a seeded permutation of the pool.

The random draws happen in a fixed order (slot permutation, then segments in
creation order -- tokens, K, V -- then queries in request order), so a given
seed always yields the same workload.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

VOCAB = 32000

CONFIG_NAMES = {
    1: "tiny_decode",
    2: "fewshot_extend",
    3: "batched_decode",
    4: "multiturn_decode",
    5: "tot_mixed_fp8",
}


@dataclass
class Segment:
    sid: int
    parent: int            # -1 for a segment hanging off the root
    tokens: np.ndarray     # int32 [n]
    k: np.ndarray          # uint16 bf16 bits [n, Hkv, d]
    v: np.ndarray          # uint16 bf16 bits [n, Hkv, d]


@dataclass
class Request:
    rid: int
    path: list             # segment ids, root-level segment first
    n_new: int             # trailing context tokens that are new in this step
    kind: str              # "extend" or "decode"
    q: np.ndarray          # uint16 bf16 bits [n_q, Hq, d]; n_q = n_new (extend) or 1 (decode)


@dataclass
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_slots: int
    dtype: str             # "bf16" or "fp8_e4m3"
    k_scale: float         # per-tensor fp8 scales (1.0 for a bf16 pool)
    v_scale: float
    sm_scale: float        # float32(1/sqrt(d)) widened to a Python float
    segments: list
    requests: list
    slot_perm: np.ndarray  # int32 permutation of [0, num_slots)
    meta: dict = field(default_factory=dict)

    def page_perm(self, page_size: int) -> np.ndarray:
        """Seeded permutation of the pool's pages of ``page_size`` slots (a paged pool's
        free list; drawn from its own stream, so the workload's other draws are unchanged)."""
        rng = np.random.default_rng([self.seed, 2, page_size])
        return rng.permutation(self.num_slots // page_size).astype(np.int32)

    def context_len(self, req: Request) -> int:
        return int(sum(len(self.segments[s].tokens) for s in req.path))

    def extend_requests(self):
        return [r for r in self.requests if r.kind == "extend"]

    def decode_requests(self):
        return [r for r in self.requests if r.kind == "decode"]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def context_tokens(w: Workload, req: Request) -> np.ndarray:
    return np.concatenate([w.segments[s].tokens for s in req.path])


def context_kv_bits(w: Workload, req: Request):
    k = np.concatenate([w.segments[s].k for s in req.path], axis=0)
    v = np.concatenate([w.segments[s].v for s in req.path], axis=0)
    return k, v


class _Builder:
    def __init__(self, seed: int, hq: int, hkv: int, d: int, num_slots: int):
        self.rng = np.random.default_rng(seed)
        self.hq, self.hkv, self.d = hq, hkv, d
        self.slot_perm = self.rng.permutation(num_slots).astype(np.int32)
        self.segments: list[Segment] = []
        self.requests: list[Request] = []
        self._first = {}

    def segment(self, parent: int, n: int) -> int:
        assert n >= 1
        toks = self.rng.integers(0, VOCAB, size=n).astype(np.int32)
        used = self._first.setdefault(parent, set())
        while int(toks[0]) in used:
            toks[0] = np.int32(self.rng.integers(0, VOCAB))
        used.add(int(toks[0]))
        shape = (n, self.hkv, self.d)
        k = to_bf16_bits(self.rng.standard_normal(shape, dtype=np.float32))
        v = to_bf16_bits(self.rng.standard_normal(shape, dtype=np.float32))
        self.segments.append(Segment(len(self.segments), parent, toks, k, v))
        return len(self.segments) - 1

    def path_to(self, sid: int) -> list:
        path = []
        while sid != -1:
            path.append(sid)
            sid = self.segments[sid].parent
        return path[::-1]

    def request(self, leaf: int, kind: str, n_new: int):
        n_q = n_new if kind == "extend" else 1
        q = to_bf16_bits(self.rng.standard_normal((n_q, self.hq, self.d), dtype=np.float32))
        self.requests.append(Request(len(self.requests), self.path_to(leaf), n_new, kind, q))

    def finish(self, name, seed, num_slots, dtype="bf16", meta=None) -> Workload:
        k_scale = v_scale = 1.0
        if dtype == "fp8_e4m3":
            amax_k = max(float(np.abs(_bits_f32(s.k)).max()) for s in self.segments)
            amax_v = max(float(np.abs(_bits_f32(s.v)).max()) for s in self.segments)
            k_scale = float(np.float32(amax_k) / np.float32(448.0))
            v_scale = float(np.float32(amax_v) / np.float32(448.0))
        sm_scale = float(np.float32(1.0) / np.sqrt(np.float32(self.d)))
        return Workload(name, seed, self.hq, self.hkv, self.d, num_slots, dtype, k_scale, v_scale,
                        sm_scale, self.segments, self.requests, self.slot_perm, meta or {})


def _bits_f32(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------------------
# the five workloads, each parameterised so tests can run scaled-down versions


def tiny_decode(seed=1, n_req=4, prefix=64, unique=16, hq=8, hkv=2, d=64, num_slots=256):
    """Decode batch: ``n_req`` requests share a ``prefix``-token segment and each owns a
    ``unique``-token tail whose last token is the query."""
    b = _Builder(seed, hq, hkv, d, num_slots)
    root = b.segment(-1, prefix)
    leaves = [b.segment(root, unique) for _ in range(n_req)]
    for leaf in leaves:
        b.request(leaf, "decode", 1)
    return b.finish("tiny_decode", seed, num_slots)


def fewshot_extend(seed=2, n_req=64, prefix=1800, suffix=200, hq=32, hkv=8, d=128,
                   num_slots=1 << 21, dtype="bf16"):
    """Extend batch: ``n_req`` requests share a cached ``prefix``-token segment (few-shot
    examples) and each extends its own ``suffix`` new tokens, causally."""
    b = _Builder(seed, hq, hkv, d, num_slots)
    root = b.segment(-1, prefix)
    leaves = [b.segment(root, suffix) for _ in range(n_req)]
    for leaf in leaves:
        b.request(leaf, "extend", suffix)
    return b.finish("fewshot_extend", seed, num_slots, dtype)


def batched_decode(seed=3, n_req=256, prefix=2048, lo=128, hi=1024, hq=32, hkv=8, d=128,
                   num_slots=1 << 21, dtype="bf16"):
    """Decode batch: a shared ``prefix``-token system prompt, then a unique tail of
    U[lo, hi] tokens per request (query token last)."""
    b = _Builder(seed, hq, hkv, d, num_slots)
    root = b.segment(-1, prefix)
    lens = b.rng.integers(lo, hi + 1, size=n_req)
    leaves = [b.segment(root, int(n)) for n in lens]
    for leaf in leaves:
        b.request(leaf, "decode", 1)
    return b.finish("batched_decode", seed, num_slots, dtype)


def multiturn_decode(seed=4, n_conv=64, turns=4, user=(300, 600), reply=(100, 400), per_turn=2,
                     hq=32, hkv=8, d=128, num_slots=1 << 21, dtype="bf16"):
    """Multi-turn chat: each conversation's history is the chain U1 R1 U2 R2 ... U_turns.
    For every turn t, ``per_turn`` sibling queries decode a fresh reply to U_t: each owns a
    partial reply of P ~ U[1, R_t] tokens (query token last), branching off after U_t."""
    b = _Builder(seed, hq, hkv, d, num_slots)
    leaves = []
    for _ in range(n_conv):
        u_len = b.rng.integers(user[0], user[1] + 1, size=turns)
        r_len = b.rng.integers(reply[0], reply[1] + 1, size=turns)
        parent = -1
        u_nodes = []
        for t in range(turns):
            u = b.segment(parent, int(u_len[t]))
            u_nodes.append(u)
            parent = b.segment(u, int(r_len[t])) if t + 1 < turns else u
        for t in range(turns):
            for _j in range(per_turn):
                p = int(b.rng.integers(1, int(r_len[t]) + 1))
                leaves.append(b.segment(u_nodes[t], p))
    for leaf in leaves:
        b.request(leaf, "decode", 1)
    return b.finish("multiturn_decode", seed, num_slots, dtype)


def tot_mixed(seed=5, root_len=4096, depth=3, branch=4, seg=256, n_new_branches=16,
              hq=32, hkv=8, d=128, num_slots=1 << 21, dtype="fp8_e4m3"):
    """Tree of thought: a ``root_len`` root, a depth-``depth`` tree with ``branch`` children
    per node and ``seg``-token segments.  Every leaf decodes one token; in the same batch one
    new child under each of the first ``n_new_branches`` depth-(depth-1) nodes extends
    ``seg`` new tokens."""
    b = _Builder(seed, hq, hkv, d, num_slots)
    root = b.segment(-1, root_len)
    level = [root]
    parents_of_leaves = []
    for lvl in range(depth):
        nxt = []
        for p in level:
            for _ in range(branch):
                nxt.append(b.segment(p, seg))
        if lvl == depth - 1:
            parents_of_leaves = level
        level = nxt
    leaves = level
    new_leaves = [b.segment(p, seg) for p in parents_of_leaves[:n_new_branches]]
    for leaf in new_leaves:
        b.request(leaf, "extend", seg)
    for leaf in leaves:
        b.request(leaf, "decode", 1)
    return b.finish("tot_mixed_fp8", seed, num_slots, dtype)


def chunked_prefill(seed=6, n_req=16, prompt=8192, chunk=1024, hq=32, hkv=8, d=128, num_slots=1 << 21,
                    dtype="bf16"):
    """Long prompts prefilled chunk by chunk: prompt i is a chain of ``chunk``-token segments
    (the last one shorter when ``chunk`` does not divide ``prompt``), with one extend request
    per segment.  Step c runs the c-th request of every prompt, over that prompt's earlier
    chunks, which steps 0 .. c-1 cached.  ``meta["chunk"]`` gives each request's step."""
    b = _Builder(seed, hq, hkv, d, num_slots)
    steps = []
    for _ in range(n_req):
        parent, pos, c = -1, 0, 0
        while pos < prompt:
            n = min(chunk, prompt - pos)
            parent = b.segment(parent, n)
            b.request(parent, "extend", n)
            steps.append(c)
            pos, c = pos + n, c + 1
    return b.finish("chunked_prefill", seed, num_slots, dtype, meta={"chunk": steps})


# --------------------------------------------------------------------------------------
# a serving stream: requests arriving over steps, each generating tokens one step at a time


@dataclass
class StreamRequest:
    rid: int
    prompt: np.ndarray      # int32 token ids
    out_len: int            # tokens to generate (one decode step each)
    arrival: int            # step at which the request joins the waiting queue
    group: int              # few-shot prompt group (shared prefix)


@dataclass
class ServingStream:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    sm_scale: float
    requests: list


def serving_stream(seed=7, n_groups=8, per_group=32, shared=1800, unique=(50, 150), out=(32, 64),
                   per_step=16, hq=32, hkv=8, d=128) -> ServingStream:
    """Few-shot serving: ``n_groups`` prompt groups, each a ``shared``-token prefix (the
    examples) followed by a unique U[unique] question per request; every request then
    generates U[out] tokens.  Requests arrive ``per_step`` at a time, the groups interleaved
    in a seeded random order, so arrival order mixes the groups."""
    rng = np.random.default_rng(seed)
    prefixes = []
    for _ in range(n_groups):
        t = rng.integers(0, VOCAB, size=shared).astype(np.int32)
        while any(len(p) and p[0] == t[0] for p in prefixes):
            t[0] = np.int32(rng.integers(0, VOCAB))
        prefixes.append(t)
    groups = rng.permutation(np.repeat(np.arange(n_groups), per_group))
    reqs = []
    for i, g in enumerate(groups):
        q = rng.integers(0, VOCAB, size=int(rng.integers(unique[0], unique[1] + 1))).astype(np.int32)
        reqs.append(StreamRequest(i, np.concatenate([prefixes[g], q]), int(rng.integers(out[0], out[1] + 1)),
                                  i // per_step, int(g)))
    sm_scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    return ServingStream("serving_stream", seed, hq, hkv, d, sm_scale, reqs)


def token_kv(seed: int, tokens, positions, hkv: int, d: int):
    """bf16 bits of K and V ([n, hkv, d] uint16) for context entries (token id, position):
    N(0, 1) values drawn from a generator keyed by (seed, token, position) alone, so equal
    prefixes have equal K/V wherever they occur."""
    n = len(tokens)
    k = np.empty((n, hkv, d), np.uint16)
    v = np.empty((n, hkv, d), np.uint16)
    for i, (t, p) in enumerate(zip(tokens, positions)):
        x = np.random.default_rng([seed, 1, int(t), int(p)]).standard_normal(2 * hkv * d, dtype=np.float32)
        k[i] = to_bf16_bits(x[:hkv * d]).reshape(hkv, d)
        v[i] = to_bf16_bits(x[hkv * d:]).reshape(hkv, d)
    return k, v


def stream_query(seed: int, rid: int, pos: int, hq: int, d: int):
    """bf16 bits [hq, d] of request rid's query at context position pos."""
    x = np.random.default_rng([seed, 3, int(rid), int(pos)]).standard_normal(hq * d, dtype=np.float32)
    return to_bf16_bits(x).reshape(hq, d)


def generated_token(seed: int, rid: int, j: int) -> int:
    """Token id of request rid's j-th generated token."""
    return int(np.random.default_rng([seed, 2, int(rid), int(j)]).integers(0, VOCAB))


def config(k: int) -> Workload:
    """The five full-size workloads, seed = configuration number."""
    return {1: tiny_decode, 2: fewshot_extend, 3: batched_decode, 4: multiturn_decode,
            5: tot_mixed}[k](seed=k)
