"""Expected outputs of one workload step, computed by contiguous recompute (oracle copy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

For every request the oracle rebuilds the request's whole context K/V by concatenating its
segments in order -- no radix tree, no pool, no slot tables -- and runs ``attention.attend``
with the causal positions of its queries.  For an fp8_e4m3 pool the context K/V are first
quantised with the oracle's own encoder and decoded back times the scale, so the
comparison charges the kernels only for their own arithmetic, not for the pool's
quantisation.  Because it never looks at slots, this recompute is independent of how the
product path shares, stores and gathers the prefix.
"""

from __future__ import annotations

import numpy as np

from .attention import attend, bf16_to_f64
from .fp8 import e4m3_decode, quantize_to_pool


def context_kv(w, req):
    """float64 K, V [L, Hkv, d] of a request's context as the pool holds them."""
    kb = np.concatenate([w.segments[s].k for s in req.path], axis=0)
    vb = np.concatenate([w.segments[s].v for s in req.path], axis=0)
    K, V = bf16_to_f64(kb), bf16_to_f64(vb)
    if w.dtype == "fp8_e4m3":
        K = e4m3_decode(quantize_to_pool(K, w.k_scale)) * w.k_scale
        V = e4m3_decode(quantize_to_pool(V, w.v_scale)) * w.v_scale
    return K, V


def query_positions(w, req):
    L = sum(len(w.segments[s].tokens) for s in req.path)
    if req.kind == "extend":
        return np.arange(L - req.n_new, L)
    return np.array([L - 1])


def request_output(w, req, query_idx=None):
    """(o [n, Hq, d], lse [n, Hq]) for all (or the listed) queries of one request."""
    K, V = context_kv(w, req)
    pos = query_positions(w, req)
    q = bf16_to_f64(req.q)
    if query_idx is not None:
        query_idx = np.asarray(query_idx, dtype=np.int64)
        pos, q = pos[query_idx], q[query_idx]
    return attend(q, K, V, w.sm_scale, pos)


def expected_outputs(w, kind):
    """All outputs of the ``kind`` ('extend' or 'decode') call of a step, in batch order:
    extend -> [sum_e, Hq, d], decode -> [B, Hq, d]."""
    outs = [request_output(w, r)[0] for r in w.requests if r.kind == kind]
    if not outs:
        return np.zeros((0, w.num_q_heads, w.head_dim))
    return np.concatenate(outs, axis=0)


def expected_sample(w, kind, picks):
    """Outputs for sampled (request-within-kind index, query index) pairs."""
    reqs = [r for r in w.requests if r.kind == kind]
    by_req = {}
    for ri, qi in picks:
        by_req.setdefault(ri, []).append(qi)
    out = {}
    for ri, qis in by_req.items():
        o, _ = request_output(w, reqs[ri], qis)
        for j, qi in enumerate(qis):
            out[(ri, qi)] = o[j]
    return out
