"""Scaled-dot-product attention over a request's token context, in float64 (oracle copy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed.  A request's context is the token sequence matched in the radix tree
followed by its uncached remainder; only the remainder is prefilled, the matched prefix's
K/V are reused ("Efficiently Programming Large Language Models using SGLang" summary,
§RadixAttention: プレフィックスマッチングアルゴリズム -- the matched length needs no
recomputation; "SGLang: Treating LLM Interactions as Programs", §Why this matters in
production).  For query token i of a request whose context has L tokens, at absolute
position t (t = p + i for an extend of the last e tokens after a p-token prefix;
t = L - 1 for a decode), and query head h with KV head g = floor(h / G), G = Hq / Hkv:

    s_j = sm_scale * <q_h, K_j,g>           for j = 0 .. t   (causal, inclusive)
    o_h = sum_j softmax(s)_j * V_j,g

The pages give no formula for this step; it is the textbook definition of causal
scaled-dot-product attention with grouped query heads, and each step below is that
definition written out with no blocking or reordering beyond one matrix product per
(request, KV head).  sm_scale defaults to 1/sqrt(d).

Partial states.  Attention over a subset of the keys returns (o, lse) with
lse = log sum_j exp(s_j); two partial states over disjoint key sets merge exactly by
``merge_states`` (the log-sum-exp identity).
"""

from __future__ import annotations

import numpy as np

from .fp8 import e4m3_decode


def bf16_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attend(q, K, V, sm_scale, positions, key_lo=0, key_hi=None):
    """q [n, Hq, d], K/V [L, Hkv, d] (float64), positions [n]: query i sees keys
    key_lo .. min(positions[i], key_hi - 1).  Returns (o [n, Hq, d], lse [n, Hq]);
    a query with no visible key gets o = 0, lse = -inf."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n, hq, d = q.shape
    L, hkv, _ = K.shape
    if key_hi is None:
        key_hi = L
    G = hq // hkv
    pos = np.asarray(positions, dtype=np.int64)
    keys = np.arange(key_lo, key_hi)
    visible = keys[None, :] <= pos[:, None]                 # [n, Lw]
    o = np.zeros((n, hq, d))
    lse = np.full((n, hq), -np.inf)
    if key_hi <= key_lo:
        return o, lse
    for g in range(hkv):
        Kg = K[key_lo:key_hi, g, :]
        Vg = V[key_lo:key_hi, g, :]
        qg = q[:, g * G:(g + 1) * G, :].reshape(n * G, d)
        s = (qg @ Kg.T).reshape(n, G, -1) * sm_scale
        s = np.where(visible[:, None, :], s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        any_vis = np.isfinite(m)
        m = np.where(any_vis, m, 0.0)
        w = np.exp(s - m)
        l = w.sum(axis=-1, keepdims=True)
        og = (w.reshape(n * G, -1) @ Vg).reshape(n, G, d)
        og = np.where(any_vis, og / np.where(l > 0, l, 1.0), 0.0)
        o[:, g * G:(g + 1) * G, :] = og
        lse[:, g * G:(g + 1) * G] = np.where(any_vis[..., 0], np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)) + m[..., 0], -np.inf)
    return o, lse


def merge_states(parts):
    """Merge partial states [(o_k, lse_k)] over disjoint key sets into (o, lse)."""
    lses = np.stack([p[1] for p in parts])                  # [k, ...]
    mx = lses.max(axis=0)
    mx_safe = np.where(np.isfinite(mx), mx, 0.0)
    wts = np.exp(lses - mx_safe)                             # exp(-inf) = 0
    tot = wts.sum(axis=0)
    o = sum(w[..., None] * p[0] for w, p in zip(wts, parts))
    o = np.where((tot > 0)[..., None], o / np.where(tot > 0, tot, 1.0)[..., None], 0.0)
    lse = np.where(tot > 0, np.log(np.where(tot > 0, tot, 1.0)) + mx_safe, -np.inf)
    return o, lse


def dequant_pool_rows(rows, dtype: str, scale: float) -> np.ndarray:
    """Pool rows (bf16 bits or e4m3 codes) -> float64 values."""
    if dtype == "bf16":
        return bf16_to_f64(rows)
    return e4m3_decode(rows) * float(scale)


def attend_pool(q, k_pool, v_pool, dtype, k_scale, v_scale, row, positions, sm_scale):
    """Attention read through one req_to_token row: key j of the context lives in pool
    slot row[j].  k_pool / v_pool hold raw pool contents [S, Hkv, d]."""
    L = int(np.max(positions)) + 1
    slots = np.asarray(row[:L], dtype=np.int64)
    K = dequant_pool_rows(k_pool[slots], dtype, k_scale)
    V = dequant_pool_rows(v_pool[slots], dtype, v_scale)
    return attend(q, K, V, sm_scale, positions)
