"""Pins for the oracle's attention: pure-Python softmax loops on tiny inputs, torch's fp64
scaled_dot_product_attention, closed-form special cases, shared-versus-duplicated prefixes,
and the log-sum-exp merge of split key ranges."""

import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep
from oracle.attention import attend, attend_pool, merge_states
from oracle.radix_tree import RadixCache


def _brute(q, K, V, sm_scale, positions):
    n, hq, d = q.shape
    hkv = K.shape[1]
    G = hq // hkv
    out = [[[0.0] * d for _ in range(hq)] for _ in range(n)]
    for i in range(n):
        for h in range(hq):
            g = h // G
            s = []
            for j in range(positions[i] + 1):
                acc = 0.0
                for c in range(d):
                    acc += float(q[i, h, c]) * float(K[j, g, c])
                s.append(acc * sm_scale)
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            for c in range(d):
                out[i][h][c] = sum(e[j] * float(V[j, g, c]) for j in range(len(e))) / tot
    return np.array(out)


@pytest.mark.parametrize("seed,hq,hkv,d,L,n", [(0, 2, 1, 4, 5, 3), (1, 4, 2, 8, 8, 4), (2, 3, 3, 2, 6, 6),
                                               (3, 8, 2, 5, 7, 1)])
def test_brute_force_tiny(seed, hq, hkv, d, L, n):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, hq, d))
    K = rng.standard_normal((L, hkv, d))
    V = rng.standard_normal((L, hkv, d))
    pos = np.arange(L - n, L)
    o, _ = attend(q, K, V, 0.37, pos)
    assert np.max(np.abs(o - _brute(q, K, V, 0.37, pos))) < 1e-12


def test_vs_torch_sdpa_fp64():
    rng = np.random.default_rng(7)
    hq, hkv, d, L, n = 8, 2, 16, 40, 9
    q = rng.standard_normal((n, hq, d))
    K = rng.standard_normal((L, hkv, d)) * 2
    V = rng.standard_normal((L, hkv, d))
    pos = np.arange(L - n, L)
    o, _ = attend(q, K, V, 1 / math.sqrt(d), pos)
    G = hq // hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)                           # [Hq, n, d]
    tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)    # [Hq, L, d]
    tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=1 / math.sqrt(d))
    assert np.max(np.abs(o - ref.permute(1, 0, 2).numpy())) < 1e-12


def test_constant_v_gives_v():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((5, 4, 8)) * 3
    K = rng.standard_normal((30, 2, 8))
    V = np.broadcast_to(rng.standard_normal((1, 2, 8)), (30, 2, 8)).copy()
    o, _ = attend(q, K, V, 0.5, np.arange(25, 30))
    want = np.stack([V[0, 0], V[0, 0], V[0, 1], V[0, 1]])
    assert np.max(np.abs(o - want[None])) < 1e-14


def test_single_key_gives_its_value():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 4, 8))
    K = rng.standard_normal((1, 1, 8))
    V = rng.standard_normal((1, 1, 8))
    o, lse = attend(q, K, V, 0.3, [0])
    assert np.array_equal(o[0], np.repeat(V[0], 4, axis=0))
    assert np.allclose(lse[0], 0.3 * (q[0] @ K[0, 0]))


def test_lse_merge_equals_unsplit():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((6, 4, 16))
    K = rng.standard_normal((100, 2, 16)) * 3
    V = rng.standard_normal((100, 2, 16))
    pos = np.arange(94, 100)
    full, lse_full = attend(q, K, V, 0.25, pos)
    cuts = [0, 13, 14, 60, 96, 100]
    parts = [attend(q, K, V, 0.25, pos, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = merge_states(parts)
    assert np.max(np.abs(o - full)) < 1e-12
    assert np.max(np.abs(lse - lse_full)) < 1e-12


def test_shared_prefix_equals_duplicated_prefix_bitwise():
    """Same values reached through shared slots or through per-request copies."""
    rng = np.random.default_rng(6)
    S, hkv, d, hq = 64, 2, 8, 4
    P, U = 10, 5
    Kp, Vp = rng.standard_normal((P, hkv, d)), rng.standard_normal((P, hkv, d))
    tails = [(rng.standard_normal((U, hkv, d)), rng.standard_normal((U, hkv, d))) for _ in range(2)]
    q = rng.standard_normal((1, hq, d))
    pos = [P + U - 1]
    # shared: both rows point at slots 0..P-1 for the prefix
    kpool, vpool = np.zeros((S, hkv, d)), np.zeros((S, hkv, d))
    kpool[:P], vpool[:P] = Kp, Vp
    rows_shared = []
    for r, (kt, vt) in enumerate(tails):
        base = P + r * U
        kpool[base:base + U], vpool[base:base + U] = kt, vt
        rows_shared.append(list(range(P)) + list(range(base, base + U)))
    # duplicated: each row has its own copy of the prefix in different slots
    kdup, vdup = np.zeros((S, hkv, d)), np.zeros((S, hkv, d))
    rows_dup = []
    for r, (kt, vt) in enumerate(tails):
        slots = list(range(63 - r * (P + U), 63 - (r + 1) * (P + U), -1))
        kdup[slots[:P]], vdup[slots[:P]] = Kp, Vp
        kdup[slots[P:]], vdup[slots[P:]] = kt, vt
        rows_dup.append(slots)
    for r in range(2):
        a, _ = _attend_f64_pool(q, kpool, vpool, rows_shared[r], pos)
        b, _ = _attend_f64_pool(q, kdup, vdup, rows_dup[r], pos)
        c, _ = attend(q, np.concatenate([Kp, tails[r][0]]), np.concatenate([Vp, tails[r][1]]), 0.3, pos)
        assert np.array_equal(a, b) and np.array_equal(a, c)


def _attend_f64_pool(q, kpool, vpool, row, pos):
    slots = np.asarray(row[:pos[0] + 1])
    return attend(q, kpool[slots], vpool[slots], 0.3, pos)


def test_step_recompute_matches_tree_and_pool_gather():
    """The step oracle's contiguous recompute equals attention read through slot tables built
    by the oracle's own radix tree and store, for a small few-shot extend and a decode tree."""
    from oracle.kv_store import kv_store_bf16
    for w in (W.fewshot_extend(seed=11, n_req=3, prefix=40, suffix=9, hq=4, hkv=2, d=8, num_slots=400),
              W.multiturn_decode(seed=12, n_conv=2, turns=2, user=(5, 9), reply=(3, 6), hq=4, hkv=2,
                                 d=8, num_slots=400)):
        tree = RadixCache()
        kpool = np.zeros((w.num_slots, w.num_kv_heads, w.head_dim), np.uint16)
        vpool = kpool.copy()
        nxt = 0
        rows = []
        for r in w.requests:
            toks = W.context_tokens(w, r)
            kb, vb = W.context_kv_bits(w, r)
            vals, _ = tree.match_prefix(toks)
            m = len(vals)
            new = w.slot_perm[nxt:nxt + len(toks) - m].tolist()
            nxt += len(toks) - m
            kpool = kv_store_bf16(kpool, kb[m:], new)
            vpool = kv_store_bf16(vpool, vb[m:], new)
            tree.insert(toks, vals + new)
            rows.append(vals + new)
        for r, row in zip(w.requests, rows):
            pos = ostep.query_positions(w, r)
            a, _ = attend_pool(W.bf16_bits_to_f64(r.q), kpool, vpool, "bf16", 1, 1, row, pos, w.sm_scale)
            b, _ = ostep.request_output(w, r)
            assert np.array_equal(a, b)
