"""Scatter of new K/V rows into token slots of the pool (oracle copy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pool is indexed per token: a radix-tree node's value is the list of KV-pool indices of
its tokens ("[SGLang] RadixAttention ...", "Radix Tree 구조도" and "핵심 자료구조: TreeNode",
value = KV cache indices).  Storing the K/V of newly computed tokens writes row
``out_cache_loc[i]`` of the pool with token i's K (and V) for every KV head; every other row
is left untouched.  For a bf16 pool the row is copied bit for bit; for an fp8_e4m3 pool
each element is quantised with the per-tensor scale (``oracle.fp8.quantize_to_pool``).
"""

from __future__ import annotations

import numpy as np

from .fp8 import quantize_to_pool


def _bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def kv_store_bf16(pool: np.ndarray, new_rows: np.ndarray, out_cache_loc) -> np.ndarray:
    """pool: uint16 [S, Hkv, d] (bf16 bits), new_rows: uint16 [n, Hkv, d]."""
    out = pool.copy()
    for i, slot in enumerate(np.asarray(out_cache_loc).tolist()):
        out[slot] = new_rows[i]
    return out


def kv_store_fp8(pool: np.ndarray, new_rows: np.ndarray, out_cache_loc, scale: float) -> np.ndarray:
    """pool: uint8 [S, Hkv, d] (e4m3 codes), new_rows: uint16 [n, Hkv, d] (bf16 bits)."""
    out = pool.copy()
    codes = quantize_to_pool(_bf16_to_f64(new_rows), scale)
    for i, slot in enumerate(np.asarray(out_cache_loc).tolist()):
        out[slot] = codes[i]
    return out
