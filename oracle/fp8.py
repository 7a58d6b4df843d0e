"""OCP FP8 E4M3 encode / decode (oracle copy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Written from the OCP "8-bit Floating Point Specification (OFP8)", E4M3 format: 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds subnormals
(0.mmm * 2^-6); no infinities; S.1111.111 is NaN, so the largest finite magnitude is
S.1111.110 = 1.75 * 2^8 = 448.

The pool stores ``e4m3(fp32(x) / fp32(scale))`` with one per-tensor scale for K and one for
V: the fp8_e4m3 KV dtype of the SGLang runtime article ("SGLang后端运行时优化细节",
§显存分级管理机制, ``--kv-cache-dtype fp8_e4m3``).  The page gives no rounding rule, so the
reading is: IEEE float32 division (round to nearest even), then round to nearest even onto
the E4M3 grid with saturation of finite values to +-448 ("satfinite").  NaN maps to 0x7F.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 0xF) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """float values (exactly representable in float64) -> uint8 codes, round to nearest
    even, finite values saturate to +-448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.int64)
    a = np.abs(np.where(nan, 0.0, x))
    # binade of |x|: a = f * 2^E with f in [0.5, 1)  ->  a in [2^(E-1), 2^E)
    _, E = np.frexp(a)
    e_unb = E.astype(np.int64) - 1                      # floor(log2 a) for a > 0
    e_unb = np.maximum(e_unb, -6)                       # below 2^-6: subnormal spacing
    quantum = np.exp2((e_unb - 3).astype(np.float64))   # 3 mantissa bits
    q = np.rint(a / quantum).astype(np.int64)           # exact division by a power of 2;
                                                        # rint rounds half to even
    # q in [0, 16]; q == 16 carries into the next binade (mantissa 0)
    carry = q >= 16
    e_unb = np.where(carry, e_unb + 1, e_unb)
    q = np.where(carry, q // 2, q)
    sub = q < 8                                         # only possible when e_unb == -6
    e_field = np.where(sub, 0, e_unb + 7)
    m_field = np.where(sub, q, q - 8)
    code = (e_field << 3) | m_field
    over = (e_field > 15) | ((e_field == 15) & (m_field == 7))
    code = np.where(over, 0x7E, code)
    code = np.where(a == 0, 0, code)
    code = code | sign
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def quantize_to_pool(x_bf16_f64, scale: float) -> np.ndarray:
    """Pool codes for bf16 inputs (given as exact float64): e4m3(fp32(x) / fp32(scale))."""
    x32 = np.asarray(x_bf16_f64, dtype=np.float64).astype(np.float32)
    y32 = x32 / np.float32(scale)                       # IEEE fp32 division, RNE
    return e4m3_encode(y32.astype(np.float64))
