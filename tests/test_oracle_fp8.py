"""Pins for the oracle's E4M3 encoder/decoder and fp8 store: torch's independent
float8_e4m3fn cast, exhaustive round trips, and the OCP format's fixed points."""

import numpy as np
import torch

from oracle.fp8 import e4m3_decode, e4m3_encode, quantize_to_pool
from oracle.kv_store import kv_store_bf16, kv_store_fp8


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _all_bf16_f64():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        return (bits << 16).view(np.float32).astype(np.float64)


def test_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_format_fixed_points():
    assert e4m3_decode([0x7E])[0] == 448.0              # largest finite
    assert e4m3_decode([0x01])[0] == 2.0 ** -9          # smallest subnormal
    assert e4m3_decode([0x08])[0] == 2.0 ** -6          # smallest normal
    assert e4m3_decode([0x38])[0] == 1.0
    assert np.isnan(e4m3_decode([0x7F])[0]) and np.isnan(e4m3_decode([0xFF])[0])
    assert e4m3_encode([1.0])[0] == 0x38 and e4m3_encode([-448.0])[0] == 0xFE


def test_round_trip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    finite = ~np.isnan(e4m3_decode(codes))
    back = e4m3_encode(e4m3_decode(codes[finite]))
    assert np.array_equal(back, codes[finite])


def test_encode_every_bf16_vs_torch_in_range():
    x = _all_bf16_f64()
    inr = np.isfinite(x) & (np.abs(x) < 464.0)           # torch turns overflow into NaN
    ours = e4m3_encode(x[inr])
    ref = torch.from_numpy(x[inr].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_saturates_and_nan():
    x = _all_bf16_f64()
    big = np.isfinite(x) & (np.abs(x) >= 464.0)
    codes = e4m3_encode(x[big])
    assert np.all((codes & 0x7F) == 0x7E)
    assert np.array_equal(codes >> 7, np.signbit(x[big]).astype(np.uint8))
    assert e4m3_encode([np.nan])[0] == 0x7F


def test_midpoints_round_to_even():
    codes = np.arange(0, 0x7E, dtype=np.uint8)          # positive finite, below max
    lo, hi = e4m3_decode(codes), e4m3_decode(codes + 1)
    mid = (lo + hi) / 2.0
    got = e4m3_encode(mid)
    even = np.where(codes % 2 == 0, codes, codes + 1)
    assert np.array_equal(got, even.astype(np.uint8))


def test_quantize_with_scale_vs_torch():
    x = _all_bf16_f64()
    for scale in (1.0, 0.0125558, 3.7, 2.0 ** -7):
        with np.errstate(over="ignore", invalid="ignore"):
            y = (x.astype(np.float32) / np.float32(scale))
        inr = np.isfinite(y) & (np.abs(y) < 464.0)
        ours = quantize_to_pool(x[inr], scale)
        t = torch.from_numpy(x[inr].astype(np.float32)) / torch.tensor(scale, dtype=torch.float32)
        ref = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours, ref), scale


def test_kv_store_scatter_semantics():
    rng = np.random.default_rng(0)
    S, H, d, n = 50, 2, 8, 7
    pool = rng.integers(0, 1 << 16, size=(S, H, d), dtype=np.uint16)
    rows = rng.integers(0, 1 << 16, size=(n, H, d), dtype=np.uint16)
    loc = rng.permutation(S)[:n]
    out = kv_store_bf16(pool, rows, loc)
    untouched = np.setdiff1d(np.arange(S), loc)
    assert np.array_equal(out[untouched], pool[untouched])
    assert np.array_equal(out[loc], rows)
    x = rng.standard_normal((n, H, d)).astype(np.float32)
    rows = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pool8 = rng.integers(0, 256, size=(S, H, d), dtype=np.uint8)
    out8 = kv_store_fp8(pool8, rows, loc, 0.01)
    assert np.array_equal(out8[untouched], pool8[untouched])
    ref = (torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).float() / torch.tensor(0.01)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(out8[loc], ref)
