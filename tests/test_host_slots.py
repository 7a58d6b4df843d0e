"""Host check of kv_store's precondition (pkv_check_out_cache_loc): within one call every
new token's slot is in the pool and no two tokens share one.  The allocator hands out
distinct free slots ("[SGLang] RadixAttention ...", "Eviction 전략": evicted slots return to
the allocator's free list), so a duplicate means a caller bug -- e.g. a slot released twice."""

import numpy as np
import pytest

import prefix_shared_kv_token_gb300 as pkv


def test_distinct_in_range_slots_pass():
    rng = np.random.default_rng(0)
    loc = rng.permutation(1 << 16)[:5000].astype(np.int32)
    assert pkv.check_out_cache_loc(loc, 1 << 16) == -1
    assert pkv.check_out_cache_loc(np.zeros(0, np.int32), 8) == -1
    assert pkv.check_out_cache_loc(np.array([0, 7], np.int32), 8) == -1   # both ends of the pool


def test_duplicate_is_reported_at_its_second_occurrence():
    loc = np.array([5, 9, 2, 9, 5, 11], np.int32)
    assert pkv.check_out_cache_loc(loc, 16) == 3      # 9 repeats at index 3 (5 repeats later, at 4)
    loc = np.array([4, 4], np.int32)
    assert pkv.check_out_cache_loc(loc, 16) == 1


def test_out_of_range_slots_are_reported():
    assert pkv.check_out_cache_loc(np.array([1, 2, 16], np.int32), 16) == 2
    assert pkv.check_out_cache_loc(np.array([1, -1, 3], np.int32), 16) == 1
    # the first offending index wins, whatever the kind
    assert pkv.check_out_cache_loc(np.array([3, 20, 3], np.int32), 16) == 1
    assert pkv.check_out_cache_loc(np.array([3, 3, 20], np.int32), 16) == 1


@pytest.mark.parametrize("pool", ["small", "huge"])
def test_matches_a_brute_force_scan(pool):
    # a small pool takes the one-pass bitmap, a huge one with a short list the sort
    rng = np.random.default_rng(1)
    for _ in range(200):
        n = int(rng.integers(0, 40))
        if pool == "small":
            S = int(rng.integers(1, 30))
            loc = rng.integers(-2, S + 2, size=n).astype(np.int32)
        else:
            S = (1 << 30) + int(rng.integers(0, 5))
            near = rng.integers(-2, 30, size=n)           # low slots, repeats likely
            loc = np.where(rng.random(n) < 0.2, S - 3 + rng.integers(0, 6, size=n), near).astype(np.int32)
        want, seen = -1, set()
        for i, s in enumerate(loc.tolist()):
            if s < 0 or s >= S or s in seen:
                want = i
                break
            seen.add(s)
        assert pkv.check_out_cache_loc(loc, S) == want, (loc, S)


def test_a_slot_released_twice_is_caught():
    a = pkv.Allocator(np.arange(8, dtype=np.int32))
    got = a.alloc(3)
    a.release(got[:1])
    a.release(got[:1])                       # caller bug: the same slot freed twice
    loc = a.alloc(a.available)               # hands slot got[0] out twice
    assert pkv.check_out_cache_loc(loc, 8) >= 0


def test_invalid_arguments():
    import ctypes as C
    from prefix_shared_kv_token_gb300 import _lib
    bad = C.c_int64(0)
    assert _lib.lib.pkv_check_out_cache_loc(None, 3, 8, C.byref(bad)) == -1
    assert _lib.lib.pkv_check_out_cache_loc(None, 0, 0, None) == -1
