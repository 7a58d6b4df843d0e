"""Pins of the oracle's paged radix tree (page size P > 1: whole blocks of P tokens only;
"Efficiently Programming Large Language Models using SGLang" (summary), §Technical Details,
whose cache insert refers to the KV by 16-token block).  Each pin checks the paged tree
against something other than itself: a hand-worked example, the token tree (already pinned
against the pages' worked example) run on one symbol per block, and the definition of a
block-granular longest cached prefix computed by brute force."""

import random

import pytest

from oracle.radix_tree import RadixCache
from oracle.schedule import peek_match_len


def test_hand_worked_example_page_2():
    t = RadixCache(page_size=2)
    # one node [1 2 | 3 4 | 5 6]
    assert t.insert([1, 2, 3, 4, 5, 6], [10, 11, 12, 13, 14, 15]) == 0
    # [1 2 | 3 9 | 5 6 | 7]: the trailing 7 is a partial block and is dropped; block (3, 9)
    # differs from (3, 4) although token 3 matches, so only one block (2 tokens) is cached
    # and the node splits after [1 2] (a token tree would split after [1 2 3])
    assert t.insert([1, 2, 3, 9, 5, 6, 7], [10, 11, 20, 21, 22, 23, 24]) == 2
    keys = sorted(tuple(n.key) for n in t._all_nodes() if n is not t.root)
    assert keys == [(1, 2), (3, 4, 5, 6), (3, 9, 5, 6)]
    # a 5-token query looks at 4 tokens; (3, 4) matches the first block of [3 4 5 6] only,
    # which splits it after 2 tokens
    vals, node = t.match_prefix([1, 2, 3, 4, 5])
    assert vals == [10, 11, 12, 13] and node.key == [3, 4]
    assert sorted(tuple(n.key) for n in t._all_nodes() if n is not t.root) == \
        [(1, 2), (3, 4), (3, 9, 5, 6), (5, 6)]
    assert t.match_prefix([1, 2, 3])[0] == [10, 11]
    assert t.match_prefix([1])[0] == [] and t.match_prefix([1])[1] is t.root
    assert t.match_prefix([1, 2, 3, 9, 5, 6])[0] == [10, 11, 20, 21, 22, 23]
    assert t.total_size() == 10


def test_keys_shorter_than_a_block_are_not_cached():
    t = RadixCache(page_size=16)
    assert t.insert(list(range(15)), list(range(15))) == 0
    assert t.total_size() == 0 and t.match_prefix(list(range(15)))[0] == []
    assert t.insert(list(range(40)), list(range(100, 140))) == 0
    assert t.total_size() == 32                       # two whole blocks of 40 tokens
    assert t.match_prefix(list(range(40)))[0] == list(range(100, 132))
    assert t.match_prefix(list(range(31)))[0] == list(range(100, 116))


@pytest.mark.parametrize("page", [2, 4, 16])
@pytest.mark.parametrize("seed", range(3))
def test_equals_token_tree_on_block_symbols(page, seed):
    """Keys made of whole blocks drawn from a few distinct blocks: the paged tree must act
    like the token tree run on one symbol per block (match lengths x page, same values)."""
    rng = random.Random(seed)
    blocks = [[rng.randint(0, 3) for _ in range(page)] for _ in range(5)]
    blocks = [b for i, b in enumerate(blocks) if b not in blocks[:i]]   # distinct contents
    paged, token = RadixCache(page_size=page), RadixCache()
    nxt = 0
    for _ in range(150):
        sym = [rng.randrange(len(blocks)) for _ in range(rng.randint(0, 6))]
        key = [t for s in sym for t in blocks[s]]
        if rng.random() < 0.5:
            vals = list(range(nxt, nxt + len(key)))
            nxt += len(key)
            assert paged.insert(key, vals) == page * token.insert(sym, vals[::page])
        else:
            vp, _ = paged.match_prefix(key)
            vt, _ = token.match_prefix(sym)
            assert len(vp) == page * len(vt)
            assert vp[::page] == vt        # the first slot of every matched block
        assert paged.total_size() == page * token.total_size()


@pytest.mark.parametrize("page", [1, 3, 4])
def test_brute_force_block_prefix(page):
    """No eviction: the matched length of q is page x the most leading blocks q shares with
    any inserted key, and the values are those of the insert that first cached each
    block-aligned prefix; insert returns the length matched just before it."""
    rng = random.Random(7 + page)
    t = RadixCache(page_size=page)
    first = {}   # block-aligned prefix -> slot values of its last block, from the first insert

    def brute(q):
        n = len(q) // page * page
        m = 0
        while m + page <= n and tuple(q[:m + page]) in first:
            m += page
        return m

    nxt = 0
    for _ in range(200):
        key = [rng.randint(0, 2) for _ in range(rng.randint(0, 14))]
        if rng.random() < 0.5:
            vals = list(range(nxt, nxt + len(key)))
            nxt += len(key)
            expect = brute(key)
            assert t.insert(key, vals) == expect
            for m in range(page, len(key) // page * page + 1, page):
                first.setdefault(tuple(key[:m]), vals[m - page:m])
        else:
            m = brute(key)
            got, _ = t.match_prefix(key)
            want = [v for j in range(page, m + 1, page) for v in first[tuple(key[:j])]]
            assert got == want
            assert peek_match_len(t, key) == m


def test_page_one_is_the_token_tree():
    a, b = RadixCache(), RadixCache(page_size=1)
    rng = random.Random(11)
    for i in range(100):
        key = [rng.randint(0, 4) for _ in range(rng.randint(0, 9))]
        v = list(range(100 * i, 100 * i + len(key)))
        assert a.insert(key, v) == b.insert(key, v)
        assert a.match_prefix(key[:5])[0] == b.match_prefix(key[:5])[0]
    assert a.dump() == b.dump()
