"""Pins of the oracle's cache-aware scheduler ("Efficiently Programming Large Language Models
using SGLang" summary, §Cache-Aware Scheduling: longest prefix match first)."""

import random

from oracle.radix_tree import RadixCache
from oracle.schedule import peek_match_len, schedule


def test_worked_queue():
    # cached: [1,2,3,4,5] and [1,2,3,13,14] (the pages' radix example)
    t = RadixCache()
    t.insert([1, 2, 3, 4, 5], [0, 1, 2, 3, 4])
    t.insert([1, 2, 3, 13, 14], [0, 1, 2, 5, 6])
    queue = [[9, 9], [1, 2, 3, 7], [1, 2], [1, 2, 3, 4, 5, 6], [1, 2, 3, 13]]
    order, lens = schedule(t, queue, "lpm")
    assert lens == [0, 3, 2, 5, 4]               # counted by hand
    assert order == [3, 4, 1, 2, 0]
    assert schedule(t, queue, "fcfs")[0] == [0, 1, 2, 3, 4]


def test_ties_keep_queue_order():
    t = RadixCache()
    t.insert([7, 8], [0, 1])
    order, lens = schedule(t, [[7, 8, 1], [5], [7, 8, 2], [6]], "lpm")
    assert lens == [2, 0, 2, 0] and order == [0, 2, 1, 3]


def test_peek_does_not_change_the_tree():
    t = RadixCache()
    t.insert([1, 2, 3, 4], [0, 1, 2, 3])
    before = t.dump()
    assert peek_match_len(t, [1, 2, 9]) == 2    # inside a node: a real match would split it
    assert t.dump() == before


def test_peek_equals_match_prefix_length():
    rng = random.Random(5)
    t = RadixCache()
    for i in range(60):
        k = [rng.randint(0, 3) for _ in range(rng.randint(1, 10))]
        t.insert(k, list(range(100 * i, 100 * i + len(k))))
    for _ in range(200):
        q = [rng.randint(0, 3) for _ in range(rng.randint(0, 12))]
        n = peek_match_len(t, q)
        vals, _ = t.match_prefix(q)
        assert n == len(vals)
