"""Pins for the oracle's radix tree: the pages' worked examples, a brute-force per-token trie,
and the invariants the radix-cache walk-through states in prose."""

import json
import os
import random

import pytest

from oracle.radix_tree import RadixCache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _shape(node, with_value=True):
    out = []
    for first in sorted(node.children):
        c = node.children[first]
        d = {"key": list(c.key), "children": _shape(c, with_value)}
        if with_value:
            d["value"] = list(c.value)
        out.append(d)
    return out


def _strip_values(tree):
    return [{"key": n["key"], "children": _strip_values(n["children"])} for n in tree]


def _sort(tree):
    return sorted(({"key": n["key"], **({"value": n["value"]} if "value" in n else {}),
                    "children": _sort(n["children"])} for n in tree), key=lambda n: n["key"][0])


def test_worked_example_tree_and_hit():
    g = json.load(open(os.path.join(GOLDEN, "radix_worked_example.json")))
    t = RadixCache()
    # build the figure's tree through the public API: the second insert finds [1,2,3]
    # already cached (3 leading tokens; the caller would free its duplicate slots)
    assert t.insert([1, 2, 3, 4, 5], [0, 1, 2, 3, 4]) == 0
    assert t.insert([1, 2, 3, 13, 14], [90, 91, 92, 5, 6]) == 3
    assert t.insert([8, 9, 10, 11, 12], [7, 8, 9, 10, 11]) == 0
    assert _shape(t.root) == _sort(g["tree"])
    values, last = t.match_prefix(g["query"])
    assert len(values) == g["hit_len"]
    assert values == g["hit_value"]
    assert last.key == [4, 5]
    # [1,2,3] stays one node shared by both branches
    shared = t.root.children[1]
    assert shared.key == [1, 2, 3] and sorted(shared.children) == [4, 13]


def test_split_example():
    g = json.load(open(os.path.join(GOLDEN, "radix_split_example.json")))
    t = RadixCache()
    t.insert([1, 2, 3, 4, 5], [10, 11, 12, 13, 14])
    assert _strip_values(_shape(t.root)) == g["before"]
    values, last = t.match_prefix([1, 2, 3, 9])     # partial match of length split_len
    assert len(values) == g["split_len"] and values == [10, 11, 12]
    assert _strip_values(_shape(t.root)) == g["after"]
    assert last.key == [1, 2, 3]
    # the split keeps every root-to-leaf concatenation (design rationale: dynamic split)
    v2, _ = t.match_prefix([1, 2, 3, 4, 5])
    assert v2 == [10, 11, 12, 13, 14]


def test_split_inherits_lock_ref():
    t = RadixCache()
    t.insert([5, 6, 7, 8], [0, 1, 2, 3])
    _, leaf = t.match_prefix([5, 6, 7, 8])
    t.inc_lock_ref(leaf)
    _, upper = t.match_prefix([5, 6, 0])
    assert upper.key == [5, 6] and upper.lock_ref == 1 and leaf.lock_ref == 1
    assert t.protected_size_ == 4 and t.evictable_size_ == 0


class BruteTrie:
    """One node per token: prefix tuple -> slot of its last token."""

    def __init__(self):
        self.slot = {}

    def insert(self, key, value):
        cached = 0
        for i in range(len(key)):
            p = tuple(key[:i + 1])
            if p in self.slot:
                cached = i + 1
            else:
                self.slot[p] = value[i]
        return cached

    def match(self, key):
        out = []
        for i in range(len(key)):
            p = tuple(key[:i + 1])
            if p not in self.slot:
                break
            out.append(self.slot[p])
        return out


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_trie_agreement(seed):
    rng = random.Random(seed)
    t, b = RadixCache(), BruteTrie()
    next_slot = 0
    for _ in range(120):
        n = rng.randint(0, 12)
        key = [rng.randint(0, 3) for _ in range(n)]
        if rng.random() < 0.5:
            vals, last = t.match_prefix(key)
            assert vals == b.match(key)
            assert len(vals) <= len(key)
        else:
            value = list(range(next_slot, next_slot + n))
            next_slot += n
            got = t.insert(key, value)
            want = b.insert(key, value)
            assert got == want
        # the insert's inserted sizes account for every cached token
        assert t.evictable_size_ + t.protected_size_ == t.total_size() == len(b.slot)


def test_lru_order_and_parent_requeue():
    t = RadixCache()
    t.insert([1, 1], [0, 1])          # tick 1
    t.insert([2, 2], [2, 3])          # tick 2
    t.insert([3, 3], [4, 5])          # tick 3
    t.match_prefix([1, 1])            # tick 4 touches [1,1]
    assert t.evict(1) == [2, 3]       # least recently used: [2,2]
    assert t.evict(2) == [4, 5]       # then [3,3] (tick 3) before [1,1] (tick 4)
    assert t.evict(10) == [0, 1]
    assert t.total_size() == 0 and t.evictable_size_ == 0


def test_evict_leaf_first_then_parent():
    t = RadixCache()
    t.insert([1, 2, 3, 4], [0, 1, 2, 3])
    t.insert([1, 2, 3, 5], [9, 9, 9, 4])      # splits: [1,2,3] -> {[4], [5]}
    freed = t.evict(100)
    assert sorted(freed) == [0, 1, 2, 3, 4]
    assert freed[-3:] == [0, 1, 2]            # the parent goes only after both leaves
    assert t.root.children == {}


def test_locked_path_never_evicted():
    t = RadixCache()
    t.insert([1, 2, 3, 4], [0, 1, 2, 3])
    t.insert([1, 2, 3, 5], [9, 9, 9, 4])
    _, leaf = t.match_prefix([1, 2, 3, 4])
    t.inc_lock_ref(leaf)
    assert t.evict(100) == [4]
    assert t.match_prefix([1, 2, 3, 4])[0] == [0, 1, 2, 3]
    assert t.protected_size_ == 4 and t.evictable_size_ == 0
    t.dec_lock_ref(leaf)
    assert t.protected_size_ == 0 and t.evictable_size_ == 4
    assert sorted(t.evict(100)) == [0, 1, 2, 3]


@pytest.mark.parametrize("seed", range(4))
def test_random_ops_invariants(seed):
    rng = random.Random(100 + seed)
    t, b = RadixCache(), BruteTrie()
    locked = []
    next_slot = 0
    for _ in range(300):
        op = rng.random()
        key = [rng.randint(0, 4) for _ in range(rng.randint(1, 10))]
        if op < 0.35:
            v = list(range(next_slot, next_slot + len(key)))
            next_slot += len(key)
            t.insert(key, v)
        elif op < 0.55:
            vals, last = t.match_prefix(key)
            if vals and rng.random() < 0.5:
                t.inc_lock_ref(last)
                locked.append((key[:len(vals)], vals, last))
        elif op < 0.7 and locked:
            k, v, node = locked.pop(rng.randrange(len(locked)))
            t.dec_lock_ref(node)
        else:
            before = t.total_size()
            freed = t.evict(rng.randint(1, 8))
            assert before - t.total_size() == len(freed)
            assert len(set(freed)) == len(freed)
        assert t.evictable_size_ + t.protected_size_ == t.total_size()
        for k, v, _ in locked:                 # a locked prefix stays cached, same slots
            assert t.match_prefix(k)[0] == v
