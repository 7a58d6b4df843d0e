"""Pins of the oracle tree's eviction policies ("[SGLang] RadixAttention ...", "Eviction 전략":
lru, lfu, slru, fifo, mru, filo, priority; node fields hit_count and priority of "핵심
자료구조: TreeNode").  Every expected order below is worked out by hand from the policy's
definition on a small history, not produced by the code under test."""

import pytest

from oracle.radix_tree import POLICIES, RadixCache


def _history(policy):
    """Three sibling leaves under the root:
         A = [1, 2, 3] (node 1, inserted at tick 1, priority 5)
         B = [4, 5]    (node 2, tick 2, priority 1)
         C = [6]       (node 3, tick 3, priority 3)
       then match A at ticks 4 and 5 (A: 2 hits, last access 5) and C at tick 6 (C: 1 hit,
       last access 6).  B keeps 0 hits and last access 2."""
    t = RadixCache(policy)
    t.insert([1, 2, 3], [10, 11, 12], priority=5)
    t.insert([4, 5], [20, 21], priority=1)
    t.insert([6], [30], priority=3)
    t.match_prefix([1, 2, 3])
    t.match_prefix([1, 2, 3, 9])
    t.match_prefix([6, 7])
    return t


# hand-derived eviction orders (values freed, one leaf per evict(1) call)
EXPECTED = {
    "lru": ["B", "A", "C"],       # last access 2 < 5 < 6
    "mru": ["C", "A", "B"],       # last access 6 > 5 > 2
    "lfu": ["B", "C", "A"],       # hits 0 < 1 < 2
    "slru": ["B", "C", "A"],      # probationary (hits < 2) B (t2), C (t6); then protected A
    "fifo": ["A", "B", "C"],      # created first: node ids 1 < 2 < 3
    "filo": ["C", "B", "A"],      # created last first
    "priority": ["B", "C", "A"],  # priorities 1 < 3 < 5
}
VALUES = {"A": [10, 11, 12], "B": [20, 21], "C": [30]}


@pytest.mark.parametrize("policy", POLICIES)
def test_policy_order_on_three_leaves(policy):
    t = _history(policy)
    order = [t.evict(1) for _ in range(3)]
    assert order == [VALUES[x] for x in EXPECTED[policy]]
    assert t.evict(1) == [] and t.total_size() == 0


def test_hit_counts_and_access_times():
    t = _history("lru")
    by_key = {tuple(n.key): n for n in t._all_nodes() if n is not t.root}
    assert (by_key[(1, 2, 3)].hit_count, by_key[(1, 2, 3)].last_access_time) == (2, 5)
    assert (by_key[(4, 5)].hit_count, by_key[(4, 5)].last_access_time) == (0, 2)
    assert (by_key[(6,)].hit_count, by_key[(6,)].last_access_time) == (1, 6)


def test_hits_count_the_whole_matched_path_after_a_split():
    t = RadixCache("lfu")
    t.insert([1, 2, 3, 4], [0, 1, 2, 3])
    _, node = t.match_prefix([1, 2, 9])        # splits [1,2,3,4] into [1,2] -> [3,4]
    assert node.key == [1, 2] and node.hit_count == 1
    assert next(iter(node.children.values())).hit_count == 0   # the lower part was not matched
    _, node2 = t.match_prefix([1, 2, 3, 4])
    assert node2.key == [3, 4] and node2.hit_count == 1 and node2.parent.hit_count == 2


def test_priority_on_insert_and_split():
    t = RadixCache("priority")
    t.insert([1, 2, 3], [0, 1, 2], priority=7)
    t.insert([1, 2, 5], [0, 1, 9], priority=2)   # splits [1,2,3]: the upper part keeps 7
    by_key = {tuple(n.key): n for n in t._all_nodes() if n is not t.root}
    assert by_key[(1, 2)].priority == 7 and by_key[(3,)].priority == 7 and by_key[(5,)].priority == 2
    assert t.root.priority == 7                  # start node raised to the insert's priority
    # lowest priority first: [5] (2), then [3] (7, older access), then its parent [1, 2]
    assert t.evict(1) == [9]
    assert t.evict(1) == [2]
    assert t.evict(1) == [0, 1]


def test_parent_requeued_under_each_policy():
    # a leaf whose parent becomes an unlocked leaf: the parent joins the heap and can be
    # evicted in the same call
    for policy in POLICIES:
        t = RadixCache(policy)
        t.insert([1, 2], [0, 1])
        t.insert([1, 2, 3], [0, 1, 2])
        assert t.evict(3) == [2, 0, 1], policy


def test_locked_nodes_survive_every_policy():
    for policy in POLICIES:
        t = _history(policy)
        _, a = t.match_prefix([1, 2, 3])
        t.inc_lock_ref(a)
        t.evict(100)
        assert [n.key for n in t._all_nodes() if n is not t.root] == [[1, 2, 3]], policy
