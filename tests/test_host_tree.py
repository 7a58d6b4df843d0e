"""The C++ radix tree and allocator (libpkv) against the oracle's tree, bit for bit: same
node ids, keys, values, lock_refs and timestamps after random operation sequences, the
pages' worked example, and eviction order."""

import random

import numpy as np
import pytest

from oracle.radix_tree import RadixCache
from prefix_shared_kv_token_gb300 import Allocator, RadixTree


def _oracle_dump(t: RadixCache):
    rows = []
    for n in t._all_nodes():
        rows.append((n.id, -1 if n.parent is None else n.parent.id, n.lock_ref, n.last_access_time,
                     tuple(n.key), tuple(n.value), len(n.children), n.hit_count, n.priority))
    return sorted(rows)


def test_worked_example_cpp():
    t = RadixTree()
    assert t.insert([1, 2, 3, 4, 5], [0, 1, 2, 3, 4]) == 0
    assert t.insert([1, 2, 3, 13, 14], [90, 91, 92, 5, 6]) == 3
    assert t.insert([8, 9, 10, 11, 12], [7, 8, 9, 10, 11]) == 0
    vals, last = t.match_prefix([1, 2, 3, 4, 5, 6])
    assert vals.tolist() == [0, 1, 2, 3, 4]
    nodes = {r[0]: r for r in t.dump()}
    assert nodes[last][4] == (4, 5)
    shared = [r for r in nodes.values() if r[4] == (1, 2, 3)]
    assert len(shared) == 1 and shared[0][6] == 2


@pytest.mark.parametrize("policy", RadixTree.POLICIES)
@pytest.mark.parametrize("seed", range(4))
def test_random_ops_bit_exact(seed, policy):
    rng = random.Random(seed)
    a, b = RadixCache(policy), RadixTree(policy)
    locked = []
    nxt = 0
    for _ in range(400):
        op = rng.random()
        key = [rng.randint(0, 5) for _ in range(rng.randint(0, 12))]
        if op < 0.35:
            v = list(range(nxt, nxt + len(key)))
            nxt += len(key)
            prio = rng.randint(0, 3)
            assert a.insert(key, v, prio) == b.insert(key, v, prio)
        elif op < 0.6:
            va, na = a.match_prefix(key)
            vb, nb = b.match_prefix(key)
            assert va == vb.tolist() and na.id == nb
            if va and rng.random() < 0.4:
                assert a.inc_lock_ref(na) == b.inc_lock_ref(nb)
                locked.append((na, nb))
        elif op < 0.72 and locked:
            na, nb = locked.pop(rng.randrange(len(locked)))
            assert a.dec_lock_ref(na) == b.dec_lock_ref(nb)
        else:
            n = rng.randint(1, 10)
            assert a.evict(n) == b.evict(n).tolist()
        s = b.sizes()
        assert (s["evictable"], s["protected"]) == (a.evictable_size_, a.protected_size_)
        assert s["total"] == a.total_size()
    assert _oracle_dump(a) == sorted(b.dump())


def test_long_sequences_and_splits():
    rng = np.random.default_rng(3)
    a, b = RadixCache(), RadixTree()
    base = rng.integers(0, 50, size=600).tolist()
    for i in range(30):
        cut = int(rng.integers(0, 600))
        key = base[:cut] + rng.integers(0, 50, size=int(rng.integers(1, 200))).tolist()
        v = list(range(10000 * i, 10000 * i + len(key)))
        assert a.insert(key, v) == b.insert(key, v)
        q = base[:int(rng.integers(0, 700))]
        va, na = a.match_prefix(q)
        vb, nb = b.match_prefix(q)
        assert va == vb.tolist() and na.id == nb
    assert _oracle_dump(a) == sorted(b.dump())


def test_lock_errors():
    t = RadixTree()
    t.insert([1, 2], [0, 1])
    _, n = t.match_prefix([1, 2])
    with pytest.raises(Exception):
        t.dec_lock_ref(n)           # nothing locked
    with pytest.raises(Exception):
        t.inc_lock_ref(12345)       # unknown node


def test_allocator_fifo():
    a = Allocator([5, 3, 9, 1])
    assert a.alloc(2).tolist() == [5, 3]
    a.release([7])
    assert a.available == 3
    assert a.alloc(3).tolist() == [9, 1, 7]
    with pytest.raises(Exception):
        a.alloc(1)


def test_cascade_spans_tile_shared_prefixes():
    t = RadixTree()
    # root segment A (10), children B (5) and C (7); B has children D (3), E (4)
    A = list(range(100, 110))
    B, C = [1, 2, 3, 4, 5], [6, 7, 8, 9, 10, 11, 12]
    D, E = [20, 21, 22], [30, 31, 32, 33]
    paths = [A + B + D, A + B + E, A + C, A + B + D[:1]]
    slot = 0
    last = []
    for p in paths:
        vals, _ = t.match_prefix(p)
        new = list(range(slot, slot + len(p) - len(vals)))
        slot += len(new)
        t.insert(p, list(vals) + new)
    for p in paths:
        vals, node = t.match_prefix(p)
        assert len(vals) == len(p)
        last.append(node)
    c = t.cascade(last)
    spans = [(int(c.span_start[s]), int(c.span_len[s]),
              sorted(c.grp_req[c.grp_indptr[s]:c.grp_indptr[s + 1]].tolist())) for s in range(c.num_spans)]
    # A shared by all 4; B by requests 0, 1, 3; D[:1] by requests 0 and 3
    assert (0, 10, [0, 1, 2, 3]) in spans
    assert (10, 5, [0, 1, 3]) in spans
    assert (15, 1, [0, 3]) in spans
    assert len(spans) == 3


@pytest.mark.parametrize("policy,order", [("lru", "BAC"), ("mru", "CAB"), ("lfu", "BCA"), ("slru", "BCA"),
                                          ("fifo", "ABC"), ("filo", "CBA"), ("priority", "BCA")])
def test_policy_orders_cpp(policy, order):
    # the hand-worked history of the oracle's policy pins, on the C++ tree
    t = RadixTree(policy)
    t.insert([1, 2, 3], [10, 11, 12], priority=5)
    t.insert([4, 5], [20, 21], priority=1)
    t.insert([6], [30], priority=3)
    t.match_prefix([1, 2, 3])
    t.match_prefix([1, 2, 3, 9])
    t.match_prefix([6, 7])
    values = {"A": [10, 11, 12], "B": [20, 21], "C": [30]}
    assert [t.evict(1).tolist() for _ in range(3)] == [values[x] for x in order]


def test_unknown_policy_rejected():
    from prefix_shared_kv_token_gb300 import _lib
    t = RadixTree()
    assert _lib.lib.pkv_tree_set_policy(t._h, 7) == -2      # PKV_E_UNSUPPORTED
    with pytest.raises(ValueError):
        RadixTree("random")


@pytest.mark.parametrize("seed", range(4))
def test_schedule_matches_oracle(seed):
    from oracle.schedule import schedule
    rng = random.Random(100 + seed)
    a, b = RadixCache(), RadixTree()
    for i in range(80):
        k = [rng.randint(0, 4) for _ in range(rng.randint(1, 14))]
        v = list(range(100 * i, 100 * i + len(k)))
        assert a.insert(k, v) == b.insert(k, v)
    queue = [[rng.randint(0, 4) for _ in range(rng.randint(0, 16))] for _ in range(50)]
    before = sorted(b.dump())
    for policy in ("lpm", "fcfs"):
        assert b.schedule(queue, policy) == schedule(a, queue, policy)
    assert sorted(b.dump()) == before            # scheduling leaves the tree as it was
    assert [b.match_len(q) for q in queue] == schedule(a, queue)[1]


@pytest.mark.parametrize("page", [2, 4, 16])
@pytest.mark.parametrize("seed", range(3))
def test_paged_random_ops_bit_exact(page, seed):
    """Paged trees (whole blocks of ``page`` tokens): C++ = oracle after random inserts,
    matches (with splits at block boundaries), locks, evictions and schedules."""
    from oracle.schedule import schedule
    rng = random.Random(1000 * page + seed)
    a, b = RadixCache("lru", page_size=page), RadixTree("lru", page_size=page)
    locked, nxt = [], 0
    for _ in range(300):
        op = rng.random()
        # few distinct tokens, so that keys often share leading tokens inside a block
        key = [rng.randint(0, 2) for _ in range(rng.randint(0, 5 * page))]
        if op < 0.4:
            v = list(range(nxt, nxt + len(key)))
            nxt += len(key)
            assert a.insert(key, v) == b.insert(key, v)
        elif op < 0.65:
            va, na = a.match_prefix(key)
            vb, nb = b.match_prefix(key)
            assert va == vb.tolist() and na.id == nb and len(va) % page == 0
            if va and rng.random() < 0.4:
                assert a.inc_lock_ref(na) == b.inc_lock_ref(nb)
                locked.append((na, nb))
        elif op < 0.75 and locked:
            na, nb = locked.pop(rng.randrange(len(locked)))
            assert a.dec_lock_ref(na) == b.dec_lock_ref(nb)
        else:
            n = rng.randint(1, 3 * page)
            assert a.evict(n) == b.evict(n).tolist()
        s = b.sizes()
        assert (s["evictable"], s["protected"], s["total"]) == (a.evictable_size_, a.protected_size_,
                                                              a.total_size())
    assert _oracle_dump(a) == sorted(b.dump())
    assert all(len(r[4]) % page == 0 for r in b.dump())
    queue = [[rng.randint(0, 2) for _ in range(rng.randint(0, 5 * page))] for _ in range(40)]
    for policy in ("lpm", "fcfs"):
        assert b.schedule(queue, policy) == schedule(a, queue, policy)


def test_page_size_only_on_an_empty_tree():
    from prefix_shared_kv_token_gb300 import _lib
    t = RadixTree()
    assert _lib.lib.pkv_tree_set_page_size(t._h, 0) == -1
    assert _lib.lib.pkv_tree_set_page_size(t._h, 16) == 0
    t.insert(list(range(20)), list(range(20)))
    assert _lib.lib.pkv_tree_set_page_size(t._h, 4) == -1   # holds nodes: refused
    assert t.match_prefix(list(range(20)))[0].tolist() == list(range(16))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_match_lock_batch_equals_single_calls(seed):
    # the batched match-and-lock leaves the same tree (splits, access times, hit counts,
    # locks) and returns the same values and nodes as match_prefix + inc_lock_ref per key
    rng = np.random.default_rng(seed)
    base = [rng.integers(0, 6, size=int(rng.integers(5, 40))) for _ in range(12)]
    trees = (RadixTree(), RadixTree())
    slot = 0
    for t in trees:
        slot = 0
        for k in base:
            t.insert(k, np.arange(slot, slot + len(k), dtype=np.int32))
            slot += len(k)
    keys = []
    for _ in range(30):   # prefixes that end inside nodes, past them, on nothing at all
        k = base[int(rng.integers(0, len(base)))]
        cut = int(rng.integers(0, len(k) + 1))
        tail = rng.integers(0, 6, size=int(rng.integers(0, 4)))
        keys.append(np.concatenate([k[:cut], tail]).astype(np.int32))
    keys.append(np.zeros(0, np.int32))
    single_v, single_n = [], []
    for k in keys:
        v, n = trees[0].match_prefix(k)
        trees[0].inc_lock_ref(n)
        single_v.append(v)
        single_n.append(n)
    batch_v, batch_n = trees[1].match_lock_batch(keys)
    assert [n for n in batch_n.tolist()] == single_n
    for a, b in zip(single_v, batch_v):
        assert np.array_equal(a, b)
    assert trees[0].dump() == trees[1].dump()
    assert trees[0].sizes() == trees[1].sizes()
    # the locks are real: unlocking every node returns both trees to the same evictable size
    for t, nodes in zip(trees, (single_n, batch_n)):
        for n in nodes:
            t.dec_lock_ref(int(n))
    assert trees[0].sizes() == trees[1].sizes() and trees[0].sizes()["protected"] == 0


def test_fill_batch_table_matches_row_by_row_construction():
    from prefix_shared_kv_token_gb300 import PkvError, fill_batch_table
    rng = np.random.default_rng(5)
    for _ in range(50):
        n = int(rng.integers(0, 12))
        cl = rng.integers(0, 30, size=n)
        fl = rng.integers(0, 5, size=n)
        cached = rng.integers(0, 1 << 20, size=int(cl.sum())).astype(np.int32)
        fresh = rng.integers(0, 1 << 20, size=int(fl.sum())).astype(np.int32)
        stride = int((cl + fl).max()) + int(rng.integers(0, 3)) if n else 4
        table = np.full((max(n, 1), stride), -7, dtype=np.int32)
        fill_batch_table(cached, cl, fresh, fl, table)
        want = np.full_like(table, -7)
        ca = fa = 0
        for i in range(n):
            want[i, :cl[i]] = cached[ca:ca + cl[i]]
            want[i, cl[i]:cl[i] + fl[i]] = fresh[fa:fa + fl[i]]
            ca += cl[i]
            fa += fl[i]
        assert np.array_equal(table, want)
    # a row past the stride is refused and nothing is written
    table = np.zeros((2, 4), dtype=np.int32)
    with pytest.raises(PkvError):
        fill_batch_table(np.arange(3, dtype=np.int32), [1, 2], np.arange(5, dtype=np.int32), [1, 4], table)
    assert not table.any()
