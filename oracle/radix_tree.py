"""Radix tree of token prefixes whose node values are KV-pool slot indices (oracle copy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "[SGLang] RadixAttention: Radix Tree 기반 프리픽스 캐싱의 핵심"
(blog.secrett2633.cloud/opensource/sglang/radix-cache), sections
  * "Radix Tree 구조도"             -- keys are token sequences, values are KV indices;
  * "핵심 자료구조: TreeNode"        -- children keyed by first token, parent, key, value,
                                      lock_ref, last_access_time;
  * "프리픽스 매칭: match_prefix"    -- longest-prefix walk, split on a partial match;
  * "노드 분할: _split_node"         -- upper part inherits lock_ref;
  * "삽입: _insert_helper"           -- walk, split, append the remainder as a leaf,
                                      return the already-cached length;
  * "Eviction 전략"                  -- heap of evictable leaves, parents re-queued;
  * "참조 카운트: lock_ref"          -- lock the whole path up to the root.

Readings where the page leaves a step open (each is also listed in the design notes):
  * page size 1: a node's child key is the first token of the child's key;
  * time is a logical clock that advances once per public operation (match_prefix,
    insert); every timestamp written inside one operation is that tick;
  * the insert walk's elided "split on partial match" splits exactly like match does and
    then continues from the upper half; only the node the walk starts from and the nodes
    it creates get the new timestamp (the printed loop touches no other node);
  * LRU priority is last_access_time, ties broken by node id (creation order);
  * the root is created with lock_ref = 1 (as in the page's diagram) and is never
    evicted or counted in the evictable / protected sizes.

Eviction policies ("Eviction 전략": lru, lfu, slru, fifo, mru, filo, priority, with the
node fields hit_count and priority of "핵심 자료구조: TreeNode").  The page prints only the
LRU ordering and how priority moves on insert and split; the other orderings are the
plainest reading of their names, smallest key evicted first, ties by node id:
  * lru       (last_access_time)
  * lfu       (hit_count, last_access_time)
  * slru      (hit_count >= SLRU_PROTECT, last_access_time): the probationary segment (fewer
              than SLRU_PROTECT hits) goes first, each segment in LRU order
  * fifo      (node id): the node created first
  * mru       (-last_access_time)
  * filo      (-node id): the node created last
  * priority  (priority, last_access_time): lowest priority first
hit_count: every node on the path a match_prefix returns (root excluded) gains one hit,
counted after any split.  priority: an insert raises its start node's priority to at least
its own and gives it to the leaf it creates; a split's upper part takes the child's
priority (as printed in "노드 분할"); new nodes otherwise start at 0 hits.

Paged tree (page_size P > 1; "Efficiently Programming Large Language Models using SGLang"
(summary), §Technical Details, whose cache insert refers to the KV by
16-token block, position / 16).  The plainest reading that keeps the rest of the tree's
behaviour: the cache holds whole blocks of P tokens only.
  * match_prefix and insert look at the key's first P * floor(len / P) tokens; a trailing
    partial block is never matched or inserted (it stays with the request that owns it);
  * tokens compare a block at a time: a block matches when all its P tokens are equal, so
    every node key, match length, split point and cached length is a multiple of P;
  * a node's child key is its first block (the tuple of its first P tokens);
  * everything else (times, hits, priorities, eviction, locking) is unchanged.
With P = 1 every rule above is the token tree's.
"""

from __future__ import annotations

import heapq


POLICIES = ("lru", "lfu", "slru", "fifo", "mru", "filo", "priority")
SLRU_PROTECT = 2  # hits that move a node into SLRU's protected segment


class TreeNode:
    def __init__(self, node_id: int, now: int, priority: int = 0):
        self.id = node_id
        self.children: dict[int, "TreeNode"] = {}
        self.parent: TreeNode | None = None
        self.key: list[int] = []
        self.value: list[int] = []
        self.lock_ref = 0
        self.last_access_time = now
        self.hit_count = 0
        self.priority = priority


def eviction_key(policy: str, n: TreeNode):
    """Heap key of an evictable leaf under ``policy`` (smallest evicted first)."""
    if policy == "lru":
        return (n.last_access_time, n.id)
    if policy == "lfu":
        return (n.hit_count, n.last_access_time, n.id)
    if policy == "slru":
        return (1 if n.hit_count >= SLRU_PROTECT else 0, n.last_access_time, n.id)
    if policy == "fifo":
        return (n.id,)
    if policy == "mru":
        return (-n.last_access_time, n.id)
    if policy == "filo":
        return (-n.id,)
    if policy == "priority":
        return (n.priority, n.last_access_time, n.id)
    raise ValueError(policy)


def _key_match(a, b, page: int = 1) -> int:
    """Number of equal leading tokens of a and b, counted in whole blocks of ``page``
    tokens (a block counts only when all of its tokens are equal)."""
    n = 0
    if page == 1:
        for x, y in zip(a, b):
            if x != y:
                break
            n += 1
        return n
    while n + page <= min(len(a), len(b)) and list(a[n:n + page]) == list(b[n:n + page]):
        n += page
    return n


class RadixCache:
    def __init__(self, policy: str = "lru", page_size: int = 1):
        if policy not in POLICIES:
            raise ValueError(policy)
        if page_size < 1:
            raise ValueError(page_size)
        self.page = page_size
        self.policy = policy
        self._next_id = 0
        self.clock = 0
        self.root = self._new_node()
        self.root.lock_ref = 1
        self.evictable_size_ = 0
        self.protected_size_ = 0

    def _new_node(self, priority: int = 0) -> TreeNode:
        n = TreeNode(self._next_id, self.clock, priority)
        self._next_id += 1
        return n

    def _child_key(self, key):
        """Key of a child in its parent's table: its first token, or its first block."""
        return key[0] if self.page == 1 else tuple(key[:self.page])

    def _aligned(self, key):
        return list(key)[:len(key) // self.page * self.page]

    # ---- match -------------------------------------------------------------------
    def match_prefix(self, key):
        """Longest cached prefix of ``key``: (concatenated slot values, last node)."""
        self.clock += 1
        key = self._aligned(key)
        node = self.root
        node.last_access_time = self.clock
        values = []
        while key and self._child_key(key) in node.children:
            child = node.children[self._child_key(key)]
            child.last_access_time = self.clock
            n = _key_match(child.key, key, self.page)
            if n < len(child.key):
                upper = self._split_node(child.key, child, n)
                values.extend(upper.value)
                node = upper
                break
            values.extend(child.value)
            node = child
            key = key[n:]
        hit = node
        while hit is not self.root:
            hit.hit_count += 1
            hit = hit.parent
        return values, node

    def _split_node(self, key, child: TreeNode, split_len: int) -> TreeNode:
        upper = self._new_node(child.priority)
        upper.children = {self._child_key(key[split_len:]): child}
        upper.parent = child.parent
        upper.lock_ref = child.lock_ref
        upper.key = child.key[:split_len]
        upper.value = child.value[:split_len]
        child.parent = upper
        child.key = child.key[split_len:]
        child.value = child.value[split_len:]
        upper.parent.children[self._child_key(key)] = upper
        return upper

    # ---- insert ------------------------------------------------------------------
    def insert(self, key, value, priority: int = 0) -> int:
        """Insert ``key`` -> ``value``; returns how many leading tokens were already cached
        (the caller frees those entries of ``value``, they duplicate cached slots)."""
        assert len(key) == len(value)
        self.clock += 1
        key, value = self._aligned(key), list(value)[:len(self._aligned(key))]
        node = self.root
        node.last_access_time = self.clock
        node.priority = max(node.priority, priority)
        total = 0
        while key and self._child_key(key) in node.children:
            node = node.children[self._child_key(key)]
            n = _key_match(node.key, key, self.page)
            total += n
            key, value = key[n:], value[n:]
            if n < len(node.key):
                node = self._split_node(node.key, node, n)
        if key:
            leaf = self._new_node(priority)
            leaf.parent = node
            leaf.key = key
            leaf.value = value
            node.children[self._child_key(key)] = leaf
            self.evictable_size_ += len(key)
        return total

    # ---- eviction ----------------------------------------------------------------
    def _all_nodes(self):
        out, stack = [], [self.root]
        while stack:
            n = stack.pop()
            out.append(n)
            stack.extend(n.children.values())
        return out

    def evict(self, num_tokens: int):
        """Free at least ``num_tokens`` slots from unlocked leaves in the policy's order
        (LRU: least recently used first); returns the freed slot values in the order they
        were freed."""
        heap = [(eviction_key(self.policy, n), n) for n in self._all_nodes()
                if n is not self.root and not n.children and n.lock_ref == 0]
        heapq.heapify(heap)
        freed, evicted = [], 0
        while evicted < num_tokens and heap:
            _, x = heapq.heappop(heap)
            freed.extend(x.value)
            evicted += len(x.value)
            parent = x.parent
            del parent.children[self._child_key(x.key)]
            self.evictable_size_ -= len(x.key)
            if not parent.children and parent.lock_ref == 0:
                heapq.heappush(heap, (eviction_key(self.policy, parent), parent))
        return freed

    # ---- locking -----------------------------------------------------------------
    def inc_lock_ref(self, node: TreeNode) -> int:
        delta = 0
        while node is not self.root:
            if node.lock_ref == 0:
                self.evictable_size_ -= len(node.key)
                self.protected_size_ += len(node.key)
                delta -= len(node.key)
            node.lock_ref += 1
            node = node.parent
        return delta

    def dec_lock_ref(self, node: TreeNode) -> int:
        delta = 0
        while node is not self.root:
            if node.lock_ref == 1:
                self.evictable_size_ += len(node.key)
                self.protected_size_ -= len(node.key)
                delta += len(node.key)
            node.lock_ref -= 1
            node = node.parent
        return delta

    # ---- inspection --------------------------------------------------------------
    def total_size(self) -> int:
        return sum(len(n.key) for n in self._all_nodes() if n is not self.root)

    def node_by_id(self, node_id: int):
        for n in self._all_nodes():
            if n.id == node_id:
                return n
        return None

    def dump(self):
        """Canonical description: sorted (id, parent id, key, value, lock_ref, time)."""
        rows = []
        for n in self._all_nodes():
            rows.append((n.id, -1 if n.parent is None else n.parent.id, tuple(n.key),
                         tuple(n.value), n.lock_ref, n.last_access_time))
        return sorted(rows)
