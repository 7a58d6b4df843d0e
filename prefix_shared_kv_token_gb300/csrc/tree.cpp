// Host radix tree of token prefixes (values = KV-pool slots) and the token-slot allocator.
//
// Semantics follow "[SGLang] RadixAttention: Radix Tree 기반 프리픽스 캐싱의 핵심"
// (blog.secrett2633.cloud/opensource/sglang/radix-cache):
//   TreeNode            -- children keyed by the first token, parent, key, value, lock_ref,
//                          last_access_time ("핵심 자료구조: TreeNode");
//   match_prefix        -- longest-prefix walk, a partial match splits the child
//                          ("프리픽스 매칭: match_prefix", "노드 분할: _split_node");
//   insert              -- walk, split on a partial match, append the remainder as a leaf,
//                          return the already-cached length ("삽입: _insert_helper");
//   evict               -- heap of unlocked leaves by last access, parents re-queued once
//                          they become unlocked leaves ("Eviction 전략");
//   inc/dec_lock_ref    -- lock the path up to the root ("참조 카운트: lock_ref").
// Readings where the page leaves a step open: page size 1; a logical clock that ticks once
// per match_prefix / insert; the insert walk only stamps the node it starts from and the
// nodes it creates; LRU ties break by node id; the root starts with lock_ref 1.
//
// Eviction policies ("Eviction 전략": lru, lfu, slru, fifo, mru, filo, priority, using the
// node fields hit_count and priority).  Only the LRU order and how priority moves on insert
// and split are printed; the rest is the plainest reading of each name, smallest key first,
// ties by node id: lru (last access), lfu (hits, last access), slru (hits >= 2, last access:
// the probationary segment first), fifo (id), mru (-last access), filo (-id), priority
// (priority, last access).  A match_prefix adds one hit to every node of the path it
// returns (after any split); an insert raises its start node's priority to its own and gives
// it to the leaf it creates; a split's upper part takes the child's priority.
//
// Paged tree (pkv_tree_set_page_size, P > 1; "Efficiently Programming Large Language Models
// using SGLang", §Technical Details: its cache's insert refers to the KV by
// 16-token block: position / 16): the cache holds whole blocks of P tokens.  match_prefix
// and insert use the key's first P * floor(n / P) tokens, tokens compare a block at a time
// (a block matches when all its tokens are equal), and a child is keyed by its first block.
// Every node key, match length, split point and cached length is then a multiple of P.
//
// The cascade extraction (pkv_tree_cascade) turns the nodes shared by several requests of a
// batch into spans for the attention kernels: the tree already knows which prefix KV is
// shared ("Radix Tree 구조도": both branches under [1,2,3] share its KV).

#include <algorithm>
#include <array>
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <queue>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace {

struct Node {
    int64_t id = 0;
    int64_t parent = -1;
    std::unordered_map<int64_t, int64_t> children;  // child key (first token / block id) -> id
    std::vector<int32_t> key;
    std::vector<int32_t> value;
    int64_t lock_ref = 0;
    int64_t last_access_time = 0;
    int64_t hit_count = 0;
    int64_t priority = 0;
    bool alive = true;
};

constexpr int64_t kSlruProtect = 2;  // hits that move a node into SLRU's protected segment
constexpr int64_t kNoBlock = INT64_MIN;  // a block that no node's key starts with

struct BlockHash {
    size_t operator()(const std::vector<int32_t> &b) const {
        uint64_t h = 1469598103934665603ull;  // FNV-1a over the tokens
        for (int32_t t : b) {
            h ^= (uint32_t)t;
            h *= 1099511628211ull;
        }
        return (size_t)h;
    }
};

}  // namespace

struct pkv_tree {
    std::vector<Node> nodes;  // indexed by id; evicted nodes stay as tombstones
    int64_t clock = 0;
    int64_t evictable = 0;
    int64_t protected_ = 0;
    int64_t live = 0;
    int policy = PKV_EVICT_LRU;
    int64_t page = 1;  // tokens per block
    // paged tree: block contents -> small id, for the child tables (a block is interned when
    // a node key first starts with it)
    std::unordered_map<std::vector<int32_t>, int64_t, BlockHash> block_ids;

    pkv_tree() {
        Node root;
        root.id = 0;
        root.lock_ref = 1;
        nodes.push_back(std::move(root));
        live = 1;
    }

    int64_t new_node(int64_t priority = 0) {
        Node n;
        n.id = (int64_t)nodes.size();
        n.last_access_time = clock;
        n.priority = priority;
        nodes.push_back(std::move(n));
        ++live;
        return nodes.back().id;
    }

    // Equal leading tokens of a and b, in whole blocks.
    int64_t key_match(const int32_t *a, int64_t na, const int32_t *b, int64_t nb) const {
        int64_t n = std::min(na, nb), i = 0;
        while (i < n && a[i] == b[i]) ++i;
        return i / page * page;
    }

    // Key of a child whose key starts at k: its first token, or its block's id (interned
    // when `create`, else kNoBlock for a block no node starts with).
    int64_t child_key(const int32_t *k, bool create) {
        if (page == 1) return k[0];
        std::vector<int32_t> b(k, k + page);
        auto it = block_ids.find(b);
        if (it != block_ids.end()) return it->second;
        if (!create) return kNoBlock;
        const int64_t id = (int64_t)block_ids.size();
        block_ids.emplace(std::move(b), id);
        return id;
    }
    int64_t find_child(int64_t node, const int32_t *k) {
        const int64_t ck = child_key(k, false);
        if (ck == kNoBlock) return -1;
        auto it = nodes[node].children.find(ck);
        return it == nodes[node].children.end() ? -1 : it->second;
    }

    // Split `child` after split_len tokens; returns the new upper node.
    int64_t split(int64_t child, int64_t split_len) {
        int64_t up = new_node(nodes[child].priority);  // may reallocate `nodes`: index by id only
        Node &c = nodes[child];
        Node &u = nodes[up];
        u.parent = c.parent;
        u.lock_ref = c.lock_ref;
        u.key.assign(c.key.begin(), c.key.begin() + split_len);
        u.value.assign(c.value.begin(), c.value.begin() + split_len);
        c.key.erase(c.key.begin(), c.key.begin() + split_len);
        c.value.erase(c.value.begin(), c.value.begin() + split_len);
        c.parent = up;
        const int64_t ck = child_key(c.key.data(), true), uk = child_key(u.key.data(), true);
        nodes[up].children[ck] = child;
        nodes[nodes[up].parent].children[uk] = up;
        return up;
    }

    int64_t match(const int32_t *key, int64_t n, std::vector<int32_t> *values) {
        ++clock;
        n = n / page * page;
        int64_t node = 0;
        nodes[0].last_access_time = clock;
        int64_t pos = 0;
        while (pos < n) {
            const int64_t child = find_child(node, key + pos);
            if (child < 0) break;
            nodes[child].last_access_time = clock;
            int64_t m = key_match(nodes[child].key.data(), (int64_t)nodes[child].key.size(),
                                  key + pos, n - pos);
            if (m < (int64_t)nodes[child].key.size()) {
                int64_t up = split(child, m);
                values->insert(values->end(), nodes[up].value.begin(), nodes[up].value.end());
                node = up;
                break;
            }
            values->insert(values->end(), nodes[child].value.begin(), nodes[child].value.end());
            node = child;
            pos += m;
        }
        for (int64_t x = node; x != 0; x = nodes[x].parent) nodes[x].hit_count += 1;
        return node;
    }

    // Cached prefix length of key without touching the tree (no split, no time, no hit).
    int64_t peek(const int32_t *key, int64_t n) {
        n = n / page * page;
        int64_t node = 0, pos = 0;
        while (pos < n) {
            const int64_t child = find_child(node, key + pos);
            if (child < 0) break;
            const Node &c = nodes[child];
            int64_t m = key_match(c.key.data(), (int64_t)c.key.size(), key + pos, n - pos);
            pos += m;
            if (m < (int64_t)c.key.size()) break;
            node = c.id;
        }
        return pos;
    }

    int64_t insert(const int32_t *key, const int32_t *value, int64_t n, int64_t priority) {
        ++clock;
        n = n / page * page;
        int64_t node = 0;
        nodes[0].last_access_time = clock;
        nodes[0].priority = std::max(nodes[0].priority, priority);
        int64_t pos = 0, total = 0;
        while (pos < n) {
            const int64_t child = find_child(node, key + pos);
            if (child < 0) break;
            node = child;
            int64_t m = key_match(nodes[node].key.data(), (int64_t)nodes[node].key.size(),
                                  key + pos, n - pos);
            total += m;
            pos += m;
            if (m < (int64_t)nodes[node].key.size()) node = split(node, m);
        }
        if (pos < n) {
            int64_t leaf = new_node(priority);
            Node &l = nodes[leaf];
            l.parent = node;
            l.key.assign(key + pos, key + n);
            l.value.assign(value + pos, value + n);
            nodes[node].children[child_key(key + pos, true)] = leaf;
            evictable += n - pos;
        }
        return total;
    }

    bool evictable_leaf(const Node &x) const {
        return x.alive && x.id != 0 && x.children.empty() && x.lock_ref == 0;
    }

    // Heap key of an evictable leaf under the tree's policy (smallest evicted first; the id
    // breaks every tie and is the last component).
    using Key = std::array<int64_t, 3>;
    Key eviction_key(const Node &x) const {
        switch (policy) {
            case PKV_EVICT_LFU: return {x.hit_count, x.last_access_time, x.id};
            case PKV_EVICT_SLRU: return {x.hit_count >= kSlruProtect ? 1 : 0, x.last_access_time, x.id};
            case PKV_EVICT_FIFO: return {x.id, 0, 0};
            case PKV_EVICT_MRU: return {-x.last_access_time, x.id, 0};
            case PKV_EVICT_FILO: return {-x.id, 0, 0};
            case PKV_EVICT_PRIORITY: return {x.priority, x.last_access_time, x.id};
            default: return {x.last_access_time, x.id, 0};
        }
    }

    void evict(int64_t num_tokens, std::vector<int32_t> *freed) {
        using Item = std::pair<Key, int64_t>;  // (key, id)
        std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
        for (const Node &x : nodes)
            if (evictable_leaf(x)) heap.push({eviction_key(x), x.id});
        int64_t evicted = 0;
        while (evicted < num_tokens && !heap.empty()) {
            int64_t id = heap.top().second;
            heap.pop();
            Node &x = nodes[id];
            freed->insert(freed->end(), x.value.begin(), x.value.end());
            evicted += (int64_t)x.value.size();
            Node &p = nodes[x.parent];
            p.children.erase(child_key(x.key.data(), false));
            evictable -= (int64_t)x.key.size();
            x.alive = false;
            x.children.clear();
            std::vector<int32_t>().swap(x.key);
            std::vector<int32_t>().swap(x.value);
            --live;
            if (p.children.empty() && p.lock_ref == 0 && p.id != 0) heap.push({eviction_key(p), p.id});
        }
    }

    int64_t inc_lock(int64_t node) {
        int64_t delta = 0;
        while (node != 0) {
            Node &x = nodes[node];
            if (x.lock_ref == 0) {
                evictable -= (int64_t)x.key.size();
                protected_ += (int64_t)x.key.size();
                delta -= (int64_t)x.key.size();
            }
            x.lock_ref += 1;
            node = x.parent;
        }
        return delta;
    }

    int64_t dec_lock(int64_t node) {
        int64_t delta = 0;
        while (node != 0) {
            Node &x = nodes[node];
            if (x.lock_ref == 1) {
                evictable += (int64_t)x.key.size();
                protected_ -= (int64_t)x.key.size();
                delta += (int64_t)x.key.size();
            }
            x.lock_ref -= 1;
            node = x.parent;
        }
        return delta;
    }

    int64_t max_leaf_len() const {
        int64_t m = 0;
        for (const Node &x : nodes)
            if (evictable_leaf(x)) m = std::max<int64_t>(m, (int64_t)x.key.size());
        return m;
    }

    bool valid(int64_t id) const { return id >= 0 && id < (int64_t)nodes.size() && nodes[id].alive; }
};

struct pkv_allocator {
    std::deque<int32_t> free_list;
};

extern "C" {

pkv_tree *pkv_tree_new(void) { return new (std::nothrow) pkv_tree(); }

void pkv_tree_free(pkv_tree *t) { delete t; }

int pkv_tree_match_prefix(pkv_tree *t, const int32_t *key, int64_t n, int32_t *values,
                          int64_t values_cap, int64_t *matched, int64_t *last_node) {
    if (!t || n < 0 || (n > 0 && !key) || !matched || !last_node) return PKV_E_INVALID;
    std::vector<int32_t> v;
    v.reserve((size_t)n);
    int64_t node = t->match(key, n, &v);
    *matched = (int64_t)v.size();
    *last_node = node;
    if (values) {
        int64_t m = std::min<int64_t>((int64_t)v.size(), values_cap);
        if (m > 0) std::memcpy(values, v.data(), sizeof(int32_t) * (size_t)m);
    }
    return PKV_OK;
}

int pkv_tree_insert(pkv_tree *t, const int32_t *key, const int32_t *value, int64_t n,
                    int64_t *prefix_len) {
    return pkv_tree_insert_priority(t, key, value, n, 0, prefix_len);
}

int pkv_tree_insert_priority(pkv_tree *t, const int32_t *key, const int32_t *value, int64_t n,
                             int64_t priority, int64_t *prefix_len) {
    if (!t || n < 0 || (n > 0 && (!key || !value))) return PKV_E_INVALID;
    int64_t total = t->insert(key, value, n, priority);
    if (prefix_len) *prefix_len = total;
    return PKV_OK;
}

int pkv_tree_set_page_size(pkv_tree *t, int32_t page_size) {
    if (!t || page_size < 1 || page_size > 4096) return PKV_E_INVALID;
    if (t->live != 1) return PKV_E_INVALID;  // only while the tree holds nothing
    t->page = page_size;
    t->block_ids.clear();
    return PKV_OK;
}

int pkv_tree_set_policy(pkv_tree *t, int policy) {
    if (!t) return PKV_E_INVALID;
    if (policy < PKV_EVICT_LRU || policy > PKV_EVICT_PRIORITY) return PKV_E_UNSUPPORTED;
    t->policy = policy;
    return PKV_OK;
}

int pkv_tree_evict(pkv_tree *t, int64_t num_tokens, int32_t *freed, int64_t freed_cap,
                   int64_t *num_freed) {
    if (!t || num_tokens < 0 || !num_freed) return PKV_E_INVALID;
    // every freed slot belongs to an unlocked node, so the evictable size bounds the output;
    // refuse up front rather than evict into a buffer that cannot hold the result
    if (freed_cap < std::min<int64_t>(t->evictable, num_tokens + t->max_leaf_len()))
        return PKV_E_WORKSPACE;
    std::vector<int32_t> f;
    t->evict(num_tokens, &f);
    if ((int64_t)f.size() > freed_cap) return PKV_E_WORKSPACE;  // unreachable by the check
    if (!f.empty()) {
        if (!freed) return PKV_E_INVALID;
        std::memcpy(freed, f.data(), sizeof(int32_t) * f.size());
    }
    *num_freed = (int64_t)f.size();
    return PKV_OK;
}

int pkv_tree_match_len(pkv_tree *t, const int32_t *key, int64_t n, int64_t *len) {
    if (!t || n < 0 || (n > 0 && !key) || !len) return PKV_E_INVALID;
    *len = t->peek(key, n);
    return PKV_OK;
}

int pkv_schedule(pkv_tree *t, const int32_t *tokens, const int64_t *offsets, int32_t n, int policy,
                 int32_t *order, int64_t *match_len) {
    if (!t || n < 0 || (n > 0 && (!offsets || !order))) return PKV_E_INVALID;
    if (policy != PKV_SCHED_LPM && policy != PKV_SCHED_FCFS) return PKV_E_UNSUPPORTED;
    std::vector<int64_t> len((size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        const int64_t a = offsets[i], b = offsets[i + 1];
        if (a < 0 || b < a || (b > a && !tokens)) return PKV_E_INVALID;
        len[(size_t)i] = t->peek(tokens + a, b - a);
    }
    for (int32_t i = 0; i < n; ++i) order[i] = i;
    if (policy == PKV_SCHED_LPM)
        std::stable_sort(order, order + n, [&](int32_t x, int32_t y) { return len[(size_t)x] > len[(size_t)y]; });
    if (match_len)
        for (int32_t i = 0; i < n; ++i) match_len[i] = len[(size_t)i];
    return PKV_OK;
}

int pkv_tree_inc_lock_ref(pkv_tree *t, int64_t node, int64_t *delta) {
    if (!t) return PKV_E_INVALID;
    if (!t->valid(node)) return PKV_E_NOTFOUND;
    int64_t d = t->inc_lock(node);
    if (delta) *delta = d;
    return PKV_OK;
}

int pkv_tree_match_lock_batch(pkv_tree *t, const int32_t *keys, const int64_t *offsets, int32_t n,
                              int32_t *values, int64_t *matched, int64_t *last_nodes) {
    if (!t || n < 0 || (n > 0 && (!offsets || !values || !matched || !last_nodes))) return PKV_E_INVALID;
    if (n > 0 && offsets[0] != 0) return PKV_E_INVALID;
    for (int32_t i = 0; i < n; ++i)
        if (offsets[i + 1] < offsets[i]) return PKV_E_INVALID;
    if (n > 0 && offsets[n] > 0 && !keys) return PKV_E_INVALID;
    std::vector<int32_t> v;
    int64_t at = 0;
    for (int32_t i = 0; i < n; ++i) {
        v.clear();
        const int64_t node = t->match(keys + offsets[i], offsets[i + 1] - offsets[i], &v);
        if (!v.empty()) std::memcpy(values + at, v.data(), sizeof(int32_t) * v.size());
        at += (int64_t)v.size();
        matched[i] = (int64_t)v.size();
        last_nodes[i] = node;
        t->inc_lock(node);
    }
    return PKV_OK;
}

int pkv_tree_dec_lock_ref(pkv_tree *t, int64_t node, int64_t *delta) {
    if (!t) return PKV_E_INVALID;
    if (!t->valid(node)) return PKV_E_NOTFOUND;
    // refuse to unlock below zero: the walk would corrupt the size bookkeeping
    for (int64_t x = node; x != 0; x = t->nodes[x].parent)
        if (t->nodes[x].lock_ref <= 0) return PKV_E_INVALID;
    int64_t d = t->dec_lock(node);
    if (delta) *delta = d;
    return PKV_OK;
}

int pkv_tree_sizes(pkv_tree *t, int64_t *evictable, int64_t *protected_size, int64_t *total,
                   int64_t *num_nodes) {
    if (!t) return PKV_E_INVALID;
    if (evictable) *evictable = t->evictable;
    if (protected_size) *protected_size = t->protected_;
    if (total) {
        int64_t s = 0;
        for (const Node &x : t->nodes)
            if (x.alive && x.id != 0) s += (int64_t)x.key.size();
        *total = s;
    }
    if (num_nodes) *num_nodes = t->live;
    return PKV_OK;
}

int pkv_tree_dump(pkv_tree *t, int64_t *out, int64_t cap, int64_t *used) {
    if (!t || !used) return PKV_E_INVALID;
    int64_t need = 0;
    for (const Node &x : t->nodes)
        if (x.alive) need += 8 + 2 * (int64_t)x.key.size();
    *used = need;
    if (!out || cap < need) return out ? PKV_E_WORKSPACE : PKV_OK;
    int64_t k = 0;
    for (const Node &x : t->nodes) {
        if (!x.alive) continue;
        out[k++] = x.id;
        out[k++] = x.parent;
        out[k++] = x.lock_ref;
        out[k++] = x.last_access_time;
        out[k++] = (int64_t)x.key.size();
        out[k++] = (int64_t)x.children.size();
        out[k++] = x.hit_count;
        out[k++] = x.priority;
        for (int32_t v : x.key) out[k++] = v;
        for (int32_t v : x.value) out[k++] = v;
    }
    return PKV_OK;
}

int pkv_tree_cascade(pkv_tree *t, const int64_t *last_nodes, int32_t batch, int32_t min_group,
                     int32_t *span_req, int32_t *span_start, int32_t *span_len,
                     int32_t *grp_indptr, int32_t *grp_req, int32_t cap_spans,
                     int32_t cap_members, int32_t *num_spans, int32_t *num_members) {
    if (!t || batch < 0 || (batch > 0 && !last_nodes) || !num_spans || !num_members)
        return PKV_E_INVALID;
    if (min_group < 2) min_group = 2;
    // paths root -> last node (root excluded), and the members of every node
    std::vector<std::vector<int64_t>> paths((size_t)batch);
    std::unordered_map<int64_t, std::vector<int32_t>> members;
    for (int32_t r = 0; r < batch; ++r) {
        int64_t x = last_nodes[r];
        if (!t->valid(x)) return PKV_E_NOTFOUND;
        for (; x != 0; x = t->nodes[x].parent) paths[r].push_back(x);
        std::reverse(paths[r].begin(), paths[r].end());
        for (int64_t n : paths[r]) members[n].push_back(r);
    }
    struct Span { int32_t req, start, len; int64_t head; };
    std::vector<Span> spans;
    std::unordered_map<int64_t, int32_t> span_of_head;  // first node of a span -> span index
    std::vector<int32_t> member_flat, indptr{0};
    for (int32_t r = 0; r < batch; ++r) {
        int64_t pos = 0;
        int64_t cur_head = -1;
        for (size_t i = 0; i < paths[r].size(); ++i) {
            int64_t n = paths[r][i];
            const auto &mem = members[n];
            int64_t len = (int64_t)t->nodes[n].key.size();
            if ((int32_t)mem.size() < min_group) break;  // shared nodes form a prefix
            bool fuse = cur_head >= 0 && members[cur_head].size() == mem.size();
            if (!fuse) {
                cur_head = n;
                auto it = span_of_head.find(n);
                if (it == span_of_head.end()) {
                    span_of_head[n] = (int32_t)spans.size();
                    spans.push_back({mem[0], (int32_t)pos, (int32_t)len, n});
                    member_flat.insert(member_flat.end(), mem.begin(), mem.end());
                    indptr.push_back((int32_t)member_flat.size());
                }
            } else if (members[cur_head][0] == r) {
                // first member extends the fused span (every member walks the same chain)
                spans[span_of_head[cur_head]].len += (int32_t)len;
            }
            pos += len;
        }
    }
    *num_spans = (int32_t)spans.size();
    *num_members = (int32_t)member_flat.size();
    if ((int32_t)spans.size() > cap_spans || (int32_t)member_flat.size() > cap_members)
        return (cap_spans == 0 && cap_members == 0) ? PKV_OK : PKV_E_WORKSPACE;
    if (!spans.empty() && (!span_req || !span_start || !span_len || !grp_indptr || !grp_req))
        return PKV_E_INVALID;
    for (size_t s = 0; s < spans.size(); ++s) {
        span_req[s] = spans[s].req;
        span_start[s] = spans[s].start;
        span_len[s] = spans[s].len;
    }
    if (grp_indptr)
        for (size_t s = 0; s <= spans.size(); ++s) grp_indptr[s] = indptr[s];
    if (!member_flat.empty()) std::memcpy(grp_req, member_flat.data(), sizeof(int32_t) * member_flat.size());
    return PKV_OK;
}

pkv_allocator *pkv_allocator_new(const int32_t *free_slots, int64_t n) {
    if (n < 0 || (n > 0 && !free_slots)) return nullptr;
    auto *a = new (std::nothrow) pkv_allocator();
    if (!a) return nullptr;
    a->free_list.assign(free_slots, free_slots + n);
    return a;
}

void pkv_allocator_free_all(pkv_allocator *a) { delete a; }

int pkv_allocator_alloc(pkv_allocator *a, int64_t n, int32_t *out) {
    if (!a || n < 0 || (n > 0 && !out)) return PKV_E_INVALID;
    if ((int64_t)a->free_list.size() < n) return PKV_E_NOSPACE;
    for (int64_t i = 0; i < n; ++i) {
        out[i] = a->free_list.front();
        a->free_list.pop_front();
    }
    return PKV_OK;
}

int pkv_allocator_release(pkv_allocator *a, const int32_t *slots, int64_t n) {
    if (!a || n < 0 || (n > 0 && !slots)) return PKV_E_INVALID;
    a->free_list.insert(a->free_list.end(), slots, slots + n);
    return PKV_OK;
}

int64_t pkv_allocator_available(const pkv_allocator *a) { return a ? (int64_t)a->free_list.size() : 0; }

}  // extern "C"
