// rx_host.cpp -- host side of librx: error layer, radix tree, slot free list,
// request admission and the decode-plan builder.
//
// The radix tree follows "SGLang: Efficient Execution of Structured Language
// Model Programs" (unite.ai, es): section "Introducción a SGLang"
// (RadixAttention: an LRU cache of KV inside a radix tree with matching,
// insertion and eviction) and section "SGLang: Modelo de programación y
// metodología" (nine-step walkthrough: token-sequence edges, an extension
// becomes a new node, a partial share splits a node, least recently used
// nodes are evicted).  Node boundaries are kept as inserts made them; nodes
// are never merged.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <map>
#include <memory>
#include <new>
#include <set>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include "rx.h"
#include "rx_internal.h"

// ---------------------------------------------------------------------------
// error layer
// ---------------------------------------------------------------------------

static thread_local std::string g_last_error;

int rx_set_error(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

extern "C" const char *rx_last_error(void) { return g_last_error.c_str(); }

// Allocation-failure hook for tests: the n-th next radix-tree node
// allocation (counting from 1) throws std::bad_alloc, as a failing host
// allocator would; 0 disables it.
static std::atomic<int64_t> g_fail_alloc_in{0};

extern "C" int rx_test_fail_alloc(int64_t n)
{
    if (n < 0) return rx_set_error(RX_ERR_INVALID, "rx_test_fail_alloc: n < 0");
    g_fail_alloc_in.store(n);
    return RX_OK;
}

// Counts one host allocation against the hook; throws when it is the one
// the hook names.
static void count_alloc()
{
    int64_t left = g_fail_alloc_in.load();
    while (left > 0) {
        if (g_fail_alloc_in.compare_exchange_weak(left, left - 1)) {
            if (left == 1) throw std::bad_alloc();
            return;
        }
    }
}
extern "C" int rx_version(void) { return RX_ABI_VERSION; }

// Layered pools: one layer's rows are num_slots * num_kv_heads * head_dim
// elements (bf16, or one byte for FP8 codes) after the previous layer's.
template <class Pool>
static int pool_layer(const Pool *in, Pool *out, int64_t elem_bytes, const char *who)
{
    *out = *in;
    const int32_t L = in->num_layers;
    if (L < 0 || in->layer < 0 || in->layer >= (L > 1 ? L : 1))
        return rx_set_error(RX_ERR_INVALID, "%s: layer %d of a pool of %d layers", who, in->layer, L);
    if (in->layer > 0) {
        const int64_t off = (int64_t)in->layer * in->num_slots * in->num_kv_heads * in->head_dim * elem_bytes;
        out->k = static_cast<char *>(in->k) + off;
        out->v = static_cast<char *>(in->v) + off;
    }
    out->num_layers = 0;
    out->layer = 0;
    return RX_OK;
}

int rx_pool_layer(const void *in, void *out, int fp8, const char *who)
{
    if (!in) return RX_OK;
    if (fp8)
        return pool_layer(static_cast<const rx_kv_pool_fp8 *>(in), static_cast<rx_kv_pool_fp8 *>(out), 1, who);
    return pool_layer(static_cast<const rx_kv_pool *>(in), static_cast<rx_kv_pool *>(out), 2, who);
}

// ---------------------------------------------------------------------------
// radix tree
// ---------------------------------------------------------------------------

namespace {

struct Node {
    int64_t id = 0;
    Node *parent = nullptr;
    std::vector<int64_t> tok;
    std::vector<int32_t> slot;
    std::vector<int32_t> lock;          // per token
    int64_t nlocked = 0;                // tokens with lock > 0
    int64_t last = 0;                   // last-access clock value
    std::unordered_map<int64_t, Node *> kids;  // keyed by first token
    bool in_leafset = false;
    std::pair<int64_t, int64_t> key{0, 0};
};

struct Walk {
    std::vector<Node *> nodes;  // nodes holding >= 1 matched token, root excluded
    int64_t matched = 0;        // tokens matched
    int64_t in_last = 0;        // tokens matched inside nodes.back()
};

}  // namespace

struct rx_tree {
    Node root;
    int64_t clock = 0;
    int64_t next_id = 1;
    int64_t cached = 0;
    int64_t n_nodes = 0;
    // evictable leaves ordered by (last access, id)
    std::set<std::pair<int64_t, int64_t>> leaves;
    std::unordered_map<int64_t, Node *> by_id;

    ~rx_tree() { free_subtree(&root); }

    void free_subtree(Node *n)
    {
        std::vector<Node *> stack;
        for (auto &kv : n->kids) stack.push_back(kv.second);
        n->kids.clear();
        while (!stack.empty()) {
            Node *x = stack.back();
            stack.pop_back();
            for (auto &kv : x->kids) stack.push_back(kv.second);
            delete x;
        }
    }

    void refresh(Node *n)
    {
        if (n == &root) return;
        if (n->in_leafset) {
            leaves.erase(n->key);
            n->in_leafset = false;
        }
        if (n->kids.empty() && n->nlocked == 0) {
            n->key = {n->last, n->id};
            leaves.insert(n->key);
            n->in_leafset = true;
        }
    }

    // A node, allocated but not yet part of the tree: operations allocate
    // every node they need before they change anything, so that a failed
    // allocation leaves the tree as it was.
    static Node *raw_node()
    {
        count_alloc();
        return new Node();
    }

    Node *adopt(Node *n, Node *parent)
    {
        n->id = next_id++;
        n->parent = parent;
        by_id[n->id] = n;
        ++n_nodes;
        return n;
    }

    Walk walk(const int64_t *t, int64_t n)
    {
        Walk w;
        Node *cur = &root;
        int64_t pos = 0;
        while (pos < n) {
            auto it = cur->kids.find(t[pos]);
            if (it == cur->kids.end()) break;
            Node *c = it->second;
            int64_t len = (int64_t)c->tok.size(), m = 0;
            while (m < len && pos + m < n && c->tok[m] == t[pos + m]) ++m;
            w.nodes.push_back(c);
            pos += m;
            w.in_last = m;
            if (m < len) break;
            cur = c;
        }
        w.matched = pos;
        return w;
    }

    void tick(const Walk &w)
    {
        for (Node *n : w.nodes) {
            n->last = clock;
            refresh(n);
        }
    }

    // Split n after its first k tokens; n keeps the upper part, the lower
    // part goes to `lo` (a node from raw_node).
    Node *split(Node *n, int64_t k, Node *lo)
    {
        adopt(lo, n);
        lo->tok.assign(n->tok.begin() + k, n->tok.end());
        lo->slot.assign(n->slot.begin() + k, n->slot.end());
        lo->lock.assign(n->lock.begin() + k, n->lock.end());
        lo->last = n->last;
        lo->kids.swap(n->kids);
        for (auto &kv : lo->kids) kv.second->parent = lo;
        n->tok.resize(k);
        n->slot.resize(k);
        n->lock.resize(k);
        n->nlocked = 0;
        for (int32_t c : n->lock) n->nlocked += c > 0;
        lo->nlocked = 0;
        for (int32_t c : lo->lock) lo->nlocked += c > 0;
        n->kids[lo->tok[0]] = lo;
        refresh(lo);
        refresh(n);
        return lo;
    }

    void remove_leaf(Node *n)
    {
        Node *p = n->parent;
        p->kids.erase(n->tok[0]);
        if (n->in_leafset) leaves.erase(n->key);
        by_id.erase(n->id);
        cached -= (int64_t)n->tok.size();
        --n_nodes;
        delete n;
        refresh(p);
    }

    // Evicts into `out` (appending) until `want` slots were appended or no
    // evictable leaf remains.  With cap >= 0, stops before a node that would
    // take out past cap and returns false.
    bool evict(int64_t want, std::vector<int32_t> &out, int64_t cap)
    {
        int64_t got = 0;
        while (got < want && !leaves.empty()) {
            Node *n = by_id[leaves.begin()->second];
            int64_t len = (int64_t)n->slot.size();
            if (cap >= 0 && (int64_t)out.size() + len > cap) return false;
            out.insert(out.end(), n->slot.begin(), n->slot.end());
            got += len;
            remove_leaf(n);
        }
        return true;
    }

    // RX_OK when every cached token of the prefix of t[0..n) holds a lock.
    int check_unlock(const int64_t *t, int64_t n)
    {
        Walk w = walk(t, n);
        for (size_t i = 0; i < w.nodes.size(); ++i) {
            Node *x = w.nodes[i];
            int64_t m = (i + 1 == w.nodes.size()) ? w.in_last : (int64_t)x->tok.size();
            for (int64_t j = 0; j < m; ++j)
                if (x->lock[j] <= 0)
                    return rx_set_error(RX_ERR_INVALID, "rx_lock_prefix: unlocking a token that is not locked");
        }
        return RX_OK;
    }

    int lock(const int64_t *t, int64_t n, int32_t delta, int64_t *len)
    {
        if (delta < 0) {
            const int rc = check_unlock(t, n);
            if (rc != RX_OK) return rc;
        }
        if (delta > 0) ++clock;
        Walk w = walk(t, n);
        for (size_t i = 0; i < w.nodes.size(); ++i) {
            Node *x = w.nodes[i];
            int64_t m = (i + 1 == w.nodes.size()) ? w.in_last : (int64_t)x->tok.size();
            for (int64_t j = 0; j < m; ++j) {
                int32_t before = x->lock[j];
                x->lock[j] += delta;
                if (before == 0 && x->lock[j] > 0) ++x->nlocked;
                if (before > 0 && x->lock[j] == 0) --x->nlocked;
            }
            if (delta > 0) x->last = clock;
            refresh(x);
        }
        if (len) *len = w.matched;
        return RX_OK;
    }

    int64_t insert(const int64_t *t, const int32_t *s, int64_t n)
    {
        Walk w = walk(t, n);
        const bool grow = w.matched < n;
        const bool cut = grow && !w.nodes.empty() && w.in_last < (int64_t)w.nodes.back()->tok.size();
        // the nodes this insert needs, before anything changes
        std::unique_ptr<Node> lo(cut ? raw_node() : nullptr);
        std::unique_ptr<Node> fresh(grow ? raw_node() : nullptr);
        ++clock;
        Node *attach = &root;
        if (!w.nodes.empty()) {
            attach = w.nodes.back();
            if (cut) split(attach, w.in_last, lo.release());  // diverges strictly inside: split
        }
        tick(w);
        if (grow) {
            Node *leaf = adopt(fresh.release(), attach);
            leaf->tok.assign(t + w.matched, t + n);
            leaf->slot.assign(s + w.matched, s + n);
            leaf->lock.assign((size_t)(n - w.matched), 0);
            leaf->last = clock;
            attach->kids[leaf->tok[0]] = leaf;
            cached += n - w.matched;
            refresh(attach);
            refresh(leaf);
        }
        return w.matched;
    }
};

extern "C" int rx_tree_create(rx_tree **out)
{
    if (!out) return rx_set_error(RX_ERR_INVALID, "rx_tree_create: null out");
    RX_TRY
    count_alloc();
    *out = new rx_tree();
    return RX_OK;
    RX_CATCH
}

extern "C" void rx_tree_destroy(rx_tree *tree) { delete tree; }

extern "C" int rx_match_prefix(rx_tree *tree, const int64_t *tokens, int64_t n, int32_t *out_slots,
                               int64_t out_cap, int64_t *out_prefix_len)
{
    if (!tree || n < 0 || (n > 0 && !tokens) || !out_prefix_len || out_cap < 0 ||
        (out_cap > 0 && !out_slots))
        return rx_set_error(RX_ERR_INVALID, "rx_match_prefix: invalid argument");
    RX_TRY
    ++tree->clock;
    Walk w = tree->walk(tokens, n);
    tree->tick(w);
    *out_prefix_len = w.matched;
    if (w.matched > out_cap)
        return rx_set_error(RX_ERR_CAPACITY, "rx_match_prefix: need %lld slots, capacity %lld",
                            (long long)w.matched, (long long)out_cap);
    int64_t pos = 0;
    for (size_t i = 0; i < w.nodes.size(); ++i) {
        Node *x = w.nodes[i];
        int64_t m = (i + 1 == w.nodes.size()) ? w.in_last : (int64_t)x->tok.size();
        std::memcpy(out_slots + pos, x->slot.data(), sizeof(int32_t) * (size_t)m);
        pos += m;
    }
    return RX_OK;
    RX_CATCH
}

extern "C" int rx_prefix_len(rx_tree *tree, const int64_t *tokens, int64_t n, int64_t *out_len)
{
    if (!tree || n < 0 || (n > 0 && !tokens) || !out_len)
        return rx_set_error(RX_ERR_INVALID, "rx_prefix_len: invalid argument");
    RX_TRY
    *out_len = tree->walk(tokens, n).matched;
    return RX_OK;
    RX_CATCH
}

// Cache-aware scheduling ("SGLang: Evaluación y resultados"): probe every
// waiting request's cached prefix, then order them -- arrival order, or
// longest cached prefix first with ties in arrival order (a stable sort).
extern "C" int rx_schedule(rx_tree *tree, const int64_t *tokens, const int64_t *offsets, int32_t n_req,
                           int32_t policy, int32_t *out_order, int64_t *out_prefix_len)
{
    if (!tree || n_req < 0 || (policy != RX_SCHED_FCFS && policy != RX_SCHED_LPM))
        return rx_set_error(RX_ERR_INVALID, "rx_schedule: invalid argument");
    if (n_req == 0) return RX_OK;
    if (!offsets || !out_order || !out_prefix_len || offsets[0] != 0)
        return rx_set_error(RX_ERR_INVALID, "rx_schedule: invalid argument");
    for (int32_t i = 0; i < n_req; ++i)
        if (offsets[i + 1] < offsets[i])
            return rx_set_error(RX_ERR_INVALID, "rx_schedule: offsets decrease at request %d", i);
    if (offsets[n_req] > 0 && !tokens) return rx_set_error(RX_ERR_INVALID, "rx_schedule: null tokens");
    RX_TRY
    std::vector<int64_t> len((size_t)n_req);
    for (int32_t i = 0; i < n_req; ++i)
        len[(size_t)i] = tree->walk(tokens + offsets[i], offsets[i + 1] - offsets[i]).matched;
    std::vector<int32_t> order((size_t)n_req);
    for (int32_t i = 0; i < n_req; ++i) order[(size_t)i] = i;
    if (policy == RX_SCHED_LPM)
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return len[(size_t)a] > len[(size_t)b]; });
    std::memcpy(out_order, order.data(), sizeof(int32_t) * (size_t)n_req);
    std::memcpy(out_prefix_len, len.data(), sizeof(int64_t) * (size_t)n_req);
    return RX_OK;
    RX_CATCH
}

// Image keys ("SGLang: Evaluación y resultados": an image's hash is its key
// in the radix tree): the FNV-1a 64-bit hash of the bytes (offset basis
// 0xcbf29ce484222325, prime 0x100000001b3) seeds a SplitMix64 generator
// (increment 0x9e3779b97f4a7c15, its published finaliser); output i + 1 with
// the top bit set is the key of image token i.
extern "C" int rx_image_keys(const uint8_t *data, int64_t nbytes, int64_t n_tokens, int64_t *out_keys)
{
    if (nbytes < 0 || n_tokens < 0 || (nbytes > 0 && !data) || (n_tokens > 0 && !out_keys))
        return rx_set_error(RX_ERR_INVALID, "rx_image_keys: invalid argument");
    uint64_t h = 0xcbf29ce484222325ull;
    for (int64_t i = 0; i < nbytes; ++i) {
        h ^= (uint64_t)data[i];
        h *= 0x100000001b3ull;
    }
    uint64_t state = h;
    for (int64_t i = 0; i < n_tokens; ++i) {
        state += 0x9e3779b97f4a7c15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        z ^= z >> 31;
        z |= 0x8000000000000000ull;
        std::memcpy(out_keys + i, &z, sizeof(z));
    }
    return RX_OK;
}

extern "C" int rx_insert(rx_tree *tree, const int64_t *tokens, const int32_t *slots, int64_t n,
                         int64_t *out_already_cached)
{
    if (!tree || n < 0 || (n > 0 && (!tokens || !slots)))
        return rx_set_error(RX_ERR_INVALID, "rx_insert: invalid argument");
    RX_TRY
    int64_t k = tree->insert(tokens, slots, n);
    if (out_already_cached) *out_already_cached = k;
    return RX_OK;
    RX_CATCH
}

extern "C" int rx_evict_lru(rx_tree *tree, int64_t num_tokens, int32_t *out_freed, int64_t out_cap,
                            int64_t *out_num_freed)
{
    if (!tree || num_tokens < 0 || out_cap < 0 || (out_cap > 0 && !out_freed) || !out_num_freed)
        return rx_set_error(RX_ERR_INVALID, "rx_evict_lru: invalid argument");
    RX_TRY
    std::vector<int32_t> got;
    bool fit = tree->evict(num_tokens, got, out_cap);
    if (!got.empty()) std::memcpy(out_freed, got.data(), sizeof(int32_t) * got.size());
    *out_num_freed = (int64_t)got.size();
    if (!fit)
        return rx_set_error(RX_ERR_CAPACITY, "rx_evict_lru: next node does not fit in %lld slots",
                            (long long)out_cap);
    if ((int64_t)got.size() < num_tokens)
        return rx_set_error(RX_ERR_NOT_ENOUGH, "rx_evict_lru: freed %lld of %lld tokens",
                            (long long)got.size(), (long long)num_tokens);
    return RX_OK;
    RX_CATCH
}

extern "C" int rx_lock_prefix(rx_tree *tree, const int64_t *tokens, int64_t n, int32_t delta,
                              int64_t *out_len)
{
    if (!tree || n < 0 || (n > 0 && !tokens) || (delta != 1 && delta != -1))
        return rx_set_error(RX_ERR_INVALID, "rx_lock_prefix: invalid argument");
    RX_TRY
    return tree->lock(tokens, n, delta, out_len);
    RX_CATCH
}

extern "C" int rx_tree_stats(rx_tree *tree, int64_t *cached_tokens, int64_t *num_nodes,
                             int64_t *evictable_tokens)
{
    if (!tree) return rx_set_error(RX_ERR_INVALID, "rx_tree_stats: null tree");
    if (cached_tokens) *cached_tokens = tree->cached;
    if (num_nodes) *num_nodes = tree->n_nodes;
    if (evictable_tokens) {
        int64_t e = 0;
        for (auto &kv : tree->by_id)
            if (kv.second->nlocked == 0) e += (int64_t)kv.second->tok.size();
        *evictable_tokens = e;
    }
    return RX_OK;
}

extern "C" int rx_tree_dump(rx_tree *tree, int64_t *out, int64_t out_cap, int64_t *out_len)
{
    if (!tree || !out_len || out_cap < 0 || (out_cap > 0 && !out))
        return rx_set_error(RX_ERR_INVALID, "rx_tree_dump: invalid argument");
    RX_TRY
    std::vector<int64_t> buf;
    std::vector<Node *> stack;
    auto push_kids = [&](Node *n) {
        std::vector<std::pair<int64_t, Node *>> ks(n->kids.begin(), n->kids.end());
        std::sort(ks.begin(), ks.end(),
                  [](const std::pair<int64_t, Node *> &a, const std::pair<int64_t, Node *> &b) {
                      return a.first > b.first;  // popped in ascending order
                  });
        for (auto &kv : ks) stack.push_back(kv.second);
    };
    push_kids(&tree->root);
    while (!stack.empty()) {
        Node *n = stack.back();
        stack.pop_back();
        buf.push_back(n->id);
        buf.push_back(n->parent == &tree->root ? -1 : n->parent->id);
        buf.push_back(n->last);
        buf.push_back((int64_t)n->tok.size());
        buf.insert(buf.end(), n->tok.begin(), n->tok.end());
        for (int32_t s : n->slot) buf.push_back(s);
        for (int32_t c : n->lock) buf.push_back(c);
        push_kids(n);
    }
    *out_len = (int64_t)buf.size();
    if ((int64_t)buf.size() > out_cap)
        return rx_set_error(RX_ERR_CAPACITY, "rx_tree_dump: need %lld words",
                            (long long)buf.size());
    if (!buf.empty()) std::memcpy(out, buf.data(), sizeof(int64_t) * buf.size());
    return RX_OK;
    RX_CATCH
}

// ---------------------------------------------------------------------------
// slot free list
// ---------------------------------------------------------------------------

struct rx_slot_alloc {
    std::deque<int32_t> q;
    int64_t num_slots = 0;
};

extern "C" int rx_slot_alloc_create(const int32_t *free_order, int64_t n, int64_t num_slots,
                                    rx_slot_alloc **out)
{
    if (!out || n < 0 || (n > 0 && !free_order) || num_slots < 0 || num_slots > INT32_MAX)
        return rx_set_error(RX_ERR_INVALID, "rx_slot_alloc_create: invalid argument");
    RX_TRY
    for (int64_t i = 0; i < n; ++i)
        if (free_order[i] < 0 || free_order[i] >= num_slots)
            return rx_set_error(RX_ERR_INVALID, "rx_slot_alloc_create: slot %d out of range",
                                free_order[i]);
    rx_slot_alloc *a = new rx_slot_alloc();
    a->q.assign(free_order, free_order + n);
    a->num_slots = num_slots;
    *out = a;
    return RX_OK;
    RX_CATCH
}

extern "C" void rx_slot_alloc_destroy(rx_slot_alloc *a) { delete a; }

extern "C" int rx_slot_alloc_take(rx_slot_alloc *a, int64_t n, int32_t *out)
{
    if (!a || n < 0 || (n > 0 && !out))
        return rx_set_error(RX_ERR_INVALID, "rx_slot_alloc_take: invalid argument");
    if ((int64_t)a->q.size() < n)
        return rx_set_error(RX_ERR_NOT_ENOUGH, "rx_slot_alloc_take: %lld free, %lld asked",
                            (long long)a->q.size(), (long long)n);
    for (int64_t i = 0; i < n; ++i) {
        out[i] = a->q.front();
        a->q.pop_front();
    }
    return RX_OK;
}

extern "C" int rx_slot_alloc_give(rx_slot_alloc *a, const int32_t *slots, int64_t n)
{
    if (!a || n < 0 || (n > 0 && !slots))
        return rx_set_error(RX_ERR_INVALID, "rx_slot_alloc_give: invalid argument");
    for (int64_t i = 0; i < n; ++i)
        if (slots[i] < 0 || slots[i] >= a->num_slots)
            return rx_set_error(RX_ERR_INVALID, "rx_slot_alloc_give: slot %d out of range", slots[i]);
    RX_TRY
    a->q.insert(a->q.end(), slots, slots + n);
    return RX_OK;
    RX_CATCH
}

extern "C" int64_t rx_slot_alloc_free_count(const rx_slot_alloc *a)
{
    return a ? (int64_t)a->q.size() : 0;
}

// ---------------------------------------------------------------------------
// request admission
// ---------------------------------------------------------------------------

extern "C" int rx_admit(rx_tree *tree, rx_slot_alloc *alloc, const int64_t *tokens, int64_t n,
                        int32_t *out_row, int64_t *out_prefix_len, int64_t *out_evicted)
{
    if (!tree || !alloc || n < 0 || (n > 0 && (!tokens || !out_row)) || !out_prefix_len)
        return rx_set_error(RX_ERR_INVALID, "rx_admit: invalid argument");
    RX_TRY
    int64_t k = 0;
    int rc = rx_match_prefix(tree, tokens, n, out_row, n, &k);
    if (rc != RX_OK) return rc;
    int64_t locked = 0;
    rc = tree->lock(tokens, k, +1, &locked);
    if (rc != RX_OK) return rc;
    int64_t need = n - k, evicted = 0;
    if ((int64_t)alloc->q.size() < need) {
        std::vector<int32_t> freed;
        tree->evict(need - (int64_t)alloc->q.size(), freed, -1);
        evicted = (int64_t)freed.size();
        alloc->q.insert(alloc->q.end(), freed.begin(), freed.end());
    }
    if (out_evicted) *out_evicted = evicted;
    if ((int64_t)alloc->q.size() < need) {
        tree->lock(tokens, locked, -1, nullptr);
        return rx_set_error(RX_ERR_NOT_ENOUGH, "rx_admit: request needs %lld slots, %lld free",
                            (long long)need, (long long)alloc->q.size());
    }
    for (int64_t i = 0; i < need; ++i) {
        out_row[k + i] = alloc->q.front();
        alloc->q.pop_front();
    }
    *out_prefix_len = k;
    return RX_OK;
    RX_CATCH
}

extern "C" int rx_commit(rx_tree *tree, rx_slot_alloc *alloc, const int64_t *tokens,
                         const int32_t *row, int64_t n, int64_t prefix_len)
{
    if (!tree || !alloc || n < 0 || prefix_len < 0 || prefix_len > n ||
        (n > 0 && (!tokens || !row)))
        return rx_set_error(RX_ERR_INVALID, "rx_commit: invalid argument");
    RX_TRY
    // check the unlock, insert (a failed allocation there changes nothing),
    // then unlock; the order of the insert and the unlock does not change
    // the resulting tree
    int rc = tree->check_unlock(tokens, prefix_len);
    if (rc != RX_OK) return rc;
    int64_t cached = tree->insert(tokens, row, n);
    tree->lock(tokens, prefix_len, -1, nullptr);
    if (cached > prefix_len) alloc->q.insert(alloc->q.end(), row + prefix_len, row + cached);
    return RX_OK;
    RX_CATCH
}

// ---------------------------------------------------------------------------
// decode plan
// ---------------------------------------------------------------------------
//
// Requests whose slot lists agree from position 0 up to some position share
// that prefix's KV.  Sorting the batch by slot list puts requests that share
// a prefix next to each other; the longest common prefixes (LCPs) of
// neighbours then nest exactly like the radix tree the slots came from: every
// LCP interval is a tree node shared by its requests.  Each interval whose own
// span (its LCP minus its parent's) is at least min_shared becomes a shared
// segment; shorter spans are folded into the segments below them.

namespace {

struct Interval {
    int64_t lcp, lb, rb;    // shared prefix length, first and last plan row
    int64_t parent_lcp;     // lcp of the enclosing interval
    int parent = -1;        // index of the enclosing reported interval (-1: root)
};

}  // namespace

extern "C" int rx_decode_plan_build(const int32_t *rtt, int64_t stride, const int32_t *req_idx,
                                    const int32_t *seq_len, int32_t batch, int32_t hq, int32_t hkv,
                                    int32_t kv_chunk, int32_t min_shared, int32_t *out_buf,
                                    int64_t out_cap, rx_decode_plan_info *info)
{
    if (!rtt || !req_idx || !seq_len || !info || batch <= 0 || stride <= 0 || hkv <= 0 ||
        hq <= 0 || hq % hkv != 0 ||
        (kv_chunk != 0 && (kv_chunk < 64 || kv_chunk % 64 != 0 || kv_chunk > RX_MAX_KV_CHUNK)) ||
        min_shared < 1 || out_cap < 0 || (out_cap > 0 && !out_buf))
        return rx_set_error(RX_ERR_INVALID, "rx_decode_plan_build: invalid argument");
    const int64_t G = hq / hkv;
    if (64 % G != 0)
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_decode_plan_build: q heads per kv head (%lld) "
                            "must divide 64", (long long)G);
    for (int32_t b = 0; b < batch; ++b)
        if (seq_len[b] <= 0 || seq_len[b] > stride || req_idx[b] < 0)
            return rx_set_error(RX_ERR_INVALID, "rx_decode_plan_build: bad request %d", b);
    RX_TRY
    const int64_t B = batch;
    auto row = [&](int64_t b) { return rtt + (int64_t)req_idx[b] * stride; };
    std::vector<int32_t> order((size_t)B);
    for (int64_t i = 0; i < B; ++i) order[(size_t)i] = (int32_t)i;
    // Any order in which rows with a common prefix sit next to each other
    // will do; the byte-wise order of the slot lists is one (a common prefix
    // of k slots is a common prefix of 4k bytes), and memcmp finds the first
    // difference of two long shared prefixes quickly.
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        const int64_t la = seq_len[a], lb = seq_len[b];
        const int c = std::memcmp(row(a), row(b), sizeof(int32_t) * (size_t)std::min(la, lb));
        return c < 0 || (c == 0 && la < lb);
    });
    // Common prefix of neighbours, at most one short of the shorter request:
    // a request's last position always stays its own, so that every request
    // ends in a private piece that can follow its length (RX_PLAN_OPEN_END).
    std::vector<int64_t> lcp((size_t)(B > 1 ? B - 1 : 0));
    for (int64_t i = 0; i + 1 < B; ++i) {
        const int32_t *x = row(order[(size_t)i]), *y = row(order[(size_t)i + 1]);
        const int64_t m = std::min(seq_len[order[(size_t)i]], seq_len[order[(size_t)i + 1]]) - 1;
        int64_t k = 0;
        while (k + 16 <= m && std::memcmp(x + k, y + k, 64) == 0) k += 16;
        while (k < m && x[k] == y[k]) ++k;
        lcp[(size_t)i] = k;
    }
    // LCP intervals, children reported before parents
    std::vector<Interval> iv;
    {
        struct Open {
            int64_t lcp, lb;
            std::vector<int> kids;
        };
        std::vector<Open> st;
        st.push_back({0, 0, {}});
        for (int64_t i = 1; i <= B; ++i) {
            int64_t l = (i < B) ? lcp[(size_t)i - 1] : 0;
            int64_t lb = i - 1;
            int last_closed = -1;
            while (l < st.back().lcp) {
                Open o = st.back();
                st.pop_back();
                Interval x{o.lcp, o.lb, i - 1, std::max(l, st.back().lcp), -1};
                int id = (int)iv.size();
                iv.push_back(x);
                for (int c : o.kids) iv[(size_t)c].parent = id;
                lb = o.lb;
                if (l <= st.back().lcp)
                    st.back().kids.push_back(id);
                else
                    last_closed = id;
            }
            if (l > st.back().lcp) {
                st.push_back({l, lb, {}});
                if (last_closed >= 0) st.back().kids.push_back(last_closed);
            }
        }
    }
    // top-down: which intervals become segments, and where each starts
    const int64_t n_iv = (int64_t)iv.size();
    std::vector<int64_t> seg_start((size_t)n_iv), eff_end((size_t)n_iv);
    std::vector<char> is_seg((size_t)n_iv, 0);
    // parents appear after their children, so walk backwards
    for (int64_t k = n_iv - 1; k >= 0; --k) {
        Interval &x = iv[(size_t)k];
        int64_t start = (x.parent >= 0) ? eff_end[(size_t)x.parent] : 0;
        seg_start[(size_t)k] = start;
        if (x.lcp - start >= min_shared) {
            is_seg[(size_t)k] = 1;
            eff_end[(size_t)k] = x.lcp;
        } else {
            eff_end[(size_t)k] = start;
        }
    }
    // deepest segment covering each plan row, and the KV rows the plan reads
    std::vector<int64_t> priv_begin((size_t)B, 0), depth_best((size_t)B, -1);
    std::vector<int64_t> deepest((size_t)B, -1);
    int64_t n_seg = 0, shared = 0, reads = 0;
    for (int64_t k = 0; k < n_iv; ++k) {
        if (!is_seg[(size_t)k]) continue;
        const Interval &x = iv[(size_t)k];
        ++n_seg;
        shared += x.lcp - seg_start[(size_t)k];
        for (int64_t r = x.lb; r <= x.rb; ++r)
            if (x.lcp > depth_best[(size_t)r]) {
                depth_best[(size_t)r] = x.lcp;
                priv_begin[(size_t)r] = x.lcp;
                deepest[(size_t)r] = k;
            }
    }
    reads = shared;
    for (int64_t r = 0; r < B; ++r) reads += seq_len[order[(size_t)r]] - priv_begin[(size_t)r];
    const bool auto_chunk = kv_chunk == 0;
    // With one q head per kv head, or with the head counts the
    // several-q-heads all-heads kernel takes, a request's own positions are
    // read across all kv heads at once (whole contiguous slot rows), as
    // single-request "wide" items; otherwise every item is per kv head.
    const bool wide = G == 1 || rx_gqa_heads(hq, hkv);
    if (auto_chunk) {
        // about RX_DECODE_TARGET_ITEMS work items over all kv heads; with wide
        // items, about RX_DECODE_TARGET_SHARED_ITEMS per-head items over the
        // shared reads only, or RX_DECODE_TARGET_GROUP_CHUNKS (kv head, chunk)
        // pairs when the shared chunks go to the all-heads kernel in groups
        const int64_t n = wide ? shared * hkv : reads * hkv;
        const int64_t target = !wide ? RX_DECODE_TARGET_ITEMS
                               : G > 1 ? RX_DECODE_TARGET_GROUP_CHUNKS : RX_DECODE_TARGET_SHARED_ITEMS;
        int64_t c = (n + target - 1) / target;
        c = std::min<int64_t>(RX_MAX_KV_CHUNK, std::max<int64_t>(64, (c + 63) / 64 * 64));
        kv_chunk = (int32_t)c;
    }
    auto nchunks = [&](int64_t len) { return (len + kv_chunk - 1) / kv_chunk; };
    // With wide items, a request's own (private) positions are cut into
    // near-equal pieces: with automatic chunking, of about priv_total /
    // RX_DECODE_TARGET_WIDE_ITEMS (or _GROUPED) positions (16 ..
    // RX_MAX_KV_CHUNK), else of at most kv_chunk.  Otherwise they are cut
    // into kv_chunk pieces.
    int64_t priv_total = 0;
    for (int64_t r = 0; r < B; ++r) priv_total += seq_len[order[(size_t)r]] - priv_begin[(size_t)r];
    // Request-group items share the all-heads kernel's queue with the
    // private pieces, longest first; with automatic chunking a private range
    // is not cut into pieces shorter than the longest group item, which
    // would only add partial results to merge, not balance.
    const bool groups = G > 1 && rx_gqa_heads(hq, hkv);
    const int64_t RG = 16 / G;
    auto grouped_seg = [&](const Interval &x) {
        return groups && (x.rb - x.lb + 1 + RG - 1) / RG <= RX_DECODE_MAX_GROUPS;
    };
    int64_t group_len = 0;
    bool per_head_segs = false;  // a shared segment goes to the per-head kernel
    for (int64_t k = 0; k < n_iv; ++k) {
        if (!is_seg[(size_t)k]) continue;
        if (grouped_seg(iv[(size_t)k]))
            group_len = std::max<int64_t>(group_len, std::min<int64_t>(kv_chunk, iv[(size_t)k].lcp - seg_start[(size_t)k]));
        else
            per_head_segs = true;
    }
    // fewer, longer private pieces when group items (and nothing else) share
    // the all-heads kernel's queue with them
    const int64_t wide_target = group_len > 0 && !per_head_segs ? RX_DECODE_TARGET_WIDE_ITEMS_GROUPED
                                                                 : RX_DECODE_TARGET_WIDE_ITEMS;
    int64_t pchunk = kv_chunk;
    if (auto_chunk && wide && priv_total > 0)
        pchunk = std::min<int64_t>(RX_MAX_KV_CHUNK, std::max<int64_t>(RX_DECODE_MIN_WIDE_CHUNK,
                                   (priv_total + wide_target - 1) / wide_target));
    auto npriv = [&](int64_t len) {
        int64_t n = (len + pchunk - 1) / pchunk;
        if (auto_chunk && wide && group_len > 0)
            n = std::max<int64_t>((len + RX_MAX_KV_CHUNK - 1) / RX_MAX_KV_CHUNK,
                                  std::min<int64_t>(n, std::max<int64_t>(1, len / group_len)));
        return n;
    };
    // start of private piece c of n over len positions: near-equal pieces for
    // wide items, whole kv_chunk pieces (64-key tiles) for per-head items
    auto piece = [&](int64_t len, int64_t n, int64_t c) {
        return wide ? len * c / n : std::min(len, c * (int64_t)kv_chunk);
    };
    // part bases of segments and per-row private ranges
    std::vector<int64_t> part_base((size_t)n_iv, 0), base_after((size_t)n_iv, 0);
    for (int64_t k = n_iv - 1; k >= 0; --k) {
        Interval &x = iv[(size_t)k];
        int64_t pb = (x.parent >= 0) ? base_after[(size_t)x.parent] : 0;
        part_base[(size_t)k] = pb;
        base_after[(size_t)k] = pb + (is_seg[(size_t)k] ? nchunks(x.lcp - seg_start[(size_t)k]) : 0);
    }
    std::vector<int64_t> priv_base((size_t)B, 0);
    for (int64_t r = 0; r < B; ++r)
        if (deepest[(size_t)r] >= 0) priv_base[(size_t)r] = base_after[(size_t)deepest[(size_t)r]];
    std::vector<int32_t> nparts((size_t)B);
    int64_t max_parts = 0;
    for (int64_t r = 0; r < B; ++r) {
        int64_t L = seq_len[order[(size_t)r]];
        int64_t np = priv_base[(size_t)r] + npriv(L - priv_begin[(size_t)r]);
        nparts[(size_t)order[(size_t)r]] = (int32_t)np;
        max_parts = std::max(max_parts, np);
    }
    // work items; `all` marks the ones for an all-heads kernel
    struct Item {
        int32_t v[8];
        bool all;
    };
    std::vector<Item> items;
    const int64_t R = 64 / G;  // requests per per-head item (64 query rows)
    // groups of up to RG = 16 / G requests (16 query rows per kv head) for
    // the several-q-heads all-heads kernel
    for (int64_t k = 0; k < n_iv; ++k) {
        if (!is_seg[(size_t)k]) continue;
        const Interval &x = iv[(size_t)k];
        const bool grouped = grouped_seg(x);
        const int64_t step = grouped ? RG : R;
        int64_t s0 = seg_start[(size_t)k], s1 = x.lcp;
        for (int64_t c = 0; c * kv_chunk < s1 - s0; ++c) {
            int64_t p0 = s0 + c * kv_chunk, p1 = std::min(s1, p0 + kv_chunk);
            for (int64_t r0 = x.lb; r0 <= x.rb; r0 += step) {
                int64_t nr = std::min(step, x.rb - r0 + 1);
                bool fin = true;
                for (int64_t r = r0; r < r0 + nr; ++r) fin = fin && nparts[(size_t)order[(size_t)r]] == 1;
                const int32_t b0 = order[(size_t)r0];
                items.push_back({{(int32_t)r0, (int32_t)nr, (int32_t)p0, (int32_t)p1,
                                  (int32_t)(part_base[(size_t)k] + c), fin ? 1 : 0, req_idx[b0], b0},
                                 grouped});
            }
        }
    }
    for (int64_t r = 0; r < B; ++r) {
        int64_t L = seq_len[order[(size_t)r]], s0 = priv_begin[(size_t)r];
        const int64_t n = npriv(L - s0);
        for (int64_t c = 0; c < n; ++c) {
            int64_t p0 = s0 + piece(L - s0, n, c), p1 = s0 + piece(L - s0, n, c + 1);
            bool fin = nparts[(size_t)order[(size_t)r]] == 1;
            const int32_t b0 = order[(size_t)r];
            // the request's last piece ends wherever its length is when the
            // plan is used
            if (c + 1 == n) p1 = RX_PLAN_OPEN_END;
            items.push_back({{(int32_t)r, 1, (int32_t)p0, (int32_t)p1,
                              (int32_t)(priv_base[(size_t)r] + c), fin ? 1 : 0, req_idx[b0], b0},
                             wide});
        }
    }
    // per-head items first, then the all-heads items (read across all kv
    // heads at once).  The per-head kernel's CTAs walk their items in a
    // static round-robin: items of several requests before single-request
    // ones, each of those longest first.  The all-heads kernel hands its
    // items out first come first served, so they go longest first whatever
    // their request count (the tail of the grid then holds the short items;
    // equal lengths keep their order, so a shared chunk's request groups stay
    // together and all but the first find it in L2).
    auto item_end = [&](const Item &x) -> int64_t {
        return x.v[3] == RX_PLAN_OPEN_END ? (int64_t)seq_len[x.v[7]] : (int64_t)x.v[3];
    };
    std::stable_sort(items.begin(), items.end(), [&](const Item &a, const Item &b) {
        if (a.all != b.all) return b.all;
        const bool sa = a.v[1] == 1, sb = b.v[1] == 1;
        if (!a.all && sa != sb) return sb;
        int64_t la = item_end(a) - a.v[2], lb = item_end(b) - b.v[2];
        if (la != lb) return la > lb;
        return a.v[1] > b.v[1];
    });
    int64_t n_wide = 0;
    for (const Item &x : items) n_wide += x.all;
    if ((int64_t)items.size() > INT32_MAX / 8)
        return rx_set_error(RX_ERR_UNSUPPORTED, "rx_decode_plan_build: too many items");
    info->kv_chunk = kv_chunk;
    info->n_items = (int32_t)items.size();
    info->max_parts = (int32_t)max_parts;
    info->n_segments = (int32_t)n_seg;
    info->shared_tokens = shared;
    info->tokens_read = reads;
    info->buf_words = 2 * B + 8 * (int64_t)items.size();
    info->n_wide = (int32_t)n_wide;
    if (info->buf_words > out_cap)
        return rx_set_error(RX_ERR_CAPACITY, "rx_decode_plan_build: need %lld words",
                            (long long)info->buf_words);
    for (int64_t r = 0; r < B; ++r) out_buf[r] = order[(size_t)r];
    for (int64_t b = 0; b < B; ++b) out_buf[B + b] = nparts[(size_t)b];
    for (size_t i = 0; i < items.size(); ++i)
        std::memcpy(out_buf + 2 * B + 8 * (int64_t)i, items[i].v, sizeof(items[i].v));
    return RX_OK;
    RX_CATCH
}
