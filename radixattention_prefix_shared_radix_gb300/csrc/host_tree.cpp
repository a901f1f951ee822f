// Host radix tree, slot allocator, batch-table builder and prefix groups.
//
// The tree is a compressed radix tree: a node holds a run of whole pages
// (tokens + page ids), children are keyed by their first page.  This is the
// structure of bhfrc.com/news/45689 §3.1 (find the child starting with the
// next token, then the longest common prefix inside it) and of
// "SGLang：从前端 DSL 到 SRT 服务运行时", section "用基数树实现前缀复用" (a node
// holds a contiguous token run paged by one token or by multi-token pages).
//
// Semantics are defined per PAGE so that the compressed tree behaves exactly
// like a one-page-per-node trie:
//   * a match or insert that ends inside a node splits it, so use stamps
//     (last_access) and reference counts are uniform over each node;
//   * every page carries a creation id; a node's pages have consecutive ids
//     (a run is created by one insert and only ever split or shortened from
//     its end), so the LRU tie-break of a per-page trie -- oldest page first
//     among equal stamps -- is (last_access, id of the node's last page);
//   * eviction removes pages one at a time from the end of the least
//     recently used unreferenced leaf; once a leaf is the minimum it stays
//     the minimum while it shrinks (its key only decreases), so a leaf is
//     drained until enough is freed or it is gone, and its parent may then
//     become a candidate (leaf-first LRU, oripoin.cn section above;
//     "SGLang 深度拆解" (chenxutan.com) §2.3 _evict; reference counts per
//     request as in bhfrc.com §3.2).

#include <algorithm>
#include <cstring>
#include <deque>
#include <memory>
#include <new>
#include <queue>
#include <unordered_map>
#include <vector>

#include "common.h"

namespace {

struct Node {
    int64_t id = 0;
    Node* parent = nullptr;
    std::vector<int32_t> tokens;   // multiple of the page size
    std::vector<int32_t> pages;    // tokens.size() / P page ids
    int64_t first_pid = 0;         // creation id of pages[0]
    int64_t ref = 0;
    int64_t last_access = 0;
    int64_t depth = 0;             // position of tokens[0]
    std::vector<Node*> children;
};

}  // namespace

struct sgl_tree {
    int32_t P = 1;
    int64_t num_pages = 0;
    std::deque<int32_t> free_pages;
    int64_t clock = 0;
    int64_t next_pid = 1;
    int64_t next_handle = 1;
    Node root;
    std::vector<Node*> handles;   // handle -> node (nullptr once removed)
    int64_t tree_tokens = 0;
    int64_t num_nodes = 0;

    ~sgl_tree() {
        std::vector<Node*> stack(root.children.begin(), root.children.end());
        while (!stack.empty()) {
            Node* n = stack.back();
            stack.pop_back();
            for (Node* c : n->children) stack.push_back(c);
            delete n;
        }
    }

    Node* node_of(sgl_node h) {
        if (h == 0) return &root;
        if (h < 0 || h >= (int64_t)handles.size()) return nullptr;
        return handles[h];
    }

    Node* new_node() {
        Node* n = new Node();
        n->id = next_handle++;
        if ((int64_t)handles.size() <= n->id) handles.resize(n->id + 1, nullptr);
        handles[n->id] = n;
        ++num_nodes;
        return n;
    }

    bool first_page_equal(const Node* c, const int32_t* toks) const {
        return std::memcmp(c->tokens.data(), toks, sizeof(int32_t) * P) == 0;
    }

    Node* find_child(Node* n, const int32_t* toks) {
        for (Node* c : n->children)
            if (first_page_equal(c, toks)) return c;
        return nullptr;
    }

    // Split `c` after k tokens (k a positive multiple of P, < its length).
    // The new upper node takes the first k tokens and c's place under the
    // parent; c keeps its handle and becomes the lower part.
    Node* split(Node* c, int64_t k) {
        Node* u = new_node();
        int64_t kp = k / P;
        u->parent = c->parent;
        u->tokens.assign(c->tokens.begin(), c->tokens.begin() + k);
        u->pages.assign(c->pages.begin(), c->pages.begin() + kp);
        u->first_pid = c->first_pid;
        u->ref = c->ref;
        u->last_access = c->last_access;
        u->depth = c->depth;
        for (Node*& slot : c->parent->children)
            if (slot == c) slot = u;
        u->children.push_back(c);
        c->parent = u;
        c->tokens.erase(c->tokens.begin(), c->tokens.begin() + k);
        c->pages.erase(c->pages.begin(), c->pages.begin() + kp);
        c->first_pid += kp;
        c->depth += k;
        return u;
    }

    int64_t common_pages(const Node* c, const int32_t* toks, int64_t avail) const {
        int64_t lim = std::min<int64_t>((int64_t)c->tokens.size(), avail);
        const int32_t* a = c->tokens.data();
        int64_t k = 0;
        // whole blocks of 256 tokens, then of 8 tokens, then token by token:
        // each level only advances over equal ranges, so k ends at the first
        // mismatch (or lim) as a token-by-token walk would
        while (k + 256 <= lim && std::memcmp(a + k, toks + k, 256 * sizeof(int32_t)) == 0) k += 256;
        while (k + 8 <= lim && std::memcmp(a + k, toks + k, 8 * sizeof(int32_t)) == 0) k += 8;
        while (k < lim && a[k] == toks[k]) ++k;
        return k / P * P;
    }

    // Longest whole-page prefix; stamps the matched nodes.
    Node* match(const int32_t* toks, int64_t n, int64_t* matched, std::vector<int32_t>* slots) {
        ++clock;
        int64_t n_full = n / P * P, pos = 0;
        Node* node = &root;
        while (pos < n_full) {
            Node* c = find_child(node, toks + pos);
            if (!c) break;
            int64_t k = common_pages(c, toks + pos, n_full - pos);
            if (k <= 0) break;
            bool partial = k < (int64_t)c->tokens.size();
            if (partial) c = split(c, k);
            c->last_access = clock;
            if (slots) {
                if (P == 1) {
                    slots->insert(slots->end(), c->pages.begin(), c->pages.end());
                } else {
                    for (int32_t pg : c->pages)
                        for (int32_t o = 0; o < P; ++o) slots->push_back(pg * P + o);
                }
            }
            pos += k;
            node = c;
            if (partial) break;
        }
        *matched = pos;
        return node;
    }

    // Insert full pages; duplicates go back to the free list.
    Node* insert(const int32_t* toks, const int32_t* pages_in, int64_t n_full, int64_t* dup) {
        return insert_from(&root, toks, pages_in, n_full, dup);
    }
    // The same, resuming at `start`, a node whose path from the root holds
    // exactly the first start->depth + |start->tokens| tokens with the
    // caller's own pages (a locked node just returned by match for these
    // tokens): the walk over that path would find the same nodes, split
    // none of them and find no duplicate page, so only its stamps are
    // applied.  pages_in holds the pages from that node's end on.
    Node* insert_from(Node* start, const int32_t* toks, const int32_t* pages_in, int64_t n_full, int64_t* dup) {
        ++clock;
        *dup = 0;
        for (Node* x = start; x != &root; x = x->parent) x->last_access = clock;
        const int64_t pos0 = start == &root ? 0 : start->depth + (int64_t)start->tokens.size();
        const int64_t pg0 = pos0 / P;   // page index of pages_in[0]
        int64_t pos = pos0;
        Node* node = start;
        while (pos < n_full) {
            Node* c = find_child(node, toks + pos);
            if (!c) {
                Node* m = new_node();
                m->parent = node;
                m->tokens.assign(toks + pos, toks + n_full);
                m->pages.assign(pages_in + (pos / P - pg0), pages_in + (n_full / P - pg0));
                m->first_pid = next_pid;
                next_pid += (n_full - pos) / P;
                m->last_access = clock;
                m->depth = pos;
                node->children.push_back(m);
                tree_tokens += n_full - pos;
                node = m;
                pos = n_full;
                break;
            }
            int64_t k = common_pages(c, toks + pos, n_full - pos);
            if (k < (int64_t)c->tokens.size()) c = split(c, k);
            for (int64_t i = 0; i < k / P; ++i) {
                int32_t mine = pages_in[pos / P - pg0 + i];
                if (c->pages[i] != mine) {
                    *dup += P;
                    free_pages.push_back(mine);
                }
            }
            c->last_access = clock;
            pos += k;
            node = c;
        }
        return node;
    }

    void lock(Node* n) {
        for (; n != &root; n = n->parent) ++n->ref;
    }

    bool unlock(Node* n) {
        for (Node* x = n; x != &root; x = x->parent)
            if (x->ref <= 0) return false;
        for (; n != &root; n = n->parent) --n->ref;
        return true;
    }

    void remove_leaf(Node* v) {
        Node* p = v->parent;
        p->children.erase(std::find(p->children.begin(), p->children.end(), v));
        handles[v->id] = nullptr;
        --num_nodes;
        delete v;
    }

    int64_t evict(int64_t want) {
        using Key = std::pair<std::pair<int64_t, int64_t>, Node*>;
        auto key = [](Node* v) {
            return std::make_pair(v->last_access, v->first_pid + (int64_t)v->pages.size() - 1);
        };
        std::priority_queue<Key, std::vector<Key>, std::greater<Key>> heap;
        std::vector<Node*> stack = root.children;
        while (!stack.empty()) {
            Node* n = stack.back();
            stack.pop_back();
            if (n->children.empty()) {
                if (n->ref == 0) heap.push({key(n), n});
            } else {
                for (Node* c : n->children) stack.push_back(c);
            }
        }
        int64_t freed = 0;
        while (freed < want && !heap.empty()) {
            Node* v = heap.top().second;
            heap.pop();
            while (!v->pages.empty() && freed < want) {
                free_pages.push_back(v->pages.back());
                v->pages.pop_back();
                v->tokens.resize(v->tokens.size() - P);
                freed += P;
                tree_tokens -= P;
            }
            if (v->pages.empty()) {
                Node* p = v->parent;
                remove_leaf(v);
                if (p != &root && p->children.empty() && p->ref == 0) heap.push({key(p), p});
            }
        }
        return freed;
    }

    bool alloc(int64_t n, std::vector<int32_t>* out) {
        int64_t need = (n + P - 1) / P;
        if ((int64_t)free_pages.size() < need) evict((need - (int64_t)free_pages.size()) * P);
        if ((int64_t)free_pages.size() < need) return false;
        for (int64_t i = 0; i < need; ++i) {
            int32_t pg = free_pages.front();
            free_pages.pop_front();
            for (int32_t o = 0; o < P && (int64_t)out->size() < n + 0; ++o) out->push_back(pg * P + o);
        }
        out->resize(n);
        return true;
    }

    bool free_slots(const int32_t* slots, int64_t n) {
        std::vector<int32_t> seen;
        for (int64_t i = 0; i < n; ++i) {
            if (slots[i] < 0 || slots[i] / P >= num_pages) return false;
        }
        for (int64_t i = 0; i < n; ++i) {
            int32_t pg = slots[i] / P;
            if (std::find(seen.begin(), seen.end(), pg) == seen.end()) seen.push_back(pg);
        }
        for (int32_t pg : seen) free_pages.push_back(pg);
        return true;
    }

    // Page ids of slots[0..n_full); false if a page's slots are not that
    // page's consecutive slots or out of range.
    bool pages_of(const int32_t* slots, int64_t n_full, std::vector<int32_t>* pages) const {
        pages->clear();
        if (P == 1) {   // a slot is its page: range checks, then one copy
            for (int64_t i = 0; i < n_full; ++i)
                if (slots[i] < 0 || slots[i] >= num_pages) return false;
            pages->assign(slots, slots + n_full);
            return true;
        }
        for (int64_t i = 0; i < n_full; i += P) {
            int32_t s = slots[i];
            if (s < 0 || s % P) return false;
            int32_t pg = s / P;
            if (pg >= num_pages) return false;
            for (int32_t o = 1; o < P; ++o)
                if (slots[i + o] != s + o) return false;
            pages->push_back(pg);
        }
        return true;
    }
};

struct sgl_groups {
    std::vector<int32_t> seg_begin, seg_end, seg_row, seg_member_ptr, seg_members;
    void clear() {
        seg_begin.clear();
        seg_end.clear();
        seg_row.clear();
        seg_member_ptr.assign(1, 0);
        seg_members.clear();
    }
};

namespace {

struct Seg {
    int32_t rep, begin, end;
    const std::vector<int32_t>* members;
};

void emit(sgl_groups* g, std::vector<Seg>& segs) {
    std::sort(segs.begin(), segs.end(), [](const Seg& a, const Seg& b) {
        return a.rep != b.rep ? a.rep < b.rep : a.begin < b.begin;
    });
    g->clear();
    for (const Seg& s : segs) {
        g->seg_begin.push_back(s.begin);
        g->seg_end.push_back(s.end);
        g->seg_row.push_back(s.rep);
        g->seg_members.insert(g->seg_members.end(), s.members->begin(), s.members->end());
        g->seg_member_ptr.push_back((int32_t)g->seg_members.size());
    }
}

}  // namespace

extern "C" {

int sgl_tree_create(int64_t num_slots, int32_t page_size, const int32_t* free_order, sgl_tree** out) {
    if (!out || page_size < 1 || num_slots < 0 || num_slots % page_size) return SGL_ERR_INVALID_ARG;
    if (num_slots / page_size > INT32_MAX || num_slots > INT32_MAX) return SGL_ERR_INVALID_ARG;
    sgl_tree* t = new (std::nothrow) sgl_tree();
    if (!t) return SGL_ERR_INVALID_ARG;
    t->P = page_size;
    t->num_pages = num_slots / page_size;
    if (free_order) {
        std::vector<char> seen(t->num_pages, 0);
        for (int64_t i = 0; i < t->num_pages; ++i) {
            int32_t p = free_order[i];
            if (p < 0 || p >= t->num_pages || seen[p]) {
                delete t;
                return SGL_ERR_INVALID_ARG;
            }
            seen[p] = 1;
            t->free_pages.push_back(p);
        }
    } else {
        for (int64_t i = 0; i < t->num_pages; ++i) t->free_pages.push_back((int32_t)i);
    }
    *out = t;
    return SGL_OK;
}

void sgl_tree_destroy(sgl_tree* tree) { delete tree; }

int sgl_tree_match(sgl_tree* t, const int32_t* tokens, int64_t n, int64_t* matched_len, int32_t* slots_out,
                   sgl_node* last) {
    if (!t || n < 0 || (n > 0 && !tokens) || !matched_len) return SGL_ERR_INVALID_ARG;
    std::vector<int32_t> slots;
    Node* node = t->match(tokens, n, matched_len, slots_out ? &slots : nullptr);
    if (slots_out && !slots.empty()) std::memcpy(slots_out, slots.data(), slots.size() * sizeof(int32_t));
    if (last) *last = node->id;
    return SGL_OK;
}

int sgl_tree_insert(sgl_tree* t, const int32_t* tokens, const int32_t* slots, int64_t n, int64_t* dup_len,
                    sgl_node* last) {
    if (!t || n < 0 || (n > 0 && (!tokens || !slots))) return SGL_ERR_INVALID_ARG;
    int64_t n_full = n / t->P * t->P;
    std::vector<int32_t> pages;
    if (!t->pages_of(slots, n_full, &pages)) return SGL_ERR_INVALID_ARG;
    int64_t dup = 0;
    Node* node = t->insert(tokens, pages.data(), n_full, &dup);
    if (dup_len) *dup_len = dup;
    if (last) *last = node->id;
    return SGL_OK;
}

int sgl_tree_lock(sgl_tree* t, sgl_node h) {
    if (!t) return SGL_ERR_INVALID_ARG;
    Node* n = t->node_of(h);
    if (!n) return SGL_ERR_STATE;
    t->lock(n);
    return SGL_OK;
}

int sgl_tree_unlock(sgl_tree* t, sgl_node h) {
    if (!t) return SGL_ERR_INVALID_ARG;
    Node* n = t->node_of(h);
    if (!n) return SGL_ERR_STATE;
    return t->unlock(n) ? SGL_OK : SGL_ERR_STATE;
}

int sgl_tree_alloc(sgl_tree* t, int64_t n, int32_t* slots_out) {
    if (!t || n < 0 || (n > 0 && !slots_out)) return SGL_ERR_INVALID_ARG;
    std::vector<int32_t> out;
    if (!t->alloc(n, &out)) return SGL_ERR_NO_SLOTS;
    if (n) std::memcpy(slots_out, out.data(), n * sizeof(int32_t));
    return SGL_OK;
}

int sgl_tree_free(sgl_tree* t, const int32_t* slots, int64_t n) {
    if (!t || n < 0 || (n > 0 && !slots)) return SGL_ERR_INVALID_ARG;
    return t->free_slots(slots, n) ? SGL_OK : SGL_ERR_INVALID_ARG;
}

int sgl_tree_evict(sgl_tree* t, int64_t num_tokens, int64_t* freed) {
    if (!t || num_tokens < 0) return SGL_ERR_INVALID_ARG;
    int64_t f = t->evict(num_tokens);
    if (freed) *freed = f;
    return SGL_OK;
}

int sgl_tree_stats(const sgl_tree* t, sgl_tree_stats_t* out) {
    if (!t || !out) return SGL_ERR_INVALID_ARG;
    out->free_pages = (int64_t)t->free_pages.size();
    out->tree_tokens = t->tree_tokens;
    out->num_nodes = t->num_nodes;
    out->clock = t->clock;
    int64_t locked = 0, evictable = 0;
    std::vector<const Node*> stack(t->root.children.begin(), t->root.children.end());
    while (!stack.empty()) {
        const Node* n = stack.back();
        stack.pop_back();
        (n->ref > 0 ? locked : evictable) += (int64_t)n->tokens.size();
        for (const Node* c : n->children) stack.push_back(c);
    }
    out->locked_tokens = locked;
    out->evictable_tokens = evictable;
    return SGL_OK;
}

int sgl_groups_create(sgl_groups** out) {
    if (!out) return SGL_ERR_INVALID_ARG;
    *out = new (std::nothrow) sgl_groups();
    if (!*out) return SGL_ERR_INVALID_ARG;
    (*out)->clear();
    return SGL_OK;
}

void sgl_groups_destroy(sgl_groups* g) { delete g; }

int sgl_groups_view(const sgl_groups* g, sgl_prefix_groups* v) {
    if (!g || !v) return SGL_ERR_INVALID_ARG;
    v->num_segments = (int32_t)g->seg_begin.size();
    v->num_members = (int32_t)g->seg_members.size();
    v->seg_begin = g->seg_begin.data();
    v->seg_end = g->seg_end.data();
    v->seg_row = g->seg_row.data();
    v->seg_member_ptr = g->seg_member_ptr.data();
    v->seg_members = g->seg_members.data();
    return SGL_OK;
}

int sgl_build_batch(sgl_tree* t, int32_t B, const int32_t* const* tokens, const int64_t* len, int32_t* req_to_token,
                    int64_t ld, int32_t* seq_lens, int32_t* prefix_lens, sgl_node* last_nodes,
                    sgl_groups* groups_out) {
    if (!t || B < 0 || (B > 0 && (!tokens || !len || !req_to_token || !seq_lens))) return SGL_ERR_INVALID_ARG;
    for (int32_t r = 0; r < B; ++r) {
        if (len[r] < 0 || len[r] > ld || len[r] > INT32_MAX || (len[r] > 0 && !tokens[r]))
            return SGL_ERR_INVALID_ARG;
    }
    const int32_t P = t->P;
    std::vector<Node*> lasts(B, nullptr);
    std::vector<int64_t> n_full(B, 0);
    std::vector<int32_t> row, pages;
    for (int32_t r = 0; r < B; ++r) {
        const int64_t L = len[r];
        int64_t m = 0;
        row.clear();
        Node* mnode = t->match(tokens[r], L, &m, &row);
        t->lock(mnode);
        std::vector<int32_t> fresh;
        if (!t->alloc(L - m, &fresh)) {
            t->unlock(mnode);
            for (int32_t q = 0; q < r; ++q) {
                t->unlock(lasts[q]);
                int64_t nf = n_full[q];
                t->free_slots(req_to_token + (int64_t)q * ld + nf, len[q] - nf);
            }
            return SGL_ERR_NO_SLOTS;
        }
        row.insert(row.end(), fresh.begin(), fresh.end());
        n_full[r] = L / P * P;
        // pages of the unmatched full pages only (the matched ones are the tree's)
        t->pages_of(row.data() + m, n_full[r] - m, &pages);
        int64_t dup = 0;
        // mnode is locked and its path holds tokens[0, m) with the slots just
        // taken from it
        Node* last = t->insert_from(mnode, tokens[r], pages.data(), n_full[r], &dup);
        t->lock(last);
        t->unlock(mnode);
        lasts[r] = last;
        int32_t* out = req_to_token + (int64_t)r * ld;
        if (L) std::memcpy(out, row.data(), L * sizeof(int32_t));
        for (int64_t j = L; j < ld; ++j) out[j] = -1;
        seq_lens[r] = (int32_t)L;
        if (prefix_lens) prefix_lens[r] = (int32_t)m;
        if (last_nodes) last_nodes[r] = last->id;
    }
    if (!groups_out) return SGL_OK;

    // Prefix groups from the tree: members of every node on the batch's
    // paths, then each request's path cut where the member count changes;
    // a private tail page is its own member set {r}.
    std::unordered_map<Node*, std::vector<int32_t>> members;
    std::vector<std::vector<Node*>> paths(B);
    for (int32_t r = 0; r < B; ++r) {
        for (Node* n = lasts[r]; n != &t->root; n = n->parent) paths[r].push_back(n);
        std::reverse(paths[r].begin(), paths[r].end());
        for (Node* n : paths[r]) members[n].push_back(r);
    }
    std::vector<std::vector<int32_t>> singles(B);
    std::vector<Seg> segs;
    for (int32_t r = 0; r < B; ++r) {
        singles[r].assign(1, r);
        const std::vector<int32_t>* cur = nullptr;
        int32_t begin = 0, end = 0;
        for (Node* n : paths[r]) {
            const std::vector<int32_t>* mem = &members[n];
            int32_t nb = (int32_t)n->depth, ne = (int32_t)(n->depth + n->tokens.size());
            if (cur && mem->size() == cur->size()) {
                end = ne;
                continue;
            }
            if (cur && (*cur)[0] == r) segs.push_back({r, begin, end, cur});
            cur = mem;
            begin = nb;
            end = ne;
        }
        if (len[r] > n_full[r]) {
            if (cur && cur->size() == 1) {
                end = (int32_t)len[r];
            } else {
                if (cur && (*cur)[0] == r) segs.push_back({r, begin, end, cur});
                cur = &singles[r];
                begin = (int32_t)n_full[r];
                end = (int32_t)len[r];
            }
        }
        if (cur && (*cur)[0] == r) segs.push_back({r, begin, end, cur});
    }
    emit(groups_out, segs);
    return SGL_OK;
}

int sgl_tree_finish(sgl_tree* t, sgl_node last, const int32_t* row, int64_t len) {
    if (!t || len < 0 || (len > 0 && !row)) return SGL_ERR_INVALID_ARG;
    Node* n = t->node_of(last);
    if (!n) return SGL_ERR_STATE;
    if (!t->unlock(n)) return SGL_ERR_STATE;
    int64_t nf = len / t->P * t->P;
    if (len > nf && !t->free_slots(row + nf, len - nf)) return SGL_ERR_INVALID_ARG;
    return SGL_OK;
}

int sgl_tree_finish_batch(sgl_tree* t, int32_t B, const sgl_node* last, const int32_t* req_to_token, int64_t ld,
                          const int32_t* seq_lens) {
    if (!t || B < 0 || ld < 0 || (B > 0 && (!last || !req_to_token || !seq_lens))) return SGL_ERR_INVALID_ARG;
    for (int32_t r = 0; r < B; ++r) {
        if (seq_lens[r] < 0 || seq_lens[r] > ld) return SGL_ERR_INVALID_ARG;
        const int st = sgl_tree_finish(t, last[r], req_to_token + (int64_t)r * ld, seq_lens[r]);
        if (st) return st;
    }
    return SGL_OK;
}

// One decode step of a running batch.  The new tokens stay out of the tree
// until their request ends (the CPU scheduler of "SGLang 深度拆解" §1.3
// caches a sequence when its request finishes; the CS349D notes §3.1 insert
// the prompt at prefill completion): each row gets one slot, from a fresh page
// when its length is a multiple of the page size, else the next slot of its
// private tail page.  The fresh pages of the step are allocated in one call
// and handed out in request order.
int sgl_batch_append(sgl_tree* t, int32_t B, int32_t* req_to_token, int64_t ld, int32_t* seq_lens,
                     sgl_groups* g) {
    if (!t || B < 0 || ld < 1 || (B > 0 && (!req_to_token || !seq_lens))) return SGL_ERR_INVALID_ARG;
    const int32_t P = t->P;
    const int64_t S = t->num_pages * P;
    int64_t need = 0;
    for (int32_t r = 0; r < B; ++r) {
        const int64_t L = seq_lens[r];
        if (L < 0 || L >= ld) return SGL_ERR_INVALID_ARG;
        if (L % P == 0) {
            ++need;
        } else {
            const int32_t prev = req_to_token[(int64_t)r * ld + L - 1];
            if (prev < 0 || prev + 1 >= S || (prev + 1) % P == 0) return SGL_ERR_INVALID_ARG;
        }
    }
    // each request's last segment: the one of its segments that ends at its length
    std::vector<int32_t> last_seg;
    if (g) {
        last_seg.assign(B, -1);
        const int32_t ns = (int32_t)g->seg_begin.size();
        for (int32_t s = 0; s < ns; ++s) {
            for (int32_t k = g->seg_member_ptr[s]; k < g->seg_member_ptr[s + 1]; ++k) {
                const int32_t m = g->seg_members[k];
                if (m < 0 || m >= B) return SGL_ERR_INVALID_ARG;
                if (g->seg_end[s] == seq_lens[m]) last_seg[m] = s;
            }
        }
        for (int32_t r = 0; r < B; ++r)
            if (seq_lens[r] > 0 && last_seg[r] < 0) return SGL_ERR_INVALID_ARG;
    }
    std::vector<int32_t> fresh;
    if (!t->alloc(need * P, &fresh)) return SGL_ERR_NO_SLOTS;
    int64_t k = 0;
    bool new_segs = false;
    for (int32_t r = 0; r < B; ++r) {
        int32_t* row = req_to_token + (int64_t)r * ld;
        const int32_t L = seq_lens[r];
        row[L] = L % P == 0 ? fresh[(k++) * P] : row[L - 1] + 1;
        seq_lens[r] = L + 1;
        if (g) {
            const int32_t s = last_seg[r];
            if (s >= 0 && g->seg_member_ptr[s + 1] - g->seg_member_ptr[s] == 1) {
                g->seg_end[s] = L + 1;   // a private trailing segment grows
                last_seg[r] = -2;
            } else {
                new_segs = true;
            }
        }
    }
    if (new_segs) {
        // requests whose context ended in a shared segment (or was empty) get
        // a private one-token segment; the order stays (seg_row, seg_begin)
        struct Row {
            int32_t rep, begin, end, m0, m1;
        };
        std::vector<Row> rows;
        const int32_t ns = (int32_t)g->seg_begin.size();
        for (int32_t s = 0; s < ns; ++s)
            rows.push_back({g->seg_row[s], g->seg_begin[s], g->seg_end[s], g->seg_member_ptr[s],
                            g->seg_member_ptr[s + 1]});
        std::vector<int32_t> solo;
        for (int32_t r = 0; r < B; ++r)
            if (last_seg[r] != -2) solo.push_back(r);
        for (int32_t r : solo) rows.push_back({r, seq_lens[r] - 1, seq_lens[r], -1 - r, 0});
        std::stable_sort(rows.begin(), rows.end(), [](const Row& a, const Row& b) {
            return a.rep != b.rep ? a.rep < b.rep : a.begin < b.begin;
        });
        sgl_groups n;
        n.clear();
        for (const Row& x : rows) {
            n.seg_begin.push_back(x.begin);
            n.seg_end.push_back(x.end);
            n.seg_row.push_back(x.rep);
            if (x.m0 < 0) {
                n.seg_members.push_back(-1 - x.m0);
            } else {
                n.seg_members.insert(n.seg_members.end(), g->seg_members.begin() + x.m0,
                                     g->seg_members.begin() + x.m1);
            }
            n.seg_member_ptr.push_back((int32_t)n.seg_members.size());
        }
        *g = std::move(n);
    }
    return SGL_OK;
}

// A request ends: its whole sequence goes into the tree ("SGLang 深度拆解"
// §1.3, completed sequences are cached), resuming at the node it holds, then
// its reference is released and a partial tail page freed.
int sgl_tree_cache_finished(sgl_tree* t, sgl_node last, const int32_t* tokens, const int32_t* row, int64_t len,
                            int64_t* dup_len) {
    if (!t || len < 0 || (len > 0 && (!tokens || !row))) return SGL_ERR_INVALID_ARG;
    Node* n = t->node_of(last);
    if (!n) return SGL_ERR_STATE;
    for (Node* x = n; x != &t->root; x = x->parent)
        if (x->ref <= 0) return SGL_ERR_STATE;
    const int32_t P = t->P;
    const int64_t end = n == &t->root ? 0 : n->depth + (int64_t)n->tokens.size();
    if (end > len) return SGL_ERR_INVALID_ARG;
    // the held path must be this sequence's own prefix, with its slots
    for (Node* x = n; x != &t->root; x = x->parent) {
        const int64_t d = x->depth, m = (int64_t)x->tokens.size();
        if (std::memcmp(x->tokens.data(), tokens + d, m * sizeof(int32_t)) != 0) return SGL_ERR_INVALID_ARG;
        for (int64_t i = 0; i < m / P; ++i)
            if (row[d + i * P] != x->pages[i] * P) return SGL_ERR_INVALID_ARG;
    }
    const int64_t n_full = len / P * P;
    std::vector<int32_t> pages;
    if (!t->pages_of(row + end, n_full - end, &pages)) return SGL_ERR_INVALID_ARG;
    if (len > n_full) {
        for (int64_t i = n_full; i < len; ++i)
            if (row[i] < 0 || row[i] / P >= t->num_pages) return SGL_ERR_INVALID_ARG;
    }
    int64_t dup = 0;
    t->insert_from(n, tokens, pages.data(), n_full, &dup);
    t->unlock(n);
    if (len > n_full) t->free_slots(row + n_full, len - n_full);
    if (dup_len) *dup_len = dup;
    return SGL_OK;
}

int sgl_tree_cache_finished_batch(sgl_tree* t, int32_t B, const int32_t* const* tokens, const sgl_node* last,
                                  const int32_t* req_to_token, int64_t ld, const int32_t* seq_lens) {
    if (!t || B < 0 || ld < 0 || (B > 0 && (!tokens || !last || !req_to_token || !seq_lens)))
        return SGL_ERR_INVALID_ARG;
    for (int32_t r = 0; r < B; ++r) {
        if (seq_lens[r] < 0 || seq_lens[r] > ld) return SGL_ERR_INVALID_ARG;
        const int st = sgl_tree_cache_finished(t, last[r], tokens[r], req_to_token + (int64_t)r * ld, seq_lens[r],
                                               nullptr);
        if (st) return st;
    }
    return SGL_OK;
}

int sgl_groups_from_table(const int32_t* table, int64_t ld, const int32_t* seq_lens, int32_t B,
                          sgl_groups* g) {
    if (!g || B < 0 || (B > 0 && (!table || !seq_lens))) return SGL_ERR_INVALID_ARG;
    for (int32_t r = 0; r < B; ++r)
        if (seq_lens[r] < 0 || seq_lens[r] > ld) return SGL_ERR_INVALID_ARG;
    // Trie over slot sequences: (parent node, slot) -> node; count rows per node.
    std::unordered_map<uint64_t, int32_t> child;
    std::vector<int32_t> count(1, 0);
    std::vector<std::vector<int32_t>> path(B);
    for (int32_t r = 0; r < B; ++r) {
        int32_t cur = 0;
        const int32_t* row = table + (int64_t)r * ld;
        path[r].reserve(seq_lens[r]);
        for (int32_t j = 0; j < seq_lens[r]; ++j) {
            uint64_t key = ((uint64_t)(uint32_t)cur << 32) | (uint32_t)row[j];
            auto it = child.find(key);
            int32_t nx;
            if (it == child.end()) {
                nx = (int32_t)count.size();
                count.push_back(0);
                child.emplace(key, nx);
            } else {
                nx = it->second;
            }
            ++count[nx];
            path[r].push_back(nx);
            cur = nx;
        }
    }
    // A segment starts where the member count changes along a row's path.
    std::unordered_map<int32_t, std::vector<int32_t>> start_members;
    std::vector<std::vector<std::pair<int32_t, int32_t>>> starts(B);  // (position, node)
    for (int32_t r = 0; r < B; ++r) {
        for (int32_t j = 0; j < seq_lens[r]; ++j) {
            int32_t v = path[r][j];
            if (j == 0 || count[v] != count[path[r][j - 1]]) {
                starts[r].push_back({j, v});
                start_members[v].push_back(r);
            }
        }
    }
    std::vector<Seg> segs;
    for (int32_t r = 0; r < B; ++r) {
        for (size_t k = 0; k < starts[r].size(); ++k) {
            int32_t v = starts[r][k].second;
            const std::vector<int32_t>* mem = &start_members[v];
            if ((*mem)[0] != r) continue;
            int32_t b = starts[r][k].first;
            int32_t e = k + 1 < starts[r].size() ? starts[r][k + 1].first : seq_lens[r];
            segs.push_back({r, b, e, mem});
        }
    }
    emit(g, segs);
    return SGL_OK;
}

}  // extern "C"
