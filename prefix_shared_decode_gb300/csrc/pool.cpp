// Prefix-aware KV cache: a trie of fixed-size chunks over a refcounted slot
// allocator ("ChunkAttention: Efficient Self-Attention with Prefix-Aware KV
// Cache and Two-Phase Partition", §3.1; explainer blog, "Prefix-Aware KV
// Cache" and "動的プレフィックス検出").
//
// Rules (the pages state the idea; these are its plainest exact form):
//  * a sequence's tokens are cut into chunks of c tokens plus a trailing
//    partial chunk;
//  * full chunks are matched child by child from the root by their exact
//    c-token tuple, so a chunk is shared only when its whole path matches; a
//    partial chunk is always a new private leaf;
//  * a matched chunk gains a reference; new chunks take the lowest free slot
//    (min-heap); a removed sequence drops one reference along its path and
//    chunks left with none give their slot back at once;
//  * children keep insertion order (the schedule walks them in that order).
#include <algorithm>
#include <functional>
#include <memory>
#include <new>

#include "ca_internal.h"

namespace ca {
namespace {

// 64-bit hash of a chunk's token tuple: four independent multiply-xorshift
// lanes over token pairs (short dependency chains), folded at the end.
uint64_t chunk_hash(const int32_t* tokens, int32_t c) {
    const uint64_t K = 0x9e3779b97f4a7c15ull;
    uint64_t h[4] = {0x6a09e667f3bcc909ull ^ (uint64_t)c, 0xbb67ae8584caa73bull,
                     0x3c6ef372fe94f82bull, 0xa54ff53a5f1d36f1ull};
    int32_t i = 0;
    for (; i + 8 <= c; i += 8) {
        for (int l = 0; l < 4; ++l) {
            const uint64_t w = (uint64_t)(uint32_t)tokens[i + 2 * l] |
                               ((uint64_t)(uint32_t)tokens[i + 2 * l + 1] << 32);
            h[l] = (h[l] ^ w) * K;
            h[l] ^= h[l] >> 29;
        }
    }
    for (; i < c; ++i) {
        h[0] = (h[0] ^ (uint64_t)(uint32_t)tokens[i]) * K;
        h[0] ^= h[0] >> 29;
    }
    uint64_t r = h[0];
    for (int l = 1; l < 4; ++l) {
        r = (r ^ h[l]) * K;
        r ^= r >> 31;
    }
    return r;
}

constexpr size_t kIndexAbove = 32;   // children before a node gets a hash index

}  // namespace

// A point where an insert or append may allocate host memory.  A test can
// make the n-th point from now fail (ca_pool_inject_alloc_failure) to check
// that the call then leaves the pool unchanged.
void alloc_point(const Pool& p) {
    if (p.fail_alloc_in < 0) return;
    if (p.fail_alloc_in-- == 0) throw std::bad_alloc();
}

namespace {

const int32_t* chunk_tokens(const Pool& p, const Node* n) {
    return p.tokens.data() + (size_t)n->slot * p.cfg.chunk;
}

Node* find_child(const Pool& p, const Node* node, const int32_t* tokens, int32_t c, uint64_t h) {
    if (node->index) {
        auto it = node->index->find(h);
        if (it == node->index->end()) return nullptr;
        Node* ch = it->second;
        return std::equal(tokens, tokens + c, chunk_tokens(p, ch)) ? ch : nullptr;
    }
    for (Node* ch : node->children)
        if (ch->matchable && ch->hash == h && std::equal(tokens, tokens + c, chunk_tokens(p, ch)))
            return ch;
    return nullptr;
}

void add_child(Node* node, Node* ch) {
    node->children.push_back(ch);
    if (node->index) {
        if (ch->matchable) node->index->emplace(ch->hash, ch);
    } else if (node->children.size() > kIndexAbove) {
        // built aside and installed whole, so a failed allocation leaves no
        // partial index behind (the linear scan stays right without one)
        auto idx = std::make_unique<std::unordered_map<uint64_t, Node*>>();
        for (Node* x : node->children)
            if (x->matchable) idx->emplace(x->hash, x);
        node->index = std::move(idx);
    }
}

void drop_child(Node* node, Node* ch) {
    auto& v = node->children;
    auto pos = std::find(v.begin(), v.end(), ch);
    if (pos != v.end()) v.erase(pos);       // absent only while undoing a failed add_child
    if (node->index && ch->matchable) {
        auto it = node->index->find(ch->hash);
        if (it != node->index->end() && it->second == ch) node->index->erase(it);
    }
}

int32_t heap_pop(std::vector<int32_t>& h) {
    std::pop_heap(h.begin(), h.end(), std::greater<int32_t>());
    const int32_t s = h.back();
    h.pop_back();
    return s;
}

void heap_push(std::vector<int32_t>& h, int32_t s) {
    h.push_back(s);
    std::push_heap(h.begin(), h.end(), std::greater<int32_t>());
}

// Walk the matched full-chunk prefix; returns the matched nodes.
void walk_matched(const Pool& p, const int32_t* tokens, int32_t n, std::vector<Node*>& out) {
    out.clear();
    if (p.cfg.flags & CA_NO_SHARING) return;
    const int32_t c = p.cfg.chunk;
    const Node* node = &p.root;
    for (int32_t i = 0; i < n / c; ++i) {
        Node* ch = find_child(p, node, tokens + (size_t)i * c, c, chunk_hash(tokens + (size_t)i * c, c));
        if (!ch) break;
        out.push_back(ch);
        node = ch;
    }
}

}  // namespace

int32_t pool_match(const Pool& p, const int32_t* tokens, int32_t n) {
    std::vector<Node*> path;
    walk_matched(p, tokens, n, path);
    return (int32_t)path.size() * p.cfg.chunk;
}

int pool_insert(Pool& p, int64_t seq_id, const int32_t* tokens, int32_t n,
                std::vector<std::pair<int32_t, int32_t>>* new_chunks, int32_t* n_shared) {
    if (n <= 0 || !tokens) return CA_ERR_INVALID;
    if (p.seqs.count(seq_id)) return CA_ERR_EXISTS;
    const int32_t c = p.cfg.chunk;
    const int32_t pieces = (n + c - 1) / c;
    Sequence seq;
    seq.length = n;
    alloc_point(p);
    walk_matched(p, tokens, n, seq.path);
    const int32_t matched = (int32_t)seq.path.size();
    const int32_t n_new = pieces - matched;
    if ((size_t)n_new > p.heap.size()) return CA_ERR_OOM;
    alloc_point(p);
    seq.path.reserve(pieces);               // nothing below pushes past it
    const size_t chunks_before = new_chunks ? new_chunks->size() : 0;
    // The sequence's map entry is allocated before anything changes and
    // filled at the end by a move that cannot throw.
    alloc_point(p);
    const auto entry = p.seqs.try_emplace(seq_id).first;

    // All or nothing: a host allocation that fails part-way (a child list or
    // hash index growing, the new-chunk list) undoes every change made so far
    // and rethrows, so the pool is as before the call.
    for (Node* m : seq.path) m->refcount += 1;
    try {
        Node* node = matched ? seq.path.back() : &p.root;
        const bool share = !(p.cfg.flags & CA_NO_SHARING);
        for (int32_t i = matched; i < pieces; ++i) {
            const int32_t a = i * c, len = std::min(c, n - a);
            const int32_t slot = heap_pop(p.heap);
            Node* ch = &p.nodes[slot];
            ch->slot = slot;
            ch->ntok = len;
            std::copy(tokens + a, tokens + a + len, p.tokens.begin() + (size_t)slot * c);
            ch->matchable = share && len == c;
            ch->hash = ch->matchable ? chunk_hash(tokens + a, c) : 0;
            ch->parent = node;
            ch->children.clear();
            ch->index.reset();
            ch->refcount = 1;
            seq.path.push_back(ch);         // reserved: cannot throw
            alloc_point(p);
            add_child(node, ch);
            node = ch;
            if (new_chunks) {
                alloc_point(p);
                new_chunks->emplace_back(a, slot);
            }
        }
    } catch (...) {
        for (size_t i = seq.path.size(); i-- > (size_t)matched;) {
            Node* x = seq.path[i];
            drop_child(x->parent, x);
            heap_push(p.heap, x->slot);
            x->children.clear();
            x->index.reset();
            x->parent = nullptr;
            x->matchable = false;
            x->refcount = 0;
        }
        for (int32_t i = 0; i < matched; ++i) seq.path[i]->refcount -= 1;
        if (new_chunks) new_chunks->resize(chunks_before);
        p.seqs.erase(entry);
        throw;
    }
    entry->second = std::move(seq);
    p.generation += 1;
    if (n_shared) *n_shared = matched * c;
    return CA_OK;
}

size_t pool_tile_bytes(const PoolCfg& c) {
    return (size_t)c.capacity_slots * c.n_layers * 2 * kv_heads(c) * c.chunk * c.head_dim * kv_elem_bytes(c);
}

size_t pool_total_bytes(const PoolCfg& c) {
    return pool_tile_bytes(c) + (((size_t)c.capacity_slots * sizeof(int32_t) + 255) & ~size_t(255));
}

int pool_append(Pool& p, int64_t seq_id, const int32_t* tokens, int32_t n,
                std::vector<ScatterChunk>* copies, AppendUndo* undo) {
    if (n <= 0 || !tokens) return CA_ERR_INVALID;
    auto it = p.seqs.find(seq_id);
    if (it == p.seqs.end()) return CA_ERR_NOT_FOUND;
    Sequence& seq = it->second;
    const int32_t c = p.cfg.chunk;
    const bool share = !(p.cfg.flags & CA_NO_SHARING);
    Node* last = seq.path.back();
    const int32_t fill = std::min(c - last->ntok, n);
    const int32_t n_new = (n - fill + c - 1) / c;
    if ((size_t)n_new > p.heap.size()) return CA_ERR_OOM;
    alloc_point(p);
    seq.path.reserve(seq.path.size() + n_new);   // nothing below pushes past it
    const AppendUndo u{last, last->ntok, last->matchable, last->hash, seq.path.size(), p.generation, seq.length};
    if (undo) *undo = u;
    const size_t copies_before = copies ? copies->size() : 0;
    // All or nothing, as for an insert: a host allocation that fails part-way
    // undoes the append and rethrows.
    try {
        if (fill > 0) {
            // the partial last chunk is private (never matched), so it grows in place
            std::copy(tokens, tokens + fill, p.tokens.begin() + (size_t)last->slot * c + last->ntok);
            if (copies) {
                alloc_point(p);
                copies->push_back({0, fill, last->slot, last->ntok});
            }
            last->ntok += fill;
            if (last->ntok == c && share) {
                const int32_t* lt = chunk_tokens(p, last);
                const uint64_t h = chunk_hash(lt, c);
                if (!find_child(p, last->parent, lt, c, h)) {
                    last->hash = h;
                    last->matchable = true;
                    if (last->parent->index) {
                        alloc_point(p);
                        last->parent->index->emplace(h, last);
                    }
                }
            }
        }
        Node* node = last;
        for (int32_t i = 0; i < n_new; ++i) {
            const int32_t a = fill + i * c, len = std::min(c, n - a);
            const int32_t slot = heap_pop(p.heap);
            Node* ch = &p.nodes[slot];
            ch->slot = slot;
            ch->ntok = len;
            std::copy(tokens + a, tokens + a + len, p.tokens.begin() + (size_t)slot * c);
            const uint64_t h = (share && len == c) ? chunk_hash(tokens + a, c) : 0;
            // an append never matches, and an equal sibling keeps its place
            ch->matchable = share && len == c && !find_child(p, node, tokens + a, c, h);
            ch->hash = h;
            ch->parent = node;
            ch->children.clear();
            ch->index.reset();
            ch->refcount = 1;
            seq.path.push_back(ch);             // reserved: cannot throw
            alloc_point(p);
            add_child(node, ch);
            if (copies) {
                alloc_point(p);
                copies->push_back({a, len, slot, 0});
            }
            node = ch;
        }
    } catch (...) {
        pool_undo_append(p, seq_id, u);
        if (copies) copies->resize(copies_before);
        throw;
    }
    seq.length += n;
    if (n_new > 0) p.generation += 1;
    return CA_OK;
}

void pool_undo_append(Pool& p, int64_t seq_id, const AppendUndo& u) {
    Sequence& seq = p.seqs.at(seq_id);
    while (seq.path.size() > u.path_size) {
        Node* x = seq.path.back();
        seq.path.pop_back();
        drop_child(x->parent, x);
        heap_push(p.heap, x->slot);
        x->children.clear();
        x->index.reset();
        x->parent = nullptr;
        x->matchable = false;
        x->refcount = 0;
    }
    Node* last = u.last;
    if (last->matchable && !u.matchable && last->parent->index) {
        auto m = last->parent->index->find(last->hash);
        if (m != last->parent->index->end() && m->second == last) last->parent->index->erase(m);
    }
    last->ntok = u.ntok;
    last->matchable = u.matchable;
    last->hash = u.hash;
    seq.length = u.length;
    p.generation = u.generation;
}

int pool_remove(Pool& p, int64_t seq_id) {
    auto it = p.seqs.find(seq_id);
    if (it == p.seqs.end()) return CA_ERR_NOT_FOUND;
    std::vector<Node*> path = std::move(it->second.path);
    p.seqs.erase(it);
    // Refcounts never grow along a path, so the chunks that drop to zero form
    // a suffix of it; detach its first node and free the whole suffix.
    size_t first_free = path.size();
    for (size_t i = 0; i < path.size(); ++i) {
        path[i]->refcount -= 1;
        if (path[i]->refcount == 0 && first_free == path.size()) first_free = i;
    }
    if (first_free < path.size()) {
        Node* top = path[first_free];
        drop_child(top->parent, top);
        for (size_t i = first_free; i < path.size(); ++i) {
            Node* x = path[i];
            heap_push(p.heap, x->slot);
            x->children.clear();
            x->index.reset();
            x->parent = nullptr;
            x->matchable = false;
        }
    }
    p.generation += 1;
    return CA_OK;
}

}  // namespace ca
