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
#include <string>

#include "ca_internal.h"

namespace ca {
namespace {

std::string chunk_key(const int32_t* tokens, int32_t c) {
    return std::string(reinterpret_cast<const char*>(tokens), sizeof(int32_t) * (size_t)c);
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

int32_t count_matched(const Pool& p, const int32_t* tokens, int32_t n, const Node** last) {
    const int32_t c = p.cfg.chunk;
    const Node* node = p.root.get();
    int32_t matched = 0;
    if (!(p.cfg.flags & CA_NO_SHARING)) {
        for (int32_t i = 0; i < n / c; ++i) {
            auto it = node->match.find(chunk_key(tokens + (size_t)i * c, c));
            if (it == node->match.end()) break;
            node = it->second;
            ++matched;
        }
    }
    if (last) *last = node;
    return matched;
}

}  // namespace

int32_t pool_match(const Pool& p, const int32_t* tokens, int32_t n) {
    return count_matched(p, tokens, n, nullptr) * p.cfg.chunk;
}

int pool_insert(Pool& p, int64_t seq_id, const int32_t* tokens, int32_t n,
                std::vector<std::pair<int32_t, int32_t>>* new_chunks, int32_t* n_shared) {
    if (n <= 0 || !tokens) return CA_ERR_INVALID;
    if (p.seqs.count(seq_id)) return CA_ERR_EXISTS;
    const int32_t c = p.cfg.chunk;
    const int32_t pieces = (n + c - 1) / c;
    const Node* last = nullptr;
    const int32_t matched = count_matched(p, tokens, n, &last);
    const int32_t n_new = pieces - matched;
    if ((size_t)n_new > p.heap.size()) return CA_ERR_OOM;

    Sequence seq;
    seq.length = n;
    seq.path.reserve(pieces);
    Node* node = p.root.get();
    for (int32_t i = 0; i < pieces; ++i) {
        const int32_t a = i * c, len = std::min(c, n - a);
        if (i < matched) {
            node = node->match.find(chunk_key(tokens + a, c))->second;
        } else {
            const int32_t slot = heap_pop(p.heap);
            std::unique_ptr<Node> ch(new Node());
            ch->slot = slot;
            ch->tokens.assign(tokens + a, tokens + a + len);
            ch->parent = node;
            node->children.push_back(ch.get());
            if (len == c && !(p.cfg.flags & CA_NO_SHARING))
                node->match.emplace(chunk_key(tokens + a, c), ch.get());
            node = ch.get();
            p.nodes_by_slot[slot] = std::move(ch);
            if (new_chunks) new_chunks->emplace_back(a, slot);
        }
        node->refcount += 1;
        seq.path.push_back(node);
    }
    p.seqs.emplace(seq_id, std::move(seq));
    p.generation += 1;
    if (n_shared) *n_shared = matched * c;
    return CA_OK;
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
        Node* parent = top->parent;
        auto& ch = parent->children;
        ch.erase(std::find(ch.begin(), ch.end(), top));
        if (top->tokens.size() == (size_t)p.cfg.chunk) {
            auto m = parent->match.find(chunk_key(top->tokens.data(), p.cfg.chunk));
            if (m != parent->match.end() && m->second == top) parent->match.erase(m);
        }
        for (size_t i = first_free; i < path.size(); ++i) {
            const int32_t slot = path[i]->slot;
            heap_push(p.heap, slot);
            p.nodes_by_slot[slot].reset();
        }
    }
    p.generation += 1;
    return CA_OK;
}

}  // namespace ca
