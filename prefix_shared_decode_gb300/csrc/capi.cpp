// The C ABI of libchunk_attention (declared in include/chunk_attention.h):
// argument checks, object lifetimes and the host side of each call.  No C++
// exception crosses this boundary.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstring>
#include <new>

#include "ca_internal.h"

using namespace ca;

struct ca_pool : Pool {};
struct ca_sched : Sched {};

namespace {

constexpr int32_t kHostOnlyGrid = 2 * 152;   // plan grid for a pool with no GPU

// An NVTX range around a host call (insert, append, remove, schedule,
// attention), so that a profiler attached to the process shows where each
// call's host work and kernels belong; without a profiler a push or pop is a
// call through a no-op pointer.
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

template <class F>
int guard(F&& f) {
    try {
        return f();
    } catch (const std::bad_alloc&) {
        return CA_ERR_OOM;
    } catch (...) {
        return CA_ERR_INVALID;
    }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cfg(const PoolCfg* c) {
    if (!c) return CA_ERR_INVALID;
    if (c->n_layers < 1 || c->n_heads < 1 || c->capacity_slots < 1) return CA_ERR_INVALID;
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return CA_ERR_UNSUPPORTED;
    // head_dim 256: chunks of at most 32 tokens (two stages of K+V must fit
    // beside the query tile), fp16 only
    if (c->head_dim == 256 && (c->chunk > 32 || (c->flags & CA_KV_FP8))) return CA_ERR_UNSUPPORTED;
    if (c->chunk != 16 && c->chunk != 32 && c->chunk != 64) return CA_ERR_UNSUPPORTED;
    if (c->flags & ~(CA_NO_SHARING | CA_KV_FP8)) return CA_ERR_INVALID;
    if (c->flags & CA_KV_FP8) {
        if (c->head_dim != 128) return CA_ERR_UNSUPPORTED;
        for (float sc : {c->k_scale, c->v_scale})
            if (!(sc == 0.f || (sc > 0.f && sc < 3.0e38f))) return CA_ERR_INVALID;
    }
    if (c->n_kv_heads < 0 || (c->n_kv_heads > 0 && c->n_heads % c->n_kv_heads)) return CA_ERR_INVALID;
    if (c->n_heads / kv_heads(*c) > max_query_rows(*c)) return CA_ERR_UNSUPPORTED;
    // TMA row coordinates are 32-bit.
    const long double rows = (long double)c->capacity_slots * c->n_layers * 2 * kv_heads(*c) * c->chunk;
    if (rows > 2147483647.0L) return CA_ERR_UNSUPPORTED;
    return CA_OK;
}

size_t pool_bytes(const PoolCfg& c) { return pool_total_bytes(c); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? CA_OK : CA_ERR_CUDA; }

// Copy the plan blob to the device through the next pinned staging buffer.
int upload_plan(Sched& s, cudaStream_t stream) {
    const int i = s.pinned_next;
    s.pinned_next ^= 1;
    cudaEvent_t& done = reinterpret_cast<cudaEvent_t&>(s.pinned_done[i]);
    if (done && cudaEventSynchronize(done) != cudaSuccess) return CA_ERR_CUDA;  // its last copy
    if (s.pinned_bytes[i] < s.blob.size()) {
        if (s.pinned[i]) cudaFreeHost(s.pinned[i]);
        s.pinned[i] = nullptr;
        s.pinned_bytes[i] = 0;
        const size_t want = s.blob.size() + s.blob.size() / 2;
        if (cudaHostAlloc(&s.pinned[i], want, cudaHostAllocDefault) != cudaSuccess) return CA_ERR_CUDA;
        s.pinned_bytes[i] = want;
    }
    if (!done && cudaEventCreateWithFlags(&done, cudaEventDisableTiming) != cudaSuccess) return CA_ERR_CUDA;
    std::memcpy(s.pinned[i], s.blob.data(), s.blob.size());
    if (cudaMemcpyAsync(s.dev, s.pinned[i], s.blob.size(), cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return CA_ERR_CUDA;
    return cuda_status(cudaEventRecord(done, stream));
}

}  // namespace

extern "C" {

int ca_pool_bytes_ex(const ca_pool_config_ex* cfg_ex, size_t* bytes_out) {
    if (!cfg_ex) return CA_ERR_INVALID;
    const PoolCfg cfg = pool_cfg(*cfg_ex);
    int st = check_cfg(&cfg);
    if (st) return st;
    if (!bytes_out) return CA_ERR_INVALID;
    *bytes_out = pool_bytes(cfg);
    return CA_OK;
}

int ca_pool_bytes(const ca_pool_config* cfg, size_t* bytes_out) {
    if (!cfg) return CA_ERR_INVALID;
    ca_pool_config_ex e{};
    e.base = *cfg;
    return ca_pool_bytes_ex(&e, bytes_out);
}

int ca_pool_create_ex(const ca_pool_config_ex* cfg_ex, void* kv_dev, size_t kv_bytes, ca_pool** pool_out) {
    return guard([&] {
        if (!cfg_ex) return CA_ERR_INVALID;
        const PoolCfg c = pool_cfg(*cfg_ex);
        const PoolCfg* cfg = &c;
        int st = check_cfg(cfg);
        if (st) return st;
        if (!pool_out) return CA_ERR_INVALID;
        *pool_out = nullptr;
        if (kv_dev && (!aligned(kv_dev, 1024) || kv_bytes < pool_bytes(*cfg))) return CA_ERR_INVALID;
        std::unique_ptr<ca_pool> p(new ca_pool());
        p->cfg = *cfg;
        p->kv = kv_dev;
        p->kv_bytes = kv_bytes;
        p->nodes.resize(cfg->capacity_slots);
        p->tokens.assign((size_t)cfg->capacity_slots * cfg->chunk, 0);
        p->heap.resize(cfg->capacity_slots);
        for (int32_t i = 0; i < cfg->capacity_slots; ++i) p->heap[i] = i;   // sorted = min-heap
        if (kv_dev) {
            if (cudaGetDevice(&p->device) != cudaSuccess) return CA_ERR_CUDA;
            if (cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess)
                return CA_ERR_CUDA;
            int ctas = 1;
            st = kernel_ctas_per_sm(*cfg, &ctas);
            if (st) return st;
            p->num_sms *= ctas;   // grid = resident CTAs
            st = make_tensor_map(*p);
            if (st) return st;
        }
        *pool_out = p.release();
        return CA_OK;
    });
}

int ca_pool_create(const ca_pool_config* cfg, void* kv_dev, size_t kv_bytes, ca_pool** pool_out) {
    if (!cfg) return CA_ERR_INVALID;
    ca_pool_config_ex e{};
    e.base = *cfg;
    return ca_pool_create_ex(&e, kv_dev, kv_bytes, pool_out);
}

int ca_pool_destroy(ca_pool* pool) {
    delete pool;
    return CA_OK;
}

int ca_match_prefix(const ca_pool* pool, const int32_t* tokens, int32_t n, int32_t* n_matched_out) {
    if (!pool || !n_matched_out || n < 0 || (n > 0 && !tokens)) return CA_ERR_INVALID;
    return guard([&] {
        *n_matched_out = pool_match(*pool, tokens, n);
        return CA_OK;
    });
}

int ca_insert_tokens(ca_pool* pool, int64_t seq_id, const int32_t* tokens, int32_t n,
                     const void* k_dev, const void* v_dev, void* stream, int32_t* n_shared_out) {
    return ca_insert_batch(pool, 1, &seq_id, tokens, &n, k_dev, v_dev, stream, n_shared_out);
}

int ca_insert_batch(ca_pool* pool, int32_t n_seqs, const int64_t* seq_ids, const int32_t* tokens,
                    const int32_t* lengths, const void* k_dev, const void* v_dev, void* stream,
                    int32_t* n_shared_out) {
    const Range range("ca_insert");
    if (!pool || n_seqs < 1 || !seq_ids || !tokens || !lengths) return CA_ERR_INVALID;
    int64_t total = 0;
    for (int32_t i = 0; i < n_seqs; ++i) {
        if (lengths[i] < 1) return CA_ERR_INVALID;
        total += lengths[i];
    }
    if (total > INT32_MAX) return CA_ERR_INVALID;
    if (pool->kv) {
        if (!k_dev || !v_dev || !aligned(k_dev, 16) || !aligned(v_dev, 16)) return CA_ERR_INVALID;
    } else if (k_dev || v_dev) {
        return CA_ERR_INVALID;
    }
    return guard([&] {
        const int64_t gen = pool->generation;
        std::vector<std::pair<int32_t, int32_t>> fresh;
        std::vector<ScatterChunk> copies;
        int32_t row0 = 0, st = CA_OK, inserted = 0;
        // The pool must be unchanged after any failure: a failed sequence
        // undoes itself (pool_insert is all or nothing, exceptions included),
        // the ones before it are removed again here.
        auto undo = [&] {
            for (int32_t j = inserted - 1; j >= 0; --j) pool_remove(*pool, seq_ids[j]);
            pool->generation = gen;
        };
        try {
            for (int32_t i = 0; i < n_seqs; ++i) {
                fresh.clear();
                int32_t shared = 0;
                st = pool_insert(*pool, seq_ids[i], tokens + row0, lengths[i], &fresh, &shared);
                if (st) break;
                ++inserted;
                for (const auto& f : fresh) {
                    alloc_point(*pool);
                    copies.push_back({row0 + f.first, std::min(pool->cfg.chunk, lengths[i] - f.first), f.second, 0});
                }
                if (n_shared_out) n_shared_out[i] = shared;
                row0 += lengths[i];
            }
            if (!st && pool->kv) st = launch_scatter(*pool, k_dev, v_dev, (int32_t)total, copies, stream);
        } catch (...) {
            undo();
            throw;
        }
        if (st) undo();
        return st;
    });
}

int ca_append_tokens(ca_pool* pool, int64_t seq_id, const int32_t* tokens, int32_t n,
                     const void* k_dev, const void* v_dev, void* stream, int32_t* n_new_chunks_out) {
    const Range range("ca_append_tokens");
    if (!pool || n <= 0 || !tokens) return CA_ERR_INVALID;
    if (pool->kv) {
        if (!k_dev || !v_dev || !aligned(k_dev, 16) || !aligned(v_dev, 16)) return CA_ERR_INVALID;
    } else if (k_dev || v_dev) {
        return CA_ERR_INVALID;
    }
    return guard([&] {
        std::vector<ScatterChunk> copies;
        AppendUndo undo;
        const size_t before = pool->seqs.count(seq_id) ? pool->seqs.at(seq_id).path.size() : 0;
        int st = pool_append(*pool, seq_id, tokens, n, &copies, &undo);
        if (st) return st;
        if (pool->kv) {
            st = launch_scatter(*pool, k_dev, v_dev, n, copies, stream);
            if (st) {
                pool_undo_append(*pool, seq_id, undo);
                return st;
            }
        }
        if (n_new_chunks_out) *n_new_chunks_out = (int32_t)(pool->seqs.at(seq_id).path.size() - before);
        return CA_OK;
    });
}

int ca_remove_seq(ca_pool* pool, int64_t seq_id) {
    const Range range("ca_remove");
    if (!pool) return CA_ERR_INVALID;
    return guard([&] { return pool_remove(*pool, seq_id); });
}

int ca_remove_batch(ca_pool* pool, int32_t n_seqs, const int64_t* seq_ids) {
    const Range range("ca_remove");
    if (!pool || n_seqs < 0 || (n_seqs > 0 && !seq_ids)) return CA_ERR_INVALID;
    return guard([&] {
        for (int32_t i = 0; i < n_seqs; ++i)
            if (!pool->seqs.count(seq_ids[i])) return CA_ERR_NOT_FOUND;
        std::vector<int64_t> sorted(seq_ids, seq_ids + n_seqs);
        std::sort(sorted.begin(), sorted.end());
        if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return CA_ERR_INVALID;
        for (int32_t i = 0; i < n_seqs; ++i) pool_remove(*pool, seq_ids[i]);
        return CA_OK;
    });
}

int ca_pool_stats(const ca_pool* pool, ca_stats* out) {
    if (!pool || !out) return CA_ERR_INVALID;
    return guard([&] {
        ca_stats s{};
        s.free_slots = (int64_t)pool->heap.size();
        s.live_slots = pool->cfg.capacity_slots - s.free_slots;
        for (const auto& n : pool->nodes) s.refcount_sum += n.refcount;
        s.live_seqs = (int64_t)pool->seqs.size();
        s.generation = pool->generation;
        *out = s;
        return CA_OK;
    });
}

int ca_seq_slots(const ca_pool* pool, int64_t seq_id, int32_t* slots, int32_t cap, int32_t* n_out) {
    if (!pool || !n_out || cap < 0 || (cap > 0 && !slots)) return CA_ERR_INVALID;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return CA_ERR_NOT_FOUND;
    const auto& path = it->second.path;
    for (int32_t i = 0; i < cap && i < (int32_t)path.size(); ++i) slots[i] = path[i]->slot;
    *n_out = (int32_t)path.size();
    return CA_OK;
}

int ca_build_schedule(ca_pool* pool, const int64_t* seq_ids, int32_t b, ca_sched** inout, void* stream) {
    return ca_build_schedule_ex(pool, seq_ids, b, 1, 0u, inout, stream);
}

int ca_build_schedule_ex(ca_pool* pool, const int64_t* seq_ids, int32_t b, int32_t q_len, uint32_t flags,
                         ca_sched** inout, void* stream) {
    const Range range("ca_build_schedule");
    if (!pool || !inout || !seq_ids || b < 1 || q_len < 1 || (flags & ~(CA_SCHED_NO_TPP | CA_SCHED_CAUSAL)))
        return CA_ERR_INVALID;
    if ((int64_t)q_len * (pool->cfg.n_heads / kv_heads(pool->cfg)) > max_query_rows(pool->cfg))
        return CA_ERR_UNSUPPORTED;
    if (q_len == 1) flags &= ~CA_SCHED_CAUSAL;       // one query token sees its whole context
    return guard([&] {
        ca_sched* s = *inout;
        if (s && s->pool == pool && s->generation == pool->generation && s->flags == flags &&
            s->q_len == q_len && (int32_t)s->seq_ids.size() == b &&
            std::equal(seq_ids, seq_ids + b, s->seq_ids.begin()))
            return CA_OK;                   // context unchanged since the tree last changed
        if (flags & CA_SCHED_CAUSAL)
            for (int32_t i = 0; i < b; ++i) {
                auto it = pool->seqs.find(seq_ids[i]);
                if (it != pool->seqs.end() && it->second.length < q_len) return CA_ERR_INVALID;
            }
        std::unique_ptr<ca_sched> fresh;
        if (!s) {
            fresh.reset(new ca_sched());
            s = fresh.get();
        }
        int st = build_tables(*pool, seq_ids, b, flags, s->t_next);
        if (st) return st;                  // s (if reused) keeps its previous tables
        std::swap(s->t, s->t_next);
        // Invalid until the plan for these tables is built and uploaded: a
        // failure from here on leaves a schedule that every later call
        // rebuilds and every decode call refuses as stale.
        s->generation = -1;
        s->pool = pool;
        s->flags = flags;
        s->q_len = q_len;
        s->seq_ids.assign(seq_ids, seq_ids + b);
        alloc_point(*pool);                 // the plan's vectors may grow below
        build_plan(*pool, s->t, pool->kv ? pool->num_sms : kHostOnlyGrid, q_len, s->plan);
        layout_plan(s->plan, b, s->layout, s->blob, s->t);
        layout_ws(s->plan, *pool, b, s->ws);
        if (pool->kv) {
            if (s->dev_bytes < s->blob.size()) {
                if (s->dev) cudaFree(s->dev);
                s->dev = nullptr;
                s->dev_bytes = 0;
                if (cudaMalloc(&s->dev, s->blob.size()) != cudaSuccess) {
                    s->generation = -1;
                    return CA_ERR_CUDA;
                }
                s->dev_bytes = s->blob.size();
            }
            st = upload_plan(*s, static_cast<cudaStream_t>(stream));
            if (st) {
                s->generation = -1;
                return st;
            }
        }
        s->generation = pool->generation;
        if (fresh) *inout = fresh.release();
        return CA_OK;
    });
}

int ca_sched_destroy(ca_sched* sched) {
    if (!sched) return CA_OK;
    for (int i = 0; i < 2; ++i) {
        if (sched->pinned_done[i]) {
            cudaEventSynchronize(static_cast<cudaEvent_t>(sched->pinned_done[i]));
            cudaEventDestroy(static_cast<cudaEvent_t>(sched->pinned_done[i]));
        }
        if (sched->pinned[i]) cudaFreeHost(sched->pinned[i]);
    }
    if (sched->dev) cudaFree(sched->dev);
    delete sched;
    return CA_OK;
}

int ca_sched_counts(const ca_sched* s, int32_t counts[6]) {
    if (!s || !counts) return CA_ERR_INVALID;
    counts[0] = s->t.b;
    counts[1] = (int32_t)(s->t.cf_rows.size() / 4);
    counts[2] = (int32_t)(s->t.cf_runs.size() / 4);
    counts[3] = (int32_t)(s->t.sf_chunks.size() / 2);
    counts[4] = (int32_t)s->t.merge_runs.size();
    counts[5] = (int32_t)s->plan.units.size();
    return CA_OK;
}

int ca_export_tables(const ca_sched* s, int32_t* seq_perm, int32_t* cf_rows, int32_t* cf_runs,
                     int32_t* sf_offsets, int32_t* sf_chunks, int32_t* merge_offsets,
                     int32_t* merge_runs) {
    if (!s) return CA_ERR_INVALID;
    auto put = [](int32_t* dst, const std::vector<int32_t>& v) {
        if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int32_t));
    };
    put(seq_perm, s->t.seq_perm);
    put(cf_rows, s->t.cf_rows);
    put(cf_runs, s->t.cf_runs);
    put(sf_offsets, s->t.sf_offsets);
    put(sf_chunks, s->t.sf_chunks);
    put(merge_offsets, s->t.merge_offsets);
    put(merge_runs, s->t.merge_runs);
    return CA_OK;
}

int ca_export_plan(const ca_sched* s, int32_t counts[4], int32_t* units, int32_t* cta_begin,
                   int32_t* pbase, int32_t* chunks) {
    if (!s || !counts) return CA_ERR_INVALID;
    counts[0] = (int32_t)s->plan.units.size();
    counts[1] = s->plan.grid;
    counts[2] = (int32_t)s->plan.pbase.size();
    counts[3] = (int32_t)s->plan.chunks.size();
    static_assert(sizeof(Unit) == 12 * sizeof(int32_t), "Unit is 12 int32");
    static_assert(sizeof(ChunkRef) == 2 * sizeof(int32_t), "ChunkRef is 2 int32");
    if (units && !s->plan.units.empty())
        std::memcpy(units, s->plan.units.data(), s->plan.units.size() * sizeof(Unit));
    if (cta_begin) std::memcpy(cta_begin, s->plan.cta_begin.data(), s->plan.cta_begin.size() * sizeof(int32_t));
    if (pbase) std::memcpy(pbase, s->plan.pbase.data(), s->plan.pbase.size() * sizeof(int32_t));
    if (chunks && !s->plan.chunks.empty())
        std::memcpy(chunks, s->plan.chunks.data(), s->plan.chunks.size() * sizeof(ChunkRef));
    return CA_OK;
}

int ca_workspace_bytes(const ca_sched* s, size_t* bytes_out) {
    if (!s || !bytes_out) return CA_ERR_INVALID;
    *bytes_out = s->ws.total;
    return CA_OK;
}

int ca_workspace_bytes_host(const ca_sched* s, size_t* bytes_out) {
    if (!s || !bytes_out) return CA_ERR_INVALID;
    *bytes_out = s->ws.total_host;
    return CA_OK;
}

static int decode_checks(const ca_pool* pool, const ca_sched* s, int32_t layer, void* ws_dev,
                         size_t ws_bytes, size_t need) {
    if (!pool || !s || !pool->kv || s->pool != pool || !s->dev) return CA_ERR_INVALID;
    if (s->generation != pool->generation) return CA_ERR_STALE;
    if (layer < 0 || layer >= pool->cfg.n_layers) return CA_ERR_INVALID;
    if (!ws_dev || !aligned(ws_dev, 256) || ws_bytes < need) return CA_ERR_INVALID;
    return CA_OK;
}

}  // extern "C"

namespace ca {
AttnParams attn_params(const Pool& pool, const Sched& s, int32_t layer, const void* q, void* out,
                       float scale, void* ws_dev) {
    unsigned char* dev = static_cast<unsigned char*>(s.dev);
    unsigned char* ws = static_cast<unsigned char*>(ws_dev);
    AttnParams a{};
    a.chunks = reinterpret_cast<const ChunkRef*>(dev + s.layout.chunks);
    a.units = reinterpret_cast<const Unit*>(dev + s.layout.units);
    a.cta_head = reinterpret_cast<const CtaHead*>(dev + s.layout.cta_head);
    a.seq_perm = reinterpret_cast<const int32_t*>(dev + s.layout.seq_perm);
    a.pbase = reinterpret_cast<const int32_t*>(dev + s.layout.pbase);
    a.slot_ntok = reinterpret_cast<const int32_t*>(static_cast<const unsigned char*>(pool.kv) +
                                                   pool_tile_bytes(pool.cfg));
    a.status = reinterpret_cast<int32_t*>(dev + s.layout.status);
    a.dyn_counter = reinterpret_cast<int32_t*>(dev + s.layout.counter);
    a.chunk_tok0 = reinterpret_cast<const int32_t*>(dev + s.layout.chunk_tok0);
    a.ctx_len = reinterpret_cast<const int32_t*>(dev + s.layout.ctx_len);
    a.q_len = s.q_len;
    a.causal = (s.flags & CA_SCHED_CAUSAL) ? 1 : 0;
    a.dyn_begin = s.plan.cta_begin[s.plan.grid];
    a.dyn_end = (int32_t)s.plan.units.size();
    a.q = static_cast<const uint16_t*>(q);
    a.out = static_cast<uint16_t*>(out);
    a.part_o = reinterpret_cast<float*>(ws + s.ws.part_o);
    a.part_ms = reinterpret_cast<float2*>(ws + s.ws.part_ms);
    a.n_layers = pool.cfg.n_layers;
    a.n_heads = pool.cfg.n_heads;
    a.n_kv_heads = kv_heads(pool.cfg);
    a.group = pool.cfg.n_heads / a.n_kv_heads;
    a.layer = layer;
    a.capacity = pool.cfg.capacity_slots;
    const bool f8 = (pool.cfg.flags & CA_KV_FP8) != 0;
    a.scale_log2 = scale * 1.4426950408889634f * (f8 ? kv_scale_of(pool.cfg.k_scale) : 1.f);
    a.out_scale = f8 ? kv_scale_of(pool.cfg.v_scale) : 1.f;
    return a;
}
}  // namespace ca

extern "C" {

static int decode_launch(const ca_pool* pool, const ca_sched* s, int32_t layer, const void* q,
                         void* out, float scale, void* ws_dev, void* stream) {
    const AttnParams a = attn_params(*pool, *s, layer, q, out, scale, ws_dev);
    return launch_attention(*pool, *s, a, stream);
}

int ca_decode_attention(const ca_pool* pool, const ca_sched* s, int32_t layer, const void* q_dev,
                        void* out_dev, float scale, void* ws_dev, size_t ws_bytes, void* stream) {
    const Range range("ca_decode_attention");
    int st = decode_checks(pool, s, layer, ws_dev, ws_bytes, s ? s->ws.total : 0);
    if (st) return st;
    if (!q_dev || !out_dev || !aligned(q_dev, 16) || !aligned(out_dev, 16)) return CA_ERR_INVALID;
    return decode_launch(pool, s, layer, q_dev, out_dev, scale, ws_dev, stream);
}

int ca_decode_attention_host(const ca_pool* pool, const ca_sched* s, int32_t layer,
                             const void* q_host, void* out_host, float scale, void* ws_dev,
                             size_t ws_bytes, void* stream) {
    const Range range("ca_decode_attention");
    int st = decode_checks(pool, s, layer, ws_dev, ws_bytes, s ? s->ws.total_host : 0);
    if (st) return st;
    if (!q_host || !out_host) return CA_ERR_INVALID;
    // Pinned host memory is mapped into the device's address space (on GB300
    // over NVLink-C2C): when both buffers have a device mapping, the kernels
    // read q from it and the merge writes out to it directly, so no copy
    // steps serialise with the kernels.  Otherwise q and out are staged in
    // the workspace with one copy each way.
    void* q_map = nullptr;
    void* out_map = nullptr;
    if (cudaHostGetDevicePointer(&q_map, const_cast<void*>(q_host), 0) == cudaSuccess &&
        cudaHostGetDevicePointer(&out_map, out_host, 0) == cudaSuccess)
        return decode_launch(pool, s, layer, q_map, out_map, scale, ws_dev, stream);
    (void)cudaGetLastError();   // the failed lookup is not an error of this call
    const size_t bytes = (size_t)s->t.b * s->q_len * pool->cfg.n_heads * pool->cfg.head_dim * 2;
    unsigned char* ws = static_cast<unsigned char*>(ws_dev);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(ws + s->ws.q_stage, q_host, bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return CA_ERR_CUDA;
    st = decode_launch(pool, s, layer, ws + s->ws.q_stage, ws + s->ws.out_stage, scale, ws_dev, stream);
    if (st) return st;
    return cuda_status(cudaMemcpyAsync(out_host, ws + s->ws.out_stage, bytes, cudaMemcpyDeviceToHost, cs));
}

int ca_sched_device_status(const ca_sched* s, void* stream) {
    if (!s) return CA_ERR_INVALID;
    if (!s->dev) {
        // A host-only pool's schedule has no device word; its host word is
        // written only by ca_sched_inject_status.
        if (!s->pool || s->pool->kv) return CA_ERR_INVALID;
        const int32_t word = s->host_status;
        s->host_status = 0;
        return word;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess) return CA_ERR_CUDA;
    int32_t word = 0;
    int32_t* dev_word = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(s->dev) + s->layout.status);
    if (cudaMemcpy(&word, dev_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return CA_ERR_CUDA;
    if (word != 0) {
        // A call that stopped early may have left the queue counter
        // mid-count: clear it with the word.
        if (cudaMemset(dev_word, 0, sizeof(word)) != cudaSuccess ||
            cudaMemset(static_cast<unsigned char*>(s->dev) + s->layout.counter, 0, sizeof(int32_t)) !=
                cudaSuccess)
            return CA_ERR_CUDA;
    }
    return word;
}

int ca_sched_inject_status(ca_sched* s, int32_t code, void* stream) {
    if (!s || code >= 0 || code < CA_ERR_SCRATCH_LIMIT) return CA_ERR_INVALID;
    if (!s->dev) {
        if (!s->pool || s->pool->kv) return CA_ERR_INVALID;
        s->host_status = code;
        return CA_OK;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t* dev_word = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(s->dev) + s->layout.status);
    if (cudaMemcpyAsync(dev_word, &code, sizeof(code), cudaMemcpyHostToDevice, cs) != cudaSuccess) return CA_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(cs));
}

int ca_sched_inject_stall(ca_sched* s, int32_t n_calls) {
    if (!s || n_calls < 0) return CA_ERR_INVALID;
    s->stall_calls = n_calls;
    return CA_OK;
}

int ca_pool_inject_alloc_failure(ca_pool* pool, int32_t after_n) {
    if (!pool) return CA_ERR_INVALID;
    pool->fail_alloc_in = after_n < 0 ? -1 : after_n;
    return CA_OK;
}

int ca_sched_set_profile_events(ca_sched* s, void* event_begin, void* event_end) {
    if (!s) return CA_ERR_INVALID;
    const bool on = event_begin && event_end;
    s->ev_begin = on ? event_begin : nullptr;
    s->ev_end = on ? event_end : nullptr;
    return CA_OK;
}

int ca_kernel_launches(uint64_t* count_out) {
    if (!count_out) return CA_ERR_INVALID;
    *count_out = ca::kernel_launches();
    return CA_OK;
}

const char* ca_error_string(int status) {
    switch (status) {
        case CA_OK: return "ok";
        case CA_ERR_INVALID: return "invalid argument or state";
        case CA_ERR_OOM: return "out of chunk slots or host memory";
        case CA_ERR_NOT_FOUND: return "unknown sequence id";
        case CA_ERR_EXISTS: return "sequence id already present";
        case CA_ERR_STALE: return "schedule is older than the pool";
        case CA_ERR_CUDA: return "CUDA call failed";
        case CA_ERR_DEVICE_BOUNDS: return "kernel saw a table index out of range";
        case CA_ERR_TIMEOUT: return "kernel wait timed out";
        case CA_ERR_UNSUPPORTED: return "shape not supported";
        case CA_ERR_SCRATCH_LIMIT: return "schedule needs more scratch than the static buffer holds";
        default: return "unknown status";
    }
}

}  // extern "C"
