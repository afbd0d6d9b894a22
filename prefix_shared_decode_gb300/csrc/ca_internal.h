// Internal declarations shared by the host library (C++17) and the CUDA
// kernels of libchunk_attention.  Nothing here is part of the public C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <memory>
#include <string>
#include <unordered_map>
#include <vector>

#include <vector_types.h>

#include "../../include/chunk_attention.h"

namespace ca {

// ---------------------------------------------------------------------------
// Work plan read by the attention kernel (uploaded to the device as one blob).
//
// A unit is one stretch of chunk-heads that one CTA streams:
//  * UNIT_CF (chunk-first): rows [c_begin, c_end) of one run of chunks shared
//    by batch positions [q_lo, q_hi) (at most 64 of them), for the heads
//    [head, head + n_per_head), one head after the other,
//    against the batched queries of those positions [ChunkAttention §3.2:
//    the queries of the sequences that share a chunk form a matrix for
//    tensor-core matmul].
//  * UNIT_SF (sequence-first): a contiguous range [c_begin, c_end) of position
//    q_lo's own (head, chunk) pairs in the order h * n_per_head + j, i.e. the
//    tail of one head's chunks, whole heads, and the start of another.
// Every unit leaves one partial triple (o, m, s) per covered (position,
// head); the partials of (position p, head h) occupy ids
// [pbase[p*H+h], pbase[p*H+h+1]).
// ---------------------------------------------------------------------------
enum : int32_t { UNIT_CF = 0, UNIT_SF = 1 };

// The full shape of a pool: the public ca_pool_config_ex flattened (its
// ca_pool_config fields, then the grouped-query and fp8 fields).
struct PoolCfg {
    int32_t n_layers, n_heads, head_dim, chunk, capacity_slots;
    uint32_t flags;
    int32_t n_kv_heads;
    float k_scale, v_scale;
};
inline PoolCfg pool_cfg(const ca_pool_config_ex& e) {
    return {e.base.n_layers, e.base.n_heads, e.base.head_dim, e.base.chunk, e.base.capacity_slots,
            e.base.flags,    e.n_kv_heads,   e.k_scale,       e.v_scale};
}
inline PoolCfg pool_cfg(const ca_pool_config& b) {
    ca_pool_config_ex e{};
    e.base = b;
    return pool_cfg(e);
}

struct ChunkRef {      // one chunk the kernel reads
    int32_t slot;      // pool slot
    int32_t ntok;      // valid tokens in it (1..c)
};

struct Unit {
    int32_t kind;      // UNIT_CF or UNIT_SF
    int32_t head;      // CF: the head; SF: first head (c_begin / n_per_head)
    int32_t q_lo;      // first batch position
    int32_t q_hi;      // one past the last batch position
    int32_t c_begin;   // CF: chunk rows in the ChunkRef list; SF: linear (head, chunk) range
    int32_t c_end;
    int32_t part;      // partial index within the first covered (position, head)
    int32_t qrow;      // SF: row of q / out of its position (seq_perm[q_lo])
    int32_t n_per_head;  // SF: chunks of the position per head; CF: number of heads
    int32_t base;      // SF: ChunkRef index of the position's first chunk
    int32_t part_next; // SF: partial index within the (position, head)s after the first
    int32_t pad;
};
constexpr int kUnitInts = (int)(sizeof(Unit) / sizeof(int32_t));

// Offsets (in bytes) of the arrays inside the device plan blob.
struct PlanLayout {
    size_t chunks, units, seq_perm, pbase, status, counter, chunk_tok0, ctx_len, cta_head, total;
};

// One 128-byte line per CTA with what its producer needs to issue its first
// copies: its static unit range, its first unit, and that unit's first
// kHeadRefs chunk refs (in walk order), so the first stages go out after one
// memory round trip instead of a chain of dependent reads.
constexpr int kHeadRefs = 8;
struct CtaHead {
    int32_t u_begin, u_end, pad0, pad1;
    Unit first;                    // units[u_begin] (zeros when the range is empty)
    ChunkRef refs[kHeadRefs];      // chunk refs of the first unit's steps 0..kHeadRefs-1
};
static_assert(sizeof(CtaHead) == 128, "one line per CTA");

// Parameters of the attention kernel (passed by value).
struct AttnParams {
    const ChunkRef* chunks;
    const Unit* units;
    const CtaHead* cta_head;     // [grid] first work of each CTA
    const int32_t* seq_perm;     // [b] position -> row of q / out
    const int32_t* pbase;        // [b*H + 1] partial-id CSR per (position, head)
    const int32_t* slot_ntok;    // [capacity] valid tokens per pool slot (device table)
    int32_t* status;             // device status word (CA_ERR_* or 0)
    int32_t* dyn_counter;        // next unit of the shared tail queue (0 between calls)
    int32_t dyn_begin, dyn_end;  // the tail queue: units [dyn_begin, dyn_end)
    const uint16_t* q;           // fp16 [b][H][D]
    uint16_t* out;               // fp16 [b][H][D]
    float* part_o;               // [P][D] unnormalised partial outputs
    float2* part_ms;             // [P] (running max in log2 units, sum of exp2)
    int32_t n_layers, n_heads, layer, capacity;   // n_heads: query heads
    int32_t n_kv_heads, group;                     // key/value heads, n_heads / n_kv_heads
    int32_t q_len, causal;                         // query tokens per position; causal mask
    const int32_t* chunk_tok0;   // [chunks] first token's offset in the context
    const int32_t* ctx_len;      // [b] context tokens of each position
    float scale_log2;            // scale * log2(e) (times the key scale of an fp8 pool)
    float out_scale;             // value scale of an fp8 pool, else 1
    int32_t n_stages;
    int32_t kv_stable;           // no insert/append wrote the pool since the last call
    int32_t test_stall;          // test hook: the producer first waits on a barrier nothing completes
};

// Workspace layout for a schedule.
struct WsLayout {
    size_t part_o, part_ms, total;                  // device-resident inputs
    size_t q_stage, out_stage, total_host;          // + staging for host I/O
};

// ---------------------------------------------------------------------------
// Host objects.
// ---------------------------------------------------------------------------
struct Node {
    int32_t slot = -1;
    int32_t ntok = 0;              // tokens in the chunk (c, or fewer for a tail)
    uint64_t hash = 0;             // full chunks: 64-bit hash of the token tuple
    bool matchable = false;        // full chunk a later insert may match
    Node* parent = nullptr;
    std::vector<Node*> children;   // insertion order (capacity kept when reused)
    // Hash index over the matchable children, built only once a node has many
    // children (a linear scan of the stored hashes is cheaper below that).
    // Should two different sibling tuples ever share a hash, the index keeps
    // the first: sharing is lost for the other, results stay exact.
    std::unique_ptr<std::unordered_map<uint64_t, Node*>> index;
    int32_t refcount = 0;
    int32_t mark = 0;              // scratch for schedule building: batch holders
    int32_t row = -1;              // scratch: chunk-first row while building
    int32_t end_begin = 0;         // scratch: batch sequences ending here, as a
    int32_t end_count = 0;         //   range of the sorted (node, seq_id) list
    int32_t owner = -1;            // scratch: batch row whose private chain starts here
};

struct Sequence {
    std::vector<Node*> path;
    int32_t length = 0;
};

struct Pool {
    PoolCfg cfg{};
    void* kv = nullptr;            // device pool (nullptr: host only)
    size_t kv_bytes = 0;
    int device = -1;
    int num_sms = 0;
    alignas(64) unsigned char tmap[128];  // CUtensorMap over the pool
    Node root;
    std::vector<Node> nodes;       // one per slot, reused; live iff refcount > 0
    std::vector<int32_t> tokens;   // [slot][c] token ids of each live chunk
    std::vector<int32_t> heap;     // min-heap of free slots
    std::unordered_map<int64_t, Sequence> seqs;
    int64_t generation = 0;
    // Set when a KV scatter (insert or append) is launched, cleared when an
    // attention launch reads it: while clear, the pool's device contents are
    // not written by any kernel the next attention call could overlap.
    mutable bool kv_written = true;
    // Stream capture (CUDA graphs): the id of the capture that last recorded
    // an attention call on this pool, and whether a KV scatter was ever
    // recorded into a graph (its replays then write the pool at times the
    // host does not see).
    mutable unsigned long long capture_id = 0;
    mutable bool captured_writes = false;
    // Test hook: allocation points to pass before one fails (-1: none fails).
    mutable int64_t fail_alloc_in = -1;
};

struct Tables {
    int32_t b = 0;
    std::vector<int32_t> seq_perm, cf_rows, cf_runs, sf_offsets, sf_chunks,
        merge_offsets, merge_runs;
    // token offset of each chunk in its sequences' contexts (cf rows, then sf
    // chunks) and each position's context length: the causal mask's inputs
    std::vector<int32_t> row_tok0, sf_tok0, ctx_len;
};

struct Plan {
    std::vector<ChunkRef> chunks;
    std::vector<int32_t> chunk_tok0;   // parallel to chunks: first token's context offset
    int32_t q_len = 1;                 // query tokens per position
    std::vector<Unit> units;       // per-CTA static lists, then the tail queue
    std::vector<int32_t> cta_begin;  // [grid + 1]; cta_begin[grid] = first queue unit
    std::vector<int32_t> pbase;
    int32_t grid = 0;
    int64_t n_partials = 0;
    // scratch kept across rebuilds so that a rebuild allocates nothing new
    std::vector<std::pair<int32_t, Unit>> tagged;   // chunk-first units with their CTA
    std::vector<Unit> sf_scratch, tail_scratch;
    std::vector<int32_t> sf_end;
};

struct Sched {
    const Pool* pool = nullptr;
    int64_t generation = -1;
    uint32_t flags = 0;
    int32_t q_len = 1;
    std::vector<int64_t> seq_ids;
    Tables t;
    Tables t_next;                     // rebuilt into, then swapped with t
    Plan plan;
    PlanLayout layout{};
    WsLayout ws{};
    std::vector<unsigned char> blob;   // host copy of the device plan
    void* dev = nullptr;               // device plan blob
    size_t dev_bytes = 0;
    // Two pinned staging buffers used in turn for the upload, each with an
    // event marking when its last copy finished, so that building the next
    // context never waits for the GPU (only for a copy two builds back).
    void* pinned[2] = {nullptr, nullptr};
    size_t pinned_bytes[2] = {0, 0};
    void* pinned_done[2] = {nullptr, nullptr};   // cudaEvent_t
    int pinned_next = 0;
    void* ev_begin = nullptr;
    void* ev_end = nullptr;
    // Test hooks: the status word of a host-only pool's schedule, and the
    // number of coming decode calls whose producer stalls (every wait then
    // gives up after its limit and the call reports CA_ERR_TIMEOUT).
    mutable int32_t host_status = 0;
    mutable int32_t stall_calls = 0;
};

// One chunk to fill: rows [src_row, src_row + n_rows) of a packed
// [L][total_rows][H][D] source go to rows [dst_row, dst_row + n_rows) of
// `slot`, whose valid-token count becomes dst_row + n_rows.
struct ScatterChunk {
    int32_t src_row, n_rows, slot, dst_row;
};

// Key/value heads of a pool (grouped-query attention; 0 in the config means
// one per query head).
inline int32_t kv_heads(const PoolCfg& c) { return c.n_kv_heads > 0 ? c.n_kv_heads : c.n_heads; }

// Device bytes of the pool: the K/V tiles, then the per-slot token counts.
// Bytes per stored K/V element (fp16, or 1 for an FP8 pool) and the
// effective dequantisation scales.
inline int kv_elem_bytes(const PoolCfg& c) { return (c.flags & CA_KV_FP8) ? 1 : 2; }
inline float kv_scale_of(float s) { return s == 0.f ? 1.f : s; }
// Query rows one tensor-core unit takes: 64, or 32 at head_dim 256.
inline int32_t max_query_rows(const PoolCfg& c) { return c.head_dim == 256 ? 32 : 64; }
size_t pool_tile_bytes(const PoolCfg& c);
size_t pool_total_bytes(const PoolCfg& c);

// What an append changed, so that a failed copy launch can undo it.
struct AppendUndo {
    Node* last = nullptr;
    int32_t ntok = 0;
    bool matchable = false;
    uint64_t hash = 0;
    size_t path_size = 0;
    int64_t generation = 0;
    int32_t length = 0;
};

// pool.cpp
void alloc_point(const Pool& p);
int pool_append(Pool& p, int64_t seq_id, const int32_t* tokens, int32_t n,
                std::vector<ScatterChunk>* copies, AppendUndo* undo);
void pool_undo_append(Pool& p, int64_t seq_id, const AppendUndo& undo);
int pool_insert(Pool& p, int64_t seq_id, const int32_t* tokens, int32_t n,
                std::vector<std::pair<int32_t, int32_t>>* new_chunks,  // (first token, slot)
                int32_t* n_shared);
int pool_remove(Pool& p, int64_t seq_id);
int32_t pool_match(const Pool& p, const int32_t* tokens, int32_t n);

// schedule.cpp
int build_tables(const Pool& p, const int64_t* seq_ids, int32_t b, uint32_t flags, Tables& t);
void build_plan(const Pool& p, const Tables& t, int32_t grid, int32_t q_len, Plan& plan);
void layout_plan(const Plan& plan, int32_t b, PlanLayout& lay, std::vector<unsigned char>& blob,
                 const Tables& t);
void layout_ws(const Plan& plan, const Pool& p, int32_t b, WsLayout& ws);

// kernels.cu
int kernel_smem_bytes(const PoolCfg& c, int* n_stages, size_t* bytes);
int kernel_ctas_per_sm(const PoolCfg& c, int* ctas);
int make_tensor_map(Pool& p);
int launch_scatter(const Pool& p, const void* k, const void* v, int32_t total_rows,
                   const std::vector<ScatterChunk>& chunks, void* stream);
int launch_attention(const Pool& p, const Sched& s, const AttnParams& prm, void* stream);
// Kernel parameters of one call: the schedule's device plan and counters,
// the pool, q / out, and the partial buffers inside `ws_dev`.
AttnParams attn_params(const Pool& pool, const Sched& s, int32_t layer, const void* q, void* out,
                       float scale, void* ws_dev);
// Kernels this process has launched through the library (all pools, all devices).
uint64_t kernel_launches();

}  // namespace ca
