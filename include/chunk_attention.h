/*
 * chunk_attention.h — C ABI of the prefix-shared decode attention library
 * (libchunk_attention.so), a GB300 (sm_103a) implementation of ChunkAttention's
 * decode hot path.
 *
 * Sources: "ChunkAttention: Efficient Self-Attention with Prefix-Aware KV Cache
 * and Two-Phase Partition" (arXiv 2402.15220v4 summary), cited [CA §n], and
 * the explainer "ACL 2024論文解説: ChunkAttention — プレフィックスKVキャッシュ共有
 * によるマルチテナント推論高速化", cited [CA-blog, <section>].
 *
 * Model of the problem [CA §2.2, §3.1]: requests join with a prompt whose
 * keys/values came from prefill, decode one token per step under iteration
 * batching, and leave when done.  Their K/V live in fixed-size chunks that form
 * a prefix tree; a chunk is stored once however many sequences share it.  Each
 * decode step runs attention for the whole batch in two phases [CA §3.2]:
 * chunk-first (every chunk shared by >= 2 batch sequences, against the batched
 * queries of its sharers, on tensor cores) and sequence-first (each sequence's
 * own chunks), whose partial results are merged by the log-sum-exp rule
 * [CA-blog, Two-Phase Partition, output-combination equation].
 *
 * Conventions
 *  - Every call returns an int status: CA_OK (0) or a negative CA_ERR_* code.
 *    No C++ exception crosses this boundary and nothing aborts the process.
 *    ca_error_string() names a code.
 *  - Pointers named *_dev are device pointers the caller owns (e.g. torch
 *    tensors); the library never frees them.  Host arrays are read during
 *    the call only.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All device work is enqueued asynchronously on it.
 *  - Objects are not thread-safe: serialise calls on one pool.
 *  - Element type of K, V, Q and out is IEEE fp16; accumulation is fp32.
 *    A pool created with CA_KV_FP8 stores K and V as 8-bit floats (below);
 *    its inputs and outputs stay fp16.
 */
#ifndef CHUNK_ATTENTION_H
#define CHUNK_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define CA_OK                 0
#define CA_ERR_INVALID       -1  /* bad argument, size, alignment or state    */
#define CA_ERR_OOM           -2  /* no free chunk slots; the pool is unchanged */
#define CA_ERR_NOT_FOUND     -3  /* unknown seq_id                             */
#define CA_ERR_EXISTS        -4  /* seq_id already present                     */
#define CA_ERR_STALE         -5  /* schedule built before the tree last changed */
#define CA_ERR_CUDA          -6  /* a CUDA runtime/driver call failed          */
#define CA_ERR_DEVICE_BOUNDS -7  /* a kernel saw a table index out of range    */
#define CA_ERR_TIMEOUT       -8  /* a kernel wait gave up after ~1 s           */
#define CA_ERR_UNSUPPORTED   -9  /* shape the kernels are not built for        */
#define CA_ERR_SCRATCH_LIMIT -10  /* schedule needs more than the library's own
                                     scratch buffer (CA_STATIC_WS_BYTES) holds  */

/* ---- pool flags -------------------------------------------------------- */
/* Never match prefixes: every sequence owns a private chain of chunks.  This
 * is the flat paged-KV layout [CA §5, PagedAttention] used as the control. */
#define CA_NO_SHARING        1u
/* Store K and V as FP8 E4M3 (OCP 8-bit float: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, largest finite 448, no infinities) instead of
 * fp16, halving the pool's bytes and the bytes every decode call reads.
 * Inserted rows are quantised on the device as
 *     code = E4M3(fp32(x) * fp32(1 / scale)),  round to nearest even,
 *     values beyond +-448 saturate to +-448,
 * with scale = k_scale for keys and v_scale for values, and read back as
 * code * scale exactly.  Attention is then the plain definition over those
 * dequantised keys and values.  Needs head_dim 128.  The pages' own kernels
 * keep fp16; this is one of the variants their tuning discussion leaves open
 * [CA §7, Model and Hardware Compatibility]. */
#define CA_KV_FP8            2u

/* ---- schedule flags ---------------------------------------------------- */
/* Treat every chunk as sequence-first even when the batch shares it (no
 * two-phase partition; shared chunks are read once per sharer).  Reproduces
 * the pages' PagedAttn* comparator: physically shared KV without TPP
 * [CA §4.1, Table 3]. */
#define CA_SCHED_NO_TPP      1u
/* Multi-token queries (ca_build_schedule_ex): query token j of a sequence
 * whose context holds n tokens sees only tokens [0, n - q_len + j]. */
#define CA_SCHED_CAUSAL      2u

typedef struct ca_pool  ca_pool;
typedef struct ca_sched ca_sched;

/* Shape of a pool [CA §3.1: K/V tensors cut into chunks of c tokens].
 * head_dim 64, 128 or 256 (256 only with chunks of 16 or 32 tokens and an
 * fp16 pool); chunk 16, 32 or 64 tokens (the paper's kernel default is 64
 * [CA §4.1]); n_layers, n_heads and capacity_slots >= 1.  Other shapes give
 * CA_ERR_UNSUPPORTED, bad counts or unknown flags CA_ERR_INVALID.  A pool
 * made from this struct has one key/value head per query head and (with
 * CA_KV_FP8) scales of 1; ca_pool_config_ex sets those too. */
typedef struct {
    int32_t  n_layers;
    int32_t  n_heads;         /* query heads (q and out)                       */
    int32_t  head_dim;
    int32_t  chunk;           /* c: tokens per chunk                           */
    int32_t  capacity_slots;  /* chunk slots in the device pool                */
    uint32_t flags;           /* CA_NO_SHARING | CA_KV_FP8, or 0               */
} ca_pool_config;

/* ca_pool_config plus the variants the summary's tuning discussion leaves
 * open [CA §7, Model and Hardware Compatibility].  n_kv_heads: key/value
 * heads stored in the pool (grouped-query attention: query head h reads
 * key/value head h / (n_heads / n_kv_heads)); 0 means n_heads; n_heads must
 * be a multiple of it and the group n_heads / n_kv_heads at most 64 (32 at
 * head_dim 256).  k_scale / v_scale: the CA_KV_FP8 scales (0 means 1.0;
 * ignored without CA_KV_FP8). */
typedef struct {
    ca_pool_config base;
    int32_t  n_kv_heads;      /* key/value heads (0: n_heads)                  */
    float    k_scale;         /* CA_KV_FP8 only: key scale (0: 1.0)            */
    float    v_scale;         /* CA_KV_FP8 only: value scale (0: 1.0)          */
} ca_pool_config_ex;

/* Occupancy of a pool (ca_pool_stats).  The storage model of prefix
 * sharing [CA-blog, Prefix-Aware KV Cache: a shared prefix of L_p tokens and
 * N private suffixes of L_s tokens take L_p + N * L_s token slots instead of
 * N * (L_p + L_s)] is what live_slots counts, in chunks. */
typedef struct {
    int64_t live_slots;       /* slots holding a chunk                         */
    int64_t free_slots;
    int64_t refcount_sum;     /* sum over live chunks of their refcount        */
    int64_t live_seqs;
    int64_t generation;       /* bumped by every insert and remove             */
} ca_stats;

/* ---- pool ----------------------------------------------------------------
 * Device layout: the K/V tiles (row-major, fp16 or with CA_KV_FP8 one byte
 * per element, head = key/value head)
 *     kv[slot][layer][K|V][head][c][head_dim]
 * so one chunk of one head is a contiguous c x head_dim tile (16 KiB at
 * c = 64, D = 128 in fp16) that the kernels fetch whole with TMA; then one int32 per
 * slot holding the chunk's valid-token count (the kernels read it, so a
 * decode-time append can grow a partial chunk without a new schedule).
 */

/* Bytes of device memory a pool with this shape needs (for kv_dev).
 * Errors: as ca_pool_create's shape checks; CA_ERR_INVALID if bytes_out is
 * NULL.  [CA §3.1: the chunks live in one preallocated pool.] */
int ca_pool_bytes(const ca_pool_config* cfg, size_t* bytes_out);
int ca_pool_bytes_ex(const ca_pool_config_ex* cfg, size_t* bytes_out);

/* Create a pool over caller-owned device memory kv_dev of kv_bytes >=
 * ca_pool_bytes(cfg); kv_dev must be 1024-byte aligned and must outlive the
 * pool.  kv_dev == NULL creates a host-only pool (trie, allocator and
 * schedule tables work; nothing touches a GPU; decode returns
 * CA_ERR_INVALID).  [CA §3.1: chunked KV tensors in a prefix tree.] */
int ca_pool_create(const ca_pool_config* cfg, void* kv_dev, size_t kv_bytes,
                   ca_pool** pool_out);
/* The same with the grouped-query and fp8 fields (ca_pool_config_ex). */
int ca_pool_create_ex(const ca_pool_config_ex* cfg, void* kv_dev, size_t kv_bytes,
                      ca_pool** pool_out);
int ca_pool_destroy(ca_pool* pool);

/* Leading tokens of tokens[0..n) whose K/V the pool already holds: the
 * longest path of full chunks matching chunk by chunk from the root (a
 * multiple of c; 0 with CA_NO_SHARING).  Lets a caller skip prefill of the
 * matched prefix.  Does not change the pool. [CA-blog, 動的プレフィックス検出] */
int ca_match_prefix(const ca_pool* pool, const int32_t* tokens, int32_t n,
                    int32_t* n_matched_out);

/* Add sequence seq_id with context tokens[0..n), n >= 1 [CA §3.1: new
 * sequences add paths].  Full chunks that match the tree along the path gain a
 * reference; every other chunk (and always the trailing partial chunk) gets a
 * new slot, lowest free index first, and its K/V rows are copied on `stream`
 * from k_dev / v_dev: fp16 [n_layers][n][n_kv_heads][head_dim], contiguous, 16-byte
 * aligned.  Rows of matched tokens are not read (the first inserter's rows are
 * kept).  k_dev/v_dev must be NULL for a host-only pool and non-NULL
 * otherwise.  n_shared_out (may be NULL) receives the matched token count.
 * Errors: CA_ERR_EXISTS, CA_ERR_OOM (not enough free slots), CA_ERR_INVALID;
 * on any error the pool is unchanged. */
int ca_insert_tokens(ca_pool* pool, int64_t seq_id, const int32_t* tokens,
                     int32_t n, const void* k_dev, const void* v_dev,
                     void* stream, int32_t* n_shared_out);

/* Insert several sequences at once (sequences joining in one iteration
 * [CA §2.2]).  Equivalent to ca_insert_tokens for seq_ids[0], seq_ids[1], ...
 * in order (a later sequence may share chunks an earlier one created), but
 * with one call and one KV copy launch per 128 new chunks.
 *   tokens   int32, the n_seqs token lists concatenated; lengths[i] >= 1
 *   k_dev / v_dev  fp16 [n_layers][sum(lengths)][n_kv_heads][head_dim]: the
 *            rows of sequence i start at row lengths[0] + ... + lengths[i-1]
 *            (a packed prefill output); rows of matched tokens are not read
 *   n_shared_out   int32[n_seqs] or NULL
 * All or nothing: on any error (CA_ERR_EXISTS, CA_ERR_OOM, CA_ERR_INVALID,
 * CA_ERR_CUDA) the pool is left exactly as before the call. */
int ca_insert_batch(ca_pool* pool, int32_t n_seqs, const int64_t* seq_ids,
                    const int32_t* tokens, const int32_t* lengths,
                    const void* k_dev, const void* v_dev, void* stream,
                    int32_t* n_shared_out);

/* Append decoded tokens to a live sequence [CA §3.1: decoding appends tokens
 * to leaf chunks or grows new chunks].  The tokens first fill the sequence's
 * partial last chunk in place, then grow new private chunks (lowest free
 * slots first); an append never matches existing chunks.  A chunk that
 * becomes full becomes shareable by later inserts (unless its parent already
 * holds an equal one).  k_dev / v_dev: fp16 [n_layers][n][n_kv_heads][head_dim]
 * for the n appended tokens.  Filling the partial chunk does not change the
 * tree's structure, so schedules stay valid (their exported ntok values are
 * as of their build; the kernels read current counts from the pool); growing
 * a chunk bumps the generation (schedules go stale), as the pages' "a full
 * chunk triggers a context copy" [CA §3.3].  n_new_chunks_out (may be NULL)
 * receives the number of chunks grown.  Errors: CA_ERR_NOT_FOUND, CA_ERR_OOM,
 * CA_ERR_INVALID, CA_ERR_CUDA; on error the pool is unchanged. */
int ca_append_tokens(ca_pool* pool, int64_t seq_id, const int32_t* tokens,
                     int32_t n, const void* k_dev, const void* v_dev,
                     void* stream, int32_t* n_new_chunks_out);

/* Remove a finished sequence [CA §3.1: completed sequences remove their
 * path].  Every chunk on its path loses one reference; chunks left with none
 * return their slot to the free list [CA-blog, 動的プレフィックス検出]. */
int ca_remove_seq(ca_pool* pool, int64_t seq_id);

/* Remove n_seqs sequences; CA_ERR_NOT_FOUND (nothing removed) if any id is
 * unknown, CA_ERR_INVALID if an id repeats. */
int ca_remove_batch(ca_pool* pool, int32_t n_seqs, const int64_t* seq_ids);

/* Occupancy counters (ca_stats above); host only, never touches the GPU.
 * CA_ERR_INVALID on NULL arguments. */
int ca_pool_stats(const ca_pool* pool, ca_stats* out);

/* Slots along seq_id's path, root first (test and inspection helper).
 * Writes min(cap, path length) entries; *n_out = path length. */
int ca_seq_slots(const ca_pool* pool, int64_t seq_id, int32_t* slots, int32_t cap,
                 int32_t* n_out);

/* ---- schedule -------------------------------------------------------------
 * The per-step context of the two-phase kernel [CA §3.2, §3.3] for the batch
 * seq_ids[0..b): which chunks are chunk-first and which sequences share each
 * (one contiguous range of a depth-first batch order), each sequence's
 * sequence-first chunks, and the merge lists; plus the kernels' work plan.
 * *inout == NULL allocates a schedule; otherwise it is reused, and when the
 * pool has not changed since it was built and the batch is identical it is
 * returned untouched (the pages: context copies are cached until the tree
 * changes [CA §3.3]).  Tables are copied to a library-owned device buffer
 * with cudaMemcpyAsync on `stream` (none for a host-only pool).
 * Errors: CA_ERR_NOT_FOUND (unknown seq_id), CA_ERR_INVALID (b < 1, duplicate
 * ids), CA_ERR_CUDA. */
int ca_build_schedule(ca_pool* pool, const int64_t* seq_ids, int32_t b,
                      ca_sched** inout, void* stream);

/* The same with flags (CA_SCHED_NO_TPP, CA_SCHED_CAUSAL; 0 is
 * ca_build_schedule) and q_len query tokens per sequence (multi-token queries: draft
 * tokens to verify, or a chunk of prompt prefilled over the trie).  The
 * blog's two-phase function takes queries of any length [CA-blog, Two-Phase
 * Partition: queries (batch, heads, seq_len, d_k)] and lets every query
 * token attend to the sequence's whole context; that is the default here.
 * With CA_SCHED_CAUSAL, query token j of a sequence whose context holds n
 * tokens attends to tokens [0, n - q_len + j] only — the form for tokens
 * whose own K/V the caller has already appended.  q and out of the decode
 * calls are then [b][q_len][n_heads][head_dim] (row i*q_len + j is token j
 * of seq_ids[i]).  q_len = 1 with flags 0 is ca_build_schedule.  Requires
 * q_len * (n_heads / n_kv_heads) <= 64 (CA_ERR_UNSUPPORTED otherwise) and,
 * with CA_SCHED_CAUSAL, every context at least q_len tokens long
 * (CA_ERR_INVALID otherwise); other errors as ca_build_schedule. */
int ca_build_schedule_ex(ca_pool* pool, const int64_t* seq_ids, int32_t b, int32_t q_len,
                         uint32_t flags, ca_sched** inout, void* stream);
int ca_sched_destroy(ca_sched* sched);

/* Table sizes, then the tables themselves (host copies; for bit-exact tests).
 * These are the per-step context the pages describe [CA §3.2: which chunks
 * the chunk-first phase takes and for which range of sequences; CA §3.3:
 * the context is kept until the tree changes], exported as built.
 * counts[0..5] = b, R (chunk-first rows), U (runs), S (sequence-first
 * chunks), M (merge entries), n_units (kernel work units). */
int ca_sched_counts(const ca_sched* sched, int32_t counts[6]);
/* Any pointer may be NULL to skip that table.  Layouts (int32):
 *   seq_perm[b]           DFS position -> row of Q / out (index into seq_ids)
 *   cf_rows[R][4]         (slot, ntok, lo, hi), DFS pre-order
 *   cf_runs[U][4]         (row0, nrows, lo, hi)
 *   sf_offsets[b+1], sf_chunks[S][2] (slot, ntok)
 *   merge_offsets[b+1], merge_runs[M] */
int ca_export_tables(const ca_sched* sched, int32_t* seq_perm, int32_t* cf_rows,
                     int32_t* cf_runs, int32_t* sf_offsets, int32_t* sf_chunks,
                     int32_t* merge_offsets, int32_t* merge_runs);

/* The kernel work plan derived from the tables (inspection and tests).
 * counts[0..3] = n_units, grid (CTAs), n_pbase (= b * q_len * n_heads + 1),
 * n_chunks.  Any array may be NULL.  Layouts (int32):
 *   units[n_units][12] (kind, head, pos_lo, pos_hi, begin, end, part, qrow,
 *                       n_per_head, base, part_next, 0).  Chunk-first (kind 0):
 *                       chunks [begin, end) of the list for the heads
 *                       [head, head + n_per_head) and positions
 *                       [pos_lo, pos_hi).  Sequence-first (kind 1):
 *                       position pos_lo's (head, chunk) pairs with linear
 *                       index h * n_per_head + j in [begin, end), chunk j at
 *                       list index base + j; its first head uses partial
 *                       index `part`, later heads `part_next`.
 *   cta_begin[grid+1]  static unit range of each CTA; units from
 *                      cta_begin[grid] to n_units form the tail queue that
 *                      CTAs drain dynamically after their static ranges
 *   pbase[n_pbase]     partial ids of (position p, query token j, head h)
 *                      are [pbase[i], pbase[i+1]) with i = (p*q_len+j)*H+h
 *   chunks[n_chunks][2] (slot, ntok) list the units index into */
int ca_export_plan(const ca_sched* sched, int32_t counts[4], int32_t* units,
                   int32_t* cta_begin, int32_t* pbase, int32_t* chunks);

/* Bytes of caller-owned device workspace ca_decode_attention needs for this
 * schedule: one partial triple (o: head_dim fp32, m, s: fp32) per piece of
 * work and (sequence, query token, head) it covers — the per-phase partial
 * results that the output-combination rule merges [CA-blog, Two-Phase
 * Partition; CA §3.2].  CA_ERR_INVALID on NULL arguments. */
int ca_workspace_bytes(const ca_sched* sched, size_t* bytes_out);

/* ---- decode attention -----------------------------------------------------
 * out[i][h][:] = sum_t softmax_t(scale * q[i][h] . k_t) v_t over every token
 * t of sequence seq_ids[i]'s context, computed by the two-phase partition
 * [CA §3.2; CA-blog, Two-Phase Partition].
 *   q_dev    fp16 [b][n_heads][head_dim], row i = seq_ids[i] of the schedule
 *            ([b][q_len][n_heads][head_dim] for a ca_build_schedule_ex
 *            schedule, masked as that call says)
 *   out_dev  same shape as q, written
 *   layer    0 <= layer < n_layers
 *   ws_dev   >= ca_workspace_bytes(sched) bytes, 256-byte aligned, caller
 *            owned; its contents need no initialisation.  Calls sharing one
 *            workspace or one schedule must not overlap on the GPU (the
 *            schedule holds the kernels' work-queue counter).
 * Two kernels run on `stream`: the two-phase kernel and a merge kernel
 * launched as its programmatic dependent (one warp per sequence and head).
 * Both are programmatic dependents of the work before them on `stream`: they
 * read q, the workspace and the queue counter only once that work has
 * completed.  The two-phase kernel starts streaming the pool before then
 * when no insert or append on this pool was launched since its last
 * attention call, so the pool's device memory must be written only through
 * this library's calls.
 * Stream capture (CUDA graphs): the call may be recorded into a graph
 * (cudaStreamBeginCapture or torch.cuda.graph on `stream`), with q_dev,
 * out_dev and ws_dev fixed at capture; the two kernels keep their
 * programmatic dependencies inside the graph.  The first call a capture
 * records for a pool does not stream the pool before its dependency wait,
 * since at replay anything may precede it.  Once an insert or append has
 * been recorded into a graph, uncaptured calls on that pool no longer do
 * either (the host cannot see when those replays write the pool).  A graph
 * stays valid while its schedule is unchanged: appends that fit the
 * sequences' partial last chunks keep it (the kernels read each chunk's
 * token count from the pool); anything that rebuilds the schedule (a grown
 * chunk, an insert or remove, another batch) needs a new capture.  Build
 * schedules outside capture (ca_build_schedule allocates).
 * Errors: CA_ERR_STALE if the pool changed after the schedule was built;
 * CA_ERR_INVALID for a host-only pool, bad layer, NULL or misaligned pointers
 * or a small workspace; CA_ERR_CUDA if a launch fails or `stream`'s capture
 * was invalidated.  Kernel-side faults
 * (an index out of range, a wait that timed out) are reported by
 * ca_sched_device_status(). */
int ca_decode_attention(const ca_pool* pool, const ca_sched* sched, int32_t layer,
                        const void* q_dev, void* out_dev, float scale,
                        void* ws_dev, size_t ws_bytes, void* stream);

/* The same computation with q and out in HOST memory, all on `stream`; the
 * caller synchronises.  When both buffers are pinned memory with a device
 * mapping (cudaHostGetDevicePointer succeeds, as for cudaHostAlloc memory
 * under unified addressing), the kernels read q from and the merge writes out
 * to host memory directly (NVLink-C2C on GB300) and no copy is issued;
 * otherwise q is copied in and out copied back through device staging.
 * Either way ws_dev needs ca_workspace_bytes_host(sched) bytes (the staging
 * for q and out lives at its end). */
int ca_workspace_bytes_host(const ca_sched* sched, size_t* bytes_out);
int ca_decode_attention_host(const ca_pool* pool, const ca_sched* sched,
                             int32_t layer, const void* q_host, void* out_host,
                             float scale, void* ws_dev, size_t ws_bytes,
                             void* stream);

/* ca_decode_attention for callers that cannot allocate device memory at the
 * point of the call (a component inside a server that has already reserved
 * the whole device memory budget for its own pool, a latency-critical path
 * where cudaMalloc / cudaFree would synchronise the device, a plugin whose
 * host forbids allocation in its callbacks).  There is no workspace
 * argument: the partial results go to a fixed buffer the library holds in
 * device memory, CA_STATIC_WS_BYTES bytes per GPU that loads the library,
 * kept until the process exits.  The call allocates nothing; the caller
 * still passes q_dev and out_dev as for ca_decode_attention.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress); make that first call outside any stream
 *     capture.  The pool's device must be current.  The address is kept
 *     for the life of the process, so resetting a device (cudaDeviceReset)
 *     after its first call is not supported.
 *   - Every call shares the one buffer: calls that overlap on the GPU
 *     (other streams, other host threads) race and corrupt each other's
 *     results.  Nothing in the buffer needs clearing between calls.
 *   - A schedule whose ca_workspace_bytes() exceeds CA_STATIC_WS_BYTES is
 *     rejected with CA_ERR_SCRATCH_LIMIT; other errors as ca_decode_attention.
 * The pages describe no such call; it exists for callers of this library. */
#define CA_STATIC_WS_BYTES (16u << 20)
int ca_decode_attention_static_ws(const ca_pool* pool, const ca_sched* sched,
                                  int32_t layer, const void* q_dev, void* out_dev,
                                  float scale, void* stream);

/* Synchronise `stream` and read the schedule's device status word: CA_OK,
 * CA_ERR_DEVICE_BOUNDS or CA_ERR_TIMEOUT (or a code written by
 * ca_sched_inject_status); a non-zero word is then cleared, together with
 * the tail-queue counter a call that stopped early may have left behind.
 * For a host-only pool's schedule: its host word (0 unless injected). */
int ca_sched_device_status(const ca_sched* sched, void* stream);

/* ---- failure injection (tests) ---------------------------------------------
 * The pages have no counterpart: these let the library's own tests exercise
 * its failure paths without faulting or hanging a GPU.
 *
 * ca_sched_inject_status: write `code` (a CA_ERR_* value, negative) into the
 * schedule's status word, as a kernel that saw a bad index or gave up a wait
 * would; the next ca_sched_device_status() returns it and clears it.  For a
 * device pool the word is written on `stream` and the call synchronises it;
 * a host-only pool's schedule keeps a host word (ca_sched_device_status then
 * reads that one).  CA_ERR_INVALID for a non-negative or unknown code.
 *
 * ca_sched_inject_stall: the next n_calls decode calls on this schedule run
 * with their producer warps first waiting for a barrier phase that nothing
 * completes.  No copy is issued; that wait and the consumers' first waits
 * give up after their limit (~1 s), the call's results are undefined and
 * ca_sched_device_status() returns CA_ERR_TIMEOUT.  Later calls run normally.
 *
 * ca_pool_inject_alloc_failure: the host allocation points of the coming
 * inserts and appends pass after_n times, then one fails as if the host were
 * out of memory; that call returns CA_ERR_OOM and leaves the pool exactly as
 * it was before the call.  after_n < 0 turns the failure off. */
int ca_sched_inject_status(ca_sched* sched, int32_t code, void* stream);
int ca_sched_inject_stall(ca_sched* sched, int32_t n_calls);
int ca_pool_inject_alloc_failure(ca_pool* pool, int32_t after_n);

/* Optional timing hook: when both are non-NULL, ca_decode_attention records
 * event_begin (a cudaEvent_t) just before its main kernel and event_end just
 * after it, on `stream`.  Pass NULLs to turn it off. */
int ca_sched_set_profile_events(ca_sched* sched, void* event_begin, void* event_end);

/* Number of kernels the library has launched in this process so far (KV
 * scatters, attention and merge kernels; every pool and device), counted
 * when each launch is accepted.  A caller reads it before and after a run
 * of calls to learn how many GPU kernels they issued.  Instrumentation
 * only: the pages have no counterpart.  CA_ERR_INVALID if count_out is
 * NULL. */
int ca_kernel_launches(uint64_t* count_out);

/* A static, human-readable name for a status code ("unknown status" for
 * codes this header does not define); never NULL.  The pages have no
 * counterpart: it only serves callers of this library. */
const char* ca_error_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* CHUNK_ATTENTION_H */
