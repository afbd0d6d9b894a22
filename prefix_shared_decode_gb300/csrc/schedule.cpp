// Per-step context of the two-phase partition ("ChunkAttention: Efficient
// Self-Attention with Prefix-Aware KV Cache and Two-Phase Partition", §3.2
// and §3.3) and the kernel work plan derived from it.
//
// Tables (the exact, testable part):
//  * depth-first batch order: children in insertion order; at a node, the
//    sequences ending there first (ascending seq_id), then its children — so
//    every chunk's sharers are one contiguous range [lo, hi) of positions;
//  * cf_rows: chunks held by >= 2 batch sequences, pre-order, with [lo, hi);
//  * cf_runs: maximal parent->child stretches of rows with the same range;
//  * sf lists: each position's chunks held by that sequence alone;
//  * merge lists: the runs covering each position.
//
// Plan (GB300-specific, verified through the outputs): chunk-first runs are
// cut into units of at most 64 query rows (32 at head_dim 256, and in small
// calls whose positions bring several rows each) and a balanced
// number of chunks; sequence-first chunk-heads are spread over the CTAs in
// contiguous pieces so that every CTA gets the same estimated time, with a
// tail of small units that CTAs claim dynamically.
#include <algorithm>
#include <cstring>
#include <numeric>

#include "ca_internal.h"

namespace ca {

int build_tables(const Pool& p, const int64_t* seq_ids, int32_t b, uint32_t flags, Tables& t) {
    if (b < 1 || !seq_ids) return CA_ERR_INVALID;
    std::vector<const Sequence*> seq_of(b);
    for (int32_t i = 0; i < b; ++i) {
        auto it = p.seqs.find(seq_ids[i]);
        if (it == p.seqs.end()) return CA_ERR_NOT_FOUND;
        seq_of[i] = &it->second;
    }
    // (end node, seq_id, caller row): sorted, so that the sequences ending at
    // one node are adjacent and in ascending seq_id (ids must be distinct).
    struct End { const Node* node; int64_t id; int32_t row; };
    std::vector<End> ends(b);
    for (int32_t i = 0; i < b; ++i) ends[i] = {seq_of[i]->path.back(), seq_ids[i], i};
    std::sort(ends.begin(), ends.end(), [](const End& x, const End& y) {
        return x.node != y.node ? std::less<const Node*>()(x.node, y.node) : x.id < y.id;
    });
    // a repeated id has one path, so its copies sit side by side here
    for (int32_t i = 1; i < b; ++i)
        if (ends[i].node == ends[i - 1].node && ends[i].id == ends[i - 1].id) return CA_ERR_INVALID;
    const bool tpp = !(flags & CA_SCHED_NO_TPP);
    // Batch holders per node.  When the batch is every live sequence (the
    // usual decode step) they are the chunks' refcounts; otherwise each
    // batch path is marked (Node::mark).
    const bool all_live = (size_t)b == p.seqs.size();
    auto holders = [all_live](const Node* n) { return all_live ? n->refcount : n->mark; };
    if (!all_live)
        for (int32_t i = 0; i < b; ++i)
            for (Node* n : seq_of[i]->path) n->mark += 1;
    for (int32_t i = 0; i < b;) {
        int32_t j = i;
        while (j < b && ends[j].node == ends[i].node) ++j;
        Node* n = const_cast<Node*>(ends[i].node);
        n->end_begin = i;
        n->end_count = j - i;
        i = j;
    }
    // Each batch sequence's private chain: the suffix of its path held by it
    // alone.  Holders never grow along a path, so its first node (the chain
    // head) is found by bisection; the head records its sequence.
    std::vector<int32_t> chain_at(b);
    for (int32_t i = 0; i < b; ++i) {
        const auto& path = seq_of[i]->path;
        size_t lo = 0, hi = path.size();
        while (lo < hi) {
            const size_t mid = (lo + hi) / 2;
            if (holders(path[mid]) >= 2) lo = mid + 1;
            else hi = mid;
        }
        chain_at[i] = (int32_t)lo;
        if (lo < path.size()) path[lo]->owner = i;
    }

    t.b = b;
    for (auto* v : {&t.seq_perm, &t.cf_rows, &t.cf_runs, &t.sf_offsets, &t.sf_chunks, &t.merge_offsets,
                    &t.merge_runs, &t.row_tok0, &t.sf_tok0, &t.ctx_len})
        v->clear();
    const int32_t c = p.cfg.chunk;
    // Depth-first order over the shared nodes only: at a node, the sequences
    // ending there, then its children in insertion order; a child held by
    // one batch sequence is that sequence's chain, which contributes exactly
    // that sequence and no chunk-first row.
    std::vector<int32_t>& order = t.seq_perm;     // DFS position -> caller row
    order.reserve(b);
    std::vector<const Node*> row_node;
    struct Frame { const Node* node; size_t next; };
    std::vector<Frame> stack;
    stack.push_back({&p.root, 0});
    while (!stack.empty()) {
        Frame& f = stack.back();
        const Node* node = f.node;
        if (f.next == 0 && node != &p.root) {
            if (tpp) {
                const_cast<Node*>(node)->row = (int32_t)row_node.size();
                row_node.push_back(node);
                t.cf_rows.insert(t.cf_rows.end(), {node->slot, node->ntok, (int32_t)order.size(), -1});
                t.row_tok0.push_back((int32_t)(stack.size() - 2) * c);   // path index x c
            }
            for (int32_t k = 0; k < node->end_count; ++k) order.push_back(ends[node->end_begin + k].row);
        }
        const auto& ch = node->children;
        size_t ci = f.next;
        for (; ci < ch.size(); ++ci) {
            const int32_t hc = holders(ch[ci]);
            if (hc >= 2) break;
            if (hc == 1) order.push_back(ch[ci]->owner);
        }
        if (ci < ch.size()) {
            f.next = ci + 1;
            stack.push_back({ch[ci], 0});
        } else {
            if (node->row >= 0) t.cf_rows[4 * node->row + 3] = (int32_t)order.size();
            stack.pop_back();
        }
    }

    // Runs.
    const int32_t R = (int32_t)row_node.size();
    for (int32_t r = 0; r < R; ++r) {
        const int32_t lo = t.cf_rows[4 * r + 2], hi = t.cf_rows[4 * r + 3];
        const size_t U = t.cf_runs.size() / 4;
        if (U > 0 && row_node[r]->parent == row_node[r - 1] && t.cf_rows[4 * (r - 1) + 2] == lo &&
            t.cf_rows[4 * (r - 1) + 3] == hi) {
            t.cf_runs[4 * (U - 1) + 1] += 1;
        } else {
            t.cf_runs.insert(t.cf_runs.end(), {r, 1, lo, hi});
        }
    }

    // Sequence-first lists: each position's private chain (its whole path
    // without the partition).
    t.sf_offsets.resize((size_t)b + 1);
    t.sf_offsets[0] = 0;
    for (int32_t pos = 0; pos < b; ++pos) {
        const int32_t i = order[pos];
        const size_t k = tpp ? (size_t)chain_at[i] : 0;
        t.sf_offsets[pos + 1] = t.sf_offsets[pos] + (int32_t)(seq_of[i]->path.size() - k);
    }
    t.sf_chunks.resize(2 * (size_t)t.sf_offsets[b]);
    t.sf_tok0.resize((size_t)t.sf_offsets[b]);
    t.ctx_len.resize(b);
    for (int32_t pos = 0; pos < b; ++pos) {
        const int32_t i = order[pos];
        const auto& path = seq_of[i]->path;
        int32_t* dst = t.sf_chunks.data() + 2 * (size_t)t.sf_offsets[pos];
        int32_t* tok0 = t.sf_tok0.data() + t.sf_offsets[pos];
        for (size_t k = tpp ? (size_t)chain_at[i] : 0; k < path.size(); ++k) {
            *dst++ = path[k]->slot;
            *dst++ = path[k]->ntok;
            *tok0++ = (int32_t)k * c;        // every chunk before the last is full
        }
        t.ctx_len[pos] = seq_of[i]->length;
    }

    // Merge lists: runs are nested intervals listed in pre-order, so a
    // position's covering runs come out in root-to-leaf order.
    t.merge_offsets.assign(1, 0);
    const int32_t U = (int32_t)(t.cf_runs.size() / 4);
    for (int32_t pos = 0; pos < b; ++pos) {
        for (int32_t u = 0; u < U; ++u)
            if (t.cf_runs[4 * u + 2] <= pos && pos < t.cf_runs[4 * u + 3]) t.merge_runs.push_back(u);
        t.merge_offsets.push_back((int32_t)t.merge_runs.size());
    }

    for (int32_t i = 0; i < b; ++i) {
        if (!all_live)
            for (Node* n : seq_of[i]->path) n->mark = 0;
        Node* e = seq_of[i]->path.back();
        e->end_begin = e->end_count = 0;
    }
    for (const Node* n : row_node) const_cast<Node*>(n)->row = -1;
    return CA_OK;
}

// ---------------------------------------------------------------------------
// Work plan.
// Cost model, in "chunk-head tiles" (one chunk of one head, K and V): a
// sequence-first tile of one query row costs 1 (HBM-bound); a tile on the
// tensor cores for m query rows costs 1 + kCfComputePer16 * ceil(m / 16)
// (tensor-core work grows with m), relative to the sequence-first tiles'
// own cost; the coefficients are fitted to traced unit times on GB300.
// ---------------------------------------------------------------------------
namespace {
constexpr double kCfComputePer16 = 0.2;
// fp8 pools: a chunk-first tile against a single-row sequence-first one
// (both on the tensor cores straight from the E4M3 bytes; the chunk-first
// tile carries m query rows of work on half the bytes of an fp16 tile);
// swept on GB300 (1.5 .. 2.8) for the fastest calls
constexpr double kF8CfFactor = 2.0;

// Share of the sequence-first tiles left to the tail queue that CTAs drain
// dynamically once their static lists are done (absorbs the run-to-run rate
// differences between SMs), and the size of a queued unit in chunk-heads.
constexpr double kTailShare = 0.12;
constexpr int32_t kTailUnitsPerCta = 2;     // aim: about this many queue units per CTA
// At least four chunk-heads per queued unit: every unit pays a fixed cost
// (its claim, query load, partial writes and one more partial to merge),
// which two-tile units did not amortise (measured: 2% slower calls).
constexpr int32_t kTailUnitMin = 4, kTailUnitMax = 8;
// Below this many tiles per CTA, positions with several query rows take
// chunk-first groups of at most 32 rows (measured on GB300: a grouped-query
// call of ~8 tiles per CTA 21.5 -> 19.3 us; a multi-token call of ~32 tiles
// per CTA was 1% slower with them).
constexpr double kSmallCallTiles = 16.0;
}  // namespace

void build_plan(const Pool& p, const Tables& t, int32_t grid, int32_t q_len, Plan& plan) {
    // Work is per key/value head (H of them); partials are per query token
    // and query head (HQ = H * G; G = 1 is multi-head attention).  Each
    // position brings RW = q_len * G query rows per key/value head; with
    // RW > 1 a sequence-first chunk-head multiplies them on tensor cores.
    const int32_t HQ = p.cfg.n_heads, H = kv_heads(p.cfg), G = HQ / H, RW = q_len * G;
    const int32_t D = p.cfg.head_dim, c = p.cfg.chunk, b = t.b;
    plan.q_len = q_len;
    const double sf_cost = (RW == 1) ? 1.0 : 1.0 + kCfComputePer16 * ((RW + 15) / 16);
    // An fp8 pool halves a tile's bytes while the chunk-first tensor work per
    // tile stays the same, so against single-row sequence-first tiles (and
    // only there) a chunk-first tile costs more.
    const double cf_mult = ((p.cfg.flags & CA_KV_FP8) && RW == 1) ? kF8CfFactor : 1.0;
    auto rows_cost = [&](int32_t m_rows) {
        return cf_mult * (1.0 + kCfComputePer16 * ((m_rows + 15) / 16)) / sf_cost;
    };
    const int32_t R = (int32_t)(t.cf_rows.size() / 4), U = (int32_t)(t.cf_runs.size() / 4);
    plan.chunks.clear();
    plan.units.clear();
    plan.cta_begin.clear();
    plan.pbase.clear();
    plan.n_partials = 0;

    // Chunk list: chunk-first rows first (index = row), then sf chunks.
    plan.chunks.resize(R + t.sf_chunks.size() / 2);
    plan.chunk_tok0.resize(plan.chunks.size());
    for (int32_t r = 0; r < R; ++r) {
        plan.chunks[r] = {t.cf_rows[4 * r], t.cf_rows[4 * r + 1]};
        plan.chunk_tok0[r] = t.row_tok0[r];
    }
    for (size_t i = 0; i < t.sf_chunks.size() / 2; ++i) {
        plan.chunks[R + i] = {t.sf_chunks[2 * i], t.sf_chunks[2 * i + 1]};
        plan.chunk_tok0[R + i] = t.sf_tok0[i];
    }

    // Totals for the per-CTA budget.  Chunk-first query groups take at most
    // max_query_rows rows; when positions bring several rows each (RW > 1)
    // and the call is small (under kSmallCallTiles tiles per CTA), groups of
    // at most 32 rows instead: twice the units, so the CTAs holding the
    // chunk-first work no longer finish long after the rest.
    const double sf_total = (double)(t.sf_chunks.size() / 2) * H;
    int32_t group_rows = max_query_rows(p.cfg);
    auto cf_cost_total = [&] {
        double total = 0;
        for (int32_t u = 0; u < U; ++u) {
            const int32_t nrows = t.cf_runs[4 * u + 1], m = t.cf_runs[4 * u + 3] - t.cf_runs[4 * u + 2];
            const int32_t max_pos = std::max(1, group_rows / RW);
            const int32_t ngroups = (m + max_pos - 1) / max_pos;
            total += (double)nrows * H * ngroups * rows_cost((m + ngroups - 1) / ngroups * RW);
        }
        return total;
    };
    double cf_total = cf_cost_total();
    // a small call whose positions bring several rows each
    const bool small_multi_row = RW > 1 && (sf_total + cf_total) < kSmallCallTiles * grid;
    if (small_multi_row && group_rows > 32) {
        group_rows = 32;
        cf_total = cf_cost_total();
    }
    const int32_t tiles_ceiling = (int32_t)std::max(1.0, sf_total + cf_total);
    grid = std::max(1, std::min(grid, tiles_ceiling));
    plan.grid = grid;
    const int64_t tail_tiles = (int64_t)(kTailShare * sf_total);
    const double sf_static = sf_total - (double)tail_tiles;
    const double avg = (sf_static + cf_total) / grid;

    // Chunk-first units: pieces per run.
    std::vector<int32_t> pieces(U, 0);
    struct CfUnit { Unit u; double cost; };
    std::vector<CfUnit> cf;
    cf.reserve((size_t)U * 8);
    for (int32_t u = 0; u < U; ++u) {
        const int32_t row0 = t.cf_runs[4 * u], nrows = t.cf_runs[4 * u + 1];
        const int32_t lo = t.cf_runs[4 * u + 2], hi = t.cf_runs[4 * u + 3], m = hi - lo;
        // query groups of at most group_rows (position, query token, query head) rows
        const int32_t max_pos = std::max(1, group_rows / RW);
        const int32_t ngroups = (m + max_pos - 1) / max_pos;
        const int32_t mg = (m + ngroups - 1) / ngroups;
        const double row_cost = rows_cost(mg * RW);
        // Enough rows per piece that partial traffic (2 x mg x G x (D+2)
        // floats) stays under 1/8 of the piece's KV bytes, but never so many
        // that one piece outweighs a CTA's share by more than a quarter: the
        // longest unit bounds the kernel, while extra partials are spread
        // over every CTA and the merge.
        const int32_t rmin = std::max(1, (int32_t)((16.0 * mg * RW * (D + 2)) / ((double)c * D) + 0.999));
        const int32_t rpar = std::max(1, (int32_t)(avg / row_cost));
        const int32_t rcap = std::max(1, (int32_t)(1.25 * avg / row_cost));
        const int32_t per = std::max(rpar, std::min(rmin, rcap));
        const int32_t np = std::max(1, (nrows + per - 1) / per);
        pieces[u] = np;
        for (int32_t g = 0; g < ngroups; ++g) {
            const int32_t qa = lo + (int32_t)((int64_t)m * g / ngroups);
            const int32_t qb = lo + (int32_t)((int64_t)m * (g + 1) / ngroups);
            for (int32_t k = 0; k < np; ++k) {
                const int32_t ra = row0 + (int32_t)((int64_t)nrows * k / np);
                const int32_t rb = row0 + (int32_t)((int64_t)nrows * (k + 1) / np);
                // A unit covers a range of heads (the kernel reloads the query
                // tile per head), as many as keep it within a CTA's share.
                const double head_cost = (rb - ra) * rows_cost((qb - qa) * RW);
                const int32_t hp = std::max(1, std::min(H, (int32_t)(avg / head_cost)));
                const int32_t nparts = (H + hp - 1) / hp;
                for (int32_t hk = 0; hk < nparts; ++hk) {
                    const int32_t h0 = (int32_t)((int64_t)H * hk / nparts);
                    const int32_t h1 = (int32_t)((int64_t)H * (hk + 1) / nparts);
                    Unit x{UNIT_CF, h0, qa, qb, ra, rb, k, 0, h1 - h0, 0, 0, 0};
                    cf.push_back({x, (h1 - h0) * head_cost});
                }
            }
        }
    }
    // Partial index base of a run for its positions: the pieces of the runs
    // before it on the same path (its ancestors), which are exactly the runs
    // preceding it in any covered position's merge list.
    std::vector<int32_t> run_base(U, 0);
    std::vector<int32_t> nk1(b, 0);
    for (int32_t pos = 0; pos < b; ++pos) {
        int32_t acc = 0;
        for (int32_t k = t.merge_offsets[pos]; k < t.merge_offsets[pos + 1]; ++k) {
            const int32_t u = t.merge_runs[k];
            run_base[u] = acc;       // identical for every position the run covers
            acc += pieces[u];
        }
        nk1[pos] = acc;
    }
    // The base depends on the unit's run: recover it from the row range.
    {
        std::vector<int32_t> run_of_row(R);
        for (int32_t u = 0; u < U; ++u)
            for (int32_t r = t.cf_runs[4 * u]; r < t.cf_runs[4 * u] + t.cf_runs[4 * u + 1]; ++r)
                run_of_row[r] = u;
        for (auto& x : cf) x.u.part = run_base[run_of_row[x.u.c_begin]] + x.u.part;
    }

    // LPT: biggest chunk-first units first, each onto the least-loaded CTA.
    // Each CTA's list is its chunk-first units (in assignment order), then
    // its sequence-first pieces (in list order); the tail queue follows.
    std::vector<std::pair<int32_t, Unit>>& cf_at = plan.tagged;    // (CTA, unit)
    cf_at.clear();
    cf_at.reserve(cf.size());
    std::vector<double> load(grid, 0.0);
    {
        // Costs in 1/64 tile units; the heap key packs (load, CTA) into one
        // integer so that ties go to the lowest CTA index (deterministic).
        std::vector<int32_t> order(cf.size());
        std::vector<int64_t> icost(cf.size());
        for (size_t i = 0; i < cf.size(); ++i) {
            order[i] = (int32_t)i;
            icost[i] = (int64_t)(cf[i].cost * 64.0 + 0.5);
        }
        std::sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
            return icost[x] != icost[y] ? icost[x] > icost[y] : x < y;
        });
        std::vector<int64_t> heap(grid);
        for (int32_t k = 0; k < grid; ++k) heap[k] = k;           // load 0
        auto greater = [](int64_t x, int64_t y) { return x > y; };
        std::make_heap(heap.begin(), heap.end(), greater);
        for (int32_t i : order) {
            std::pop_heap(heap.begin(), heap.end(), greater);
            const int64_t top = heap.back();
            const int32_t k = (int32_t)(top & 0xfffff);
            const int64_t l = (top >> 20) + icost[i];
            cf_at.emplace_back(k, cf[i].u);
            load[k] = l / 64.0;
            heap.back() = (l << 20) | k;
            std::push_heap(heap.begin(), heap.end(), greater);
        }
    }

    // Sequence-first pieces.  Position p's work is its n_p own chunks for each
    // of the H heads, in the order h * n_p + j; positions are laid end to end
    // and each CTA takes a contiguous stretch up to its share (cumulative
    // rounding places every tile), cut into one unit per position it touches.
    // A head split between two units gets one partial per piece.  The walk
    // keeps (head, chunk) of the point reached, so it needs no division.
    std::vector<int32_t> npart((size_t)b * H, 0);
    for (int32_t pos = 0; pos < b; ++pos)
        for (int32_t h = 0; h < H; ++h) npart[(size_t)pos * H + h] = nk1[pos];
    std::vector<Unit>& sf_units = plan.sf_scratch;     // static pieces, in CTA order
    std::vector<Unit>& tail_units = plan.tail_scratch;
    std::vector<int32_t>& sf_end = plan.sf_end;        // sf_units after CTA k
    sf_units.clear();
    tail_units.clear();
    sf_end.assign(grid, 0);
    {
        std::vector<double> quota(grid);
        double qsum = 0;
        for (int32_t k = 0; k < grid; ++k) { quota[k] = std::max(0.0, avg - load[k]); qsum += quota[k]; }
        const double scale = qsum > 0 ? sf_static / qsum : 0.0;
        auto seg_len = [&](int32_t ps) { return t.sf_offsets[ps + 1] - t.sf_offsets[ps]; };
        auto unit_at = [&](int32_t pos, int32_t h0, int32_t a, int32_t z, int32_t before) {
            return Unit{UNIT_SF, h0, pos, pos + 1, a, z, nk1[pos] + before, t.seq_perm[pos], seg_len(pos),
                        R + t.sf_offsets[pos], nk1[pos], 0};
        };
        int64_t placed = 0;
        double cum = 0;
        int32_t pos = 0, hd = 0, jd = 0;    // point reached: chunk jd of head hd of `pos`
        int32_t head_pieces = 0;            // pieces already placed of head hd
        auto next_pos = [&]() {
            hd = jd = head_pieces = 0;
            ++pos;
            while (pos < b && seg_len(pos) == 0) ++pos;
        };
        while (pos < b && seg_len(pos) == 0) ++pos;
        int32_t k = 0;
        for (; k < grid && pos < b; ++k) {
            cum += quota[k] * scale;
            const int64_t target = (k == grid - 1) ? (int64_t)sf_static : (int64_t)(cum + 0.5);
            int64_t room = target - placed;
            while (room > 0 && pos < b) {
                const int32_t n = seg_len(pos);
                const int64_t left = (int64_t)(H - hd) * n - jd;
                const int32_t take = (int32_t)std::min<int64_t>(room, left);
                const int32_t a = hd * n + jd, h0 = hd;
                const int32_t before = (jd == 0) ? 0 : head_pieces;
                sf_units.push_back(unit_at(pos, h0, a, a + take, before));
                // every head the piece touches gets one more partial
                int32_t rem = take, step = std::min(rem, n - jd);
                npart[(size_t)pos * H + hd] += 1;
                rem -= step;
                jd += step;
                while (rem > 0) {
                    ++hd;
                    npart[(size_t)pos * H + hd] += 1;
                    step = std::min(rem, n);
                    rem -= step;
                    jd = step;
                }
                if (jd == n) {
                    ++hd;
                    jd = 0;
                    head_pieces = 0;
                } else {
                    head_pieces = (hd == h0) ? before + 1 : 1;
                }
                placed += take;
                room -= take;
                if (hd == H) next_pos();
            }
            sf_end[k] = (int32_t)sf_units.size();
        }
        for (; k < grid; ++k) sf_end[k] = (int32_t)sf_units.size();
        // The rest of the list becomes the tail queue: units of at most
        // `tail_unit` chunk-heads that never cross a head boundary.  In a
        // small multi-row call, whose CTAs hold only a few tiles each, the
        // last 2 x grid chunk-heads (the queue's last claims) go in units of
        // two, so that the CTAs' finish times spread less.
        const int32_t tail_unit = std::max<int32_t>(
            kTailUnitMin, std::min<int32_t>(kTailUnitMax, (int32_t)((tail_tiles + kTailUnitsPerCta * grid - 1) /
                                                                   ((int64_t)kTailUnitsPerCta * grid))));
        int64_t remaining = 0;                       // chunk-heads left for the queue
        for (int32_t ps = pos; ps < b; ++ps) remaining += (int64_t)H * seg_len(ps);
        if (pos < b) remaining -= (int64_t)hd * seg_len(pos) + jd;
        const int64_t split_zone = small_multi_row ? 2 * (int64_t)grid : 0;
        while (pos < b) {
            const int32_t n = seg_len(pos);
            const int32_t unit_now = remaining <= split_zone ? std::min<int32_t>(2, tail_unit) : tail_unit;
            const int32_t a = hd * n + jd, len = std::min(unit_now, n - jd);
            remaining -= len;
            const int32_t before = (jd == 0) ? 0 : head_pieces;
            tail_units.push_back(unit_at(pos, hd, a, a + len, before));
            npart[(size_t)pos * H + hd] += 1;
            jd += len;
            if (jd == n) {
                ++hd;
                jd = 0;
                head_pieces = 0;
            } else {
                head_pieces = before + 1;
            }
            if (hd == H) next_pos();
        }
    }

    // partial ids per (position, query token, query head); every query token
    // and the G query heads of a key/value head have the same pieces
    plan.pbase.resize((size_t)b * q_len * HQ + 1);
    {
        int32_t acc = 0;
        size_t i = 0;
        plan.pbase[0] = 0;
        for (int32_t pos = 0; pos < b; ++pos)
            for (int32_t j = 0; j < q_len; ++j)
                for (int32_t h = 0; h < H; ++h) {
                    const int32_t np = npart[(size_t)pos * H + h];
                    for (int32_t g = 0; g < G; ++g) plan.pbase[++i] = (acc += np);
                }
    }
    plan.n_partials = plan.pbase.back();
    // Lay the lists out: per CTA its chunk-first units, then its pieces.
    plan.cta_begin.resize((size_t)grid + 1);
    std::vector<int32_t> cur(grid, 0);
    for (const auto& x : cf_at) cur[x.first] += 1;
    int32_t off = 0;
    for (int32_t k = 0; k < grid; ++k) {
        plan.cta_begin[k] = off;
        off += cur[k] + sf_end[k] - (k ? sf_end[k - 1] : 0);
        cur[k] = plan.cta_begin[k];
    }
    plan.cta_begin[grid] = off;
    plan.units.resize((size_t)off + tail_units.size());
    for (const auto& x : cf_at) plan.units[cur[x.first]++] = x.second;
    for (int32_t k = 0; k < grid; ++k)
        std::copy(sf_units.begin() + (k ? sf_end[k - 1] : 0), sf_units.begin() + sf_end[k],
                  plan.units.begin() + cur[k]);
    std::copy(tail_units.begin(), tail_units.end(), plan.units.begin() + off);
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

void layout_plan(const Plan& plan, int32_t b, PlanLayout& lay, std::vector<unsigned char>& blob,
                 const Tables& t) {
    size_t off = 0;
    lay.chunks = off;    off = align256(off + plan.chunks.size() * sizeof(ChunkRef));
    lay.units = off;     off = align256(off + plan.units.size() * sizeof(Unit));
    lay.seq_perm = off;  off = align256(off + (size_t)b * sizeof(int32_t));
    lay.pbase = off;     off = align256(off + plan.pbase.size() * sizeof(int32_t));
    lay.status = off;    off = align256(off + sizeof(int32_t));
    lay.counter = off;   off = align256(off + sizeof(int32_t));
    lay.chunk_tok0 = off; off = align256(off + plan.chunk_tok0.size() * sizeof(int32_t));
    lay.ctx_len = off;   off = align256(off + (size_t)b * sizeof(int32_t));
    lay.cta_head = off;  off = align256(off + (size_t)plan.grid * sizeof(CtaHead));
    lay.total = off;
    blob.assign(off, 0);
    std::memcpy(blob.data() + lay.chunks, plan.chunks.data(), plan.chunks.size() * sizeof(ChunkRef));
    std::memcpy(blob.data() + lay.units, plan.units.data(), plan.units.size() * sizeof(Unit));
    std::memcpy(blob.data() + lay.seq_perm, t.seq_perm.data(), (size_t)b * sizeof(int32_t));
    std::memcpy(blob.data() + lay.pbase, plan.pbase.data(), plan.pbase.size() * sizeof(int32_t));
    std::memcpy(blob.data() + lay.chunk_tok0, plan.chunk_tok0.data(), plan.chunk_tok0.size() * sizeof(int32_t));
    std::memcpy(blob.data() + lay.ctx_len, t.ctx_len.data(), (size_t)b * sizeof(int32_t));
    // Each CTA's first work, with the chunk refs of its first unit's steps
    // (a unit walks the linear (head, chunk) range [L0, L1); step L reads
    // chunk base + L % n, as the kernel's producer does).
    CtaHead* heads = reinterpret_cast<CtaHead*>(blob.data() + lay.cta_head);
    for (int32_t c = 0; c < plan.grid; ++c) {
        CtaHead h{};
        h.u_begin = plan.cta_begin[c];
        h.u_end = plan.cta_begin[c + 1];
        if (h.u_begin < h.u_end) {
            const Unit& u = plan.units[h.u_begin];
            h.first = u;
            const bool sf = u.kind == UNIT_SF;
            const int32_t n = sf ? u.n_per_head : u.c_end - u.c_begin;
            const int32_t base = sf ? u.base : u.c_begin;
            const int32_t L0 = sf ? u.c_begin : u.head * n;
            const int32_t L1 = sf ? u.c_end : (u.head + u.n_per_head) * n;
            for (int32_t k = 0; k < kHeadRefs && L0 + k < L1; ++k) h.refs[k] = plan.chunks[base + (L0 + k) % n];
        }
        heads[c] = h;
    }
}

void layout_ws(const Plan& plan, const Pool& p, int32_t b, WsLayout& ws) {
    const size_t H = p.cfg.n_heads, D = p.cfg.head_dim;   // q and out use the query heads
    size_t off = 0;
    ws.part_o = off;   off = align256(off + (size_t)plan.n_partials * D * sizeof(float));
    ws.part_ms = off;  off = align256(off + (size_t)plan.n_partials * 2 * sizeof(float));
    ws.total = off;
    ws.q_stage = off;  off = align256(off + (size_t)b * plan.q_len * H * D * 2);
    ws.out_stage = off; off = align256(off + (size_t)b * plan.q_len * H * D * 2);
    ws.total_host = off;
}

}  // namespace ca
