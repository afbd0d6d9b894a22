// Device code of libchunk_attention: the two-phase decode attention kernel,
// its merge kernel, and the KV scatter used by inserts and appends.  sm_103a
// (GB300).
//
// Method: ChunkAttention's two-phase partition ("ChunkAttention: Efficient
// Self-Attention with Prefix-Aware KV Cache and Two-Phase Partition", §3.2).
// A shared chunk is multiplied against the batched queries of every sequence
// holding it (chunk-first, tensor cores); each sequence's own chunks are
// processed per query (sequence-first: CUDA cores with warp-shuffle
// reductions on an fp16 pool; tensor cores, with the bytes widened straight
// into fragments, on an fp8 pool with 64-token chunks; tensor cores too when
// a position brings several query rows per key/value head: grouped query
// heads or several query tokens).  On an fp8 pool the chunk-first products
// also take their operands straight from the E4M3 bytes.  Every
// piece of work leaves a partial triple (o, m, s) that is
// combined by the rescaled-sum rule of the explainer blog's "Two-Phase
// Partition" section.
//
// GB300 design (not the paper's A100 kernel):
//  * one persistent launch holds both phases: CTAs take a host-balanced list
//    of chunk-first and sequence-first units, so the tensor-core work of the
//    shared chunks overlaps the HBM stream of the private chunks on the same
//    SMs (two CTAs per SM);
//  * a producer warp streams every chunk-head tile (c x D, fp16 or E4M3,
//    contiguous in the pool) into a ring of shared-memory stages with 2-D TMA
//    loads, 128-byte swizzled, completing on mbarriers; four consumer warps
//    compute (at head_dim 256 in pairs that split the head dims);
//  * every unit stores its partials with plain stores (no fences, atomics or
//    waits between units); a small merge kernel, launched as a programmatic
//    dependent of the main kernel so that its launch overlaps the main
//    kernel's tail, combines the partials of each (sequence, head);
//  * the main kernel is itself a programmatic dependent of the work before
//    it: its CTAs become resident as the previous grid drains and, when no
//    insert or append wrote the pool since the last call, start streaming
//    their static tiles at once, before the dependency wait that guards q,
//    the workspace and the queue counter;
//  * every wait is bounded (~1 s) and reports CA_ERR_TIMEOUT instead of
//    hanging.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <atomic>
#include <cstdio>
#include <cstring>

#include "ca_internal.h"

namespace ca {
namespace dev {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxStages = 8;
constexpr int kQRows = 64;                 // query rows per tensor-core unit, max (D <= 128)
// Query rows of the Q tile: 32 at head_dim 256 (the tile stays 16 KiB).
template <int D>
__host__ __device__ constexpr int q_rows() { return D == 256 ? 32 : kQRows; }
constexpr int kRing = 16;                  // unit announcements (producer -> consumers)
// Merge CTAs: one warp per pair, 16 warps a CTA (fewer CTAs to retire at
// the hand-over than 4-warp CTAs; measured 2% faster calls at 72 MB of KV)
constexpr int kMergeWarps = 16;
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for an mbarrier phase; false after about a second (never hangs).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t spin = 0; spin < (1u << 28); ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63) == 63 && global_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void consumer_sync() {   // named barrier over the 4 consumer warps
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
__device__ __forceinline__ float ex2(float x) {      // 2^x, hardware approximation
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t r;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r) : "r"(addr));
    return r;
}
__device__ __forceinline__ void lds64(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// The 8x8 b16 matrix held in fragment layout (lane L: row L/4, columns
// 2(L%4), 2(L%4)+1) transposed across the warp.
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
// FP8 E4M3 <-> fp16/fp32 conversions (hardware cvt, round to nearest even).
// In a packed pair the byte at the lower address is the low half.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t v16) {
    uint32_t r;
    const uint16_t v = (uint16_t)v16;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// A lane's DPL consecutive values: fp16 loads as packed pairs, fp32 loads and
// stores (DPL = 2, 4 or 8).
template <int DPL>
__device__ __forceinline__ void ld_h(const void* src, uint32_t (&w)[DPL / 2]) {
    if constexpr (DPL == 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (DPL == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t*>(src);
    }
}
template <int DPL>
__device__ __forceinline__ void ldcg_f(const float* src, float (&v)[DPL]) {
    if constexpr (DPL >= 4) {
#pragma unroll
        for (int i = 0; i < DPL; i += 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + i));
            v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
    } else {
        const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
        v[0] = x.x; v[1] = x.y;
    }
}
template <int DPL>
__device__ __forceinline__ void st_f(float* dst, const float (&v)[DPL]) {
    if constexpr (DPL >= 4) {
#pragma unroll
        for (int i = 0; i < DPL; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
        *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
    }
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
    atomicCAS(status, 0, code);
}

// Byte offset of 16-byte column chunk k of row r inside a tile stored as
// boxes of `rows` x 128 B (a row's bytes split 128 at a time), each 128-byte
// swizzled (TMA SWIZZLE_128B: chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int r, int k, int rows) {
    return (uint32_t)((k >> 3) * rows * 128 + r * 128 + (((k & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------
// Merge kernel: all partials of one (position, query token, head) combined by the
// explainer's output-combination rule, m* = max m_j,
// out = sum 2^{m_j-m*} o_j / sum 2^{m_j-m*} s_j (m in log2 units), taken a
// few partials at a time with the running maximum rescaled as it grows.  One
// warp per pair; lane L owns D/32 output dims; lane j of a group loads (m, s)
// of its partial while every lane loads its values of all the group's
// partials, so a group costs one memory round trip.  Launched as a
// programmatic dependent of the main kernel:
// `griddepcontrol.wait` returns once the main grid has completed and its
// stores are visible.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_partials_kernel(const AttnParams p, int n_pairs) {
    constexpr int DPL = D / 32;
    constexpr int KB = 4;                          // partials whose loads are in flight together
    const int gw = blockIdx.x * kMergeWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    // The next call's kernels may be scheduled now: they wait for this grid
    // before touching anything it writes, and their prologue overlaps it.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Plan entries may be read before the dependency wait; partials only after.
    int a = 0, n = 0, row = 0;
    if (gw < n_pairs) {
        a = p.pbase[gw];
        n = p.pbase[gw + 1] - a;
        // pair gw = (position, query token, head); out row = that position's
        // row of q times q_len plus the token
        row = p.seq_perm[gw / (p.q_len * p.n_heads)] * p.q_len + (gw / p.n_heads) % p.q_len;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.dyn_counter = 0;   // the main grid is done with it
    if (gw >= n_pairs) return;
    float M = -INFINITY, S = 0.f, acc[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
    for (int j = 0; j < n; j += KB) {
        const int cnt = min(KB, n - j);
        float2 ms = make_float2(-INFINITY, 0.f);
        if (lane < cnt) ms = __ldcg(&p.part_ms[a + j + lane]);
        float o[KB][DPL];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            ldcg_f<DPL>(p.part_o + (size_t)(a + j + min(k, cnt - 1)) * D + lane * DPL, o[k]);
        }
        float mk[KB], sk[KB], mg = M;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            mk[k] = __shfl_sync(kFull, ms.x, k);
            sk[k] = __shfl_sync(kFull, ms.y, k);
            if (k < cnt) mg = fmaxf(mg, mk[k]);
        }
        const float mu = (mg == -INFINITY) ? 0.f : mg;
        const float alpha = ex2(M - mu);            // 0 while nothing is accumulated
        S *= alpha;
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[d] *= alpha;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const float w = (k < cnt && mk[k] != -INFINITY) ? ex2(mk[k] - mu) : 0.f;
            S += w * sk[k];
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[d] += w * o[k][d];
        }
        M = mg;
    }
    const float inv = p.out_scale / S;          // an fp8 pool's value scale, else 1
    uint16_t* dst = p.out + ((size_t)row * p.n_heads + gw % p.n_heads) * D + lane * DPL;
    uint32_t h[DPL / 2];
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) h[i] = pack_half2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    if constexpr (DPL == 8) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
    } else if constexpr (DPL == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(h[0], h[1]);
    } else {
        *reinterpret_cast<uint32_t*>(dst) = h[0];
    }
}

// ---------------------------------------------------------------------------
// Sequence-first: one chunk-head tile against one query, warp w taking
// tokens [w*NT, (w+1)*NT) of the chunk.  Lane L owns dims [L*DPL, (L+1)*DPL).
// Scores are reduce-scattered across the warp so that each lane ends with
// the score of token (L >> (5 - log2 NT)); online softmax in log2 units.
// ---------------------------------------------------------------------------
template <int C, int D, int EB>
__device__ __forceinline__ void sf_chunk(const uint8_t* kt, const uint8_t* vt, int ntok,
                                         const float (&q)[D / 32], float& m, float& s,
                                         float (&o)[D / 32], int w, int lane) {
    constexpr int DPL = D / 32;
    constexpr int NT = C / kConsumerWarps;
    constexpr int LOGNT = NT == 16 ? 4 : NT == 8 ? 3 : 2;
    constexpr int BPL = DPL * EB;                     // bytes per lane per row
    const int kidx = (lane * BPL) >> 4, within = (lane * BPL) & 15;

    float part[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int r = w * NT + t;
        const uint8_t* src = kt + swz(r, kidx, C) + within;
        if constexpr (EB == 1) {                      // fp8: four bytes, two converts
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
            const uint32_t lo = f16x2_from_e4m3x2(raw & 0xffffu), hi = f16x2_from_e4m3x2(raw >> 16);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            part[t] = q[0] * a.x + q[1] * a.y + q[2] * b.x + q[3] * b.y;
        } else if constexpr (DPL == 8) {
            uint32_t raw[4];
            ld_h<8>(src, raw);
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw[i]));
                acc += q[2 * i] * a.x + q[2 * i + 1] * a.y;
            }
            part[t] = acc;
        } else if constexpr (DPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(src);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            part[t] = q[0] * a.x + q[1] * a.y + q[2] * b.x + q[3] * b.y;
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
            part[t] = q[0] * a.x + q[1] * a.y;
        }
    }
    // Reduce-scatter: after log2(NT) halving stages lane L holds the sum of
    // token (L >> (5-LOGNT)) over the lanes differing in its top bits; the
    // remaining stages sum over the low bits.
#pragma unroll
    for (int n = NT, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = upper ? part[i + n / 2] : part[i];
            const float send = upper ? part[i] : part[i + n / 2];
            part[i] = keep + __shfl_xor_sync(kFull, send, off);
        }
    }
#pragma unroll
    for (int off = 16 >> LOGNT; off >= 1; off >>= 1) part[0] += __shfl_xor_sync(kFull, part[0], off);

    const int j = lane >> (5 - LOGNT);
    float x = (w * NT + j < ntok) ? part[0] : -INFINITY;
    float mx = x;
#pragma unroll
    for (int off = 16; off >= (32 >> LOGNT); off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    const float mnew = fmaxf(m, mx);
    const float mu = (mnew == -INFINITY) ? 0.f : mnew;
    const float alpha = ex2(m - mu);
    const float pj = ex2(x - mu);
    float ps = pj;
#pragma unroll
    for (int off = 16; off >= (32 >> LOGNT); off >>= 1) ps += __shfl_xor_sync(kFull, ps, off);
    s = s * alpha + ps;
    m = mnew;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] *= alpha;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float pt = __shfl_sync(kFull, pj, t << (5 - LOGNT));
        const uint8_t* src = vt + swz(w * NT + t, kidx, C) + within;
        if constexpr (EB == 1) {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
            const uint32_t lo = f16x2_from_e4m3x2(raw & 0xffffu), hi = f16x2_from_e4m3x2(raw >> 16);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            o[0] += pt * a.x; o[1] += pt * a.y; o[2] += pt * b.x; o[3] += pt * b.y;
        } else if constexpr (DPL == 8) {
            uint32_t raw[4];
            ld_h<8>(src, raw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw[i]));
                o[2 * i] += pt * a.x;
                o[2 * i + 1] += pt * a.y;
            }
        } else if constexpr (DPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(src);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            o[0] += pt * a.x; o[1] += pt * a.y; o[2] += pt * b.x; o[3] += pt * b.y;
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
            o[0] += pt * a.x; o[1] += pt * a.y;
        }
    }
}

// ---------------------------------------------------------------------------
// Sequence-first on an fp8 pool with 64-token chunks: the same product on
// the tensor cores.  One query row against a chunk-head tile is a matrix-
// vector product, but on CUDA cores the E4M3 widening and the cross-lane
// reductions made this path issue-bound (half the issue slots busy, HBM at
// half its rate), so warp w multiplies its 16 tokens [16w, 16w + 16) with
// mma.sync m16n8k16, the query replicated over the 8 columns, and the bytes
// widened straight into fragment registers (fp32 accumulation throughout).
// Lane (g, t) = (lane / 4, lane % 4).
//  * S = K q: A = the 16-token x 16-dim key block of step kk with the dims
//    permuted inside the step, fragment column 2t (+1) <-> dim 16kk + 4t (+1)
//    and 2t + 8 (+9) <-> 16kk + 4t + 2 (+3), so that one 32-bit load of row g
//    (and g + 8) gives the lane its four bytes; qb[kk] holds the query's
//    dims in the same order.  The result rows are whole scores: tokens g and
//    g + 8, in every lane of the group.
//  * O^T += V^T p: per pair of 16-dim blocks, fragment row g <-> dims
//    32qd + 4g (+2) and row g + 8 <-> 32qd + 4g + 1 (+3); fragment column
//    (token) 2t, 2t + 1, 2t + 8, 2t + 9 <-> tokens t, 4 + t, 8 + t, 12 + t.
//    Each lane loads 4 bytes of those four tokens and pairs them per dim with
//    byte permutes; p arrives in the same token order by two shuffles.
// Only columns 0 (c0, c2) of the output fragments are read, so only they are
// rescaled.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void sf_chunk_f8_tc(const uint8_t* kt, const uint8_t* vt, int ntok,
                                               const uint32_t (&qb)[8][2], float scale_log2, float& m,
                                               float& s, float (&oc)[8][4], int w, int lane) {
    constexpr int C = 64;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * w + g, r1 = r0 + 8;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(kt + swz(r0, kk, C) + 4 * t);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(kt + swz(r1, kk, C) + 4 * t);
        const uint32_t a[4] = {f16x2_from_e4m3x2(w0 & 0xffffu), f16x2_from_e4m3x2(w1 & 0xffffu),
                               f16x2_from_e4m3x2(w0 >> 16), f16x2_from_e4m3x2(w1 >> 16)};
        mma16816(acc, a, qb[kk][0], qb[kk][1]);
    }
    const float x0 = (r0 < ntok) ? acc[0] * scale_log2 : -INFINITY;   // token r0
    const float x1 = (r1 < ntok) ? acc[2] * scale_log2 : -INFINITY;   // token r1
    float mx = fmaxf(x0, x1);
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    const float mnew = fmaxf(m, mx);
    const float mu = (mnew == -INFINITY) ? 0.f : mnew;
    const float alpha = ex2(m - mu);
    const float p0 = ex2(x0 - mu), p1 = ex2(x1 - mu);
    float ps = p0 + p1;
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) ps += __shfl_xor_sync(kFull, ps, off);
    s = s * alpha + ps;
    m = mnew;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
        oc[mb][0] *= alpha;
        oc[mb][2] *= alpha;
    }
    // p of tokens (t, 4 + t) and (8 + t, 12 + t), as the B fragment
    const uint32_t p2 = pack_half2(p0, p1);                   // (p[g], p[g + 8])
    const uint32_t u = __shfl_sync(kFull, p2, 4 * t);         // (p[t], p[t + 8])
    const uint32_t v = __shfl_sync(kFull, p2, 16 + 4 * t);    // (p[4 + t], p[12 + t])
    const uint32_t pb0 = __byte_perm(u, v, 0x5410), pb1 = __byte_perm(u, v, 0x7632);
    const int t0 = 16 * w + t;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
        const int kc = 2 * qd + (g >> 2), off = 4 * (g & 3);
        const uint32_t x0b = *reinterpret_cast<const uint32_t*>(vt + swz(t0, kc, C) + off);
        const uint32_t x1b = *reinterpret_cast<const uint32_t*>(vt + swz(t0 + 4, kc, C) + off);
        const uint32_t x2b = *reinterpret_cast<const uint32_t*>(vt + swz(t0 + 8, kc, C) + off);
        const uint32_t x3b = *reinterpret_cast<const uint32_t*>(vt + swz(t0 + 12, kc, C) + off);
        // bytes 0/1 of each token's word: dims 32qd + 4g (+1); bytes 2/3: +2 (+3)
        const uint32_t za = __byte_perm(x0b, x1b, 0x5140), zb = __byte_perm(x2b, x3b, 0x5140);
        const uint32_t zc = __byte_perm(x0b, x1b, 0x7362), zd = __byte_perm(x2b, x3b, 0x7362);
        const uint32_t a0[4] = {f16x2_from_e4m3x2(za & 0xffffu), f16x2_from_e4m3x2(za >> 16),
                                f16x2_from_e4m3x2(zb & 0xffffu), f16x2_from_e4m3x2(zb >> 16)};
        mma16816(oc[2 * qd], a0, pb0, pb1);
        const uint32_t a1[4] = {f16x2_from_e4m3x2(zc & 0xffffu), f16x2_from_e4m3x2(zc >> 16),
                                f16x2_from_e4m3x2(zd & 0xffffu), f16x2_from_e4m3x2(zd >> 16)};
        mma16816(oc[2 * qd + 1], a1, pb0, pb1);
    }
}

// ---------------------------------------------------------------------------
// Tensor-core path (chunk-first units, and sequence-first units with several
// query rows): one chunk-head tile against a 16-row block of the Q tile with
// mma.sync m16n8k16 (fp16 in, fp32 accumulate).  The warp takes tokens
// [tok0, tok0 + NT) of the chunk.  Row state per thread: rows g = lane/4 and
// g + 8 of the block.
// ---------------------------------------------------------------------------
// Scores of a 16-row block against NT tokens [tok0, tok0 + NT) of a chunk
// tile, over the head dims [16 kk0, 16 kk1): S = Q K^T with the Q fragments
// read from the swizzled Q tile (row lane%16, 16-byte chunk 2kk + lane/16).
template <int C, int D, int NT, bool F8 = false>
__device__ __forceinline__ void cf_scores(uint32_t kt, int tok0, uint32_t qrow_addr_base, int kk0, int kk1,
                                          float (&sacc)[NT / 8][4], int lane) {
#pragma unroll
    for (int i = 0; i < NT / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
    if constexpr (F8) {
        // E4M3 keys (128-byte rows, 16-byte chunk kk of row r at chunk
        // kk ^ (r % 8)).  Inside each 16-dim step the fragment columns are
        // permuted, 2t (+1) <-> dim 16kk + 4t (+1) and 2t + 8 (+9) <->
        // 16kk + 4t + 2 (+3), on both operands: one 32-bit load gives a
        // lane's four key bytes of token g, one 64-bit load its four query
        // dims of a row.  The scores come out in the usual layout.
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int kk = kk0; kk < kk1; ++kk) {
            uint32_t qa[4];
            lds64(qrow_addr_base + swz(g, 2 * kk + (t >> 1), q_rows<D>()) + 8 * (t & 1), qa[0], qa[2]);
            lds64(qrow_addr_base + swz(g + 8, 2 * kk + (t >> 1), q_rows<D>()) + 8 * (t & 1), qa[1], qa[3]);
#pragma unroll
            for (int j = 0; j < NT / 8; ++j) {
                const int row = tok0 + 8 * j + g;
                const uint32_t wd = lds32(kt + row * 128 + ((kk ^ (row & 7)) << 4) + 4 * t);
                mma16816(sacc[j], qa, f16x2_from_e4m3x2(wd & 0xffffu), f16x2_from_e4m3x2(wd >> 16));
            }
        }
        return;
    }
#pragma unroll
    for (int kk = kk0; kk < kk1; ++kk) {
        uint32_t qa[4];
        {
            const int qr = (lane & 15), qc = 2 * kk + (lane >> 4);
            ldsm_x4(qrow_addr_base + swz(qr, qc, q_rows<D>()), qa[0], qa[1], qa[2], qa[3]);
        }
#pragma unroll
        for (int np = 0; np < NT / 16; ++np) {
            const int tok = tok0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int kc = 2 * kk + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + swz(tok, kc, C), b0, b1, b2, b3);
            mma16816(sacc[2 * np], qa, b0, b1);
            mma16816(sacc[2 * np + 1], qa, b2, b3);
        }
    }
}

// Online softmax of a scored 16-row block (log2 units; columns past ntok,
// and under the causal mask past each row's limit, are masked), then
// O += P V for the OD output dims [16 dp0, 16 dp0 + OD).
template <int C, int NT, int OD, bool F8 = false>
__device__ __forceinline__ void cf_softmax_pv(uint32_t vt, int ntok, int tok0, int ctx0, int lim0, int lim1,
                                              float scale_log2, float (&sacc)[NT / 8][4], int dp0,
                                              float (&m)[2], float (&s)[2], float (&o)[OD / 8][4], int lane) {
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NT / 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = tok0 + nt * 8 + 2 * (lane & 3) + (e & 1);
            // a column counts if it holds a token and, under the causal
            // mask, that token is at or before the row's limit
            const bool ok = col < ntok && ctx0 + col <= ((e >> 1) ? lim1 : lim0);
            const float x = ok ? sacc[nt][e] * scale_log2 : -INFINITY;
            sacc[nt][e] = x;
            mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
    }
    // The row's reference maximum m is raised lazily: only when the chunk's
    // maximum exceeds it by more than 2^8 (P then stays below 256, exact in
    // fp16), so most chunks leave O unscaled; o and s always refer to the
    // same m, which the partial carries.
    float alpha[2], mu[2];
    bool grow = false;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 2));
        alpha[r] = 1.f;
        if (mx[r] > m[r] + 8.f) {                   // also the first finite maximum
            alpha[r] = ex2(m[r] - mx[r]);           // 0 while m is -inf
            m[r] = mx[r];
            s[r] *= alpha[r];
            grow = true;
        }
        mu[r] = (m[r] == -INFINITY) ? 0.f : m[r];
    }
    uint32_t pa[NT / 16][4];
#pragma unroll
    for (int nt = 0; nt < NT / 8; ++nt) {
        const float p0 = ex2(sacc[nt][0] - mu[0]), p1 = ex2(sacc[nt][1] - mu[0]);
        const float p2 = ex2(sacc[nt][2] - mu[1]), p3 = ex2(sacc[nt][3] - mu[1]);
        s[0] += p0 + p1;
        s[1] += p2 + p3;
        // accumulator layout of n-tile nt == A-operand layout of k-step nt/2
        pa[nt >> 1][(nt & 1) * 2 + 0] = pack_half2(p0, p1);
        pa[nt >> 1][(nt & 1) * 2 + 1] = pack_half2(p2, p3);
    }
    if (__any_sync(kFull, grow)) {
#pragma unroll
        for (int dt = 0; dt < OD / 8; ++dt) {
            o[dt][0] *= alpha[0]; o[dt][1] *= alpha[0];
            o[dt][2] *= alpha[1]; o[dt][3] *= alpha[1];
        }
    }
    if constexpr (F8) {
        // E4M3 values: n-tile 4dq + i holds output dims 32dq + 4n + i
        // (n = the fragment column), so a lane's B operand for dims
        // 32dq + 4g .. + 3 of its four tokens (16j + 2t, + 1, + 8, + 9) is
        // four 32-bit loads paired per dim by byte permutes.  The
        // accumulator of lane (g, t) then holds dims 32dq + 8t .. + 7 of its
        // rows: o[4dq + i][c] <-> dim 32dq + 8t + 4c' + i (c' = c % 2).
        static_assert(OD == 128, "fp8 pools have head_dim 128");
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int j = 0; j < NT / 16; ++j) {
            const int r0 = tok0 + 16 * j + 2 * t;
#pragma unroll
            for (int dq = 0; dq < 4; ++dq) {
                const int kc = 2 * dq + (g >> 2);
                const uint32_t off = 4 * (g & 3);
                const uint32_t wa = lds32(vt + r0 * 128 + ((kc ^ (r0 & 7)) << 4) + off);
                const uint32_t wb = lds32(vt + (r0 + 1) * 128 + ((kc ^ ((r0 + 1) & 7)) << 4) + off);
                const uint32_t wc = lds32(vt + (r0 + 8) * 128 + ((kc ^ (r0 & 7)) << 4) + off);
                const uint32_t wd = lds32(vt + (r0 + 9) * 128 + ((kc ^ ((r0 + 1) & 7)) << 4) + off);
                const uint32_t x01 = __byte_perm(wa, wb, 0x5140), x23 = __byte_perm(wa, wb, 0x7362);
                const uint32_t y01 = __byte_perm(wc, wd, 0x5140), y23 = __byte_perm(wc, wd, 0x7362);
                mma16816(o[4 * dq + 0], pa[j], f16x2_from_e4m3x2(x01 & 0xffffu), f16x2_from_e4m3x2(y01 & 0xffffu));
                mma16816(o[4 * dq + 1], pa[j], f16x2_from_e4m3x2(x01 >> 16), f16x2_from_e4m3x2(y01 >> 16));
                mma16816(o[4 * dq + 2], pa[j], f16x2_from_e4m3x2(x23 & 0xffffu), f16x2_from_e4m3x2(y23 & 0xffffu));
                mma16816(o[4 * dq + 3], pa[j], f16x2_from_e4m3x2(x23 >> 16), f16x2_from_e4m3x2(y23 >> 16));
            }
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < NT / 16; ++j) {
#pragma unroll
        for (int dq = 0; dq < OD / 16; ++dq) {
            const int tok = tok0 + 16 * j + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int kc = 2 * (dp0 + dq) + (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vt + swz(tok, kc, C), b0, b1, b2, b3);
            mma16816(o[2 * dq], pa[j], b0, b1);
            mma16816(o[2 * dq + 1], pa[j], b2, b3);
        }
    }
}

// One warp, one 16-row block, NT tokens, every head dim.
// F8: K and V are the stage's E4M3 bytes (head_dim 128), and o comes out
// with its dims permuted as cf_softmax_pv describes.
template <int C, int D, int NT, bool F8 = false>
__device__ __forceinline__ void cf_chunk(uint32_t kt, uint32_t vt, int ntok, int tok0, int ctx0, int lim0,
                                         int lim1, uint32_t qrow_addr_base, float scale_log2,
                                         float (&m)[2], float (&s)[2], float (&o)[D / 8][4], int lane) {
    float sacc[NT / 8][4];
    cf_scores<C, D, NT, F8>(kt, tok0, qrow_addr_base, 0, D / 16, sacc, lane);
    cf_softmax_pv<C, NT, D, F8>(vt, ntok, tok0, ctx0, lim0, lim1, scale_log2, sacc, 0, m, s, o, lane);
}

// head_dim 256: two warps share a 16-row block, warp `half` owning head dims
// [128 half, 128 half + 128) (128 fp32 accumulators per thread for all 256
// would not fit the register budget).  Each scores the block over its dims,
// the pair adds the two halves through shared memory (xs_w its own slot,
// xs_p the partner's; the slots alternate by chunk parity, so one pair
// barrier per chunk keeps the next chunk's writes clear of this chunk's
// reads), both take the same softmax, and each accumulates P V for its dims.
template <int C, int NT>
__device__ __forceinline__ void cf_chunk_split(uint32_t kt, uint32_t vt, int ntok, int tok0, int ctx0, int lim0,
                                               int lim1, uint32_t qrow_addr_base, float scale_log2, int half,
                                               float* xs_w, const float* xs_p, int bar_id,
                                               float (&m)[2], float (&s)[2], float (&o)[16][4], int lane) {
    float sacc[NT / 8][4];
    cf_scores<C, 256, NT>(kt, tok0, qrow_addr_base, 8 * half, 8 * half + 8, sacc, lane);
#pragma unroll
    for (int i = 0; i < NT / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) xs_w[(i * 4 + e) * 32 + lane] = sacc[i][e];
    asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
#pragma unroll
    for (int i = 0; i < NT / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[i][e] += xs_p[(i * 4 + e) * 32 + lane];
    cf_softmax_pv<C, NT, 128>(vt, ntok, tok0, ctx0, lim0, lim1, scale_log2, sacc, 8 * half, m, s, o, lane);
}

// An fp8 chunk-head tile (C rows of 128 one-byte dims, 128-byte swizzled as
// TMA stores it) widened to the fp16 tile layout the transposed few-row
// products read (chunk-first tiles read the bytes directly)
// (two 64-dim boxes, each 128-byte swizzled).  E4M3 values are exact in fp16.
// All consumer threads take part.
template <int C>
__device__ __forceinline__ void f8_tile_to_f16(const uint8_t* src, uint8_t* dst, int tid) {
#pragma unroll 2
    for (int i = tid; i < C * 8; i += kConsumerWarps * 32) {
        const int r = i >> 3, kc = i & 7;
        const uint4 v = *reinterpret_cast<const uint4*>(src + r * 128 + ((kc ^ (r & 7)) << 4));
        uint4 a, b;
        a.x = f16x2_from_e4m3x2(v.x & 0xffffu); a.y = f16x2_from_e4m3x2(v.x >> 16);
        a.z = f16x2_from_e4m3x2(v.y & 0xffffu); a.w = f16x2_from_e4m3x2(v.y >> 16);
        b.x = f16x2_from_e4m3x2(v.z & 0xffffu); b.y = f16x2_from_e4m3x2(v.z >> 16);
        b.z = f16x2_from_e4m3x2(v.w & 0xffffu); b.w = f16x2_from_e4m3x2(v.w >> 16);
        *reinterpret_cast<uint4*>(dst + swz(r, 2 * kc, C)) = a;
        *reinterpret_cast<uint4*>(dst + swz(r, 2 * kc + 1, C)) = b;
    }
}

// Shared-memory map of one CTA.  EB: bytes per stored K/V element (2 for
// fp16, 1 for fp8, which adds an fp16 copy of one stage for the transposed
// few-row products).
template <int C, int D, int EB>
struct Smem {
    static constexpr int kTile = C * D * EB;    // one K or V tile of one chunk-head
    static constexpr int kStage = 2 * kTile;    // K then V
    static constexpr int kConvBytes = EB == 1 ? 2 * C * D * 2 : 0;
    static constexpr int kQBytes = q_rows<D>() * D * 2;
    // head_dim 256: score halves exchanged by warp pairs, two chunk parities
    static constexpr int kXsBytes = D == 256 ? 2 * kConsumerWarps * (C / 8) * 4 * 32 * 4 : 0;
    static constexpr int kXmsBytes = 512;
    static constexpr int kBarBytes = 2 * kMaxStages * 8;
    static constexpr int kRingBytes = kRing * 4 + 2 * kMaxStages * 4;   // ids, then ntok and tok0 per stage
    static size_t bytes(int stages) {
        return (size_t)stages * kStage + kConvBytes + kXsBytes + kQBytes + kXmsBytes + kBarBytes + kRingBytes;
    }
};

// ---------------------------------------------------------------------------
// A sequence-first unit of one position with at most 8 query rows per key/
// value head (grouped query heads or several query tokens).  The products
// are taken transposed, tokens on the mma rows and the query rows on its 8
// columns: S^T = K Q^T and O^T += V^T P^T, so no mma row is padding (a
// 16-row block would hold 4 live rows at G = 4).  Warp w < T takes tokens
// [16w, 16w + 16) of each chunk; lane (g, t) holds the scores of tokens g
// and g + 8 for query rows 2t and 2t + 1, and O^T for dims 16db + g (+8) of
// the same rows.  Q^T fragments are read from the Q tile with ldmatrix each
// chunk; P^T fragments are the score fragments transposed in registers
// (movmatrix).  The warps' states are tree-combined through the Q tile at
// each head boundary and warp 0 writes the rows' partials.  It is compiled
// only into the kernel variant for such schedules, so that its registers do
// not weigh on the single-row kernel.  Walks [L, L_end) of the unit's
// (head, chunk) range; false on a timeout.
// ---------------------------------------------------------------------------
template <int C, int D, int EB>
__device__ __forceinline__ bool sf_rows_transposed(
    const AttnParams& p, uint8_t* stages, uint8_t* conv, uint8_t* qreg, float* xms, uint32_t full0,
    uint32_t empty0, const volatile int32_t* stage_ntok, const volatile int32_t* stage_tok0, int S, int& it_io,
    int& L_io, int L_end, int n, int q_lo, int m_rows, int part_first, int part_rest, int w, int lane) {
    using SM = Smem<C, D, EB>;
    const int H = p.n_heads, G = p.group, QL = p.q_len;
    const int Tr = min(kConsumerWarps, C / 16);
    const bool act = w < Tr;
    const int g = lane >> 2, t = lane & 3;
    int it = it_io, L = L_io;
    int limr[2] = {INT_MAX, INT_MAX};               // causal limits of rows 2t, 2t + 1
    if (p.causal) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (2 * t + r < m_rows) limr[r] = p.ctx_len[q_lo] - QL + (2 * t + r) / G;
    }
    bool ok = true;
    for (bool first = true; L < L_end && ok; first = false) {
        const int kvh = L / n;
        const int seg_end = min(L_end, (kvh + 1) * n);
        const int upart = first ? part_first : part_rest;
        if (!first) consumer_sync();   // the previous head's exchange reads are done
        for (int idx = threadIdx.x; idx < m_rows * (D / 8); idx += kConsumerWarps * 32) {
            const int r = idx / (D / 8), k = idx % (D / 8);
            const size_t qrow_tok = (size_t)p.seq_perm[q_lo] * QL + r / G;
            const uint16_t* src = p.q + (qrow_tok * H + kvh * G + r % G) * D + k * 8;
            cp_async16(smem_u32(qreg + swz(r, k, q_rows<D>())), src);
        }
        cp_async_wait_all();
        consumer_sync();
        float ot[D / 16][4], m[2] = {-INFINITY, -INFINITY}, s[2] = {0.f, 0.f};
#pragma unroll
        for (int db = 0; db < D / 16; ++db) ot[db][0] = ot[db][1] = ot[db][2] = ot[db][3] = 0.f;
        for (; L < seg_end; ++L, ++it) {
            const int st = it % S;
            if (!mbar_wait(full0 + 8 * st, (uint32_t)(it / S) & 1u)) {
                set_status(p.status, CA_ERR_TIMEOUT);
                ok = false;
                break;
            }
            uint32_t kt = smem_u32(stages + (size_t)st * SM::kStage);
            uint32_t vt = kt + SM::kTile;
            const int ntok = stage_ntok[st];
            const int ctx0 = stage_tok0[st];
            if constexpr (EB == 1) {
                consumer_sync();
                const uint8_t* sk = stages + (size_t)st * SM::kStage;
                f8_tile_to_f16<C>(sk, conv, threadIdx.x);
                f8_tile_to_f16<C>(sk + SM::kTile, conv + SM::kConvBytes / 2, threadIdx.x);
                consumer_sync();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
                kt = smem_u32(conv);
                vt = kt + SM::kConvBytes / 2;
            }
            if (act) {
                const int tok0 = 16 * w;
                float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // Q^T as the B operand: n = query row (lane & 7), k = 16 dims
                    uint32_t a[4], qb0, qb1;
                    ldsm_x2(smem_u32(qreg) + swz(lane & 7, 2 * kk + ((lane >> 3) & 1), q_rows<D>()), qb0, qb1);
                    ldsm_x4(kt + swz(tok0 + (lane & 15), 2 * kk + (lane >> 4), C), a[0], a[1], a[2], a[3]);
                    mma16816(sacc, a, qb0, qb1);
                }
                // sacc: (token g, rows 2t, 2t+1), (token g + 8, rows 2t, 2t+1)
                float x[4], mx[2];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = tok0 + g + 8 * (i >> 1), row = 2 * t + (i & 1);
                    const bool valid = tok < ntok && row < m_rows && ctx0 + tok <= limr[i & 1];
                    x[i] = valid ? sacc[i] * p.scale_log2 : -INFINITY;
                }
                mx[0] = fmaxf(x[0], x[2]);
                mx[1] = fmaxf(x[1], x[3]);
                bool grow = false;
                float alpha[2] = {1.f, 1.f}, mu[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
#pragma unroll
                    for (int off = 4; off <= 16; off <<= 1) mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], off));
                    // the reference maximum is raised lazily, as in cf_softmax_pv
                    if (mx[r] > m[r] + 8.f) {
                        alpha[r] = ex2(m[r] - mx[r]);
                        m[r] = mx[r];
                        s[r] *= alpha[r];
                        grow = true;
                    }
                    mu[r] = (m[r] == -INFINITY) ? 0.f : m[r];
                }
                if (__any_sync(kFull, grow)) {
#pragma unroll
                    for (int db = 0; db < D / 16; ++db) {
                        ot[db][0] *= alpha[0]; ot[db][1] *= alpha[1];
                        ot[db][2] *= alpha[0]; ot[db][3] *= alpha[1];
                    }
                }
                const float p0 = ex2(x[0] - mu[0]), p1 = ex2(x[1] - mu[1]);
                const float p2 = ex2(x[2] - mu[0]), p3 = ex2(x[3] - mu[1]);
                float ps[2] = {p0 + p2, p1 + p3};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
#pragma unroll
                    for (int off = 4; off <= 16; off <<= 1) ps[r] += __shfl_xor_sync(kFull, ps[r], off);
                    s[r] += ps[r];
                }
                // P^T fragments: k = tokens, n = query rows
                const uint32_t b0 = movm_trans(pack_half2(p0, p1));   // tokens 0..7
                const uint32_t b1 = movm_trans(pack_half2(p2, p3));   // tokens 8..15
#pragma unroll
                for (int db = 0; db < D / 16; ++db) {
                    uint32_t a[4];
                    ldsm_x4_t(vt + swz(tok0 + (lane & 7) + ((lane >> 4) << 3), 2 * db + ((lane >> 3) & 1), C),
                              a[0], a[1], a[2], a[3]);
                    mma16816(ot[db], a, b0, b1);
                }
            }
            if constexpr (EB == 2) {
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * st);
            }
        }
        if (!ok) break;
        // Combine the Tr warps' states through the Q tile (free once every
        // warp has left the chunk loop: the barrier opening each round).
        float* xo = reinterpret_cast<float*>(qreg);
        for (int half = Tr / 2; half >= 1; half /= 2) {
            consumer_sync();
            if (w >= half && w < 2 * half) {
                float* dst = xo + (size_t)(w - half) * (D / 16) * 4 * 32;
#pragma unroll
                for (int db = 0; db < D / 16; ++db)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[(db * 4 + e) * 32 + lane] = ot[db][e];
                if (g == 0) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        xms[(w - half) * 16 + (2 * t + r) * 2] = m[r];
                        xms[(w - half) * 16 + (2 * t + r) * 2 + 1] = s[r];
                    }
                }
            }
            consumer_sync();
            if (w < half) {
                const float* so = xo + (size_t)w * (D / 16) * 4 * 32;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float m2 = xms[w * 16 + (2 * t + r) * 2], s2 = xms[w * 16 + (2 * t + r) * 2 + 1];
                    const float M = fmaxf(m[r], m2);
                    const float Mu = (M == -INFINITY) ? 0.f : M;
                    const float a1 = ex2(m[r] - Mu), a2 = ex2(m2 - Mu);
                    s[r] = s[r] * a1 + s2 * a2;
                    m[r] = M;
#pragma unroll
                    for (int db = 0; db < D / 16; ++db) {
                        ot[db][r] = ot[db][r] * a1 + so[(db * 4 + r) * 32 + lane] * a2;
                        ot[db][r + 2] = ot[db][r + 2] * a1 + so[(db * 4 + r + 2) * 32 + lane] * a2;
                    }
                }
            }
        }
        if (w == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = 2 * t + r;
                if (row < m_rows) {
                    const int pid = p.pbase[((size_t)q_lo * QL + row / G) * H + kvh * G + row % G] + upart;
                    float* dst = p.part_o + (size_t)pid * D;
#pragma unroll
                    for (int db = 0; db < D / 16; ++db) {
                        dst[16 * db + g] = ot[db][r];
                        dst[16 * db + g + 8] = ot[db][r + 2];
                    }
                    if (g == 0) p.part_ms[pid] = make_float2(m[r], s[r]);
                }
            }
        }
    }
    it_io = it;
    L_io = L;
    return ok;
}

// ---------------------------------------------------------------------------
// The persistent two-phase kernel.
// ---------------------------------------------------------------------------
// kRows: the variant for schedules whose positions bring 2..8 query rows per
// key/value head (head_dim <= 128): it has the transposed few-row path and
// no single-row sequence-first path; the other variant the reverse.
template <int C, int D, int EB, bool kRows>
__global__ void __launch_bounds__(kThreads, 2)
two_phase_attention_kernel(const __grid_constant__ CUtensorMap tmap, const AttnParams p) {
    using SM = Smem<C, D, EB>;
    constexpr int DPL = D / 32;
    constexpr int BOXES = D * EB / 128;   // 128-byte boxes per tile row
    // single-row sequence-first work of an fp8 pool with 64-token chunks
    // runs on the tensor cores (sf_chunk_f8_tc), elsewhere on CUDA cores
    constexpr bool kF8Tc = EB == 1 && C == 64 && D == 128;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = p.n_stages;
    uint8_t* stages = smem;
    uint8_t* conv = smem + (size_t)S * SM::kStage;       // fp8 pools: fp16 copy of one stage
    float* xs = reinterpret_cast<float*>(conv + SM::kConvBytes);   // head_dim 256 score exchange
    uint8_t* qreg = conv + SM::kConvBytes + SM::kXsBytes;
    float* xms = reinterpret_cast<float*>(qreg + SM::kQBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xms) + SM::kXmsBytes);
    volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(bars + 2 * kMaxStages);
    volatile int32_t* stage_ntok = ring + kRing;          // valid tokens of each stage's chunk
    volatile int32_t* stage_tok0 = stage_ntok + kMaxStages;   // its first token's context offset
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The merge kernel may be scheduled now; it waits for this grid itself.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((smem_u32(smem) & 1023u) != 0 || S < 1 || S > kMaxStages) {   // uniform across the CTA
        if (threadIdx.x == 0) set_status(p.status, CA_ERR_INVALID);
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    // this CTA's first work: one 128-byte line (its unit range, first unit
    // and that unit's first chunk refs)
    const CtaHead* hd = p.cta_head + blockIdx.x;
    const int2 range = *reinterpret_cast<const int2*>(hd);
    const int u_begin = range.x, u_end = range.y;
    const int H = p.n_heads;            // query heads (q, out, partials)
    const int HK = p.n_kv_heads;        // key/value heads (pool tiles, units)
    const int G = p.group;              // query heads per key/value head
    const int QL = p.q_len;             // query tokens per position
    const int RW = QL * G;              // query rows per position and key/value head

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane != 0) return;
        // the tensor map's descriptor is fetched while the plan line loads
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
        if (p.test_stall) {
            // Test hook (ca_sched_inject_stall): wait for stage 0's first
            // phase, which nothing completes since no copy has been issued;
            // the wait gives up after its limit and the producer leaves
            // without issuing anything.  The consumers' first waits give up
            // the same way.
            if (!mbar_wait(full0, 0u)) set_status(p.status, CA_ERR_TIMEOUT);
            return;
        }
        const uint64_t pol = policy_evict_first();
        int it = 0;
        bool ok = true;
        // Work: this CTA's static units [u_begin, u_end), then units claimed
        // one at a time from the shared tail queue [dyn_begin, dyn_end).  A
        // queue unit is claimed only once this CTA has issued all its earlier
        // work (at most one claim ahead), so slow CTAs do not hoard the tail.
        // Each unit's id is written to the ring before its first chunk is
        // issued (that chunk's barrier arrival publishes it); after the last
        // unit a stage carries the id -1.  The plan may be read before the
        // dependency wait; the queue counter (reset by the previous call's
        // merge kernel) only after it, and the pool too unless p.kv_stable.
        // Both kinds walk a linear (head, chunk) range: step L covers chunk
        // base + L % n of head L / n.  A chunk-first unit's n is its row count
        // and its range spans its heads.
        auto lin_n = [](const Unit& X) { return X.kind == UNIT_SF ? X.n_per_head : X.c_end - X.c_begin; };
        auto lin_base = [](const Unit& X) { return X.kind == UNIT_SF ? X.base : X.c_begin; };
        auto lin_begin = [&](const Unit& X) { return X.kind == UNIT_SF ? X.c_begin : X.head * lin_n(X); };
        auto lin_end = [&](const Unit& X) {
            return X.kind == UNIT_SF ? X.c_end : (X.head + X.n_per_head) * lin_n(X);
        };
        auto first_chunk = [&](const Unit& X) { return lin_base(X) + lin_begin(X) % lin_n(X); };
        int s_next = u_begin;
        // The previous kernel in the stream (normally the previous call's
        // merge) may still run.  The queue counter it resets is read only after
        // the dependency wait, and so is the pool unless no insert or append
        // wrote it since the last call: then this CTA's static tiles stream
        // at once, overlapping that kernel and the previous grid's tail.
        bool dep_done = false;
        auto dep_wait = [&]() {
            if (!dep_done) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                dep_done = true;
            }
        };
        auto claim = [&]() -> int {
            if (s_next < u_end) return s_next++;
            dep_wait();
            const int k = atomicAdd(p.dyn_counter, 1);
            return (p.dyn_begin + k < p.dyn_end) ? p.dyn_begin + k : -1;
        };
        int cur = (u_begin < u_end) ? s_next++ : -1;
        // The first static unit and its first kHeadRefs chunk refs come from
        // the CTA's line, so its first stages are issued without waiting on
        // further plan reads.
        bool from_head = cur >= 0;
        Unit Un = (cur >= 0) ? hd->first : Unit{};
        ChunkRef chn = (cur >= 0) ? hd->refs[0] : ChunkRef{0, 0};
        // context offsets matter only under the causal mask
        int tkn = (cur >= 0 && p.causal) ? p.chunk_tok0[first_chunk(Un)] : 0;
        if (!p.kv_stable) dep_wait();
        if (cur < 0) {
            cur = claim();
            if (cur >= 0) {
                Un = p.units[cur];
                chn = p.chunks[first_chunk(Un)];
                if (p.causal) tkn = p.chunk_tok0[first_chunk(Un)];
            }
        }
        int seq = 0;
        for (; cur >= 0 && ok; ++seq) {
            const Unit U = Un;
            ring[seq % kRing] = cur;
            // The next unit (the next static one, or in the tail phase a
            // claim) is taken when two chunks of this one remain: late
            // enough not to hold queue work long, early enough to hide the
            // claim and descriptor latency (three measured slower on every
            // workload but one, level there).
            int nxt = -1;
            bool have_next = false;
            const int n = lin_n(U), base = lin_base(U);
            const int L0 = lin_begin(U), L1 = lin_end(U);
            const int claim_at = max(L0, L1 - 2);
            int h = L0 / n;
            int j = L0 - h * n;
            for (int L = L0; L < L1; ++L, ++it) {
                if (!have_next && L >= claim_at) {
                    nxt = claim();
                    if (nxt >= 0) Un = p.units[nxt];
                    have_next = true;
                }
                const ChunkRef ch = chn;
                const int tok0 = tkn;
                // the chunk's token count comes from the pool's device table
                // (appends grow partial chunks in place); the load is in
                // flight while the producer waits for the stage
                const bool slot_ok = ch.slot >= 0 && ch.slot < p.capacity;
                const int ntok = slot_ok ? p.slot_ntok[ch.slot] : 0;
                const int head = h;
                if (++j == n) { j = 0; ++h; }
                if (L + 1 < L1) {
                    chn = (from_head && L + 1 - L0 < kHeadRefs) ? hd->refs[L + 1 - L0] : p.chunks[base + j];
                    if (p.causal) tkn = p.chunk_tok0[base + j];
                } else if (nxt >= 0) {
                    chn = p.chunks[first_chunk(Un)];
                    if (p.causal) tkn = p.chunk_tok0[first_chunk(Un)];
                }
                const int st = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                if (!mbar_wait(empty0 + 8 * st, ph ^ 1u)) {
                    set_status(p.status, CA_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                const uint32_t fb = full0 + 8 * st;
                if (!slot_ok || head < 0 || head >= HK) {
                    set_status(p.status, CA_ERR_DEVICE_BOUNDS);
                    stage_ntok[st] = 0;
                    mbar_arrive(fb);          // release the consumers without data
                    continue;
                }
                // The copies go out first; the stage completes once they have
                // landed and the token count (whose load may still be in
                // flight) has been written and the producer has arrived.
                mbar_expect_tx_only(fb, SM::kStage);
                const uint32_t dst = smem_u32(stages + (size_t)st * SM::kStage);
                const int rowK = (((ch.slot * p.n_layers + p.layer) * 2 + 0) * HK + head) * C;
                const int rowV = rowK + HK * C;
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx) {
                    tma_load_2d(dst + bx * C * 128, &tmap, bx * (128 / EB), rowK, fb, pol);
                    tma_load_2d(dst + SM::kTile + bx * C * 128, &tmap, bx * (128 / EB), rowV, fb, pol);
                }
                stage_ntok[st] = min(max(ntok, 0), C);
                stage_tok0[st] = tok0;
                mbar_arrive(fb);
            }
            if (!have_next) {                 // left early on a timeout
                nxt = -1;
            }
            from_head = false;
            cur = nxt;
        }
        if (ok) {
            // end of work: one more stage, without data, carries the id -1
            const int st = it % S;
            if (mbar_wait(empty0 + 8 * st, ((uint32_t)(it / S) & 1u) ^ 1u)) {
                ring[seq % kRing] = -1;
                mbar_arrive(full0 + 8 * st);
            } else {
                set_status(p.status, CA_ERR_TIMEOUT);
                ok = false;
            }
        }
        if (!ok) {
            // Give the copies already issued a bounded chance to land before
            // the CTA can exit.
            for (int k = (it > S ? it - S : 0); k < it; ++k)
                mbar_wait(full0 + 8 * (k % S), (uint32_t)(k / S) & 1u);
        }
        return;
    }

    // ------------------------------ consumers --------------------------------
    const int w = warp;
    int it = 0;
    // Unit descriptors are held lane-distributed (lane i keeps field i) and
    // run two units ahead; query rows of sequence-first heads are fetched one
    // head ahead, so no unit or head starts on a dependent global load.
    enum { F_KIND = 0, F_HEAD, F_QLO, F_QHI, F_CB, F_CE, F_PART, F_QROW, F_N, F_BASE, F_PNEXT };
    auto load_desc = [&](int u) -> int32_t {
        return lane < kUnitInts ? reinterpret_cast<const int32_t*>(p.units + u)[lane] : 0;
    };
    auto fld = [&](int32_t d, int i) -> int32_t { return __shfl_sync(kFull, d, i); };
    auto load_q = [&](int qrow, int head) -> uint4 {
        const uint16_t* qp = p.q + ((size_t)qrow * H + head) * D + lane * DPL;
        if constexpr (DPL == 8) return *reinterpret_cast<const uint4*>(qp);
        else if constexpr (DPL == 4) {
            const uint2 v = *reinterpret_cast<const uint2*>(qp);
            return make_uint4(v.x, v.y, 0u, 0u);
        } else {
            return make_uint4(*reinterpret_cast<const uint32_t*>(qp), 0u, 0u, 0u);
        }
    };
    uint4 qn = make_uint4(0u, 0u, 0u, 0u);   // prefetched query row ...
    int qn_row = -1, qn_head = -1;        // ... and which (row, head) it is
    auto prefetch_q = [&](int qrow, int head) {
        qn = load_q(qrow, head);
        qn_row = qrow;
        qn_head = head;
    };
    auto take_q = [&](int qrow, int head) -> uint4 {
        return (qrow == qn_row && head == qn_head) ? qn : load_q(qrow, head);
    };
    // Unit ids come from the ring (the producer writes each before the
    // unit's first chunk; -1 ends the work).  Static ids are known from the
    // plan, so their descriptors and first query rows are fetched one unit
    // ahead; a queue unit's descriptor is read when its id arrives.
    const int n_static = u_end - u_begin;
    int32_t dn = (n_static > 0) ? load_desc(u_begin) : 0;   // descriptor of unit `seq`
    asm volatile("griddepcontrol.wait;" ::: "memory");     // q and the pool after this
    if (n_static > 0 && fld(dn, F_KIND) == UNIT_SF) prefetch_q(fld(dn, F_QROW), fld(dn, F_HEAD));
    int flush = 0;                        // sequence-first partials written (exchange parity)
    for (int seq = 0;; ++seq) {
        // The unit's first stage (or the closing one) carries its id.
        if (!mbar_wait(full0 + 8 * (it % S), (uint32_t)(it / S) & 1u)) {
            set_status(p.status, CA_ERR_TIMEOUT);
            return;
        }
        const int cur = ring[seq % kRing];
        if (cur < 0) break;
        const int32_t dc = (seq < n_static) ? dn : load_desc(cur);
        // the next unit, when it is static: its descriptor now, its query later
        const bool next_static = seq + 1 < n_static;
        if (next_static) dn = load_desc(u_begin + seq + 1);
        const int32_t d0 = dn;
        const bool next_sf = next_static && fld(d0, F_KIND) == UNIT_SF;
        consumer_sync();   // previous unit (and its exchange reads) finished
        if (!kRows && fld(dc, F_KIND) == UNIT_SF && G == 1 && QL == 1) {
            const int pos = fld(dc, F_QLO), n = fld(dc, F_N), base = fld(dc, F_BASE);
            const int qrow = fld(dc, F_QROW), c_end = fld(dc, F_CE), part_next = fld(dc, F_PNEXT);
            int L = fld(dc, F_CB), h = fld(dc, F_HEAD), part = fld(dc, F_PART);
            while (L < c_end) {                   // one head's piece at a time
                const int seg_end = min(c_end, (h + 1) * n);
                const uint4 qraw = take_q(qrow, h);
                if (seg_end < c_end) prefetch_q(qrow, h + 1);
                else if (next_sf) prefetch_q(fld(d0, F_QROW), fld(d0, F_HEAD));
                float* xo = reinterpret_cast<float*>(qreg) + (flush & 1) * kConsumerWarps * D;
                float* xm = xms + (flush & 1) * 2 * kConsumerWarps;
                float m = -INFINITY, s = 0.f;
                if constexpr (kF8Tc) {
                    // The query in fragment order: lane L holds dims 4L .. 4L + 3,
                    // step kk wants dims 16kk + 4t .. + 3, i.e. lane 4kk + t's.
                    uint32_t qb[8][2];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        qb[kk][0] = __shfl_sync(kFull, qraw.x, 4 * kk + (lane & 3));
                        qb[kk][1] = __shfl_sync(kFull, qraw.y, 4 * kk + (lane & 3));
                    }
                    float oc[8][4];
#pragma unroll
                    for (int mb = 0; mb < 8; ++mb) oc[mb][0] = oc[mb][1] = oc[mb][2] = oc[mb][3] = 0.f;
                    for (; L < seg_end; ++L, ++it) {
                        const int st = it % S;
                        if (!mbar_wait(full0 + 8 * st, (uint32_t)(it / S) & 1u)) {
                            set_status(p.status, CA_ERR_TIMEOUT);
                            return;
                        }
                        const int ntok = stage_ntok[st];
                        const uint8_t* kt = stages + (size_t)st * SM::kStage;
                        sf_chunk_f8_tc(kt, kt + SM::kTile, ntok, qb, p.scale_log2, m, s, oc, w, lane);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(empty0 + 8 * st);
                    }
                    // lane (g, 0) holds dims 32qd + 4g .. + 3 (see sf_chunk_f8_tc)
                    if ((lane & 3) == 0) {
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd)
                            *reinterpret_cast<float4*>(xo + w * D + 32 * qd + 4 * (lane >> 2)) =
                                make_float4(oc[2 * qd][0], oc[2 * qd][2], oc[2 * qd + 1][0], oc[2 * qd + 1][2]);
                    }
                } else {
                    float q[DPL], o[DPL];
                    {
                        const uint32_t qw[4] = {qraw.x, qraw.y, qraw.z, qraw.w};
#pragma unroll
                        for (int i = 0; i < DPL / 2; ++i) {
                            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&qw[i]));
                            q[2 * i] = a.x;
                            q[2 * i + 1] = a.y;
                        }
#pragma unroll
                        for (int d = 0; d < DPL; ++d) { q[d] *= p.scale_log2; o[d] = 0.f; }
                    }
                    for (; L < seg_end; ++L, ++it) {
                        const int st = it % S;
                        if (!mbar_wait(full0 + 8 * st, (uint32_t)(it / S) & 1u)) {
                            set_status(p.status, CA_ERR_TIMEOUT);
                            return;
                        }
                        const int ntok = stage_ntok[st];
                        const uint8_t* kt = stages + (size_t)st * SM::kStage;
                        sf_chunk<C, D, EB>(kt, kt + SM::kTile, ntok, q, m, s, o, w, lane);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(empty0 + 8 * st);
                    }
#pragma unroll
                    for (int d = 0; d < DPL; ++d) xo[w * D + lane * DPL + d] = o[d];
                }
                // Combine the four warps' states and write the partial.  The
                // exchange area alternates between two halves, so the next
                // head's writes never meet this head's reads.
                if (lane == 0) { xm[2 * w] = m; xm[2 * w + 1] = s; }
                consumer_sync();
                if (w == 0) {
                    float M = -INFINITY;
#pragma unroll
                    for (int v = 0; v < kConsumerWarps; ++v) M = fmaxf(M, xm[2 * v]);
                    float acc[DPL], sum = 0.f;
#pragma unroll
                    for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
#pragma unroll
                    for (int v = 0; v < kConsumerWarps; ++v) {
                        const float mv = xm[2 * v];
                        const float wt = (mv == -INFINITY) ? 0.f : ex2(mv - M);
                        sum += wt * xm[2 * v + 1];
#pragma unroll
                        for (int d = 0; d < DPL; ++d) acc[d] += wt * xo[v * D + lane * DPL + d];
                    }
                    const int pid = p.pbase[pos * H + h] + part;
                    st_f<DPL>(p.part_o + (size_t)pid * D + lane * DPL, acc);
                    if (lane == 0) p.part_ms[pid] = make_float2(M, sum);
                }
                ++flush;
                ++h;
                part = part_next;
            }
        } else {
            // ------------------------- tensor-core path -------------------------
            // Chunk-first units, and sequence-first units when a position has
            // several query rows per key/value head (grouped query heads or
            // several query tokens).  Rows of the query tile are (position,
            // query token, query head): row r is position q_lo + r / RW, token
            // (r % RW) / G, query head kvh * G + r % G.  The unit is walked as
            // its linear (key/value head, chunk) range, one head's piece at a
            // time.
            const bool is_sf = fld(dc, F_KIND) == UNIT_SF;
            const int q_lo = fld(dc, F_QLO), q_hi = fld(dc, F_QHI);
            const int cb = fld(dc, F_CB), ce = fld(dc, F_CE);
            const int n = is_sf ? fld(dc, F_N) : ce - cb;
            const int base = is_sf ? fld(dc, F_BASE) : cb;
            int L = is_sf ? cb : fld(dc, F_HEAD) * n;
            const int L_end = is_sf ? ce : (fld(dc, F_HEAD) + fld(dc, F_N)) * n;
            const int part_first = fld(dc, F_PART), part_rest = is_sf ? fld(dc, F_PNEXT) : part_first;
            if (next_sf) prefetch_q(fld(d0, F_QROW), fld(d0, F_HEAD));
            const int m_rows = (q_hi - q_lo) * RW;
            const int rblocks = m_rows <= 16 ? 1 : m_rows <= 32 ? 2 : 4;
            // head_dim 256: warp pairs split the head dims (at most 32 rows)
            constexpr bool kSplit = D == 256;
            constexpr int OD = kSplit ? 128 : D;          // output dims per warp
            int T = kSplit ? 1 : kConsumerWarps / rblocks;   // warps splitting a chunk's tokens
            if (T * 16 > C) T = C / 16;
            const int rb = kSplit ? (w >> 1) : w / T, tp = kSplit ? 0 : w % T;
            const int dhalf = kSplit ? (w & 1) : 0;
            const bool active = rb < rblocks && rb * 16 < m_rows;
            // Causal mask: the last context token each of this thread's two
            // rows (rb*16 + lane/4 and 8 below) may see; the rows are the same
            // for every head of the unit.
            int lim[2] = {INT_MAX, INT_MAX};
            if (p.causal) {
#pragma unroll
                for (int r2 = 0; r2 < 2; ++r2) {
                    const int row = rb * 16 + (lane >> 2) + 8 * r2;
                    if (row < m_rows) lim[r2] = p.ctx_len[q_lo + row / RW] - QL + (row % RW) / G;
                }
            }
            if (kRows && !kSplit && is_sf && m_rows <= 8) {
                // a sequence-first position with at most 8 query rows:
                // the products transposed (sf_rows_transposed)
                if (!sf_rows_transposed<C, D, EB>(p, stages, conv, qreg, xms, full0, empty0, stage_ntok,
                                                  stage_tok0, S, it, L, L_end, n, q_lo, m_rows, part_first,
                                                  part_rest, w, lane))
                    return;
            } else {
            for (bool first = true; L < L_end; first = false) {
                const int kvh = L / n;
                const int seg_end = min(L_end, (kvh + 1) * n);
                const int upart = first ? part_first : part_rest;
                if (!first) consumer_sync();   // the previous head's exchange reads are done
                // Copy the rows' queries into the swizzled Q tile with 16-byte
                // asynchronous copies, all in flight at once.  Rows past m_rows
                // are left as they are: each mma row is independent and such
                // rows are never written out.
                for (int idx = threadIdx.x; idx < m_rows * (D / 8); idx += kConsumerWarps * 32) {
                    const int r = idx / (D / 8), k = idx % (D / 8);
                    const size_t qrow_tok = (size_t)p.seq_perm[q_lo + r / RW] * QL + (r % RW) / G;
                    const uint16_t* src = p.q + (qrow_tok * H + kvh * G + r % G) * D + k * 8;
                    cp_async16(smem_u32(qreg + swz(r, k, q_rows<D>())), src);
                }
                cp_async_wait_all();
                consumer_sync();
                float o[OD / 8][4], m[2] = {-INFINITY, -INFINITY}, s[2] = {0.f, 0.f};
#pragma unroll
                for (int dt = 0; dt < OD / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
                // Row block rb starts at a multiple of 8 rows, so its swizzle
                // pattern is the tile's shifted by rb * 16 rows of 128 bytes.
                const uint32_t qblock = smem_u32(qreg) + rb * 16 * 128;
                const int NTw = C / T;
                for (; L < seg_end; ++L, ++it) {
                    const int st = it % S;
                    if (!mbar_wait(full0 + 8 * st, (uint32_t)(it / S) & 1u)) {
                        set_status(p.status, CA_ERR_TIMEOUT);
                        return;
                    }
                    uint32_t kt = smem_u32(stages + (size_t)st * SM::kStage);
                    uint32_t vt = kt + SM::kTile;
                    const int ntok = stage_ntok[st];
                    const int ctx0 = stage_tok0[st];
                    // an fp8 stage is read as E4M3 bytes, straight into the
                    // fragments (cf_chunk<..., true>)
                    if constexpr (kSplit) {
                        if (active) {
                            constexpr int kXs = (C / 8) * 4 * 32;     // floats per warp slot
                            float* xw = xs + ((it & 1) * kConsumerWarps + w) * kXs;
                            const float* xp = xs + ((it & 1) * kConsumerWarps + (w ^ 1)) * kXs;
                            cf_chunk_split<C, C>(kt, vt, ntok, 0, ctx0, lim[0], lim[1], qblock, p.scale_log2,
                                                 dhalf, xw, xp, 2 + rb, m, s, o, lane);
                        }
                    } else if (active) {
                        if (NTw == 16) {
                            cf_chunk<C, D, 16, EB == 1>(kt, vt, ntok, tp * 16, ctx0, lim[0], lim[1], qblock,
                                                        p.scale_log2, m, s, o, lane);
                        } else if constexpr (C >= 32) {
                            // 32 tokens at a time keeps the score tile in registers
                            for (int t0 = tp * NTw; t0 < (tp + 1) * NTw; t0 += 32)
                                cf_chunk<C, D, 32, EB == 1>(kt, vt, ntok, t0, ctx0, lim[0], lim[1], qblock,
                                                            p.scale_log2, m, s, o, lane);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty0 + 8 * st);
                }
                // Row sums are per thread so far: reduce over the quad.
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    s[r] += __shfl_xor_sync(kFull, s[r], 1);
                    s[r] += __shfl_xor_sync(kFull, s[r], 2);
                }
                // Tree-combine the T warps that split the tokens of one row block,
                // through the (now free) Q tile: round `half` moves warps with
                // tp in [half, 2*half) onto tp - half.
                float* xo = reinterpret_cast<float*>(qreg);
                for (int half = T / 2; half >= 1; half /= 2) {
                    consumer_sync();
                    const bool writer = active && tp >= half && tp < 2 * half;
                    const int slot = rb * (T / 2) + (tp - half);    // < 2 writers per round
                    if (writer) {
                        float* dst = xo + (size_t)slot * (16 * D);
#pragma unroll
                        for (int dt = 0; dt < OD / 8; ++dt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) dst[(dt * 4 + e) * 32 + lane] = o[dt][e];
                        if ((lane & 3) == 0) {
                            const int g = lane >> 2;
                            xms[slot * 64 + g * 4 + 0] = m[0];
                            xms[slot * 64 + g * 4 + 1] = s[0];
                            xms[slot * 64 + g * 4 + 2] = m[1];
                            xms[slot * 64 + g * 4 + 3] = s[1];
                        }
                    }
                    consumer_sync();
                    if (active && tp < half) {
                        const int src = rb * (T / 2) + tp;
                        const float* so = xo + (size_t)src * (16 * D);
                        const int g = lane >> 2;
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const float m2 = xms[src * 64 + g * 4 + 2 * r];
                            const float s2 = xms[src * 64 + g * 4 + 2 * r + 1];
                            const float M = fmaxf(m[r], m2);
                            const float Mu = (M == -INFINITY) ? 0.f : M;
                            const float a1 = ex2(m[r] - Mu), a2 = ex2(m2 - Mu);
                            s[r] = s[r] * a1 + s2 * a2;
                            m[r] = M;
#pragma unroll
                            for (int dt = 0; dt < OD / 8; ++dt) {
                                o[dt][2 * r] = o[dt][2 * r] * a1 + so[(dt * 4 + 2 * r) * 32 + lane] * a2;
                                o[dt][2 * r + 1] =
                                    o[dt][2 * r + 1] * a1 + so[(dt * 4 + 2 * r + 1) * 32 + lane] * a2;
                            }
                        }
                    }
                }
                // Warps with tp == 0 now hold their row block (at head_dim 256,
                // each warp of a pair its half of the dims): write one partial
                // per valid row.
                if (active && tp == 0) {
                    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int row = rb * 16 + g + 8 * r;
                        if (row < m_rows) {
                            const int pos = q_lo + row / RW, jq = (row % RW) / G, qh = kvh * G + row % G;
                            const int pid = p.pbase[((size_t)pos * QL + jq) * H + qh] + upart;
                            float* dst = p.part_o + (size_t)pid * D + dhalf * OD;
                            if constexpr (EB == 1) {
                                // o[4dq + i][2r + c] holds dim 32dq + 8t + 4c + i
#pragma unroll
                                for (int dq = 0; dq < OD / 32; ++dq) {
                                    *reinterpret_cast<float4*>(dst + 32 * dq + 8 * t4) =
                                        make_float4(o[4 * dq][2 * r], o[4 * dq + 1][2 * r], o[4 * dq + 2][2 * r],
                                                    o[4 * dq + 3][2 * r]);
                                    *reinterpret_cast<float4*>(dst + 32 * dq + 8 * t4 + 4) =
                                        make_float4(o[4 * dq][2 * r + 1], o[4 * dq + 1][2 * r + 1],
                                                    o[4 * dq + 2][2 * r + 1], o[4 * dq + 3][2 * r + 1]);
                                }
                            } else {
#pragma unroll
                                for (int dt = 0; dt < OD / 8; ++dt)
                                    *reinterpret_cast<float2*>(dst + dt * 8 + 2 * t4) =
                                        make_float2(o[dt][2 * r], o[dt][2 * r + 1]);
                            }
                            if (t4 == 0 && dhalf == 0) p.part_ms[pid] = make_float2(m[r], s[r]);
                        }
                    }
                }
            }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// KV scatter for inserts: each listed chunk copies rows [src_row, src_row +
// n_rows) of k/v [L][total_rows][H][D] into rows [0, n_rows) of its slot's
// K and V tiles.  One CTA per (chunk, layer); 16-byte vectors.
// ---------------------------------------------------------------------------
constexpr int kScatterMaxChunks = 128;    // chunks per launch (small parameter block)
struct ScatterArgs {
    const uint4* k;
    const uint4* v;
    void* pool;
    int32_t* slot_ntok;
    int32_t total_rows, chunk, n_layers, n_heads, vec_per_row, n_chunks;
    float inv_k, inv_v;                   // fp8 pools: 1 / scale (fp32)
    ScatterChunk ch[kScatterMaxChunks];
};

// One CTA per (chunk, layer, head): a c x D tile of K and one of V, eight
// elements per step.  An fp8 pool stores E4M3(fp32(x) * inv_scale).  A chunk
// written from its first row (a new chunk) gets zeros in the rows past its
// tokens: the kernels give those rows weight 0, which must not meet a NaN.
template <bool F8>
__global__ void __launch_bounds__(256) kv_scatter_kernel(const __grid_constant__ ScatterArgs a) {
    const int h = blockIdx.x % a.n_heads;
    const int rest = blockIdx.x / a.n_heads;
    const int ci = rest % a.n_chunks, l = rest / a.n_chunks;
    const ScatterChunk c = a.ch[ci];
    const int total = (c.dst_row == 0 ? a.chunk : c.n_rows) * a.vec_per_row;
    if (h == 0 && l == 0 && threadIdx.x == 0) a.slot_ntok[c.slot] = c.dst_row + c.n_rows;
    const long long tile = ((((long long)c.slot * a.n_layers + l) * 2 * a.n_heads + h) * a.chunk +
                            c.dst_row) * a.vec_per_row;
    const long long vtile = tile + (long long)a.n_heads * a.chunk * a.vec_per_row;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int r = i / a.vec_per_row, vec = i % a.vec_per_row;
        if (r >= c.n_rows) {                     // past the tokens of a new chunk
            if constexpr (F8) {
                static_cast<uint2*>(a.pool)[tile + i] = make_uint2(0u, 0u);
                static_cast<uint2*>(a.pool)[vtile + i] = make_uint2(0u, 0u);
            } else {
                static_cast<uint4*>(a.pool)[tile + i] = make_uint4(0u, 0u, 0u, 0u);
                static_cast<uint4*>(a.pool)[vtile + i] = make_uint4(0u, 0u, 0u, 0u);
            }
            continue;
        }
        const long long src = (((long long)l * a.total_rows + c.src_row + r) * a.n_heads + h) * a.vec_per_row + vec;
        if constexpr (F8) {
            auto pack = [](const uint4 x, float inv) {
                const __half2* hp = reinterpret_cast<const __half2*>(&x);
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __half22float2(hp[k]);
                    w[k] = e4m3x2_from_f32(f.x * inv, f.y * inv);
                }
                return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
            };
            uint2* pool = static_cast<uint2*>(a.pool);
            pool[tile + i] = pack(a.k[src], a.inv_k);
            pool[vtile + i] = pack(a.v[src], a.inv_v);
        } else {
            uint4* pool = static_cast<uint4*>(a.pool);
            pool[tile + i] = a.k[src];
            pool[vtile + i] = a.v[src];
        }
    }
}

}  // namespace dev

// ---------------------------------------------------------------------------
// Host launchers.
// ---------------------------------------------------------------------------
namespace {
template <int C, int D, int EB, bool R>
void* kernel_ptr() {
    return reinterpret_cast<void*>(&dev::two_phase_attention_kernel<C, D, EB, R>);
}
template <int C, int D, int EB>
void* kernel_ptr(bool rows) {
    if constexpr (D <= 128) {
        if (rows) return kernel_ptr<C, D, EB, true>();
    }
    return kernel_ptr<C, D, EB, false>();
}
// rows: the schedule brings 2..8 query rows per position and key/value head
// (the few-row variant exists for head_dim <= 128).
void* pick_kernel(const PoolCfg& c, bool rows = false) {
    if (kv_elem_bytes(c) == 1) {
        if (c.head_dim != 128) return nullptr;
        if (c.chunk == 64) return kernel_ptr<64, 128, 1>(rows);
        if (c.chunk == 32) return kernel_ptr<32, 128, 1>(rows);
        if (c.chunk == 16) return kernel_ptr<16, 128, 1>(rows);
    } else if (c.head_dim == 256) {                 // chunks of 16 or 32 tokens
        if (c.chunk == 32) return kernel_ptr<32, 256, 2>(false);
        if (c.chunk == 16) return kernel_ptr<16, 256, 2>(false);
    } else if (c.head_dim == 128) {
        if (c.chunk == 64) return kernel_ptr<64, 128, 2>(rows);
        if (c.chunk == 32) return kernel_ptr<32, 128, 2>(rows);
        if (c.chunk == 16) return kernel_ptr<16, 128, 2>(rows);
    } else if (c.head_dim == 64) {
        if (c.chunk == 64) return kernel_ptr<64, 64, 2>(rows);
        if (c.chunk == 32) return kernel_ptr<32, 64, 2>(rows);
        if (c.chunk == 16) return kernel_ptr<16, 64, 2>(rows);
    }
    return nullptr;
}
// The kernel's dynamic shared memory (the Smem map above, computed here).
size_t smem_for(const PoolCfg& c, int stages) {
    const size_t eb = (size_t)kv_elem_bytes(c), cd = (size_t)c.chunk * c.head_dim;
    const size_t conv = eb == 1 ? 2 * cd * 2 : 0;
    const size_t qrows = c.head_dim == 256 ? 32 : dev::kQRows;
    const size_t xs = c.head_dim == 256 ? (size_t)2 * dev::kConsumerWarps * (c.chunk / 8) * 4 * 32 * 4 : 0;
    return (size_t)stages * 2 * cd * eb + conv + xs + qrows * c.head_dim * 2 + 512 +
           2 * dev::kMaxStages * 8 + 4 * dev::kRing + 2 * 4 * dev::kMaxStages;
}
}  // namespace

// Stages that fit two CTAs per SM (113 KiB each, at most 8).
int kernel_smem_bytes(const PoolCfg& c, int* n_stages, size_t* bytes) {
    if (!pick_kernel(c)) return CA_ERR_UNSUPPORTED;
    const size_t budget = 113 * 1024;
    int st = dev::kMaxStages;
    while (st > 1 && smem_for(c, st) > budget) --st;
    *n_stages = st;
    *bytes = smem_for(c, st);
    return CA_OK;
}

int kernel_ctas_per_sm(const PoolCfg& c, int* ctas) {
    void* fn = pick_kernel(c);
    if (!fn) return CA_ERR_UNSUPPORTED;
    int st;
    size_t bytes;
    kernel_smem_bytes(c, &st, &bytes);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return CA_ERR_CUDA;
    // the few-row variant takes the same shared memory (and, by its launch
    // bounds, the same two CTAs per SM)
    void* fr = pick_kernel(c, true);
    if (fr != fn && cudaFuncSetAttribute(fr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return CA_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, dev::kThreads, bytes) != cudaSuccess)
        return CA_ERR_CUDA;
    *ctas = n < 1 ? 1 : n;
    return CA_OK;
}

int make_tensor_map(Pool& p) {
    using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return CA_ERR_CUDA;
    const PoolCfg& c = p.cfg;
    // The pool as a 2-D tensor: rows of head_dim elements (fp16, or bytes for
    // an fp8 pool), one row per (slot, layer, K|V, head, token-in-chunk);
    // boxes of 128 bytes x c rows.
    const int eb = kv_elem_bytes(c);
    const cuuint64_t rows = (cuuint64_t)c.capacity_slots * c.n_layers * 2 * kv_heads(c) * c.chunk;
    const cuuint64_t dims[2] = {(cuuint64_t)c.head_dim, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)c.head_dim * eb};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / eb), (cuuint32_t)c.chunk};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap* map = reinterpret_cast<CUtensorMap*>(p.tmap);
    CUresult r = reinterpret_cast<EncodeFn>(fn)(
        map, eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.kv, dims, strides,
        box, estr,
        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? CA_OK : CA_ERR_CUDA;
}

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

uint64_t kernel_launches() { return g_launches.load(std::memory_order_relaxed); }

int launch_scatter(const Pool& p, const void* k, const void* v, int32_t total_rows,
                   const std::vector<ScatterChunk>& chunks, void* stream) {
    const PoolCfg& c = p.cfg;
    p.kv_written = true;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess) return CA_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) p.captured_writes = true;
    for (size_t i = 0; i < chunks.size(); i += dev::kScatterMaxChunks) {
        const size_t cnt = std::min<size_t>(dev::kScatterMaxChunks, chunks.size() - i);
        dev::ScatterArgs a;
        a.k = static_cast<const uint4*>(k);
        a.v = static_cast<const uint4*>(v);
        a.pool = p.kv;
        a.slot_ntok = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(p.kv) + pool_tile_bytes(c));
        a.total_rows = total_rows;
        a.chunk = c.chunk;
        a.n_layers = c.n_layers;
        a.n_heads = kv_heads(c);
        a.vec_per_row = c.head_dim / 8;
        a.n_chunks = (int32_t)cnt;
        a.inv_k = 1.f / kv_scale_of(c.k_scale);
        a.inv_v = 1.f / kv_scale_of(c.v_scale);
        std::copy(chunks.begin() + i, chunks.begin() + i + cnt, a.ch);
        const unsigned blocks = (unsigned)(cnt * c.n_layers * a.n_heads);
        if (kv_elem_bytes(c) == 1)
            dev::kv_scatter_kernel<true><<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
        else
            dev::kv_scatter_kernel<false><<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
        if (cudaGetLastError() != cudaSuccess) return CA_ERR_CUDA;
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    return CA_OK;
}

int launch_attention(const Pool& p, const Sched& s, const AttnParams& prm, void* stream) {
    // positions with 2..8 query rows per key/value head: the few-row variant
    const int rw = s.q_len * (p.cfg.n_heads / kv_heads(p.cfg));
    void* fn = pick_kernel(p.cfg, rw >= 2 && rw <= 8);
    if (!fn) return CA_ERR_UNSUPPORTED;
    int st;
    size_t bytes;
    kernel_smem_bytes(p.cfg, &st, &bytes);   // attribute set at pool creation
    AttnParams a = prm;
    a.n_stages = st;
    // The kernel may read the pool before its dependency wait only when no
    // KV scatter was launched since the last attention launch: every kernel
    // this launch can overlap then leaves the pool alone.  Under stream
    // capture, the first attention call a graph records for this pool may
    // follow anything when the graph is replayed, so it waits; and once a
    // scatter has been recorded into a graph, the host no longer knows when
    // the pool is written, so uncaptured calls always wait.
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    unsigned long long cap_id = 0;
    if (cudaStreamGetCaptureInfo(cs, &cap, &cap_id) != cudaSuccess) return CA_ERR_CUDA;
    bool stable = !p.kv_written;
    if (cap == cudaStreamCaptureStatusActive) {
        if (p.capture_id != cap_id) stable = false;
        p.capture_id = cap_id;
    } else if (cap != cudaStreamCaptureStatusNone) {
        return CA_ERR_CUDA;                       // an invalidated capture
    } else if (p.captured_writes) {
        stable = false;
    }
    a.kv_stable = stable ? 1 : 0;
    a.test_stall = 0;
    if (s.stall_calls > 0) {
        a.test_stall = 1;
        --s.stall_calls;
    }
    p.kv_written = false;
    const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(p.tmap);
    void* args[] = {const_cast<CUtensorMap*>(map), &a};
    // Both kernels are programmatic dependents of whatever precedes them in
    // the stream: their launch overlaps the previous kernel's tail and each
    // waits (griddepcontrol.wait) before touching data that kernel may write.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t mc = {};
    mc.gridDim = dim3((unsigned)s.plan.grid);
    mc.blockDim = dim3(dev::kThreads);
    mc.dynamicSmemBytes = bytes;
    mc.stream = cs;
    mc.attrs = attr;
    mc.numAttrs = 1;
    if (s.ev_begin) cudaEventRecord(static_cast<cudaEvent_t>(s.ev_begin), cs);
    cudaError_t e = cudaLaunchKernelExC(&mc, fn, args);
    if (s.ev_end) cudaEventRecord(static_cast<cudaEvent_t>(s.ev_end), cs);
    if (e != cudaSuccess) return CA_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    // Merge: one warp per (position, head).
    const int n_pairs = s.t.b * s.q_len * p.cfg.n_heads;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((n_pairs + dev::kMergeWarps - 1) / dev::kMergeWarps));
    lc.blockDim = dim3(dev::kMergeWarps * 32);
    lc.dynamicSmemBytes = 0;
    lc.stream = cs;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (p.cfg.head_dim == 256)
        e = cudaLaunchKernelEx(&lc, dev::merge_partials_kernel<256>, a, n_pairs);
    else if (p.cfg.head_dim == 128)
        e = cudaLaunchKernelEx(&lc, dev::merge_partials_kernel<128>, a, n_pairs);
    else
        e = cudaLaunchKernelEx(&lc, dev::merge_partials_kernel<64>, a, n_pairs);
    if (e != cudaSuccess) {
        cudaMemsetAsync(a.dyn_counter, 0, sizeof(int32_t), cs);   // keep the next call's queue clean
        return CA_ERR_CUDA;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return CA_OK;
}

}  // namespace ca
