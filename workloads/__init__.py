"""Seeded synthetic inputs for prefix-shared decode attention.

This module only draws numbers and lays out token segments.  It holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle may take
their inputs from it without sharing any of the method.

A workload is a set of token *segments* (a shared system prompt, a branch
segment, a private suffix) and a list of sequences, each an ordered list of
segment ids.  Every segment draws its token ids from its own id range, so two
sequences share a prefix exactly when they list the same leading segments
(ChunkAttention, §3.1: sharing requires the common prompt at the start of the
sequence).  The K/V rows of a segment are drawn once from a generator keyed by
(workload seed, segment id), so identical prefixes carry identical K/V, which
is what a prefix-aware cache assumes when it keeps the first inserter's rows.

Values: Q, K, V are i.i.d. N(0, 1) drawn in float32 by numpy's PCG64 and
rounded to float16 (round-to-nearest-even).  Layouts: K/V of a segment are
[L, n, H, D]; queries of a step are [b, H, D].
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

TOKEN_ID_STRIDE = 1 << 16  # token ids of segment s are s * stride + [0, n)


def segment_tokens(seg_id: int, n: int) -> np.ndarray:
    """Token ids of segment ``seg_id``: a range no other segment uses."""
    if n >= TOKEN_ID_STRIDE or seg_id >= (1 << 15):
        raise ValueError("segment too long or id out of range")
    return (np.arange(n, dtype=np.int64) + seg_id * TOKEN_ID_STRIDE).astype(np.int32)


def segment_kv(seed: int, seg_id: int, n: int, n_layers: int, n_heads: int,
               head_dim: int) -> tuple[np.ndarray, np.ndarray]:
    """K and V rows of one segment, float16 [L, n, H, D], N(0, 1)."""
    rng = np.random.default_rng([seed, 1, seg_id])
    shape = (n_layers, n, n_heads, head_dim)
    k = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    v = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    return k, v


def step_queries(seed: int, step: int, b: int, n_heads: int, head_dim: int,
                 layer: int = 0, q_len: int = 1) -> np.ndarray:
    """Decode queries of one step, float16 [b, H, D] ([b, q_len, H, D] for
    several query tokens per sequence), N(0, 1)."""
    rng = np.random.default_rng([seed, 2, step, layer])
    shape = (b, n_heads, head_dim) if q_len == 1 else (b, q_len, n_heads, head_dim)
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


@dataclass
class Workload:
    """A prefix tree of token segments plus the sequences that walk it."""
    name: str
    n_layers: int
    n_heads: int
    head_dim: int
    chunk: int
    seed: int
    n_kv_heads: int = 0            # key/value heads (0: one per query head)
    kv_dtype: str = "fp16"         # pool storage: "fp16", or "fp8" (E4M3, scales 1)
    q_len: int = 1                 # query tokens per sequence (> 1: causal, the last q_len tokens)
    seg_len: dict[int, int] = field(default_factory=dict)
    seqs: dict[int, list[int]] = field(default_factory=dict)  # seq_id -> segment ids
    churn: int = 0  # sequences removed and inserted per step (multi-tenant tree)
    description: str = ""
    _kv_cache: dict = field(default_factory=dict, repr=False)
    _rng_state: object = field(default=None, repr=False)
    _next_seg: int = 0
    _next_seq: int = 0
    _slots_of: dict = field(default_factory=dict, repr=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def kv_heads(self) -> int:
        return self.n_kv_heads or self.n_heads

    def seq_ids(self) -> list[int]:
        return sorted(self.seqs)

    def seq_len(self, seq_id: int) -> int:
        return sum(self.seg_len[s] for s in self.seqs[seq_id])

    def tokens(self, seq_id: int) -> np.ndarray:
        return np.concatenate([segment_tokens(s, self.seg_len[s]) for s in self.seqs[seq_id]])

    def segment(self, seg_id: int) -> tuple[np.ndarray, np.ndarray]:
        if seg_id not in self._kv_cache:
            self._kv_cache[seg_id] = segment_kv(self.seed, seg_id, self.seg_len[seg_id],
                                                self.n_layers, self.kv_heads, self.head_dim)
        return self._kv_cache[seg_id]

    def kv_rows(self, seq_id: int, start: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """K/V [L, n - start, H, D] of the sequence's tokens from ``start`` on."""
        ks, vs, pos = [], [], 0
        for s in self.seqs[seq_id]:
            n = self.seg_len[s]
            if pos + n > start:
                k, v = self.segment(s)
                a = max(0, start - pos)
                ks.append(k[:, a:])
                vs.append(v[:, a:])
            pos += n
        if not ks:
            shape = (self.n_layers, 0, self.kv_heads, self.head_dim)
            return np.zeros(shape, np.float16), np.zeros(shape, np.float16)
        return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1)

    def queries(self, step: int, b: int | None = None, layer: int = 0) -> np.ndarray:
        return step_queries(self.seed, step, len(self.seqs) if b is None else b,
                            self.n_heads, self.head_dim, layer, self.q_len)

    def unique_tokens(self) -> int:
        """Tokens of the distinct segments the live sequences use."""
        used = {s for segs in self.seqs.values() for s in segs}
        return sum(self.seg_len[s] for s in used)

    # -- multi-tenant churn -------------------------------------------------
    def _new_seg(self, n: int) -> int:
        sid = self._next_seg
        self._next_seg += 1
        self.seg_len[sid] = n
        return sid

    def churn_step(self) -> tuple[list[int], list[int]]:
        """Remove ``churn`` live sequences chosen uniformly and insert as many
        new ones into the freed (tenant, branch) positions, each with a fresh
        private suffix.  Returns (removed seq ids, inserted seq ids)."""
        rng = self._rng_state
        live = sorted(self.seqs)
        pick = sorted(rng.choice(len(live), size=self.churn, replace=False).tolist())
        removed = [live[i] for i in pick]
        inserted = []
        for sid in removed:
            segs = self.seqs.pop(sid)
            self._kv_cache.pop(segs[-1], None)
            plen = int(rng.integers(256, 1024, endpoint=True))
            new_id = self._next_seq
            self._next_seq += 1
            self.seqs[new_id] = segs[:-1] + [self._new_seg(plen)]
            inserted.append(new_id)
        return removed, inserted


def _shared_prefix(name, seed, b, n_shared, n_private, n_heads=32, head_dim=128,
                   chunk=64, description="", n_kv_heads=0) -> Workload:
    w = Workload(name, 1, n_heads, head_dim, chunk, seed, description=description,
                 n_kv_heads=n_kv_heads)
    if n_shared:
        pre = w._new_seg(n_shared)
    for i in range(b):
        segs = ([pre] if n_shared else []) + [w._new_seg(n_private)]
        w.seqs[i] = segs
    w._next_seq = b
    return w


def _multi_tenant(seed: int) -> Workload:
    w = Workload("multi_tenant", 1, 32, 128, 64, seed, churn=8,
                 description="4 tenants x 2048-token prompt, 2 branches x 256 shared "
                             "tokens each, 8 sequences per branch, private suffix "
                             "U{256..1024}; per step 8 removed and 8 inserted")
    rng = np.random.default_rng([seed, 3])
    w._rng_state = rng
    sid = 0
    for t in range(4):
        prompt = w._new_seg(2048)
        for br in range(2):
            branch = w._new_seg(256)
            for _ in range(8):
                plen = int(rng.integers(256, 1024, endpoint=True))
                w.seqs[sid] = [prompt, branch, w._new_seg(plen)]
                sid += 1
    w._next_seq = sid
    return w


def make(name: str) -> Workload:
    """The synthetic workloads, by name.

    tiny            1 layer, 2 heads, head_dim 64, chunk 16; a 64-token shared
                    prefix and 4 sequences with 16 private tokens each; seed 0.
    llama7b_p1024   32 heads, head_dim 128, chunk 64; 32 sequences sharing a
                    1024-token prefix, 512 private tokens each; seed 1.
    sweep_s{2048,4096}_b{32,64}
                    the same layer with a 2048- or 4096-token shared prefix and
                    batch 32 or 64, 512 private tokens each; seeds 2-5.
    no_sharing      32 sequences with fully private 2048-token contexts; seed 6.
    multi_tenant    the multi-tenant tree with churn; seed 7.
    gqa_p1024       llama7b_p1024's tree with grouped-query attention: 32 query
                    heads over 8 key/value heads; seed 8.
    llama7b_p1024_fp8, sweep_s4096_b64_fp8
                    those trees (same seeds) in a pool that stores K/V as FP8
                    E4M3 with scales 1 (the inputs stay fp16 N(0, 1)).
    d256_p1024      head_dim 256: 16 heads, chunk 32, llama7b_p1024's tree
                    shape (same KV bytes per token); seed 9.
    llama7b_p1024_q4
                    llama7b_p1024 with 4 query tokens per sequence (draft
                    tokens being verified): causal, token j sees the context
                    up to its own position, the last 4 tokens.
    """
    if name.endswith("_q4"):
        w = make(name[:-3])
        w.name, w.q_len = name, 4
        w.description += "; 4 query tokens per sequence under the causal mask (the last 4 context tokens)"
        return w
    if name.endswith("_fp8"):
        w = make(name[:-4])
        w.name, w.kv_dtype = name, "fp8"
        w.description += "; K/V stored as FP8 E4M3 (scales 1)"
        return w
    if name == "tiny":
        return _shared_prefix(name, 0, 4, 64, 16, n_heads=2, head_dim=64, chunk=16,
                              description="2 heads, D 64, chunk 16; 64-token prefix + 4 x 16 private")
    if name == "llama7b_p1024":
        return _shared_prefix(name, 1, 32, 1024, 512,
                              description="32 heads, D 128, chunk 64; 32 seqs share 1024 tokens, 512 private each")
    sweep = {"sweep_s2048_b32": (2, 32, 2048), "sweep_s2048_b64": (3, 64, 2048),
             "sweep_s4096_b32": (4, 32, 4096), "sweep_s4096_b64": (5, 64, 4096)}
    if name in sweep:
        seed, b, ns = sweep[name]
        return _shared_prefix(name, seed, b, ns, 512,
                              description=f"32 heads, D 128, chunk 64; {b} seqs share {ns} tokens, 512 private each")
    if name == "no_sharing":
        return _shared_prefix(name, 6, 32, 0, 2048,
                              description="32 heads, D 128, chunk 64; 32 fully private 2048-token contexts")
    if name == "multi_tenant":
        return _multi_tenant(7)
    if name == "d256_p1024":
        return _shared_prefix(name, 9, 32, 1024, 512, n_heads=16, head_dim=256, chunk=32,
                              description="16 heads, D 256, chunk 32 (the same KV bytes per token as 32 x 128); "
                                          "32 seqs share 1024 tokens, 512 private each")
    if name == "gqa_p1024":
        return _shared_prefix(name, 8, 32, 1024, 512, n_kv_heads=8,
                              description="32 query heads sharing 8 key/value heads (grouped-query, "
                                          "Llama-3-8B-like), D 128, chunk 64; 32 seqs share 1024 "
                                          "tokens, 512 private each")
    raise KeyError(name)


ALL = ["tiny", "llama7b_p1024", "sweep_s2048_b32", "sweep_s2048_b64",
       "sweep_s4096_b32", "sweep_s4096_b64", "no_sharing", "multi_tenant", "gqa_p1024",
       "llama7b_p1024_fp8", "sweep_s4096_b64_fp8", "llama7b_p1024_q4", "d256_p1024"]
