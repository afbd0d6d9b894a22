"""Oracle decode attention in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Decode attention has a plain definition that the two-phase partition reaches
exactly, up to rounding order [CA-blog, Two-Phase Partition: the split keeps
FlashAttention-style online-softmax compatibility]:

    out_{i,h} = sum_t softmax_t(scale * q_{i,h} . k_{t,h}) v_{t,h}

over every token t of sequence i's context (reading R7: the tokens inserted
for it; no causal mask inside one decode query).  With grouped-query
attention (fewer key/value heads than query heads, the "other model
configurations" of [CA-summary §7]) query head h reads key/value head
h // (Hq / Hkv).  ``decode_attention`` is that
definition written out.  The partial triple and the merge follow the pages'
statement of the two phases:

  partial (o, m, s) of a query over a set of tokens [CA-blog, Two-Phase
  Partition, Phase 1 / Phase 2 equations and the two-phase function]:
      x_t = scale * q . k_t,   m = max_t x_t,
      s = sum_t exp(x_t - m),  o = sum_t exp(x_t - m) v_t   (unnormalised)
  merge of partials j [CA-blog, output-combination equation, written with the
  function's rescaled sums; reading R1]:
      m* = max_j m_j,   out = sum_j e^{m_j - m*} o_j / sum_j e^{m_j - m*} s_j

Reading R1: the blog's equation weights *normalised* phase outputs by e^{m}
and calls m a log-sum-exp term; that is the same quantity as the form above
when m is the log-sum-exp.  The oracle keeps the unnormalised (o, max, sum)
triple that the blog's function keeps, generalised to any number of parts.
Reading R9: an empty part is (o = 0, m = -inf, s = 0) and carries no weight; a
context of zero tokens is an error.
"""
from __future__ import annotations

import numpy as np

from .pakv import OracleError, OracleTrie


def kv_head_of(n_q_heads: int, n_kv_heads: int) -> np.ndarray:
    """Grouped-query attention: query head h reads key/value head h // G,
    G = n_q_heads / n_kv_heads (G = 1 is multi-head attention)."""
    if n_kv_heads <= 0 or n_q_heads % n_kv_heads:
        raise OracleError("invalid", "query heads must be a multiple of key/value heads")
    return np.arange(n_q_heads) // (n_q_heads // n_kv_heads)


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """One query per head against a dense context.

    q [Hq, D]; k, v [n, Hkv, D] with Hq a multiple of Hkv  ->  [Hq, D],
    all float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if k.shape[0] == 0:
        raise OracleError("invalid", "empty context")
    g = kv_head_of(q.shape[0], k.shape[1])
    k, v = k[:, g], v[:, g]                             # each query head's key/value head
    x = scale * np.einsum("hd,nhd->hn", q, k)          # scores [H, n]
    w = np.exp(x - x.max(axis=1, keepdims=True))        # softmax numerators
    w /= w.sum(axis=1, keepdims=True)
    return np.einsum("hn,nhd->hd", w, v)


def decode_attention(trie: OracleTrie, seq_ids, layer: int, q: np.ndarray,
                     scale: float) -> np.ndarray:
    """Decode attention for a batch: row i of ``q`` [b, H, D] is sequence
    ``seq_ids[i]``; its context is materialised densely from the trie."""
    q = np.asarray(q, dtype=np.float64)
    out = np.empty(q.shape, dtype=np.float64)
    for i, s in enumerate(seq_ids):
        k, v = trie.materialize(int(s), layer)
        out[i] = softmax_attention(q[i], k, v, scale)
    return out


def decode_attention_multi(trie: OracleTrie, seq_ids, layer: int, q: np.ndarray, scale: float,
                           causal: bool = False) -> np.ndarray:
    """Several query tokens per sequence: q [b, q_len, H, D] -> [b, q_len, H, D].

    The blog's two-phase function takes queries of any length and lets every
    query token attend to the whole prefix and suffix [CA-blog, Two-Phase
    Partition]; that is the default.  Reading R16 (causal): when the query
    tokens are the last q_len tokens of the context (their K/V appended
    first), token j of a sequence with n context tokens attends to its first
    n - q_len + j + 1 tokens."""
    q = np.asarray(q, dtype=np.float64)
    b, q_len = q.shape[:2]
    out = np.empty(q.shape, dtype=np.float64)
    for i, s in enumerate(seq_ids):
        k, v = trie.materialize(int(s), layer)
        n = k.shape[0]
        for j in range(q_len):
            lim = n - q_len + j + 1 if causal else n
            if lim < 1:
                raise OracleError("invalid", "causal context shorter than the query tokens")
            out[i, j] = softmax_attention(q[i, j], k[:lim], v[:lim], scale)
    return out


def partial(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """The partial-result triple of one query per head over a token set.

    q [H, D]; k, v [n, H, D]  ->  o [H, D] (unnormalised), m [H], s [H].
    """
    q = np.asarray(q, dtype=np.float64)
    H, D = q.shape
    if k.shape[0] == 0:
        return np.zeros((H, D)), np.full(H, -np.inf), np.zeros(H)
    g = kv_head_of(H, k.shape[1])
    k = np.asarray(k, dtype=np.float64)[:, g]
    v = np.asarray(v, dtype=np.float64)[:, g]
    x = scale * np.einsum("hd,nhd->hn", q, k)
    m = x.max(axis=1)
    e = np.exp(x - m[:, None])
    s = e.sum(axis=1)
    o = np.einsum("hn,nhd->hd", e, v)
    return o, m, s


def merge(parts) -> np.ndarray:
    """Combine partial triples of disjoint token sets into the attention output."""
    parts = list(parts)
    ms = np.stack([p[1] for p in parts])                # [J, H]
    mstar = ms.max(axis=0)
    if np.any(np.isneginf(mstar)):
        raise OracleError("invalid", "every part empty")
    num = np.zeros_like(parts[0][0])
    den = np.zeros_like(parts[0][2])
    for o, m, s in parts:
        w = np.where(np.isneginf(m), 0.0, np.exp(m - mstar))
        num += w[:, None] * o
        den += w * s
    return num / den[:, None]


def two_phase_single_prefix(queries, prefix_k, prefix_v, suffix_k, suffix_v, scale):
    """The blog's two-phase formulation for one shared prefix.

    Phase 1 runs every query of the batch against the shared prefix at once;
    phase 2 runs each query against its own suffix; the two partial results
    are combined by the rescaled-sum rule.  queries [b, H, D]; prefix_k/v
    [n_s, H, D]; suffix_k/v lists of [n_i, H, D].
    """
    queries = np.asarray(queries, dtype=np.float64)
    out = np.empty_like(queries)
    for i in range(queries.shape[0]):
        shared = partial(queries[i], prefix_k, prefix_v, scale)
        own = partial(queries[i], suffix_k[i], suffix_v[i], scale)
        out[i] = merge([shared, own])
    return out


def _chunk_kv(trie: OracleTrie, slots_ntok, layer: int):
    by_slot = {}
    stack = [trie.root]
    while stack:
        n = stack.pop()
        if n.slot >= 0:
            by_slot[n.slot] = n
        stack.extend(n.children)
    ks = [by_slot[int(s)].k[layer][:int(t)] for s, t in slots_ntok]
    vs = [by_slot[int(s)].v[layer][:int(t)] for s, t in slots_ntok]
    if not ks:
        return None, None
    return np.concatenate(ks, 0).astype(np.float64), np.concatenate(vs, 0).astype(np.float64)


def two_phase_attention(trie: OracleTrie, tables: dict, layer: int, q: np.ndarray,
                        scale: float) -> np.ndarray:
    """Decode attention evaluated the two-phase way over the schedule tables
    [CA-summary §3.2]: chunk-first partials per run and sharer, one
    sequence-first partial per sequence over its own chunks, then the merge.
    Equal to ``decode_attention`` iff the tables cover every context exactly
    once."""
    q = np.asarray(q, dtype=np.float64)
    b, H, D = q.shape
    perm = tables["seq_perm"]
    rows, runs = tables["cf_rows"], tables["cf_runs"]
    run_parts = {}
    for u, (row0, nrows, lo, hi) in enumerate(runs):
        k, v = _chunk_kv(trie, rows[row0:row0 + nrows, :2], layer)
        for p in range(lo, hi):
            run_parts[(u, p)] = partial(q[perm[p]], k, v, scale)
    out = np.empty_like(q)
    for p in range(b):
        parts = [run_parts[(int(u), p)] for u in
                 tables["merge_runs"][tables["merge_offsets"][p]:tables["merge_offsets"][p + 1]]]
        a, z = tables["sf_offsets"][p], tables["sf_offsets"][p + 1]
        if z > a:
            k, v = _chunk_kv(trie, tables["sf_chunks"][a:z], layer)
            parts.append(partial(q[perm[p]], k, v, scale))
        out[perm[p]] = merge(parts)
    return out


def unique_kv_tokens(trie: OracleTrie, seq_ids) -> int:
    """Tokens held by the distinct chunks the batch's sequences use."""
    seen, total = set(), 0
    for s in seq_ids:
        for n in trie.paths[int(s)]:
            if id(n) not in seen:
                seen.add(id(n))
                total += n.ntok
    return total
