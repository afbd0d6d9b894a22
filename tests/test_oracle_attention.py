"""Pins of the oracle's attention arithmetic against things other than itself:
brute force in plain Python loops, closed forms, and the merge identity.

The definitions being pinned: decode attention out = sum_t softmax_t(scale q.k_t)
v_t; the partial triple (o unnormalised, m = max, s = sum exp) of each phase
and their rescaled-sum merge [ChunkAttention explainer blog, "Two-Phase
Partition": phase equations, output combination and the two-phase function].
"""
import math
import random

import numpy as np
import pytest

from oracle import attention as A
from oracle.pakv import OracleError, OracleTrie


def brute_force(q, k, v, scale):
    """Plain-Python triple loop: for each head, scores, exponentials, weighted
    sum.  No numpy, no max shift (inputs are kept small enough not to
    overflow)."""
    n, H, D = len(k), len(q), len(q[0])
    out = []
    for h in range(H):
        e = []
        for t in range(n):
            dot = 0.0
            for d in range(D):
                dot += q[h][d] * k[t][h][d]
            e.append(math.exp(scale * dot))
        z = sum(e)
        out.append([sum(e[t] * v[t][h][d] for t in range(n)) / z for d in range(D)])
    return out


def rand(shape, rng, lo=-1.0, hi=1.0):
    return rng.uniform(lo, hi, size=shape)


def test_hand_computed_two_token_example():
    # q = (1, 0), keys (1, 0) and (0, 0), values (1, 2) and (3, 4), scale 1:
    # scores 1 and 0, weights e/(1+e) and 1/(1+e).
    q = np.array([[1.0, 0.0]])
    k = np.array([[[1.0, 0.0]], [[0.0, 0.0]]])
    v = np.array([[[1.0, 2.0]], [[3.0, 4.0]]])
    e = math.e
    want = np.array([[(e + 3) / (1 + e), (2 * e + 4) / (1 + e)]])
    np.testing.assert_allclose(A.softmax_attention(q, k, v, 1.0), want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("n,H,D", [(1, 1, 1), (3, 2, 4), (17, 3, 5), (40, 2, 8)])
def test_softmax_attention_matches_brute_force(n, H, D):
    rng = np.random.default_rng(n * 100 + H * 10 + D)
    q, k, v = rand((H, D), rng), rand((n, H, D), rng), rand((n, H, D), rng)
    scale = 1 / math.sqrt(D)
    got = A.softmax_attention(q, k, v, scale)
    want = brute_force(q.tolist(), k.tolist(), v.tolist(), scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_constant_v_returns_v():
    rng = np.random.default_rng(1)
    H, D, n = 3, 16, 50
    q, k = rand((H, D), rng, -4, 4), rand((n, H, D), rng, -4, 4)
    row = rand((H, D), rng)
    v = np.broadcast_to(row, (n, H, D))
    np.testing.assert_allclose(A.softmax_attention(q, k, v, 0.7), row, rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_v():
    rng = np.random.default_rng(2)
    H, D, n = 2, 8, 33
    k, v = rand((n, H, D), rng), rand((n, H, D), rng)
    got = A.softmax_attention(np.zeros((H, D)), k, v, 0.3)
    np.testing.assert_allclose(got, v.mean(axis=0), rtol=0, atol=1e-14)


def test_single_token_context_returns_its_value():
    rng = np.random.default_rng(3)
    q, k, v = rand((4, 8), rng), rand((1, 4, 8), rng), rand((1, 4, 8), rng)
    np.testing.assert_allclose(A.softmax_attention(q, k, v, 2.0), v[0], rtol=0, atol=1e-15)


def test_dominant_key_returns_its_value():
    rng = np.random.default_rng(4)
    H, D, n = 2, 8, 20
    q = np.ones((H, D))
    k, v = rand((n, H, D), rng, -0.1, 0.1), rand((n, H, D), rng)
    k[7] = 10.0                                     # score 80 * scale above the rest
    np.testing.assert_allclose(A.softmax_attention(q, k, v, 1.0), v[7], rtol=0, atol=1e-30 + 1e-12)


def test_scores_use_the_scale():
    # Doubling the scale equals doubling q; a missing or misplaced scale fails.
    rng = np.random.default_rng(5)
    q, k, v = rand((2, 4), rng), rand((9, 2, 4), rng), rand((9, 2, 4), rng)
    np.testing.assert_allclose(A.softmax_attention(q, k, v, 2.0),
                               A.softmax_attention(2 * q, k, v, 1.0), rtol=1e-13, atol=1e-14)
    assert not np.allclose(A.softmax_attention(q, k, v, 2.0), A.softmax_attention(q, k, v, 1.0))


def test_partial_triple_against_brute_force():
    rng = np.random.default_rng(6)
    H, D, n = 2, 4, 11
    q, k, v = rand((H, D), rng), rand((n, H, D), rng), rand((n, H, D), rng)
    o, m, s = A.partial(q, k, v, 0.5)
    for h in range(H):
        x = [0.5 * sum(q[h][d] * k[t][h][d] for d in range(D)) for t in range(n)]
        mm = max(x)
        assert m[h] == pytest.approx(mm, abs=1e-15)
        assert s[h] == pytest.approx(sum(math.exp(xi - mm) for xi in x), rel=1e-14)
        for d in range(D):
            want = sum(math.exp(x[t] - mm) * v[t][h][d] for t in range(n))
            assert o[h][d] == pytest.approx(want, rel=1e-13, abs=1e-15)


@pytest.mark.parametrize("seed", range(8))
def test_merge_identity_any_split(seed):
    """Splitting a context into parts and merging their partials equals the
    softmax over the whole context (the merge rule), including empty parts."""
    rng = np.random.default_rng(100 + seed)
    H, D, n = 3, 8, int(rng.integers(1, 60))
    q, k, v = rand((H, D), rng, -3, 3), rand((n, H, D), rng, -3, 3), rand((n, H, D), rng)
    cuts = sorted(rng.integers(0, n + 1, size=int(rng.integers(0, 6))).tolist())
    bounds = [0] + cuts + [n]
    parts = [A.partial(q, k[a:z], v[a:z], 0.9) for a, z in zip(bounds[:-1], bounds[1:])]
    random.Random(seed).shuffle(parts)                 # order of parts is free
    np.testing.assert_allclose(A.merge(parts), A.softmax_attention(q, k, v, 0.9),
                               rtol=1e-12, atol=1e-13)


def test_merge_of_only_empty_parts_is_an_error():
    q = np.zeros((1, 2))
    empty = A.partial(q, np.zeros((0, 1, 2)), np.zeros((0, 1, 2)), 1.0)
    with pytest.raises(OracleError):
        A.merge([empty, empty])


def test_merge_needs_the_rescale():
    # Parts whose maxima differ by a lot: a merge that skipped e^{m_j - m*}
    # would weight the small part as much as the large one.
    q = np.array([[1.0]])
    k1, v1 = np.array([[[10.0]]]), np.array([[[1.0]]])
    k2, v2 = np.array([[[0.0]]]), np.array([[[-1.0]]])
    got = A.merge([A.partial(q, k1, v1, 1.0), A.partial(q, k2, v2, 1.0)])
    w = math.exp(10) / (math.exp(10) + 1)
    assert got[0, 0] == pytest.approx(w - (1 - w), rel=1e-14)


def test_two_phase_single_prefix_equals_definition():
    rng = np.random.default_rng(7)
    b, H, D, ns = 5, 2, 8, 13
    q = rand((b, H, D), rng, -2, 2)
    pk, pv = rand((ns, H, D), rng, -2, 2), rand((ns, H, D), rng)
    sk = [rand((int(rng.integers(0, 9)), H, D), rng, -2, 2) for _ in range(b)]
    sv = [rand((x.shape[0], H, D), rng) for x in sk]
    got = A.two_phase_single_prefix(q, pk, pv, sk, sv, 0.4)
    for i in range(b):
        want = brute_force(q[i].tolist(), np.concatenate([pk, sk[i]]).tolist(),
                           np.concatenate([pv, sv[i]]).tolist(), 0.4)
        np.testing.assert_allclose(got[i], want, rtol=1e-12, atol=1e-13)


def test_decode_attention_over_trie_matches_brute_force():
    rng = np.random.default_rng(8)
    L, H, D, c = 2, 2, 4, 3
    trie = OracleTrie(c, 64)
    prefix = list(range(7))
    pk, pv = rand((L, 7, H, D), rng), rand((L, 7, H, D), rng)
    ctx = {}
    for s in range(4):
        tail = [100 + 10 * s + i for i in range(s + 1)]
        tk, tv = rand((L, len(tail), H, D), rng), rand((L, len(tail), H, D), rng)
        k, v = np.concatenate([pk, tk], 1), np.concatenate([pv, tv], 1)
        trie.insert(s, prefix + tail, k, v)
        ctx[s] = (k, v)
    q = rand((4, H, D), rng)
    for layer in range(L):
        out = A.decode_attention(trie, [3, 1, 0, 2], layer, q, 0.5)
        for i, s in enumerate([3, 1, 0, 2]):
            k, v = ctx[s]
            want = brute_force(q[i].tolist(), k[layer].tolist(), v[layer].tolist(), 0.5)
            np.testing.assert_allclose(out[i], want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_grouped_query_attention_equals_repeated_kv(G):
    """GQA equals multi-head attention with each key/value head repeated for
    its G query heads; brute force checks one head directly."""
    rng = np.random.default_rng(20 + G)
    Hkv, D, n = 2, 4, 9
    q = rand((Hkv * G, D), rng, -2, 2)
    k, v = rand((n, Hkv, D), rng, -2, 2), rand((n, Hkv, D), rng)
    got = A.softmax_attention(q, k, v, 0.6)
    want = A.softmax_attention(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), 0.6)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)
    h = Hkv * G - 1                                       # last query head -> last kv head
    bf = brute_force(q[h:h + 1].tolist(), k[:, Hkv - 1:Hkv].tolist(), v[:, Hkv - 1:Hkv].tolist(), 0.6)
    np.testing.assert_allclose(got[h], bf[0], rtol=1e-12, atol=1e-13)
    o, m, s = A.partial(q, k, v, 0.6)
    np.testing.assert_allclose(A.merge([(o, m, s)]), got, rtol=1e-13, atol=1e-14)


def test_grouped_query_heads_must_divide():
    with pytest.raises(OracleError):
        A.softmax_attention(np.zeros((3, 2)), np.zeros((1, 2, 2)), np.zeros((1, 2, 2)), 1.0)


def _trie_with(rng, n_seqs, lengths, H=2, D=4, c=3):
    trie = OracleTrie(c, 200)
    for s in range(n_seqs):
        toks = list(range(7)) + [100 + 20 * s + i for i in range(lengths[s])]
        trie.insert(s, toks, rand((1, len(toks), H, D), rng), rand((1, len(toks), H, D), rng))
    return trie


@pytest.mark.parametrize("causal", [False, True])
def test_multi_token_queries_with_one_token_are_decode_attention(causal):
    rng = np.random.default_rng(30)
    trie = _trie_with(rng, 3, [2, 5, 1])
    q = rand((3, 1, 2, 4), rng)
    np.testing.assert_allclose(A.decode_attention_multi(trie, [2, 0, 1], 0, q, 0.5, causal)[:, 0],
                               A.decode_attention(trie, [2, 0, 1], 0, q[:, 0], 0.5), rtol=1e-13, atol=1e-14)


def test_multi_token_queries_without_mask_are_independent_queries():
    # every token sees the whole context: each token row is its own decode query
    rng = np.random.default_rng(31)
    trie = _trie_with(rng, 2, [4, 3])
    q = rand((2, 3, 2, 4), rng)
    got = A.decode_attention_multi(trie, [0, 1], 0, q, 0.7)
    for j in range(3):
        np.testing.assert_allclose(got[:, j], A.decode_attention(trie, [0, 1], 0, q[:, j], 0.7),
                                   rtol=1e-13, atol=1e-14)


def test_causal_queries_over_a_whole_sequence_are_causal_self_attention():
    # q_len = n: token j attends to tokens 0..j (brute force per token)
    rng = np.random.default_rng(32)
    H, D, n = 2, 4, 9
    trie = OracleTrie(4, 10)
    k, v = rand((1, n, H, D), rng), rand((1, n, H, D), rng)
    trie.insert(0, list(range(n)), k, v)
    q = rand((1, n, H, D), rng)
    got = A.decode_attention_multi(trie, [0], 0, q, 0.6, causal=True)
    for j in range(n):
        want = brute_force(q[0, j].tolist(), k[0, :j + 1].tolist(), v[0, :j + 1].tolist(), 0.6)
        np.testing.assert_allclose(got[0, j], want, rtol=1e-12, atol=1e-13)
    # the last token sees everything, the first only itself
    np.testing.assert_allclose(got[0, -1], A.softmax_attention(q[0, -1], k[0], v[0], 0.6), rtol=1e-13)
    np.testing.assert_allclose(got[0, 0], v[0, 0], rtol=0, atol=1e-15)


def test_multi_token_queries_match_the_two_phase_form():
    # the blog's two-phase function over a shared prefix, token by token
    rng = np.random.default_rng(33)
    b, H, D, ns, ql = 3, 2, 4, 6, 2
    pk, pv = rand((ns, H, D), rng), rand((ns, H, D), rng)
    sk = [rand((int(rng.integers(1, 5)), H, D), rng) for _ in range(b)]
    sv = [rand((x.shape[0], H, D), rng) for x in sk]
    trie = OracleTrie(ns, 50)
    for i in range(b):
        toks = list(range(ns)) + [1000 + 10 * i + t for t in range(sk[i].shape[0])]
        trie.insert(i, toks, np.concatenate([pk, sk[i]])[None], np.concatenate([pv, sv[i]])[None])
    q = rand((b, ql, H, D), rng)
    got = A.decode_attention_multi(trie, list(range(b)), 0, q, 0.4)
    for j in range(ql):
        np.testing.assert_allclose(got[:, j], A.two_phase_single_prefix(q[:, j], pk, pv, sk, sv, 0.4),
                                   rtol=1e-12, atol=1e-13)


def test_causal_context_shorter_than_the_queries_is_an_error():
    rng = np.random.default_rng(34)
    trie = OracleTrie(3, 10)
    trie.insert(0, [1, 2], rand((1, 2, 1, 2), rng), rand((1, 2, 1, 2), rng))
    with pytest.raises(OracleError):
        A.decode_attention_multi(trie, [0], 0, rand((1, 3, 1, 2), rng), 1.0, causal=True)
