"""The kernel work plan, checked on CPU: evaluate every exported unit with the
oracle's partial triple and merge it through the exported partial-id CSR, in
float64, and compare with the plain definition.  Any chunk dropped or counted
twice, or a partial written to the wrong id, changes the result
[ChunkAttention (arXiv 2402.15220v4 summary) §3.2]."""
import numpy as np
import pytest

from oracle import attention as A
from oracle.pakv import OracleTrie
from tests.treegen import random_segment_sequences


def simulate(plan, tables, trie, q, scale, H, G=1):
    by_slot = {}
    stack = [trie.root]
    while stack:
        n = stack.pop()
        if n.slot >= 0:
            by_slot[n.slot] = n
        stack.extend(n.children)
    perm, pbase = tables["seq_perm"], plan["pbase"]
    parts = {}
    cover = {}
    HQ = H * G

    def emit(pos, kvh, part, chunks):
        # one partial per query head of the key/value head
        k = np.concatenate([by_slot[s].k[0][:t, kvh] for s, t in chunks])[:, None, :]
        v = np.concatenate([by_slot[s].v[0][:t, kvh] for s, t in chunks])[:, None, :]
        for qh in range(kvh * G, (kvh + 1) * G):
            pid = pbase[pos * HQ + qh] + part
            assert pbase[pos * HQ + qh] <= pid < pbase[pos * HQ + qh + 1]
            assert pid not in parts
            parts[pid] = A.partial(q[perm[pos], qh][None, :], k, v, scale)
            cover.setdefault((pos, qh), []).extend(int(s) for s, _ in chunks)

    for kind, h, lo, hi, cb, ce, part, qrow, n, base, part_next, _ in plan["units"]:
        assert lo < hi and cb < ce
        if kind == 0:
            assert 0 <= h and h + n <= H and n >= 1 and (hi - lo) * G <= 64
            for hh in range(h, h + n):
                for pos in range(lo, hi):
                    emit(pos, hh, part, plan["chunks"][cb:ce])
        else:
            assert hi == lo + 1 and qrow == perm[lo] and h == cb // n
            L = cb
            while L < ce:                      # one head's piece at a time
                hh, j = divmod(L, n)
                z = min(ce, (hh + 1) * n)
                emit(lo, hh, part if hh == h else part_next, plan["chunks"][base + j:base + j + (z - L)])
                L = z
    assert len(parts) == pbase[-1]
    out = np.empty(q.shape)
    b = len(perm)
    for pos in range(b):
        for h in range(HQ):
            ids = range(pbase[pos * HQ + h], pbase[pos * HQ + h + 1])
            out[perm[pos], h] = A.merge([parts[i] for i in ids])[0]
    return out, cover


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("c", [16, 32])
def test_plan_reproduces_the_definition(lib, seed, c):
    from prefix_shared_decode_gb300 import Pool
    H, D = 3, 64
    rng = np.random.default_rng(seed)
    seqs = random_segment_sequences(seed, 10, c)
    pool = Pool(1, H, D, c, 500, host_only=True)
    trie = OracleTrie(c, 500)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), H, D))
        v = rng.standard_normal((1, len(toks), H, D))
        pool.insert(i, toks)
        trie.insert(i, toks, k, v)
    batch = [int(x) for x in rng.permutation(10)[:8]]
    q = rng.standard_normal((len(batch), H, D))
    for no_tpp in (False, True):
        sched = pool.schedule(batch, no_tpp=no_tpp)
        plan = sched.plan()
        assert plan["cta_begin"][0] == 0 and plan["cta_begin"][-1] <= len(plan["units"])
        assert np.all(np.diff(plan["cta_begin"]) >= 0)
        out, cover = simulate(plan, sched.tables(), trie, q, 0.125, H)
        np.testing.assert_allclose(out, A.decode_attention(trie, batch, 0, q, 0.125),
                                   rtol=1e-10, atol=1e-12)
        # every (sequence, head) sees exactly its own path's chunks
        for pos, s in enumerate(sched.tables()["seq_perm"]):
            for h in range(H):
                assert sorted(cover[(pos, h)]) == sorted(trie.slots(batch[s]))


def test_plan_splits_large_runs_and_query_groups(lib):
    # 70 sequences share 40 chunks: query groups of <= 64 and several row
    # pieces; private chunks spread over many CTAs.
    from prefix_shared_decode_gb300 import Pool
    c, H = 64, 4
    pool = Pool(1, H, 128, c, 4000, host_only=True)
    prefix = list(range(40 * c))
    for i in range(70):
        pool.insert(i, prefix + [10**6 + 1000 * i + j for j in range(100 + i)])
    sched = pool.schedule(list(range(70)))
    plan = sched.plan()
    cf = plan["units"][plan["units"][:, 0] == 0]
    sf = plan["units"][plan["units"][:, 0] == 1]
    static = plan["units"][:plan["cta_begin"][-1]]
    tail = plan["units"][plan["cta_begin"][-1]:]
    assert (static[:, 0] == 1).sum() <= 70 + 2 * 304        # about one unit per position and CTA
    assert len(tail) > 0 and (tail[:, 0] == 1).all() and (tail[:, 5] - tail[:, 4]).max() <= 8
    assert cf[:, 3].max() - cf[:, 2].min() == 70
    assert (cf[:, 3] - cf[:, 2]).max() <= 64
    assert len(np.unique(cf[:, 2])) == 2                   # two query groups
    assert plan["grid"] == 304
    units_per_cta = np.diff(plan["cta_begin"])
    assert (units_per_cta > 0).sum() > 250


@pytest.mark.parametrize("G", [2, 4, 8])
def test_plan_with_grouped_query_heads(lib, G):
    """Units per key/value head, partials per query head, query groups of at
    most 64 (position, query head) rows."""
    from prefix_shared_decode_gb300 import Pool
    Hkv, D, c = 2, 64, 16
    rng = np.random.default_rng(30 + G)
    seqs = random_segment_sequences(30 + G, 12, c)
    pool = Pool(1, Hkv * G, D, c, 500, host_only=True, n_kv_heads=Hkv)
    trie = OracleTrie(c, 500)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), Hkv, D))
        trie.insert(i, toks, k, k * 0.5)
        pool.insert(i, toks)
    batch = [int(x) for x in rng.permutation(12)[:10]]
    q = rng.standard_normal((len(batch), Hkv * G, D))
    sched = pool.schedule(batch)
    out, _ = simulate(sched.plan(), sched.tables(), trie, q, 0.125, Hkv, G)
    np.testing.assert_allclose(out, A.decode_attention(trie, batch, 0, q, 0.125), rtol=1e-10, atol=1e-12)



def simulate_multi(plan, tables, trie, batch, q, scale, H, G, q_len, causal):
    """The exported plan evaluated for q_len query tokens per position: rows
    (position, token, query head); under the causal mask a chunk's row r at
    context offset depth * c counts for token j iff offset + r <= n - q_len + j."""
    c = trie.chunk
    node_of, depth = {}, {}
    stack = [(trie.root, -1)]
    while stack:
        n, d = stack.pop()
        if n.slot >= 0:
            node_of[n.slot], depth[n.slot] = n, d
        stack.extend((ch, d + 1) for ch in n.children)
    perm, pbase = tables["seq_perm"], plan["pbase"]
    HQ = H * G
    n_ctx = [trie.lengths[batch[perm[pos]]] for pos in range(len(perm))]
    parts = {}

    def emit(pos, kvh, part, chunks):
        for j in range(q_len):
            lim = n_ctx[pos] - q_len + j if causal else 1 << 30
            ks, vs = [], []
            for s, t in chunks:
                rows = [r for r in range(int(t)) if depth[int(s)] * c + r <= lim]
                ks.append(node_of[int(s)].k[0][rows, kvh])
                vs.append(node_of[int(s)].v[0][rows, kvh])
            k = np.concatenate(ks)[:, None, :]
            v = np.concatenate(vs)[:, None, :]
            for qh in range(kvh * G, (kvh + 1) * G):
                i = (pos * q_len + j) * HQ + qh
                pid = pbase[i] + part
                assert pbase[i] <= pid < pbase[i + 1]
                assert pid not in parts
                parts[pid] = A.partial(q[perm[pos], j, qh][None, :], k, v, scale)

    for kind, h, lo, hi, cb, ce, part, qrow, n, base, part_next, _ in plan["units"]:
        if kind == 0:
            assert (hi - lo) * q_len * G <= 64
            for hh in range(h, h + n):
                for pos in range(lo, hi):
                    emit(pos, hh, part, plan["chunks"][cb:ce])
        else:
            L = cb
            while L < ce:
                hh, j = divmod(L, n)
                z = min(ce, (hh + 1) * n)
                emit(lo, hh, part if hh == h else part_next, plan["chunks"][base + j:base + j + (z - L)])
                L = z
    assert len(parts) == pbase[-1]
    out = np.empty(q.shape)
    for pos in range(len(perm)):
        for j in range(q_len):
            for h in range(HQ):
                i = (pos * q_len + j) * HQ + h
                out[perm[pos], j, h] = A.merge([parts[x] for x in range(pbase[i], pbase[i + 1])])[0]
    return out


@pytest.mark.parametrize("q_len,causal,G", [(2, False, 1), (3, True, 1), (5, True, 2), (4, False, 2), (8, True, 1)])
@pytest.mark.parametrize("seed", range(3))
def test_plan_with_multi_token_queries(lib, q_len, causal, G, seed):
    from prefix_shared_decode_gb300 import Pool
    Hkv, D, c = 2, 64, 16
    rng = np.random.default_rng(70 + seed)
    seqs = random_segment_sequences(70 + seed, 10, c)
    pool = Pool(1, Hkv * G, D, c, 600, host_only=True, n_kv_heads=Hkv)
    trie = OracleTrie(c, 600)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), Hkv, D))
        trie.insert(i, toks, k, k * 0.3 + 1)
        pool.insert(i, toks)
    # a causal batch needs every context at least q_len tokens long
    batch = [int(x) for x in rng.permutation(10) if len(seqs[x]) >= q_len][:8]
    q = rng.standard_normal((len(batch), q_len, Hkv * G, D))
    for no_tpp in (False, True):
        sched = pool.schedule(batch, no_tpp=no_tpp, q_len=q_len, causal=causal)
        out = simulate_multi(sched.plan(), sched.tables(), trie, batch, q, 0.125, Hkv, G, q_len, causal)
        want = A.decode_attention_multi(trie, batch, 0, q, 0.125, causal)
        np.testing.assert_allclose(out, want, rtol=1e-10, atol=1e-12)


def test_multi_token_schedule_limits(lib):
    from prefix_shared_decode_gb300 import CAError, Pool
    pool = Pool(1, 8, 64, 16, 50, host_only=True, n_kv_heads=2)       # G = 4
    pool.insert(0, list(range(20)))
    pool.insert(1, list(range(3)))
    with pytest.raises(CAError) as e:
        pool.schedule([0], q_len=17)                                     # 17 * 4 rows > 64
    assert e.value.name == "CA_ERR_UNSUPPORTED"
    with pytest.raises(CAError) as e:
        pool.schedule([0, 1], q_len=4, causal=True)                      # a 3-token context
    assert e.value.name == "CA_ERR_INVALID"
    pool.schedule([0, 1], q_len=4)                                       # no mask: fine
    assert len(pool.schedule([0], q_len=16).plan()["pbase"]) == 16 * 8 + 1


def test_schedule_reuse_fast_path_and_staleness_key(lib):
    """The per-step ``pool.schedule(batch, reuse=s)`` keeps the batch's int64
    copy; a batch list changed in place, or another list, is converted again
    (the tables follow the new batch).  ``Schedule._key`` (what a captured
    CUDA graph is checked against) stays put across appends that fit the
    partial last chunks and changes when a chunk grows or the batch changes."""
    from prefix_shared_decode_gb300 import Pool
    c, H, D = 16, 2, 64
    pool = Pool(1, H, D, c, 200, host_only=True)
    shared = list(range(2 * c))
    for i in range(4):
        pool.insert(i, shared + [1000 + 100 * i + j for j in range(c // 2 + i)])
    batch = [0, 1, 2, 3]
    s = pool.schedule(batch)
    key, perm = s._key(), s.tables()["seq_perm"].copy()
    assert pool.schedule(batch, reuse=s) is s and s._key() == key
    assert pool.append(2, [5000]) == 0                      # fits the partial last chunk
    assert pool.schedule(list(batch), reuse=s)._key() == key
    batch.reverse()                                          # the same list object, changed in place
    pool.schedule(batch, reuse=s)
    assert s._key() != key
    np.testing.assert_array_equal(s.tables()["seq_perm"], [3 - p for p in perm])
    key = s._key()
    assert pool.append(0, [6000 + j for j in range(c)]) == 1  # grows a chunk
    assert s._key() != key
    pool.schedule(batch, reuse=s)
    assert s._key() != key and pool.schedule(batch, reuse=s)._key() == s._key()
