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

