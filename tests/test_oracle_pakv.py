"""Pins of the oracle's prefix-aware KV cache: counts fixed by the pages'
storage model, brute-force prefix sharing, refcount bookkeeping and rollback.

[ChunkAttention (arXiv 2402.15220v4 summary) §3.1; ChunkAttention explainer
blog, "Prefix-Aware KV Cache" (tokens stored: L_p + N * L_s instead of
N * L_p) and "動的プレフィックス検出" (refcounts, collection at zero).]
"""
import json
import math
import os

import numpy as np
import pytest

from oracle.pakv import OracleError, OracleTrie
from tests.treegen import lcp_chunks, random_token_lists

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_storage_model_lp_plus_n_ls():
    # N sequences sharing a chunk-aligned prefix of L_p tokens, each with L_s
    # private tokens: L_p + N * L_s tokens stored, against N * (L_p + L_s).
    for c, Lp, N, Ls in [(16, 64, 4, 16), (64, 1024, 32, 512), (4, 12, 7, 9)]:
        trie = OracleTrie(c, 10_000)
        prefix = list(range(Lp))
        for i in range(N):
            trie.insert(i, prefix + [10_000 + 100 * i + t for t in range(Ls)])
        chunks = trie.live_slots()
        assert chunks == Lp // c + N * math.ceil(Ls / c)
        tokens = Lp + N * Ls
        held = sum(n.ntok for n in {id(n): n for p in trie.paths.values() for n in p}.values())
        assert held == tokens
        flat = OracleTrie(c, 10_000, no_sharing=True)
        for i in range(N):
            flat.insert(i, prefix + [10_000 + 100 * i + t for t in range(Ls)])
        assert flat.live_slots() == N * math.ceil((Lp + Ls) / c)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("c", [1, 2, 4])
def test_sharing_matches_brute_force(seed, c):
    seqs = random_token_lists(seed, 9, c)
    trie = OracleTrie(c, 1000)
    for i, t in enumerate(seqs):
        shared = trie.insert(i, t)
        # the shared tokens are the longest full-chunk prefix any live sequence has
        want = max([lcp_chunks(t, seqs[j], c) for j in range(i)], default=0) * c
        assert shared == want
    # every pair shares exactly its longest common full-chunk prefix
    for i in range(len(seqs)):
        for j in range(i + 1, len(seqs)):
            si, sj = trie.slots(i), trie.slots(j)
            common = 0
            while common < min(len(si), len(sj)) and si[common] == sj[common]:
                common += 1
            assert common == lcp_chunks(seqs[i], seqs[j], c)
    # distinct full-chunk prefixes + one slot per partial tail
    prefixes = {tuple(t[:k * c]) for t in seqs for k in range(1, len(t) // c + 1)}
    tails = sum(1 for t in seqs if len(t) % c)
    assert trie.live_slots() == len(prefixes) + tails
    assert trie.refcount_sum() == sum(math.ceil(len(t) / c) for t in seqs)


@pytest.mark.parametrize("seed", range(6))
def test_remove_everything_frees_every_slot(seed):
    c = 2
    seqs = random_token_lists(seed, 10, c)
    trie = OracleTrie(c, 200)
    for i, t in enumerate(seqs):
        trie.insert(i, t)
    rng = np.random.default_rng(seed)
    for i in rng.permutation(len(seqs)):
        trie.remove(int(i))
    assert trie.live_slots() == 0
    assert sorted(trie.free) == list(range(200))
    assert trie.root.children == [] and trie.root.match == {}


def test_lowest_free_slot_first_and_reuse():
    trie = OracleTrie(2, 8)
    trie.insert(1, [1, 2, 3, 4])          # slots 0, 1
    trie.insert(2, [5, 6, 7])             # slots 2, 3
    trie.remove(1)                        # frees 0, 1
    trie.insert(3, [9, 9, 9, 9, 9])       # takes 0, 1, then 4
    assert trie.slots(3) == [0, 1, 4]


def test_partial_tail_is_never_shared():
    trie = OracleTrie(4, 16)
    assert trie.insert(1, [1, 2, 3, 4, 5, 6]) == 0
    assert trie.insert(2, [1, 2, 3, 4, 5, 6]) == 4       # only the full chunk
    assert trie.slots(1)[0] == trie.slots(2)[0]
    assert trie.slots(1)[1] != trie.slots(2)[1]
    assert trie.match_prefix([1, 2, 3, 4, 5, 6, 7, 8]) == 4


def test_no_sharing_makes_private_chains():
    trie = OracleTrie(2, 32, no_sharing=True)
    trie.insert(1, [1, 2, 3, 4])
    assert trie.insert(2, [1, 2, 3, 4]) == 0
    assert set(trie.slots(1)).isdisjoint(trie.slots(2))


def test_oom_leaves_the_trie_unchanged():
    trie = OracleTrie(2, 5)
    trie.insert(1, [1, 2, 3, 4, 5, 6])     # 3 slots
    before = (sorted(trie.free), trie.refcount_sum(), trie.generation)
    with pytest.raises(OracleError) as e:
        trie.insert(2, [1, 2, 7, 8, 9, 10, 11])   # shares 1, needs 3 more, 2 free
    assert e.value.code == "oom"
    assert (sorted(trie.free), trie.refcount_sum(), trie.generation) == before
    assert 2 not in trie.paths


def test_error_codes():
    trie = OracleTrie(2, 8)
    trie.insert(1, [1])
    for call, code in [(lambda: trie.insert(1, [2]), "exists"),
                       (lambda: trie.insert(2, []), "invalid"),
                       (lambda: trie.remove(7), "not_found")]:
        with pytest.raises(OracleError) as e:
            call()
        assert e.value.code == code


def test_first_inserter_rows_are_kept():
    # Rows of matched tokens are not read: the second insert passes different
    # K/V for the shared chunk, and the stored chunk keeps the first.
    L, H, D = 1, 1, 2
    k1 = np.arange(8, dtype=np.float64).reshape(L, 4, H, D)
    k2 = -k1
    trie = OracleTrie(2, 8)
    trie.insert(1, [1, 2, 3, 4], k1, k1)
    trie.insert(2, [1, 2, 5, 6], k2, k2)
    k, _ = trie.materialize(2)
    np.testing.assert_array_equal(k[:2], k1[0, :2])
    np.testing.assert_array_equal(k[2:], k2[0, 2:])


def test_golden_ops_slots_and_stats():
    for g in json.load(open(os.path.join(GOLDEN, "schedule_tiny_tree.json")))["scenarios"]:
        run_golden_ops(g)


def run_golden_ops(g):
    trie = OracleTrie(g["chunk"], g["capacity"])
    for op in g["ops"]:
        if op["op"] == "insert":
            assert trie.insert(op["seq_id"], op["tokens"]) == op["n_shared"]
            assert trie.slots(op["seq_id"]) == op["slots"]
        elif op["op"] == "remove":
            trie.remove(op["seq_id"])
        elif op["op"] == "append":
            n_new = trie.append(op["seq_id"], op["tokens"])
            if "n_new" in op:
                assert n_new == op["n_new"]
                assert trie.slots(op["seq_id"]) == op["slots"]
        elif op["op"] == "append_oom":
            with pytest.raises(OracleError) as e:
                trie.append(op["seq_id"], op["tokens"])
            assert e.value.code == "oom"
        elif op["op"] == "stats":
            assert trie.live_slots() == op["live_slots"]
            assert trie.refcount_sum() == op["refcount_sum"]
            if "generation" in op:
                assert trie.generation == op["generation"]


@pytest.mark.parametrize("seed", range(6))
def test_appends_keep_counts_and_context(seed):
    """After random inserts and appends, every sequence's materialised K/V is
    its inserted rows followed by its appended rows, and the refcount sum is
    the sum of ceil(len / c)."""
    rng = np.random.default_rng(seed)
    c, L, H, D = 2, 1, 1, 2
    seqs = random_token_lists(seed, 6, c)
    trie = OracleTrie(c, 500)
    full = {}
    for i, t in enumerate(seqs):
        k = rng.standard_normal((L, len(t), H, D))
        trie.insert(i, t, k, k + 1)
        full[i] = (list(t), k)
    # identical K/V for identical prefixes: rebuild each context from the trie's
    # view of the inserted part, then append
    for i in full:
        full[i] = (full[i][0], trie.materialize(i)[0][None])
    for step in range(12):
        i = int(rng.integers(0, 6))
        add = rng.integers(0, 3, size=int(rng.integers(1, 6))).tolist()
        k = rng.standard_normal((L, len(add), H, D))
        grown = trie.append(i, add, k, k + 1)
        toks, kk = full[i]
        full[i] = (toks + add, np.concatenate([kk, k], 1))
        assert grown == -(-(len(toks) + len(add)) // c) - -(-len(toks) // c)
    for i, (toks, kk) in full.items():
        got_k, got_v = trie.materialize(i)
        np.testing.assert_array_equal(got_k, kk[0])
        np.testing.assert_array_equal(got_v, kk[0] + 1)
        assert trie.lengths[i] == len(toks)
    assert trie.refcount_sum() == sum(-(-len(t) // c) for t, _ in full.values())


def test_append_errors_leave_the_trie_unchanged():
    trie = OracleTrie(2, 3)
    trie.insert(1, [1, 2, 3])                 # 2 slots, last chunk partial
    with pytest.raises(OracleError) as e:
        trie.append(1, [4, 5, 6, 7, 8])       # fills 1, needs 2 more, 1 free
    assert e.value.code == "oom"
    assert trie.paths[1][-1].tokens == (3,) and trie.lengths[1] == 3 and len(trie.free) == 1
    for call, code in [(lambda: trie.append(9, [1]), "not_found"), (lambda: trie.append(1, []), "invalid")]:
        with pytest.raises(OracleError) as e:
            call()
        assert e.value.code == code
