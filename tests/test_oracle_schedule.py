"""Pins of the oracle's two-phase schedule tables: a hand-derived fixture,
coverage invariants, and the two-phase evaluation over the tables against the
plain definition.

[ChunkAttention (arXiv 2402.15220v4 summary) §3.2: chunk-first over chunks the
batch shares, then sequence-first over the rest; §3.3: tables rebuilt when the
tree changes.]
"""
import json
import os

import numpy as np
import pytest

from oracle import attention as A
from oracle.pakv import OracleError, OracleTrie
from oracle.schedule import build_schedule
from tests.treegen import random_token_lists

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TABLES = ["seq_perm", "cf_rows", "cf_runs", "sf_offsets", "sf_chunks",
          "merge_offsets", "merge_runs"]


def test_golden_schedule_tables():
    n_sched = 0
    for g in json.load(open(os.path.join(GOLDEN, "schedule_tiny_tree.json")))["scenarios"]:
        n_sched += run_golden_schedules(g)
    assert n_sched == 6


def run_golden_schedules(g):
    trie = OracleTrie(g["chunk"], g["capacity"])
    n_sched = 0
    for op in g["ops"]:
        if op["op"] == "insert":
            trie.insert(op["seq_id"], op["tokens"])
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
        elif op["op"] == "schedule":
            t = build_schedule(trie, op["seq_ids"])
            for name in TABLES:
                want = np.array(op[name], dtype=np.int32).reshape(t[name].shape)
                np.testing.assert_array_equal(t[name], want, err_msg=name)
            n_sched += 1
    return n_sched


def check_invariants(trie, seq_ids, t):
    b = len(seq_ids)
    perm = t["seq_perm"]
    assert sorted(perm.tolist()) == list(range(b))
    order = [seq_ids[i] for i in perm]
    holders = {}
    for p, s in enumerate(order):
        for node in trie.paths[s]:
            holders.setdefault(node.slot, []).append(p)
    # each chunk-first row's range is exactly its sharers, and it has >= 2
    for slot, ntok, lo, hi in t["cf_rows"]:
        assert holders[slot] == list(range(lo, hi))
        assert hi - lo >= 2
    # runs tile the rows in order
    cover = []
    for row0, nrows, lo, hi in t["cf_runs"]:
        cover += list(range(row0, row0 + nrows))
        for r in range(row0, row0 + nrows):
            assert list(t["cf_rows"][r][2:]) == [lo, hi]
    assert cover == list(range(len(t["cf_rows"])))
    # every (sequence, chunk) incidence is covered exactly once
    for p, s in enumerate(order):
        got = []
        for u in t["merge_runs"][t["merge_offsets"][p]:t["merge_offsets"][p + 1]]:
            row0, nrows, lo, hi = t["cf_runs"][u]
            assert lo <= p < hi
            got += [int(x) for x in t["cf_rows"][row0:row0 + nrows, 0]]
        got += [int(x) for x in t["sf_chunks"][t["sf_offsets"][p]:t["sf_offsets"][p + 1], 0]]
        assert got == trie.slots(s)
        ntok = (sum(int(t["cf_rows"][r][1]) for u in t["merge_runs"][t["merge_offsets"][p]:t["merge_offsets"][p + 1]]
                    for r in range(t["cf_runs"][u][0], t["cf_runs"][u][0] + t["cf_runs"][u][1]))
                + int(t["sf_chunks"][t["sf_offsets"][p]:t["sf_offsets"][p + 1], 1].sum()))
        assert ntok == trie.lengths[s]


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("c", [1, 2, 3])
def test_random_tree_tables_and_two_phase_equal_definition(seed, c):
    rng = np.random.default_rng(seed)
    L, H, D = 1, 2, 4
    seqs = random_token_lists(seed, 10, c)
    trie = OracleTrie(c, 500)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((L, len(toks), H, D))
        v = rng.standard_normal((L, len(toks), H, D))
        trie.insert(i, toks, k, v)
    # drop a few to exercise removal, then schedule a random subset
    for i in rng.choice(10, size=3, replace=False):
        trie.remove(int(i))
    live = sorted(trie.paths)
    batch = [int(x) for x in rng.permutation(live)[: max(1, len(live) - 1)]]
    t = build_schedule(trie, batch)
    check_invariants(trie, batch, t)
    q = rng.standard_normal((len(batch), H, D))
    np.testing.assert_allclose(A.two_phase_attention(trie, t, 0, q, 0.5),
                               A.decode_attention(trie, batch, 0, q, 0.5),
                               rtol=1e-11, atol=1e-12)


def test_batch_permutation_invariance():
    rng = np.random.default_rng(3)
    c, L, H, D = 2, 1, 2, 4
    seqs = random_token_lists(3, 8, c)
    trie = OracleTrie(c, 200)
    for i, toks in enumerate(seqs):
        trie.insert(i, toks, rng.standard_normal((L, len(toks), H, D)),
                    rng.standard_normal((L, len(toks), H, D)))
    batch = list(range(8))
    q = rng.standard_normal((8, H, D))
    ref = A.two_phase_attention(trie, build_schedule(trie, batch), 0, q, 0.7)
    p = rng.permutation(8)
    got = A.two_phase_attention(trie, build_schedule(trie, [batch[i] for i in p]), 0, q[p], 0.7)
    np.testing.assert_allclose(got, ref[p], rtol=1e-12, atol=1e-13)
    # the DFS order itself does not depend on the caller's order
    assert (build_schedule(trie, batch)["cf_rows"].tolist()
            == build_schedule(trie, [batch[i] for i in p])["cf_rows"].tolist())


def test_sharing_off_gives_identical_outputs():
    rng = np.random.default_rng(4)
    c, L, H, D = 4, 1, 2, 8
    prefix = list(range(16))
    shared, flat = OracleTrie(c, 100), OracleTrie(c, 100, no_sharing=True)
    pk, pv = rng.standard_normal((L, 16, H, D)), rng.standard_normal((L, 16, H, D))
    for i in range(5):
        tail = [100 + 10 * i + j for j in range(i + 2)]
        k = np.concatenate([pk, rng.standard_normal((L, len(tail), H, D))], 1)
        v = np.concatenate([pv, rng.standard_normal((L, len(tail), H, D))], 1)
        shared.insert(i, prefix + tail, k, v)
        flat.insert(i, prefix + tail, k, v)
    q = rng.standard_normal((5, H, D))
    ts, tf = build_schedule(shared, range(5)), build_schedule(flat, range(5))
    assert len(ts["cf_rows"]) == 4 and len(tf["cf_rows"]) == 0
    np.testing.assert_allclose(A.two_phase_attention(shared, ts, 0, q, 0.3),
                               A.two_phase_attention(flat, tf, 0, q, 0.3), rtol=1e-12, atol=1e-13)
    assert np.array_equal(A.decode_attention(shared, range(5), 0, q, 0.3),
                          A.decode_attention(flat, range(5), 0, q, 0.3))


def test_schedule_errors():
    trie = OracleTrie(2, 8)
    trie.insert(1, [1, 2])
    for batch, code in [([], "invalid"), ([1, 1], "invalid"), ([1, 2], "not_found")]:
        with pytest.raises(OracleError) as e:
            build_schedule(trie, batch)
        assert e.value.code == code
