"""The C library's host side against the oracle, on CPU (host-only pools: no
GPU is touched).  Tables, slots, shared-token counts and pool statistics must
match bit for bit [ChunkAttention (arXiv 2402.15220v4 summary) §3.1-§3.3]."""
import json
import os
import re

import numpy as np
import pytest

from oracle.pakv import OracleTrie
from oracle.schedule import build_schedule
from tests.treegen import random_segment_sequences

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLES = ["seq_perm", "cf_rows", "cf_runs", "sf_offsets", "sf_chunks", "merge_offsets", "merge_runs"]


def header_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(ca_\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_symbol(lib):
    from prefix_shared_decode_gb300 import capi
    declared = header_functions()
    assert declared == set(capi.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.ca_error_string(-5) == b"schedule is older than the pool"


def make_pools(c, cap, no_sharing=False, H=2, D=64):
    from prefix_shared_decode_gb300 import Pool
    return (Pool(1, H, D, c, cap, no_sharing=no_sharing, host_only=True),
            OracleTrie(c, cap, no_sharing=no_sharing))


def assert_tables_equal(sched, want):
    got = sched.tables()
    for name in TABLES:
        np.testing.assert_array_equal(got[name], want[name].reshape(got[name].shape), err_msg=name)


def test_golden_fixture_through_the_c_api(lib):
    # The fixture uses c = 2; the library supports c in {16, 32, 64}.  Expand
    # every fixture token to 16 tokens and use c = 32: chunk boundaries and
    # sharing are preserved, token counts scale by 16.
    from prefix_shared_decode_gb300 import Pool
    X = 16
    g_all = json.load(open(os.path.join(ROOT, "tests", "golden", "schedule_tiny_tree.json")))
    for g in g_all["scenarios"]:
        pool = Pool(1, 2, 64, g["chunk"] * X, g["capacity"], host_only=True)
        expand = lambda toks: [t * X + j for t in toks for j in range(X)]
        for op in g["ops"]:
            if op["op"] == "insert":
                assert pool.insert(op["seq_id"], expand(op["tokens"])) == op["n_shared"] * X
                assert pool.seq_slots(op["seq_id"]) == op["slots"]
            elif op["op"] == "remove":
                pool.remove(op["seq_id"])
            elif op["op"] == "append":
                assert pool.append(op["seq_id"], expand(op["tokens"])) == op["n_new"]
                assert pool.seq_slots(op["seq_id"]) == op["slots"]
            elif op["op"] == "append_oom":
                from prefix_shared_decode_gb300 import CAError
                with pytest.raises(CAError) as e:
                    pool.append(op["seq_id"], expand(op["tokens"]))
                assert e.value.name == "CA_ERR_OOM"
            elif op["op"] == "stats":
                st = pool.stats()
                assert st["live_slots"] == op["live_slots"]
                assert st["refcount_sum"] == op["refcount_sum"]
                if "generation" in op:
                    assert st["generation"] == op["generation"]
            elif op["op"] == "schedule":
                t = pool.schedule(op["seq_ids"]).tables()
                for name in TABLES:
                    want = np.array(op[name], dtype=np.int32).reshape(t[name].shape)
                    if name in ("cf_rows", "sf_chunks") and want.size:
                        want[:, 1] *= X
                    np.testing.assert_array_equal(t[name], want, err_msg=name)


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("c", [16, 32])
def test_random_trees_bit_exact_with_oracle(lib, seed, c):
    seqs = random_segment_sequences(seed, 12, c)
    pool, ref = make_pools(c, 400)
    for i, toks in enumerate(seqs):
        assert pool.match_prefix(toks) == ref.match_prefix(toks)
        assert pool.insert(100 + i, toks) == ref.insert(100 + i, toks)
        assert pool.seq_slots(100 + i) == ref.slots(100 + i)
    rng = np.random.default_rng(seed)
    for step in range(3):
        live = sorted(ref.paths)
        batch = [int(x) for x in rng.permutation(live)[: max(1, len(live) - step)]]
        assert_tables_equal(pool.schedule(batch), build_schedule(ref, batch))
        # churn: remove two, insert two new ones reusing stems of the removed
        for sid in [int(x) for x in rng.choice(live, size=min(2, len(live) - 1), replace=False)]:
            pool.remove(sid)
            ref.remove(sid)
        for j in range(2):
            toks = random_segment_sequences(seed * 10 + step * 2 + j, 1, c)[0]
            sid = 1000 + step * 2 + j
            assert pool.insert(sid, toks) == ref.insert(sid, toks)
            assert pool.seq_slots(sid) == ref.slots(sid)
        st = pool.stats()
        assert st["live_slots"] == ref.live_slots()
        assert st["refcount_sum"] == ref.refcount_sum()
        assert st["generation"] == ref.generation


def test_no_sharing_pool_matches_oracle(lib):
    seqs = random_segment_sequences(3, 10, 16)
    pool, ref = make_pools(16, 500, no_sharing=True)
    for i, toks in enumerate(seqs):
        assert pool.insert(i, toks) == ref.insert(i, toks) == 0
        assert pool.seq_slots(i) == ref.slots(i)
    assert_tables_equal(pool.schedule(range(10)), build_schedule(ref, range(10)))
    assert pool.schedule(range(10)).counts()["cf_rows"] == 0


def test_no_tpp_schedule_makes_everything_sequence_first(lib):
    from prefix_shared_decode_gb300 import Pool
    pool = Pool(1, 2, 64, 16, 64, host_only=True)
    prefix = list(range(48))
    for i in range(4):
        pool.insert(i, prefix + [1000 + 100 * i + j for j in range(5)])
    t = pool.schedule([0, 1, 2, 3], no_tpp=True).tables()
    assert len(t["cf_rows"]) == 0 and len(t["merge_runs"]) == 0
    for p in range(4):
        s = t["seq_perm"][p]
        chunks = t["sf_chunks"][t["sf_offsets"][p]:t["sf_offsets"][p + 1]]
        assert list(chunks[:, 0]) == pool.seq_slots(s)
        assert chunks[:, 1].sum() == 53


def test_kernel_launch_counter_on_host_only_pools(lib):
    from prefix_shared_decode_gb300 import Pool, kernel_launches
    before = kernel_launches()
    pool = Pool(1, 2, 64, 16, 8, host_only=True)
    pool.insert(1, list(range(40)))                     # host-only: no KV scatter launched
    pool.schedule([1])
    assert kernel_launches() == before
    assert lib.ca_kernel_launches(None) == -1            # CA_ERR_INVALID


def test_head_dim_256_shape_limits(lib):
    from prefix_shared_decode_gb300 import CAError, Pool
    for chunk, kv in ((64, "fp16"), (32, "fp8")):
        with pytest.raises(CAError) as e:
            Pool(1, 2, 256, chunk, 10, host_only=True, kv_dtype=kv)
        assert e.value.name == "CA_ERR_UNSUPPORTED"
    pool = Pool(1, 8, 256, 32, 20, host_only=True, n_kv_heads=1)       # G = 8
    pool.insert(0, list(range(40)))
    with pytest.raises(CAError) as e:
        pool.schedule([0], q_len=5)                                     # 5 * 8 rows > 32
    assert e.value.name == "CA_ERR_UNSUPPORTED"
    plan = pool.schedule([0], q_len=4).plan()                           # 32 rows: fine
    assert len(plan["pbase"]) == 4 * 8 + 1


def test_errors_and_rollback(lib):
    from prefix_shared_decode_gb300 import CAError, Pool
    pool = Pool(1, 2, 64, 16, 5, host_only=True)
    pool.insert(1, list(range(40)))                     # 3 slots
    before = pool.stats()
    with pytest.raises(CAError) as e:
        pool.insert(2, list(range(16)) + list(range(100, 150)))   # shares 1, needs 4
    assert e.value.name == "CA_ERR_OOM"
    assert pool.stats() == before
    for fn, name in [(lambda: pool.insert(1, [5]), "CA_ERR_EXISTS"),
                     (lambda: pool.insert(3, []), "CA_ERR_INVALID"),
                     (lambda: pool.remove(9), "CA_ERR_NOT_FOUND"),
                     (lambda: pool.schedule([1, 1]), "CA_ERR_INVALID"),
                     (lambda: pool.schedule([7]), "CA_ERR_NOT_FOUND"),
                     (lambda: pool.schedule([]), "CA_ERR_INVALID")]:
        with pytest.raises(CAError) as e:
            fn()
        assert e.value.name == name
    with pytest.raises(CAError) as e:
        Pool(1, 2, 96, 16, 5, host_only=True)
    assert e.value.name == "CA_ERR_UNSUPPORTED"


def test_schedule_is_cached_until_the_tree_changes(lib):
    from prefix_shared_decode_gb300 import Pool
    pool = Pool(1, 2, 64, 16, 64, host_only=True)
    pool.insert(1, list(range(40)))
    pool.insert(2, list(range(40)) + [7])
    s = pool.schedule([1, 2])
    h = s.handle.value
    t0 = s.tables()
    assert pool.schedule([1, 2], reuse=s).handle.value == h
    pool.insert(3, [9] * 20)                            # tree changed: rebuilt in place
    s2 = pool.schedule([1, 2, 3], reuse=s)
    assert s2.handle.value == h and s2.counts()["b"] == 3
    np.testing.assert_array_equal(pool.schedule([1, 2], reuse=s).tables()["cf_rows"], t0["cf_rows"])


def test_remove_all_frees_everything(lib):
    seqs = random_segment_sequences(5, 15, 16)
    pool, ref = make_pools(16, 600)
    for i, toks in enumerate(seqs):
        pool.insert(i, toks)
    for i in np.random.default_rng(5).permutation(15):
        pool.remove(int(i))
    st = pool.stats()
    assert st["live_slots"] == 0 and st["free_slots"] == 600 and st["refcount_sum"] == 0
    # the allocator restarts from slot 0
    pool.insert(99, list(range(33)))
    assert pool.seq_slots(99) == [0, 1, 2]


def test_insert_batch_equals_sequential_inserts(lib):
    from prefix_shared_decode_gb300 import Pool
    seqs = random_segment_sequences(21, 12, 16)
    one, many = Pool(1, 2, 64, 16, 400, host_only=True), Pool(1, 2, 64, 16, 400, host_only=True)
    want = [one.insert(100 + i, t) for i, t in enumerate(seqs)]
    got = many.insert_batch([100 + i for i in range(12)], seqs)
    assert got == want
    for i in range(12):
        assert many.seq_slots(100 + i) == one.seq_slots(100 + i)
    assert many.stats() == one.stats()
    many.remove_batch([100, 105, 107])
    for s in (100, 105, 107):
        one.remove(s)
    assert many.stats() == one.stats()


def test_insert_batch_is_all_or_nothing(lib):
    from prefix_shared_decode_gb300 import CAError, Pool
    pool = Pool(1, 2, 64, 16, 10, host_only=True)
    pool.insert(1, list(range(40)))                       # 3 slots
    before = pool.stats()
    slots1 = pool.seq_slots(1)
    # second entry collides with an existing id
    with pytest.raises(CAError) as e:
        pool.insert_batch([2, 1], [list(range(20)), [7]])
    assert e.value.name == "CA_ERR_EXISTS"
    assert pool.stats() == before and pool.seq_slots(1) == slots1
    # the third entry runs out of slots after two succeeded
    with pytest.raises(CAError) as e:
        pool.insert_batch([3, 4, 5], [list(range(16)) + [500] * 20, [900] * 40, [901] * 100])
    assert e.value.name == "CA_ERR_OOM"
    assert pool.stats() == before
    with pytest.raises(CAError) as e:
        pool.remove_batch([1, 42])
    assert e.value.name == "CA_ERR_NOT_FOUND"
    assert pool.stats() == before
    with pytest.raises(CAError) as e:
        pool.remove_batch([1, 1])
    assert e.value.name == "CA_ERR_INVALID"
    # a later sequence of the batch shares chunks an earlier one created
    assert pool.insert_batch([6, 7], [[3] * 33, [3] * 40]) == [0, 32]


@pytest.mark.parametrize("seed", range(12))
def test_random_scripts_with_appends_bit_exact(lib, seed):
    """Inserts, appends (filling partial chunks, growing new ones, making
    chunks shareable) and removes through the C ABI, against the oracle."""
    from prefix_shared_decode_gb300 import Pool
    c = 16
    rng = np.random.default_rng(seed)
    pool, ref = Pool(1, 2, 64, c, 2000, host_only=True), OracleTrie(c, 2000)
    seqs = random_segment_sequences(seed, 10, c)
    for i, t in enumerate(seqs):
        assert pool.insert(i, t) == ref.insert(i, t)
    next_id = 100
    for step in range(40):
        live = sorted(ref.paths)
        r = rng.random()
        if r < 0.55:
            sid = int(rng.choice(live))
            add = rng.integers(0, 3, size=int(rng.integers(1, 2 * c))).tolist()
            assert pool.append(sid, add) == ref.append(sid, add)
            assert pool.seq_slots(sid) == ref.slots(sid)
        elif r < 0.8 or len(live) < 3:
            # a new sequence reusing the tokens of a live one (with a tail), so
            # chunks filled by appends get matched
            base = list(ref.paths[int(rng.choice(live))][0].tokens)
            src = int(rng.choice(live))
            toks = [t for n in ref.paths[src] for t in n.tokens]
            toks = toks[: int(rng.integers(1, len(toks) + 1))] + rng.integers(0, 3, size=int(rng.integers(0, c))).tolist()
            assert pool.match_prefix(toks) == ref.match_prefix(toks)
            assert pool.insert(next_id, toks) == ref.insert(next_id, toks)
            assert pool.seq_slots(next_id) == ref.slots(next_id)
            next_id += 1
        else:
            sid = int(rng.choice(live))
            pool.remove(sid)
            ref.remove(sid)
        st = pool.stats()
        assert (st["live_slots"], st["refcount_sum"], st["generation"]) == (
            ref.live_slots(), ref.refcount_sum(), ref.generation)
        if step % 5 == 4:
            batch = sorted(ref.paths)
            assert_tables_equal(pool.schedule(batch), build_schedule(ref, batch))
