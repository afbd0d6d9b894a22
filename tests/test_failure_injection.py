"""Failure paths, exercised without faulting or hanging a GPU.

* The status word: a kernel that sees a table index out of range or gives up
  a wait records CA_ERR_DEVICE_BOUNDS / CA_ERR_TIMEOUT; ca_sched_device_status
  returns the code once and clears it.  Here a test hook writes the word (on
  CPU: a host-only pool's host word; on a GPU: the device word).
* Host allocation failures: an insert or append that runs out of host memory
  part-way (a child list, a hash index, the copy list, the sequence map)
  returns CA_ERR_OOM and leaves the pool exactly as before.  Every allocation
  point of the call is made to fail in turn, and after each failure the pool
  must behave bit for bit like one that never saw the call: same slots, same
  statistics, same schedule tables (checked against the oracle's trie too).
* On a GPU: a decode call whose producer waits for a barrier phase that
  nothing completes (no copy issued) gives up after the ~1 s limit, reports
  CA_ERR_TIMEOUT, and the next call is correct.
"""
import numpy as np
import pytest

from oracle.pakv import OracleTrie
from oracle.schedule import build_schedule

ERR_INVALID, ERR_OOM, ERR_BOUNDS, ERR_TIMEOUT = -1, -2, -7, -8
TABLES = ["seq_perm", "cf_rows", "cf_runs", "sf_offsets", "sf_chunks", "merge_offsets", "merge_runs"]


def host_pool(c=16, cap=400):
    from prefix_shared_decode_gb300 import Pool
    return Pool(1, 2, 64, c, cap, host_only=True)


def test_status_word_is_decoded_once_and_cleared_host_only(lib):
    pool = host_pool()
    pool.insert(0, list(range(40)))
    pool.insert(1, list(range(32)) + [900, 901])
    sched = pool.schedule([0, 1])
    assert sched.device_status() == 0
    for code in (ERR_BOUNDS, ERR_TIMEOUT):
        assert lib.ca_sched_inject_status(sched.handle, code, None) == 0
        assert sched.device_status() == code
        assert sched.device_status() == 0                    # cleared by the read
    for bad in (0, 3, -11):
        assert lib.ca_sched_inject_status(sched.handle, bad, None) == ERR_INVALID
    assert lib.ca_sched_inject_status(None, ERR_BOUNDS, None) == ERR_INVALID
    assert lib.ca_sched_inject_stall(sched.handle, -1) == ERR_INVALID
    assert lib.ca_pool_inject_alloc_failure(None, 0) == ERR_INVALID


def snapshot(pool, live, probes):
    """Everything a caller can observe of the pool."""
    s = pool.stats()
    slots = {sid: pool.seq_slots(sid) for sid in live}
    matched = [pool.match_prefix(t) for t in probes]
    tables = pool.schedule(sorted(live)).tables() if live else None
    return s, slots, matched, tables


def same(a, b):
    sa, sb = a, b
    assert sa[0] == sb[0] and sa[1] == sb[1] and sa[2] == sb[2]
    if sa[3] is None:
        assert sb[3] is None
    else:
        for k in TABLES:
            np.testing.assert_array_equal(sa[3][k], sb[3][k], err_msg=k)


def build_tree(pool, trie, c):
    """40 sequences with distinct first chunks (the root gets a hash index),
    plus a stem with a partial tail shared by several sequences."""
    live = []
    for i in range(40):
        toks = [10_000 + 100 * i + j for j in range(c + 3)]
        pool.insert(i, toks)
        trie.insert(i, toks)
        live.append(i)
    stem = [7 for _ in range(2 * c)]
    for i in range(40, 44):
        toks = stem + [20_000 + 50 * i + j for j in range(i % 5 + 1)]
        pool.insert(i, toks)
        trie.insert(i, toks)
        live.append(i)
    return live


def new_batch(c):
    stem = [7 for _ in range(2 * c)]
    return {100: stem + [555] * (c + 2),                           # shares the stem, grows two chunks
            101: [30_000 + j for j in range(3 * c + 1)],           # a new root child (indexed root)
            102: [10_000 + j for j in range(c)] + [31_000 + j for j in range(c)]}   # shares sequence 0's chunk


def test_injected_allocation_failure_rolls_back_insert_batch(lib):
    c = 16
    batch = new_batch(c)
    probes = list(batch.values()) + [[7] * (2 * c), [10_000 + j for j in range(c)]]
    ref_pool, ref_trie = host_pool(c), OracleTrie(c, 400)
    live = build_tree(ref_pool, ref_trie, c)
    before = snapshot(ref_pool, live, probes)
    failures = 0
    for k in range(200):
        pool = host_pool(c)
        build_tree(pool, OracleTrie(c, 400), c)
        assert lib.ca_pool_inject_alloc_failure(pool.handle, k) == 0
        try:
            pool.insert_batch(list(batch), list(batch.values()))
        except Exception as e:                                  # CAError
            assert getattr(e, "name", "") == "CA_ERR_OOM", e
            failures += 1
            assert lib.ca_pool_inject_alloc_failure(pool.handle, -1) == 0
            same(snapshot(pool, live, probes), before)
            # the same call now succeeds and the pool matches the oracle's trie
            pool.insert_batch(list(batch), list(batch.values()))
            trie = OracleTrie(c, 400)
            build_tree(host_pool(c), trie, c)
            for sid, toks in batch.items():
                trie.insert(sid, toks)
            ids = sorted(live + list(batch))
            got = pool.schedule(ids).tables()
            want = build_schedule(trie, ids)
            for name in TABLES:
                np.testing.assert_array_equal(got[name], want[name].reshape(got[name].shape), err_msg=name)
            for sid in ids:
                assert pool.seq_slots(sid) == trie.slots(sid)
            continue
        break                                                   # k passed every allocation point
    assert failures >= 20, failures                             # 30 allocation points in this call


def test_injected_allocation_failure_rolls_back_append(lib):
    c = 16
    probes = [[7] * (2 * c) + [1, 2, 3] + [44] * c]
    ref_pool = host_pool(c)
    live = build_tree(ref_pool, OracleTrie(c, 400), c)
    before = snapshot(ref_pool, live, probes)
    tail = [44] * (2 * c + 5)                                 # fills sequence 42's chunk, grows three
    failures = 0
    for k in range(100):
        pool = host_pool(c)
        build_tree(pool, OracleTrie(c, 400), c)
        assert lib.ca_pool_inject_alloc_failure(pool.handle, k) == 0
        try:
            pool.append(42, tail)
        except Exception as e:
            assert getattr(e, "name", "") == "CA_ERR_OOM", e
            failures += 1
            assert lib.ca_pool_inject_alloc_failure(pool.handle, -1) == 0
            same(snapshot(pool, live, probes), before)
            pool.append(42, tail)
            ref = host_pool(c)
            build_tree(ref, OracleTrie(c, 400), c)
            ref.append(42, tail)
            same(snapshot(pool, live, probes), snapshot(ref, live, probes))
            continue
        break
    assert failures >= 5, failures                              # 6 allocation points in this call


@pytest.mark.gpu
def test_device_status_and_stalled_call_on_the_gpu(lib):
    """The device word decodes and clears each code; a stalled call (its
    producer waits for a barrier phase nothing completes; no copy issued)
    gives up after ~1 s with CA_ERR_TIMEOUT, and the next call matches the
    oracle."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import time

    import workloads
    from oracle import attention as A
    from prefix_shared_decode_gb300 import Pool, decode_attention
    from workloads.device import capacity_for, insert_sequence
    wl = workloads.make("tiny")
    pool = Pool(wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, capacity_for(wl))
    trie = OracleTrie(wl.chunk, 1000)
    for sid in wl.seq_ids():
        insert_sequence(pool, wl, sid)
        trie.insert(sid, wl.tokens(sid), *wl.kv_rows(sid))
    batch = wl.seq_ids()
    sched = pool.schedule(batch)
    stream = torch.cuda.current_stream().cuda_stream
    for code in (ERR_BOUNDS, ERR_TIMEOUT):
        assert lib.ca_sched_inject_status(sched.handle, code, stream) == 0
        assert sched.device_status() == code
        assert sched.device_status() == 0
    q = wl.queries(0)
    want = A.decode_attention(trie, batch, 0, q, wl.scale)
    qd = torch.from_numpy(q).cuda()
    assert lib.ca_sched_inject_stall(sched.handle, 1) == 0
    t0 = time.perf_counter()
    decode_attention(pool, sched, qd)
    assert sched.device_status() == ERR_TIMEOUT
    assert 0.5 < time.perf_counter() - t0 < 30
    for _ in range(2):                                           # the next calls run normally
        got = decode_attention(pool, sched, qd).cpu().numpy().astype(np.float64)
        assert sched.device_status() == 0
        err = np.abs(got - want)
        assert err.max() <= 2e-3 and err.mean() <= 2e-4


@pytest.mark.gpu
def test_decode_call_argument_errors_launch_nothing(lib):
    """Bad arguments to the decode call are refused on the host with
    CA_ERR_INVALID before any kernel is launched: missing or misaligned q /
    out, a workspace that is too small or not 256-byte aligned, a layer out
    of range, a schedule of another pool.  A valid call then succeeds."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import workloads
    from oracle import attention as A
    from prefix_shared_decode_gb300 import Pool, capi, kernel_launches
    from workloads.device import capacity_for, insert_sequence
    wl = workloads.make("tiny")
    pools = []
    for _ in range(2):
        p = Pool(wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, capacity_for(wl))
        for sid in wl.seq_ids():
            insert_sequence(p, wl, sid)
        pools.append(p)
    pool, other = pools
    sched, other_sched = pool.schedule(wl.seq_ids()), other.schedule(wl.seq_ids())
    q = torch.from_numpy(wl.queries(0)).cuda()
    out = torch.empty_like(q)
    need = sched.workspace_bytes()
    ws = torch.zeros(need + 4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    L = capi.lib()

    def call(sch=sched, layer=0, qp=q.data_ptr(), op=out.data_ptr(), wp=ws.data_ptr(), wb=ws.numel()):
        return L.ca_decode_attention(pool.handle, sch.handle, layer, qp, op, float(wl.scale), wp, wb, stream)

    torch.cuda.synchronize()
    n0 = kernel_launches()
    for what, st in [("q NULL", call(qp=None)), ("out NULL", call(op=None)),
                     ("q misaligned", call(qp=q.data_ptr() + 2)), ("out misaligned", call(op=out.data_ptr() + 8)),
                     ("workspace short", call(wb=need - 1)), ("workspace NULL", call(wp=None)),
                     ("workspace misaligned", call(wp=ws.data_ptr() + 16, wb=need + 16)),
                     ("layer past the end", call(layer=wl.n_layers)), ("negative layer", call(layer=-1)),
                     ("another pool's schedule", call(sch=other_sched))]:
        assert st == ERR_INVALID, (what, st)
    assert kernel_launches() == n0
    assert call() == 0
    assert sched.device_status() == 0
    trie = OracleTrie(wl.chunk, 1000)
    for sid in wl.seq_ids():
        trie.insert(sid, wl.tokens(sid), *wl.kv_rows(sid))
    err = np.abs(out.cpu().numpy().astype(np.float64) - A.decode_attention(trie, wl.seq_ids(), 0, wl.queries(0),
                                                                          wl.scale))
    assert err.max() <= 2e-3 and err.mean() <= 2e-4


def test_failed_schedule_rebuild_is_never_reused(lib):
    """A schedule rebuild that fails part-way (host allocation) on a reused
    schedule, with the tree unchanged, must not leave new tables beside the
    old plan: the next call for the same batch rebuilds, and its plan equals
    a fresh schedule's."""
    from prefix_shared_decode_gb300 import CAError
    c = 16
    pool = host_pool(c)
    build_tree(pool, OracleTrie(c, 400), c)
    a, b = list(range(0, 44, 2)), list(range(1, 44, 3))
    sched = pool.schedule(a)
    assert lib.ca_pool_inject_alloc_failure(pool.handle, 0) == 0
    with pytest.raises(CAError) as e:
        pool.schedule(b, reuse=sched)
    assert e.value.name == "CA_ERR_OOM"
    assert lib.ca_pool_inject_alloc_failure(pool.handle, -1) == 0
    again = pool.schedule(b, reuse=sched).plan()
    fresh = pool.schedule(b).plan()
    for k in ("units", "cta_begin", "pbase", "chunks"):
        np.testing.assert_array_equal(again[k], fresh[k], err_msg=k)
