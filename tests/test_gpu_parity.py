"""GPU parity of the two-phase decode attention kernel with the fp64 oracle.

Bar: max |out - oracle| <= 2e-3 and mean |out - oracle| <= 2e-4 on fp16
outputs computed with fp32 accumulation; tables and slots bit-exact.  Small
cases compare every output with the oracle's trie-based decode attention;
the full-size workloads compare every output (all sequences, heads and query
tokens) with the plain definition over each sequence's K/V [ChunkAttention explainer blog,
Two-Phase Partition; ChunkAttention (arXiv 2402.15220v4 summary) §3.2]."""
import numpy as np
import pytest

import workloads
from oracle import attention as A
from oracle import fp8 as F8
from oracle.pakv import OracleTrie
from oracle.schedule import build_schedule
from tests.oracle_parallel import plain_definition
from tests.treegen import random_segment_sequences
from workloads.device import capacity_for, insert_sequence

pytestmark = pytest.mark.gpu
TOL_MAX, TOL_MEAN = 2e-3, 2e-4


@pytest.fixture(scope="module")
def torch_cuda(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def assert_close(got, want, what=""):
    err = np.abs(got.astype(np.float64) - want)
    assert np.isfinite(got).all(), what
    assert err.max() <= TOL_MAX, f"{what}: max err {err.max():.3g}"
    assert err.mean() <= TOL_MEAN, f"{what}: mean err {err.mean():.3g}"


def load(torch, wl, no_sharing=False, capacity=None):
    from prefix_shared_decode_gb300 import Pool
    pool = Pool(wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, capacity or capacity_for(wl),
                no_sharing=no_sharing, n_kv_heads=wl.kv_heads, kv_dtype=wl.kv_dtype)
    staging = {}
    for sid in wl.seq_ids():
        insert_sequence(pool, wl, sid, staging=staging)
    return pool


def run(torch, pool, batch, q, no_tpp=False, layer=0, scale=None, q_len=1):
    from prefix_shared_decode_gb300 import decode_attention
    sched = pool.schedule(batch, no_tpp=no_tpp, q_len=q_len, causal=q_len > 1)
    out = decode_attention(pool, sched, torch.from_numpy(q).cuda(), layer=layer, scale=scale)
    assert sched.device_status() == 0
    return out.cpu().numpy(), sched


def oracle_trie(wl):
    trie = OracleTrie(wl.chunk, 100_000)
    for sid in wl.seq_ids():
        k, v = wl.kv_rows(sid)
        trie.insert(sid, wl.tokens(sid), k, v)
    return trie


def test_tiny_workload_every_output(torch_cuda):
    wl = workloads.make("tiny")
    pool = load(torch_cuda, wl)
    batch = wl.seq_ids()
    q = wl.queries(0)
    trie = oracle_trie(wl)
    want = A.decode_attention(trie, batch, 0, q, wl.scale)
    for no_tpp in (False, True):
        got, sched = run(torch_cuda, pool, batch, q, no_tpp=no_tpp)
        assert_close(got, want, f"tiny no_tpp={no_tpp}")
    # the tables the kernel ran on are the oracle's, bit for bit
    t = pool.schedule(batch).tables()
    ref = build_schedule(trie, batch)
    for name in ["seq_perm", "cf_rows", "cf_runs", "sf_offsets", "sf_chunks", "merge_offsets", "merge_runs"]:
        np.testing.assert_array_equal(t[name], ref[name].reshape(t[name].shape), err_msg=name)
    # sharing off (flat paged layout) gives the same attention
    flat = load(torch_cuda, wl, no_sharing=True)
    got, _ = run(torch_cuda, flat, batch, q)
    assert_close(got, want, "tiny no_sharing")


@pytest.mark.parametrize("c,D", [(16, 64), (32, 128), (64, 128), (64, 64), (16, 128), (32, 64)])
@pytest.mark.parametrize("seed", range(3))
def test_random_trees_every_output(torch_cuda, c, D, seed):
    from prefix_shared_decode_gb300 import Pool
    torch = torch_cuda
    H = 4
    rng = np.random.default_rng(seed)
    seqs = random_segment_sequences(seed, 12, c, n_segments=10)
    pool = Pool(2, H, D, c, 600)
    trie = OracleTrie(c, 600)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((2, len(toks), H, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((2, len(toks), H, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = [int(x) for x in rng.permutation(12)[:10]]
    q = rng.standard_normal((10, H, D), dtype=np.float32).astype(np.float16)
    for layer in (0, 1):
        want = A.decode_attention(trie, batch, layer, q, 1 / np.sqrt(D))
        got, _ = run(torch, pool, batch, q, layer=layer)
        assert_close(got, want, f"c={c} D={D} layer={layer}")


@pytest.mark.parametrize("G,Hkv,c,D", [(2, 2, 32, 128), (4, 2, 64, 128), (8, 1, 64, 64), (8, 2, 16, 128)])
def test_grouped_query_attention_every_output(torch_cuda, G, Hkv, c, D):
    """Grouped-query attention: G query heads per key/value head; the
    sequence-first phase then multiplies G rows per chunk on tensor cores."""
    from prefix_shared_decode_gb300 import Pool
    torch = torch_cuda
    rng = np.random.default_rng(40 + G + c)
    seqs = random_segment_sequences(40 + G, 12, c, n_segments=10)
    pool = Pool(1, Hkv * G, D, c, 600, n_kv_heads=Hkv)
    trie = OracleTrie(c, 600)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((1, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = [int(x) for x in rng.permutation(12)[:11]]
    q = rng.standard_normal((11, Hkv * G, D), dtype=np.float32).astype(np.float16)
    got, _ = run(torch, pool, batch, q)
    assert_close(got, A.decode_attention(trie, batch, 0, q, 1 / np.sqrt(D)), f"G={G}")


def _fp8_rows(rng, L, n, Hkv, D, scale):
    """fp16 N(0, 1) rows, their E4M3 codes and the dequantised rows."""
    x = rng.standard_normal((L, n, Hkv, D), dtype=np.float32).astype(np.float16)
    return x, F8.dequantize(F8.quantize(x, scale), scale)


def _check_fp8_bytes(pool, trie, k_scale, v_scale):
    """Every live chunk's stored codes equal the oracle's quantisation of its
    rows (scales are powers of two, so the dequantised rows divide back)."""
    kv = pool.kv_view().cpu().numpy()
    stack, n_checked = [trie.root], 0
    while stack:
        node = stack.pop()
        stack.extend(node.children)
        if node.slot < 0:
            continue
        t = node.ntok
        for kvi, (rows, sc) in enumerate(((node.k, k_scale), (node.v, v_scale))):
            want = F8.encode(np.transpose(rows / sc, (0, 2, 1, 3)))        # [L, H, t, D]
            np.testing.assert_array_equal(kv[node.slot, :, kvi, :, :t, :], want,
                                          err_msg=f"slot {node.slot} {'KV'[kvi]}")
        n_checked += 1
    assert n_checked > 0


@pytest.mark.parametrize("c,G,k_scale,v_scale", [(16, 1, 1.0, 1.0), (32, 1, 0.5, 2.0), (64, 1, 1.0, 0.25),
                                                 (64, 4, 2.0, 1.0), (32, 8, 1.0, 0.5)])
def test_fp8_pool_bytes_and_every_output(torch_cuda, c, G, k_scale, v_scale):
    """An FP8 pool: the stored codes match the oracle's E4M3 quantisation bit
    for bit, and attention matches the definition over the dequantised K/V,
    before and after decode-time appends (which quantise too)."""
    from prefix_shared_decode_gb300 import Pool, decode_attention
    torch = torch_cuda
    Hkv, D, L = 2, 128, 2
    rng = np.random.default_rng(60 + c + G)
    seqs = random_segment_sequences(60 + c, 12, c, n_segments=10)
    pool = Pool(L, Hkv * G, D, c, 700, n_kv_heads=Hkv, kv_dtype="fp8", k_scale=k_scale, v_scale=v_scale)
    trie = OracleTrie(c, 700)
    for i, toks in enumerate(seqs):
        k16, kq = _fp8_rows(rng, L, len(toks), Hkv, D, k_scale)
        v16, vq = _fp8_rows(rng, L, len(toks), Hkv, D, v_scale)
        trie.insert(i, toks, kq, vq)
        pool.insert(i, toks, torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda())
    torch.cuda.synchronize()
    _check_fp8_bytes(pool, trie, k_scale, v_scale)
    batch = [int(x) for x in rng.permutation(12)[:10]]
    q = rng.standard_normal((10, Hkv * G, D), dtype=np.float32).astype(np.float16)
    for layer in range(L):
        want = A.decode_attention(trie, batch, layer, q, 1 / np.sqrt(D))
        for no_tpp in (False, True):
            got, _ = run(torch, pool, batch, q, layer=layer, no_tpp=no_tpp)
            assert_close(got, want, f"fp8 c={c} G={G} layer={layer} no_tpp={no_tpp}")
    for step, n_add in enumerate((1, c + 3)):            # fill in place, then grow chunks
        for sid in batch:
            toks = [10**6 + 1000 * step + sid * 50 + j for j in range(n_add)]
            k16, kq = _fp8_rows(rng, L, n_add, Hkv, D, k_scale)
            v16, vq = _fp8_rows(rng, L, n_add, Hkv, D, v_scale)
            trie.append(sid, toks, kq, vq)
            pool.append(sid, toks, torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda())
        sched = pool.schedule(batch)
        got = decode_attention(pool, sched, torch.from_numpy(q).cuda(), layer=1).cpu().numpy()
        assert sched.device_status() == 0
        assert_close(got, A.decode_attention(trie, batch, 1, q, 1 / np.sqrt(D)), f"fp8 append {step}")
    torch.cuda.synchronize()
    _check_fp8_bytes(pool, trie, k_scale, v_scale)


def test_fp8_pool_shape_limits(torch_cuda):
    from prefix_shared_decode_gb300 import CAError, Pool
    with pytest.raises(CAError) as e:
        Pool(1, 2, 64, 16, 10, kv_dtype="fp8")            # fp8 needs head_dim 128
    assert e.value.name == "CA_ERR_UNSUPPORTED"
    with pytest.raises(CAError) as e:
        Pool(1, 2, 128, 16, 10, kv_dtype="fp8", k_scale=-1.0)
    assert e.value.name == "CA_ERR_INVALID"
    p = Pool(1, 2, 128, 16, 10, kv_dtype="fp8")
    assert p.kv_view().dtype == torch_cuda.uint8 and p.kv_bytes < Pool(1, 2, 128, 16, 10).kv_bytes


@pytest.mark.parametrize("q_len,causal,G,c,kv_dtype", [(2, False, 1, 16, "fp16"), (4, True, 1, 64, "fp16"),
                                                      (3, True, 2, 32, "fp16"), (8, True, 1, 32, "fp16"),
                                                      (2, True, 4, 64, "fp16"), (16, True, 4, 16, "fp16"),
                                                      (4, True, 1, 64, "fp8")])
def test_multi_token_queries_every_output(torch_cuda, q_len, causal, G, c, kv_dtype):
    """Several query tokens per sequence (q / out [b, q_len, H, D]), with and
    without the causal mask, against the definition."""
    from prefix_shared_decode_gb300 import Pool, decode_attention, decode_attention_host
    torch = torch_cuda
    Hkv, D, L = 2, 128, 2
    rng = np.random.default_rng(80 + q_len + c)
    seqs = random_segment_sequences(80 + q_len, 12, c, n_segments=10)
    pool = Pool(L, Hkv * G, D, c, 700, n_kv_heads=Hkv, kv_dtype=kv_dtype)
    trie = OracleTrie(c, 700)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((L, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((L, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        if kv_dtype == "fp8":
            trie.insert(i, toks, F8.dequantize(F8.quantize(k, 1.0), 1.0), F8.dequantize(F8.quantize(v, 1.0), 1.0))
        else:
            trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = [int(x) for x in rng.permutation(12) if len(seqs[x]) >= q_len][:10]
    q = rng.standard_normal((len(batch), q_len, Hkv * G, D), dtype=np.float32).astype(np.float16)
    for layer in range(L):
        want = A.decode_attention_multi(trie, batch, layer, q, 1 / np.sqrt(D), causal)
        for no_tpp in (False, True):
            sched = pool.schedule(batch, no_tpp=no_tpp, q_len=q_len, causal=causal)
            got = decode_attention(pool, sched, torch.from_numpy(q).cuda(), layer=layer).cpu().numpy()
            assert sched.device_status() == 0
            assert_close(got, want, f"q_len={q_len} causal={causal} G={G} layer={layer} no_tpp={no_tpp}")
    # the host-buffer entry point with the same schedule
    qh = torch.from_numpy(q).pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    decode_attention_host(pool, sched, qh, oh, layer=1)
    torch.cuda.synchronize()
    assert_close(oh.numpy(), A.decode_attention_multi(trie, batch, 1, q, 1 / np.sqrt(D), causal), "host io")


def test_speculative_verification_over_appended_drafts(torch_cuda):
    """Draft tokens are appended to each sequence (filling and growing
    chunks), then all of them are verified in one causal multi-token call;
    then they are accepted one more step."""
    from prefix_shared_decode_gb300 import Pool, decode_attention
    torch = torch_cuda
    c, H, D, q_len = 64, 4, 128, 5
    rng = np.random.default_rng(90)
    seqs = random_segment_sequences(90, 8, c, n_segments=6)
    pool, trie = Pool(1, H, D, c, 500), OracleTrie(c, 500)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = list(range(8))
    for step in range(3):
        for sid in batch:
            toks = [10**6 + 1000 * step + 50 * sid + j for j in range(q_len)]
            k = rng.standard_normal((1, q_len, H, D), dtype=np.float32).astype(np.float16)
            v = rng.standard_normal((1, q_len, H, D), dtype=np.float32).astype(np.float16)
            trie.append(sid, toks, k, v)
            pool.append(sid, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        q = rng.standard_normal((8, q_len, H, D), dtype=np.float32).astype(np.float16)
        sched = pool.schedule(batch, q_len=q_len, causal=True)
        got = decode_attention(pool, sched, torch.from_numpy(q).cuda()).cpu().numpy()
        assert sched.device_status() == 0
        assert_close(got, A.decode_attention_multi(trie, batch, 0, q, 1 / np.sqrt(D), causal=True),
                     f"step {step}")


@pytest.mark.parametrize("c,G,q_len,causal", [(16, 1, 1, False), (32, 1, 1, False), (32, 4, 1, False),
                                              (16, 2, 4, True), (32, 1, 8, True)])
def test_head_dim_256_every_output(torch_cuda, c, G, q_len, causal):
    """head_dim 256 (chunks of 16 or 32): the sequence-first lanes own 8 dims;
    on the tensor cores warp pairs split the head dims and add their score
    halves through shared memory."""
    from prefix_shared_decode_gb300 import Pool, decode_attention
    torch = torch_cuda
    Hkv, D, L = 2, 256, 2
    rng = np.random.default_rng(100 + c + G + q_len)
    seqs = random_segment_sequences(100 + c + q_len, 12, c, n_segments=10)
    pool = Pool(L, Hkv * G, D, c, 900, n_kv_heads=Hkv)
    trie = OracleTrie(c, 900)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((L, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((L, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = [int(x) for x in rng.permutation(12) if len(seqs[x]) >= q_len][:10]
    shape = (len(batch), Hkv * G, D) if q_len == 1 else (len(batch), q_len, Hkv * G, D)
    q = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    for layer in range(L):
        if q_len == 1:
            want = A.decode_attention(trie, batch, layer, q, 1 / np.sqrt(D))
        else:
            want = A.decode_attention_multi(trie, batch, layer, q, 1 / np.sqrt(D), causal)
        for no_tpp in (False, True):
            sched = pool.schedule(batch, no_tpp=no_tpp, q_len=q_len, causal=causal)
            got = decode_attention(pool, sched, torch.from_numpy(q).cuda(), layer=layer).cpu().numpy()
            assert sched.device_status() == 0
            assert_close(got, want, f"D=256 c={c} G={G} q_len={q_len} layer={layer} no_tpp={no_tpp}")


def test_edge_cases(torch_cuda):
    """One-token contexts, exactly one chunk, one chunk plus one token,
    identical sequences (no sequence-first work at all), a batch of one."""
    from prefix_shared_decode_gb300 import Pool
    torch = torch_cuda
    c, H, D = 64, 2, 128
    rng = np.random.default_rng(11)
    cases = {0: [1], 1: list(range(64)), 2: list(range(65)), 3: list(range(128)),
             4: list(range(128)), 5: list(range(64)) + [777], 6: [5, 6, 7]}
    pool = Pool(1, H, D, c, 64)
    trie = OracleTrie(c, 64)
    for sid, toks in cases.items():
        k = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
        trie.insert(sid, toks, k, v)
        pool.insert(sid, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    for batch in ([0], [3, 4], list(cases), [6, 2, 1]):
        q = rng.standard_normal((len(batch), H, D), dtype=np.float32).astype(np.float16)
        want = A.decode_attention(trie, batch, 0, q, 0.1)
        got, _ = run(torch, pool, batch, q, scale=0.1)
        assert_close(got, want, f"batch {batch}")
    # a one-token context returns that token's value exactly (up to fp16)
    q = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
    got, _ = run(torch, pool, [0], q)
    np.testing.assert_array_equal(got[0], trie.paths[0][0].v[0][0])


def test_more_than_64_sharers(torch_cuda):
    """A shared run with 70 sequences is split into query groups of <= 64."""
    from prefix_shared_decode_gb300 import Pool
    torch = torch_cuda
    c, H, D, b = 64, 2, 128, 70
    rng = np.random.default_rng(12)
    pool = Pool(1, H, D, c, 400)
    trie = OracleTrie(c, 400)
    pk = rng.standard_normal((1, 300, H, D), dtype=np.float32).astype(np.float16)
    pv = rng.standard_normal((1, 300, H, D), dtype=np.float32).astype(np.float16)
    for i in range(b):
        n_own = 1 + (i * 7) % 90
        k = np.concatenate([pk, rng.standard_normal((1, n_own, H, D), dtype=np.float32).astype(np.float16)], 1)
        v = np.concatenate([pv, rng.standard_normal((1, n_own, H, D), dtype=np.float32).astype(np.float16)], 1)
        toks = list(range(300)) + [10_000 * (i + 1) + j for j in range(n_own)]
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = list(range(b))[::-1]
    q = rng.standard_normal((b, H, D), dtype=np.float32).astype(np.float16)
    got, _ = run(torch, pool, batch, q)
    assert_close(got, A.decode_attention(trie, batch, 0, q, 1 / np.sqrt(D)), "70 sharers")


def test_kv_scatter_round_trip(torch_cuda):
    """Rows copied into the pool sit in kv[slot][layer][K|V][head][row][:]."""
    from prefix_shared_decode_gb300 import Pool
    torch = torch_cuda
    c, H, D, L = 32, 3, 64, 2
    rng = np.random.default_rng(13)
    pool = Pool(L, H, D, c, 32)
    toks = list(range(70))
    k = rng.standard_normal((L, 70, H, D), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((L, 70, H, D), dtype=np.float32).astype(np.float16)
    pool.insert(1, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    kv = pool.kv_view().cpu().numpy()          # [slots, L, 2, H, c, D]
    for i, slot in enumerate(pool.seq_slots(1)):
        n = min(c, 70 - i * c)
        for l in range(L):
            np.testing.assert_array_equal(kv[slot, l, 0, :, :n], k[l, i * c:i * c + n].transpose(1, 0, 2))
            np.testing.assert_array_equal(kv[slot, l, 1, :, :n], v[l, i * c:i * c + n].transpose(1, 0, 2))
    # a second insert sharing the first chunk copies only its own rows
    k2, v2 = -k, -v
    assert pool.insert(2, toks[:32] + [999] * 5, torch.from_numpy(np.ascontiguousarray(k2[:, :37])).cuda(),
                       torch.from_numpy(np.ascontiguousarray(v2[:, :37])).cuda()) == 32
    torch.cuda.synchronize()
    kv = pool.kv_view().cpu().numpy()
    s0, s1 = pool.seq_slots(2)
    np.testing.assert_array_equal(kv[s0, 0, 0, :, :32], k[0, :32].transpose(1, 0, 2))
    np.testing.assert_array_equal(kv[s1, 0, 0, :, :5], k2[0, 32:37].transpose(1, 0, 2))


def test_insert_batch_packed_rows(torch_cuda):
    """ca_insert_batch copies each sequence's rows out of one packed K/V
    buffer; attention over the result matches the oracle."""
    from prefix_shared_decode_gb300 import Pool
    torch = torch_cuda
    c, H, D, L = 32, 4, 128, 2
    rng = np.random.default_rng(14)
    seqs = random_segment_sequences(14, 9, c, n_segments=6)
    total = sum(len(t) for t in seqs)
    k = rng.standard_normal((L, total, H, D), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((L, total, H, D), dtype=np.float32).astype(np.float16)
    pool = Pool(L, H, D, c, 300)
    trie = OracleTrie(c, 300)
    shared = pool.insert_batch(list(range(9)), seqs, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    row = 0
    for i, t in enumerate(seqs):
        assert trie.insert(i, t, k[:, row:row + len(t)], v[:, row:row + len(t)]) == shared[i]
        row += len(t)
    batch = [8, 3, 0, 5, 1]
    q = rng.standard_normal((5, H, D), dtype=np.float32).astype(np.float16)
    for layer in (0, 1):
        got, _ = run(torch, pool, batch, q, layer=layer)
        assert_close(got, A.decode_attention(trie, batch, layer, q, 1 / np.sqrt(D)), f"layer {layer}")


def test_decode_time_appends(torch_cuda):
    """One decoded token per sequence per step: appends that only fill a
    partial chunk keep the cached schedule valid (the kernels read the
    chunk's token count from the pool), appends that grow a chunk make it
    stale and it is rebuilt; every step matches the oracle."""
    from prefix_shared_decode_gb300 import CAError, Pool, decode_attention
    torch = torch_cuda
    c, H, D = 32, 4, 128
    rng = np.random.default_rng(15)
    seqs = random_segment_sequences(15, 6, c, n_segments=5)
    pool, trie = Pool(1, H, D, c, 500), OracleTrie(c, 500)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = list(range(6))
    sched = pool.schedule(batch)
    cached_steps = rebuilt_steps = 0
    for step in range(45):
        grew = False
        for sid in batch:
            n_add = 1 if step % 15 else 40               # now and then a multi-token append
            toks = [10**6 + 1000 * step + sid * 50 + j for j in range(n_add)]
            k = rng.standard_normal((1, n_add, H, D), dtype=np.float32).astype(np.float16)
            v = rng.standard_normal((1, n_add, H, D), dtype=np.float32).astype(np.float16)
            g1 = trie.append(sid, toks, k, v)
            g2 = pool.append(sid, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
            assert g1 == g2
            grew |= g2 > 0
        handle = sched.handle.value
        if grew:
            q = torch.zeros((6, H, D), dtype=torch.float16, device="cuda")
            with pytest.raises(CAError):
                decode_attention(pool, sched, q)               # stale after growth
        sched = pool.schedule(batch, reuse=sched)
        if grew:
            rebuilt_steps += 1
        else:
            assert sched.handle.value == handle
            cached_steps += 1
        q = rng.standard_normal((6, H, D), dtype=np.float32).astype(np.float16)
        got = decode_attention(pool, sched, torch.from_numpy(q).cuda()).cpu().numpy()
        assert sched.device_status() == 0
        assert_close(got, A.decode_attention(trie, batch, 0, q, 1 / np.sqrt(D)), f"step {step}")
    assert cached_steps > 20 and rebuilt_steps > 2


def test_back_to_back_calls_and_pool_writes(torch_cuda):
    """Calls issued back to back with no host synchronisation.  While no
    insert or append has written a pool since its last call, a call streams
    the pool before the previous kernel in the stream has finished; the first
    call after an append waits for it.  Calls alternating between two pools,
    then an append to one of them followed at once by calls on it, all match
    the oracle (each call against the trie state it was issued on)."""
    from prefix_shared_decode_gb300 import Pool, decode_attention
    torch = torch_cuda
    c, H, D = 32, 4, 128
    rng = np.random.default_rng(23)
    seqs = random_segment_sequences(23, 8, c, n_segments=5)
    pools, tries = [], []
    for _ in range(2):
        pool, trie = Pool(1, H, D, c, 600), OracleTrie(c, 600)
        for i, toks in enumerate(seqs):
            k = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
            v = rng.standard_normal((1, len(toks), H, D), dtype=np.float32).astype(np.float16)
            trie.insert(i, toks, k, v)
            pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
        pools.append(pool)
        tries.append(trie)
    batch = list(range(8))
    scheds = [p.schedule(batch) for p in pools]
    qs = [rng.standard_normal((8, H, D), dtype=np.float32).astype(np.float16) for _ in range(8)]
    qd = [torch.from_numpy(q).cuda() for q in qs]
    add = {sid: ([2 * 10**6 + sid], rng.standard_normal((1, 1, H, D), dtype=np.float32).astype(np.float16),
                 rng.standard_normal((1, 1, H, D), dtype=np.float32).astype(np.float16)) for sid in batch}
    add_d = {sid: (torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()) for sid, (_, k, v) in add.items()}
    torch.cuda.synchronize()
    outs = [decode_attention(pools[i % 2], scheds[i % 2], qd[i]) for i in range(6)]
    for sid in batch:                                   # appends, right behind the calls
        pools[0].append(sid, add[sid][0], *add_d[sid])
    sched0 = pools[0].schedule(batch, reuse=scheds[0])
    outs += [decode_attention(pools[0], sched0, qd[i]) for i in (6, 7)]
    torch.cuda.synchronize()
    assert scheds[1].device_status() == 0 and sched0.device_status() == 0
    for i in range(6):
        want = A.decode_attention(tries[i % 2], batch, 0, qs[i], 1 / np.sqrt(D))
        assert_close(outs[i].cpu().numpy(), want, f"call {i}")
    for sid in batch:
        tries[0].append(sid, *add[sid])
    for j, i in enumerate((6, 7)):
        want = A.decode_attention(tries[0], batch, 0, qs[i], 1 / np.sqrt(D))
        assert_close(outs[6 + j].cpu().numpy(), want, f"call {i} after the append")


def test_host_io_entry_and_repeat_calls(torch_cuda):
    from prefix_shared_decode_gb300 import decode_attention, decode_attention_host
    torch = torch_cuda
    wl = workloads.make("tiny")
    pool = load(torch, wl)
    sched = pool.schedule(wl.seq_ids())
    q = torch.from_numpy(wl.queries(3)).cuda()
    a = decode_attention(pool, sched, q).cpu()
    b = decode_attention(pool, sched, q).cpu()
    assert torch.equal(a, b)                           # counters reset, deterministic merge
    qh = q.cpu().pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    decode_attention_host(pool, sched, qh, oh)
    torch.cuda.synchronize()
    assert torch.equal(oh, a)
    assert sched.device_status() == 0


def test_kernel_launch_counter(torch_cuda):
    """Each decode call launches two kernels (attention, merge); an insert
    launches one KV scatter per 128 new chunks."""
    from prefix_shared_decode_gb300 import decode_attention, kernel_launches
    torch = torch_cuda
    wl = workloads.make("tiny")
    pool = load(torch, wl)
    sched = pool.schedule(wl.seq_ids())
    q = torch.from_numpy(wl.queries(0)).cuda()
    n0 = kernel_launches()
    for _ in range(3):
        decode_attention(pool, sched, q)
    assert kernel_launches() - n0 == 6
    n1 = kernel_launches()
    k = torch.zeros((1, 40, wl.kv_heads, wl.head_dim), dtype=torch.float16, device="cuda")
    pool.insert(1000, list(range(900000, 900040)), k, k)   # 3 new chunks of 16
    torch.cuda.synchronize()
    assert kernel_launches() - n1 == 1


def test_two_ctas_per_sm(torch_cuda):
    """The persistent grid holds two CTAs per SM (registers and shared memory
    of the largest instantiation fit twice)."""
    from prefix_shared_decode_gb300 import Pool
    pool = Pool(1, 32, 128, 64, 64)
    toks = list(range(64 * 40))
    k = torch_cuda.zeros((1, len(toks), 32, 128), dtype=torch_cuda.float16, device="cuda")
    pool.insert(0, toks, k, k)
    sms = torch_cuda.cuda.get_device_properties(0).multi_processor_count
    assert pool.schedule([0]).plan()["grid"] == min(2 * sms, 40 * 32)


def test_stale_schedule_is_rejected(torch_cuda):
    from prefix_shared_decode_gb300 import CAError, decode_attention
    torch = torch_cuda
    wl = workloads.make("tiny")
    pool = load(torch, wl)
    sched = pool.schedule(wl.seq_ids())
    pool.remove(wl.seq_ids()[0])
    with pytest.raises(CAError) as e:
        decode_attention(pool, sched, torch.from_numpy(wl.queries(0)).cuda())
    assert e.value.name == "CA_ERR_STALE"


@pytest.mark.parametrize("name", ["llama7b_p1024", "sweep_s2048_b32", "sweep_s2048_b64",
                                  "sweep_s4096_b32", "sweep_s4096_b64", "no_sharing", "gqa_p1024",
                                  "llama7b_p1024_fp8", "sweep_s4096_b64_fp8", "llama7b_p1024_q4",
                                  "d256_p1024"])
def test_full_size_workloads_every_output(torch_cuda, name):
    """The benchmark's launch configuration at full size (the same pool,
    schedule and kernel variant the benchmark times): every sequence, head
    and query token is compared with the oracle; max and mean are taken over
    all outputs of the call."""
    wl = workloads.make(name)
    pool = load(torch_cuda, wl)
    batch = wl.seq_ids()
    q = wl.queries(0)
    got, sched = run(torch_cuda, pool, batch, q, q_len=wl.q_len)
    assert_close(got, plain_definition(wl, batch, q), name)


def test_multi_tenant_with_churn_every_output(torch_cuda):
    """The multi-tenant tree with four churn steps (8 sequences removed and
    8 inserted each, the schedule rebuilt and uploaded through both plan
    staging buffers twice): every output of every step against the oracle."""
    from prefix_shared_decode_gb300 import decode_attention
    torch = torch_cuda
    wl = workloads.make("multi_tenant")
    pool = load(torch, wl)
    staging = {}
    sched = None
    for step in range(5):
        if step:
            removed, inserted = wl.churn_step()
            for sid in removed:
                pool.remove(sid)
            for sid in inserted:
                insert_sequence(pool, wl, sid, staging=staging)
        batch = wl.seq_ids()
        sched = pool.schedule(batch, reuse=sched)
        q = wl.queries(step)
        got = decode_attention(pool, sched, torch.from_numpy(q).cuda()).cpu().numpy()
        assert sched.device_status() == 0
        assert_close(got, plain_definition(wl, batch, q), f"multi_tenant step {step}")
