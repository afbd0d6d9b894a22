"""ca_decode_attention_static_ws: decode attention that allocates nothing.

Some callers of this library cannot allocate device memory when they run
attention: a component inside a server that has already reserved the whole
device memory budget for its own pool, code on a latency-critical path where
cudaMalloc / cudaFree would synchronise the device, or a plugin whose host
forbids allocation inside its callbacks.  For them the library keeps its own
fixed scratch buffer (CA_STATIC_WS_BYTES per GPU) for the partial results, so
the call needs no workspace argument.

These tests call that entry point through the C ABI, two calls in a row,
and compare each output with ca_decode_attention (caller-provided workspace)
on the same inputs and with the fp64 oracle, within the parity tolerance
used by every GPU test (max abs 2e-3, mean abs 2e-4).  The shared buffer
keeps the last call's contents, so a schedule with a smaller, differently
laid out set of partials also runs right after a large one.  The file is
named to be collected last."""
import numpy as np
import pytest

import workloads
from oracle import attention as A
from oracle.pakv import OracleTrie
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


def static_call(lib, pool, sched, q, out, scale, stream):
    return lib.ca_decode_attention_static_ws(pool.handle, sched.handle, 0, q.data_ptr(),
                                             out.data_ptr(), float(scale), stream)


def assert_close(got, want, what):
    err = np.abs(got.astype(np.float64) - want)
    assert np.isfinite(got).all(), what
    assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (what, err.max(), err.mean())


def run_static_twice(lib, torch, pool, sched, queries, scale, oracle_out):
    """Two static-scratch calls in a row, each compared with the workspace
    entry point and with the oracle."""
    from prefix_shared_decode_gb300 import decode_attention
    stream = torch.cuda.current_stream().cuda_stream
    for call, qn in enumerate(queries):
        q = torch.from_numpy(qn).cuda()
        want_ws = decode_attention(pool, sched, q, scale=scale).cpu().numpy().astype(np.float64)
        out = torch.full_like(q, float("nan"))
        assert static_call(lib, pool, sched, q, out, scale, stream) == 0
        assert sched.device_status() == 0
        got = out.cpu().numpy()
        assert_close(got, want_ws, f"call {call} vs workspace entry point")
        assert_close(got, oracle_out(qn), f"call {call} vs oracle")


def test_static_scratch_matches_workspace_entry_and_oracle_two_calls(lib, torch_cuda):
    from prefix_shared_decode_gb300 import Pool, capi
    wl = workloads.make("llama7b_p1024")
    pool = Pool(wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, capacity_for(wl))
    staging = {}
    for sid in wl.seq_ids():
        insert_sequence(pool, wl, sid, staging=staging)
    batch = wl.seq_ids()
    sched = pool.schedule(batch)
    assert sched.workspace_bytes() <= capi.CA_STATIC_WS_BYTES
    def oracle_out(q):
        return plain_definition(wl, batch, q)

    run_static_twice(lib, torch_cuda, pool, sched, [wl.queries(0), wl.queries(1)], wl.scale, oracle_out)


def test_static_scratch_smaller_layout_after_a_large_one(lib, torch_cuda):
    """A large call first leaves the buffer full of its partials; then a
    small grouped-query, multi-token causal schedule (other partial ids,
    other counts per pair) runs through the same buffer, twice."""
    from prefix_shared_decode_gb300 import Pool, decode_attention
    torch = torch_cuda
    big = workloads.make("sweep_s2048_b64")
    pool_big = Pool(big.n_layers, big.n_heads, big.head_dim, big.chunk, capacity_for(big))
    staging = {}
    for sid in big.seq_ids():
        insert_sequence(pool_big, big, sid, staging=staging)
    sched_big = pool_big.schedule(big.seq_ids())
    q_big = torch.from_numpy(big.queries(0)).cuda()
    out_big = torch.empty_like(q_big)
    stream = torch.cuda.current_stream().cuda_stream
    assert static_call(lib, pool_big, sched_big, q_big, out_big, big.scale, stream) == 0
    assert sched_big.device_status() == 0
    want_big = decode_attention(pool_big, sched_big, q_big, scale=big.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_big, want_big)          # same kernels, same partial order: bitwise

    G, Hkv, D, c, q_len = 4, 2, 128, 32, 2
    rng = np.random.default_rng(77)
    seqs = random_segment_sequences(77, 9, c, n_segments=8)
    pool = Pool(1, Hkv * G, D, c, 400, n_kv_heads=Hkv)
    trie = OracleTrie(c, 400)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((1, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((1, len(toks), Hkv, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    batch = [i for i in range(9) if len(seqs[i]) >= q_len][:7]
    sched = pool.schedule(batch, q_len=q_len, causal=True)
    assert sched.workspace_bytes() < sched_big.workspace_bytes()
    qs = [rng.standard_normal((len(batch), q_len, Hkv * G, D), dtype=np.float32).astype(np.float16)
          for _ in range(2)]

    def oracle_out(q):
        return A.decode_attention_multi(trie, batch, 0, q, 1 / np.sqrt(D), causal=True)

    run_static_twice(lib, torch, pool, sched, qs, 1 / np.sqrt(D), oracle_out)


def test_static_scratch_rejects_schedules_that_do_not_fit(lib, torch_cuda):
    """640 sequences x 32 heads x 2 partials of 520 bytes is 21 MB of
    partials, more than the 16 MiB buffer: the call must refuse it."""
    from prefix_shared_decode_gb300 import Pool, capi
    torch = torch_cuda
    b, H, D, c = 640, 32, 128, 16
    pool = Pool(1, H, D, c, b + 8)
    k = torch.zeros((1, c + 1, H, D), dtype=torch.float16, device="cuda")
    for i in range(b):
        pool.insert(i, list(range(c)) + [100_000 + i], k, k)
    sched = pool.schedule(list(range(b)))
    assert sched.workspace_bytes() > capi.CA_STATIC_WS_BYTES
    q = torch.zeros((b, H, D), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    st = static_call(lib, pool, sched, q, out, 0.1, torch.cuda.current_stream().cuda_stream)
    assert capi.ERRORS.get(st) == "CA_ERR_SCRATCH_LIMIT"
