"""Decode attention recorded into CUDA graphs and replayed: every replay
matches the fp64 oracle (and the same call issued directly, bit for bit),
across decode-time appends that keep the schedule, and a replay after a
schedule rebuild is refused [ChunkAttention (arXiv 2402.15220v4 summary)
§3.1 and §3.2: the prefix tree grows by a token per sequence per step, and
its context is rebuilt only when the tree's chunk structure changes]."""
import numpy as np
import pytest

from oracle import attention as A
from oracle.pakv import OracleTrie
from tests.test_gpu_parity import assert_close
from tests.treegen import random_segment_sequences

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda(lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _tree(torch, seed, n_seqs, c, H, D, L, capacity):
    from prefix_shared_decode_gb300 import Pool
    rng = np.random.default_rng(seed)
    seqs = random_segment_sequences(seed, n_seqs, c, n_segments=5)
    pool, trie = Pool(L, H, D, c, capacity), OracleTrie(c, capacity)
    for i, toks in enumerate(seqs):
        k = rng.standard_normal((L, len(toks), H, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((L, len(toks), H, D), dtype=np.float32).astype(np.float16)
        trie.insert(i, toks, k, v)
        pool.insert(i, toks, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    return pool, trie, rng


def test_graph_replay_over_decode_steps(torch_cuda):
    """Two layers' calls in one graph.  Each step appends one token per
    sequence, writes new queries into the captured q buffers and replays.
    Appends inside the partial last chunks keep the graph valid; a grown
    chunk makes the replay raise, and the graph is captured again on the
    rebuilt schedule."""
    from prefix_shared_decode_gb300 import CAError, DecodeGraph, decode_attention, kernel_launches
    torch = torch_cuda
    c, H, D, L, b = 32, 4, 128, 2, 6
    pool, trie, rng = _tree(torch, 31, b, c, H, D, L, 500)
    batch = list(range(b))
    sched = pool.schedule(batch)
    qb = [torch.zeros((b, H, D), dtype=torch.float16, device="cuda") for _ in range(L)]
    ob = [torch.zeros((b, H, D), dtype=torch.float16, device="cuda") for _ in range(L)]
    graph = DecodeGraph(pool, sched, [(layer, qb[layer], ob[layer]) for layer in range(L)])
    replays = captures = 0
    for step in range(40):
        grew = False
        for sid in batch:
            tok = [10**6 + 1000 * step + sid]
            k = rng.standard_normal((L, 1, H, D), dtype=np.float32).astype(np.float16)
            v = rng.standard_normal((L, 1, H, D), dtype=np.float32).astype(np.float16)
            g1 = trie.append(sid, tok, k, v)
            g2 = pool.append(sid, tok, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
            assert g1 == g2
            grew |= g2 > 0
        if grew:
            with pytest.raises(CAError):
                graph.replay()
            sched = pool.schedule(batch, reuse=sched)
            graph = DecodeGraph(pool, sched, [(layer, qb[layer], ob[layer]) for layer in range(L)])
            captures += 1
        q = [rng.standard_normal((b, H, D), dtype=np.float32).astype(np.float16) for _ in range(L)]
        for layer in range(L):
            qb[layer].copy_(torch.from_numpy(q[layer]))
        before = kernel_launches()
        graph.replay()
        assert kernel_launches() == before          # no launch went through the host path
        torch.cuda.synchronize()
        assert sched.device_status() == 0
        replays += 1
        for layer in range(L):
            got = ob[layer].cpu().numpy()
            assert_close(got, A.decode_attention(trie, batch, layer, q[layer], 1 / np.sqrt(D)),
                         f"step {step} layer {layer}")
            direct = decode_attention(pool, sched, qb[layer], layer=layer).cpu().numpy()
            np.testing.assert_array_equal(got, direct, err_msg=f"step {step} layer {layer}")
    assert replays == 40 and captures >= 1


def test_graph_of_many_calls_replayed_back_to_back(torch_cuda):
    """Sixteen calls in one graph (layers alternating, each with its own
    query buffer), replayed five times with no host synchronisation in
    between: inside the graph the kernels of consecutive calls overlap
    through their programmatic dependencies."""
    from prefix_shared_decode_gb300 import DecodeGraph
    torch = torch_cuda
    c, H, D, L, b, n = 64, 8, 128, 2, 8, 16
    pool, trie, rng = _tree(torch, 47, b, c, H, D, L, 400)
    batch = list(range(b))
    sched = pool.schedule(batch)
    q = [rng.standard_normal((b, H, D), dtype=np.float32).astype(np.float16) for _ in range(n)]
    qb = [torch.from_numpy(x).cuda() for x in q]
    ob = [torch.zeros((b, H, D), dtype=torch.float16, device="cuda") for _ in range(n)]
    graph = DecodeGraph(pool, sched, [(i % L, qb[i], ob[i]) for i in range(n)])
    for x in ob:
        x.zero_()
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    assert sched.device_status() == 0
    for i in range(n):
        assert_close(ob[i].cpu().numpy(), A.decode_attention(trie, batch, i % L, q[i], 1 / np.sqrt(D)),
                     f"call {i}")


def test_default_stream_is_torchs_current_stream(torch_cuda):
    """Calls without a stream argument run on torch's current stream: the
    default stream, a side stream, and the capture stream of a graph."""
    from prefix_shared_decode_gb300 import _stream_ptr
    torch = torch_cuda
    assert _stream_ptr(None) == (torch.cuda.current_stream().cuda_stream or None)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert _stream_ptr(None) == side.cuda_stream
    g = torch.cuda.CUDAGraph()
    x = torch.zeros(4, device="cuda")
    with torch.cuda.graph(g):
        seen = _stream_ptr(None)
        x.add_(1)
        assert seen == torch.cuda.current_stream().cuda_stream
    g.replay()
    torch.cuda.synchronize()
    assert x.sum().item() == 4
