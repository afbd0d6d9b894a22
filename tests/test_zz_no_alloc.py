"""ca_decode_attention_static_ws: decode attention that allocates nothing.

Some callers of this library cannot allocate device memory when they run
attention: a component inside a server that has already reserved the whole
device memory budget for its own pool, code on a latency-critical path where
cudaMalloc / cudaFree would synchronise the device, or a plugin whose host
forbids allocation inside its callbacks.  For them the library keeps its own
fixed scratch buffer (CA_STATIC_WS_BYTES per GPU) for the partial results, so
the call needs no workspace argument.

These tests call that entry point through the C ABI and compare it with
ca_decode_attention (caller-provided workspace) on the same inputs, for two
calls in a row, within the parity tolerance used by every GPU test (max abs
2e-3, mean abs 2e-4).  The file is named to be collected last."""
import numpy as np
import pytest

import workloads
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


def test_static_scratch_matches_workspace_entry_two_calls(lib, torch_cuda):
    from prefix_shared_decode_gb300 import Pool, capi, decode_attention
    torch = torch_cuda
    wl = workloads.make("llama7b_p1024")
    pool = Pool(wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, capacity_for(wl))
    staging = {}
    for sid in wl.seq_ids():
        insert_sequence(pool, wl, sid, staging=staging)
    sched = pool.schedule(wl.seq_ids())
    assert sched.workspace_bytes() <= capi.CA_STATIC_WS_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        q = torch.from_numpy(wl.queries(call)).cuda()
        want = decode_attention(pool, sched, q, scale=wl.scale).cpu().numpy().astype(np.float64)
        out = torch.full_like(q, float("nan"))
        assert static_call(lib, pool, sched, q, out, wl.scale, stream) == 0
        assert sched.device_status() == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        err = np.abs(got - want)
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN, (call, err.max(), err.mean())


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
