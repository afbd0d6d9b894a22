"""Opt-in soak: many steps of the multi-tenant tree with churn (8 removes and
8 inserts per step, the schedule rebuilt every step through the two plan
staging buffers, the tail-queue counter reset by every merge), the device
status read and the output compared with the oracle every 100 steps.  Runs
only when CA_SOAK_STEPS is set (e.g. 2000: ~7 minutes, mostly drawing the
inserted rows on the host)."""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.skipif(not os.environ.get("CA_SOAK_STEPS"), reason="set CA_SOAK_STEPS to run the soak")
def test_multi_tenant_soak():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import workloads
    from prefix_shared_decode_gb300 import Pool, decode_attention
    from tests.oracle_parallel import plain_definition
    from workloads.device import capacity_for, insert_sequence
    steps = int(os.environ["CA_SOAK_STEPS"])
    wl = workloads.make("multi_tenant")
    pool = Pool(wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, capacity_for(wl, headroom=1.5))
    staging = {}
    for sid in wl.seq_ids():
        insert_sequence(pool, wl, sid, staging=staging)
    sched = None
    for step in range(steps):
        if step:
            removed, inserted = wl.churn_step()
            pool.remove_batch(removed)
            for sid in inserted:
                insert_sequence(pool, wl, sid, staging=staging)
        batch = wl.seq_ids()
        sched = pool.schedule(batch, reuse=sched)
        q = wl.queries(step % 7)
        out = decode_attention(pool, sched, torch.from_numpy(q).cuda())
        if step % 100 == 0 or step == steps - 1:
            assert sched.device_status() == 0, step
            err = np.abs(out.cpu().numpy().astype(np.float64) - plain_definition(wl, batch, q))
            assert err.max() <= 2e-3 and err.mean() <= 2e-4, (step, err.max(), err.mean())
    assert pool.stats()["live_seqs"] == len(wl.seqs)
