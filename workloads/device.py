"""Load a synthetic workload into a device pool (harness code: token lists
and K/V rows only, no attention arithmetic)."""
from __future__ import annotations

import numpy as np


def insert_sequence(pool, wl, seq_id: int, stream=None, staging: dict | None = None) -> int:
    """Insert one sequence of workload ``wl`` into ``pool``.  Only the rows
    past the pool's matched prefix are generated and copied to the device
    (the library does not read matched rows).  Returns the shared tokens."""
    import torch
    toks = wl.tokens(seq_id)
    n = len(toks)
    matched = pool.match_prefix(toks)
    k_new, v_new = wl.kv_rows(seq_id, start=matched)
    shape = (wl.n_layers, n, wl.kv_heads, wl.head_dim)
    key = ("kv", shape)
    if staging is not None and key in staging:
        k_dev, v_dev = staging[key]
    else:
        k_dev = torch.empty(shape, dtype=torch.float16, device="cuda")
        v_dev = torch.empty(shape, dtype=torch.float16, device="cuda")
        if staging is not None:
            staging[key] = (k_dev, v_dev)
    if n > matched:
        k_dev[:, matched:].copy_(torch.from_numpy(np.ascontiguousarray(k_new)), non_blocking=False)
        v_dev[:, matched:].copy_(torch.from_numpy(np.ascontiguousarray(v_new)), non_blocking=False)
    shared = pool.insert(seq_id, toks, k_dev, v_dev, stream=stream)
    assert shared == matched
    return shared


def capacity_for(wl, headroom: float = 1.25, extra: int = 64) -> int:
    """Chunk slots for the workload's live sequences (with room for churn)."""
    c = wl.chunk
    seen, slots = set(), 0
    for segs in wl.seqs.values():
        pos = 0
        for s in segs:
            pos += wl.seg_len[s]
        slots += -(-pos // c)
    return int(slots * headroom) + extra
