"""The oracle's plain definition over a whole batch, one sequence per task,
spread over the host cores (test infrastructure).

Each task carries what identifies its inputs (the workload seed, the
sequence's segment ids and lengths, the shape) and its query rows; the
worker draws the segments' K/V from ``workloads.segment_kv`` (the generator
both sides use) and calls ``oracle.attention.softmax_attention`` on them:
the oracle's arithmetic, unchanged, only called in several processes.  The
pool is started with ``spawn``, so it is safe after CUDA has been
initialised in the parent."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_pool = None
_segments: dict = {}          # worker-side cache: (seed, seg_id, n, L, H, D) -> (k, v)


def _segment(key):
    if key not in _segments:
        import workloads
        if len(_segments) > 16:
            _segments.clear()
        _segments[key] = workloads.segment_kv(*key)
    return _segments[key]


def _one(task):
    from oracle import attention as A
    from oracle import fp8 as F8
    seed, segs, L, Hkv, D, kv_dtype, q_len, scale, q = task
    ks, vs = [], []
    for seg_id, n in segs:
        k, v = _segment((seed, seg_id, n, L, Hkv, D))
        ks.append(k[0])
        vs.append(v[0])
    k, v = np.concatenate(ks), np.concatenate(vs)
    if kv_dtype == "fp8":                              # the dequantised rows (scales 1)
        k, v = F8.dequantize(F8.quantize(k, 1.0), 1.0), F8.dequantize(F8.quantize(v, 1.0), 1.0)
    if q_len == 1:
        return A.softmax_attention(q, k, v, scale)
    n = k.shape[0]
    return np.stack([A.softmax_attention(q[j], k[:n - q_len + j + 1], v[:n - q_len + j + 1], scale)
                     for j in range(q_len)])


def workers() -> int:
    return max(1, min(16, len(os.sched_getaffinity(0))))


def pool():
    global _pool
    if _pool is None:
        _pool = mp.get_context("spawn").Pool(workers())
    return _pool


def plain_definition(wl, batch, q) -> np.ndarray:
    """Layer-0 decode attention of every sequence of ``batch`` (rows of
    ``q``) by the plain definition: [b, H, D], or [b, q_len, H, D] where
    token j of n context tokens sees the first n - q_len + j + 1."""
    tasks = [(wl.seed, [(s, wl.seg_len[s]) for s in wl.seqs[sid]], wl.n_layers, wl.kv_heads,
              wl.head_dim, wl.kv_dtype, wl.q_len, wl.scale, q[i]) for i, sid in enumerate(batch)]
    return np.stack(pool().map(_one, tasks, chunksize=1))
