"""Prefix-shared decode attention (ChunkAttention's hot path) for GB300.

A thin binding over libchunk_attention (include/chunk_attention.h): every
step of the path runs in the library's C++ host code and sm_103a CUDA
kernels; this module only marshals arguments.  PyTorch supplies device
memory and streams.

    pool = Pool(n_layers=1, n_heads=32, head_dim=128, chunk=64, capacity_slots=...)
    pool.insert(seq_id, tokens, k, v)          # K/V fp16 [L, n, H, D] on the GPU
    sched = pool.schedule(seq_ids)             # per-step two-phase tables
    out = decode_attention(pool, sched, q)     # q fp16 [b, H, D] on the GPU
"""
from __future__ import annotations

import ctypes as C
import math

import numpy as np

from . import capi
from .capi import CAError, check

__all__ = ["Pool", "Schedule", "DecodeGraph", "decode_attention", "decode_attention_host", "kernel_launches",
           "CAError"]


_cuda_ok = None


def _stream_ptr(stream) -> int | None:
    """The raw handle of ``stream`` (default: torch's current stream on the
    current device; 0 / None is the legacy default stream)."""
    if stream is None:
        global _cuda_ok
        import torch
        if _cuda_ok is None:
            _cuda_ok = torch.cuda.is_available()
        if not _cuda_ok:
            return None
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)   # no Stream object per call
        if raw is not None:
            return raw(torch.cuda.current_device()) or None
        stream = torch.cuda.current_stream()
    return int(getattr(stream, "cuda_stream", stream)) or None


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class Pool:
    """A prefix-aware KV cache: the chunk trie and its device pool.

    With ``host_only=True`` no GPU memory is touched (trie, allocator and
    schedule tables only).  ``kv_dtype="fp8"`` stores K and V as FP8 E4M3
    with the given scales (inserted rows stay fp16; the library quantises)."""

    def __init__(self, n_layers: int, n_heads: int, head_dim: int, chunk: int,
                 capacity_slots: int, no_sharing: bool = False, host_only: bool = False,
                 device=None, n_kv_heads: int | None = None, kv_dtype: str = "fp16",
                 k_scale: float = 1.0, v_scale: float = 1.0):
        L = capi.lib()
        if kv_dtype not in ("fp16", "fp8"):
            raise ValueError("kv_dtype must be 'fp16' or 'fp8'")
        flags = (capi.CA_NO_SHARING if no_sharing else 0) | (capi.CA_KV_FP8 if kv_dtype == "fp8" else 0)
        self.cfg = capi.PoolConfigEx(capi.PoolConfig(n_layers, n_heads, head_dim, chunk, capacity_slots, flags),
                                     n_kv_heads or 0, float(k_scale), float(v_scale))
        self.kv_dtype, self.k_scale, self.v_scale = kv_dtype, float(k_scale), float(v_scale)
        self.n_layers, self.n_heads, self.head_dim, self.chunk = n_layers, n_heads, head_dim, chunk
        self.n_kv_heads = n_kv_heads or n_heads
        self.capacity_slots = capacity_slots
        nbytes = C.c_size_t()
        check(L.ca_pool_bytes_ex(C.byref(self.cfg), C.byref(nbytes)), "ca_pool_bytes_ex")
        self.kv_bytes = nbytes.value
        self._kv = None
        ptr = None
        if not host_only:
            import torch
            dev = torch.device(device if device is not None else "cuda")
            # over-allocate so the pool can start on a 1024-byte boundary
            self._kv = torch.empty(self.kv_bytes + 1024, dtype=torch.uint8, device=dev)
            base = self._kv.data_ptr()
            ptr = (base + 1023) // 1024 * 1024
            self._kv_offset = ptr - base
        self.host_only = host_only
        h = C.c_void_p()
        check(L.ca_pool_create_ex(C.byref(self.cfg), ptr, self.kv_bytes, C.byref(h)), "ca_pool_create_ex")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            capi.lib().ca_pool_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def _tile_bytes(self) -> int:
        eb = 1 if self.kv_dtype == "fp8" else 2
        return self.capacity_slots * self.n_layers * 2 * self.n_kv_heads * self.chunk * self.head_dim * eb

    def kv_view(self):
        """The device pool's K/V tiles as [slots, L, 2, H, c, D] (a view):
        fp16, or the E4M3 codes as uint8 for an fp8 pool."""
        import torch
        t = self._kv[self._kv_offset:self._kv_offset + self._tile_bytes()]
        if self.kv_dtype == "fp16":
            t = t.view(torch.float16)
        return t.view(self.capacity_slots, self.n_layers, 2, self.n_kv_heads, self.chunk, self.head_dim)

    def slot_ntok_view(self):
        """The pool's per-slot valid-token counts, int32 [slots] (a view)."""
        import torch
        a = self._kv_offset + self._tile_bytes()
        return self._kv[a:a + 4 * self.capacity_slots].view(torch.int32)

    def match_prefix(self, tokens) -> int:
        tok = _i32(tokens)
        n = C.c_int32()
        check(capi.lib().ca_match_prefix(self._h, tok.ctypes.data_as(C.POINTER(C.c_int32)),
                                          len(tok), C.byref(n)), "ca_match_prefix")
        return n.value

    def insert(self, seq_id: int, tokens, k=None, v=None, stream=None) -> int:
        """Insert a sequence; k, v are fp16 device tensors [L, n, Hkv, D]
        (None for a host-only pool).  Returns the number of shared tokens."""
        tok = _i32(tokens)
        kp = vp = None
        if k is not None:
            assert k.is_contiguous() and v.is_contiguous()
            assert tuple(k.shape) == (self.n_layers, len(tok), self.n_kv_heads, self.head_dim)
            kp, vp = k.data_ptr(), v.data_ptr()
        shared = C.c_int32()
        check(capi.lib().ca_insert_tokens(self._h, int(seq_id), tok.ctypes.data_as(C.POINTER(C.c_int32)),
                                          len(tok), kp, vp,
                                          None if self.host_only else _stream_ptr(stream),
                                          C.byref(shared)), "ca_insert_tokens")
        return shared.value

    def insert_batch(self, seq_ids, token_lists, k=None, v=None, stream=None, lengths=None) -> list[int]:
        """Insert several sequences in one call; k, v are fp16 device tensors
        [L, sum(lengths), H, D] holding the sequences' rows back to back (None
        for a host-only pool).  All or nothing.  Returns the shared tokens.
        ``token_lists`` is a list of token arrays, or (with ``lengths``) the
        already concatenated tokens."""
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        if lengths is None:
            lens = np.ascontiguousarray(np.array([len(t) for t in token_lists], dtype=np.int32))
            tok = np.ascontiguousarray(np.concatenate([np.asarray(t, dtype=np.int32) for t in token_lists]))
        else:
            lens = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
            tok = np.ascontiguousarray(np.asarray(token_lists, dtype=np.int32))
        kp = vp = None
        if k is not None:
            assert k.is_contiguous() and v.is_contiguous()
            assert tuple(k.shape) == (self.n_layers, int(lens.sum()), self.n_kv_heads, self.head_dim)
            kp, vp = k.data_ptr(), v.data_ptr()
        shared = np.zeros(len(ids), dtype=np.int32)
        P32 = C.POINTER(C.c_int32)
        check(capi.lib().ca_insert_batch(self._h, len(ids), ids.ctypes.data_as(C.POINTER(C.c_int64)),
                                         tok.ctypes.data_as(P32), lens.ctypes.data_as(P32), kp, vp,
                                         None if self.host_only else _stream_ptr(stream),
                                         shared.ctypes.data_as(P32)), "ca_insert_batch")
        return shared.tolist()

    def append(self, seq_id: int, tokens, k=None, v=None, stream=None) -> int:
        """Append decoded tokens to a sequence; k, v are fp16 device tensors
        [L, n, H, D] for the new tokens (None for a host-only pool).  Returns
        the number of chunks grown (0: the partial last chunk took them)."""
        tok = _i32(tokens)
        kp = vp = None
        if k is not None:
            assert k.is_contiguous() and v.is_contiguous()
            assert tuple(k.shape) == (self.n_layers, len(tok), self.n_kv_heads, self.head_dim)
            kp, vp = k.data_ptr(), v.data_ptr()
        grown = C.c_int32()
        check(capi.lib().ca_append_tokens(self._h, int(seq_id), tok.ctypes.data_as(C.POINTER(C.c_int32)),
                                          len(tok), kp, vp, None if self.host_only else _stream_ptr(stream),
                                          C.byref(grown)), "ca_append_tokens")
        return grown.value

    def remove(self, seq_id: int) -> None:
        check(capi.lib().ca_remove_seq(self._h, int(seq_id)), "ca_remove_seq")

    def remove_batch(self, seq_ids) -> None:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        check(capi.lib().ca_remove_batch(self._h, len(ids), ids.ctypes.data_as(C.POINTER(C.c_int64))),
              "ca_remove_batch")

    def _generation(self) -> int:
        st = self.__dict__.setdefault("_stats_buf", capi.Stats())
        check(capi.lib().ca_pool_stats(self._h, C.byref(st)), "ca_pool_stats")
        return st.generation

    def stats(self) -> dict:
        s = capi.Stats()
        check(capi.lib().ca_pool_stats(self._h, C.byref(s)), "ca_pool_stats")
        return {f: getattr(s, f) for f, _ in capi.Stats._fields_}

    def seq_slots(self, seq_id: int) -> list[int]:
        n = C.c_int32()
        check(capi.lib().ca_seq_slots(self._h, int(seq_id), None, 0, C.byref(n)), "ca_seq_slots")
        buf = (C.c_int32 * max(1, n.value))()
        check(capi.lib().ca_seq_slots(self._h, int(seq_id), buf, n.value, C.byref(n)), "ca_seq_slots")
        return list(buf)[:n.value]

    def schedule(self, seq_ids, no_tpp: bool = False, reuse: "Schedule | None" = None,
                 stream=None, q_len: int = 1, causal: bool = False) -> "Schedule":
        """Per-step tables for the batch ``seq_ids`` (rows of q / out in that
        order).  Passing the previous schedule reuses it when nothing changed.
        ``q_len`` > 1: that many query tokens per sequence (q / out become
        [b, q_len, H, D]); ``causal``: token j sees context tokens
        [0, len - q_len + j] only."""
        s = reuse if reuse is not None else Schedule(self)
        # A decode loop passes the same batch list every step: its int64 copy
        # (and that copy's address) is kept, so the per-step call converts
        # nothing; the library itself decides whether the tables are current.
        if isinstance(seq_ids, list) and s._ids_list is not None and seq_ids == s._ids_list:
            ids = s._ids
        else:
            ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        h = s._h if s._h is not None else C.c_void_p()
        flags = (capi.CA_SCHED_NO_TPP if no_tpp else 0) | (capi.CA_SCHED_CAUSAL if causal else 0)
        check(capi.lib().ca_build_schedule_ex(self._h, ids.__array_interface__["data"][0] if ids is not s._ids
                                              else s._ids_ptr, len(ids), int(q_len), flags, C.byref(h),
                                              None if self.host_only else _stream_ptr(stream)),
              "ca_build_schedule_ex")
        s._h = h
        s.b = len(ids)
        s.q_len = int(q_len)
        if ids is not s._ids:
            s._ids, s._ids_ptr = ids, ids.__array_interface__["data"][0]
            s._ids_list = list(seq_ids) if isinstance(seq_ids, list) else None
        s._flags = flags
        return s


class Schedule:
    """The two-phase context of one batch (owned by the library)."""

    def __init__(self, pool: Pool):
        self.pool = pool
        self._h = None
        self.b = 0
        self.q_len = 1
        self._ws = None
        self._ids, self._ids_ptr, self._ids_list, self._flags = None, None, None, 0

    def _key(self) -> tuple:
        """What the library's tables depend on: the batch, the flags, q_len and
        the pool's generation (the library rebuilds them when one changes)."""
        return (self._ids.tobytes(), self._flags, self.q_len, self.pool._generation())

    def __del__(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            capi.lib().ca_sched_destroy(self._h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def counts(self) -> dict:
        c = (C.c_int32 * 6)()
        check(capi.lib().ca_sched_counts(self._h, c), "ca_sched_counts")
        return dict(zip(["b", "cf_rows", "cf_runs", "sf_chunks", "merge_runs", "units"], list(c)))

    def tables(self) -> dict[str, np.ndarray]:
        n = self.counts()
        b, R, U, S, M = n["b"], n["cf_rows"], n["cf_runs"], n["sf_chunks"], n["merge_runs"]
        out = {"seq_perm": np.zeros(b, np.int32), "cf_rows": np.zeros((R, 4), np.int32),
               "cf_runs": np.zeros((U, 4), np.int32), "sf_offsets": np.zeros(b + 1, np.int32),
               "sf_chunks": np.zeros((S, 2), np.int32), "merge_offsets": np.zeros(b + 1, np.int32),
               "merge_runs": np.zeros(M, np.int32)}
        ptr = lambda a: a.ctypes.data_as(C.POINTER(C.c_int32))
        check(capi.lib().ca_export_tables(self._h, *[ptr(out[k]) for k in
                                                     ["seq_perm", "cf_rows", "cf_runs", "sf_offsets",
                                                      "sf_chunks", "merge_offsets", "merge_runs"]]),
              "ca_export_tables")
        return out

    def plan(self) -> dict[str, np.ndarray]:
        """The kernel work plan (units, per-CTA ranges, partial-id CSR, chunk list)."""
        cnt = (C.c_int32 * 4)()
        L = capi.lib()
        check(L.ca_export_plan(self._h, cnt, None, None, None, None), "ca_export_plan")
        n_units, grid, n_pbase, n_chunks = list(cnt)
        out = {"units": np.zeros((n_units, 12), np.int32), "cta_begin": np.zeros(grid + 1, np.int32),
               "pbase": np.zeros(n_pbase, np.int32), "chunks": np.zeros((n_chunks, 2), np.int32)}
        ptr = lambda a: a.ctypes.data_as(C.POINTER(C.c_int32))
        check(L.ca_export_plan(self._h, cnt, ptr(out["units"]), ptr(out["cta_begin"]),
                               ptr(out["pbase"]), ptr(out["chunks"])), "ca_export_plan")
        out["grid"] = grid
        return out

    def workspace_bytes(self, host_io: bool = False) -> int:
        n = C.c_size_t()
        fn = capi.lib().ca_workspace_bytes_host if host_io else capi.lib().ca_workspace_bytes
        check(fn(self._h, C.byref(n)), "ca_workspace_bytes")
        return n.value

    def workspace(self, host_io: bool = False):
        """A zero-filled device workspace large enough for this schedule
        (cached and grown on demand)."""
        import torch
        need = self.workspace_bytes(host_io)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.pool._kv.device)
        return self._ws

    def device_status(self, stream=None) -> int:
        return capi.lib().ca_sched_device_status(self._h, _stream_ptr(stream))

    def set_profile_events(self, begin=None, end=None) -> None:
        bp = begin.cuda_event if begin is not None else None
        ep = end.cuda_event if end is not None else None
        if begin is not None and not (bp and ep):
            raise ValueError("record the events once before handing them to the library")
        check(capi.lib().ca_sched_set_profile_events(self._h, bp, ep), "ca_sched_set_profile_events")


def decode_attention(pool: Pool, sched: Schedule, q, out=None, layer: int = 0, scale: float | None = None,
                     workspace=None, stream=None):
    """out[i, h] = softmax(scale q[i, h] . K^T) V over sequence seq_ids[i]'s
    context, via the two-phase kernel.  q: fp16 [b, H, D] on the GPU
    ([b, q_len, H, D] for a multi-token schedule)."""
    import torch
    if q.dtype != torch.float16 or not q.is_contiguous():
        raise ValueError("q must be a contiguous fp16 tensor")
    want = ((sched.b, pool.n_heads, pool.head_dim) if sched.q_len == 1
            else (sched.b, sched.q_len, pool.n_heads, pool.head_dim))
    if q.shape != want:
        raise ValueError(f"q has shape {tuple(q.shape)}, the schedule needs {want}")
    if out is None:
        out = torch.empty_like(q)
    if scale is None:
        scale = 1.0 / math.sqrt(pool.head_dim)
    ws = workspace if workspace is not None else sched.workspace()
    check(capi.lib().ca_decode_attention(pool._h, sched._h, layer, q.data_ptr(), out.data_ptr(),
                                         float(scale), ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
          "ca_decode_attention")
    return out


def decode_attention_host(pool: Pool, sched: Schedule, q_host, out_host, layer: int = 0,
                          scale: float | None = None, workspace=None, stream=None):
    """The same with q / out in (pinned) host memory; copies in, computes and
    copies out on ``stream``; the caller synchronises."""
    if scale is None:
        scale = 1.0 / math.sqrt(pool.head_dim)
    ws = workspace if workspace is not None else sched.workspace(host_io=True)
    check(capi.lib().ca_decode_attention_host(pool._h, sched._h, layer, q_host.data_ptr(),
                                              out_host.data_ptr(), float(scale), ws.data_ptr(),
                                              ws.numel(), _stream_ptr(stream)),
          "ca_decode_attention_host")
    return out_host


class DecodeGraph:
    """Decode-attention calls recorded once into a CUDA graph and replayed
    with one launch: the per-call host work (argument checks, two kernel
    launches each) is paid at capture only.  ``calls`` lists (layer, q, out)
    device tensors, run in that order on one schedule and workspace; the
    graph keeps those buffers, so new queries are written into the same q
    tensors before each replay.  The kernels keep their programmatic
    dependencies inside the graph.  A replay is valid while the schedule is
    the one captured: appending tokens that fit the sequences' partial last
    chunks keeps it (the kernels read each chunk's token count from the pool),
    while anything that rebuilds the schedule (a grown chunk, an insert or
    remove, another batch) makes ``replay`` raise; capture again then."""

    def __init__(self, pool: Pool, sched: Schedule, calls, workspace=None, scale: float | None = None):
        import torch
        self.pool, self.sched = pool, sched
        self.calls = [(int(layer), q, out) for layer, q, out in calls]
        self.workspace = workspace if workspace is not None else sched.workspace()
        self.scale = scale
        self._key = sched._key()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._record()                       # one uncaptured pass first
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._record()

    def _record(self):
        for layer, q, out in self.calls:
            decode_attention(self.pool, self.sched, q, out=out, layer=layer, scale=self.scale,
                             workspace=self.workspace)

    def replay(self) -> None:
        """Run every recorded call on the current stream."""
        if self.sched._key() != self._key:
            raise CAError(capi.CA_ERR_STALE, "DecodeGraph: the pool or the schedule changed after capture")
        self.graph.replay()


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    n = C.c_uint64(0)
    check(capi.lib().ca_kernel_launches(C.byref(n)), "ca_kernel_launches")
    return int(n.value)
