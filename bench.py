#!/usr/bin/env python3
"""Benchmark: prefix-shared decode attention (ChunkAttention's two-phase
kernel) on one GB300.

One step = one decode step of the whole hot path for the batch: the
per-step schedule lookup (cached while the tree is unchanged, as in the
pages' "context copies cached until the tree changes") and one layer's
two-phase attention call.  The multi-tenant workload adds its per-step churn
(8 removes, 8 inserts with KV scatter, schedule rebuild) to the step.

Prints one JSON line.  The headline workload (default) is the largest
shared-prefix configuration: 64 sequences sharing a 4096-token prefix with
512 private tokens each, 32 heads, head_dim 128, chunk 64, fp16
(ChunkAttention §4.1, Table 3's shared-prompt sweep at its largest prompt,
with twice its batch).  The same line carries a `per_config` block with
every other configuration (the tiny correctness case, the 1024-token
Llama-7B-like layer, the prompt/batch sweep, the no-sharing control, the
multi-tenant tree with churn) and the variant workloads (grouped-query
attention, an fp8 pool, 4 query tokens, head_dim 256).

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/layer call; effective HBM GB/s on unique KV vs GB300 peak"
UNIT = "us/call"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
CPU_SAMPLE_SECONDS = 12.0
HEADLINE = "sweep_s4096_b64"
# Configuration number of each workload (the five configurations: tiny
# correctness case, 1024-token prompt, shared-prompt sweep, no-sharing
# control, multi-tenant tree), then the variant workloads.
CONFIGS = {"tiny": "1", "llama7b_p1024": "2", "sweep_s2048_b32": "3a", "sweep_s2048_b64": "3b",
           "sweep_s4096_b32": "3c", "sweep_s4096_b64": "3d", "no_sharing": "4", "multi_tenant": "5"}
VARIANTS = ["gqa_p1024", "llama7b_p1024_fp8", "sweep_s4096_b64_fp8", "llama7b_p1024_q4", "d256_p1024"]
CONFIG_STEPS, CONFIG_WARMUP = 200, 20
KERNEL_LAUNCHES = 32            # isolated, event-bracketed launches for the kernel's own time
ISOLATED_CALLS, ISOLATED_WARMUP = 200, 20


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip the flat-paged / no-TPP comparisons")
    ap.add_argument("--no-per-config", action="store_true", help="headline workload only")
    ap.add_argument("--configs", default="", help="comma-separated workloads for the per_config block "
                                                  "(default: every configuration and variant)")
    ap.add_argument("--quick", action="store_true",
                    help="the workload's W warm-up + K back-to-back steps only (for profiler captures)")
    return ap.parse_args(argv)


def max_over_ranks(values, device=None):
    """Element-wise maximum of the per-rank values, on every rank (under one
    process, the values unchanged).  A job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_per_call(us_per_step: float, world: int) -> float:
    """Every rank runs one layer call per step, so the job finishes `world`
    calls per step: whole-job time per call."""
    return us_per_step / max(1, world)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_config(wl, world: int = 1) -> dict:
    """The workload as both arms report it: what defines the work, nothing
    about the machine or the launch."""
    eb = 1 if wl.kv_dtype == "fp8" else 2
    return {"workload": wl.name, "description": wl.description, "batch": len(wl.seqs), "q_len": wl.q_len,
            "n_heads": wl.n_heads, "n_kv_heads": wl.kv_heads, "head_dim": wl.head_dim, "chunk": wl.chunk,
            "kv_dtype": wl.kv_dtype, "layers_per_call": 1, "unique_kv_tokens": wl.unique_tokens(),
            "unique_kv_bytes": wl.unique_tokens() * wl.kv_heads * wl.head_dim * 2 * eb,
            "l2": "no flush between steps: steps run back to back over pool copies holding >= 4 x L2 of "
                  "unique KV in total; KV loads carry an evict-first L2 hint",
            "parallelism": "replicas" if world > 1 else "single GPU"}


# ---------------------------------------------------------------------------
# Oracle CPU baseline (bounded sample of the same workload), one thread and
# over the host cores
# ---------------------------------------------------------------------------
_cpu_trie = None
_cpu_wl = None
_cpu_q = None


def _cpu_setup(name: str):
    """Worker set-up: the workload and the oracle's trie of all its sequences."""
    global _cpu_trie, _cpu_wl, _cpu_q
    import workloads
    from oracle.pakv import OracleTrie
    wl = workloads.make(name)
    trie = OracleTrie(wl.chunk, 1 << 20)
    for sid in wl.seq_ids():
        k, v = wl.kv_rows(sid)
        if wl.kv_dtype == "fp8":             # the oracle attends over the dequantised rows
            from oracle import fp8
            k, v = fp8.dequantize(fp8.quantize(k, 1.0), 1.0), fp8.dequantize(fp8.quantize(v, 1.0), 1.0)
        trie.insert(sid, wl.tokens(sid), k, v)
    _cpu_trie, _cpu_wl, _cpu_q = trie, wl, wl.queries(0)


def _cpu_one(i: int):
    """The oracle's decode attention for batch row i (query step 0)."""
    from oracle import attention as A
    wl, trie = _cpu_wl, _cpu_trie
    sid = wl.seq_ids()[i]
    q = _cpu_q[i:i + 1]
    if wl.q_len == 1:
        return A.decode_attention(trie, [sid], 0, q, wl.scale)
    return A.decode_attention_multi(trie, [sid], 0, q, wl.scale, causal=True)


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


class OraclePool:
    """The oracle's per-sequence calls spread over the host cores: one
    spawn-started process per core, each with its own trie of the workload
    (spawn: safe after CUDA is initialised in the parent)."""

    def __init__(self, name: str, cores: int | None = None):
        import multiprocessing as mp
        self.cores = cores or host_cores()
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_cpu_setup, initargs=(name,))

    def call(self, rows, timeout: float = 600.0):
        """Wall time (s) to compute the given batch rows through the pool.
        Bounded: a worker whose set-up keeps failing would otherwise make the
        pool respawn it for ever."""
        t0 = time.perf_counter()
        self.pool.map_async(_cpu_one, rows, chunksize=1).get(timeout)
        return time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()


def cpu_baseline_single(name: str, seconds: float = CPU_SAMPLE_SECONDS) -> dict:
    """One thread: single-sequence oracle calls for a bounded time, scaled to
    one layer call over the batch."""
    _cpu_setup(name)
    b = len(_cpu_wl.seqs)
    times, done = [], 0
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < seconds or done == 0:
        t0 = time.perf_counter()
        _cpu_one(done % b)
        times.append(time.perf_counter() - t0)
        done += 1
    us = sum(times) / len(times) * b * 1e6
    return {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} single-sequence fp64 oracle decode calls on one thread (materialise K/V from "
                      f"the oracle trie + softmax attention), {sum(times):.1f} s, scaled x{b} sequences "
                      f"to one layer call"}


def cpu_baseline(name: str, seconds: float = CPU_SAMPLE_SECONDS) -> dict:
    """The oracle over every host core (the figure reported), with the
    one-thread figure beside it.  A failure here is reported in the line
    rather than stopping the GPU measurement."""
    try:
        return _cpu_baseline(name, seconds)
    except Exception as e:                       # noqa: BLE001 (reported, not raised)
        return {"value": None, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                "error": f"{type(e).__name__}: {e}"[:300]}


def _cpu_baseline(name: str, seconds: float) -> dict:
    import workloads
    b = len(workloads.make(name).seqs)
    op = OraclePool(name)
    try:
        rows = list(range(b))
        op.call(rows)                                         # warm-up: workers build their tries
        times = []
        t_start = time.perf_counter()
        while time.perf_counter() - t_start < seconds or not times:
            times.append(op.call(rows))
    finally:
        op.close()
    us = statistics.median(times) * 1e6
    single = cpu_baseline_single(name, seconds)
    return {"value": us, "unit": UNIT, "cores": op.cores, "kind": "oracle",
            "sample": f"{len(times)} full layer calls ({b} sequences each) of the fp64 oracle decode "
                      f"(materialise K/V from the oracle trie + softmax attention), sequences spread over "
                      f"{op.cores} worker processes (one per host core), {sum(times):.1f} s; median",
            "single_thread": single}


# ---------------------------------------------------------------------------
# Clock sampling during the timed regions
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 10 ms, each
    with its timestamp, so that the samples inside the timed windows (wall
    clock, added with window()) can be told from the rest."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NEAR_S = 0.1                # a window with no sample inside takes those within 100 ms of it

    def __init__(self, device_index: int):
        import tempfile
        self.idx = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"ca_bench_clocks_{os.getpid()}.csv")
        self.windows: dict[str, list] = {}
        self.rows = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def window(self, label: str, t0: float, t1: float):
        self.windows.setdefault(label, []).append((t0, t1))

    def stop(self):
        import datetime
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]),
                             {n for n, v in zip(names, parts[6:10]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        try:
            os.remove(self.path)
        except OSError:
            pass
        self.rows = rows

    def summary(self, labels=None) -> dict:
        if self.rows is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        wins = [w for k, ws in self.windows.items() if labels is None or k in labels for w in ws]
        inside = [r for r in self.rows if any(a <= r[0] <= z for a, z in wins)]
        near = [r for r in self.rows if any(a - self.NEAR_S <= r[0] <= z + self.NEAR_S for a, z in wins)]
        use = inside or near or self.rows
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(set().union(*(r[3] for r in use))) if use else [],
                "samples": len(self.rows), "samples_in_timed_region": len(inside),
                "samples_used": len(use),
                "basis": ("samples inside the timed region" if inside else
                          f"samples within {int(self.NEAR_S * 1e3)} ms of the timed region (it is shorter "
                          f"than the 10 ms sampling period)" if near else "all samples of the run")}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def source_fingerprint(path: str) -> str:
    """sha256[:16] of a C++/CUDA source with comments and whitespace removed,
    so that only code changes (not comment edits) change it."""
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = re.sub(r"\s+", " ", text)
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def profile_record(key: str):
    """The committed ncu record for a kernel on a workload, if it was taken on
    the current kernel code (None otherwise)."""
    h = source_fingerprint(os.path.join(ROOT, "prefix_shared_decode_gb300", "csrc", "kernels.cu"))
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except ValueError:
        return None
    e = d.get(key)
    if not e or e.get("kernels_cu_code_sha256_16") != h:
        return None
    return e


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class WorkloadRun:
    """One workload loaded on the GPU: its pool copies, schedules,
    workspaces and query buffers, and the timing methods."""

    def __init__(self, name: str, dev, stream, max_steps: int):
        import numpy as np
        import torch
        import workloads
        from prefix_shared_decode_gb300 import Pool
        from workloads.device import capacity_for, insert_sequence
        t0 = time.perf_counter()
        self.torch, self.dev, self.stream = torch, dev, stream
        self.wl = wl = workloads.make(name)
        self.L, self.H, self.D, self.c, self.HK = wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk, wl.kv_heads
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.churn = wl.churn > 0
        self.batch = wl.seq_ids()
        self.b = len(self.batch)
        self.eb = 1 if wl.kv_dtype == "fp8" else 2              # bytes per stored K/V element
        self.kv_bytes = wl.unique_tokens() * self.HK * self.D * 2 * self.eb   # one layer's K and V
        self.io_bytes = 2 * self.b * wl.q_len * self.H * self.D * 2          # q in, out
        self.alg_bytes = self.kv_bytes + self.io_bytes
        self._staging = {}
        self._Pool, self._insert, self._capacity = Pool, insert_sequence, capacity_for
        self.n_copies = 1 if self.churn else self.copies_for(self.kv_bytes)
        self.pools = self.make_pools(self.n_copies)
        torch.cuda.synchronize()
        self.skw = {"q_len": wl.q_len, "causal": wl.q_len > 1}  # several query tokens: causal
        self.scheds = [p.schedule(self.batch, **self.skw) for p in self.pools]
        # Workspace with headroom so a schedule rebuilt after churn fits without
        # allocating inside the timed steps (grown, zero-filled, only if needed).
        self.wss = [torch.zeros(2 * s.workspace_bytes() + (1 << 20), dtype=torch.uint8, device=dev)
                    for s in self.scheds]
        self.qs = [torch.from_numpy(wl.queries(i)).to(dev) for i in range(4)]
        self.out = torch.empty_like(self.qs[0])
        self.host_split = {"remove": [], "insert": [], "schedule": []}
        self.step_no = 0
        if self.churn:
            # Draw every step's churn (ids, tokens) before timing.  Inserted
            # rows come from device-resident N(0,1) fp16 blocks (one packed
            # buffer per step, as a batched prefill would leave them), so the
            # timed step does only what a serving step does: remove, insert
            # (trie + KV scatter), reschedule, attend.  (Churn parity with the
            # real generator is a GPU test.)
            self.plan_churn = []
            for _ in range(max_steps):
                removed, inserted = wl.churn_step()
                toks = [wl.tokens(sid) for sid in inserted]
                self.plan_churn.append((np.array(removed, dtype=np.int64), np.array(inserted, dtype=np.int64),
                                        np.concatenate(toks), np.array([len(t) for t in toks], dtype=np.int32),
                                        wl.seq_ids()))
            nmax = max(int(p[3].sum()) for p in self.plan_churn)
            g = torch.Generator(device=dev).manual_seed(wl.seed)
            kblk = torch.randn((self.L, nmax, self.HK, self.D), generator=g, device=dev).half()
            vblk = torch.randn((self.L, nmax, self.HK, self.D), generator=g, device=dev).half()
            self.kv_views = [(kblk[:, :int(p[3].sum())], vblk[:, :int(p[3].sum())]) for p in self.plan_churn]
        torch.cuda.synchronize()
        self.setup_s = time.perf_counter() - t0

    def copies_for(self, nbytes: int) -> int:
        """Independent pool copies to rotate through so that the steps touch
        at least 4 x L2 of KV in total (1 when one copy already does; at
        most 8, so the 64 KiB tiny case stays L2-resident)."""
        return 1 if nbytes >= 4 * self.l2 else min(8, -(-4 * self.l2 // nbytes))

    def make_pools(self, n, no_sharing=False, headroom=1.5):
        ps = []
        for _ in range(n):
            pc = self._Pool(self.L, self.H, self.D, self.c, self._capacity(self.wl, headroom=headroom),
                            no_sharing=no_sharing, n_kv_heads=self.HK, kv_dtype=self.wl.kv_dtype)
            for sid in self.batch:
                self._insert(pc, self.wl, sid, staging=self._staging)
            ps.append(pc)
        return ps

    @property
    def kernel_name(self) -> str:
        """The main kernel variant the library launches: the few-row one when
        positions bring 2..8 query rows per key/value head (head_dim <= 128)."""
        rows_per_kv = self.wl.q_len * (self.H // self.HK)
        few_rows = 2 <= rows_per_kv <= 8 and self.D <= 128
        return f"two_phase_attention_kernel<{self.c},{self.D},{self.eb},{'true' if few_rows else 'false'}>"

    def step(self):
        """One decode step (with the churn of the multi-tenant workload)."""
        from prefix_shared_decode_gb300 import decode_attention
        i = self.step_no
        self.step_no += 1
        r = i % self.n_copies
        pool, sched, ws = self.pools[r], self.scheds[r], self.wss[r]
        if self.churn:
            th = time.perf_counter()
            removed, inserted, toks, lens, live = self.plan_churn[i]
            pool.remove_batch(removed)
            t1 = time.perf_counter()
            pool.insert_batch(inserted, toks, *self.kv_views[i], lengths=lens, stream=self.stream)
            t2 = time.perf_counter()
            self.batch = live
        sched = self.scheds[r] = pool.schedule(self.batch, reuse=sched, stream=self.stream, **self.skw)
        if self.churn:
            t3 = time.perf_counter()
            self.host_split["remove"].append((t1 - th) * 1e6)
            self.host_split["insert"].append((t2 - t1) * 1e6)
            self.host_split["schedule"].append((t3 - t2) * 1e6)
        if sched.workspace_bytes() > ws.numel():
            ws = self.wss[r] = self.torch.zeros(2 * sched.workspace_bytes(), dtype=self.torch.uint8,
                                                device=self.dev)
        decode_attention(pool, sched, self.qs[i % 4], out=self.out, scale=self.wl.scale, workspace=ws,
                         stream=self.stream)

    def check_status(self, what: str):
        if any(s.device_status() != 0 for s in self.scheds):
            raise RuntimeError(f"device status after {what}")

    def back_to_back(self, steps: int, warmup: int, clocks=None, label="", world=1):
        """Steps run back to back, as in a decode loop: one event pair around
        exactly `steps` steps after `warmup` untimed ones.  Consecutive steps
        touch more than twice the L2 (the pool copies hold >= 4 x L2 of KV)
        and every KV load carries an evict-first L2 hint, so no flush is
        needed between steps; nothing else is recorded inside the loop."""
        from prefix_shared_decode_gb300 import kernel_launches
        torch = self.torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        self.check_status("warm-up")
        ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        win0 = time.time()
        n0 = kernel_launches()
        ev_a.record(self.stream)
        for _ in range(steps):
            self.step()
        enqueue = time.perf_counter() - wall0
        ev_b.record(self.stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if clocks is not None:
            clocks.window(label, win0, time.time())
        launches = kernel_launches() - n0
        if world > 1:
            torch.distributed.barrier()
        self.check_status("timed steps")
        return {"us": ev_a.elapsed_time(ev_b) * 1e3 / steps, "enqueue_us": enqueue * 1e6 / steps,
                "wall_s": wall, "launches": launches}

    def kernel_isolated(self, n: int = KERNEL_LAUNCHES, clocks=None, label=""):
        """The main kernel's own duration: CUDA events recorded by the library
        just before and after its launch (the event hook), one launch at a
        time (the events break the programmatic overlap with the neighbours),
        consecutive launches rotating over the pool copies so that L2 holds
        none of a launch's KV.  Median over n launches after 4 warm-up ones."""
        from prefix_shared_decode_gb300 import decode_attention
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n + 4)]
        for a, z in evs:        # torch creates the CUDA event on first record; the library re-records it
            a.record(self.stream)
            z.record(self.stream)
        torch.cuda.synchronize()
        win0 = time.time()
        for i, (a, z) in enumerate(evs):
            r = i % self.n_copies
            self.scheds[r].set_profile_events(a, z)
            decode_attention(self.pools[r], self.scheds[r], self.qs[i % 4], out=self.out, scale=self.wl.scale,
                             workspace=self.wss[r], stream=self.stream)
            self.scheds[r].set_profile_events(None, None)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.window(label, win0, time.time())
        self.check_status("isolated kernel launches")
        us = [a.elapsed_time(z) * 1e3 for a, z in evs[4:]]
        return {"median_us": statistics.median(us), "min_us": min(us), "max_us": max(us), "launches": len(us)}

    def isolated_call(self, n: int = ISOLATED_CALLS, warmup: int = ISOLATED_WARMUP, clocks=None, label=""):
        """One call at a time: CUDA events around the call only, the median of
        n after `warmup` calls, L2 flushed before each call (a 2 x L2 buffer
        written, outside the event pair).  Also the same with the flush
        followed by a read of another 2 x L2 buffer, which leaves L2 holding
        clean lines, so the call does not pay for writing the flush's dirty
        lines back."""
        from prefix_shared_decode_gb300 import decode_attention
        torch = self.torch
        flush = torch.empty(2 * self.l2, dtype=torch.uint8, device=self.dev)
        clean = torch.ones(2 * self.l2 // 4, dtype=torch.float32, device=self.dev)
        sink = torch.empty((), dtype=torch.float32, device=self.dev)
        res = {}
        win0 = time.time()
        for mode in ("write", "write_then_read"):
            evs = []
            for i in range(n + warmup):
                r = i % self.n_copies
                flush.zero_()
                if mode == "write_then_read":
                    torch.sum(clean, dim=0, out=sink)
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
                decode_attention(self.pools[r], self.scheds[r], self.qs[i % 4], out=self.out,
                                 scale=self.wl.scale, workspace=self.wss[r], stream=self.stream)
                z.record(self.stream)
                if i >= warmup:
                    evs.append((a, z))
            torch.cuda.synchronize()
            res[mode] = statistics.median(a.elapsed_time(z) * 1e3 for a, z in evs)
        if clocks is not None:
            clocks.window(label, win0, time.time())
        self.check_status("isolated calls")
        del flush, clean
        return res

    def e2e(self, steps: int):
        """End to end through the host-buffer entry point: q read from and out
        written to pinned host memory inside each step's event pair."""
        from prefix_shared_decode_gb300 import decode_attention_host
        torch = self.torch
        qh = [q.cpu().pin_memory() for q in self.qs]
        oh = torch.empty_like(qh[0]).pin_memory()
        wshs = [s.workspace(host_io=True) for s in self.scheds]
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            r = i % self.n_copies
            eev[i][0].record(self.stream)
            self.scheds[r] = self.pools[r].schedule(self.batch, reuse=self.scheds[r], stream=self.stream,
                                                    **self.skw)
            decode_attention_host(self.pools[r], self.scheds[r], qh[i % 4], oh, scale=self.wl.scale,
                                  workspace=wshs[r], stream=self.stream)
            eev[i][1].record(self.stream)
        torch.cuda.synchronize()
        self.check_status("host-buffer calls")
        return sum(a.elapsed_time(z) for a, z in eev) / steps * 1e3

    def graph_replay(self, ng: int = 32, rg: int = 16):
        """The same calls recorded into one CUDA graph (ng calls rotating over
        the pool copies as the timed loop does) and replayed back to back."""
        from prefix_shared_decode_gb300 import decode_attention
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(self.stream)
        with torch.cuda.graph(g, stream=side):
            for i in range(ng):
                r = i % self.n_copies
                decode_attention(self.pools[r], self.scheds[r], self.qs[i % 4], out=self.out, scale=self.wl.scale,
                                 workspace=self.wss[r])
        self.stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ga, gz = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        ga.record(self.stream)
        for _ in range(rg):
            g.replay()
        gz.record(self.stream)
        host_us = (time.perf_counter() - h0) * 1e6 / (rg * ng)
        torch.cuda.synchronize()
        self.check_status("graph replays")
        del g
        return {"us_per_call": round(ga.elapsed_time(gz) * 1e3 / (rg * ng), 3), "calls_per_graph": ng,
                "replays": rg, "host_us_per_call": round(host_us, 2),
                "method": "decode_attention calls recorded into one CUDA graph (torch.cuda.graph), "
                          "replayed back to back; one event pair around all replays"}

    def context(self, n: int = 100):
        """The same batch through the flat paged layout (no sharing) and
        through physically shared KV without the two-phase partition."""
        from prefix_shared_decode_gb300 import decode_attention
        torch = self.torch

        def time_calls(ps, ss):
            ws_ = [s.workspace() for s in ss]
            m = len(ps)
            for i in range(10):
                decode_attention(ps[i % m], ss[i % m], self.qs[i % 4], out=self.out, scale=self.wl.scale,
                                 workspace=ws_[i % m], stream=self.stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for i in range(n):
                decode_attention(ps[i % m], ss[i % m], self.qs[i % 4], out=self.out, scale=self.wl.scale,
                                 workspace=ws_[i % m], stream=self.stream)
            e1.record(self.stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n * 1e3

        no_tpp = [p.schedule(self.batch, no_tpp=True, **self.skw) for p in self.pools]
        us_no_tpp = time_calls(self.pools, no_tpp)
        del no_tpp
        flat_bytes = sum(self.wl.seq_len(sid) for sid in self.batch) * self.HK * self.D * 2 * self.eb
        flats = self.make_pools(self.copies_for(flat_bytes), no_sharing=True, headroom=1.05)
        us_flat = time_calls(flats, [f.schedule(self.batch, **self.skw) for f in flats])
        del flats
        torch.cuda.empty_cache()
        return {"paged_flat_us": round(us_flat, 2), "paged_shared_no_tpp_us": round(us_no_tpp, 2)}

    def close(self):
        for name in ("pools", "scheds", "wss", "qs", "out", "kv_views", "_staging"):
            if hasattr(self, name):
                delattr(self, name)
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def config_entry(run: WorkloadRun, b2b: dict, kern: dict, iso: dict, ctx: dict | None, peak: float) -> dict:
    """One workload's figures for the per_config block."""
    us = b2b["us"]
    e = {"config": CONFIGS.get(run.wl.name, "variant"), "description": run.wl.description,
         "us_per_call": round(us, 2),
         "unique_kv_bytes": run.kv_bytes, "algorithmic_bytes": run.alg_bytes,
         "unique_kv_gbs": round(run.kv_bytes / (us * 1e-6) / 1e9, 1),
         "frac_of_measured_peak": round(run.alg_bytes / (us * 1e-6) / 1e9 / peak, 4),
         "frac_of_8tbs": round(run.alg_bytes / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
         "isolated_call_us": round(iso["write"], 2),
         "isolated_call_clean_l2_us": round(iso["write_then_read"], 2),
         "isolated_call_frac_of_8tbs": round(run.alg_bytes / (iso["write"] * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
         "kernel": run.kernel_name, "kernel_us": round(kern["median_us"], 2),
         "kernel_frac_of_measured_peak": round(run.alg_bytes / (kern["median_us"] * 1e-6) / 1e9 / peak, 4),
         "pool_copies": run.n_copies, "partial_scratch_bytes": run.scheds[0].workspace_bytes(),
         "steps": b2b.get("steps"), "warmup": b2b.get("warmup")}
    if run.churn:
        e["us_per_call"] = None
        e["us_per_step_incl_churn"] = round(us, 2)
        e["churn_per_step"] = run.wl.churn
        e["churn_host_split_us"] = {k: round(statistics.median(v), 1) for k, v in run.host_split.items() if v}
        e["attention_note"] = ("kernel_us and isolated_call_us time the attention call alone on the final "
                               "schedule; the step also runs 8 removes, 8 inserts (KV scatter) and a rebuild")
        for k in ("unique_kv_gbs", "frac_of_measured_peak", "frac_of_8tbs"):
            e[k] = None
        e["attention_frac_of_8tbs_isolated"] = e.pop("isolated_call_frac_of_8tbs")
    if ctx:
        e["context"] = ctx
        if not run.churn:
            e["context"]["speedup_vs_paged_flat"] = round(ctx["paged_flat_us"] / us, 2)
            e["context"]["speedup_vs_paged_shared_no_tpp"] = round(ctx["paged_shared_no_tpp_us"] / us, 2)
    if run.wl.name == "tiny":
        e["note"] = "64 KiB of KV: latency-bound and L2-resident (parity case; µs reported only)"
        for k in ("unique_kv_gbs", "frac_of_measured_peak", "frac_of_8tbs", "isolated_call_frac_of_8tbs",
                  "kernel_frac_of_measured_peak"):
            e[k] = None
    return e


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    from prefix_shared_decode_gb300 import build
    build.build()
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peak()
    K, W = args.steps, args.warmup
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)

    # -- headline: exactly K steps back to back after W warm-up steps --------
    run = WorkloadRun(args.workload, dev, stream, max_steps=W + K + 64)
    b2b = run.back_to_back(K, W, clocks=clocks, label="headline", world=world)
    ms_per_step = b2b["us"] / 1e3
    if args.quick:
        clocks.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(whole_job_per_call(b2b["us"], world), 3),
                              "unit": UNIT, "steps": K, "warmup": W, "quick": True,
                              "config": workload_config(run.wl, world), "gpu_launches": b2b["launches"]}),
                  flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    kern = run.kernel_isolated(clocks=clocks, label="kernel")
    iso = run.isolated_call(clocks=clocks, label="isolated")
    e2e_us = run.e2e(min(K, 200))
    graph = None if run.churn else run.graph_replay()
    graph_us = graph["us_per_call"] if graph else 0.0
    ms_per_step, kern_us, e2e_us, iso_w, iso_c, graph_us = max_over_ranks(
        [ms_per_step, kern["median_us"], e2e_us, iso["write"], iso["write_then_read"], graph_us], device=dev)
    kern["median_us"] = kern_us
    iso = {"write": iso_w, "write_then_read": iso_c}
    if graph:
        graph["us_per_call"] = round(graph_us, 3)
    ctx = None if (args.no_context or run.churn) else run.context()
    headline_entry = config_entry(run, dict(b2b, steps=K, warmup=W), kern, iso, ctx, peak)
    head = run
    run_setup = run.setup_s
    cfg = workload_config(run.wl, world)
    launch = {"grid_ctas": run.scheds[0].plan()["grid"],
              "partial_scratch_bytes": run.scheds[0].workspace_bytes(),
              "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
              "pool_copies": run.n_copies, "l2_bytes": run.l2,
              "l2_note": ("no flush: steps run back to back over %d pool cop%s (%d MB of unique KV each, "
                          "%d MB L2), so consecutive steps touch more than twice the L2; KV loads carry an "
                          "evict-first L2 hint" % (run.n_copies, "y" if run.n_copies == 1 else "ies",
                                                   run.kv_bytes >> 20, run.l2 >> 20))}
    host_split = ({k: round(statistics.median(v), 1) for k, v in run.host_split.items() if v}
                  if run.churn else None)
    kname, alg_bytes, kv_bytes, b, wl = run.kernel_name, run.alg_bytes, run.kv_bytes, run.b, run.wl
    run.close()
    del run

    # -- every other configuration and variant -----------------------------
    per_config = {wl.name: headline_entry}
    if not args.no_per_config:
        names = ([n for n in args.configs.split(",") if n] if args.configs
                 else list(CONFIGS) + VARIANTS)
        for name in names:
            if name == wl.name:
                continue
            r = WorkloadRun(name, dev, stream, max_steps=CONFIG_WARMUP + CONFIG_STEPS + 64)
            bb = r.back_to_back(CONFIG_STEPS, CONFIG_WARMUP, clocks=clocks, label="per_config", world=world)
            kk = r.kernel_isolated(clocks=clocks, label="per_config")
            ii = r.isolated_call(clocks=clocks, label="per_config")
            cc = None if (args.no_context or r.churn or name == "tiny") else r.context()
            bb_us, kk_us, ii_w, ii_c = max_over_ranks([bb["us"], kk["median_us"], ii["write"],
                                                       ii["write_then_read"]], device=dev)
            bb["us"], kk["median_us"] = bb_us, kk_us
            ii = {"write": ii_w, "write_then_read": ii_c}
            per_config[name] = config_entry(r, dict(bb, steps=CONFIG_STEPS, warmup=CONFIG_WARMUP), kk, ii, cc, peak)
            per_config[name]["setup_s"] = round(r.setup_s, 2)
            r.close()
            del r
    clocks.stop()

    if world > 1 and rank != 0:
        torch.distributed.destroy_process_group()
        return

    us = ms_per_step * 1e3
    rec = profile_record(f"{kname}:{wl.name}")
    achieved = alg_bytes / (kern["median_us"] * 1e-6) / 1e9
    res = {
        "metric": METRIC,
        "value": round(whole_job_per_call(us, world), 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f16 q/out, fp8 e4m3 K/V storage (fp32 accumulate)" if wl.kv_dtype == "fp8"
                  else "f16 (fp32 accumulate)"),
        "data": "synthetic (seeded N(0,1) fp16 Q/K/V; token segments shaped like ChunkAttention's shared "
                "system prompts)",
        "config": cfg,
        "launch": launch,
        "effective_hbm_gbs": round(alg_bytes / (us * 1e-6) / 1e9, 1),
        "unique_kv_gbs": round(kv_bytes / (us * 1e-6) / 1e9, 1),
        "frac_of_8tbs": round(alg_bytes / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs (of {peak_kind})",
                     "traffic": rec.get("dram_bytes_per_launch") if rec else None,
                     "traffic_source": rec.get("source") if rec else None,
                     "kernel": kname,
                     "kernel_us": round(kern["median_us"], 3),
                     "kernel_timing": f"isolated launches: median of {kern['launches']} launches of the main "
                                      "kernel, each bracketed by CUDA events the library records just before "
                                      "and after it, one launch at a time, rotating over the pool copies "
                                      "(L2 holds none of a launch's KV); outside the headline loop",
                     "algorithmic_bytes": alg_bytes,
                     "per_call": {"us": round(us, 3), "achieved": round(alg_bytes / (us * 1e-6) / 1e9, 1),
                                  "frac": round(alg_bytes / (us * 1e-6) / 1e9 / peak, 4),
                                  "basis": "algorithmic bytes / ms_per_step (back-to-back calls, main kernel "
                                           "+ merge + the overlap between calls)"}},
        "e2e": {"value": round(whole_job_per_call(e2e_us, world), 3), "unit": UNIT,
                "h2d_bytes_per_step": b * wl.q_len * wl.n_heads * wl.head_dim * 2,
                "d2h_bytes_per_step": b * wl.q_len * wl.n_heads * wl.head_dim * 2,
                "path": "ca_decode_attention_host: q read from and out written to pinned host memory by the "
                        "kernels through its device mapping (NVLink-C2C), inside each step's event pair"},
        "isolated_call": {"median_us": round(iso["write"], 2), "reps": ISOLATED_CALLS,
                          "clean_l2_median_us": round(iso["write_then_read"], 2),
                          "method": "one call at a time: CUDA events around the call only, median of 200 "
                                    "after 20 warm-up calls, L2 flushed (2 x L2 written) before each call; "
                                    "clean_l2: the flush followed by a read of another 2 x L2 buffer"},
        "graph_replay": graph,
        "gpu_launches": b2b["launches"],
        "gpu_launches_source": "library launch counter (ca_kernel_launches) read around the timed loop",
        "clocks": clocks.summary(["headline"]),
        "clocks_all_timed_regions": clocks.summary(),
        "wall_s_timed_loop": round(b2b["wall_s"], 4),
        "host_enqueue_us_per_step": round(b2b["enqueue_us"], 1),
        "setup_s": round(run_setup, 2),
    }
    if host_split:
        res["config"]["churn_per_step"] = wl.churn
        res["churn_host_split_us"] = host_split
    if ctx:
        res["context"] = dict(ctx)
        res["context"]["note"] = ("same kernel with every chunk sequence-first: flat = private copy of the "
                                  "prefix per sequence (PagedAttention layout), shared_no_tpp = one copy read "
                                  "once per sharer (ChunkAttention's PagedAttn* comparator)")
        res["context"]["speedup_vs_paged_flat"] = round(ctx["paged_flat_us"] / us, 2)
        res["context"]["speedup_vs_paged_shared_no_tpp"] = round(ctx["paged_shared_no_tpp_us"] / us, 2)
    res["per_config"] = per_config
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl.name)
    print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The reference arm: the fp64 CPU oracle over the host cores (one
    process per core), on the same workload, metric and step count.  A step
    is one layer call over a bounded sample of the batch's sequences,
    scaled to the whole batch."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import workloads
    wl = workloads.make(args.workload)
    b = len(wl.seqs)
    try:
        per_step, n, t_warm, cores = _reference_steps(wl, args)
    except Exception as e:                       # noqa: BLE001
        print(json.dumps({"impl": "reference", "unavailable": f"the CPU oracle failed: {type(e).__name__}: {e}"[:300]}),
              flush=True)
        return
    v = statistics.median(per_step)
    cb = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
          "sample": f"each step: the fp64 oracle decode (materialise K/V from the oracle trie + softmax "
                    f"attention) of {n} of the {b} sequences, spread over {cores} worker processes (one per "
                    f"host core), scaled x{b}/{n} to one layer call; median of {args.steps} steps after "
                    f"{args.warmup} warm-up (set-up {t_warm:.1f} s untimed)"}
    res = {"metric": METRIC, "value": round(v, 1), "unit": UNIT, "impl": "reference",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) fp16 Q/K/V; token segments shaped like ChunkAttention's shared "
                   "system prompts)",
           "config": workload_config(wl, world),
           "cpu_baseline": cb,
           "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "note": "ChunkAttention's pages publish no code: the reference arm is the fp64 CPU oracle on the host "
                   "cores, timed on a bounded sample and scaled to one layer call"}
    print(json.dumps(res), flush=True)


def _reference_steps(wl, args):
    """Per-step µs of the reference arm (one layer call over a bounded
    sample of the batch, scaled to the whole batch)."""
    b = len(wl.seqs)
    op = OraclePool(wl.name)
    try:
        t_warm = op.call(list(range(b)))                         # workers build their tries
        # sample size: whole rounds of one sequence per core, so that the
        # K + W steps take about two minutes at most
        per_round = op.call(list(range(min(b, op.cores))))
        rounds = max(1, min(-(-b // op.cores), int(120.0 / max(1e-3, per_round) / max(1, args.steps + args.warmup))))
        n = min(b, rounds * op.cores)
        rows = list(range(n))
        for _ in range(args.warmup):
            op.call(rows)
        per_step = [op.call(rows) * 1e6 * b / n for _ in range(args.steps)]
    finally:
        op.close()
    return per_step, n, t_warm, op.cores


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
