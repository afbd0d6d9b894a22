#!/usr/bin/env python3
"""Benchmark: prefix-shared decode attention (ChunkAttention's two-phase
kernel) on one GB300.

One step = one decode step of the whole hot path for the batch: the
per-step schedule lookup (cached while the tree is unchanged, as in the
pages' "context copies cached until the tree changes") and one layer's
two-phase attention call.  The multi-tenant workload adds its per-step churn
(8 removes, 8 inserts with KV scatter, schedule rebuild) to the step.

Prints one JSON line.  Default workload: 32 sequences sharing a 1024-token
prefix with 512 private tokens each, 32 heads, head_dim 128, chunk 64, fp16.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
CPU_SAMPLE_SECONDS = 12.0


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama7b_p1024")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip the flat-paged / no-TPP comparisons")
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


# ---------------------------------------------------------------------------
# Oracle CPU baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------
def cpu_baseline(wl, seconds: float = CPU_SAMPLE_SECONDS) -> dict:
    import numpy as np
    from oracle import attention as A
    from oracle.pakv import OracleTrie

    trie = OracleTrie(wl.chunk, 1 << 20)
    for sid in wl.seq_ids():
        k, v = wl.kv_rows(sid)
        if wl.kv_dtype == "fp8":             # the oracle attends over the dequantised rows
            from oracle import fp8
            k, v = fp8.dequantize(fp8.quantize(k, 1.0), 1.0), fp8.dequantize(fp8.quantize(v, 1.0), 1.0)
        trie.insert(sid, wl.tokens(sid), k, v)
    batch = wl.seq_ids()
    q = wl.queries(0)
    times, done = [], 0
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < seconds or done == 0:
        i = done % len(batch)
        t0 = time.perf_counter()
        if wl.q_len == 1:
            A.decode_attention(trie, [batch[i]], 0, q[i:i + 1], wl.scale)
        else:
            A.decode_attention_multi(trie, [batch[i]], 0, q[i:i + 1], wl.scale, causal=True)
        times.append(time.perf_counter() - t0)
        done += 1
    per_seq = sum(times) / len(times)
    us_per_call = per_seq * len(batch) * 1e6
    return {"value": us_per_call, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} single-sequence fp64 oracle decode calls (materialise K/V from the "
                      f"oracle trie + softmax attention, one numpy thread), "
                      f"{sum(times):.1f} s, scaled x{len(batch)} sequences to one layer call"}


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 10 ms, each
    with its timestamp, so that the samples inside the timed window (wall
    clock, set with window()) can be told from the rest."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        import tempfile
        self.idx = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"ca_bench_clocks_{os.getpid()}.csv")
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def stop(self) -> dict:
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(set().union(*(r[3] for r in use))) if use else [],
                "samples": len(rows), "samples_in_timed_region": len(inside)}


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


def kernel_traffic(kernel_name: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel code (null otherwise)."""
    h = source_fingerprint(os.path.join(ROOT, "prefix_shared_decode_gb300", "csrc", "kernels.cu"))
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except ValueError:
        return None
    e = d.get(kernel_name)
    if not e or e.get("kernels_cu_code_sha256_16") != h:
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    import workloads
    from prefix_shared_decode_gb300 import Pool, build, decode_attention, decode_attention_host, kernel_launches
    from workloads.device import capacity_for, insert_sequence
    build.build()

    wl = workloads.make(args.workload)
    L, H, D, c = wl.n_layers, wl.n_heads, wl.head_dim, wl.chunk
    t0 = time.perf_counter()
    HK = wl.kv_heads
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    churn = wl.churn > 0
    batch = wl.seq_ids()
    b = len(batch)
    staging = {}

    def copies_for(nbytes):
        """Independent copies to rotate through so that consecutive steps
        touch more than twice the L2 (1 when one copy already does)."""
        return 1 if nbytes >= 2 * l2 else -(-2 * l2 // nbytes)

    def make_pools(n, no_sharing=False, headroom=1.5):
        ps = []
        for _ in range(n):
            pc = Pool(L, H, D, c, capacity_for(wl, headroom=headroom), no_sharing=no_sharing, n_kv_heads=HK,
                      kv_dtype=wl.kv_dtype)
            for sid in batch:
                insert_sequence(pc, wl, sid, staging=staging)
            ps.append(pc)
        return ps

    eb = 1 if wl.kv_dtype == "fp8" else 2                       # bytes per stored K/V element
    kv_bytes = wl.unique_tokens() * HK * D * 2 * eb             # one layer's K and V
    n_copies = 1 if churn else copies_for(kv_bytes)
    pools = make_pools(n_copies)
    pool = pools[0]
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t0

    skw = {"q_len": wl.q_len, "causal": wl.q_len > 1}        # several query tokens: causal
    scheds = [p.schedule(batch, **skw) for p in pools]
    sched = scheds[0]
    # Workspace with headroom so a schedule rebuilt after churn fits without
    # allocating inside the timed steps (grown, zero-filled, only if needed).
    wss = [torch.zeros(2 * s_.workspace_bytes() + (1 << 20), dtype=torch.uint8, device=dev) for s_ in scheds]
    stream = torch.cuda.current_stream()
    qs = [torch.from_numpy(wl.queries(i)).to(dev) for i in range(4)]
    out = torch.empty_like(qs[0])
    churn_host_us = []
    host_split = {"remove": [], "insert": [], "schedule": []}
    if churn:
        # Draw every step's churn (ids, tokens) before timing.  Inserted rows
        # come from device-resident N(0,1) fp16 blocks (one packed buffer per
        # step, as a batched prefill would leave them), so the timed step does
        # only what a serving step does: remove, insert (trie + KV scatter),
        # reschedule, attend.  (Churn parity with the real generator is a GPU
        # test.)
        plan_churn = []
        for i in range(args.warmup + args.steps):
            removed, inserted = wl.churn_step()
            toks = [wl.tokens(sid) for sid in inserted]
            plan_churn.append((np.array(removed, dtype=np.int64), np.array(inserted, dtype=np.int64),
                               np.concatenate(toks), np.array([len(t) for t in toks], dtype=np.int32),
                               wl.seq_ids()))
        nmax = max(int(p[3].sum()) for p in plan_churn)
        g = torch.Generator(device=dev).manual_seed(wl.seed)
        kblk = torch.randn((L, nmax, HK, D), generator=g, device=dev).half()
        vblk = torch.randn((L, nmax, HK, D), generator=g, device=dev).half()
        kv_views = [(kblk[:, :int(p[3].sum())], vblk[:, :int(p[3].sum())]) for p in plan_churn]

    def step(i):
        nonlocal batch
        r = i % n_copies
        pool, sched, ws = pools[r], scheds[r], wss[r]
        if churn:
            th = time.perf_counter()
            removed, inserted, toks, lens, live = plan_churn[i]
            pool.remove_batch(removed)
            t1 = time.perf_counter()
            pool.insert_batch(inserted, toks, *kv_views[i], lengths=lens, stream=stream)
            t2 = time.perf_counter()
            batch = live
        sched = scheds[r] = pool.schedule(batch, reuse=sched, stream=stream, **skw)
        if churn:
            t3 = time.perf_counter()
            host_split["remove"].append((t1 - th) * 1e6)
            host_split["insert"].append((t2 - t1) * 1e6)
            host_split["schedule"].append((t3 - t2) * 1e6)
            churn_host_us.append((t3 - th) * 1e6)
        if sched.workspace_bytes() > ws.numel():
            ws = wss[r] = torch.zeros(2 * sched.workspace_bytes(), dtype=torch.uint8, device=dev)
        decode_attention(pool, sched, qs[i % 4], out=out, scale=wl.scale, workspace=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if any(s_.device_status() != 0 for s_ in scheds):
        raise RuntimeError("device status after warm-up")

    K = args.steps
    # Steps run back to back, as in a decode loop.  Consecutive steps touch
    # more than twice the L2 (the unique KV of one pool, or of the pool copies
    # the steps rotate through) and every KV load carries an evict-first L2
    # hint, so no flush is needed between steps.  One event pair brackets all K steps; the main
    # kernel is additionally timed on every 32nd step through the library's
    # event hook.  Event records between kernels break the programmatic
    # launch overlap (the next kernel's early start and its pool prefetch), so
    # a timed step runs the kernel in isolation and costs a few µs; they are
    # kept sparse to leave the back-to-back steps undisturbed.
    KEV = 32
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range((K + KEV - 1) // KEV)]
    for a, z in kev:        # torch creates the CUDA event on first record; the library re-records it
        a.record(stream)
        z.record(stream)
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    win0 = time.time()
    ev_a.record(stream)
    launches0 = kernel_launches()
    for i in range(K):
        r = (args.warmup + i) % n_copies
        if i % KEV == 0:
            scheds[r].set_profile_events(*kev[i // KEV])
        step(args.warmup + i)
        if i % KEV == 0:
            scheds[r].set_profile_events(None, None)
    enqueue = time.perf_counter() - wall0         # host time to issue the K steps
    ev_b.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks.window(win0, time.time())
    launches = kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.2)
    clk = clocks.stop()
    status = max((s_.device_status() for s_ in scheds), key=abs)
    if status != 0:
        raise RuntimeError(f"device status {status}")
    ms_per_step = ev_a.elapsed_time(ev_b) / K
    kern_ms = [a.elapsed_time(z) for a, z in kev]
    kern_ms_avg = sum(kern_ms) / len(kern_ms)

    # An isolated-call measure beside the back-to-back number: one call at a
    # time, CUDA events around the call only, 20 warm-up calls then the
    # median of 200, L2 flushed (a 2 x L2 buffer written) before every call,
    # outside the event pair.
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    iso = []
    for i in range(220):
        r = i % n_copies
        flush.zero_()
        a_, z_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        decode_attention(pools[r], scheds[r], qs[i % 4], out=out, scale=wl.scale, workspace=wss[r], stream=stream)
        z_.record(stream)
        if i >= 20:
            iso.append((a_, z_))
    torch.cuda.synchronize()
    iso_us = statistics.median(a_.elapsed_time(z_) * 1e3 for a_, z_ in iso)
    del flush

    # End to end through the host-buffer entry point: H2D q, kernel, D2H out.
    qh = [q.cpu().pin_memory() for q in qs]
    oh = torch.empty_like(qh[0]).pin_memory()
    wshs = [s_.workspace(host_io=True) for s_ in scheds]
    Ke = min(K, 200)
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
    for i in range(Ke):
        r = i % n_copies
        eev[i][0].record(stream)
        scheds[r] = pools[r].schedule(batch, reuse=scheds[r], stream=stream, **skw)
        decode_attention_host(pools[r], scheds[r], qh[i % 4], oh, scale=wl.scale, workspace=wshs[r],
                              stream=stream)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_us = sum(a.elapsed_time(z) for a, z in eev) / Ke * 1e3

    # The same calls recorded into one CUDA graph (NG calls rotating over the
    # pool copies as the timed loop does) and replayed: one host launch per
    # NG calls instead of two kernel launches and the argument checks per
    # call.  Not for the churn workload, whose schedule changes every step.
    graph_us = graph_host_us = 0.0
    NG, RG = 32, 16
    if not churn:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.graph(g, stream=side):
            for i in range(NG):
                r = i % n_copies
                decode_attention(pools[r], scheds[r], qs[i % 4], out=out, scale=wl.scale, workspace=wss[r])
        stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ga, gz = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        ga.record(stream)
        for _ in range(RG):
            g.replay()
        gz.record(stream)
        graph_host_us = (time.perf_counter() - h0) * 1e6 / (RG * NG)
        torch.cuda.synchronize()
        graph_us = ga.elapsed_time(gz) * 1e3 / (RG * NG)
        if max((s_.device_status() for s_ in scheds), key=abs) != 0:
            raise RuntimeError("device status after graph replays")
        del g
    # the slowest rank's times (one rank: unchanged)
    ms_per_step, kern_ms_avg, e2e_us, iso_us, graph_us = max_over_ranks(
        [ms_per_step, kern_ms_avg, e2e_us, iso_us, graph_us], device=dev)

    # Context: the same batch through the flat paged layout (no sharing) and
    # through physically shared KV without the two-phase partition.
    context = None
    if not args.no_context and not churn:
        def time_calls(ps, ss, n=100):
            ws_ = [s_.workspace() for s_ in ss]
            m = len(ps)
            for i in range(10):
                decode_attention(ps[i % m], ss[i % m], qs[i % 4], out=out, scale=wl.scale, workspace=ws_[i % m],
                                 stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n):
                decode_attention(ps[i % m], ss[i % m], qs[i % 4], out=out, scale=wl.scale, workspace=ws_[i % m],
                                 stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n * 1e3
        no_tpp = [p_.schedule(batch, no_tpp=True, **skw) for p_ in pools]
        us_no_tpp = time_calls(pools, no_tpp)
        del no_tpp
        flat_bytes = sum(wl.seq_len(sid) for sid in batch) * HK * D * 2 * eb
        flats = make_pools(copies_for(flat_bytes), no_sharing=True, headroom=1.05)
        us_flat = time_calls(flats, [f.schedule(batch, **skw) for f in flats])
        del flats
        torch.cuda.empty_cache()
        context = {"paged_flat_us": round(us_flat, 2), "paged_shared_no_tpp_us": round(us_no_tpp, 2),
                   "note": "same kernel with every chunk sequence-first: flat = private copy of the "
                           "prefix per sequence (PagedAttention layout), shared_no_tpp = one copy read "
                           "once per sharer (ChunkAttention's PagedAttn* comparator)"}

    if world > 1 and rank != 0:
        torch.distributed.destroy_process_group()
        return

    unique_tokens = wl.unique_tokens()
    io_bytes = 2 * b * wl.q_len * H * D * 2                    # q in, out
    # the kernel variant the library launches: the few-row one when positions
    # bring 2..8 query rows per key/value head (head_dim <= 128)
    rows_per_kv = wl.q_len * (H // HK)
    few_rows = 2 <= rows_per_kv <= 8 and D <= 128
    kname = f"two_phase_attention_kernel<{c},{D},{eb},{'true' if few_rows else 'false'}>"
    alg_bytes = kv_bytes + io_bytes
    us = ms_per_step * 1e3
    peak, peak_kind = measured_peak()
    achieved = alg_bytes / (kern_ms_avg * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(whole_job_per_call(us, world), 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f16 q/out, fp8 e4m3 K/V storage (fp32 accumulate)" if wl.kv_dtype == "fp8"
                  else "f16 (fp32 accumulate)"),
        "data": "synthetic (seeded N(0,1) fp16 Q/K/V; token segments shaped like ChunkAttention's shared system prompts)",
        "config": {"workload": wl.name, "description": wl.description, "batch": b, "q_len": wl.q_len,
                   "n_heads": H,
                   "n_kv_heads": HK,
                   "head_dim": D, "chunk": c, "layers_per_call": 1,
                   "unique_kv_tokens": unique_tokens, "unique_kv_bytes": kv_bytes,
                   "l2": ("no flush: steps run back to back over %d pool cop%s (%d MB of unique KV each, "
                          "%d MB L2), so consecutive steps touch more than twice the L2; KV loads carry "
                          "an evict-first L2 hint" % (n_copies, "y" if n_copies == 1 else "ies",
                                                        kv_bytes >> 20, l2 >> 20)),
                   "pool_copies": n_copies,
                   "grid_ctas": scheds[0].plan()["grid"], "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "effective_hbm_gbs": round(alg_bytes / (us * 1e-6) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": kernel_traffic(f"{kname}:{wl.name}"),
                     "kernel": kname,
                     "kernel_us": round(kern_ms_avg * 1e3, 3),
                     "kernel_timing": f"CUDA events around the main kernel on {len(kev)} of the {K} timed steps",
                     "algorithmic_bytes": alg_bytes},
        "e2e": {"value": round(whole_job_per_call(e2e_us, world), 3), "unit": UNIT, "h2d_bytes_per_step": b * wl.q_len * H * D * 2,
                "d2h_bytes_per_step": b * wl.q_len * H * D * 2,
                "path": "ca_decode_attention_host: q read from and out written to pinned host memory by the "
                        "kernels through its device mapping (NVLink-C2C), inside each step's event pair"},
        "isolated_call": {"median_us": round(iso_us, 2), "reps": len(iso),
                          "method": "one call at a time: CUDA events around the call only, median of 200 "
                                    "after 20 warm-up calls, L2 flushed (2 x L2 written) before each call"},
        "graph_replay": ({"us_per_call": round(graph_us, 3), "calls_per_graph": NG, "replays": RG,
                          "host_us_per_call": round(graph_host_us, 2),
                          "method": "decode_attention calls recorded into one CUDA graph (torch.cuda.graph), "
                                    "replayed back to back; one event pair around all replays"}
                         if not churn else None),
        "gpu_launches": launches,
        "gpu_launches_source": "library launch counter (ca_kernel_launches) read around the timed loop",
        "clocks": clk,
        "wall_s_timed_loop": round(wall, 3),
        "host_enqueue_us_per_step": round(enqueue * 1e6 / K, 1),
        "setup_s": round(setup_s, 2),
    }
    if churn:
        res["config"]["churn_per_step"] = wl.churn
        res["churn_host_us"] = round(statistics.median(churn_host_us), 1)
        res["churn_host_split_us"] = {k: round(statistics.median(v), 1) for k, v in host_split.items()}
    if context:
        res["context"] = context
        res["context"]["speedup_vs_paged_flat"] = round(context["paged_flat_us"] / us, 2)
        res["context"]["speedup_vs_paged_shared_no_tpp"] = round(context["paged_shared_no_tpp_us"] / us, 2)
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import workloads
    wl = workloads.make(args.workload)
    per_step = []
    cb = None
    steps = max(1, min(args.steps, 3))
    for _ in range(steps):
        cb = cpu_baseline(wl, seconds=CPU_SAMPLE_SECONDS / steps)
        per_step.append(cb["value"])
    v = statistics.median(per_step)
    cb["value"] = v
    res = {"metric": METRIC, "value": round(v, 1), "unit": UNIT, "impl": "reference",
           "n_gpus": world, "steps": steps, "warmup": args.warmup,
           "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "description": wl.description},
           "cpu_baseline": cb,
           "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "note": "ChunkAttention's pages publish no code: the reference arm is the fp64 CPU oracle, timed on a "
                   "bounded sample and scaled to one layer call"}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
