"""The benchmark's multi-process path on CPU: under torchrun every rank runs
an independent replica of the step (no collective on the data path); the
job's times are the slowest rank's (a max-reduction over `gloo` ranks here,
NCCL on GPUs), and the whole-job time per call divides by the ranks."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        q.put((rank, bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank])))
    finally:
        dist.destroy_process_group()


def test_times_are_the_slowest_ranks_over_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [2.0, 10.0, 0.5]


def test_one_process_and_whole_job_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]          # no process group
    assert bench.whole_job_per_call(100.0, 4) == 25.0
    assert bench.whole_job_per_call(100.0, 1) == 100.0


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""


def test_reference_arm_reports_the_same_config_and_steps(capsys):
    """The reference arm (the oracle over the host cores) prints the same
    workload config the GPU arm prints and times exactly --steps steps."""
    sys.path.insert(0, ROOT)
    import json

    import bench
    import workloads
    args = bench.parse(["--impl", "reference", "--workload", "tiny", "--steps", "4", "--warmup", "1"])
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 4 and line["warmup"] == 1
    assert line["config"] == bench.workload_config(workloads.make("tiny"))
    assert line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["e2e"]["value"] == line["value"] and line["unit"] == bench.UNIT


def test_cpu_baseline_over_the_host_cores_with_one_thread_figure():
    sys.path.insert(0, ROOT)
    import bench
    cb = bench.cpu_baseline("tiny", seconds=0.3)
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() and cb["value"] > 0
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0


def test_oracle_pool_calls_are_bounded_when_worker_setup_fails():
    """A pool whose workers cannot set up (an unknown workload here) makes
    multiprocessing respawn them for ever; the benchmark's calls give up
    after their limit instead of hanging, and the CPU baseline reports the
    failure in the line instead of raising."""
    import multiprocessing
    import time
    sys.path.insert(0, ROOT)
    import bench
    op = bench.OraclePool("no_such_workload", cores=2)
    t0 = time.perf_counter()
    try:
        with pytest.raises(multiprocessing.TimeoutError):
            op.call([0, 1], timeout=3.0)
    finally:
        op.close()
    assert time.perf_counter() - t0 < 60
    cb = bench.cpu_baseline("no_such_workload", seconds=0.1)
    assert cb["value"] is None and "KeyError" in cb["error"]
