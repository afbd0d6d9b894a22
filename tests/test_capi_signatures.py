"""The five calls of the problem statement, called with exactly the
signatures include/chunk_attention.h declares: ca_pool_create,
ca_insert_tokens, ca_remove_seq, ca_build_schedule and ca_decode_attention.

* From C: tests/c_abi_five_calls.c is compiled against the header (the
  compiler checks every argument type) and run on a host-only pool.
* From Python: the argument types are read off the header's prototypes (not
  off the binding's table) and the calls are made through a separate ctypes
  handle, on a host-only pool and, on a GPU, on a device pool whose output is
  compared with the fp64 oracle [ChunkAttention (arXiv 2402.15220v4 summary)
  §3.1-§3.2; explainer blog, Two-Phase Partition]."""
import ctypes as C
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "chunk_attention.h")
FIVE = ["ca_pool_create", "ca_insert_tokens", "ca_remove_seq", "ca_build_schedule", "ca_decode_attention"]


class PoolConfig(C.Structure):
    """ca_pool_config as the header lays it out (six 32-bit fields)."""
    _fields_ = [("n_layers", C.c_int32), ("n_heads", C.c_int32), ("head_dim", C.c_int32),
                ("chunk", C.c_int32), ("capacity_slots", C.c_int32), ("flags", C.c_uint32)]


CTYPES = {
    "const ca_pool_config*": C.POINTER(PoolConfig),
    "void*": C.c_void_p, "const void*": C.c_void_p,
    "size_t": C.c_size_t, "float": C.c_float,
    "ca_pool*": C.c_void_p, "const ca_pool*": C.c_void_p, "const ca_sched*": C.c_void_p,
    "ca_pool**": C.POINTER(C.c_void_p), "ca_sched**": C.POINTER(C.c_void_p),
    "int64_t": C.c_int64, "int32_t": C.c_int32,
    "const int32_t*": C.POINTER(C.c_int32), "int32_t*": C.POINTER(C.c_int32),
    "const int64_t*": C.POINTER(C.c_int64),
}


def header_prototypes() -> dict[str, list[str]]:
    """name -> parameter types, from the header's declarations."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^int\s+(ca_\w+)\s*\(([^;]*?)\);", src, flags=re.M | re.S):
        params = []
        for p in m.group(2).split(","):
            p = " ".join(p.split())
            if p.endswith("]"):                                # "int32_t counts[6]": a pointer
                p = re.sub(r"\s*(\w+)\[\d*\]$", r"* \1", p)
            p = re.sub(r"\s*\*\s*", "*", p)                 # "ca_pool* pool" -> "ca_pool*pool"
            t = re.match(r"^(.*?[\*\s])\s*\w+$", p).group(1).strip()
            params.append(t.replace("* ", "*"))
        out[m.group(1)] = params
    return out


def five_calls_lib(lib):
    """A ctypes handle on the library whose five calls carry the header's
    argument types (independent of the binding's own table)."""
    from prefix_shared_decode_gb300 import capi
    L = C.CDLL(capi.LIB_PATH)
    protos = header_prototypes()
    for name in FIVE:
        fn = getattr(L, name)
        fn.argtypes = [CTYPES[t] for t in protos[name]]
        fn.restype = C.c_int
    return L, protos


def test_header_declares_the_five_calls_as_specified(lib):
    _, protos = five_calls_lib(lib)
    assert protos["ca_pool_create"] == ["const ca_pool_config*", "void*", "size_t", "ca_pool**"]
    assert protos["ca_insert_tokens"] == ["ca_pool*", "int64_t", "const int32_t*", "int32_t", "const void*",
                                          "const void*", "void*", "int32_t*"]
    assert protos["ca_remove_seq"] == ["ca_pool*", "int64_t"]
    assert protos["ca_build_schedule"] == ["ca_pool*", "const int64_t*", "int32_t", "ca_sched**", "void*"]
    assert protos["ca_decode_attention"] == ["const ca_pool*", "const ca_sched*", "int32_t", "const void*",
                                             "void*", "float", "void*", "size_t", "void*"]
    assert C.sizeof(PoolConfig) == 24


def test_c_program_calls_the_five_calls(lib, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from prefix_shared_decode_gb300 import capi
    libdir = os.path.dirname(capi.LIB_PATH)
    exe = str(tmp_path / "five_calls")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_five_calls.c"), "-o", exe, "-L", libdir,
                        "-l:libchunk_attention.so", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "five calls ok" in r.stdout


def test_ctypes_five_calls_host_only(lib):
    L, _ = five_calls_lib(lib)
    cfg = PoolConfig(1, 2, 64, 16, 64, 0)
    pool = C.c_void_p()
    assert L.ca_pool_create(C.byref(cfg), None, 0, C.byref(pool)) == 0
    toks = [np.arange(48, dtype=np.int32), np.r_[np.arange(32), 500 + np.arange(20)].astype(np.int32)]
    shared = C.c_int32(-1)
    P32 = C.POINTER(C.c_int32)
    for sid, t in enumerate(toks):
        assert L.ca_insert_tokens(pool, sid, t.ctypes.data_as(P32), len(t), None, None, None, C.byref(shared)) == 0
    assert shared.value == 32
    ids = np.array([1, 0], dtype=np.int64)
    sched = C.c_void_p()
    assert L.ca_build_schedule(pool, ids.ctypes.data_as(C.POINTER(C.c_int64)), 2, C.byref(sched), None) == 0
    assert L.ca_decode_attention(pool, sched, 0, None, None, 0.125, None, 0, None) == -1   # host-only pool
    assert L.ca_remove_seq(pool, 0) == 0
    assert L.ca_remove_seq(pool, 0) == -3                                                  # CA_ERR_NOT_FOUND
    # the schedule predates the remove: a device call would be refused as stale,
    # and a rebuild over the remaining sequence succeeds
    one = np.array([1], dtype=np.int64)
    assert L.ca_build_schedule(pool, one.ctypes.data_as(C.POINTER(C.c_int64)), 1, C.byref(sched), None) == 0
    lib.ca_sched_destroy(sched)
    lib.ca_pool_destroy(pool)


@pytest.mark.gpu
def test_ctypes_five_calls_on_the_gpu_match_the_oracle(lib):
    """A device pool driven only through the five calls with the header's
    signatures: two sequences sharing a 64-token prefix, then one removed;
    each decode output is compared with the fp64 oracle."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle import attention as A
    from prefix_shared_decode_gb300 import capi
    L, _ = five_calls_lib(lib)
    H, D, c = 4, 128, 16
    cfg = PoolConfig(1, H, D, c, 64, 0)
    nbytes = C.c_size_t()
    assert capi.lib().ca_pool_bytes(C.byref(capi.PoolConfig(1, H, D, c, 64, 0)), C.byref(nbytes)) == 0
    kv = torch.zeros(nbytes.value + 1024, dtype=torch.uint8, device="cuda")
    base = (kv.data_ptr() + 1023) // 1024 * 1024
    pool = C.c_void_p()
    assert L.ca_pool_create(C.byref(cfg), base, nbytes.value, C.byref(pool)) == 0
    rng = np.random.default_rng(11)
    prefix_k = rng.standard_normal((64, H, D), dtype=np.float32).astype(np.float16)
    prefix_v = rng.standard_normal((64, H, D), dtype=np.float32).astype(np.float16)
    seqs = {}
    P32 = C.POINTER(C.c_int32)
    stream = torch.cuda.current_stream().cuda_stream
    for sid, n_own in ((0, 37), (1, 21)):
        toks = np.r_[np.arange(64), 10_000 * (sid + 1) + np.arange(n_own)].astype(np.int32)
        k = np.concatenate([prefix_k, rng.standard_normal((n_own, H, D), dtype=np.float32).astype(np.float16)])
        v = np.concatenate([prefix_v, rng.standard_normal((n_own, H, D), dtype=np.float32).astype(np.float16)])
        seqs[sid] = (k, v)
        kd, vd = torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda()
        shared = C.c_int32(-1)
        assert L.ca_insert_tokens(pool, sid, toks.ctypes.data_as(P32), len(toks), kd.data_ptr(), vd.data_ptr(),
                                  stream, C.byref(shared)) == 0
        assert shared.value == (0 if sid == 0 else 64)
        torch.cuda.synchronize()
    scale = 1 / np.sqrt(D)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    sched = C.c_void_p()
    for batch in ([1, 0], [1]):
        ids = np.array(batch, dtype=np.int64)
        assert L.ca_build_schedule(pool, ids.ctypes.data_as(C.POINTER(C.c_int64)), len(ids), C.byref(sched),
                                   stream) == 0
        q = rng.standard_normal((len(batch), H, D), dtype=np.float32).astype(np.float16)
        qd = torch.from_numpy(q).cuda()
        out = torch.empty_like(qd)
        assert L.ca_decode_attention(pool, sched, 0, qd.data_ptr(), out.data_ptr(), scale, ws.data_ptr(),
                                     ws.numel(), stream) == 0
        assert capi.lib().ca_sched_device_status(sched, stream) == 0
        got = out.cpu().numpy().astype(np.float64)
        for i, sid in enumerate(batch):
            want = A.softmax_attention(q[i], *seqs[sid], scale)
            err = np.abs(got[i] - want)
            assert err.max() <= 2e-3 and err.mean() <= 2e-4, (batch, sid, err.max(), err.mean())
        if batch == [1, 0]:
            assert L.ca_remove_seq(pool, 0) == 0
    capi.lib().ca_sched_destroy(sched)
    capi.lib().ca_pool_destroy(pool)
    del kv
