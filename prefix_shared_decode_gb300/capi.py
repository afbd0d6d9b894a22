"""ctypes declarations of the C ABI in include/chunk_attention.h.

Loading fails loudly when libchunk_attention.so has not been built: there is
no fallback implementation of any call."""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libchunk_attention.so")

CA_OK = 0
CA_ERR_STALE = -5
ERRORS = {
    -1: "CA_ERR_INVALID", -2: "CA_ERR_OOM", -3: "CA_ERR_NOT_FOUND", -4: "CA_ERR_EXISTS",
    -5: "CA_ERR_STALE", -6: "CA_ERR_CUDA", -7: "CA_ERR_DEVICE_BOUNDS", -8: "CA_ERR_TIMEOUT",
    -9: "CA_ERR_UNSUPPORTED", -10: "CA_ERR_SCRATCH_LIMIT",
}
CA_STATIC_WS_BYTES = 16 << 20
CA_NO_SHARING = 1
CA_KV_FP8 = 2
CA_SCHED_NO_TPP = 1
CA_SCHED_CAUSAL = 2

# Every symbol the header declares, in header order.
EXPORTS = [
    "ca_pool_bytes", "ca_pool_bytes_ex", "ca_pool_create", "ca_pool_create_ex", "ca_pool_destroy", "ca_match_prefix", "ca_insert_tokens",
    "ca_insert_batch", "ca_append_tokens", "ca_remove_seq", "ca_remove_batch", "ca_pool_stats", "ca_seq_slots", "ca_build_schedule", "ca_build_schedule_ex", "ca_sched_destroy",
    "ca_sched_counts", "ca_export_tables", "ca_export_plan", "ca_workspace_bytes", "ca_decode_attention",
    "ca_workspace_bytes_host", "ca_decode_attention_host", "ca_decode_attention_static_ws",
    "ca_sched_device_status", "ca_sched_inject_status", "ca_sched_inject_stall", "ca_pool_inject_alloc_failure",
    "ca_sched_set_profile_events", "ca_kernel_launches", "ca_error_string",
]


class PoolConfig(C.Structure):
    """ca_pool_config."""
    _fields_ = [("n_layers", C.c_int32), ("n_heads", C.c_int32), ("head_dim", C.c_int32),
                ("chunk", C.c_int32), ("capacity_slots", C.c_int32), ("flags", C.c_uint32)]


class PoolConfigEx(C.Structure):
    """ca_pool_config_ex: a ca_pool_config, then the grouped-query and fp8 fields."""
    _fields_ = [("base", PoolConfig), ("n_kv_heads", C.c_int32), ("k_scale", C.c_float),
                ("v_scale", C.c_float)]


class Stats(C.Structure):
    _fields_ = [("live_slots", C.c_int64), ("free_slots", C.c_int64), ("refcount_sum", C.c_int64),
                ("live_seqs", C.c_int64), ("generation", C.c_int64)]


class CAError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        self.name = ERRORS.get(code, str(code))
        super().__init__(f"{what}: {self.name}" if what else self.name)


_lib = None


def lib() -> C.CDLL:
    """The loaded library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with prefix_shared_decode_gb300.build.build() "
            "(there is no fallback path)")
    L = C.CDLL(LIB_PATH)
    i32, u32, i64, sz, vp = C.c_int32, C.c_uint32, C.c_int64, C.c_size_t, C.c_void_p
    P = C.POINTER
    sig = {
        "ca_pool_bytes": [P(PoolConfig), P(sz)],
        "ca_pool_bytes_ex": [P(PoolConfigEx), P(sz)],
        "ca_pool_create": [P(PoolConfig), vp, sz, P(vp)],
        "ca_pool_create_ex": [P(PoolConfigEx), vp, sz, P(vp)],
        "ca_pool_destroy": [vp],
        "ca_match_prefix": [vp, P(i32), i32, P(i32)],
        "ca_insert_tokens": [vp, i64, P(i32), i32, vp, vp, vp, P(i32)],
        "ca_insert_batch": [vp, i32, P(i64), P(i32), P(i32), vp, vp, vp, P(i32)],
        "ca_append_tokens": [vp, i64, P(i32), i32, vp, vp, vp, P(i32)],
        "ca_remove_seq": [vp, i64],
        "ca_remove_batch": [vp, i32, P(i64)],
        "ca_pool_stats": [vp, P(Stats)],
        "ca_seq_slots": [vp, i64, P(i32), i32, P(i32)],
        "ca_build_schedule": [vp, P(i64), i32, P(vp), vp],
        "ca_build_schedule_ex": [vp, vp, i32, i32, u32, P(vp), vp],     # seq_ids: int64 array address
        "ca_sched_destroy": [vp],
        "ca_sched_counts": [vp, P(i32)],
        "ca_export_tables": [vp] + [P(i32)] * 7,
        "ca_export_plan": [vp, P(i32), P(i32), P(i32), P(i32), P(i32)],
        "ca_workspace_bytes": [vp, P(sz)],
        "ca_workspace_bytes_host": [vp, P(sz)],
        "ca_decode_attention": [vp, vp, i32, vp, vp, C.c_float, vp, sz, vp],
        "ca_decode_attention_host": [vp, vp, i32, vp, vp, C.c_float, vp, sz, vp],
        "ca_decode_attention_static_ws": [vp, vp, i32, vp, vp, C.c_float, vp],
        "ca_sched_device_status": [vp, vp],
        "ca_sched_inject_status": [vp, i32, vp],
        "ca_sched_inject_stall": [vp, i32],
        "ca_pool_inject_alloc_failure": [vp, i32],
        "ca_sched_set_profile_events": [vp, vp, vp],
        "ca_kernel_launches": [vp],
        "ca_error_string": [C.c_int],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = C.c_char_p if name == "ca_error_string" else C.c_int
    _lib = L
    return L


def check(status: int, what: str = "") -> int:
    if status != CA_OK:
        raise CAError(status, what)
    return status
