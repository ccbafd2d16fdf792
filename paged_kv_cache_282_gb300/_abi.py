"""ctypes declarations of the libpkv C ABI (include/pkv.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

c_int32, c_int64, c_uint64, c_void_p, c_size_t, c_float, c_double = (
    ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float,
    ctypes.c_double)

PKV_OK = 0
STATUS_NAMES = {
    0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_OUT_OF_BLOCKS",
    4: "PKV_ERR_OUT_OF_SEQS", 5: "PKV_ERR_CUDA", 6: "PKV_ERR_TIMEOUT", 7: "PKV_ERR_DEVICE_ASSERT",
    8: "PKV_ERR_NO_DEVICE", 9: "PKV_ERR_WORKSPACE", 10: "PKV_ERR_HOST_MEMORY", 11: "PKV_ERR_UNDRAINED",
}
KV_DTYPES = {"fp32": 0, "bf16": 1, "fp8": 2, "fp8_e4m3": 2, "int8": 3}
MASKS = {"full": 0, "sliding": 1, "sink_window": 2}
KERNELS = ["cow_copy", "append", "decode", "combine", "h2o_score", "h2o_select", "table_patch", "swap_copy",
           "compact", "prefix_decode"]


class PKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class pkv_pool_config(ctypes.Structure):
    _fields_ = [("num_blocks", c_int32), ("block_size", c_int32), ("n_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("max_seqs", c_int32),
                ("max_blocks_per_seq", c_int32), ("kv_dtype", c_int32), ("alloc_seed", c_uint64),
                ("free_order", c_void_p)]


class pkv_pool_buffers(ctypes.Structure):
    _fields_ = [("k_pool", c_void_p), ("v_pool", c_void_p), ("k_scale", c_void_p), ("v_scale", c_void_p),
                ("block_tables", c_void_p), ("status", c_void_p)]


class pkv_buffer_sizes(ctypes.Structure):
    _fields_ = [("k_pool", c_size_t), ("v_pool", c_size_t), ("k_scale", c_size_t), ("v_scale", c_size_t),
                ("block_tables", c_size_t), ("status", c_size_t)]


class pkv_stats(ctypes.Structure):
    _fields_ = [("num_blocks", c_int64), ("free_blocks", c_int64), ("used_blocks", c_int64),
                ("shared_blocks", c_int64), ("active_seqs", c_int64), ("cow_copies", c_int64),
                ("blocks_allocated", c_int64), ("blocks_freed", c_int64)]


_P = ctypes.POINTER
SIGNATURES = {
    "pkv_pool_required_bytes": [_P(pkv_pool_config), _P(pkv_buffer_sizes)],
    "pkv_pool_create": [_P(pkv_pool_config), _P(pkv_pool_buffers), _P(c_void_p)],
    "pkv_pool_destroy": [c_void_p],
    "pkv_seq_add": [c_void_p, _P(c_int32)],
    "pkv_seq_fork": [c_void_p, c_int32, _P(c_int32)],
    "pkv_seq_free": [c_void_p, c_int32],
    "pkv_seq_truncate": [c_void_p, c_int32, c_int32],
    "pkv_seq_truncate_many": [c_void_p, c_int32, c_void_p, c_void_p],
    "pkv_seq_evict": [c_void_p, c_int32, c_int32, c_int32],
    "pkv_seq_len": [c_void_p, c_int32, _P(c_int32)],
    "pkv_get_block_table": [c_void_p, c_int32, c_void_p, c_int32, _P(c_int32)],
    "pkv_pool_stats": [c_void_p, _P(pkv_stats)],
    "pkv_reserve_slots": [c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_void_p, c_int32, _P(c_int32)],
    "pkv_append": [c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_void_p, c_void_p],
    "pkv_decode_workspace_size": [c_void_p, c_int32, c_int32, _P(c_size_t)],
    "pkv_decode_attn": [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_float, c_int32, c_int32, c_int32,
                        c_int32, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_size_t],
    "pkv_decode_attn_static": [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_float, c_int32, c_int32,
                               c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_int64],
    "pkv_h2o_scores": [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int64, c_void_p, c_int32, c_int32,
                       c_int32, c_void_p, c_int64],
    "pkv_h2o_select": [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int64, c_int32, c_int32, c_void_p,
                       c_int64, c_void_p],
    "pkv_policy_select": [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int64, c_int32, c_int32, c_int32,
                          c_void_p, c_int64, c_void_p],
    "pkv_seq_compact": [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_int64],
    "pkv_sync_status": [c_void_p, c_void_p],
    "pkv_timing_enable": [c_void_p, c_int32],
    "pkv_timing_read": [c_void_p, c_void_p, c_void_p],
    "pkv_launch_count": [c_void_p, _P(c_int64)],
    "pkv_set_wait_limit": [c_void_p, c_int64],
    "pkv_set_cascade": [c_void_p, c_int32],
    "pkv_set_channel_scales": [c_void_p, c_void_p, c_void_p],
    "pkv_swap_space_create": [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p],
    "pkv_swap_out": [c_void_p, c_void_p, c_int32, c_void_p],
    "pkv_swap_in": [c_void_p, c_void_p, c_int32, c_void_p],
    "pkv_seq_swapped": [c_void_p, c_int32, c_void_p],
    "pkv_get_host_block_table": [c_void_p, c_int32, c_void_p, c_int32, c_void_p],
    "pkv_host_free_blocks": [c_void_p, c_void_p],
    "pkv_test_starve_next_decode": [c_void_p, c_int32],
    "pkv_test_starve_next_select": [c_void_p],
    "pkv_test_set_geometry": [c_void_p, c_int32, c_int32, c_int32, c_int32],
    "pkv_test_plan_bytes": [c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p,
                            c_size_t, c_void_p, c_void_p],
    "pkv_test_cow_waves": [c_void_p, c_int32, c_void_p, c_void_p, c_int32, _P(c_int32)],
    "pkv_test_take_patches": [c_void_p, c_int32, c_void_p, c_int32, _P(c_int32)],
    "pkv_last_error": [],
    "pkv_version": [],
}

_lib = None


def load():
    """Loads the in-tree libpkv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpkv.so is not built ({LIB_PATH}); run `python -c 'import __graft_entry__ as g; "
                          f"g.build()'` or `python -m paged_kv_cache_282_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.pkv_pool_destroy.restype = None
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def check(status: int) -> None:
    if status != PKV_OK:
        raise PKVError(status, load().pkv_last_error().decode(errors="replace"))
