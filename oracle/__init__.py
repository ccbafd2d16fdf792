"""CPU oracle for decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
timed CPU baseline in ``bench.py`` may import this package; the product
library never does.  It shares no code with the CUDA path.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64); this module only
marshals numpy arrays into it, plus the KV-size formulas, which are one line
each.

Sources (page title, section):
  [LC] "长上下文优化：注意力稀疏化与 KV Cache 管理" -- KV bytes per token
       formula and the ``kv_cache_gb`` helper; sliding-window mask;
       StreamingKVCache; H2OEviction.
  [PA] "KV Cache 与 PagedAttention：显存复用与长上下文推理" -- ``kv_cache_size``
       formula (Llama-2-70B table); block table, allocator, refcount + COW;
       FP8 E4M3 per-token quantisation.
  [SO] "系统优化" -- StreamingLLM keep-set and H2O ``evict_tokens``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

KV_FP32, KV_BF16, KV_FP8, KV_INT8 = 0, 1, 2, 3
MASK_FULL, MASK_SLIDING, MASK_SINK_WINDOW = 0, 1, 2
BLOCK = 16

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # ORACLE_LIB points at another build of pkv_oracle.c (the mutation
        # tests load deliberately broken copies to show the pins catch them)
        lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        c_int, c_dbl, vp = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = c_dbl
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_row_bf16.argtypes = [vp, c_int, vp, vp]
        lib.oracle_keep.argtypes = [c_int] * 5
        lib.oracle_keep.restype = c_int
        lib.oracle_scatter.argtypes = [vp, c_int, c_int, c_int, vp, c_int, vp]
        lib.oracle_quantize_scatter.argtypes = [vp, vp, c_int, c_int, vp, c_int, vp, c_int, vp]
        lib.oracle_quantize_row_channel.argtypes = [vp, c_int, vp, c_int, vp, vp]
        lib.oracle_int8_encode.argtypes = [ctypes.c_float]
        lib.oracle_int8_encode.restype = ctypes.c_int8
        lib.oracle_quantize_row_int8.argtypes = [vp, c_int, vp, vp]
        lib.oracle_copy_block.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int]
        lib.oracle_decode.argtypes = [c_int, c_int, c_int, c_int, c_int, vp, vp, vp, vp, c_int,
                                      vp, c_int, vp, c_int, vp, c_dbl, c_int, c_int, c_int,
                                      vp, vp, vp, c_int, c_int, vp, vp]
        lib.oracle_decode.restype = c_int
        lib.oracle_h2o_update.argtypes = [c_int, c_int, vp, vp, c_int, vp, c_int, c_int, c_int,
                                          vp, c_int]
        lib.oracle_h2o_select.argtypes = [c_int, c_int, c_int, vp, vp]
        lib.oracle_h2o_select.restype = c_int
        lib.oracle_policy_select.argtypes = [c_int, c_int, c_int, c_int, vp, vp]
        lib.oracle_policy_select.restype = c_int
        lib.oracle_splitmix64.argtypes = [ctypes.c_uint64, c_int, vp]
        lib.oracle_alloc_create.argtypes = [c_int, c_int, c_int, ctypes.c_uint64, vp]
        lib.oracle_alloc_create.restype = vp
        lib.oracle_alloc_destroy.argtypes = [vp]
        lib.oracle_alloc_seq_add.argtypes = [vp]
        lib.oracle_alloc_seq_add.restype = c_int
        lib.oracle_alloc_append.argtypes = [vp, c_int, vp, c_int, vp, vp, vp]
        lib.oracle_alloc_append.restype = c_int
        for name in ("oracle_alloc_fork", "oracle_alloc_free"):
            getattr(lib, name).argtypes = [vp, c_int]
            getattr(lib, name).restype = c_int
        lib.oracle_alloc_truncate.argtypes = [vp, c_int, c_int]
        lib.oracle_alloc_truncate.restype = c_int
        lib.oracle_alloc_compact.argtypes = [vp, c_int, vp, vp, vp]
        lib.oracle_alloc_compact.restype = c_int
        lib.oracle_copy_rows.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, vp, vp, c_int]
        lib.oracle_alloc_set_swap_space.argtypes = [vp, c_int]
        lib.oracle_alloc_set_swap_space.restype = c_int
        lib.oracle_alloc_swap_out.argtypes = [vp, c_int, vp, vp]
        lib.oracle_alloc_swap_out.restype = c_int
        lib.oracle_alloc_swap_in.argtypes = [vp, c_int, vp, vp]
        lib.oracle_alloc_swap_in.restype = c_int
        lib.oracle_alloc_swapped.argtypes = [vp, c_int]
        lib.oracle_alloc_swapped.restype = c_int
        lib.oracle_alloc_host_refcount.argtypes = [vp, c_int]
        lib.oracle_alloc_host_refcount.restype = c_int
        lib.oracle_alloc_num_host_free.argtypes = [vp]
        lib.oracle_alloc_num_host_free.restype = c_int
        lib.oracle_alloc_host_table.argtypes = [vp, c_int, vp]
        lib.oracle_alloc_host_table.restype = c_int
        lib.oracle_copy_blocks_between.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, vp, c_int]
        lib.oracle_alloc_evict.argtypes = [vp, c_int, c_int, c_int]
        lib.oracle_alloc_evict.restype = c_int
        lib.oracle_alloc_len.argtypes = [vp, c_int]
        lib.oracle_alloc_len.restype = c_int
        lib.oracle_alloc_table.argtypes = [vp, c_int, vp]
        lib.oracle_alloc_table.restype = c_int
        lib.oracle_alloc_refcount.argtypes = [vp, c_int]
        lib.oracle_alloc_refcount.restype = c_int
        lib.oracle_alloc_num_free.argtypes = [vp]
        lib.oracle_alloc_num_free.restype = c_int
        lib.oracle_alloc_free_list.argtypes = [vp, vp]
        lib.oracle_alloc_free_list.restype = c_int
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# KV-size formulas ([LC] "KV bytes per token" and kv_cache_gb; [PA]
# kv_cache_size).  Plain arithmetic, no rounding.
# --------------------------------------------------------------------------

def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """2 (K and V) x layers x kv_heads x head_dim x bytes per element."""
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes


def kv_cache_gib(n_layers: int, n_kv_heads: int, head_dim: int, max_len: int, batch: int = 1,
                 dtype_bytes: int = 2) -> float:
    """[LC] kv_cache_gb: per-token bytes x max_len x batch / 1024**3."""
    return kv_bytes_per_token(n_layers, n_kv_heads, head_dim, dtype_bytes) * max_len * batch / 1024 ** 3


def kv_cache_size_bytes(layers: int, kv_heads: int, head_dim: int, seq_len: int, bytes_per: int = 2) -> int:
    """[PA] kv_cache_size: 2 x layers x kv_heads x head_dim x seq_len x bytes."""
    return 2 * layers * kv_heads * head_dim * seq_len * bytes_per


# --------------------------------------------------------------------------
# FP8 E4M3 codec and quantiser.
# --------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_e4m3_encode(float(v)) for v in flat), dtype=np.uint8,
                       count=flat.size).reshape(np.shape(x))


def int8_encode(x: float) -> int:
    return int(_load().oracle_int8_encode(float(x)))


def quantize_row_int8(row_bits: np.ndarray):
    """row_bits: uint16 bf16 bit patterns [D] -> (codes int8 [D], scale fp32)."""
    lib = _load()
    row_bits = _c(row_bits, np.uint16)
    codes = np.empty(row_bits.size, dtype=np.int8)
    scale = np.zeros(1, dtype=np.float32)
    lib.oracle_quantize_row_int8(_ptr(row_bits), row_bits.size, _ptr(codes), _ptr(scale))
    return codes, float(scale[0])


def quantize_row_channel(row_bits: np.ndarray, channel, kv_dtype: int):
    """Per-channel + per-token quantisation of one row: row_bits uint16 bf16
    bit patterns [D], channel fp32 [D] (or None) -> (codes [D], scale fp32)."""
    lib = _load()
    row_bits = _c(row_bits, np.uint16)
    ch = None if channel is None else _c(channel, np.float32)
    codes = np.empty(row_bits.size, dtype=np.int8 if kv_dtype == KV_INT8 else np.uint8)
    scale = np.zeros(1, dtype=np.float32)
    lib.oracle_quantize_row_channel(_ptr(row_bits), row_bits.size, _ptr(ch), kv_dtype, _ptr(codes), _ptr(scale))
    return codes, float(scale[0])


def quantize_row_bf16(row_bits: np.ndarray):
    """row_bits: uint16 bf16 bit patterns [D] -> (codes uint8 [D], scale fp32)."""
    lib = _load()
    row_bits = _c(row_bits, np.uint16)
    codes = np.empty(row_bits.size, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.float32)
    lib.oracle_quantize_row_bf16(_ptr(row_bits), row_bits.size, _ptr(codes), _ptr(scale))
    return codes, float(scale[0])


# --------------------------------------------------------------------------
# Keep-set predicate.
# --------------------------------------------------------------------------

def keep(L: int, mode: int, num_sinks: int, window: int, j: int) -> bool:
    return bool(_load().oracle_keep(L, mode, num_sinks, window, j))


def keep_set(L: int, mode: int, num_sinks: int = 0, window: int = 0) -> list[int]:
    return [j for j in range(L) if keep(L, mode, num_sinks, window, j)]


# --------------------------------------------------------------------------
# Paged pool built by the oracle itself.
# --------------------------------------------------------------------------

class OraclePool:
    """Host arrays laid out [NB][Hk][16][D] (+ scales [NB][Hk][16] for FP8)."""

    def __init__(self, num_blocks: int, n_kv_heads: int, head_dim: int, kv_dtype: int):
        self.NB, self.Hk, self.D, self.kv_dtype = num_blocks, n_kv_heads, head_dim, kv_dtype
        self.k_channel = self.v_channel = None  # per-channel scales [Hk][D] (FP8 / INT8), or None
        dt = {KV_FP32: np.float32, KV_BF16: np.uint16, KV_FP8: np.uint8, KV_INT8: np.int8}[kv_dtype]
        shape = (num_blocks, n_kv_heads, BLOCK, head_dim)
        self.k = np.zeros(shape, dtype=dt)
        self.v = np.zeros(shape, dtype=dt)
        if kv_dtype in (KV_FP8, KV_INT8):
            self.k_scale = np.zeros(shape[:3], dtype=np.float32)
            self.v_scale = np.zeros(shape[:3], dtype=np.float32)
        else:
            self.k_scale = self.v_scale = None

    def write(self, slots: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray) -> None:
        """Place T new tokens at their slots.  k_rows/v_rows: [T][Hk][D] raw
        element bits (fp32 values, or bf16 bit patterns as uint16)."""
        lib = _load()
        slots = _c(slots, np.int64)
        T = slots.size
        if self.kv_dtype in (KV_FP8, KV_INT8):
            kb, vb = _c(k_rows, np.uint16), _c(v_rows, np.uint16)
            lib.oracle_quantize_scatter(_ptr(self.k), _ptr(self.k_scale), self.Hk, self.D,
                                        _ptr(slots), T, _ptr(kb), self.kv_dtype, _ptr(self.k_channel))
            lib.oracle_quantize_scatter(_ptr(self.v), _ptr(self.v_scale), self.Hk, self.D,
                                        _ptr(slots), T, _ptr(vb), self.kv_dtype, _ptr(self.v_channel))
        else:
            dt = np.float32 if self.kv_dtype == KV_FP32 else np.uint16
            kb, vb = _c(k_rows, dt), _c(v_rows, dt)
            es = 4 if self.kv_dtype == KV_FP32 else 2
            lib.oracle_scatter(_ptr(self.k), self.Hk, self.D, es, _ptr(slots), T, _ptr(kb))
            lib.oracle_scatter(_ptr(self.v), self.Hk, self.D, es, _ptr(slots), T, _ptr(vb))

    def set_channel_scales(self, k_channel, v_channel) -> None:
        """Per-channel scales [Hk][D] fp32 for K and V (FP8 / INT8 pools), or
        None for both: the per-token scheme."""
        if k_channel is None:
            self.k_channel = self.v_channel = None
            return
        self.k_channel = _c(k_channel, np.float32).reshape(self.Hk, self.D)
        self.v_channel = _c(v_channel, np.float32).reshape(self.Hk, self.D)

    def copy_rows(self, src_slots, dst_slots) -> None:
        es = {KV_FP32: 4, KV_BF16: 2, KV_FP8: 1, KV_INT8: 1}[self.kv_dtype]
        src, dst = _c(src_slots, np.int64), _c(dst_slots, np.int64)
        _load().oracle_copy_rows(_ptr(self.k), _ptr(self.v), _ptr(self.k_scale), _ptr(self.v_scale), self.Hk,
                                 self.D, es, _ptr(src), _ptr(dst), src.size)

    def add_host_pool(self, num_host_blocks: int) -> None:
        """Host-side swap space with the device pool's layout."""
        self.NH = num_host_blocks
        self.hk = np.zeros((num_host_blocks,) + self.k.shape[1:], dtype=self.k.dtype)
        self.hv = np.zeros_like(self.hk)
        if self.k_scale is not None:
            self.hk_scale = np.zeros((num_host_blocks,) + self.k_scale.shape[1:], dtype=np.float32)
            self.hv_scale = np.zeros_like(self.hk_scale)
        else:
            self.hk_scale = self.hv_scale = None

    def swap_copy(self, pairs: np.ndarray, out: bool) -> None:
        """Block copies device -> host (out) or host -> device."""
        pairs = _c(pairs, np.int32)
        es = {KV_FP32: 4, KV_BF16: 2, KV_FP8: 1, KV_INT8: 1}[self.kv_dtype]
        src = (self.k, self.v, self.k_scale, self.v_scale)
        dst = (self.hk, self.hv, self.hk_scale, self.hv_scale)
        if not out:
            src, dst = dst, src
        _load().oracle_copy_blocks_between(*(_ptr(x) for x in src), *(_ptr(x) for x in dst), self.Hk, self.D, es,
                                           _ptr(pairs), pairs.size // 2)

    def copy_block(self, src: int, dst: int) -> None:
        es = {KV_FP32: 4, KV_BF16: 2, KV_FP8: 1, KV_INT8: 1}[self.kv_dtype]
        _load().oracle_copy_block(_ptr(self.k), _ptr(self.v), _ptr(self.k_scale),
                                  _ptr(self.v_scale), self.Hk, self.D, es, src, dst)


def decode(pool: OraclePool, tables: np.ndarray, lens: np.ndarray, q: np.ndarray, q_dtype: int,
           n_heads: int, scale: float, mask_mode: int = MASK_FULL, num_sinks: int = 0,
           window: int = 0, want_logits: bool = False, logits_stride: int | None = None,
           n_threads: int | None = None):
    """fp64 decode attention over the pool gathered through ``tables``.

    q: [n][H][D] (fp32 values, or bf16 bit patterns as uint16 with q_dtype=KV_BF16).
    Returns (out [n][H][D] f64, lse [n][H] f64, logits [n][H][stride] f64 or None).
    Logits are the natural-unit scaled scores of kept positions (NaN elsewhere).
    """
    lib = _load()
    tables = _c(tables, np.int32)
    lens = _c(lens, np.int32)
    n, max_blocks = tables.shape
    q = _c(q, np.float32 if q_dtype == KV_FP32 else np.uint16)
    out = np.zeros((n, n_heads, pool.D), dtype=np.float64)
    lse = np.zeros((n, n_heads), dtype=np.float64)
    logits = None
    if want_logits:
        logits_stride = int(logits_stride or max(1, int(lens.max()) if n else 1))
        logits = np.full((n, n_heads, logits_stride), np.nan, dtype=np.float64)
    threads = n_threads or os.cpu_count() or 1
    bad = lib.oracle_decode(n, n_heads, pool.Hk, pool.D, pool.kv_dtype, _ptr(pool.k), _ptr(pool.v),
                            _ptr(pool.k_scale), _ptr(pool.v_scale), pool.NB, _ptr(tables),
                            max_blocks, _ptr(lens), q_dtype, _ptr(q), float(scale), mask_mode,
                            num_sinks, window, _ptr(out), _ptr(lse), _ptr(logits),
                            int(logits_stride or 0), threads, _ptr(pool.k_channel), _ptr(pool.v_channel))
    if bad:
        raise ValueError("a kept token maps to an invalid physical block")
    return out, lse, logits


# --------------------------------------------------------------------------
# H2O.
# --------------------------------------------------------------------------

def h2o_update(acc: np.ndarray, lens: np.ndarray, logits: np.ndarray, lse: np.ndarray,
               mask_mode: int = MASK_FULL, num_sinks: int = 0, window: int = 0) -> np.ndarray:
    """acc [n][stride] f64 updated in place with this step's mean-over-heads weights."""
    lib = _load()
    assert acc.dtype == np.float64 and acc.flags.c_contiguous
    lens = _c(lens, np.int32)
    logits = _c(logits, np.float64)
    lse = _c(lse, np.float64)
    n, H, lstride = logits.shape
    lib.oracle_h2o_update(n, H, _ptr(lens), _ptr(logits), lstride, _ptr(lse), mask_mode,
                          num_sinks, window, _ptr(acc), acc.shape[1])
    return acc


def policy_select(L: int, sinks: int, window: int, heavy: int, scores: np.ndarray) -> np.ndarray:
    """The combined sink + recent window + heavy-hitter keep-set (ascending)."""
    lib = _load()
    scores = _c(scores, np.float64)
    out = np.empty(max(L, 1), dtype=np.int32)
    n = lib.oracle_policy_select(L, sinks, window, heavy, _ptr(scores), _ptr(out))
    return out[:n].copy()


def h2o_select(L: int, budget: int, recent: int, scores: np.ndarray) -> np.ndarray:
    lib = _load()
    scores = _c(scores, np.float64)
    out = np.empty(max(L, 1), dtype=np.int32)
    n = lib.oracle_h2o_select(L, budget, recent, _ptr(scores), _ptr(out))
    return out[:n].copy()


# --------------------------------------------------------------------------
# Allocator replay.
# --------------------------------------------------------------------------

def splitmix64_stream(seed: int, n: int) -> list[int]:
    out = np.zeros(n, dtype=np.uint64)
    _load().oracle_splitmix64(ctypes.c_uint64(seed & (2 ** 64 - 1)), n, _ptr(out))
    return [int(x) for x in out]


class OracleAllocator:
    def __init__(self, num_blocks: int, max_seqs: int, max_blocks_per_seq: int, seed: int = 0,
                 order=None):
        self._lib = _load()
        self._order = None if order is None else _c(order, np.int32)
        self._h = self._lib.oracle_alloc_create(num_blocks, max_seqs, max_blocks_per_seq,
                                                ctypes.c_uint64(seed & (2 ** 64 - 1)),
                                                _ptr(self._order))
        self.NB, self.max_seqs, self.max_blocks = num_blocks, max_seqs, max_blocks_per_seq

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.oracle_alloc_destroy(h)
            self._h = None

    def seq_add(self) -> int:
        s = self._lib.oracle_alloc_seq_add(self._h)
        if s < 0:
            raise RuntimeError("no free sequence id")
        return s

    def append(self, seq_ids, T: int):
        """Returns (slots int64 [n*T], cow_pairs int32 [ncow][2]) or raises."""
        ids = _c(seq_ids, np.int32)
        slots = np.empty(max(ids.size * T, 1), dtype=np.int64)
        cow = np.empty((max(ids.size * T, 1), 2), dtype=np.int32)
        ncow = ctypes.c_int(0)
        r = self._lib.oracle_alloc_append(self._h, ids.size, _ptr(ids), T, _ptr(slots), _ptr(cow),
                                          ctypes.byref(ncow))
        if r == -1:
            raise MemoryError("out of blocks")
        if r != 0:
            raise ValueError("invalid append")
        return slots[: ids.size * T].copy(), cow[: ncow.value].copy()

    def fork(self, src: int) -> int:
        r = self._lib.oracle_alloc_fork(self._h, src)
        if r < 0:
            raise ValueError("fork failed")
        return r

    def free(self, s: int) -> None:
        if self._lib.oracle_alloc_free(self._h, s):
            raise ValueError("free failed")

    def truncate(self, s: int, new_len: int) -> None:
        if self._lib.oracle_alloc_truncate(self._h, s, new_len):
            raise ValueError("truncate failed")

    def evict(self, s: int, num_sinks: int, window: int) -> None:
        if self._lib.oracle_alloc_evict(self._h, s, num_sinks, window):
            raise ValueError("evict failed")

    def set_swap_space(self, num_host_blocks: int) -> None:
        if self._lib.oracle_alloc_set_swap_space(self._h, num_host_blocks):
            raise ValueError("swap space in use")
        self.NH = num_host_blocks

    def _swap(self, fn, seq_ids) -> np.ndarray:
        ids = _c(seq_ids, np.int32)
        out = np.empty((max(self.NB, getattr(self, "NH", 0), 1), 2), dtype=np.int32)
        r = fn(self._h, ids.size, _ptr(ids), _ptr(out))
        if r == -1:
            raise MemoryError("out of blocks")
        if r < 0:
            raise ValueError("invalid swap")
        return out[:r].copy()

    def swap_out(self, seq_ids) -> np.ndarray:
        """CPU swap-out; returns the (device block, host block) copies."""
        return self._swap(self._lib.oracle_alloc_swap_out, seq_ids)

    def swap_in(self, seq_ids) -> np.ndarray:
        """CPU swap-in; returns the (host block, device block) copies."""
        return self._swap(self._lib.oracle_alloc_swap_in, seq_ids)

    def swapped(self, s: int) -> bool:
        return bool(self._lib.oracle_alloc_swapped(self._h, s))

    def host_refcount(self, b: int) -> int:
        return self._lib.oracle_alloc_host_refcount(self._h, b)

    def num_host_free(self) -> int:
        return self._lib.oracle_alloc_num_host_free(self._h)

    def host_table(self, s: int) -> np.ndarray:
        out = np.empty(max(self.max_blocks, 1), dtype=np.int32)
        n = self._lib.oracle_alloc_host_table(self._h, s, _ptr(out))
        return out[:n].copy()

    def compact(self, seq_ids, counts) -> list:
        """H2O compaction of the allocator state; returns each sequence's
        fresh blocks."""
        ids, cnt = _c(seq_ids, np.int32), _c(counts, np.int32)
        total = int(sum((int(c) + 15) // 16 for c in cnt))
        out = np.empty(max(total, 1), dtype=np.int32)
        r = self._lib.oracle_alloc_compact(self._h, ids.size, _ptr(ids), _ptr(cnt), _ptr(out))
        if r == -1:
            raise MemoryError("out of blocks")
        if r != 0:
            raise ValueError("invalid compaction")
        res, pos = [], 0
        for c in cnt:
            nb = (int(c) + 15) // 16
            res.append(out[pos: pos + nb].copy())
            pos += nb
        return res

    def length(self, s: int) -> int:
        return self._lib.oracle_alloc_len(self._h, s)

    def table(self, s: int) -> np.ndarray:
        out = np.empty(self.max_blocks, dtype=np.int32)
        n = self._lib.oracle_alloc_table(self._h, s, _ptr(out))
        return out[:n].copy()

    def refcount(self, b: int) -> int:
        return self._lib.oracle_alloc_refcount(self._h, b)

    def num_free(self) -> int:
        return self._lib.oracle_alloc_num_free(self._h)

    def free_list(self) -> np.ndarray:
        out = np.empty(max(self.NB, 1), dtype=np.int32)
        n = self._lib.oracle_alloc_free_list(self._h, _ptr(out))
        return out[:n].copy()

    def tables_matrix(self, seq_ids) -> np.ndarray:
        """Dense [n][max_blocks] int32 table for the given sequences (-1 padded)."""
        m = np.full((len(seq_ids), self.max_blocks), -1, dtype=np.int32)
        for i, s in enumerate(seq_ids):
            t = self.table(s)
            m[i, : t.size] = t
        return m
