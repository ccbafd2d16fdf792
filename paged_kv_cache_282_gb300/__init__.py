"""paged_kv_cache_282_gb300 -- decode attention over a paged KV cache on GB300.

A thin Python binding over ``libpkv.so`` (C ABI in ``include/pkv.h``).  Every
step of the path runs in the library's CUDA kernels; this module only
allocates device buffers with torch, passes pointers and the current stream,
and turns status codes into exceptions.  There is no CPU fallback: without the
built library every call raises.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from . import _abi
from ._abi import KERNELS, KV_DTYPES, MASKS, PKVError, load

__all__ = ["PagedKVCache", "PKVError", "load", "KERNELS", "version"] + [n for n in _abi.SIGNATURES]

BLOCK_SIZE = 16


def version() -> str:
    return load().pkv_version().decode()


def _stream_ptr(stream) -> int:
    """The CUDA stream handle for a call: `stream`, else torch's current stream
    on the current device (read straight from torch's C layer when it offers
    that, which costs far less per call than building a Stream object)."""
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return int(raw(torch._C._cuda_getDevice()))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _i32_array(values) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(values, dtype=np.int32))


def _ptr(arr: np.ndarray) -> int:
    """The address of a host array for a `void*` argument.  A plain integer
    (cheaper than a ctypes pointer object), so the caller keeps `arr` alive
    across the call: every caller passes an array held in a local name."""
    return arr.ctypes.data


# Raw C-ABI entry points, re-exported under their own names (marshalling is
# the caller's: ctypes arguments as declared in _abi.SIGNATURES).
def __getattr__(name):
    if name in _abi.SIGNATURES:
        return getattr(load(), name)
    raise AttributeError(name)


class PagedKVCache:
    """One KV pool: device buffers (torch-allocated), the library handle, and
    methods that forward to the C ABI.

    kv_dtype: "fp32" | "bf16" | "fp8" | "int8".  host_only=True creates the allocator
    without device buffers (allocator calls only)."""

    def __init__(self, num_blocks: int, n_heads: int, n_kv_heads: int, head_dim: int, max_seqs: int,
                 max_blocks_per_seq: int, kv_dtype: str = "bf16", alloc_seed: int = 0, free_order=None,
                 device="cuda", host_only: bool = False):
        self.lib = load()
        self.kv_dtype = kv_dtype
        self.n_heads, self.n_kv_heads, self.head_dim = n_heads, n_kv_heads, head_dim
        self.group = n_heads // n_kv_heads
        self.num_blocks, self.max_seqs, self.max_blocks_per_seq = num_blocks, max_seqs, max_blocks_per_seq
        self._order = None if free_order is None else _i32_array(free_order)
        self.cfg = _abi.pkv_pool_config(num_blocks, BLOCK_SIZE, n_heads, n_kv_heads, head_dim, max_seqs,
                                        max_blocks_per_seq, KV_DTYPES[kv_dtype], alloc_seed & (2 ** 64 - 1),
                                        None if self._order is None else _ptr(self._order))
        self._h = ctypes.c_void_p()
        self.host_only = host_only
        self._workspace = None
        if host_only:
            _abi.check(self.lib.pkv_pool_create(ctypes.byref(self.cfg), None, ctypes.byref(self._h)))
            return
        import torch
        self.device = torch.device(device)
        sizes = _abi.pkv_buffer_sizes()
        _abi.check(self.lib.pkv_pool_required_bytes(ctypes.byref(self.cfg), ctypes.byref(sizes)))
        dt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8, "int8": torch.int8}[kv_dtype]
        shape = (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim)
        with torch.cuda.device(self.device):
            self.k_pool = torch.empty(shape, dtype=dt, device=self.device)
            self.v_pool = torch.empty(shape, dtype=dt, device=self.device)
            if kv_dtype in ("fp8", "int8"):
                self.k_scale = torch.empty(shape[:3], dtype=torch.float32, device=self.device)
                self.v_scale = torch.empty(shape[:3], dtype=torch.float32, device=self.device)
            else:
                self.k_scale = self.v_scale = None
            self.block_tables = torch.empty((max_seqs, max_blocks_per_seq), dtype=torch.int32, device=self.device)
            self.status = torch.zeros(4, dtype=torch.int32, device=self.device)
            bufs = _abi.pkv_pool_buffers(self.k_pool.data_ptr(), self.v_pool.data_ptr(),
                                         self.k_scale.data_ptr() if self.k_scale is not None else None,
                                         self.v_scale.data_ptr() if self.v_scale is not None else None,
                                         self.block_tables.data_ptr(), self.status.data_ptr())
            _abi.check(self.lib.pkv_pool_create(ctypes.byref(self.cfg), ctypes.byref(bufs), ctypes.byref(self._h)))

    # ---- lifetime ---------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            self.lib.pkv_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # ---- sequences --------------------------------------------------------
    def seq_add(self) -> int:
        s = ctypes.c_int32()
        _abi.check(self.lib.pkv_seq_add(self._h, ctypes.byref(s)))
        return s.value

    def seq_fork(self, src: int) -> int:
        d = ctypes.c_int32()
        _abi.check(self.lib.pkv_seq_fork(self._h, src, ctypes.byref(d)))
        return d.value

    def seq_free(self, seq: int) -> None:
        _abi.check(self.lib.pkv_seq_free(self._h, seq))

    def seq_truncate(self, seq: int, new_len: int) -> None:
        _abi.check(self.lib.pkv_seq_truncate(self._h, seq, new_len))

    def seq_truncate_many(self, seq_ids, new_lens) -> None:
        ids, lens = _i32_array(seq_ids), _i32_array(new_lens)
        assert ids.size == lens.size
        _abi.check(self.lib.pkv_seq_truncate_many(self._h, ids.size, _ptr(ids), _ptr(lens)))

    def seq_evict(self, seq: int, num_sinks: int, window: int) -> None:
        _abi.check(self.lib.pkv_seq_evict(self._h, seq, num_sinks, window))

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int32()
        _abi.check(self.lib.pkv_seq_len(self._h, seq, ctypes.byref(n)))
        return n.value

    def block_table(self, seq: int) -> np.ndarray:
        out = np.empty(self.max_blocks_per_seq, dtype=np.int32)
        n = ctypes.c_int32()
        _abi.check(self.lib.pkv_get_block_table(self._h, seq, _ptr(out), out.size, ctypes.byref(n)))
        return out[: n.value].copy()

    # ---- CPU swap space ---------------------------------------------------
    def swap_space(self, num_host_blocks: int) -> None:
        """Gives the pool a host swap pool of num_host_blocks blocks in pinned
        host memory (allocator only on a host-only pool)."""
        import torch
        self.num_host_blocks = num_host_blocks
        if self.host_only:
            _abi.check(self.lib.pkv_swap_space_create(self._h, num_host_blocks, None, None, None, None))
            return
        shape = (num_host_blocks, self.n_kv_heads, BLOCK_SIZE, self.head_dim)
        self.host_k = torch.empty(shape, dtype=self.k_pool.dtype, pin_memory=True)
        self.host_v = torch.empty(shape, dtype=self.k_pool.dtype, pin_memory=True)
        if self.k_scale is not None:
            self.host_k_scale = torch.empty(shape[:3], dtype=torch.float32, pin_memory=True)
            self.host_v_scale = torch.empty(shape[:3], dtype=torch.float32, pin_memory=True)
        else:
            self.host_k_scale = self.host_v_scale = None
        with torch.cuda.device(self.device):
            _abi.check(self.lib.pkv_swap_space_create(
                self._h, num_host_blocks, self.host_k.data_ptr(), self.host_v.data_ptr(),
                self.host_k_scale.data_ptr() if self.host_k_scale is not None else None,
                self.host_v_scale.data_ptr() if self.host_v_scale is not None else None))

    def swap_out(self, seq_ids, stream=None) -> None:
        ids = _i32_array(seq_ids)
        _abi.check(self.lib.pkv_swap_out(self._h, None if self.host_only else _stream_ptr(stream), ids.size,
                                         _ptr(ids)))

    def swap_in(self, seq_ids, stream=None) -> None:
        ids = _i32_array(seq_ids)
        _abi.check(self.lib.pkv_swap_in(self._h, None if self.host_only else _stream_ptr(stream), ids.size,
                                        _ptr(ids)))

    def swapped(self, seq: int) -> bool:
        v = ctypes.c_int32()
        _abi.check(self.lib.pkv_seq_swapped(self._h, seq, ctypes.byref(v)))
        return bool(v.value)

    def host_block_table(self, seq: int) -> np.ndarray:
        out = np.empty(self.max_blocks_per_seq, dtype=np.int32)
        n = ctypes.c_int32()
        _abi.check(self.lib.pkv_get_host_block_table(self._h, seq, _ptr(out), out.size, ctypes.byref(n)))
        return out[: n.value].copy()

    def host_free_blocks(self) -> int:
        v = ctypes.c_int64()
        _abi.check(self.lib.pkv_host_free_blocks(self._h, ctypes.byref(v)))
        return int(v.value)

    def stats(self) -> dict:
        st = _abi.pkv_stats()
        _abi.check(self.lib.pkv_pool_stats(self._h, ctypes.byref(st)))
        return {f: getattr(st, f) for f, _ in st._fields_}

    def reserve_slots(self, seq_ids, T: int):
        ids = _i32_array(seq_ids)
        slots = np.empty(max(ids.size * T, 1), dtype=np.int64)
        cap = max(ids.size * T, 1)
        cow = np.empty((cap, 2), dtype=np.int32)
        ncow = ctypes.c_int32()
        _abi.check(self.lib.pkv_reserve_slots(self._h, ids.size, _ptr(ids), T, _ptr(slots), _ptr(cow), cap,
                                              ctypes.byref(ncow)))
        return slots[: ids.size * T].copy(), cow[: ncow.value].copy()

    # ---- device work ------------------------------------------------------
    def append(self, seq_ids, k_new, v_new, stream=None) -> None:
        """k_new, v_new: device tensors [n][T][n_kv_heads][head_dim]."""
        ids = _i32_array(seq_ids)
        T = int(k_new.shape[1]) if k_new.dim() == 4 else 1
        assert k_new.is_contiguous() and v_new.is_contiguous()
        _abi.check(self.lib.pkv_append(self._h, _stream_ptr(stream), ids.size, _ptr(ids), T, k_new.data_ptr(),
                                       v_new.data_ptr()))

    def workspace_bytes(self, n_seqs: int, num_splits: int = 0) -> int:
        b = ctypes.c_size_t()
        _abi.check(self.lib.pkv_decode_workspace_size(self._h, n_seqs, num_splits, ctypes.byref(b)))
        return b.value

    def workspace(self, n_seqs: int, num_splits: int = 0):
        import torch
        need = max(self.workspace_bytes(n_seqs, num_splits), 16)
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._workspace

    def decode(self, seq_ids, q, scale: float | None = None, mask: str = "full", num_sinks: int = 0,
               window: int = 0, num_splits: int = 0, out=None, lse=None, logits=None, logits_stride: int = 0,
               workspace=None, stream=None):
        """Decode attention; returns (out, lse).  q: [n][n_heads][head_dim]."""
        import torch
        ids = _i32_array(seq_ids)
        n = ids.size
        if scale is None:
            scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((n, self.n_heads), dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(n, num_splits)
        _abi.check(self.lib.pkv_decode_attn(
            self._h, _stream_ptr(stream), n, _ptr(ids), q.data_ptr(), float(scale), MASKS[mask], num_sinks, window,
            num_splits, out.data_ptr(), lse.data_ptr() if lse is not False else None,
            logits.data_ptr() if logits is not None else None, int(logits_stride),
            ws.data_ptr() if ws is not None else None, ws.numel() * ws.element_size() if ws is not None else 0))
        return out, lse

    def decode_static(self, seq_ids, q, scale: float | None = None, mask: str = "full", num_sinks: int = 0,
                      window: int = 0, num_splits: int = 0, out=None, lse=None, logits=None, logits_stride: int = 0,
                      stream=None):
        """pkv_decode_attn_static: decode whose scratch is the library's fixed
        device array (no workspace argument); returns (out, lse)."""
        import torch
        ids = _i32_array(seq_ids)
        if scale is None:
            scale = 1.0 / math.sqrt(self.head_dim)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((ids.size, self.n_heads), dtype=torch.float32, device=q.device)
        _abi.check(self.lib.pkv_decode_attn_static(
            self._h, _stream_ptr(stream), ids.size, _ptr(ids), q.data_ptr(), float(scale), MASKS[mask], num_sinks,
            window, num_splits, out.data_ptr(), lse.data_ptr(), logits.data_ptr() if logits is not None else None,
            int(logits_stride)))
        return out, lse

    def h2o_scores(self, seq_ids, logits, logits_stride: int, lse, acc, acc_stride: int, mask: str = "full",
                   num_sinks: int = 0, window: int = 0, stream=None) -> None:
        ids = _i32_array(seq_ids)
        _abi.check(self.lib.pkv_h2o_scores(self._h, _stream_ptr(stream), ids.size, _ptr(ids), logits.data_ptr(),
                                           int(logits_stride), lse.data_ptr(), MASKS[mask], num_sinks, window,
                                           acc.data_ptr(), int(acc_stride)))

    def h2o_select(self, seq_ids, acc, acc_stride: int, budget: int, recent: int, keep_idx, keep_stride: int,
                   keep_count, stream=None) -> None:
        """H2O keep-sets of the listed sequences (lengths from the pool); acc
        row i belongs to seq_ids[i]."""
        ids = _i32_array(seq_ids)
        _abi.check(self.lib.pkv_h2o_select(self._h, _stream_ptr(stream), ids.size, _ptr(ids), acc.data_ptr(),
                                           int(acc_stride), budget, recent, keep_idx.data_ptr(), int(keep_stride),
                                           keep_count.data_ptr()))

    def policy_select(self, seq_ids, acc, acc_stride: int, sink_size: int, window_size: int, h2o_size: int, keep_idx,
                      keep_stride: int, keep_count, stream=None) -> None:
        """Combined keep rule: first sink_size positions, last window_size,
        and the h2o_size highest scores over all positions (lengths from the
        pool; acc row i belongs to seq_ids[i])."""
        ids = _i32_array(seq_ids)
        _abi.check(self.lib.pkv_policy_select(self._h, _stream_ptr(stream), ids.size, _ptr(ids), acc.data_ptr(),
                                              int(acc_stride), sink_size, window_size, h2o_size, keep_idx.data_ptr(),
                                              int(keep_stride), keep_count.data_ptr()))

    def set_channel_scales(self, k_channel=None, v_channel=None) -> None:
        """Per-channel scales (FP8 / INT8 pools): device fp32 tensors
        [n_kv_heads][head_dim] for K and V, or None for both.  Set while the
        pool holds no token; the pool keeps references to them."""
        if k_channel is not None:
            assert k_channel.is_contiguous() and v_channel.is_contiguous()
        self._channel = (k_channel, v_channel)
        _abi.check(self.lib.pkv_set_channel_scales(
            self._h, k_channel.data_ptr() if k_channel is not None else None,
            v_channel.data_ptr() if v_channel is not None else None))

    def set_cascade(self, mode) -> None:
        """Shared-prefix decode: 0 / False off, 1 / True sequence pairs (the
        default), 2 group prefixes through the multi-query kernel."""
        mode = 1 if mode is True else 0 if mode is False else int(mode)
        _abi.check(self.lib.pkv_set_cascade(self._h, mode))

    def seq_compact(self, seq_ids, counts, keep_idx=None, keep_stride: int = 0, acc=None, acc_stride: int = 0,
                    stream=None) -> None:
        """H2O compaction: keep_idx device [n][keep_stride] int32 (ascending
        positions), counts host; acc optional device scores to compact."""
        ids, cnt = _i32_array(seq_ids), _i32_array(counts)
        _abi.check(self.lib.pkv_seq_compact(
            self._h, None if self.host_only else _stream_ptr(stream), ids.size, _ptr(ids),
            keep_idx.data_ptr() if keep_idx is not None else None, int(keep_stride), _ptr(cnt),
            acc.data_ptr() if acc is not None else None, int(acc_stride)))

    def sync_status(self, stream=None) -> None:
        _abi.check(self.lib.pkv_sync_status(self._h, _stream_ptr(stream)))

    # ---- measurement ------------------------------------------------------
    def timing_enable(self, on=True) -> None:
        """on: True (every kernel), False, or an iterable of kernel names."""
        if on is True:
            mask = -1
        elif not on:
            mask = 0
        else:
            mask = 0
            for name in on:
                mask |= 1 << KERNELS.index(name)
        _abi.check(self.lib.pkv_timing_enable(self._h, mask))

    def timing_read(self) -> dict:
        ms = np.zeros(len(KERNELS), dtype=np.float64)
        cnt = np.zeros(len(KERNELS), dtype=np.int64)
        _abi.check(self.lib.pkv_timing_read(self._h, _ptr(ms), _ptr(cnt)))
        return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNELS)}

    def launch_count(self) -> int:
        n = ctypes.c_int64()
        _abi.check(self.lib.pkv_launch_count(self._h, ctypes.byref(n)))
        return n.value
