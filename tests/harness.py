"""Builds the same paged cache twice -- in libpkv on the GPU and in the CPU
oracle -- from the same seeded inputs and the same sequence of allocator
operations.  Nothing here computes the method: it only replays operations
and moves bytes."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads
from paged_kv_cache_282_gb300 import PagedKVCache

KV_CODE = {"fp32": oracle.KV_FP32, "bf16": oracle.KV_BF16, "fp8": oracle.KV_FP8}
MASK_CODE = {"full": oracle.MASK_FULL, "sliding": oracle.MASK_SLIDING, "sink_window": oracle.MASK_SINK_WINDOW}
TOL = {"fp32": 1e-4, "bf16": 1e-2, "fp8": 2e-2}  # max abs error on N(0,1) inputs


class Twin:
    """A libpkv pool and an oracle pool kept in step."""

    def __init__(self, wl: workloads.Workload, num_blocks: int, max_seqs: int, max_blocks: int, seed: int = 0,
                 free_order=None, device="cuda"):
        self.wl = wl
        self.dev = torch.device(device)
        self.cache = PagedKVCache(num_blocks, wl.n_heads, wl.n_kv_heads, wl.head_dim, max_seqs, max_blocks,
                                  kv_dtype=wl.kv_dtype, alloc_seed=seed, free_order=free_order, device=self.dev)
        self.alloc = oracle.OracleAllocator(num_blocks, max_seqs, max_blocks, seed=seed, order=free_order)
        self.pool = oracle.OraclePool(num_blocks, wl.n_kv_heads, wl.head_dim, KV_CODE[wl.kv_dtype])

    def add(self) -> int:
        a, b = self.cache.seq_add(), self.alloc.seq_add()
        assert a == b
        return a

    def fork(self, s: int) -> int:
        a, b = self.cache.seq_fork(s), self.alloc.fork(s)
        assert a == b
        return a

    def free(self, s: int) -> None:
        self.cache.seq_free(s)
        self.alloc.free(s)

    def evict(self, s: int, S: int, W: int) -> None:
        self.cache.seq_evict(s, S, W)
        self.alloc.evict(s, S, W)

    def truncate(self, s: int, n: int) -> None:
        self.cache.seq_truncate(s, n)
        self.alloc.truncate(s, n)

    def append(self, seq_ids, k: torch.Tensor, v: torch.Tensor, k_dev=None, v_dev=None, mirror: bool = True):
        """k, v: CPU [n][T][Hk][D] of the input dtype (mirrored into the oracle
        pool); k_dev / v_dev: the same data already on the device (optional)."""
        T = k.shape[1]
        kd = k_dev if k_dev is not None else k.to(self.dev)
        vd = v_dev if v_dev is not None else v.to(self.dev)
        self.cache.append(list(seq_ids), kd.contiguous(), vd.contiguous())
        slots, cow = self.alloc.append(list(seq_ids), T)
        for src, dst in cow:
            self.pool.copy_block(int(src), int(dst))
        if mirror:
            self.pool.write(slots, workloads.as_bits(k.reshape(-1, *k.shape[2:])),
                            workloads.as_bits(v.reshape(-1, *v.shape[2:])))
        return slots, cow

    def tables(self, seq_ids) -> np.ndarray:
        return self.alloc.tables_matrix(list(seq_ids))

    def oracle_decode(self, seq_ids, q: torch.Tensor, mask="full", S=0, W=0, want_logits=False, logits_stride=None):
        lens = [self.alloc.length(s) for s in seq_ids]
        qdt = oracle.KV_FP32 if self.wl.kv_dtype == "fp32" else oracle.KV_BF16
        return oracle.decode(self.pool, self.tables(seq_ids), lens, workloads.as_bits(q), qdt, self.wl.n_heads,
                             self.wl.scale, MASK_CODE[mask], S, W, want_logits=want_logits,
                             logits_stride=logits_stride)


def fill_sequences(tw: Twin, lens, data_keys=None, chunk: int = 8192):
    """Adds one sequence per length and appends its seeded K/V rows."""
    ids = []
    for b, L in enumerate(lens):
        s = tw.add()
        ids.append(s)
        key = b if data_keys is None else data_keys[b]
        for t0 in range(0, L, chunk):
            n = min(chunk, L - t0)
            k, v = workloads.kv_rows(tw.wl, key, t0, n)
            tw.append([s], k[None], v[None])
    return ids


def max_err(a: torch.Tensor, b: np.ndarray) -> float:
    return float(np.abs(a.float().cpu().numpy().astype(np.float64) - b).max()) if b.size else 0.0


def lse_err(a: torch.Tensor, b: np.ndarray) -> float:
    x = a.cpu().numpy().astype(np.float64)
    both_inf = np.isneginf(x) & np.isneginf(b)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(x - b))
    return float(d.max()) if d.size else 0.0
