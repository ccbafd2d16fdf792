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

KV_CODE = {"fp32": oracle.KV_FP32, "bf16": oracle.KV_BF16, "fp8": oracle.KV_FP8, "int8": oracle.KV_INT8}
MASK_CODE = {"full": oracle.MASK_FULL, "sliding": oracle.MASK_SLIDING, "sink_window": oracle.MASK_SINK_WINDOW}
TOL = {"fp32": 1e-4, "bf16": 1e-2, "fp8": 2e-2, "int8": 2e-2}  # max abs error on N(0,1) inputs
# Accumulated H2O scores against the oracle's fp64 ones: relative error.  Each
# term exp(s - lse) is evaluated from fp32 logits and lse, whose absolute
# errors (a few ulp of |s| and |lse|, below 1e-6 for the unit-scale logits of
# these inputs) become the term's relative error, as does the rounding of its
# exponent (about |s - lse| 2^-24, taken base 2) and the exponential's own
# (about 2^-22 relative): a few 1e-6 at most.
H2O_RTOL = 1e-5


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

    def set_channel_scales(self, k_channel: np.ndarray, v_channel: np.ndarray) -> None:
        """Per-channel scales [Hk][D] on both sides (before any token)."""
        self.cache.set_channel_scales(torch.from_numpy(np.ascontiguousarray(k_channel, np.float32)).to(self.dev),
                                      torch.from_numpy(np.ascontiguousarray(v_channel, np.float32)).to(self.dev))
        self.pool.set_channel_scales(k_channel, v_channel)

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

    def compact(self, seq_ids, keeps, acc=None, acc_stride: int = 0):
        """H2O compaction on both sides: keeps[i] (ascending positions) become
        sequence seq_ids[i]'s whole contents.  The oracle moves the same rows
        through its own allocator and row copy."""
        seq_ids = list(seq_ids)
        counts = [len(k) for k in keeps]
        stride = max([1] + counts)
        kd = torch.full((len(seq_ids), stride), -1, dtype=torch.int32)
        for i, k in enumerate(keeps):
            kd[i, : len(k)] = torch.as_tensor(np.asarray(k, dtype=np.int32))
        self.cache.seq_compact(seq_ids, counts, kd.to(self.dev), stride, acc, acc_stride)
        src = []
        for s, k in zip(seq_ids, keeps):
            t = self.alloc.table(s)
            src += [int(t[p // 16]) * 16 + p % 16 for p in k]
        fresh = self.alloc.compact(seq_ids, counts)
        dst = [int(f[i // 16]) * 16 + i % 16 for f, c in zip(fresh, counts) for i in range(c)]
        self.pool.copy_rows(src, dst)
        return fresh

    def swap_space(self, num_host_blocks: int) -> None:
        self.cache.swap_space(num_host_blocks)
        self.alloc.set_swap_space(num_host_blocks)
        self.pool.add_host_pool(num_host_blocks)

    def swap_out(self, seq_ids) -> np.ndarray:
        self.cache.swap_out(list(seq_ids))
        pairs = self.alloc.swap_out(list(seq_ids))
        self.pool.swap_copy(pairs, out=True)
        return pairs

    def swap_in(self, seq_ids) -> np.ndarray:
        self.cache.swap_in(list(seq_ids))
        pairs = self.alloc.swap_in(list(seq_ids))
        self.pool.swap_copy(pairs, out=False)
        return pairs

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


def length_only_pool(lens, device="cuda"):
    """A device pool whose sequences have the given lengths, placed by the
    allocator alone (no K/V written): for the calls that read only lengths,
    such as the keep-set selections.  Returns (cache, seq_ids)."""
    nb = sum((L + 15) // 16 for L in lens) + 1
    maxb = max([(L + 15) // 16 for L in lens] + [1])
    cache = PagedKVCache(nb, 1, 1, 64, len(lens), maxb, kv_dtype="bf16", device=torch.device(device))
    ids = []
    for L in lens:
        s = cache.seq_add()
        ids.append(s)
        if L:
            cache.reserve_slots([s], L)
    return cache, ids


def dequantised(tw: "Twin", which: str) -> np.ndarray:
    """The oracle pool's K or V as float64 [NB][Hk][16][D] (codes times
    token and channel scales for FP8 / INT8; unwritten slots may hold
    anything)."""
    x = tw.pool.k if which == "k" else tw.pool.v
    sc = tw.pool.k_scale if which == "k" else tw.pool.v_scale
    ch = tw.pool.k_channel if which == "k" else tw.pool.v_channel
    ch = 1.0 if ch is None else ch.astype(np.float64)[None, :, None, :]  # per-channel scales [Hk][D]
    if tw.wl.kv_dtype == "fp8":
        table = np.array([oracle.e4m3_decode(c) for c in range(256)], dtype=np.float64)
        return table[x] * sc[..., None] * ch
    if tw.wl.kv_dtype == "int8":
        return x.astype(np.float64) * sc[..., None] * ch
    if tw.wl.kv_dtype == "bf16":
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    return x.astype(np.float64)


def output_bounds(tw: "Twin", ids, q: torch.Tensor, logits: np.ndarray, lse: np.ndarray, rel: float) -> np.ndarray:
    """Error bound of every output row [n][H] against the fp64 oracle:
    sum_j p_j max_d |V_j| (rel + expm1(e_j + ebar)) over the kept keys j,
    with p the oracle's softmax weights exp(logit - lse) and ebar =
    sum_k p_k e_k.  rel covers the roundings of the weights and of the
    output; e_j = 2^-18 (1 + scale sum_d |q_d K_jd|) bounds the error of
    logit j, an fp32 sum of exact products, which grows with the logit's
    magnitude.  Errors e_k in the logits move weight j by a factor within
    exp(+-(e_j + ebar)) (its own term and the normalisation's)."""
    G, scale = tw.wl.group, tw.wl.scale
    r = 2.0 ** -18
    K = dequantised(tw, "k")
    vmax = np.nan_to_num(np.abs(dequantised(tw, "v")).max(axis=-1), nan=0.0, posinf=0.0)
    qa = np.abs(q.double().numpy())
    out = np.zeros(lse.shape)
    for b, s in enumerate(ids):
        L = tw.alloc.length(s)
        if L == 0:
            continue
        pos = np.arange(L)
        blk = tw.alloc.table(s)[pos // 16]
        for h in range(lse.shape[1]):
            lg = logits[b, h, :L]
            kept = ~np.isnan(lg)
            if not kept.any():
                continue
            g = h // G
            k_abs = np.abs(K[blk[kept], g, pos[kept] % 16])  # [kept][D]
            e = r * (1.0 + scale * (k_abs @ qa[b, h]))
            p = np.exp(lg[kept] - lse[b, h])
            ebar = float((p * e).sum())
            out[b, h] = float((p * vmax[blk[kept], g, pos[kept] % 16] * (rel + np.expm1(e + ebar))).sum())
    return out


def max_err(a: torch.Tensor, b: np.ndarray) -> float:
    return float(np.abs(a.float().cpu().numpy().astype(np.float64) - b).max()) if b.size else 0.0


def lse_err(a: torch.Tensor, b: np.ndarray) -> float:
    x = a.cpu().numpy().astype(np.float64)
    both_inf = np.isneginf(x) & np.isneginf(b)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(x - b))
    return float(d.max()) if d.size else 0.0


def pool_bytes_equal(tw: Twin, ids, every: int = 1):
    """K/V bytes (and FP8 scales) of written slots equal the oracle's, for
    every `every`-th block of each sequence."""
    c = tw.cache
    NB, Hk = tw.pool.NB, tw.wl.n_kv_heads
    pairs = [(c.k_pool, tw.pool.k), (c.v_pool, tw.pool.v)]
    if tw.wl.kv_dtype in ("fp8", "int8"):
        pairs += [(c.k_scale, tw.pool.k_scale), (c.v_scale, tw.pool.v_scale)]
    for dt, ht in pairs:
        d = dt.view(torch.uint8).reshape(NB, Hk, 16, -1) if dt.dtype != torch.uint8 else dt.reshape(NB, Hk, 16, -1)
        h = ht.view(np.uint8).reshape(NB, Hk, 16, -1)
        for s in ids:
            L = tw.alloc.length(s)
            t = tw.alloc.table(s)
            sel = [lb for lb in range(0, len(t), every) if t[lb] >= 0]
            if not sel:
                continue
            blks = torch.tensor([int(t[lb]) for lb in sel], dtype=torch.long, device=d.device)
            got = d.index_select(0, blks).cpu().numpy()
            for i, lb in enumerate(sel):
                n = min(16, L - 16 * lb)
                assert np.array_equal(got[i, :, :n], h[t[lb], :, :n]), (s, lb, int(t[lb]))


def build_streaming(wl: workloads.Workload, device="cuda", chunk: int = 4096):
    """Sequences of logical length L that hold only the blocks intersecting
    the sink + window keep-set: block 0 and the window are real seeded data,
    the middle is zero filler appended in chunks and evicted as it leaves the
    window (the oracle replays the same operations; filler is not mirrored)."""
    S, W = wl.num_sinks, wl.window
    per_seq = 1 + (W + 15) // 16 + 2 + chunk // 16 + 2
    maxb = max((L + 15) // 16 for L in wl.lens) + 4
    tw = Twin(wl, len(wl.lens) * per_seq + 64, len(wl.lens), maxb, seed=wl.seed, device=device)
    zc = torch.zeros((1, chunk, wl.n_kv_heads, wl.head_dim), dtype=torch.bfloat16)
    zd = zc.to(tw.dev)
    ids = []
    for b, L in enumerate(wl.lens):
        s = tw.add()
        ids.append(s)
        tail = (L - W) // 16 * 16 if L > S + W else 0
        if tail < 32:
            k, v = workloads.kv_rows(wl, b, 0, L)
            tw.append([s], k[None], v[None])
            continue
        k, v = workloads.kv_rows(wl, b, 0, 16)
        tw.append([s], k[None], v[None])
        pos = 16
        while pos < tail:
            n = min(chunk, tail - pos)
            tw.append([s], zc[:, :n], zc[:, :n], k_dev=zd[:, :n], v_dev=zd[:, :n], mirror=False)
            pos += n
            tw.evict(s, S, W)
        k, v = workloads.kv_rows(wl, b, tail, L - tail)
        tw.append([s], k[None], v[None])
        tw.evict(s, S, W)
    return tw, ids


def build_prefix(wl: workloads.Workload, device="cuda", fork_parents: bool = True):
    """Groups sharing a 2048-token prefix through refcounted blocks; each
    parent adds a private suffix and (by default) is forked once."""
    ex = wl.extra
    groups, ppg, prefix = ex["groups"], ex["parents_per_group"], ex["prefix"]
    need = groups * (prefix // 16) + sum((s + 15) // 16 + 1 for s in ex["suffix"]) * 2 + 64
    maxb = max((L + 15) // 16 for L in wl.lens) + 4
    tw = Twin(wl, need, 2 * groups * ppg + groups, maxb, seed=wl.seed, device=device)
    parents = []
    for gi in range(groups):
        holder = tw.add()
        k, v = workloads.kv_rows(wl, 10_000 + gi, 0, prefix)
        tw.append([holder], k[None], v[None])
        kids = [tw.fork(holder) for _ in range(ppg)]
        tw.free(holder)
        for j, s in enumerate(kids):
            pidx = gi * ppg + j
            k, v = workloads.kv_rows(wl, pidx, prefix, ex["suffix"][pidx])
            tw.append([s], k[None], v[None])
        parents += kids
    ids = sorted(parents + [tw.fork(p) for p in parents]) if fork_parents else sorted(parents)
    return tw, ids
