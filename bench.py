"""Benchmark: paged decode attention on GB300 (one layer, one decode step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pkv|reference]

A step is one pass of the hot path over one batch: the allocator places one
new token per sequence and the append kernel scatters its K/V (plus the
copy-on-write copies when a shared block is written), then decode attention
runs over every sequence's full context (decode kernel + log-sum-exp combine;
H2O score and keep-set selection too on the streaming workload).  After each
step the appended token is rolled back on the host (the block table is
truncated), so every timed step sees the same context lengths.

Metric: algorithmic KV bytes read per second (each kept token's K and V bytes
per (sequence, kv head) once, plus FP8 / INT8 scales; a physical block shared
by several sequences counts once) and decode tokens per second
(sequences / step time).  Inputs stay resident in HBM; the KV pool of the
default workload (~1.1 GB) is far larger than L2, so no flush is needed.

With --gpus N under torchrun every rank runs its own replica of the workload
on its own GPU (no collective on the data path); the line reports the sum
over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode KV GB/s (frac of HBM peak) and tokens/s, 1×GB300"
FALLBACK_HBM_GBS = 6800.0
BYTES = {"fp32": 4, "bf16": 2, "fp8": 1, "int8": 1}


# --------------------------------------------------------------------------
# workload setup on the device
# --------------------------------------------------------------------------

def _kv_bytes_per_token(wl) -> int:
    b = 2 * wl.n_kv_heads * wl.head_dim * BYTES[wl.kv_dtype]
    if wl.kv_dtype in ("fp8", "int8"):
        b += 2 * wl.n_kv_heads * 4  # per-token K and V scales
    return b


def _kept(L, wl) -> int:
    if wl.mask == "sliding":
        return min(L, wl.window + 1)
    if wl.mask == "sink_window" and L > wl.num_sinks + wl.window:
        return wl.num_sinks + wl.window
    return L


class Setup:
    """Pool + sequences of one workload on one GPU, filled from the seeded
    generator through the library's own append path."""

    def __init__(self, wl, dev, headroom_blocks: int | None = None, extra_seqs: int = 0, channel_scales=False):
        from paged_kv_cache_282_gb300 import PagedKVCache
        self.wl, self.dev = wl, dev
        self.channel_scales = channel_scales
        self.extra = {}
        self.extra_seqs = extra_seqs  # sequence ids left free (forks of the workload's sequences)
        name = wl.name
        if name == "prefix_append":
            self._setup_prefix(PagedKVCache)
        elif name == "streaming_h2o":
            self._setup_streaming(PagedKVCache)
        else:
            lens = list(wl.lens)
            need = sum((L + 15) // 16 for L in lens)
            hb = headroom_blocks if headroom_blocks is not None else len(lens) + 8
            maxb = max((L + 15) // 16 for L in lens) + 4
            self.cache = PagedKVCache(need + hb, wl.n_heads, wl.n_kv_heads, wl.head_dim, len(lens), maxb,
                                      kv_dtype=wl.kv_dtype, alloc_seed=wl.seed, device=dev)
            self._set_channel_scales()
            self.ids = []
            for b, L in enumerate(lens):
                s = self.cache.seq_add()
                self.ids.append(s)
                for t0 in range(0, L, 16384):
                    n = min(16384, L - t0)
                    k, v = workloads.kv_rows(wl, b, t0, n)
                    self.cache.append([s], k[None].to(dev), v[None].to(dev))
        torch.cuda.synchronize(dev)
        self.lens = [self.cache.seq_len(s) for s in self.ids]

    def _set_channel_scales(self):
        """Per-channel scales (FP8 / INT8 pools, when asked for): seeded powers
        of two 2^-2 .. 2^2 per (kv head, channel), standing in for calibrated
        ones."""
        if not self.channel_scales:
            return
        wl = self.wl
        g = torch.Generator().manual_seed(wl.seed + 7)
        kc, vc = (2.0 ** torch.randint(-2, 3, (wl.n_kv_heads, wl.head_dim), generator=g).float() for _ in range(2))
        self.k_channel, self.v_channel = kc.to(self.dev), vc.to(self.dev)
        self.cache.set_channel_scales(self.k_channel, self.v_channel)

    def _setup_prefix(self, PagedKVCache):
        wl = self.wl
        ex = wl.extra
        groups, ppg, prefix = ex["groups"], ex["parents_per_group"], ex["prefix"]
        need = groups * (prefix // 16) + sum((s + 15) // 16 + 1 for s in ex["suffix"]) * 2 + 64
        maxb = max((L + 15) // 16 for L in wl.lens) + 4
        n_seqs = 2 * groups * ppg + groups
        self.cache = c = PagedKVCache(need, wl.n_heads, wl.n_kv_heads, wl.head_dim, n_seqs, maxb,
                                      kv_dtype=wl.kv_dtype, alloc_seed=wl.seed, device=self.dev)
        parents = []
        for gi in range(groups):
            holder = c.seq_add()
            k, v = workloads.kv_rows(wl, 10_000 + gi, 0, prefix)
            c.append([holder], k[None].to(self.dev), v[None].to(self.dev))
            kids = [c.seq_fork(holder) for _ in range(ppg)]
            c.seq_free(holder)
            for j, s in enumerate(kids):
                pidx = gi * ppg + j
                k, v = workloads.kv_rows(wl, pidx, prefix, ex["suffix"][pidx])
                c.append([s], k[None].to(self.dev), v[None].to(self.dev))
            parents += kids
        self.ids = sorted(parents + [c.seq_fork(p) for p in parents])

    def _setup_streaming(self, PagedKVCache):
        """Sequences of logical length L hold only the blocks that intersect
        the sink + window keep-set: the middle is appended as zero filler in
        chunks and evicted as it falls out of the window."""
        wl = self.wl
        S, W = wl.num_sinks, wl.window
        chunk = 4096
        per_seq = 1 + (W + 15) // 16 + 2 + chunk // 16 + 2
        maxb = max((L + 15) // 16 for L in wl.lens) + 4
        self.cache = c = PagedKVCache(len(wl.lens) * per_seq + 64, wl.n_heads, wl.n_kv_heads, wl.head_dim,
                                      len(wl.lens) + self.extra_seqs, maxb, kv_dtype=wl.kv_dtype,
                                      alloc_seed=wl.seed, device=self.dev)
        zeros = torch.zeros((1, chunk, wl.n_kv_heads, wl.head_dim), dtype=torch.bfloat16, device=self.dev)
        self.ids = []
        for b, L in enumerate(wl.lens):
            s = c.seq_add()
            self.ids.append(s)
            # first position of the first block that intersects the window
            tail = (L - W) // 16 * 16 if L > S + W else 0
            if tail < 32:  # the window reaches block 0 or 1: everything is real
                k, v = workloads.kv_rows(wl, b, 0, L)
                c.append([s], k[None].to(self.dev), v[None].to(self.dev))
                continue
            k, v = workloads.kv_rows(wl, b, 0, 16)  # block 0 holds the sinks
            c.append([s], k[None].to(self.dev), v[None].to(self.dev))
            pos = 16
            while pos < tail:
                n = min(chunk, tail - pos)
                c.append([s], zeros[:, :n], zeros[:, :n])
                pos += n
                c.seq_evict(s, S, W)
            k, v = workloads.kv_rows(wl, b, tail, L - tail)
            c.append([s], k[None].to(self.dev), v[None].to(self.dev))
            c.seq_evict(s, S, W)

    def algorithmic_bytes(self, lens=None) -> int:
        lens = self.lens if lens is None else lens
        return sum(_kept(L, self.wl) for L in lens) * _kv_bytes_per_token(self.wl)

    def kv_bytes_read_per_step(self) -> int:
        """KV bytes one step must read: each sequence's kept tokens, except
        that a physical block shared by several sequences counts once."""
        if self.wl.name != "prefix_append":
            return self.algorithmic_bytes([L + 1 for L in self.lens])
        return self.unique_bytes_per_step()

    def unique_bytes_per_step(self) -> int:
        """KV bytes of distinct physical blocks the step reads (blocks shared
        by several sequences count once), plus each sequence's new token."""
        fill = {}
        for s, L in zip(self.ids, self.lens):
            for lb, blk in enumerate(self.cache.block_table(s)):
                if blk >= 0:
                    fill[int(blk)] = max(fill.get(int(blk), 0), min(16, L - 16 * lb))
        return (sum(fill.values()) + len(self.ids)) * _kv_bytes_per_token(self.wl)


# --------------------------------------------------------------------------
# one step
# --------------------------------------------------------------------------

class Stepper:
    def __init__(self, setup: Setup, num_splits: int):
        wl, dev = setup.wl, setup.dev
        self.s, self.wl, self.dev = setup, wl, dev
        self.cache = setup.cache
        # int32 arrays once, so the per-step calls marshal nothing
        self.ids = np.asarray(setup.ids, dtype=np.int32)
        self.lens = np.asarray(setup.lens, dtype=np.int32)
        self.lens1 = self.lens + 1
        n = len(self.ids)
        self.num_splits = num_splits
        self.q = workloads.queries(wl, n).to(dev)
        k, v = workloads.new_tokens(wl, n, 0)
        self.k_new, self.v_new = k.to(dev), v.to(dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((n, wl.n_heads), dtype=torch.float32, device=dev)
        self.ws = self.cache.workspace(n, num_splits)
        self.h2o = wl.budget > 0
        if self.h2o:
            self.stride = max(setup.lens) + 1
            self.logits = torch.zeros((n, wl.n_kv_heads, self.stride, wl.group), dtype=torch.float32, device=dev)
            self.acc = torch.zeros((n, self.stride), dtype=torch.float32, device=dev)
            self.keep = torch.zeros((n, wl.budget), dtype=torch.int32, device=dev)
            self.keep_n = torch.zeros(n, dtype=torch.int32, device=dev)

    def step(self, q=None, k_new=None, v_new=None, out=None):
        c, wl = self.cache, self.wl
        c.append(self.ids, self.k_new if k_new is None else k_new, self.v_new if v_new is None else v_new)
        o = self.out if out is None else out
        if self.h2o:
            c.decode(self.ids, self.q if q is None else q, scale=wl.scale, mask=wl.mask, num_sinks=wl.num_sinks,
                     window=wl.window, num_splits=self.num_splits, out=o, lse=self.lse, logits=self.logits,
                     logits_stride=self.stride, workspace=self.ws)
            c.h2o_scores(self.ids, self.logits, self.stride, self.lse, self.acc, self.stride, mask=wl.mask,
                         num_sinks=wl.num_sinks, window=wl.window)
            c.h2o_select(self.ids, self.acc, self.stride, wl.budget, wl.recent, self.keep, wl.budget, self.keep_n)
        else:
            c.decode(self.ids, self.q if q is None else q, scale=wl.scale, mask=wl.mask, num_sinks=wl.num_sinks,
                     window=wl.window, num_splits=self.num_splits, out=o, lse=self.lse, workspace=self.ws)
        c.seq_truncate_many(self.ids, self.lens)  # roll the appended token back (host only)


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def _stats(rows):
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower().startswith("active")})
        return sm, mx, reasons

    def summary(self, t0, t1):
        """Clocks of the samples taken inside [t0, t1].  A region shorter than
        the sampling period may hold none: it is then reported as unsampled,
        with the samples just before and after it listed apart."""
        rows = [r for (t, r) in self.samples if t0 <= t <= t1]
        if not rows:
            before = [r for (t, r) in self.samples if t < t0][-1:]
            after = [r for (t, r) in self.samples if t > t1][:1]
            sm, mx, reasons = self._stats(before + after)
            return {"sm_mhz": None, "sm_max_mhz": max(mx) if mx else None, "reasons": ["unsampled"], "samples": 0,
                    "adjacent": {"sm_mhz": sm, "reasons": reasons}}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_HEADERS = ("async_copy.cuh", "pkv_internal.h")
DECODE_SOURCES = ("decode_tc.cuh",)


def kernel_source_sha(kernel_files=DECODE_SOURCES) -> str:
    """sha256 of the kernel's source files followed by the library headers
    they include."""
    csrc = os.path.join(ROOT, "paged_kv_cache_282_gb300", "csrc")
    h = hashlib.sha256()
    for name in tuple(kernel_files) + KERNEL_HEADERS:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel recorded from an ncu capture
    in profiles/, valid only while the kernel source is unchanged (its sha256,
    with the headers it includes, recorded beside it)."""
    path = os.path.join(ROOT, "profiles", f"decode_tc_{workload}.md")
    try:
        text = open(path).read()
        sha = kernel_source_sha()
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        if m_sha and m_tr and m_sha.group(1) == sha:
            return float(m_tr.group(1))
    except Exception:
        pass
    return None


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, dev) -> float:
    """Maximum of x over the ranks (the slowest rank's time)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    on_cpu = dist.get_backend() == "gloo"
    t = torch.tensor([x], dtype=torch.float64, device="cpu" if on_cpu else dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(ws: int, bytes_per_rank_step: int, ms_per_step_max: float) -> float:
    """GB/s of the whole job: every rank's bytes over the slowest rank's time."""
    return ws * bytes_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# --------------------------------------------------------------------------

def oracle_baseline(wl, n_sample: int, repeats: int = 1):
    import oracle
    lens = list(wl.lens)[:n_sample]
    nb = sum((L + 15) // 16 for L in lens)
    kvd = {"fp32": oracle.KV_FP32, "bf16": oracle.KV_BF16, "fp8": oracle.KV_FP8, "int8": oracle.KV_INT8}[wl.kv_dtype]
    alloc = oracle.OracleAllocator(nb, len(lens), max((L + 15) // 16 for L in lens) + 1, seed=wl.seed)
    pool = oracle.OraclePool(nb, wl.n_kv_heads, wl.head_dim, kvd)
    ids = []
    for b, L in enumerate(lens):
        s = alloc.seq_add()
        ids.append(s)
        k, v = workloads.kv_rows(wl, b, 0, L)
        slots, _ = alloc.append([s], L)
        pool.write(slots, workloads.as_bits(k), workloads.as_bits(v))
    q = workloads.as_bits(workloads.queries(wl, len(lens)))
    tables = alloc.tables_matrix(ids)
    qdt = oracle.KV_FP32 if wl.kv_dtype == "fp32" else oracle.KV_BF16
    masks = {"full": oracle.MASK_FULL, "sliding": oracle.MASK_SLIDING, "sink_window": oracle.MASK_SINK_WINDOW}
    cores = os.cpu_count() or 1
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        oracle.decode(pool, tables, lens, q, qdt, wl.n_heads, wl.scale, masks[wl.mask], wl.num_sinks, wl.window,
                      n_threads=cores)
        times.append(time.perf_counter() - t0)
    t = min(times)
    byts = sum(_kept(L, wl) for L in lens) * _kv_bytes_per_token(wl)
    return {"value": byts / t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(lens)} of {wl.batch} sequences of {wl.name} ({sum(lens)} tokens), fp64 oracle decode, "
                      f"{t:.2f} s", "seconds": t, "tokens_per_s": len(lens) / t}


# --------------------------------------------------------------------------
# main
# --------------------------------------------------------------------------

def measure(args, wl, label, splits, dev, ws, rank, cascade, headline=True):
    """Times one workload's decode step (the timed region, per-step spread,
    a sustained leg, end to end through host buffers) and returns its JSON
    fields (rank 0; None elsewhere or in profile mode)."""
    setup = Setup(wl, dev, channel_scales=args.channel_scales)
    setup.cache.set_cascade(cascade)
    st = Stepper(setup, splits)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        st.step()
    setup.cache.sync_status()
    if args.profile_steps:
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_push("profiled_steps")  # ncu --nvtx-include "profiled_steps/"
        for _ in range(args.profile_steps):
            st.step()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_steps": args.profile_steps, "workload": wl.name}))
        return None

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3)
    # ---- device-resident timed region (kernel timing events on) ----
    setup.cache.timing_enable(True if args.time_kernels else ["decode", "prefix_decode"])
    setup.cache.timing_read()
    launches0 = setup.cache.launch_count()
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        st.step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(ws)
    ms = e0.elapsed_time(e1)
    launches = setup.cache.launch_count() - launches0
    ktimes = setup.cache.timing_read()
    setup.cache.timing_enable(False)
    setup.cache.sync_status()
    ms_max = reduce_max(ms, ws, dev)

    # ---- sustained leg: the same step repeated for at least a second, in
    # chunks of steps bracketed by events (per-step median from the chunks),
    # with its own clock record
    sus = None
    if not args.no_sustained:
        per = max(ms / max(args.steps, 1), 1e-3)
        chunk = max(1, int(math.ceil(2.0 / per)))  # about 2 ms per chunk
        n_chunks = max(20, int(math.ceil(args.sustain_s * 1e3 / (per * chunk))))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_chunks + 1)]
        barrier(ws)
        torch.cuda.synchronize(dev)
        s_wall0 = time.time()
        evs[0].record(stream)
        for i in range(n_chunks):
            for _ in range(chunk):
                st.step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        s_wall1 = time.time()
        barrier(ws)
        per_chunk = [evs[i].elapsed_time(evs[i + 1]) / chunk for i in range(n_chunks)]
        sus_ms = reduce_max(evs[0].elapsed_time(evs[-1]), ws, dev) / (n_chunks * chunk)
        sus = {"steps": n_chunks * chunk, "seconds": round(evs[0].elapsed_time(evs[-1]) * 1e-3, 3),
               "ms_per_step": round(sus_ms, 5), "ms_per_step_p50": round(statistics.median(per_chunk), 5),
               "sus_wall": (s_wall0, s_wall1)}
        setup.cache.sync_status()

    # ---- per-step spread (separate from the timed region): events around
    # each of up to 50 steps, for the median and the 10th / 90th percentiles
    pct = None
    if rank == 0:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(50, args.steps))]
        for a0, a1 in evs:
            a0.record(stream)
            st.step()
            a1.record(stream)
        torch.cuda.synchronize(dev)
        t = sorted(a0.elapsed_time(a1) for a0, a1 in evs)
        q = lambda f: round(t[min(len(t) - 1, int(f * len(t)))], 5)
        pct = {"steps": len(t), "p10": q(0.1), "p50": q(0.5), "p90": q(0.9)}

    # ---- end to end through host buffers ----
    # Every step copies its inputs (queries, new K/V) from pinned host memory
    # and its output back, as a serving loop does: double-buffered, uploads and
    # downloads on two copy streams, so that step i + 1's inputs upload and
    # step i's output downloads while the neighbouring step decodes.  The
    # timed region spans the first upload to the last download.
    e2e = None
    if not args.no_e2e:
        n = len(setup.ids)
        # a step's inputs (queries, new K, new V) packed in one buffer: one copy each way
        parts = (st.q, st.k_new, st.v_new)
        assert all(t.dtype == st.q.dtype for t in parts)
        sizes = [t.numel() for t in parts]

        def packed(pin):
            flat = torch.empty(sum(sizes), dtype=st.q.dtype, device="cpu" if pin else dev)
            if pin:
                flat = flat.pin_memory()
            views, off = [], 0
            for t, nel in zip(parts, sizes):
                views.append(flat[off:off + nel].view(t.shape))
                off += nel
            return flat, views

        in_h, (q_h, k_h, v_h) = packed(True)
        q_h.copy_(st.q.cpu())
        k_h.copy_(st.k_new.cpu())
        v_h.copy_(st.v_new.cpu())
        out_h = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(2)]
        bufs = []
        for _ in range(2):
            flat_d, (qd_, kd_, vd_) = packed(False)
            bufs.append((flat_d, qd_, kd_, vd_, torch.empty_like(st.out)))
        cs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)  # uploads, downloads
        fetched = [torch.cuda.Event() for _ in range(2)]
        loaded = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def upload(i):  # inputs of step i into buffer set i % 2, on the copy stream
            flat_d = bufs[i % 2][0]
            with torch.cuda.stream(cs):
                if i >= 2:
                    cs.wait_event(done[i % 2])  # step i - 2 read this set
                flat_d.copy_(in_h, non_blocking=True)
                loaded[i % 2].record(cs)

        def run(steps):
            upload(0)
            for i in range(steps):
                if i + 1 < steps:
                    upload(i + 1)
                _, qd, kd, vd, od = bufs[i % 2]
                stream.wait_event(loaded[i % 2])
                if i >= 2:
                    stream.wait_event(fetched[i % 2])  # step i - 2's output has left this buffer
                st.step(q=qd, k_new=kd, v_new=vd, out=od)
                done[i % 2].record(stream)
                with torch.cuda.stream(ds):
                    ds.wait_event(done[i % 2])
                    out_h[i % 2].copy_(od, non_blocking=True)
                    fetched[i % 2].record(ds)
            stream.wait_stream(cs)
            stream.wait_stream(ds)

        e2e_steps = max(10, args.steps // 4)
        run(3)
        barrier(ws)
        torch.cuda.synchronize(dev)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        cs.wait_stream(stream)
        ds.wait_stream(stream)
        run(e2e_steps)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        e2e_ms = reduce_max(a0.elapsed_time(a1), ws, dev) / e2e_steps
        bi = (q_h.numel() * q_h.element_size() + k_h.numel() * k_h.element_size() +
              v_h.numel() * v_h.element_size())
        bo = out_h[0].numel() * out_h[0].element_size()
        step_bytes = setup.kv_bytes_read_per_step()
        e2e = {"value": round(ws * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 5),
               "tokens_per_s": round(ws * n / (e2e_ms * 1e-3), 1)}

    if clocks:
        clocks.stop()
    if rank != 0:
        return None

    peak, peak_kind = hbm_peak()
    lens_step = [L + 1 for L in setup.lens]
    logical = setup.algorithmic_bytes(lens_step)
    step_bytes = setup.kv_bytes_read_per_step()
    ms_step = ms_max / args.steps
    value = whole_job_rate(ws, step_bytes, ms_step)
    # decode time per step: the main decode kernel plus, with shared-prefix
    # groups, the multi-query kernel that runs before it
    dec_ms, dec_n = ktimes["decode"]
    dec_ms += ktimes["prefix_decode"][0]
    dec_avg = dec_ms / max(dec_n, 1)
    achieved = step_bytes / (dec_avg * 1e-3) / 1e9 if dec_n else None
    # the captures in profiles/ ran with the default shared-prefix mode (1)
    traffic = profiled_traffic(label) if cascade == 1 else None
    decode_share = round(dec_ms / max(ms, 1e-9), 4)
    cpu = None
    if headline and not args.no_cpu_baseline and ws == 1:
        cpu = oracle_baseline(wl, min(args.cpu_sample, wl.batch))
    clk = clocks.summary(t_wall0, t_wall1) if clocks else None
    if sus is not None:
        w0, w1 = sus.pop("sus_wall")
        sus["value"] = round(whole_job_rate(ws, step_bytes, sus["ms_per_step"]), 2)
        sus["frac_of_hbm_peak"] = round(sus["value"] / ws / peak, 4)
        sus["clocks"] = clocks.summary(w0, w1) if clocks else None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_step, 5),
        "step_ms_percentiles": pct,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.kv_dtype,
        "data": "synthetic (seeded N(0,1) K/V/Q; seeded uniform lengths)",
        "config": {"workload": label, "batch": len(setup.ids), "n_heads": wl.n_heads,
                   "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "kv_dtype": wl.kv_dtype,
                   "channel_scales": bool(args.channel_scales),
                   "mask": wl.mask, "num_splits": splits, "cascade": cascade,
                   "context_tokens": sum(lens_step),
                   "kv_bytes_per_step": step_bytes, "l2": "KV pool larger than L2 (no flush needed)",
                   "parallelism": f"replicas x{ws}"},
        "tokens_per_s": round(ws * len(setup.ids) / (ms_step * 1e-3), 1),
        "frac_of_hbm_peak": round(value / ws / peak, 4),
        "roofline": {"bound": "hbm",
                     "kernel": "decode_tc_kernel" + (" + prefix_decode_kernel" if ktimes["prefix_decode"][1] else ""), "achieved": round(achieved, 2) if achieved else None,
                     "peak": peak, "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
                     "frac": round(achieved / peak, 4) if achieved else None, "traffic": traffic,
                     "algorithmic_bytes_per_launch": step_bytes, "avg_launch_ms": round(dec_avg, 5)},
        "decode_share_of_step": decode_share,
        "kernel_ms_per_step": {k: round(v[0] / args.steps, 5) for k, v in ktimes.items() if v[1]}
        if args.time_kernels else None,
        "logical_kv_bytes_per_step": logical if logical != step_bytes else None,
        "value_logical_gbs": round(ws * logical / (ms_step * 1e-3) / 1e9, 2) if logical != step_bytes else None,
        "gpu_launches": launches,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clk,
        "sustained": sus,
    }
    if not headline:
        keep = ("value", "unit", "ms_per_step", "step_ms_percentiles", "dtype", "config", "tokens_per_s",
                "frac_of_hbm_peak", "roofline", "gpu_launches", "e2e", "clocks", "sustained")
        line = {k: line[k] for k in keep}
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="llama3_8b_b64", choices=sorted(workloads.ALL))
    ap.add_argument("--num-splits", type=int, default=None)
    ap.add_argument("--cpu-sample", type=int, default=16, help="sequences in the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=0, help="run N untimed steps and exit (for ncu)")
    ap.add_argument("--kv-dtype", default=None, choices=["bf16", "fp8", "int8"],
                    help="run the workload with another KV storage type")
    ap.add_argument("--no-cascade", action="store_true",
                    help="every sequence reads its own blocks (no shared-prefix decode)")
    ap.add_argument("--cascade", type=int, default=1, choices=[0, 1, 2],
                    help="shared-prefix decode: 0 off, 1 sequence pairs, 2 group prefixes (multi-query kernel)")
    ap.add_argument("--time-kernels", action="store_true",
                    help="bracket every kernel (not only decode) with events; adds gaps to the step")
    ap.add_argument("--head-dim", type=int, default=None, choices=[64, 128],
                    help="run the workload with another head_dim")
    ap.add_argument("--max-len", type=int, default=None,
                    help="cap every sequence's length (a smaller case of the workload, e.g. for profiling)")
    ap.add_argument("--channel-scales", action="store_true",
                    help="FP8 / INT8: per-channel scales on top of the per-token ones")
    ap.add_argument("--no-sustained", action="store_true", help="skip the sustained (>= 1 s) leg")
    ap.add_argument("--sustain-s", type=float, default=1.0, help="seconds of the sustained leg")
    ap.add_argument("--no-long-ctx", action="store_true",
                    help="default workload only: skip the 128K FP8 leg reported inside the same line")
    ap.add_argument("--op", default="step", choices=["step", "compact", "swap"],
                    help="step: the decode step (default); compact: H2O compaction of the streaming workload's "
                         "sequences to their keep-sets; swap: every sequence to pinned host memory and back")
    args = ap.parse_args()

    wl = workloads.ALL[args.workload]()
    label = wl.name
    if args.kv_dtype and args.kv_dtype != wl.kv_dtype:
        import dataclasses
        wl = dataclasses.replace(wl, kv_dtype=args.kv_dtype)
        label = f"{wl.name}_{args.kv_dtype}"
    if args.head_dim and args.head_dim != wl.head_dim:
        import dataclasses
        wl = dataclasses.replace(wl, head_dim=args.head_dim)
        label = f"{label}_d{args.head_dim}"
    if args.channel_scales:
        if wl.kv_dtype not in ("fp8", "int8"):
            raise SystemExit("--channel-scales needs an FP8 or INT8 workload (--kv-dtype)")
        label = f"{label}_channel"
    if args.max_len:
        import dataclasses
        wl = dataclasses.replace(wl, lens=tuple(min(L, args.max_len) for L in wl.lens))
        label = f"{label}_max{args.max_len}"
    splits = wl.num_splits if args.num_splits is None else args.num_splits
    ws, rank, local = dist_info()

    if args.impl == "reference":
        if rank != 0:
            return
        return run_reference(args, wl, label)

    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import paged_kv_cache_282_gb300 as pkv
    pkv.load()
    if args.op != "step":
        if ws > 1:
            raise SystemExit("--op compact / swap run on one GPU")
        return run_op(args, wl, label, dev)

    cascade = 0 if args.no_cascade else args.cascade
    line = measure(args, wl, label, splits, dev, ws, rank, cascade, headline=True)
    if args.profile_steps:
        return
    # The second throughput target: the 128K-context FP8 batch (64 splits),
    # measured in the same process (every rank) and reported inside the same line.
    if (args.workload == "llama3_8b_b64" and not args.kv_dtype and not args.no_long_ctx and
            args.num_splits is None and not args.head_dim and not args.max_len and not args.channel_scales):
        wl2 = workloads.long_context_fp8()
        leg = measure(args, wl2, wl2.name, wl2.num_splits, dev, ws, rank, cascade, headline=False)
        if line is not None and leg is not None:
            line["long_ctx_fp8"] = leg
    if rank == 0 and line is not None:
        print(json.dumps(line))


def run_op(args, wl, label, dev):
    """Throughput of the NEXT-row data movers on a workload-sized pool.

    compact: the streaming workload's sequences are forked (sharing every
    block) and each fork is compacted to its H2O keep-set (2048 positions
    out of the sink + window set); per round the kept rows are read and
    written once (K and V, + scales), algorithmic bytes = 2 x the kept rows'
    bytes, against the HBM copy peak.  The forks are freed between rounds;
    their score arrays are not compacted (no acc argument).  The timed call
    includes the host's table rewrite (the dropped entries of a long, mostly
    evicted sequence become -1) and its upload.
    swap: every sequence of the workload moves to pinned host memory and
    back; bytes per direction = the blocks' K/V (+ scales); the copies run
    through the host pool's device-mapped address, so the bound is the
    host link (no measured peak for it: peak null)."""
    import torch
    from paged_kv_cache_282_gb300 import BLOCK_SIZE
    if args.op == "compact" and wl.name != "streaming_h2o":
        wl = workloads.streaming_h2o()
        label = wl.name
    setup = Setup(wl, dev, extra_seqs=len(wl.lens) if args.op == "compact" else 0)
    c = setup.cache
    stream = torch.cuda.current_stream(dev)
    rounds = max(3, min(args.steps, 50))
    peak, peak_kind = hbm_peak()
    row_bytes = wl.head_dim * BYTES[wl.kv_dtype] + (4 if wl.kv_dtype in ("fp8", "int8") else 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    time.sleep(0.3)
    if args.op == "compact":
        st = Stepper(setup, wl.num_splits)
        for _ in range(max(3, args.warmup)):
            st.step()  # decode + H2O scores accumulate into st.acc
        n = len(setup.ids)
        keep = torch.zeros((n, wl.budget), dtype=torch.int32, device=dev)
        cnt = torch.zeros(n, dtype=torch.int32, device=dev)
        c.h2o_select(st.ids, st.acc, st.stride, wl.budget, wl.recent, keep, wl.budget, cnt)
        c.sync_status()
        counts = cnt.cpu().numpy()
        moved = int(counts.sum()) * wl.n_kv_heads * 2 * row_bytes  # K and V rows read (and as many written)

        q0 = st.q[:0]

        def one_round(timed):
            forks = [c.seq_fork(s) for s in setup.ids]
            c.decode([], q0)  # an empty call flushes the forks' queued table writes before the timed call
            if timed:
                e0.record(stream)
            c.seq_compact(forks, counts, keep, wl.budget)
            if timed:
                e1.record(stream)
            c.sync_status()
            for f in forks:
                c.seq_free(f)
            return e0.elapsed_time(e1) if timed else 0.0

        for _ in range(3):
            one_round(False)
        c.timing_enable(["compact"])
        c.timing_read()
        t_wall0 = time.time()
        ms = [one_round(True) for _ in range(rounds)]
        t_wall1 = time.time()
        kt = c.timing_read()["compact"]
        c.timing_enable(False)
        algo = 2 * moved
        call_ms = statistics.median(ms)
        kern_ms = kt[0] / max(kt[1], 1)
        line = {"metric": "H2O compaction GB/s (kept rows read + written, frac of HBM peak)",
                "value": round(algo / (call_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "op": "compact",
                "n_gpus": 1, "steps": rounds, "warmup": max(3, args.warmup), "ms_per_op": round(call_ms, 5),
                "higher_is_better": True, "dtype": wl.kv_dtype, "data": "synthetic",
                "config": {"workload": label, "sequences": n, "kept_rows": int(counts.sum()),
                           "bytes_per_op": algo},
                "roofline": {"bound": "hbm", "kernel": "compact_gather_kernel",
                             "achieved": round(algo / (kern_ms * 1e-3) / 1e9, 2), "peak": peak,
                             "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
                             "frac": round(algo / (kern_ms * 1e-3) / 1e9 / peak, 4),
                             "avg_launch_ms": round(kern_ms, 5)}}
    else:
        blocks = 0
        for s in setup.ids:
            blocks += int((c.block_table(s) >= 0).sum())
        c.swap_space(blocks + 16)
        per_dir = blocks * wl.n_kv_heads * BLOCK_SIZE * 2 * row_bytes

        def one_round(timed):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            c.swap_out(setup.ids)
            ev[1].record(stream)
            c.swap_in(setup.ids)
            ev[2].record(stream)
            c.sync_status()
            return (ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])) if timed else (0.0, 0.0)

        for _ in range(3):
            one_round(False)
        c.timing_enable(["swap_copy"])
        c.timing_read()
        t_wall0 = time.time()
        ms = [one_round(True) for _ in range(rounds)]
        t_wall1 = time.time()
        kt = c.timing_read()["swap_copy"]
        c.timing_enable(False)
        out_ms = statistics.median([a for a, _ in ms])
        in_ms = statistics.median([b for _, b in ms])
        kern_ms = kt[0] / max(kt[1], 1)
        line = {"metric": "CPU swap GB/s per direction (device pool <-> pinned host pool)",
                "value": round(2 * per_dir / ((out_ms + in_ms) * 1e-3) / 1e9, 2), "unit": "GB/s", "op": "swap",
                "n_gpus": 1, "steps": rounds, "warmup": 3, "ms_per_op": round(out_ms + in_ms, 5),
                "higher_is_better": True, "dtype": wl.kv_dtype, "data": "synthetic",
                "config": {"workload": label, "sequences": len(setup.ids), "blocks": blocks,
                           "bytes_per_direction": per_dir},
                "swap_out_gbs": round(per_dir / (out_ms * 1e-3) / 1e9, 2),
                "swap_in_gbs": round(per_dir / (in_ms * 1e-3) / 1e9, 2),
                "roofline": {"bound": "host link", "kernel": "block_copy_kernel",
                             "achieved": round(per_dir / (kern_ms * 1e-3) / 1e9, 2), "peak": None,
                             "unit": "GB/s", "frac": None, "avg_launch_ms": round(kern_ms, 5)}}
    clocks.stop()
    line["clocks"] = clocks.summary(t_wall0, t_wall1)
    print(json.dumps(line))


def run_reference(args, wl, label):
    """The CPU oracle as it stands, timed on this machine's cores, each step a
    bounded sample of the workload."""
    n = min(args.cpu_sample, wl.batch)
    res = [oracle_baseline(wl, n) for _ in range(max(1, args.warmup and 1))]  # warm-up (page in, threads)
    times = []
    for _ in range(args.steps):
        r = oracle_baseline(wl, n)
        times.append(r["seconds"])
    t = sum(times) / len(times)
    lens = list(wl.lens)[:n]
    byts = sum(_kept(L, wl) for L in lens) * _kv_bytes_per_token(wl)
    value = byts / t / 1e9
    cores = os.cpu_count() or 1
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": label, "batch": wl.batch, "sample_sequences": n},
        "tokens_per_s": round(n / t, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": res[0]["sample"]},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    main()
