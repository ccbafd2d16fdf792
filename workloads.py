"""Seeded synthetic inputs for paged decode attention.

This module only draws numbers and fixes shapes; it holds none of the
method's arithmetic (no slots, no masks, no quantisation, no attention).
Both the CPU oracle and the CUDA library consume exactly these bytes.

Shapes follow the model shapes the pages quote: Llama-3-8B (32 query heads,
8 KV heads, head_dim 128) and Llama-2-70B (64 query heads, 8 KV heads,
head_dim 128).  No public dataset is involved: every value is N(0, 1) drawn
from a seeded CPU generator (optionally with each row's magnitude spread over
several decades, for range tests), and lengths are uniform integers from a
seeded ``random.Random``.

K/V rows are drawn per (sequence, 256-token chunk) from their own seed, so
any position range of any sequence can be produced on its own and the oracle
can be run on a subset of sequences.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field

import torch

CHUNK = 256  # tokens per independently seeded chunk of K/V rows


@dataclass(frozen=True)
class Workload:
    name: str
    n_heads: int
    n_kv_heads: int
    head_dim: int
    kv_dtype: str  # "fp32" | "bf16" | "fp8" | "int8" (fp8 and int8 are quantised from bf16 rows)
    seed: int
    lens: tuple  # context length of each sequence (including the current token)
    mask: str = "full"  # "full" | "sliding" | "sink_window"
    num_sinks: int = 0
    window: int = 0
    num_splits: int = 0  # 0 = automatic
    budget: int = 0  # H2O (0 = no H2O pass)
    recent: int = 0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def batch(self) -> int:
        return len(self.lens)

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def input_dtype(self) -> torch.dtype:
        return torch.float32 if self.kv_dtype == "fp32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


def _uniform_lengths(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = random.Random(seed)
    return tuple(rng.randint(lo, hi) for _ in range(n))


def tiny() -> Workload:
    """4 query heads, 2 KV heads, head_dim 64, fp32; lengths 35, 10, 70 in a
    16-block pool (the lengths of requests A, B, C in the PagedAttention
    page's physical-layout example)."""
    return Workload("tiny", 4, 2, 64, "fp32", seed=1, lens=(35, 10, 70),
                    extra={"num_blocks": 16})


def llama3_8b_batch64(batch: int = 64) -> Workload:
    """Llama-3-8B-shaped decode layer, bf16, batch 64, L ~ U[512, 8192]."""
    return Workload("llama3_8b_b64", 32, 8, 128, "bf16", seed=2,
                    lens=_uniform_lengths(2, batch, 512, 8192))


def long_context_fp8() -> Workload:
    """Batch 4 at 131072 tokens, FP8-E4M3 KV quantised from bf16, 64 splits."""
    return Workload("long_ctx_fp8", 32, 8, 128, "fp8", seed=3, lens=(131072,) * 4,
                    num_splits=64)


def streaming_h2o() -> Workload:
    """Batch 128, logical L ~ U[4096, 131072], 4 sinks + 4096 window, then
    H2O scores with budget 2048 and 512 recent positions forced."""
    return Workload("streaming_h2o", 32, 8, 128, "bf16", seed=4,
                    lens=_uniform_lengths(4, 128, 4096, 131072), mask="sink_window",
                    num_sinks=4, window=4096, budget=2048, recent=512)


def prefix_append(groups: int = 4, parents_per_group: int = 32) -> Workload:
    """Llama-2-70B-shaped layer (64/8/128), bf16.  Each group shares a
    2048-token prefix; each parent adds a private suffix U[100, 4000] and is
    then forked once (parallel sampling), giving 2 x groups x parents
    sequences.  ``lens`` lists the parents' lengths before the fork."""
    suffix = _uniform_lengths(5, groups * parents_per_group, 100, 4000)
    return Workload("prefix_append", 64, 8, 128, "bf16", seed=5,
                    lens=tuple(2048 + s for s in suffix),
                    extra={"groups": groups, "parents_per_group": parents_per_group,
                           "prefix": 2048, "suffix": suffix})


ALL = {"tiny": tiny, "llama3_8b_b64": llama3_8b_batch64, "long_ctx_fp8": long_context_fp8,
       "streaming_h2o": streaming_h2o, "prefix_append": prefix_append}


def small(kv_dtype: str = "bf16", lens=(1, 15, 16, 17, 33, 200, 517, 1000), n_heads: int = 32,
          n_kv_heads: int = 8, head_dim: int = 128, seed: int = 11, **kw) -> Workload:
    """Small ragged case (several tiles, ragged tails) for parity tests."""
    return Workload(f"small_{kv_dtype}", n_heads, n_kv_heads, head_dim, kv_dtype, seed=seed,
                    lens=tuple(lens), **kw)


# --------------------------------------------------------------------------
# Value generators.
# --------------------------------------------------------------------------

def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed & (2 ** 63 - 1))
    return g


def _chunk_seed(wl_seed: int, stream: int, seq: int, chunk: int) -> int:
    return (((wl_seed * 1_000_003 + stream) * 1_000_033 + seq) * 1_048_583 + chunk)


def _normal(shape, seed: int, dtype: torch.dtype, spread: float = 0.0) -> torch.Tensor:
    """N(0, 1) values; with spread > 0 every row along the last axis is
    multiplied by its own factor 10^U(-spread, spread) (drawn after the values
    from the same generator), before the conversion to ``dtype``."""
    g = _gen(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if spread > 0:
        u = torch.rand(tuple(shape[:-1]) + (1,), generator=g, dtype=torch.float64)
        x = x * (10.0 ** ((2.0 * u - 1.0) * spread)).to(torch.float32)
    return x.to(dtype)


def _spread(wl: Workload) -> float:
    """Decades of magnitude spread of the workload's rows (0: plain N(0, 1))."""
    return float(wl.extra.get("spread", 0.0))


def kv_rows(wl: Workload, seq_key: int, start: int, count: int, stream: int = 0):
    """K and V rows for positions [start, start+count) of the sequence whose
    data key is ``seq_key``: two tensors [count][Hk][D] of the input dtype."""
    out = []
    for which in (0, 1):
        parts = []
        pos = start
        end = start + count
        while pos < end:
            c = pos // CHUNK
            lo = c * CHUNK
            hi = min(end, lo + CHUNK)
            full = _normal((CHUNK, wl.n_kv_heads, wl.head_dim),
                           _chunk_seed(wl.seed, 2 * stream + which, seq_key, c), wl.input_dtype, _spread(wl))
            parts.append(full[pos - lo: hi - lo])
            pos = hi
        if parts:
            out.append(torch.cat(parts, 0).contiguous())
        else:
            out.append(torch.empty((0, wl.n_kv_heads, wl.head_dim), dtype=wl.input_dtype))
    return out[0], out[1]


def queries(wl: Workload, n: int | None = None, step: int = 0) -> torch.Tensor:
    """Decode queries [n][H][D] of the input dtype (bf16 for bf16/FP8 KV)."""
    n = wl.batch if n is None else n
    return _normal((n, wl.n_heads, wl.head_dim), _chunk_seed(wl.seed, 100 + step, 0, 0),
                   wl.input_dtype, _spread(wl)).contiguous()


def new_tokens(wl: Workload, n: int, step: int):
    """One new K/V row per sequence for an append step: [n][1][Hk][D] each."""
    k = _normal((n, 1, wl.n_kv_heads, wl.head_dim), _chunk_seed(wl.seed, 200 + 2 * step, 0, 0),
                wl.input_dtype, _spread(wl))
    v = _normal((n, 1, wl.n_kv_heads, wl.head_dim), _chunk_seed(wl.seed, 201 + 2 * step, 0, 0),
                wl.input_dtype, _spread(wl))
    return k.contiguous(), v.contiguous()


def h2o_scores_input(n: int, length: int, seed: int, tie_fraction: float = 0.25) -> torch.Tensor:
    """Non-negative fp32 accumulated-score arrays [n][length] with deliberate
    ties and zeros, for testing top-k selection on its own."""
    g = _gen(seed)
    base = torch.rand((n, length), generator=g, dtype=torch.float32)
    levels = torch.randint(0, 8, (n, length), generator=g).to(torch.float32) / 8.0
    pick = torch.rand((n, length), generator=g) < tie_fraction
    zero = torch.rand((n, length), generator=g) < 0.1
    x = torch.where(pick, levels, base)
    return torch.where(zero, torch.zeros_like(x), x).contiguous()


def as_bits(t: torch.Tensor):
    """Raw element bits as a numpy array (uint16 for bf16, float32 as is)."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view("uint16")
    return t.contiguous().numpy()
