"""Pins for the CPU oracle: every check here compares the oracle with something
other than itself -- numbers the pages print, literal re-runs of the pages'
own snippets on tiny inputs, exhaustive search, closed forms, invariants and
library routines (torch's float8 codec and scaled_dot_product_attention).

Pages (title, section):
  [LC] "长上下文优化：注意力稀疏化与 KV Cache 管理"
  [PA] "KV Cache 与 PagedAttention：显存复用与长上下文推理"
  [SO] "系统优化"
"""
import itertools
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden_kv():
    vals = {}
    with open(os.path.join(GOLDEN, "kv_sizes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (x.strip() for x in line.split("="))
                vals[k] = float(v)
    return vals


def _read_golden_layout():
    rows = {}
    with open(os.path.join(GOLDEN, "page_layout_example.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                parts = line.split()
                rows[parts[0]] = (int(parts[1]), [int(x) for x in parts[2:]])
    return rows


# --------------------------------------------------------------------------
# KV sizes ([LC] KV bytes per token, kv_cache_gb; [PA] 显存公式, 收益评估)
# --------------------------------------------------------------------------

def test_kv_bytes_per_token_llama3_8b():
    g = _read_golden_kv()
    assert oracle.kv_bytes_per_token(32, 8, 128, 2) == g["llama3_8b_bytes_per_token"]
    # "128000 x 128KB ~ 16 GB": decimal gigabytes, approximate.
    gb = 128000 * oracle.kv_bytes_per_token(32, 8, 128, 2) / 1e9
    assert abs(gb - g["llama3_8b_128000_tokens_gb_approx"]) / 16 < 0.06


def test_kv_cache_gb_printouts_are_twice_the_formula():
    """The page's printed comments are exactly 2x what its own formula
    returns; the formula is taken as authoritative (the printouts are read as
    a slip in the page)."""
    g = _read_golden_kv()
    f8k = oracle.kv_cache_gib(32, 8, 128, 8192)
    f128k = oracle.kv_cache_gib(32, 8, 128, 131072)
    f128k8 = oracle.kv_cache_gib(32, 8, 128, 131072, dtype_bytes=1)
    assert (f8k, f128k, f128k8) == (1.0, 16.0, 8.0)
    assert g["printed_kv_cache_gb_8192"] == 2 * f8k
    assert g["printed_kv_cache_gb_131072"] == 2 * f128k
    assert g["printed_kv_cache_gb_131072_fp8"] == 2 * f128k8


def test_llama2_70b_table():
    g = _read_golden_kv()
    vals = [oracle.kv_cache_size_bytes(80, 8, 128, s) / 1024 ** 3 for s in (2048, 8192, 32768)]
    assert vals == [0.625, 2.5, 10.0]
    # 0.625 is an exact binary tie; the page shows 0.63 (half-up), Python's
    # two-decimal format gives 0.62 (half-even).  Both are 0.625 rounded.
    assert abs(vals[0] - g["printed_llama2_70b_gib_2048"]) <= 0.005 + 1e-12
    assert round(vals[1], 2) == g["printed_llama2_70b_gib_8192"]
    assert round(vals[2], 2) == g["printed_llama2_70b_gib_32768"]
    assert 8 * oracle.kv_cache_size_bytes(80, 8, 128, 32768) / 1024 ** 3 == g["llama2_70b_batch8_32k_gib"]
    assert oracle.kv_cache_size_bytes(80, 8, 128, 32768, 2) / 1024 ** 3 == g["seq32k_80layers_fp16_gib"]
    assert oracle.kv_cache_size_bytes(80, 8, 128, 32768, 1) / 1024 ** 3 == g["seq32k_80layers_int8_gib"]


# --------------------------------------------------------------------------
# FP8 E4M3 codec ([PA] KV 量化: FP16 -> FP8 (E4M3), per-token scaling).
# torch's float8_e4m3fn conversion is the library routine it reduces to.
# --------------------------------------------------------------------------

def _torch_e4m3_value(code: int) -> float:
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float())


def _torch_e4m3_code(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_all_codes():
    for c in range(256):
        got = oracle.e4m3_decode(c)
        ref = _torch_e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(got) and math.isnan(ref)
        else:
            assert got == ref, hex(c)
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_roundtrip_finite_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_ties_round_to_even():
    finite = sorted({oracle.e4m3_decode(c) for c in range(0x00, 0x7F)})
    for lo, hi in zip(finite[:-1], finite[1:]):
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exactly representable
        code = oracle.e4m3_encode(float(mid))
        assert code % 2 == 0, (lo, hi, code)
        assert oracle.e4m3_decode(code) in (lo, hi)
        assert oracle.e4m3_encode(-float(mid)) == code | 0x80


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    mags = np.exp2(rng.uniform(-12, math.log2(448.0), 60000)).astype(np.float32)
    sub = rng.uniform(0, 2.0 ** -6, 20000).astype(np.float32)
    vals = np.concatenate([mags, sub, np.float32([0.0, 448.0, 2.0 ** -9, 2.0 ** -10, 2.0 ** -6])])
    vals = np.concatenate([vals, -vals])
    got = oracle.e4m3_encode_array(vals)
    ref = _torch_e4m3_code(vals)
    assert np.array_equal(got, ref)


def test_e4m3_saturates():
    for x in (448.0001, 460.0, 464.0, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_quantize_row_per_token_scale():
    rng = np.random.default_rng(3)
    for trial in range(200):
        D = 128 if trial % 2 else 64
        x = torch.from_numpy(rng.standard_normal(D).astype(np.float32) * 10 ** rng.uniform(-3, 3))
        bits = workloads.as_bits(x.to(torch.bfloat16))
        xf = x.to(torch.bfloat16).float().numpy()
        codes, s = oracle.quantize_row_bf16(bits)
        amax = float(np.max(np.abs(xf)))
        i = int(np.argmax(np.abs(xf)))
        # the largest magnitude lands on the largest finite code
        assert codes[i] == (0xFE if xf[i] < 0 else 0x7E)
        assert abs(s * 448.0 - amax) <= amax * 2 ** -22
        # every code is the library's E4M3 rounding of x / s
        assert np.array_equal(codes, _torch_e4m3_code(xf / np.float32(s)))
        # dequantisation error within half an E4M3 step
        deq = np.array([oracle.e4m3_decode(c) for c in codes]) * s
        tol = np.maximum(np.abs(xf) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
        assert np.all(np.abs(deq - xf) <= tol)
    codes, s = oracle.quantize_row_bf16(np.zeros(128, dtype=np.uint16))
    assert s == 1.0 and not codes.any()


def _channel_restatement(xf, c, kv):
    """Per-channel + per-token quantisation written again with numpy float32
    arithmetic (IEEE division) and the library codecs: y = x / c, s =
    absmax(y) / qmax, code = Q(y / s)."""
    qmax = np.float32(127.0 if kv == "int8" else 448.0)
    y = np.asarray(xf, np.float32) / np.asarray(c, np.float32)
    amax = np.float32(np.max(np.abs(y)))
    s = np.float32(1.0) if amax == 0 else np.float32(amax / qmax)
    z = (y / s).astype(np.float32)
    if kv == "int8":
        return np.clip(np.rint(z.astype(np.float64)), -127, 127).astype(np.int8), float(s)
    return _torch_e4m3_code(z), float(s)


@pytest.mark.parametrize("kv", ["fp8", "int8"])
def test_quantize_row_channel_scales(kv):
    """Per-channel scaling ([PA] KV quantisation names per-channel and
    per-token scaling): codes and scale equal an independent restatement;
    unit channel scales (or none) reproduce the per-token quantiser byte for
    byte; dequantisation code * s * c lies within half a step of x."""
    rng = np.random.default_rng(5 if kv == "fp8" else 6)
    kvc = oracle.KV_INT8 if kv == "int8" else oracle.KV_FP8
    per_token = oracle.quantize_row_int8 if kv == "int8" else oracle.quantize_row_bf16
    for trial in range(200):
        D = 128 if trial % 2 else 64
        x = torch.from_numpy(rng.standard_normal(D).astype(np.float32) * 10 ** rng.uniform(-2, 2))
        bits = workloads.as_bits(x.to(torch.bfloat16))
        xf = x.to(torch.bfloat16).float().numpy()
        c = (10.0 ** rng.uniform(-1.5, 1.5, D)).astype(np.float32)
        if trial % 3 == 0:
            c = (2.0 ** rng.integers(-4, 5, D)).astype(np.float32)  # exact powers of two
        codes, s = oracle.quantize_row_channel(bits, c, kvc)
        want, ws = _channel_restatement(xf, c, kv)
        assert s == ws and np.array_equal(codes, want), trial
        # no channel scales, or all ones: the per-token scheme exactly
        pc, ps = per_token(bits)
        for cc in (None, np.ones(D, np.float32)):
            c1, s1 = oracle.quantize_row_channel(bits, cc, kvc)
            assert s1 == ps and np.array_equal(c1, pc)
        # dequantisation within half a step (times the channel scale)
        if kv == "int8":
            deq = codes.astype(np.float64) * s * c
            tol = 0.5 * s * c.astype(np.float64) * (1 + 1e-6)
        else:
            deq = np.array([oracle.e4m3_decode(int(v)) for v in codes]) * s * c
            y = np.abs(xf.astype(np.float64) / c)
            tol = np.maximum(y * 2.0 ** -4, s * 2.0 ** -10) * c * (1 + 1e-6)
        assert np.all(np.abs(deq - xf) <= tol + 1e-30), trial


@pytest.mark.parametrize("kv,ratio", [("int8", 100.0), ("fp8", 1e5)])
def test_channel_scales_tame_outlier_channels(kv, ratio):
    """What per-channel scales are for: keys with a few outlier channels lose
    the small channels under per-token scaling (INT8's uniform steps already
    at 100x; FP8's floating steps only once the small channels fall into its
    subnormal range); dividing each channel by its own magnitude first keeps
    their precision."""
    rng = np.random.default_rng(9)
    D, T = 128, 64
    mag = np.ones(D, np.float32)
    mag[[3, 40, 77, 120]] = ratio
    x = rng.standard_normal((T, D)).astype(np.float32) * mag
    xb = torch.from_numpy(x).to(torch.bfloat16)
    xf = xb.float().numpy()
    kvc = oracle.KV_INT8 if kv == "int8" else oracle.KV_FP8
    err_tok, err_ch = [], []
    for t in range(T):
        bits = workloads.as_bits(xb[t])
        for c, errs in ((None, err_tok), (mag, err_ch)):
            codes, s = oracle.quantize_row_channel(bits, c, kvc)
            vals = codes.astype(np.float64) if kv == "int8" else np.array([oracle.e4m3_decode(int(v)) for v in codes])
            deq = vals * s * (1.0 if c is None else c)
            errs.append(np.abs(deq - xf[t])[mag == 1.0].mean())
    assert np.mean(err_ch) < 0.2 * np.mean(err_tok)


def test_int8_encode_rounds_half_to_even_and_clamps():
    for x, want in ((0.5, 0), (1.5, 2), (2.5, 2), (-2.5, -2), (-3.5, -4), (126.5, 126), (0.49999997, 0),
                    (127.0, 127), (127.4, 127), (127.6, 127), (300.0, 127), (-1e9, -127), (float("inf"), 127),
                    (-0.0, 0), (float("nan"), 0)):
        assert oracle.int8_encode(x) == want, x


def test_int8_encode_matches_numpy_rounding():
    rng = np.random.default_rng(17)
    x = (rng.standard_normal(100_000) * 60).astype(np.float32)
    x[:2000] = np.round(x[:2000]) + 0.5  # exact ties
    want = np.clip(np.rint(x.astype(np.float64)), -127, 127).astype(np.int8)
    got = np.array([oracle.int8_encode(float(v)) for v in x], dtype=np.int8)
    assert np.array_equal(got, want)


def test_quantize_row_int8_per_token_scale():
    rng = np.random.default_rng(4)
    for trial in range(200):
        D = 128 if trial % 2 else 64
        x = torch.from_numpy(rng.standard_normal(D).astype(np.float32) * 10 ** rng.uniform(-3, 3))
        bits = workloads.as_bits(x.to(torch.bfloat16))
        xf = x.to(torch.bfloat16).float().numpy()
        codes, s = oracle.quantize_row_int8(bits)
        amax = float(np.max(np.abs(xf)))
        i = int(np.argmax(np.abs(xf)))
        # the largest magnitude lands on +-127; the scale is absmax / 127
        assert codes[i] == (-127 if xf[i] < 0 else 127)
        assert abs(s * 127.0 - amax) <= amax * 2 ** -22
        # every code is numpy's half-to-even rounding of the fp32 quotient
        q = (xf / np.float32(s)).astype(np.float32)
        assert np.array_equal(codes, np.clip(np.rint(q), -127, 127).astype(np.int8))
        # dequantisation error within half a step (plus the quotient's rounding)
        assert np.all(np.abs(codes.astype(np.float64) * s - xf) <= s * (0.5 + 1e-5))
    codes, s = oracle.quantize_row_int8(np.zeros(128, dtype=np.uint16))
    assert s == 1.0 and not codes.any()

@pytest.mark.parametrize("kv", ["fp8", "int8"])
def test_quantised_scatter_places_codes_and_scale_at_the_token_slot(kv):
    """Each (token, kv head) row lands at the token's slot: the codes and the
    scale stored there are the pinned per-token quantisation of that row,
    and every slot nobody wrote stays zero."""
    kvd = {"fp8": oracle.KV_FP8, "int8": oracle.KV_INT8}[kv]
    quant = oracle.quantize_row_bf16 if kv == "fp8" else oracle.quantize_row_int8
    rng = np.random.default_rng(21)
    NB, Hk, D, T = 6, 3, 64, 37
    pool = oracle.OraclePool(NB, Hk, D, kvd)
    slots = rng.choice(NB * 16, size=T, replace=False)

    def rows():
        x = rng.standard_normal((T, Hk, D)) * 10 ** rng.uniform(-2, 2, (T, Hk, 1))
        return workloads.as_bits(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16))

    kb, vb = rows(), rows()
    pool.write(slots, kb, vb)
    written = np.zeros((NB, 16), dtype=bool)
    for t, sl in enumerate(slots):
        b, o = divmod(int(sl), 16)
        written[b, o] = True
        for g in range(Hk):
            for codes_arr, scale_arr, src in ((pool.k, pool.k_scale, kb), (pool.v, pool.v_scale, vb)):
                codes, sc = quant(src[t, g])
                assert np.array_equal(codes_arr[b, g, o], codes)
                assert scale_arr[b, g, o] == np.float32(sc)
    for arr in (pool.k, pool.v):
        assert not arr.transpose(0, 2, 1, 3)[~written].any()
    for arr in (pool.k_scale, pool.v_scale):
        assert not arr.transpose(0, 2, 1)[~written].any()


# --------------------------------------------------------------------------
# Keep-sets versus the pages' own snippets, re-run literally on tiny inputs.
# --------------------------------------------------------------------------

def _visible_by_distance(L, window):
    """Row L-1 of the symmetric distance mask of the [LC] sliding-window
    snippet: key j is visible to query i when |i - j| <= window."""
    i = np.full(L, L - 1)
    j = np.arange(L)
    return [int(x) for x in j[np.abs(i - j) <= window]]


def _streaming_keep_by_simulation(L, num_sinks, window):
    """Feed token indices one at a time into a list that, whenever it grows
    past num_sinks + window entries, is cut down to its first num_sinks and
    last window entries -- what the [LC] StreamingKVCache snippet does."""
    kept = []
    for tok in range(L):
        kept.append(tok)
        if len(kept) > num_sinks + window:
            kept = kept[:num_sinks] + kept[len(kept) - window:]
    return kept


def test_sliding_window_matches_page_mask():
    for L in range(1, 65):
        for W in range(0, 41):
            assert oracle.keep_set(L, oracle.MASK_SLIDING, 0, W) == _visible_by_distance(L, W), (L, W)


def test_sink_window_matches_page_streaming_cache():
    for S in range(0, 7):
        for W in range(1, 41):
            for L in range(1, 65):
                got = oracle.keep_set(L, oracle.MASK_SINK_WINDOW, S, W)
                assert got == _streaming_keep_by_simulation(L, S, W), (S, W, L)


def test_full_mask_keeps_everything():
    for L in (0, 1, 17, 100):
        assert oracle.keep_set(L, oracle.MASK_FULL) == list(range(L))


# --------------------------------------------------------------------------
# H2O ([LC] H2OEviction, [SO] evict_tokens).
# --------------------------------------------------------------------------

def _exhaustive_select(scores, L, budget, recent):
    keep = budget - recent
    if L <= budget or L - recent <= keep:
        return list(range(L))
    cand = range(0, L - recent)
    best, best_key = None, None
    for sub in itertools.combinations(cand, keep):
        total = sum(scores[j] for j in sub)
        key = (total, [-j for j in sub])  # max sum, then lexicographically smallest
        if best_key is None or key > best_key:
            best, best_key = list(sub), key
    return sorted(set(best) | set(range(L - recent, L)))


def test_h2o_select_exhaustive():
    rng = random.Random(12)
    for _ in range(400):
        L = rng.randint(1, 12)
        budget = rng.randint(1, 12)
        recent = rng.randint(0, budget)
        scores = [float(rng.randint(0, 3)) for _ in range(L)]  # many ties
        got = oracle.h2o_select(L, budget, recent, np.array(scores)).tolist()
        assert got == _exhaustive_select(scores, L, budget, recent), (L, budget, recent, scores)


def test_h2o_select_page_variant_without_recent():
    # [SO] evict_tokens keeps topk(budget) of the summed scores: recent = 0
    rng = np.random.default_rng(5)
    s = rng.random(50)
    got = oracle.h2o_select(50, 10, 0, s)
    assert got.tolist() == sorted(np.argsort(-s, kind="stable")[:10].tolist())


def test_policy_select_reduces_to_parts():
    """The combined rule is the union of three independently pinned pieces:
    the sinks, the recent window, and the plain top-k of all positions (the
    select with recent = 0), and also numpy's stable ranking of all scores."""
    rng = np.random.default_rng(8)
    for L in (1, 3, 4, 5, 40, 260, 300, 700):
        for sinks, window, heavy in ((4, 256, 252), (0, 0, 7), (2, 3, 0), (0, 5, 5), (6, 0, 1000)):
            s = np.floor(rng.random(L) * 6)  # many ties
            got = oracle.policy_select(L, sinks, window, heavy, s).tolist()
            top = oracle.h2o_select(L, heavy, 0, s).tolist() if heavy else []
            ranked = np.argsort(-s, kind="stable")[:heavy].tolist()
            assert sorted(top) == sorted(ranked)
            want = sorted(set(range(min(sinks, L))) | set(range(max(L - window, 0), L)) | set(top))
            assert got == want, (L, sinks, window, heavy)


def test_policy_select_printed_configuration():
    """Sink 4, window 256, 512 - 4 - 256 = 252 heavy hitters.  Scores that
    put the 252 largest strictly inside the middle keep exactly 512
    positions; scores that put them in the window keep only 4 + 256."""
    L = 2000
    s = np.zeros(L)
    mid = np.arange(100, 100 + 252 * 5, 5)
    s[mid] = 1.0 + np.arange(252)
    got = oracle.policy_select(L, 4, 256, 512 - 4 - 256, s)
    assert got.size == 512
    assert got.tolist() == sorted([0, 1, 2, 3] + mid.tolist() + list(range(L - 256, L)))
    s = np.zeros(L)
    s[L - 256:] = 5.0
    got = oracle.policy_select(L, 4, 256, 252, s)
    assert got.tolist() == [0, 1, 2, 3] + list(range(L - 256, L))


def _accumulate_h2o(weights_per_step):
    """[LC] H2OEviction.update_scores restated: each step's weights [heads,
    q_len, kv_len] are reduced to one value per position (sum over queries,
    mean over heads) and added to a running total that is zero-extended to
    the step's kv_len."""
    total = torch.zeros(0, dtype=torch.float64)
    for w in weights_per_step:
        per_pos = torch.einsum("hqk->k", w) / w.shape[0]
        grown = torch.zeros(max(per_pos.numel(), total.numel()), dtype=torch.float64)
        grown[: total.numel()] += total
        grown[: per_pos.numel()] += per_pos
        total = grown
    return total


def _dense_attention_weights(q, K, scale, keep_mask, G):
    # softmax over kept keys, per query head: [H, 1, L]
    Kh = K.repeat_interleave(G, dim=1)  # [L][H][D]
    s = torch.einsum("hd,lhd->hl", q, Kh) * scale
    s = s.masked_fill(~keep_mask[None, :], float("-inf"))
    return torch.softmax(s, dim=-1)[:, None, :]


def _build_oracle_cache(wl, lens, seed, order=None):
    """Allocate and fill an oracle pool for sequences of the given lengths."""
    nb = sum((L + 15) // 16 for L in lens) + 4
    alloc = oracle.OracleAllocator(nb, len(lens), max((L + 15) // 16 for L in lens) + 1, seed=seed,
                                   order=order)
    kvd = {"fp32": oracle.KV_FP32, "bf16": oracle.KV_BF16, "fp8": oracle.KV_FP8,
           "int8": oracle.KV_INT8}[wl.kv_dtype]
    pool = oracle.OraclePool(nb, wl.n_kv_heads, wl.head_dim, kvd)
    ids = [alloc.seq_add() for _ in lens]
    dense = []
    for b, L in enumerate(lens):
        k, v = workloads.kv_rows(wl, b, 0, L)
        slots, cow = alloc.append([ids[b]], L)
        assert cow.size == 0
        pool.write(slots, workloads.as_bits(k), workloads.as_bits(v))
        dense.append((k, v))
    return alloc, pool, ids, dense


def test_h2o_update_matches_page_algorithm():
    wl = workloads.small("fp32", lens=(40,), n_heads=4, n_kv_heads=2, head_dim=16)
    L0 = 30
    alloc, pool, ids, dense = _build_oracle_cache(wl, (40,), seed=9)
    k, v = dense[0]
    attn_steps = []
    acc = np.zeros((1, 64))
    for step, L in enumerate(range(L0, 41, 5)):
        alloc.truncate(ids[0], L)  # view the first L tokens
        q = workloads.queries(wl, 1, step=step)
        tables = alloc.tables_matrix(ids)
        out, lse, logits = oracle.decode(pool, tables, [L], workloads.as_bits(q), oracle.KV_FP32,
                                         wl.n_heads, wl.scale, want_logits=True, logits_stride=64)
        oracle.h2o_update(acc, [L], logits, lse)
        attn = _dense_attention_weights(q[0].double(), k[:L].double(), wl.scale,
                                        torch.ones(L, dtype=torch.bool), wl.group)
        attn_steps.append(attn)
        # softmax rows sum to one, so each step adds exactly 1 to the total
        assert abs(acc.sum() - (step + 1)) < 1e-12
        alloc, pool, ids, _ = _build_oracle_cache(wl, (40,), seed=9)  # restore full length
    ref = _accumulate_h2o(attn_steps).numpy()
    assert np.allclose(acc[0, : ref.size], ref, rtol=1e-12, atol=1e-15)



@pytest.mark.parametrize("mask,S,W", [("sliding", 0, 7), ("sink_window", 4, 9)])
def test_h2o_update_gives_masked_positions_no_weight(mask, S, W):
    """Under a mask, a position outside the keep-set gets no attention weight,
    whatever the logits buffer holds there: the update adds nothing to it,
    the step still adds exactly 1 in total, and the kept positions get the
    masked softmax weights (mean over heads) of textbook attention."""
    wl = workloads.small("fp32", lens=(40,), n_heads=4, n_kv_heads=2, head_dim=16)
    L = 40
    alloc, pool, ids, dense = _build_oracle_cache(wl, (L,), seed=11)
    k, _ = dense[0]
    mode = {"sliding": oracle.MASK_SLIDING, "sink_window": oracle.MASK_SINK_WINDOW}[mask]
    q = workloads.queries(wl, 1, step=3)
    _, lse, logits = oracle.decode(pool, alloc.tables_matrix(ids), [L], workloads.as_bits(q), oracle.KV_FP32,
                                   wl.n_heads, wl.scale, mode, S, W, want_logits=True, logits_stride=64)
    kept = torch.zeros(L, dtype=torch.bool)
    kept[oracle.keep_set(L, mode, S, W)] = True
    assert 0 < int(kept.sum()) < L
    ref = _accumulate_h2o([_dense_attention_weights(q[0].double(), k[:L].double(), wl.scale, kept,
                                                    wl.group)]).numpy()
    dropped = ~kept.numpy()
    for fill in (None, 0.0, 50.0):  # masked logits as the decode left them, or finite values
        lg = logits.copy()
        if fill is not None:
            lg[:, :, :L][:, :, dropped] = fill
        acc = np.zeros((1, 64))
        oracle.h2o_update(acc, [L], lg, lse, mode, S, W)
        assert np.all(acc[0, :L][dropped] == 0.0)
        assert abs(acc.sum() - 1.0) < 1e-12
        assert np.allclose(acc[0, :L], ref, rtol=1e-12, atol=1e-15)

# --------------------------------------------------------------------------
# Attention: closed forms, textbook attention (SDPA) and paging invariance.
# --------------------------------------------------------------------------

def _sdpa(q, K, V, G, keep_mask, scale):
    """Library attention on a dense contiguous layout: q [H][D], K/V [L][Hk][D]."""
    Kh = K.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]  # [1][H][L][D]
    Vh = V.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    qh = q[None, :, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qh, Kh, Vh, attn_mask=keep_mask[None, None, None, :],
                                                         scale=scale)
    return o[0, :, 0, :]


def _dequant_dense(wl, pool, alloc, sid, L):
    """Dequantised dense [L][Hk][D]: codes through torch's float8 decoder
    (library) or as plain integers, times the per-token scales."""
    t = alloc.table(sid)
    ks, vs = [], []
    for j in range(L):
        b, o = t[j // 16], j % 16
        if wl.kv_dtype == "int8":
            kc = torch.from_numpy(pool.k[b, :, o, :].astype(np.float64))
            vc = torch.from_numpy(pool.v[b, :, o, :].astype(np.float64))
        else:
            kc = torch.from_numpy(pool.k[b, :, o, :].copy()).view(torch.float8_e4m3fn).double()
            vc = torch.from_numpy(pool.v[b, :, o, :].copy()).view(torch.float8_e4m3fn).double()
        ks.append(kc * torch.from_numpy(pool.k_scale[b, :, o].astype(np.float64))[:, None])
        vs.append(vc * torch.from_numpy(pool.v_scale[b, :, o].astype(np.float64))[:, None])
    return torch.stack(ks), torch.stack(vs)


@pytest.mark.parametrize("kv", ["fp8", "int8"])
def test_decode_with_channel_scales_matches_library_attention(kv):
    """FP8 / INT8 pools with per-channel scales (different per kv head): the
    oracle's decode equals library attention on the dense layout dequantised
    here as code * token scale * channel scale, and the stored codes equal the
    per-row quantiser's."""
    lens = (1, 17, 50, 97)
    wl = workloads.small(kv, lens=lens, n_heads=8, n_kv_heads=2, head_dim=32, seed=23)
    rng = np.random.default_rng(41)
    kc = (10.0 ** rng.uniform(-1, 1, (2, 32))).astype(np.float32)
    vc = (10.0 ** rng.uniform(-1, 1, (2, 32))).astype(np.float32)
    nb = sum((L + 15) // 16 for L in lens) + 2
    alloc = oracle.OracleAllocator(nb, len(lens), 8, seed=4)
    kvc = oracle.KV_INT8 if kv == "int8" else oracle.KV_FP8
    pool = oracle.OraclePool(nb, 2, 32, kvc)
    pool.set_channel_scales(kc, vc)
    ids = [alloc.seq_add() for _ in lens]
    for b, L in enumerate(lens):
        k, v = workloads.kv_rows(wl, b, 0, L)
        slots, _ = alloc.append([ids[b]], L)
        pool.write(slots, workloads.as_bits(k), workloads.as_bits(v))
        # codes at the slots equal the per-row quantiser with the same channel scales
        j = L - 1
        blk, off = int(slots[j] // 16), int(slots[j] % 16)
        for g in range(2):
            ck, sk = oracle.quantize_row_channel(workloads.as_bits(k[j, g]), kc[g], kvc)
            assert np.array_equal(pool.k[blk, g, off], ck) and pool.k_scale[blk, g, off] == sk
    q = workloads.queries(wl)
    qd = q.float().double()
    out, lse, _ = oracle.decode(pool, alloc.tables_matrix(ids), lens, workloads.as_bits(q), oracle.KV_BF16,
                                wl.n_heads, wl.scale)
    for b, L in enumerate(lens):
        K, V = _dequant_dense(wl, pool, alloc, ids[b], L)
        K = K * torch.from_numpy(kc.astype(np.float64))[None]
        V = V * torch.from_numpy(vc.astype(np.float64))[None]
        keep = torch.ones(L, dtype=torch.bool)
        ref = _sdpa(qd[b], K, V, wl.group, keep, wl.scale)
        assert torch.allclose(torch.from_numpy(out[b]), ref, rtol=1e-10, atol=1e-12), (b, L)


@pytest.mark.parametrize("kv", ["fp32", "bf16", "fp8", "int8"])
@pytest.mark.parametrize("mask", ["full", "sliding", "sink_window"])
def test_decode_matches_library_attention(kv, mask):
    lens = (1, 16, 17, 50, 97)
    wl = workloads.small(kv, lens=lens, n_heads=8, n_kv_heads=2, head_dim=32, seed=21)
    mode = {"full": oracle.MASK_FULL, "sliding": oracle.MASK_SLIDING,
            "sink_window": oracle.MASK_SINK_WINDOW}[mask]
    S, W = (3, 20) if mask == "sink_window" else (0, 24)
    alloc, pool, ids, dense = _build_oracle_cache(wl, lens, seed=33)
    q = workloads.queries(wl)
    qd = q.double() if kv == "fp32" else q.float().double()
    out, lse, _ = oracle.decode(pool, alloc.tables_matrix(ids), lens, workloads.as_bits(q),
                                oracle.KV_FP32 if kv == "fp32" else oracle.KV_BF16, wl.n_heads,
                                wl.scale, mode, S, W)
    for b, L in enumerate(lens):
        if kv in ("fp8", "int8"):
            K, V = _dequant_dense(wl, pool, alloc, ids[b], L)
        else:
            K, V = dense[b][0].double(), dense[b][1].double()
        keep = torch.tensor([oracle.keep(L, mode, S, W, j) for j in range(L)])
        ref = _sdpa(qd[b], K, V, wl.group, keep, wl.scale)
        assert torch.allclose(torch.from_numpy(out[b]), ref, rtol=1e-10, atol=1e-12), (b, L)
        # lse against the library's logsumexp of the kept logits
        Kh = K.repeat_interleave(wl.group, dim=1)
        s = torch.einsum("hd,lhd->hl", qd[b], Kh) * wl.scale
        ref_lse = torch.logsumexp(s[:, keep], dim=-1)
        assert torch.allclose(torch.from_numpy(lse[b]), ref_lse, rtol=1e-12, atol=1e-12)


def test_decode_closed_forms():
    wl = workloads.small("fp32", lens=(1, 40, 40), n_heads=4, n_kv_heads=2, head_dim=16, seed=4)
    alloc = oracle.OracleAllocator(16, 3, 4, seed=2)
    pool = oracle.OraclePool(16, 2, 16, oracle.KV_FP32)
    ids = [alloc.seq_add() for _ in range(3)]
    q = workloads.queries(wl)
    g = torch.Generator().manual_seed(0)
    # seq 0: L = 1 -> out = V_0
    k0, v0 = torch.randn(1, 2, 16, generator=g), torch.randn(1, 2, 16, generator=g)
    # seq 1: every K equal -> uniform weights -> out = mean of V
    k1 = torch.randn(1, 2, 16, generator=g).expand(40, 2, 16).contiguous()
    v1 = torch.randn(40, 2, 16, generator=g)
    # seq 2: key 17 aligned with every query head of its group, huge logit -> out = V_17
    k2 = torch.randn(40, 2, 16, generator=g) * 1e-3
    v2 = torch.randn(40, 2, 16, generator=g)
    for h in range(4):
        k2[17, h // 2] += q[2, h] * 200.0
    for sid, (k, v) in zip(ids, ((k0, v0), (k1, v1), (k2, v2))):
        slots, _ = alloc.append([sid], k.shape[0])
        pool.write(slots, k.numpy(), v.numpy())
    out, lse, _ = oracle.decode(pool, alloc.tables_matrix(ids), [1, 40, 40], q.numpy(),
                                oracle.KV_FP32, 4, wl.scale)
    for h in range(4):
        assert np.array_equal(out[0, h], v0[0, h // 2].double().numpy())
        assert abs(lse[0, h] - wl.scale * float(q[0, h].double() @ k0[0, h // 2].double())) < 1e-12
        assert np.allclose(out[1, h], v1[:, h // 2].double().mean(0).numpy(), rtol=0, atol=1e-12)
        assert abs(lse[1, h] - (wl.scale * float(q[1, h].double() @ k1[0, h // 2].double()) + math.log(40))) < 1e-10
    # huge-logit case: the two heads of group 0 and 1 both pick token 17
    for h in range(4):
        assert np.allclose(out[2, h], v2[17, h // 2].double().numpy(), atol=1e-9)


def test_decode_invariant_to_physical_placement():
    lens = (5, 33, 64, 100)
    wl = workloads.small("bf16", lens=lens, n_heads=8, n_kv_heads=4, head_dim=32, seed=8)
    q = workloads.as_bits(workloads.queries(wl))
    results = []
    for seed in (0, 1, 2, 99):
        alloc, pool, ids, _ = _build_oracle_cache(wl, lens, seed=seed)
        out, lse, _ = oracle.decode(pool, alloc.tables_matrix(ids), lens, q, oracle.KV_BF16,
                                    wl.n_heads, wl.scale)
        results.append((out, lse))
    tabs = [_build_oracle_cache(wl, lens, seed=s)[0].tables_matrix(range(4)) for s in (0, 1)]
    assert not np.array_equal(tabs[0], tabs[1])  # the placements really differ
    for out, lse in results[1:]:
        assert np.array_equal(out, results[0][0]) and np.array_equal(lse, results[0][1])


def test_decode_rejects_unmapped_kept_block():
    wl = workloads.small("fp32", lens=(20,), n_heads=2, n_kv_heads=1, head_dim=16)
    alloc, pool, ids, _ = _build_oracle_cache(wl, (20,), seed=1)
    t = alloc.tables_matrix(ids)
    t[0, 0] = -1
    with pytest.raises(ValueError):
        oracle.decode(pool, t, [20], workloads.as_bits(workloads.queries(wl)), oracle.KV_FP32, 2, 0.25)


def test_empty_keep_set():
    wl = workloads.small("fp32", lens=(20,), n_heads=2, n_kv_heads=1, head_dim=16)
    alloc, pool, ids, _ = _build_oracle_cache(wl, (20,), seed=1)
    out, lse, _ = oracle.decode(pool, alloc.tables_matrix(ids), [0],
                                workloads.as_bits(workloads.queries(wl)), oracle.KV_FP32, 2, 0.25)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# --------------------------------------------------------------------------
# Allocator ([PA] PagedAttention design, three runtime components, COW).
# --------------------------------------------------------------------------

def test_splitmix64_published_vector():
    # first outputs of splitmix64 seeded with 0 (Vigna's reference generator)
    assert oracle.splitmix64_stream(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                               0x06C45D188009454F]


def test_page_physical_layout_example():
    rows = _read_golden_layout()
    order = [7, 12, 3, 5, 8, 1, 2, 0, 9, 4, 6, 10, 11, 13, 14, 15]
    a = oracle.OracleAllocator(16, 4, 8, order=order)
    for name in ("A", "B", "C"):
        L, blocks = rows[name]
        s = a.seq_add()
        slots, _ = a.append([s], L)
        assert a.table(s).tolist() == blocks, name
        # consecutive positions fill a block before moving on
        assert slots.tolist() == [blocks[p // 16] * 16 + p % 16 for p in range(L)]
    # request A's last block holds 35 - 32 = 3 tokens
    assert rows["A"][0] - 16 * (len(rows["A"][1]) - 1) == 3
    L, blocks = rows["LC"]
    b = oracle.OracleAllocator(32, 1, 4, order=blocks + [x for x in range(32) if x not in blocks])
    s = b.seq_add()
    b.append([s], L)
    assert b.table(s).tolist() == blocks



@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_block_row_and_swap_copies_move_every_array(kv):
    """A copy-on-write block copy makes the destination block equal to the
    source in K, V and both scale arrays and changes nothing else; a row copy
    does the same for single token slots; swap copies move whole blocks
    between the device and host pools in the direction asked."""
    kvd = {"bf16": oracle.KV_BF16, "fp8": oracle.KV_FP8, "int8": oracle.KV_INT8}[kv]
    rng = np.random.default_rng(5)
    pool = oracle.OraclePool(5, 2, 32, kvd)

    def arrays():
        return [x for x in (pool.k, pool.v, pool.k_scale, pool.v_scale) if x is not None]

    for a in arrays():
        if a.dtype == np.float32:
            a[...] = rng.standard_normal(a.shape)
        else:
            info = np.iinfo(a.dtype)
            a[...] = rng.integers(info.min, info.max, a.shape, endpoint=True, dtype=a.dtype)
    before = [a.copy() for a in arrays()]
    pool.copy_block(1, 3)
    for a, b0 in zip(arrays(), before):
        want = b0.copy()
        want[3] = b0[1]
        assert np.array_equal(a, want)
    before = [a.copy() for a in arrays()]
    src, dst = [5, 17, 40], [70, 2, 33]
    pool.copy_rows(src, dst)
    for a, b0 in zip(arrays(), before):
        want = b0.copy()
        for s_, d_ in zip(src, dst):
            want[d_ // 16, :, d_ % 16] = b0[s_ // 16, :, s_ % 16]
        assert np.array_equal(a, want)
    pool.add_host_pool(4)
    host = [x for x in (pool.hk, pool.hv, pool.hk_scale, pool.hv_scale) if x is not None]
    dev = [a.copy() for a in arrays()]
    pool.swap_copy(np.array([[4, 2], [0, 1]]), out=True)
    for h, d0 in zip(host, dev):
        assert np.array_equal(h[2], d0[4]) and np.array_equal(h[1], d0[0])
        assert not h[0].any() and not h[3].any()
    assert all(np.array_equal(a, d0) for a, d0 in zip(arrays(), dev))
    pool.swap_copy(np.array([[2, 3]]), out=False)
    for a, d0 in zip(arrays(), dev):
        want = d0.copy()
        want[3] = d0[4]
        assert np.array_equal(a, want)

def test_free_pool_initial_order():
    a = oracle.OracleAllocator(50, 1, 4, seed=0)
    assert a.free_list().tolist() == list(range(50))
    b = oracle.OracleAllocator(50, 1, 4, seed=1234)
    fl = b.free_list().tolist()
    assert sorted(fl) == list(range(50)) and fl != list(range(50))



def test_smallest_free_sequence_id_and_last_freed_block_first():
    """The allocator's determinism rules on tiny inputs: a new sequence takes
    the smallest id not in use; freed blocks go back to the front of the free
    pool in ascending logical order, so the last one freed is reused first."""
    a = oracle.OracleAllocator(8, 4, 4, seed=0)
    assert [a.seq_add() for _ in range(3)] == [0, 1, 2]
    a.free(1)
    assert a.seq_add() == 1
    a.free(2)
    a.free(0)
    assert [a.seq_add(), a.seq_add(), a.seq_add()] == [0, 2, 3]
    b = oracle.OracleAllocator(8, 4, 4, seed=0)  # identity order: block 0 at the front
    x, y = b.seq_add(), b.seq_add()
    b.append([x], 20)
    b.append([y], 1)
    assert b.table(x).tolist() == [0, 1] and b.table(y).tolist() == [2]
    b.free(x)  # releases block 0, then block 1
    assert b.free_list().tolist() == [1, 0, 3, 4, 5, 6, 7]
    z = b.seq_add()
    b.append([z], 17)
    assert b.table(z).tolist() == [1, 0]

def _check_invariants(a, live):
    NB = a.NB
    held, host_held = {}, {}
    for s in live:
        t = a.table(s)
        assert t.size == (a.length(s) + 15) // 16
        if getattr(a, "NH", 0) and a.swapped(s):
            assert not (t >= 0).any()  # a swapped-out sequence holds no device block
            for hb in a.host_table(s):
                if hb >= 0:
                    host_held[hb] = host_held.get(hb, 0) + 1
        for blk in t:
            if blk >= 0:
                held[blk] = held.get(blk, 0) + 1
    if getattr(a, "NH", 0):
        assert a.num_host_free() + len(host_held) == a.NH
        for hb in range(a.NH):
            assert a.host_refcount(hb) == host_held.get(hb, 0)
    free = a.free_list().tolist()
    assert len(set(free)) == len(free)
    assert set(free).isdisjoint(held)
    assert set(free) | set(held) == set(range(NB))
    for blk in range(NB):
        assert a.refcount(blk) == held.get(blk, 0)


def test_allocator_random_ops_invariants_and_contents():
    """Random add/append/fork/free/evict/H2O-compact/truncate/CPU swap; a
    content model (token ids written through slots, COW pairs applied as
    whole-block copies, compaction as row moves into the returned fresh
    blocks, swaps as block copies between the device and host pools) must
    give every sequence exactly its own history."""
    rng = random.Random(2024)
    for trial in range(30):
        NB = rng.randint(8, 60)
        a = oracle.OracleAllocator(NB, 12, 40, seed=rng.randint(0, 10 ** 9))
        NH = rng.randint(4, 60)
        a.set_swap_space(NH)
        data = np.full((NB, 16), -1, dtype=np.int64)  # physical content: token labels
        hdata = np.full((NH, 16), -1, dtype=np.int64)  # host swap space content
        hist = {}  # seq -> list of labels (or None for evicted positions)
        label = 0
        for op in range(120):
            r = rng.random()
            if r < 0.1 and hist:
                # CPU swap: move some sequences out or back in
                out = rng.random() < 0.5
                cand = [s for s in hist if a.swapped(s) != out]
                if cand:
                    ids = rng.sample(cand, rng.randint(1, len(cand)))
                    before = (a.free_list().tolist(), a.num_host_free())
                    try:
                        pairs = a.swap_out(ids) if out else a.swap_in(ids)
                    except MemoryError:
                        assert (a.free_list().tolist(), a.num_host_free()) == before
                        continue
                    for src, dst in pairs:
                        if out:
                            hdata[dst] = data[src]
                        else:
                            data[dst] = hdata[src]
                    with pytest.raises(ValueError):  # not twice to the same place
                        a.swap_out(ids[:1]) if out else a.swap_in(ids[:1])
                    if out:  # device-side operations refuse a swapped-out sequence
                        with pytest.raises(ValueError):
                            a.append(ids[:1], 1)
                        with pytest.raises(ValueError):
                            a.fork(ids[0])
                        with pytest.raises(ValueError):
                            a.truncate(ids[0], 0)
                _check_invariants(a, list(hist))
                continue
            live = [s for s in hist if not a.swapped(s)]
            r = rng.random()
            if r >= 0.15 and not live:
                continue
            if r < 0.15 or not live:
                try:
                    s = a.seq_add()
                except RuntimeError:
                    continue
                hist[s] = []
            elif r < 0.65:
                ids = rng.sample(live, rng.randint(1, len(live)))
                T = rng.randint(1, 20)
                if any(len(hist[s]) + T > 40 * 16 for s in ids):
                    continue
                before = a.free_list().tolist()
                try:
                    slots, cow = a.append(ids, T)
                except MemoryError:
                    assert a.free_list().tolist() == before  # unchanged on failure
                    continue
                for src, dst in cow:
                    data[dst] = data[src]
                for i, s in enumerate(ids):
                    for t in range(T):
                        sl = slots[i * T + t]
                        data[sl // 16, sl % 16] = label
                        hist[s].append(label)
                        label += 1
            elif r < 0.75:
                s = rng.choice(live)
                try:
                    d = a.fork(s)
                except ValueError:
                    continue
                hist[d] = list(hist[s])
            elif r < 0.85:
                s = rng.choice(list(hist))  # swapped-out sequences can be freed too
                a.free(s)
                del hist[s]
            elif r < 0.91:
                s = rng.choice(live)
                S, W = rng.randint(0, 5), rng.randint(1, 30)
                a.evict(s, S, W)
                L = len(hist[s])
                if L > S + W:
                    for lb in range((L + 15) // 16):
                        lo, hi = lb * 16, min(L, lb * 16 + 16)
                        if not any(j < S or j >= L - W for j in range(lo, hi)):
                            for j in range(lo, hi):
                                hist[s][j] = None
            elif r < 0.96:
                ids = rng.sample(live, rng.randint(1, len(live)))
                keeps = []
                for s in ids:
                    held = [j for j, lab in enumerate(hist[s]) if lab is not None]
                    keeps.append(sorted(rng.sample(held, rng.randint(0, len(held)))))
                src = [[int(a.table(s)[j // 16]) * 16 + j % 16 for j in k] for s, k in zip(ids, keeps)]
                before = a.free_list().tolist()
                try:
                    fresh = a.compact(ids, [len(k) for k in keeps])
                except MemoryError:
                    assert a.free_list().tolist() == before
                    continue
                for s, k, sl, f in zip(ids, keeps, src, fresh):
                    assert len(f) == (len(k) + 15) // 16 and set(f.tolist()) <= set(before)
                    moved = [data[x // 16, x % 16] for x in sl]
                    for i, lab in enumerate(moved):
                        data[f[i // 16], i % 16] = lab
                    hist[s] = [hist[s][j] for j in k]
            else:
                s = rng.choice(live)
                n = rng.randint(0, len(hist[s]))
                if n % 16 and hist[s][n - 1] is None:
                    with pytest.raises(ValueError):
                        a.truncate(s, n)
                    continue
                a.truncate(s, n)
                hist[s] = hist[s][:n]
            _check_invariants(a, list(hist))
            for s, h in hist.items():
                swapped = a.swapped(s)
                t = a.host_table(s) if swapped else a.table(s)
                mem = hdata if swapped else data
                for j, lab in enumerate(h):
                    if lab is None:
                        assert t[j // 16] == -1
                    else:
                        assert mem[t[j // 16], j % 16] == lab, (trial, op, s, j)


def test_cow_fires_once_per_shared_partial_block():
    a = oracle.OracleAllocator(16, 4, 8, seed=0)
    p = a.seq_add()
    a.append([p], 20)  # blocks 0, 1 (second partially filled)
    f = a.fork(p)
    assert a.refcount(1) == 2
    slots, cow = a.append([p, f], 1)
    assert cow.tolist() == [[1, 2]]  # parent copies its shared last block
    assert a.table(p).tolist() == [0, 2] and a.table(f).tolist() == [0, 1]
    assert a.refcount(1) == 1 and a.refcount(2) == 1 and a.refcount(0) == 2
    assert slots.tolist() == [2 * 16 + 4, 1 * 16 + 4]  # sibling writes in place
    # a fork at a block boundary needs no copy: the next token opens a block
    a2 = oracle.OracleAllocator(16, 4, 8, seed=0)
    p = a2.seq_add()
    a2.append([p], 32)
    f = a2.fork(p)
    _, cow = a2.append([p, f], 1)
    assert cow.size == 0


def test_append_all_or_nothing():
    a = oracle.OracleAllocator(4, 3, 8, seed=5)
    s0, s1 = a.seq_add(), a.seq_add()
    a.append([s0], 40)  # 3 blocks
    before = (a.free_list().tolist(), a.table(s0).tolist(), a.length(s0))
    with pytest.raises(MemoryError):
        a.append([s0, s1], 20)  # needs 1 + 2 blocks, 1 free
    assert (a.free_list().tolist(), a.table(s0).tolist(), a.length(s0)) == before
    assert a.length(s1) == 0
