"""GPU parity: libpkv (through the C ABI) against the CPU oracle on the same
seeded inputs.  Bit-exact for block tables, slot placement, COW copies, FP8
codes and scales, and H2O keep-sets on a given score array; attention output
within max abs error 1e-2 (BF16 KV) / 2e-2 (FP8 KV) / 1e-4 (FP32 KV)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import H2O_RTOL, TOL, Twin, fill_sequences, length_only_pool, lse_err, max_err, output_bounds
from paged_kv_cache_282_gb300 import _abi

pytestmark = pytest.mark.gpu


def _pool_bytes_equal(tw: Twin, ids):
    """K/V bytes (and FP8 scales) of every written slot of every live sequence
    equal the oracle's; unwritten slots hold whatever the memory held."""
    c = tw.cache
    NB, Hk = tw.pool.NB, tw.wl.n_kv_heads
    dev = [c.k_pool, c.v_pool]
    host = [tw.pool.k, tw.pool.v]
    if tw.wl.kv_dtype in ("fp8", "int8"):
        dev += [c.k_scale, c.v_scale]
        host += [tw.pool.k_scale, tw.pool.v_scale]
    for dt, ht in zip(dev, host):
        d = dt.contiguous().view(torch.uint8).reshape(NB, Hk, 16, -1).cpu().numpy()
        h = ht.view(np.uint8).reshape(NB, Hk, 16, -1)
        for s in ids:
            L = tw.alloc.length(s)
            for lb, blk in enumerate(tw.alloc.table(s)):
                if blk >= 0:
                    n = min(16, L - 16 * lb)
                    assert np.array_equal(d[blk, :, :n], h[blk, :, :n]), (s, lb, blk)


# --------------------------------------------------------------------------
# tiny configuration: fp32, 4/2/64, lengths 35, 10, 70 in a 16-block pool
# --------------------------------------------------------------------------

@pytest.mark.parametrize("placement", ["page_literal", "seeded"])
def test_tiny_fp32(placement):
    wl = workloads.tiny()
    order = [7, 12, 3, 5, 8, 1, 2, 0, 9, 4, 6, 10, 11, 13, 14, 15] if placement == "page_literal" else None
    tw = Twin(wl, 16, 3, 8, seed=wl.seed, free_order=order)
    ids = fill_sequences(tw, wl.lens)
    if placement == "page_literal":
        assert [tw.cache.block_table(s).tolist() for s in ids] == [[7, 12, 3], [5], [8, 1, 2, 0, 9]]
    for s in ids:
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    _pool_bytes_equal(tw, ids)
    q = workloads.queries(wl)
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale)
    tw.cache.sync_status()
    ref, ref_lse, _ = tw.oracle_decode(ids, q)
    assert max_err(out, ref) <= TOL["fp32"]
    assert lse_err(lse, ref_lse) <= 1e-4
    test_tiny_fp32.outputs = getattr(test_tiny_fp32, "outputs", []) + [out.cpu()]
    if len(test_tiny_fp32.outputs) == 2:  # both placements: identical bits
        assert torch.equal(test_tiny_fp32.outputs[0], test_tiny_fp32.outputs[1])


# --------------------------------------------------------------------------
# small ragged cases across dtypes, group sizes, masks and split counts
# --------------------------------------------------------------------------

LENS = (1, 15, 16, 17, 33, 200, 517, 1000, 2049)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_small_full_mask(kv, G, D):
    wl = workloads.small(kv, lens=LENS, n_heads=8 * G, n_kv_heads=8, head_dim=D, seed=30 + G)
    nb = sum((L + 15) // 16 for L in LENS) + 5
    tw = Twin(wl, nb, len(LENS), 160, seed=123)
    ids = fill_sequences(tw, LENS)
    _pool_bytes_equal(tw, ids)
    q = workloads.queries(wl)
    ref, ref_lse, _ = tw.oracle_decode(ids, q)
    outs = []
    for splits in (0, 1, 3, 64):
        out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, num_splits=splits)
        tw.cache.sync_status()
        assert max_err(out, ref) <= TOL[kv], (splits, max_err(out, ref))
        assert lse_err(lse, ref_lse) <= 2e-3, splits
        outs.append(out.float().cpu())
    # split count changes only the merge order
    for o in outs[1:]:
        assert (o - outs[0]).abs().max() <= 8e-3


@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("mask,S,W", [("sliding", 0, 0), ("sliding", 0, 37), ("sliding", 0, 600),
                                      ("sink_window", 4, 100), ("sink_window", 0, 64), ("sink_window", 20, 3),
                                      ("sink_window", 0, 0)])
@pytest.mark.parametrize("D", [128, 64])
def test_small_masks(kv, mask, S, W, D):
    wl = workloads.small(kv, lens=LENS, head_dim=D, seed=50)
    nb = sum((L + 15) // 16 for L in LENS)
    tw = Twin(wl, nb, len(LENS), 160, seed=9)
    ids = fill_sequences(tw, LENS)
    q = workloads.queries(wl)
    ref, ref_lse, _ = tw.oracle_decode(ids, q, mask, S, W)
    for splits in (0, 2):
        out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, mask=mask, num_sinks=S, window=W,
                                   num_splits=splits)
        tw.cache.sync_status()
        assert max_err(out, ref) <= TOL[kv]
        assert lse_err(lse, ref_lse) <= 2e-3


# Error allowed relative to each output row's natural scale (output_bounds):
# the output's bf16 rounding (2^-9 relative) plus the rounding of the softmax
# weights for the PV product (bf16, 2^-9, on BF16 pools; fp16, 2^-12, on FP8 /
# INT8 pools), with some room; output_bounds adds the fp32 logits' part.
WIDE_TOL = {"bf16": 6e-3, "fp8": 4e-3, "int8": 4e-3}


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("kv", ["fp8", "int8", "bf16"])
def test_wide_magnitudes(kv, D):
    """Every K and V row (token, kv head) and every query head carries its own
    magnitude 10^U(-3, 3): the fp16 operands of the one-byte path must
    neither overflow nor flush.  Each output row matches the oracle within
    output_bounds (a fixed fraction of its natural scale sum_j p_j max_d |V_j|
    plus the fp32 logits' share), and lse within a relative bound."""
    lens = (1, 2, 17, 200, 517, 1000, 2049)
    wl = workloads.small(kv, lens=lens, head_dim=D, seed=95 + D, extra={"spread": 3.0})
    tw = Twin(wl, sum((L + 15) // 16 for L in lens) + 4, len(lens), 160, seed=8)
    if kv != "bf16" and D == 64:  # per-channel scales 2^-7 .. 2^7 as well
        rng = np.random.default_rng(12)
        tw.set_channel_scales((2.0 ** rng.integers(-7, 8, (8, D))).astype(np.float32),
                              (2.0 ** rng.integers(-7, 8, (8, D))).astype(np.float32))
    ids = fill_sequences(tw, lens)
    stride = max(lens)
    for step in (0, 1):
        q = workloads.queries(wl, step=step)
        ref, ref_lse, ref_lg = tw.oracle_decode(ids, q, want_logits=True, logits_stride=stride)
        bound = output_bounds(tw, ids, q, ref_lg, ref_lse, WIDE_TOL[kv])
        for splits in (0, 3):
            out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, num_splits=splits)
            tw.cache.sync_status()
            err = np.abs(out.float().cpu().numpy().astype(np.float64) - ref).max(axis=2)
            bad = np.argwhere(err > bound)
            assert bad.size == 0, (step, splits, bad[:4].tolist(), err[tuple(bad[0])], bound[tuple(bad[0])])
            got_lse = lse.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got_lse - ref_lse) <= 2e-5 * (1.0 + np.abs(ref_lse))), (step, splits)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("kv", ["fp8", "int8"])
def test_channel_scales(kv, D):
    """Per-channel scales (one power of two per kv head and channel, 2^-4 ..
    2^4) on top of the per-token ones: stored codes and token scales
    bit-exact against the oracle's quantiser with the same channel scales;
    decode within the dtype's bound for several keep-sets and splits and
    through the static-scratch entry; logits within 2e-3; lse within 2e-3.
    Scales that are not powers of two, and changing the scales while tokens
    are stored, are refused."""
    wl = workloads.small(kv, lens=LENS, head_dim=D, seed=71)
    tw = Twin(wl, sum((L + 15) // 16 for L in LENS) + 4, len(LENS), 160, seed=3)
    rng = np.random.default_rng(D + (kv == "int8"))
    kc = (2.0 ** rng.integers(-4, 5, (wl.n_kv_heads, D))).astype(np.float32)
    vc = (2.0 ** rng.integers(-4, 5, (wl.n_kv_heads, D))).astype(np.float32)
    bad = kc.copy()
    bad[1, 3] = 3.0
    with pytest.raises(_abi.PKVError) as e:
        tw.cache.set_channel_scales(torch.from_numpy(bad).cuda(), torch.from_numpy(vc).cuda())
    assert e.value.status == 1
    tw.set_channel_scales(kc, vc)
    ids = fill_sequences(tw, LENS)
    _pool_bytes_equal(tw, ids)
    q = workloads.queries(wl)
    stride = max(LENS)
    for mask, S, W, splits in (("full", 0, 0, 0), ("full", 0, 0, 3), ("sink_window", 4, 100, 0), ("sliding", 0, 37, 2)):
        ref, ref_lse, ref_lg = tw.oracle_decode(ids, q, mask, S, W, want_logits=True, logits_stride=stride)
        lg = torch.full((len(ids), wl.n_kv_heads, stride, wl.group), float("nan"), device="cuda")
        out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, mask=mask, num_sinks=S, window=W,
                                   num_splits=splits, logits=lg, logits_stride=stride)
        tw.cache.sync_status()
        assert max_err(out, ref) <= TOL[kv], (mask, splits, max_err(out, ref))
        assert lse_err(lse, ref_lse) <= 2e-3
        got = lg.permute(0, 1, 3, 2).reshape(len(ids), wl.n_heads, stride).cpu().numpy()
        kept = ~np.isnan(ref_lg)
        assert np.array_equal(kept, ~np.isnan(got)) and np.abs(got[kept] - ref_lg[kept]).max() <= 2e-3
    out, lse = tw.cache.decode_static(ids, q.cuda(), scale=wl.scale)
    tw.cache.sync_status()
    ref, ref_lse, _ = tw.oracle_decode(ids, q)
    assert max_err(out, ref) <= TOL[kv] and lse_err(lse, ref_lse) <= 2e-3
    with pytest.raises(_abi.PKVError) as e:
        tw.cache.set_channel_scales(None, None)
    assert e.value.status == 1


@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_physical_placement_invariance(kv):
    """The output depends only on logical order: two different physical
    placements give bit-identical results."""
    wl = workloads.small(kv, lens=LENS, seed=60)
    nb = sum((L + 15) // 16 for L in LENS) + 40
    q = workloads.queries(wl).cuda()
    res = []
    for seed in (1, 2):
        tw = Twin(wl, nb, len(LENS), 160, seed=seed)
        ids = fill_sequences(tw, LENS)
        res.append(tw.cache.decode(ids, q, scale=wl.scale))
        tables = [tw.cache.block_table(s).tolist() for s in ids]
        res[-1] = res[-1] + (tables,)
    assert res[0][2] != res[1][2]
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_logits_match_oracle():
    wl = workloads.small("bf16", lens=LENS, seed=61)
    nb = sum((L + 15) // 16 for L in LENS)
    tw = Twin(wl, nb, len(LENS), 160, seed=4)
    ids = fill_sequences(tw, LENS)
    q = workloads.queries(wl)
    stride = max(LENS)
    for mask, S, W in (("full", 0, 0), ("sink_window", 4, 300)):
        logits = torch.full((len(LENS), wl.n_kv_heads, stride, wl.group), float("nan"), device="cuda")
        tw.cache.decode(ids, q.cuda(), scale=wl.scale, mask=mask, num_sinks=S, window=W, logits=logits,
                        logits_stride=stride)
        _, _, ref = tw.oracle_decode(ids, q, mask, S, W, want_logits=True, logits_stride=stride)
        got = logits.permute(0, 1, 3, 2).reshape(len(LENS), wl.n_heads, stride).cpu().numpy()
        kept = ~np.isnan(ref)
        assert np.array_equal(kept, ~np.isnan(got))
        assert np.abs(got[kept] - ref[kept]).max() <= 2e-3


def test_empty_and_zero_length():
    wl = workloads.small("bf16", lens=(0, 5, 40), seed=62)
    tw = Twin(wl, 8, 3, 8, seed=1)
    ids = fill_sequences(tw, wl.lens)
    q = workloads.queries(wl)
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale)
    ref, ref_lse, _ = tw.oracle_decode(ids, q)
    assert max_err(out, ref) <= TOL["bf16"] and lse_err(lse, ref_lse) <= 2e-3
    assert torch.isneginf(lse[0]).all() and (out[0] == 0).all()
    # sink + window with nothing kept
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, mask="sink_window", num_sinks=0, window=0)
    assert (out[1:] == 0).all() and torch.isneginf(lse[1:]).all()


# --------------------------------------------------------------------------
# copy-on-write and append bit-exactness
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_fork_append_cow(kv):
    wl = workloads.small(kv, lens=(40, 64, 77), seed=70)
    tw = Twin(wl, 64, 8, 16, seed=17)
    ids = fill_sequences(tw, wl.lens)
    kids = [tw.fork(s) for s in ids]
    batch = [x for pair in zip(ids, kids) for x in pair]
    for step in range(20):
        k, v = workloads.new_tokens(wl, len(batch), step)
        _, cow = tw.append(batch, k, v)
        if step == 0:
            # the parent of each pair with a partial, shared last block copies it
            assert len(cow) == sum(1 for L in wl.lens if L % 16)
    assert tw.cache.stats()["cow_copies"] == sum(1 for L in wl.lens if L % 16)
    for s in batch:
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    _pool_bytes_equal(tw, batch)
    q = workloads.queries(wl, len(batch))
    out, lse = tw.cache.decode(batch, q.cuda(), scale=wl.scale)
    ref, ref_lse, _ = tw.oracle_decode(batch, q)
    assert max_err(out, ref) <= TOL[kv] and lse_err(lse, ref_lse) <= 2e-3


def test_evicted_block_in_keep_set_is_rejected():
    wl = workloads.small("bf16", lens=(300,), seed=71)
    tw = Twin(wl, 32, 2, 32, seed=3)
    ids = fill_sequences(tw, wl.lens)
    tw.evict(ids[0], 4, 64)
    q = workloads.queries(wl).cuda()
    with pytest.raises(Exception) as e:
        tw.cache.decode(ids, q, scale=wl.scale)
    assert getattr(e.value, "status", None) == 1
    out, lse = tw.cache.decode(ids, q, scale=wl.scale, mask="sink_window", num_sinks=4, window=64)
    ref, ref_lse, _ = tw.oracle_decode(ids, workloads.queries(wl), "sink_window", 4, 64)
    assert max_err(out, ref) <= TOL["bf16"]


def test_workspace_too_small_is_rejected():
    wl = workloads.small("bf16", lens=(3000, 3000), seed=72)
    tw = Twin(wl, 400, 2, 200, seed=3)
    ids = fill_sequences(tw, wl.lens)
    q = workloads.queries(wl).cuda()
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Exception) as e:
        tw.cache.decode(ids, q, scale=wl.scale, num_splits=8, workspace=ws)
    assert getattr(e.value, "status", None) == 9


# --------------------------------------------------------------------------
# H2O select on its own: bit-exact keep-sets on given score arrays
# --------------------------------------------------------------------------

@pytest.mark.parametrize("budget,recent", [(2048, 512), (64, 0), (100, 100), (37, 5)])
def test_h2o_select_bit_exact(budget, recent):
    lens = [0, 1, 50, budget, budget + 1, 3000, 20000, 131072]
    stride = max(lens)
    acc = workloads.h2o_scores_input(len(lens), stride, seed=budget + recent)
    cache, ids = length_only_pool(lens)
    keep = torch.full((len(lens), budget), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(len(lens), dtype=torch.int32, device="cuda")
    cache.h2o_select(ids, acc.cuda(), stride, budget, recent, keep, budget, cnt)
    cache.sync_status()
    keep, cnt = keep.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens):
        ref = oracle.h2o_select(L, budget, recent, acc[b, :L].double().numpy())
        assert cnt[b] == ref.size
        assert np.array_equal(keep[b, : cnt[b]], ref), (b, L)


@pytest.mark.parametrize("sinks,window,heavy", [(4, 256, 252), (0, 0, 64), (2, 3, 0), (16, 1024, 1000),
                                                (0, 512, 2048), (7, 0, 20000)])
def test_policy_select_bit_exact(sinks, window, heavy):
    """The combined sink + window + heavy-hitter rule on seeded score arrays
    with many ties, every length regime: all kept, ranking smaller than the
    heavy count, and long sequences whose candidates overflow shared memory."""
    lens = [0, 1, 50, 259, 260, 261, 512, 513, 3000, 20000, 131072]
    stride = max(lens)
    acc = workloads.h2o_scores_input(len(lens), stride, seed=sinks + window + heavy)
    cache, ids = length_only_pool(lens)
    width = min(sinks + window + heavy, stride)
    keep = torch.full((len(lens), width), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((len(lens),), -1, dtype=torch.int32, device="cuda")
    cache.policy_select(ids, acc.cuda(), stride, sinks, window, heavy, keep, width, cnt)
    cache.sync_status()
    keep, cnt = keep.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens):
        ref = oracle.policy_select(L, sinks, window, heavy, acc[b, :L].double().numpy())
        assert cnt[b] == ref.size, (b, L)
        assert np.array_equal(keep[b, : cnt[b]], ref), (b, L)


@pytest.mark.parametrize("pad,offset", [(1, 0), (3, 1)])
def test_select_rows_not_16_byte_aligned(pad, offset):
    """Score rows that do not start on a 16-byte boundary (a row stride that
    is not a multiple of four floats, a base pointer one float in) take the
    plain-load gather instead of the bulk-copy ring: same keep-sets."""
    lens = [3000, 20000, 70001, 131072]
    stride = max(lens) + pad
    base = workloads.h2o_scores_input(len(lens), stride, seed=11 + pad)
    cache, ids = length_only_pool(lens)
    flat = torch.zeros(offset + len(lens) * stride, dtype=torch.float32, device="cuda")
    flat[offset:] = base.reshape(-1).cuda()
    acc = flat[offset:].view(len(lens), stride)
    for sinks, window, heavy in ((4, 512, 1536), (0, 0, 9000)):
        width = sinks + window + heavy
        keep = torch.full((len(lens), width), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((len(lens),), -1, dtype=torch.int32, device="cuda")
        cache.policy_select(ids, acc, stride, sinks, window, heavy, keep, width, cnt)
        cache.sync_status()
        k, c = keep.cpu().numpy(), cnt.cpu().numpy()
        for b, L in enumerate(lens):
            ref = oracle.policy_select(L, sinks, window, heavy, base[b, :L].double().numpy())
            assert c[b] == ref.size, (b, L)
            assert np.array_equal(k[b, : c[b]], ref), (b, L)


def test_patches_and_cow_chains_in_one_flush():
    """Several host-side changes queued before one device call: a table entry
    set to -1 and back (truncate + re-append), and a copy-on-write whose source
    is the destination of an earlier queued copy."""
    wl = workloads.small("bf16", lens=(32, 20), seed=73)
    tw = Twin(wl, 32, 8, 8, seed=5)
    a, b = fill_sequences(tw, wl.lens)
    k, v = workloads.new_tokens(wl, 1, 0)
    for _ in range(3):  # truncate + re-append the block-opening token
        tw.append([a], k, v)
        tw.truncate(a, 32)
    tw.append([a], k, v)
    # chain: b's partial last block is shared, copied; the copy is shared and
    # copied again, all before any device call
    c1 = tw.fork(b)
    s1, cow1 = tw.cache.reserve_slots([b], 1)
    o1, ocow1 = tw.alloc.append([b], 1)
    c2 = tw.fork(b)
    s2, cow2 = tw.cache.reserve_slots([b], 1)
    o2, ocow2 = tw.alloc.append([b], 1)
    assert np.array_equal(cow1, ocow1) and np.array_equal(cow2, ocow2) and cow2[0, 0] == cow1[0, 1]
    for src, dst in list(ocow1) + list(ocow2):
        tw.pool.copy_block(int(src), int(dst))
    q = workloads.queries(wl, 1)
    out, lse = tw.cache.decode([a], q.cuda(), scale=wl.scale)  # flushes everything queued
    tw.cache.sync_status()
    ref, ref_lse, _ = tw.oracle_decode([a], q)
    assert max_err(out, ref) <= TOL["bf16"]
    assert np.array_equal(tw.cache.block_table(a), tw.alloc.table(a))
    for s in (a, c1, c2):
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    dst = int(cow2[0, 1])
    # b's last block holds tokens 16..19 in slots 0..3 (the rest is unwritten)
    d = tw.cache.k_pool.view(torch.int16)[dst, :, :4].cpu().numpy().view(np.uint16)
    assert np.array_equal(d, tw.pool.k[dst, :, :4])



def test_copy_into_a_block_freed_after_it_was_queued_as_a_source():
    """A queued copy-on-write reads block A; A is then freed and, before any
    device call, comes back as the destination of a second copy.  The device
    must keep the queue's order: the first copy reads A before the second
    one overwrites it."""
    wl = workloads.small("bf16", lens=(20, 20), seed=74)
    tw = Twin(wl, 16, 8, 8, seed=0)
    a, b = fill_sequences(tw, wl.lens)
    fb = tw.fork(b)  # b's part-filled last block A is shared
    _, cow1 = tw.cache.reserve_slots([b], 1)
    _, ocow1 = tw.alloc.append([b], 1)  # copy A -> B queued; fb still holds A
    tw.free(fb)  # A goes back to the front of the free pool
    fa = tw.fork(a)  # a's part-filled last block is shared
    _, cow2 = tw.cache.reserve_slots([a], 1)
    _, ocow2 = tw.alloc.append([a], 1)  # its copy lands in A
    assert np.array_equal(cow1, ocow1) and np.array_equal(cow2, ocow2)
    assert cow2[0, 1] == cow1[0, 0]
    for src, dst in list(ocow1) + list(ocow2):
        tw.pool.copy_block(int(src), int(dst))
    q = workloads.queries(wl, 1)
    tw.cache.decode([], q[:0].cuda())  # flushes everything queued
    tw.cache.sync_status()
    for s in (a, b, fa):
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    for blk in (int(cow1[0, 1]), int(cow2[0, 1])):  # slots 0..3 hold tokens 16..19
        for dev_pool, host_pool in ((tw.cache.k_pool, tw.pool.k), (tw.cache.v_pool, tw.pool.v)):
            d = dev_pool.view(torch.int16)[blk, :, :4].cpu().numpy().view(np.uint16)
            assert np.array_equal(d, host_pool[blk, :, :4]), blk

def test_bounded_wait_reports_timeout_and_context_survives():
    """A stage whose copies are never issued makes its bounded wait run out:
    the kernel returns, the status word reports the expiry, and the next
    decode on the same context is correct."""
    wl = workloads.small("bf16", lens=(300, 700), seed=80)
    tw = Twin(wl, 80, 2, 64, seed=3)
    ids = fill_sequences(tw, wl.lens)
    q = workloads.queries(wl)
    _abi.check(tw.cache.lib.pkv_set_wait_limit(tw.cache.handle, 50_000_000))  # 50 ms
    _abi.check(tw.cache.lib.pkv_test_starve_next_decode(tw.cache.handle, 0))
    tw.cache.decode(ids, q.cuda(), scale=wl.scale)
    with pytest.raises(_abi.PKVError) as e:
        tw.cache.sync_status()
    assert e.value.status == 6
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale)
    tw.cache.sync_status()
    ref, ref_lse, _ = tw.oracle_decode(ids, q)
    assert max_err(out, ref) <= TOL["bf16"] and lse_err(lse, ref_lse) <= 2e-3


@pytest.mark.parametrize("pad", [0, 5])
def test_select_chunk_boundaries(pad):
    """Ranked lengths on and around the streamed gather's 8192-key chunks,
    the last ragged chunk under 16 bytes, and the sampled path's 16384-key
    threshold, on row starts aligned to 128 bytes (pad 0) and not (pad 5):
    keep-sets exact for plain H2O and the combined rule."""
    base = [16384, 16385, 16386, 24575, 24576, 24577, 24579, 32768 + 3, 40961, 65536]
    lens = [L + 512 for L in base]  # ranked part [0, L - 512) hits the sizes above
    stride = max(lens) + pad
    acc = workloads.h2o_scores_input(len(lens), stride, seed=31 + pad)
    cache, ids = length_only_pool(lens)
    keep = torch.full((len(lens), 2048), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((len(lens),), -1, dtype=torch.int32, device="cuda")
    cache.h2o_select(ids, acc.cuda(), stride, 2048, 512, keep, 2048, cnt)
    cache.sync_status()
    k, c = keep.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens):
        ref = oracle.h2o_select(L, 2048, 512, acc[b, :L].double().numpy())
        assert c[b] == ref.size and np.array_equal(k[b, : c[b]], ref), (b, L)
    width = 4 + 256 + 4000
    keep2 = torch.full((len(lens), width), -7, dtype=torch.int32, device="cuda")
    cache.policy_select(ids, acc.cuda(), stride, 4, 256, 4000, keep2, width, cnt)
    cache.sync_status()
    k, c = keep2.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens):
        ref = oracle.policy_select(L, 4, 256, 4000, acc[b, :L].double().numpy())
        assert c[b] == ref.size and np.array_equal(k[b, : c[b]], ref), (b, L)


def test_default_stream_is_torchs_current_stream():
    """Calls without a stream argument run on torch's current stream,
    including inside a torch.cuda.stream context."""
    import paged_kv_cache_282_gb300 as pkv
    side = torch.cuda.Stream()
    assert pkv._stream_ptr(None) == torch.cuda.current_stream().cuda_stream
    with torch.cuda.stream(side):
        assert pkv._stream_ptr(None) == side.cuda_stream
    assert pkv._stream_ptr(side) == side.cuda_stream


def test_select_bounded_wait_reports_timeout_and_context_survives():
    """The first row's first streamed chunk is never copied: its bounded wait
    runs out, the status word reports the expiry, that row's count is 0, and
    the next selection on the same context is exact."""
    lens = [40000, 3000, 70001]
    stride = max(lens)
    acc = workloads.h2o_scores_input(len(lens), stride, seed=21)
    cache, ids = length_only_pool(lens)
    keep = torch.full((len(lens), 2048), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((len(lens),), -1, dtype=torch.int32, device="cuda")
    _abi.check(cache.lib.pkv_set_wait_limit(cache.handle, 50_000_000))  # 50 ms
    _abi.check(cache.lib.pkv_test_starve_next_select(cache.handle))
    cache.h2o_select(ids, acc.cuda(), stride, 2048, 512, keep, 2048, cnt)
    with pytest.raises(_abi.PKVError) as e:
        cache.sync_status()
    assert e.value.status == 6
    assert int(cnt[0]) == 0
    cache.h2o_select(ids, acc.cuda(), stride, 2048, 512, keep, 2048, cnt)
    cache.sync_status()
    k, c = keep.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens):
        ref = oracle.h2o_select(L, 2048, 512, acc[b, :L].double().numpy())
        assert c[b] == ref.size and np.array_equal(k[b, : c[b]], ref), b


# --------------------------------------------------------------------------
# H2O compaction: the keep-set becomes the whole sequence
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_h2o_compaction(kv):
    """Keep-sets from the oracle's selection on seeded scores; one sequence
    shares its blocks with a fork, one keeps nothing, one keeps everything.
    After compaction: tables and free counts equal the oracle's, every kept
    row is byte-equal, the scores moved with their tokens, decode over the
    compacted sequences matches the oracle, and appends continue after it."""
    lens = (3000, 700, 1, 257, 40)
    wl = workloads.small(kv, lens=lens, seed=81)
    tw = Twin(wl, 800, 8, 220, seed=19)
    ids = fill_sequences(tw, wl.lens)
    twin_fork = tw.fork(ids[0])
    stride = max(lens)
    acc = workloads.h2o_scores_input(len(lens), stride, seed=81)
    keeps = [oracle.h2o_select(L, 300, 64, acc[b, :L].double().numpy()) for b, L in enumerate(lens)]
    keeps[2] = np.zeros(0, dtype=np.int32)
    keeps[4] = np.arange(40, dtype=np.int32)
    acc_dev = acc.cuda()
    tw.compact(ids, keeps, acc_dev, stride)
    tw.cache.sync_status()
    for s in ids + [twin_fork]:
        assert tw.cache.seq_len(s) == tw.alloc.length(s)
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    assert tw.cache.stats()["free_blocks"] == tw.alloc.num_free()
    _pool_bytes_equal(tw, ids + [twin_fork])
    got = acc_dev.cpu().numpy()
    for b, L in enumerate(lens):
        n = len(keeps[b])
        assert np.array_equal(got[b, :n], acc.numpy()[b, keeps[b]])
        assert not got[b, n:L].any()
        assert np.array_equal(got[b, L:], acc.numpy()[b, L:])
    live = [s for s in ids if tw.alloc.length(s) > 0] + [twin_fork]
    q = workloads.queries(wl, n=len(live)).cuda()
    out, lse = tw.cache.decode(live, q, scale=wl.scale)
    ref, ref_lse, _ = tw.oracle_decode(live, q.cpu())
    assert max_err(out, ref) <= TOL[kv] and lse_err(lse, ref_lse) <= 1e-3
    k, v = workloads.new_tokens(wl, len(live), 5)
    tw.append(live, k, v)
    out, _ = tw.cache.decode(live, q, scale=wl.scale)
    ref, _, _ = tw.oracle_decode(live, q.cpu())
    assert max_err(out, ref) <= TOL[kv]
    _pool_bytes_equal(tw, live)


def test_h2o_compaction_refuses_out_of_range_positions():
    """A keep position at or past the sequence length is flagged by the
    gather (status word) instead of reading another sequence's rows."""
    wl = workloads.small("bf16", lens=(64,), seed=82)
    tw = Twin(wl, 20, 2, 8, seed=1)
    ids = fill_sequences(tw, wl.lens)
    bad = torch.tensor([[0, 5, 64]], dtype=torch.int32, device="cuda")
    tw.cache.seq_compact(ids, [3], bad, 3)
    with pytest.raises(Exception) as e:
        tw.cache.sync_status()
    assert getattr(e.value, "status", None) == 7


@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_policy_scores_select_compact_chain(kv):
    """Decode with logits, accumulate the heavy-hitter scores, keep 4 sinks +
    256 recent + 252 heavy hitters, compact, decode again.  Each side runs
    its own chain; the keep-sets may differ only where scores tie within
    fp32 rounding, and both sides compact with the oracle's keep-set."""
    lens = (3000, 700, 5000, 300, 520)
    S, W, Hh = 4, 256, 252
    wl = workloads.small(kv, lens=lens, seed=83)
    tw = Twin(wl, 1000, 6, 340, seed=23)
    ids = fill_sequences(tw, wl.lens)
    stride = max(lens)
    q = workloads.queries(wl)
    logits = torch.zeros((len(ids), wl.n_kv_heads, stride, wl.group), device="cuda")
    _, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, logits=logits, logits_stride=stride)
    acc = torch.zeros((len(ids), stride), device="cuda")
    tw.cache.h2o_scores(ids, logits, stride, lse, acc, stride)
    keep = torch.full((len(ids), S + W + Hh), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(len(ids), dtype=torch.int32, device="cuda")
    tw.cache.policy_select(ids, acc, stride, S, W, Hh, keep, S + W + Hh, cnt)
    tw.cache.sync_status()

    _, ref_lse, ref_logits = tw.oracle_decode(ids, q, want_logits=True, logits_stride=stride)
    ref_acc = np.zeros((len(ids), stride))
    oracle.h2o_update(ref_acc, list(lens), ref_logits, ref_lse, oracle.MASK_FULL, 0, 0)
    assert np.allclose(acc.cpu().numpy().astype(np.float64), ref_acc, rtol=H2O_RTOL, atol=1e-9)
    keeps = []
    gk, gc = keep.cpu().numpy(), cnt.cpu().numpy()
    for b, L in enumerate(lens):
        want = oracle.policy_select(L, S, W, Hh, ref_acc[b, :L])
        keeps.append(want)
        got = set(gk[b, : gc[b]].tolist())
        if L > Hh:
            kth = np.sort(ref_acc[b, :L])[::-1][Hh - 1]
            for j in got ^ set(want.tolist()):
                assert abs(ref_acc[b, j] - kth) <= H2O_RTOL * kth + 1e-9, (b, j)
        else:
            assert got == set(range(L))
    tw.compact(ids, keeps)
    tw.cache.sync_status()
    for s in ids:
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    _pool_bytes_equal(tw, ids)
    q2 = workloads.queries(wl, step=1)
    out, lse = tw.cache.decode(ids, q2.cuda(), scale=wl.scale)
    ref, ref_lse, _ = tw.oracle_decode(ids, q2)
    assert max_err(out, ref) <= TOL[kv] and lse_err(lse, ref_lse) <= 2e-3
