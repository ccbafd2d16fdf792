"""Parity at the full sizes of the five workloads, in the launch
configuration bench.py times (automatic splits; 64 splits for the 128K FP8
case).  The oracle computes every output of every sequence; pool bytes are
compared on a sample of blocks."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from harness import (H2O_RTOL, TOL, Twin, build_prefix, build_streaming, fill_sequences, lse_err, max_err,
                     pool_bytes_equal)

pytestmark = pytest.mark.gpu


def _decode_and_compare(tw, ids, wl, splits, mask="full", S=0, W=0):
    q = workloads.queries(wl, len(ids))
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, mask=mask, num_sinks=S, window=W, num_splits=splits)
    tw.cache.sync_status()
    ref, ref_lse, _ = tw.oracle_decode(ids, q, mask, S, W)
    err = max_err(out, ref)
    assert err <= TOL[wl.kv_dtype], err
    assert lse_err(lse, ref_lse) <= 2e-3
    return err


def test_llama3_8b_batch64():
    wl = workloads.llama3_8b_batch64()
    nb = sum((L + 15) // 16 for L in wl.lens)  # a pool sized to fit exactly
    tw = Twin(wl, nb, wl.batch, max((L + 15) // 16 for L in wl.lens), seed=wl.seed)
    ids = fill_sequences(tw, wl.lens, chunk=16384)
    assert tw.cache.stats()["free_blocks"] == 0
    for s in ids:
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    pool_bytes_equal(tw, ids, every=7)
    _decode_and_compare(tw, ids, wl, splits=0)
    _decode_and_compare(tw, ids, wl, splits=8)


def test_long_context_fp8():
    wl = workloads.long_context_fp8()
    nb = sum((L + 15) // 16 for L in wl.lens)
    tw = Twin(wl, nb, wl.batch, max((L + 15) // 16 for L in wl.lens), seed=wl.seed)
    ids = fill_sequences(tw, wl.lens, chunk=16384)
    pool_bytes_equal(tw, ids, every=61)
    _decode_and_compare(tw, ids, wl, splits=64)
    _decode_and_compare(tw, ids, wl, splits=0)


def test_streaming_h2o():
    wl = workloads.streaming_h2o()
    tw, ids = build_streaming(wl)
    S, W = wl.num_sinks, wl.window
    lens = [tw.alloc.length(s) for s in ids]
    assert lens == list(wl.lens)
    for s in ids:
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    # only blocks that intersect the keep-set hold storage
    assert all((tw.alloc.table(s) >= 0).sum() <= 2 + (W + 15) // 16 for s in ids)
    pool_bytes_equal(tw, ids, every=5)
    stride = max(lens)
    q = workloads.queries(wl, len(ids))
    logits = torch.zeros((len(ids), wl.n_kv_heads, stride, wl.group), device="cuda")
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale, mask="sink_window", num_sinks=S, window=W,
                               logits=logits, logits_stride=stride)
    acc = torch.zeros((len(ids), stride), device="cuda")
    tw.cache.h2o_scores(ids, logits, stride, lse, acc, stride, mask="sink_window", num_sinks=S, window=W)
    keep = torch.full((len(ids), wl.budget), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(len(ids), dtype=torch.int32, device="cuda")
    tw.cache.h2o_select(ids, acc, stride, wl.budget, wl.recent, keep, wl.budget, cnt)
    tw.cache.sync_status()

    ref, ref_lse, ref_logits = tw.oracle_decode(ids, q, "sink_window", S, W, want_logits=True, logits_stride=stride)
    assert max_err(out, ref) <= TOL["bf16"] and lse_err(lse, ref_lse) <= 2e-3
    ref_acc = np.zeros((len(ids), stride))
    oracle.h2o_update(ref_acc, lens, ref_logits, ref_lse, oracle.MASK_SINK_WINDOW, S, W)
    got_acc = acc.cpu().numpy().astype(np.float64)
    assert np.allclose(got_acc, ref_acc, rtol=H2O_RTOL, atol=1e-9)
    keep, cnt = keep.cpu().numpy(), cnt.cpu().numpy()
    k = wl.budget - wl.recent
    for b, L in enumerate(lens):
        got = set(keep[b, : cnt[b]].tolist())
        want = set(oracle.h2o_select(L, wl.budget, wl.recent, ref_acc[b, :L]).tolist())
        assert cnt[b] == len(want) == wl.budget
        cand = np.sort(ref_acc[b, : L - wl.recent])[::-1]
        kth = cand[k - 1]
        # the selections may differ only where scores tie within fp32 error
        for j in got ^ want:
            assert abs(ref_acc[b, j] - kth) <= H2O_RTOL * kth + 1e-9, (b, j, ref_acc[b, j], kth)


def test_prefix_sharing_append_cow():
    wl = workloads.prefix_append()
    tw, ids = build_prefix(wl)
    assert len(ids) == 256
    st = tw.cache.stats()
    assert st["shared_blocks"] >= 4 * 128  # every group prefix block is shared
    k, v = workloads.new_tokens(wl, len(ids), 0)
    _, cow = tw.append(ids, k, v)
    expected = sum(1 for s in wl.extra["suffix"] if (2048 + s) % 16)
    assert len(cow) == expected and tw.cache.stats()["cow_copies"] == expected
    for s in ids:
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
    pool_bytes_equal(tw, ids, every=9)
    for mode in (1, 2, 0):  # sequence pairs, group prefixes (multi-query kernel), off
        tw.cache.set_cascade(mode)
        _decode_and_compare(tw, ids, wl, splits=0)
    tw.cache.set_cascade(1)


def test_prefix_sharing_literal_shapes_never_copy():
    """Without the fork, no shared block is ever last (the prefix is exactly
    128 blocks), so an append copies nothing."""
    wl = workloads.prefix_append(groups=2, parents_per_group=4)
    tw, ids = build_prefix(wl, fork_parents=False)
    k, v = workloads.new_tokens(wl, len(ids), 0)
    _, cow = tw.append(ids, k, v)
    assert len(cow) == 0 and tw.cache.stats()["cow_copies"] == 0
    _decode_and_compare(tw, ids, wl, splits=0)
