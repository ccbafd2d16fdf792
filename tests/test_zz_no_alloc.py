"""pkv_decode_attn_static: decode that takes no workspace and allocates no
device memory -- its split-KV scratch is a fixed array inside the library --
for callers that cannot allocate device memory themselves (a framework
allocator owns the device budget, or cudaMalloc / cudaFree would stall a
latency-critical loop).  Its results must agree with pkv_decode_attn
(caller-supplied workspace) on consecutive calls.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from harness import TOL, Twin, fill_sequences, lse_err, max_err
from paged_kv_cache_282_gb300 import _abi

pytestmark = pytest.mark.gpu


def _call_static(cache, ids, q, out, lse, num_splits, mask=0, S=0, W=0):
    arr = np.ascontiguousarray(ids, dtype=np.int32)
    st = cache.lib.pkv_decode_attn_static(cache.handle, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                          arr.size, arr.ctypes.data_as(ctypes.c_void_p), q.data_ptr(),
                                          1.0 / np.sqrt(cache.head_dim), mask, S, W, num_splits, out.data_ptr(),
                                          lse.data_ptr(), None, 0)
    _abi.check(st)


@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_static_scratch_matches_workspace_decode(kv):
    lens = (1, 16, 20, 300, 1000, 2049, 4000)
    wl = workloads.small(kv, lens=lens, seed=90)
    tw = Twin(wl, sum((L + 15) // 16 for L in lens) + 8, len(lens) + 4, 300, seed=6)
    ids = fill_sequences(tw, lens)
    cache = tw.cache
    # two calls in a row, with different queries, split counts and keep-sets
    for call, (splits, mask, S, W) in enumerate([(0, 0, 0, 0), (5, 2, 4, 700)]):
        # allocator work that waits in the queue for the next device call,
        # which is the static one: a fork of a sequence whose last block is
        # partial, a one-token reservation that copies the now shared block
        # (copy-on-write), and a truncation back to the old length
        parent = ids[2 + call]
        n0 = tw.alloc.length(parent)
        fork = tw.fork(parent)
        _, cow = cache.reserve_slots([parent], 1)
        _, ocow = tw.alloc.append([parent], 1)
        assert len(cow) == 1 and np.array_equal(cow, ocow)
        tw.pool.copy_block(int(ocow[0, 0]), int(ocow[0, 1]))
        tw.truncate(parent, n0)
        batch = ids + [fork]
        mname = ["full", "sliding", "sink_window"][mask]
        q = workloads.queries(wl, n=len(batch), step=call)
        qd = q.cuda()
        out = torch.full_like(qd, float("nan"))
        lse = torch.full((len(batch), wl.n_heads), float("nan"), device="cuda")
        _call_static(cache, batch, qd, out, lse, splits, mask, S, W)
        cache.sync_status()
        assert torch.isfinite(out.float()).all()
        ref_out, ref_lse = cache.decode(batch, qd, mask=mname, num_sinks=S, window=W, num_splits=splits)
        err = (out.float() - ref_out.float()).abs().max().item()
        assert err <= TOL[kv], (call, err)
        assert lse_err(lse, ref_lse.cpu().numpy().astype(np.float64)) <= 2e-3
        # and against the oracle, which replayed the same allocator steps
        ref, o_lse, _ = tw.oracle_decode(batch, q, mname, S, W)
        assert max_err(out, ref) <= TOL[kv], call
        assert lse_err(lse, o_lse) <= 2e-3


def test_static_scratch_rejects_oversized_request():
    lens = (20000,) * 3
    wl = workloads.small("bf16", lens=lens, seed=91)
    tw = Twin(wl, sum((L + 15) // 16 for L in lens), 3, 1300, seed=2)
    ids = fill_sequences(tw, lens)
    q = workloads.queries(wl).cuda()
    out = torch.empty_like(q)
    lse = torch.empty((3, wl.n_heads), device="cuda")
    with pytest.raises(_abi.PKVError) as e:
        _call_static(tw.cache, ids, q, out, lse, num_splits=1200)  # 3 x 8 x 1200 partial records
    assert e.value.status == 9 and "static scratch" in str(e.value)
