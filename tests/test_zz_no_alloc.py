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
from harness import TOL, Twin, fill_sequences, lse_err
from paged_kv_cache_282_gb300 import _abi

pytestmark = pytest.mark.gpu


def _call_static(cache, ids, q, out, lse, num_splits, mask=0, S=0, W=0):
    arr = np.ascontiguousarray(ids, dtype=np.int32)
    st = cache.lib.pkv_decode_attn_static(cache.handle, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                          arr.size, arr.ctypes.data_as(ctypes.c_void_p), q.data_ptr(),
                                          1.0 / np.sqrt(cache.head_dim), mask, S, W, num_splits, out.data_ptr(),
                                          lse.data_ptr(), None, 0)
    _abi.check(st)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_static_scratch_matches_workspace_decode(kv):
    lens = (1, 16, 17, 300, 1000, 2049, 4000)
    wl = workloads.small(kv, lens=lens, seed=90)
    tw = Twin(wl, sum((L + 15) // 16 for L in lens) + 4, len(lens), 300, seed=6)
    ids = fill_sequences(tw, lens)
    cache = tw.cache
    # two calls in a row, with different queries, split counts and keep-sets
    for call, (splits, mask, S, W) in enumerate([(0, 0, 0, 0), (5, 2, 4, 700)]):
        q = workloads.queries(wl, step=call).cuda()
        ref_out, ref_lse = cache.decode(ids, q, mask=["full", "sliding", "sink_window"][mask], num_sinks=S,
                                        window=W, num_splits=splits)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((len(ids), wl.n_heads), float("nan"), device="cuda")
        _call_static(cache, ids, q, out, lse, splits, mask, S, W)
        cache.sync_status()
        assert torch.isfinite(out.float()).all()
        err = (out.float() - ref_out.float()).abs().max().item()
        assert err <= TOL[kv], (call, err)
        assert lse_err(lse, ref_lse.cpu().numpy().astype(np.float64)) <= 2e-3


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
