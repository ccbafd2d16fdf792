"""GPU parity of CPU swap: sequences move between the device pool and a
pinned host pool by block copies (one kernel per call that reads or writes
the host pool through its device-mapped address).  Host and device bytes,
tables and free counts must equal the oracle's after every move, and decode
before, during and after must match it."""
import numpy as np
import pytest
import torch

import workloads
from harness import TOL, Twin, fill_sequences, lse_err, max_err, pool_bytes_equal

pytestmark = pytest.mark.gpu


def _host_bytes_equal(tw: Twin, ids):
    c, pool = tw.cache, tw.pool
    pairs = [(c.host_k, pool.hk), (c.host_v, pool.hv)]
    if pool.hk_scale is not None:
        pairs += [(c.host_k_scale, pool.hk_scale), (c.host_v_scale, pool.hv_scale)]
    for dt, ht in pairs:
        d = dt.contiguous().view(torch.uint8).reshape(pool.NH, tw.wl.n_kv_heads, 16, -1).numpy()
        h = ht.view(np.uint8).reshape(pool.NH, tw.wl.n_kv_heads, 16, -1)
        for s in ids:
            L = tw.alloc.length(s)
            for lb, hb in enumerate(tw.alloc.host_table(s)):
                if hb >= 0:
                    n = min(16, L - 16 * lb)
                    assert np.array_equal(d[hb, :, :n], h[hb, :, :n]), (s, lb, hb)


def _state_equal(tw: Twin, ids):
    for s in ids:
        assert tw.cache.swapped(s) == tw.alloc.swapped(s)
        assert np.array_equal(tw.cache.block_table(s), tw.alloc.table(s))
        if tw.alloc.swapped(s):
            assert np.array_equal(tw.cache.host_block_table(s), tw.alloc.host_table(s))
    assert tw.cache.stats()["free_blocks"] == tw.alloc.num_free()
    assert tw.cache.host_free_blocks() == tw.alloc.num_host_free()


def _decode_equal(tw: Twin, wl, ids, step):
    q = workloads.queries(wl, n=len(ids), step=step)
    out, lse = tw.cache.decode(ids, q.cuda(), scale=wl.scale)
    tw.cache.sync_status()
    ref, ref_lse, _ = tw.oracle_decode(ids, q)
    assert max_err(out, ref) <= TOL[wl.kv_dtype]
    assert lse_err(lse, ref_lse) <= 2e-3


@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
def test_swap_out_and_in(kv):
    """Swap out a forked parent (its fork stays), a fork pair together (their
    shared blocks go out once) and a lone sequence; decode and append on the
    rest; swap back in two calls; everything must equal the oracle."""
    wl = workloads.small(kv, lens=(1000, 333, 17, 64, 700), seed=88)
    tw = Twin(wl, 320, 12, 80, seed=7)
    ids = fill_sequences(tw, wl.lens)
    f0, f1 = tw.fork(ids[0]), tw.fork(ids[1])
    k, v = workloads.new_tokens(wl, 2, 0)
    tw.append([ids[0], f1], k, v)  # copy-on-write of shared partial last blocks
    everyone = ids + [f0, f1]
    tw.swap_space(200)
    out = [ids[0], f1, ids[1], ids[3]]
    pairs = tw.swap_out(out)
    # f1 and ids[1] share all but one block: those go to the host once
    assert len(pairs) < sum((tw.alloc.length(s) + 15) // 16 for s in out)
    tw.cache.sync_status()
    _state_equal(tw, everyone)
    _host_bytes_equal(tw, out)
    stay = [s for s in everyone if s not in out]
    pool_bytes_equal(tw, stay)
    _decode_equal(tw, wl, stay, step=1)
    with pytest.raises(Exception) as e:  # device work refuses a swapped-out sequence
        tw.cache.decode([ids[0]], workloads.queries(wl, n=1).cuda(), scale=wl.scale)
    assert getattr(e.value, "status", None) == 1
    # the freed device blocks are reused while the others are out
    k, v = workloads.new_tokens(wl, len(stay), 2)
    tw.append(stay, k, v)
    k, v = workloads.kv_rows(wl, 99, 0, 200)
    extra = tw.add()
    tw.append([extra], k[None], v[None])
    stay.append(extra)
    everyone.append(extra)
    _decode_equal(tw, wl, stay, step=2)
    tw.swap_in([f1, ids[0]])
    tw.swap_in([ids[1], ids[3]])
    tw.cache.sync_status()
    _state_equal(tw, everyone)
    pool_bytes_equal(tw, everyone)
    _decode_equal(tw, wl, everyone, step=3)
    # and once more, with appends after the round trip
    k, v = workloads.new_tokens(wl, len(everyone), 4)
    tw.append(everyone, k, v)
    _decode_equal(tw, wl, everyone, step=4)


def test_swap_refusals_leave_state_unchanged():
    wl = workloads.small("bf16", lens=(100, 50), seed=89)
    tw = Twin(wl, 40, 4, 16, seed=2)
    ids = fill_sequences(tw, wl.lens)
    tw.swap_space(8)  # 100 + 50 tokens need 7 + 4 host blocks
    with pytest.raises(Exception) as e:
        tw.cache.swap_out(ids)
    assert getattr(e.value, "status", None) == 3
    _state_equal(tw, ids)
    tw.swap_out(ids[:1])
    tw.cache.sync_status()
    with pytest.raises(Exception) as e:
        tw.cache.swap_out(ids[:1])
    assert getattr(e.value, "status", None) == 1
    _state_equal(tw, ids)
    _host_bytes_equal(tw, ids[:1])
    tw.free(ids[0])  # a swapped-out sequence gives its host blocks back
    assert tw.cache.host_free_blocks() == tw.alloc.num_host_free() == 8
