"""GPU parity of shared-prefix (cascade) decode: sequences that share leading
blocks through forks are paired, and each pair's shared blocks are read once
for both.  Outputs, lse and logits must match the oracle exactly as without
pairing (within the same tolerances), for BF16 and FP8 KV and every GQA
group size, in the allocating and the static-scratch entry points."""
import numpy as np
import pytest
import torch

import workloads
from harness import TOL, Twin, lse_err, max_err

pytestmark = pytest.mark.gpu


def _shared_batch(kv: str, n_heads: int, seed: int, head_dim: int = 128):
    """Three prefix groups (100, 37 and 512 tokens) forked into children
    with private suffixes; some children forked again with no new token
    (tables identical up to the partial last block); one unrelated sequence,
    one of 5 tokens and one empty.  Then one token is appended to every
    non-empty sequence, which copies each shared partial last block."""
    wl = workloads.small(kv, lens=(1,), n_heads=n_heads, head_dim=head_dim, seed=seed)
    tw = Twin(wl, 900, 40, 80, seed=seed)
    rng = np.random.default_rng(seed)
    key = 0
    ids = []

    def put(s, t0, n):
        nonlocal key
        k, v = workloads.kv_rows(wl, key, t0, n)
        key += 1
        tw.append([s], k[None], v[None])

    for prefix, kids in ((100, 5), (37, 3), (512, 6)):
        holder = tw.add()
        put(holder, 0, prefix)
        children = [tw.fork(holder) for _ in range(kids)]
        tw.free(holder)
        for j, s in enumerate(children):
            if j % 3 != 2:
                put(s, prefix, int(rng.integers(1, 300)))
        ids += children
        ids += [tw.fork(children[0]), tw.fork(children[1])]
    lone = tw.add()
    put(lone, 0, 700)
    short = tw.add()
    put(short, 0, 5)
    empty = tw.add()
    ids += [lone, short, empty]
    live = [s for s in ids if tw.alloc.length(s) > 0]
    k, v = workloads.new_tokens(wl, len(live), 3)
    tw.append(live, k, v)
    return wl, tw, sorted(ids)


def _decode_both(tw, wl, ids, cascade, static: bool = False, logits: bool = False):
    tw.cache.set_cascade(cascade)
    q = workloads.queries(wl, n=len(ids), step=2)
    stride = max(tw.alloc.length(s) for s in ids)
    lg = torch.full((len(ids), wl.n_kv_heads, stride, wl.group), 7.0, device="cuda") if logits else None
    fn = tw.cache.decode_static if static else tw.cache.decode
    out, lse = fn(ids, q.cuda(), scale=wl.scale, logits=lg, logits_stride=stride if logits else 0)
    tw.cache.sync_status()
    ref, ref_lse, ref_lg = tw.oracle_decode(ids, q, want_logits=logits, logits_stride=stride if logits else None)
    assert max_err(out, ref) <= TOL[wl.kv_dtype]
    assert lse_err(lse, ref_lse) <= 2e-3
    if logits:
        # [n][Hk][stride][G] -> [n][H][stride], the oracle's layout
        got = lg.permute(0, 1, 3, 2).reshape(len(ids), wl.n_heads, stride).cpu().numpy().astype(np.float64)
        for b, s in enumerate(ids):
            L = tw.alloc.length(s)
            if L:
                assert np.abs(got[b, :, :L] - ref_lg[b, :, :L]).max() <= 2e-3, b
    return out


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("kv", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("n_heads", [64, 32, 16, 8])
def test_cascade_matches_oracle(kv, n_heads, D):
    """Mode 2: group prefixes (BF16, head_dim 128) and pairs; mode 1: pairs
    only; 0: off."""
    wl, tw, ids = _shared_batch(kv, n_heads, seed=90 + n_heads, head_dim=D)
    groups = _decode_both(tw, wl, ids, cascade=2)
    pairs = _decode_both(tw, wl, ids, cascade=1)
    off = _decode_both(tw, wl, ids, cascade=0)
    for x in (groups, pairs):
        assert max_err(x, off.float().cpu().numpy()) <= 2 * TOL[kv]


@pytest.mark.parametrize("n_heads", [64, 32])
def test_cascade_logits_and_static_entry(n_heads):
    wl, tw, ids = _shared_batch("bf16", n_heads, seed=97)
    _decode_both(tw, wl, ids, cascade=2, logits=True)
    _decode_both(tw, wl, ids, cascade=2, static=True)
    _decode_both(tw, wl, ids, cascade=1, logits=True)


@pytest.mark.parametrize("n_heads", [64, 32, 16, 8])
def test_group_prefix_only(n_heads):
    """Forty sequences that are the same 700-token prefix plus one private
    token each: the group prefix (43 full blocks) is the multi-query kernel's
    whole work but for one block per sequence; 40 x G rows span several row
    tiles for small G."""
    wl = workloads.small("bf16", lens=(1,), n_heads=n_heads, seed=99)
    tw = Twin(wl, 600, 48, 60, seed=5)
    base = tw.add()
    k, v = workloads.kv_rows(wl, 0, 0, 700)
    tw.append([base], k[None], v[None])
    ids = [tw.fork(base) for _ in range(40)]
    tw.free(base)
    k, v = workloads.new_tokens(wl, len(ids), 6)
    tw.append(ids, k, v)
    _decode_both(tw, wl, ids, cascade=2)
    _decode_both(tw, wl, ids, cascade=2, logits=True)


def test_cascade_identical_forks_share_everything():
    """Forks with no new token have identical tables: the pair covers every
    full block, and a length that is a multiple of 16 leaves no remainder."""
    wl = workloads.small("bf16", lens=(1,), n_heads=64, seed=98)
    tw = Twin(wl, 200, 8, 40, seed=3)
    base = tw.add()
    k, v = workloads.kv_rows(wl, 0, 0, 320)
    tw.append([base], k[None], v[None])
    ids = [base] + [tw.fork(base) for _ in range(4)]
    _decode_both(tw, wl, ids, cascade=True)
