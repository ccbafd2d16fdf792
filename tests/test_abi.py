"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/pkv.h, and its host allocator replays bit-exactly
against the oracle's allocator (same seeds, same operations)."""
import os
import random
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_282_gb300 import build
    build.build()
    import paged_kv_cache_282_gb300 as m
    m.load()
    return m


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(pkv):
    names = _declared_functions()
    assert len(names) >= 20
    lib = pkv.load()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pkv._abi.SIGNATURES), "binding and header disagree"
    assert b"sm_103a" in lib.pkv_version()


def test_required_bytes(pkv):
    import ctypes
    from paged_kv_cache_282_gb300 import _abi
    cfg = _abi.pkv_pool_config(100, 16, 32, 8, 128, 4, 64, 2, 0, None)
    sz = _abi.pkv_buffer_sizes()
    _abi.check(pkv.load().pkv_pool_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)))
    assert sz.k_pool == 100 * 8 * 16 * 128 and sz.k_scale == 100 * 8 * 16 * 4
    assert sz.block_tables == 4 * 64 * 4 and sz.status == 16


def test_required_bytes_int8(pkv):
    import ctypes
    from paged_kv_cache_282_gb300 import _abi
    cfg = _abi.pkv_pool_config(100, 16, 32, 8, 128, 4, 64, 3, 0, None)
    sz = _abi.pkv_buffer_sizes()
    _abi.check(pkv.load().pkv_pool_required_bytes(ctypes.byref(cfg), ctypes.byref(sz)))
    assert sz.k_pool == 100 * 8 * 16 * 128 and sz.k_scale == 100 * 8 * 16 * 4


@pytest.mark.parametrize("bad", [dict(block_size=8), dict(n_heads=24, n_kv_heads=8),
                                 dict(head_dim=96), dict(kv_dtype=7)])
def test_config_rejected(pkv, bad):
    import ctypes
    from paged_kv_cache_282_gb300 import _abi
    kw = dict(num_blocks=10, block_size=16, n_heads=32, n_kv_heads=8, head_dim=128, max_seqs=2,
              max_blocks_per_seq=4, kv_dtype=1, alloc_seed=0, free_order=None)
    kw.update(bad)
    cfg = _abi.pkv_pool_config(**kw)
    h = ctypes.c_void_p()
    st = pkv.load().pkv_pool_create(ctypes.byref(cfg), None, ctypes.byref(h))
    assert st in (1, 2)
    assert pkv.load().pkv_last_error()


def test_host_only_pool_refuses_device_work(pkv):
    c = pkv.PagedKVCache(8, 4, 2, 64, 2, 4, kv_dtype="fp32", host_only=True)
    s = c.seq_add()
    with pytest.raises(pkv.PKVError) as e:
        c.decode.__func__  # noqa: B018 (bound method exists)
        import ctypes
        ids = np.array([s], dtype=np.int32)
        pkv._abi.check(c.lib.pkv_decode_attn(c.handle, None, 1, ids.ctypes.data_as(ctypes.c_void_p), None, 1.0,
                                             0, 0, 0, 0, None, None, None, 0, None, 0))
    assert e.value.status == 8


def test_page_layout_example_via_library(pkv):
    order = [7, 12, 3, 5, 8, 1, 2, 0, 9, 4, 6, 10, 11, 13, 14, 15]
    c = pkv.PagedKVCache(16, 4, 2, 64, 4, 8, kv_dtype="fp32", free_order=order, host_only=True)
    got = {}
    for name, L in (("A", 35), ("B", 10), ("C", 70)):
        s = c.seq_add()
        c.reserve_slots([s], L)
        got[name] = c.block_table(s).tolist()
    assert got == {"A": [7, 12, 3], "B": [5], "C": [8, 1, 2, 0, 9]}


def _replay(pkv, seed):
    rng = random.Random(seed)
    NB = rng.randint(8, 80)
    aseed = rng.randint(0, 2 ** 63)
    lib = pkv.PagedKVCache(NB, 4, 2, 64, 10, 48, kv_dtype="fp32", alloc_seed=aseed, host_only=True)
    ora = oracle.OracleAllocator(NB, 10, 48, seed=aseed)
    NH = rng.randint(4, 80)
    lib.swap_space(NH)
    ora.set_swap_space(NH)
    seqs = []  # every live sequence, swapped out or not
    for op in range(150):
        if seqs and rng.random() < 0.12:
            out = rng.random() < 0.5
            cand = [s for s in seqs if ora.swapped(s) != out]
            if cand:
                ids = rng.sample(cand, rng.randint(1, len(cand)))
                try:
                    (lib.swap_out if out else lib.swap_in)(ids)
                    ok = True
                except pkv.PKVError as e:
                    ok = e.status
                try:
                    ora.swap_out(ids) if out else ora.swap_in(ids)
                    ok2 = True
                except MemoryError:
                    ok2 = 3
                assert ok == ok2
                if out and ok is True:  # device-side operations refuse it
                    for call in (lambda: lib.reserve_slots(ids[:1], 1), lambda: lib.seq_fork(ids[0]),
                                 lambda: lib.seq_truncate(ids[0], 0), lambda: lib.seq_evict(ids[0], 1, 4),
                                 lambda: lib.seq_compact(ids[:1], [0])):
                        with pytest.raises(pkv.PKVError) as e:
                            call()
                        assert e.value.status == 1
            continue
        live = [s for s in seqs if not ora.swapped(s)]
        r = rng.random()
        if r < 0.15 or not live:
            try:
                a = lib.seq_add()
            except pkv.PKVError as e:
                assert e.status == 4
                with pytest.raises(RuntimeError):
                    ora.seq_add()
                continue
            assert a == ora.seq_add()
            seqs.append(a)
        elif r < 0.65:
            ids = rng.sample(live, rng.randint(1, len(live)))
            T = rng.randint(1, 24)
            try:
                s1, c1 = lib.reserve_slots(ids, T)
                ok = True
            except pkv.PKVError as e:
                ok = e.status
            try:
                s2, c2 = ora.append(ids, T)
                ok2 = True
            except MemoryError:
                ok2 = 3
            except ValueError:
                ok2 = 1
            assert ok == ok2
            if ok is True:
                assert np.array_equal(s1, s2) and np.array_equal(c1, c2)
        elif r < 0.75:
            s = rng.choice(live)
            try:
                d = lib.seq_fork(s)
            except pkv.PKVError as e:
                assert e.status == 4
                with pytest.raises(ValueError):
                    ora.fork(s)
                continue
            assert d == ora.fork(s)
            seqs.append(d)
        elif r < 0.85:
            s = rng.choice(seqs)  # swapped-out sequences can be freed too
            lib.seq_free(s)
            ora.free(s)
            seqs.remove(s)
        elif r < 0.91:
            s = rng.choice(live)
            S, W = rng.randint(0, 5), rng.randint(1, 40)
            lib.seq_evict(s, S, W)
            ora.evict(s, S, W)
        elif r < 0.96:
            ids = rng.sample(live, rng.randint(1, len(live)))
            counts = [rng.randint(0, lib.seq_len(s)) for s in ids]
            try:
                lib.seq_compact(ids, counts)
                ok = True
            except pkv.PKVError as e:
                ok = e.status
            try:
                ora.compact(ids, counts)
                ok2 = True
            except MemoryError:
                ok2 = 3
            assert ok == ok2
        else:
            s = rng.choice(live)
            n = rng.randint(0, lib.seq_len(s))
            try:
                lib.seq_truncate(s, n)
                ok = True
            except pkv.PKVError:
                ok = False
            try:
                ora.truncate(s, n)
                ok2 = True
            except ValueError:
                ok2 = False
            assert ok == ok2
        for s in seqs:
            assert lib.seq_len(s) == ora.length(s)
            assert np.array_equal(lib.block_table(s), ora.table(s)), (seed, op, s)
            assert lib.swapped(s) == ora.swapped(s)
            if ora.swapped(s):
                assert np.array_equal(lib.host_block_table(s), ora.host_table(s)), (seed, op, s)
        st = lib.stats()
        assert st["free_blocks"] == ora.num_free()
        assert lib.host_free_blocks() == ora.num_host_free()
        assert st["shared_blocks"] == sum(1 for b in range(NB) if ora.refcount(b) > 1)


@pytest.mark.parametrize("seed", range(12))
def test_allocator_matches_oracle_replay(pkv, seed):
    """Random adds, appends (with copy-on-write), forks, frees, evictions,
    H2O compactions, truncations and CPU swaps, the same on both sides."""
    _replay(pkv, seed)


def test_workload_sized_pool_tables_match_oracle(pkv):
    """The pool of the Llama-3-8B-shaped batch: a seeded permutation of a pool
    sized to fit exactly; every table entry must agree with the oracle."""
    import workloads
    wl = workloads.llama3_8b_batch64()
    nb = sum((L + 15) // 16 for L in wl.lens)
    lib = pkv.PagedKVCache(nb, 32, 8, 128, 64, 512, kv_dtype="bf16", alloc_seed=wl.seed, host_only=True)
    ora = oracle.OracleAllocator(nb, 64, 512, seed=wl.seed)
    for L in wl.lens:
        a, b = lib.seq_add(), ora.seq_add()
        s1, _ = lib.reserve_slots([a], L)
        s2, _ = ora.append([b], L)
        assert np.array_equal(s1, s2)
    assert lib.stats()["free_blocks"] == 0
    with pytest.raises(pkv.PKVError) as e:
        lib.reserve_slots([0], 16)
    assert e.value.status == 3


def test_truncate_many_matches_single_truncates(pkv):
    rng = random.Random(77)
    lib = pkv.PagedKVCache(200, 4, 2, 64, 8, 40, kv_dtype="fp32", alloc_seed=3, host_only=True)
    ora = oracle.OracleAllocator(200, 8, 40, seed=3)
    ids = [lib.seq_add() for _ in range(6)]
    for s in ids:
        assert ora.seq_add() == s
        L = rng.randint(1, 300)
        lib.reserve_slots([s], L)
        ora.append([s], L)
    ids.append(lib.seq_fork(ids[0]))
    assert ora.fork(ids[0]) == ids[-1]
    new = [rng.randint(0, lib.seq_len(s)) for s in ids]
    lib.seq_truncate_many(ids, new)
    for s, L in zip(ids, new):
        ora.truncate(s, L)
    for s in ids:
        assert np.array_equal(lib.block_table(s), ora.table(s))
    assert lib.stats()["free_blocks"] == ora.num_free()
    with pytest.raises(pkv.PKVError):  # duplicates are refused before anything changes
        lib.seq_truncate_many([ids[0], ids[0]], [0, 0])
    assert lib.seq_len(ids[0]) == new[0]


def test_compaction_refusals_leave_state_unchanged(pkv):
    lib = pkv.PagedKVCache(10, 4, 2, 64, 4, 8, kv_dtype="fp32", alloc_seed=5, host_only=True)
    a, b = lib.seq_add(), lib.seq_add()
    lib.reserve_slots([a], 64)
    lib.reserve_slots([b], 40)
    before = (lib.block_table(a).tolist(), lib.block_table(b).tolist(), lib.stats()["free_blocks"])
    for ids, counts, status in (([a, b], [64, 40], 3),   # 7 fresh blocks, 3 free
                                ([a, a], [1, 1], 1),     # listed twice
                                ([a], [65], 1),          # more than the length
                                ([3], [0], 1)):          # not a live sequence
        with pytest.raises(pkv.PKVError) as e:
            lib.seq_compact(ids, counts)
        assert e.value.status == status
        assert (lib.block_table(a).tolist(), lib.block_table(b).tolist(), lib.stats()["free_blocks"]) == before
    lib.seq_compact([b], [17])
    assert lib.seq_len(b) == 17 and len(lib.block_table(b)) == 2


def _plan(pkv, c, ids, mode, S, W, splits, general):
    import ctypes
    buf = ctypes.create_string_buffer(16 << 20)
    size = ctypes.c_size_t()
    info = (ctypes.c_int32 * 9)()
    arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    pkv._abi.check(c.lib.pkv_test_plan_bytes(c._h, arr.size, arr.ctypes.data_as(ctypes.c_void_p), mode, S, W, splits,
                                             general, buf, len(buf), ctypes.byref(size), info))
    return buf.raw[: size.value], tuple(info)


@pytest.mark.parametrize("seed", range(8))
def test_one_pass_planner_matches_general_planner(pkv, seed):
    """The one-pass decode planner (one sequence per warp; sequence pairs)
    writes the same plan bytes as the general planner: random batches with
    empty and short sequences, forked pairs with private suffixes, every mask,
    two GQA widths and both warp geometries."""
    rng = random.Random(seed)
    Hk = (2, 8)[seed % 2]
    c = pkv.PagedKVCache(60000, Hk * 4, Hk, 128, 300, 1300, host_only=True, alloc_seed=seed)
    pkv._abi.check(c.lib.pkv_test_set_geometry(c._h, 152, 16 if seed % 3 == 0 else 12, 12, 4))
    ids = []
    if seed % 2:  # parents forked once, then private suffixes on some of each
        for _ in range(rng.randint(2, 40)):
            s = c.seq_add()
            c.reserve_slots([s], rng.randint(1, 3000))
            f = c.seq_fork(s)
            ids += [s, f]
            for x in (s, f):
                if rng.random() < 0.7:
                    c.reserve_slots([x], rng.randint(1, 700))
    else:
        for _ in range(rng.randint(1, 150)):
            s = c.seq_add()
            L = 0 if rng.random() < 0.1 else rng.randint(1, 9000 if rng.random() < 0.8 else 40)
            if L:
                c.reserve_slots([s], L)
            ids.append(s)
    pairs_seen = False
    for mode, S, W in [(0, 0, 0), (1, 0, rng.randint(0, 3000)), (2, rng.randint(0, 40), rng.randint(0, 3000)),
                       (2, 0, 0)]:
        fast, info = _plan(pkv, c, ids, mode, S, W, 0, 0)
        general, ginfo = _plan(pkv, c, ids, mode, S, W, 0, 1)
        assert info == ginfo and fast == general, (mode, S, W)
        pairs_seen |= info[3] == 2
    assert pairs_seen == bool(seed % 2)


@pytest.mark.parametrize("spare", [0, 1])
def test_append_to_shared_block_needs_one_copy_fewer_than_sharers(pkv, spare):
    """Four sequences share a part-filled block. When all four append in one
    call, three copy it and the last one finds it its own: the call needs
    three free blocks, not four. One block fewer refuses it, with nothing
    changed; library and oracle agree either way."""
    free_after_forks = 3 - 1 + spare          # 2 (refused) or 3 (fits)
    nb = 2 + free_after_forks                 # 17 tokens take 2 blocks
    lib = pkv.PagedKVCache(nb, 4, 2, 64, 8, 8, kv_dtype="fp32", alloc_seed=9, host_only=True)
    ora = oracle.OracleAllocator(nb, 8, 8, seed=9)
    a = lib.seq_add()
    assert ora.seq_add() == a
    lib.reserve_slots([a], 17)
    ora.append([a], 17)
    ids = [a]
    for _ in range(3):
        ids.append(lib.seq_fork(a))
        assert ora.fork(a) == ids[-1]
    assert lib.stats()["free_blocks"] == ora.num_free() == free_after_forks
    tables = [lib.block_table(s).tolist() for s in ids]
    if spare:
        s1, c1 = lib.reserve_slots(ids, 1)
        s2, c2 = ora.append(ids, 1)
        assert np.array_equal(s1, s2) and np.array_equal(c1, c2) and len(c1) == 3
        for s in ids:
            assert np.array_equal(lib.block_table(s), ora.table(s))
        assert lib.stats()["free_blocks"] == ora.num_free() == 0
    else:
        with pytest.raises(pkv.PKVError) as e:
            lib.reserve_slots(ids, 1)
        assert e.value.status == 3
        with pytest.raises(MemoryError):
            ora.append(ids, 1)
        assert [lib.block_table(s).tolist() for s in ids] == tables
        assert [lib.seq_len(s) for s in ids] == [17] * 4
    with pytest.raises(pkv.PKVError) as e:  # a sequence listed twice
        lib.reserve_slots([ids[1], ids[1]], 1)
    assert e.value.status == 1


# The uploaded plan's records, as laid out by the library (see the test
# hook's declaration): int32 fields in declaration order.
_PIECE = np.dtype([(f, "<i4") for f in ("seq_slot", "q_row", "kv_head", "lo", "hi", "ctx_len", "out_index", "flags",
                                        "q_row1", "out_index1", "item1", "stream_from")])
_COMBINE = np.dtype([(f, "<i4") for f in ("q_row", "kv_head", "first", "n")])
_EMPTY = np.dtype([(f, "<i4") for f in ("q_row", "kv_head")])
_PITEM = np.dtype([(f, "<i4") for f in ("kv_head", "table_seq", "lo", "hi", "member_begin", "n_members", "p0", "p1")])
_PMEMBER = np.dtype([(f, "<i4") for f in ("q_row", "out_index", "item", "pad")])


def _parse_plan(raw, info):
    warps, _, _, _, n_pieces, n_combine, n_empty, n_items, n_members = info
    up = lambda x: (x + 31) & ~31  # noqa: E731
    off = {"wb": 0}
    off["pieces"] = up(4 * (warps + 1))
    off["combine"] = up(off["pieces"] + n_pieces * _PIECE.itemsize)
    off["counters"] = up(off["combine"] + n_combine * _COMBINE.itemsize)
    off["empty"] = up(off["counters"] + 4 * n_combine)
    off["pitems"] = up(off["empty"] + n_empty * _EMPTY.itemsize)
    off["pmembers"] = up(off["pitems"] + n_items * _PITEM.itemsize)
    assert len(raw) == off["pmembers"] + n_members * _PMEMBER.itemsize
    arr = lambda dt, key, cnt: np.frombuffer(raw, dtype=dt, count=cnt, offset=off[key])  # noqa: E731
    return (arr("<i4", "wb", warps + 1), arr(_PIECE, "pieces", n_pieces), arr(_COMBINE, "combine", n_combine),
            arr("<i4", "counters", n_combine), arr(_EMPTY, "empty", n_empty), arr(_PITEM, "pitems", n_items),
            arr(_PMEMBER, "pmembers", n_members))


def _check_plan(c, ids, Hk, mode, S, W, splits, raw, info, wpc):
    """What any decode plan must satisfy, stated from the keep-sets alone:
    every kept logical block of every (sequence, kv head) is read exactly
    once (by a piece of the sequence, as the second sequence of a pair whose
    table holds the same physical blocks, or by a group prefix all of whose
    members hold them); each (sequence, kv head) either writes its output
    directly from one run or has one merge item whose records are written
    exactly once; runs end at warp ends; stream-K warps differ by at most one
    block of work."""
    wb, pieces, combine, counters, empty, pitems, pmembers = _parse_plan(raw, info)
    n = len(ids)
    lens = [c.seq_len(s) for s in ids]
    tables = [c.block_table(s) for s in ids]
    assert info[0] == len(wb) - 1 and (info[0] == 0 or info[0] == info[1] * wpc)
    assert wb[0] == 0 and wb[-1] == len(pieces) and np.all(np.diff(wb) >= 0)
    assert not counters.any()
    item_of = {(int(ci["q_row"]), int(ci["kv_head"])): k for k, ci in enumerate(combine)}
    assert len(item_of) == len(combine)
    spans = sorted((int(ci["first"]), int(ci["n"])) for ci in combine)
    assert all(nn >= 1 for _, nn in spans)
    assert [f for f, _ in spans] == list(np.cumsum([0] + [nn for _, nn in spans])[:-1])
    assert sum(nn for _, nn in spans) == info[2]
    # blocks read once by the call (no other holder, or only the pair): a
    # piece's stream_from starts the longest tail of its segment held by at
    # most that many sequences, counted over the listed sequences' tables
    # (every live sequence is listed); with no block held twice it is the
    # segment's start
    holders = {}
    for t in tables:
        for blk in t[t >= 0].tolist():
            holders[blk] = holders.get(blk, 0) + 1
    any_shared = any(v > 1 for v in holders.values())
    for pc in pieces:
        limit = 2 if pc["q_row1"] >= 0 else 1
        row = tables[int(pc["q_row"])]
        sf = int(pc["stream_from"])
        for lb in range(max(sf, int(pc["lo"])), int(pc["hi"])):
            assert holders[int(row[lb])] <= limit, (lb, sf)
        if any_shared and int(pc["lo"]) <= sf - 1 < int(pc["hi"]):
            assert holders[int(row[sf - 1])] > limit, (sf, int(pc["lo"]))
        if not any_shared:
            assert sf <= int(pc["lo"])
    read = {(b, g): [] for b in range(n) for g in range(Hk)}
    written = {(b, g): [] for b in range(n) for g in range(Hk)}
    direct = {(b, g): 0 for b in range(n) for g in range(Hk)}
    for w in range(len(wb) - 1):
        run = []
        units = 0
        for pc in pieces[wb[w]:wb[w + 1]]:
            b, g = int(pc["q_row"]), int(pc["kv_head"])
            assert pc["seq_slot"] == ids[b] and pc["ctx_len"] == lens[b] and pc["lo"] < pc["hi"]
            blocks = list(range(int(pc["lo"]), int(pc["hi"])))
            units += len(blocks)
            assert all(tables[b][blocks] >= 0)
            read[(b, g)] += blocks
            if pc["q_row1"] >= 0:
                b1 = int(pc["q_row1"])
                assert np.array_equal(tables[b1][blocks], tables[b][blocks])
                read[(b1, g)] += blocks
            run.append(pc)
            if not pc["flags"] & 1:
                continue
            key = {(int(x["q_row"]), int(x["kv_head"]), int(x["q_row1"]), int(x["out_index"]), int(x["out_index1"]),
                    int(x["flags"]) >> 1, int(x["item1"])) for x in run}
            assert len(key) == 1, "a run's pieces share sequence, head and records"
            if pc["out_index"] >= 0:
                assert pc["flags"] >> 1 == item_of[(b, g)]
                written[(b, g)].append(int(pc["out_index"]))
            else:
                direct[(b, g)] += 1
            if pc["q_row1"] >= 0:
                b1 = int(pc["q_row1"])
                assert pc["out_index1"] >= 0 and pc["item1"] == item_of[(b1, g)]
                written[(b1, g)].append(int(pc["out_index1"]))
            run = []
        assert not run, "a warp's last piece ends its run"
    for it in pitems:
        g, lo, hi = int(it["kv_head"]), int(it["lo"]), int(it["hi"])
        members = pmembers[int(it["member_begin"]):int(it["member_begin"]) + int(it["n_members"])]
        assert len(members) == it["n_members"] > 0 and lo < hi
        ref = c.block_table(int(it["table_seq"]))[lo:hi]
        for m in members:
            b = int(m["q_row"])
            assert np.array_equal(tables[b][lo:hi], ref) and all(ref >= 0)
            assert m["item"] == item_of[(b, g)]
            read[(b, g)] += list(range(lo, hi))
            written[(b, g)].append(int(m["out_index"]))
    empties = {(int(e["q_row"]), int(e["kv_head"])) for e in empty}
    assert len(empties) == len(empty)
    for b in range(n):
        kept = sorted({j // 16 for j in oracle.keep_set(lens[b], mode, S, W)})
        for g in range(Hk):
            assert sorted(read[(b, g)]) == kept, (b, g)
            assert ((b, g) in empties) == (not kept)
            if (b, g) in item_of:
                ci = combine[item_of[(b, g)]]
                assert direct[(b, g)] == 0
                assert sorted(written[(b, g)]) == list(range(int(ci["first"]), int(ci["first"]) + int(ci["n"])))
                if splits > 0:
                    assert ci["n"] == min(splits, len(kept))
            elif kept:
                assert direct[(b, g)] == 1 and not written[(b, g)]
    if splits == 0 and not len(pitems):
        per_warp = [sum(int(x["hi"] - x["lo"]) for x in pieces[wb[w]:wb[w + 1]]) for w in range(len(wb) - 1)]
        busy = [u for u in per_warp if u]
        assert not busy or max(busy) - min(busy) <= 1


@pytest.mark.parametrize("seed", range(10))
def test_decode_plans_read_every_kept_block_once(pkv, seed):
    """Plans from both planner paths, checked against the keep-sets: random
    batches (empty, short and long sequences; forks with private suffixes;
    streaming eviction matching the mask), every mask, explicit splits,
    sequence pairs and, on some seeds, group prefixes."""
    rng = random.Random(100 + seed)
    Hk = (2, 8)[seed % 2]
    wpc, wpc2 = (16, 12) if seed % 3 == 0 else (12, 12)
    c = pkv.PagedKVCache(60000, Hk * 4, Hk, 128, 300, 1300, kv_dtype="bf16", host_only=True, alloc_seed=seed)
    pkv._abi.check(c.lib.pkv_test_set_geometry(c._h, 152 if seed % 4 else 7, wpc, wpc2, 4))
    if seed % 5 == 4:
        c.set_cascade(2)
    ids = []
    for _ in range(rng.randint(1, 30)):
        s = c.seq_add()
        L = 0 if rng.random() < 0.1 else rng.randint(1, 5000 if rng.random() < 0.8 else 40)
        if L:
            c.reserve_slots([s], L)
        ids.append(s)
        for _ in range(rng.choice([0, 0, 1, 5])):  # forks, some with private suffixes
            f = c.seq_fork(s)
            if rng.random() < 0.5:
                c.reserve_slots([f], rng.randint(1, 300))
            ids.append(f)
    rng.shuffle(ids)
    S, W = rng.randint(0, 40), rng.randint(1, 3000)
    evicted = [s for s in ids if rng.random() < 0.2]
    cases = [(0, 0, 0, 0), (0, 0, 0, rng.randint(1, 70)), (1, 0, rng.randint(0, 3000), 0), (1, 0, 500, 16),
             (1, 0, 0, 0), (2, S, W, 0), (2, 0, 0, 0), (2, 5, 0, 0), (2, 0, 7, 3), (2, 17, 15, 0)]
    for mode, s_, w_, splits in cases:
        for general in (0, 1):
            raw, info = _plan(pkv, c, ids, mode, s_, w_, splits, general)
            _check_plan(c, ids, Hk, mode, s_, w_, splits, raw, info, wpc2 if info[3] == 2 else wpc)
    for s in evicted:  # sink + window eviction: the same mask's plans skip the freed blocks
        c.seq_evict(s, S, W)
    for general in (0, 1):
        raw, info = _plan(pkv, c, ids, 2, S, W, 0, general)
        _check_plan(c, ids, Hk, 2, S, W, 0, raw, info, wpc)


def _cow_waves(pkv, c, pairs):
    import ctypes
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1))
    cap = len(pairs) + 2
    out = np.zeros(cap, dtype=np.int32)
    n = ctypes.c_int32()
    pkv._abi.check(c.lib.pkv_test_cow_waves(c._h, len(pairs), arr.ctypes.data, out.ctypes.data, cap, ctypes.byref(n)))
    return out[: n.value].tolist()


def test_copy_waves_run_like_the_queue_in_order(pkv):
    """The queued copy-on-write copies run in waves; the copies of a wave run
    in parallel.  Each wave must be free of conflicts (no copy reads a block
    another one writes, no two write the same block), so that any order
    inside a wave gives what the queue gives one by one; and a wave ends only
    where the next copy conflicts with it."""
    c = pkv.PagedKVCache(12, 4, 2, 64, 4, 4, kv_dtype="fp32", host_only=True)
    # a block freed after it was queued as a source comes back as a destination
    assert _cow_waves(pkv, c, [(3, 5), (7, 3)]) == [0, 1, 2]
    assert _cow_waves(pkv, c, [(3, 5), (5, 6)]) == [0, 1, 2]   # reads an earlier copy's result
    assert _cow_waves(pkv, c, [(3, 5), (4, 5)]) == [0, 1, 2]   # writes an earlier copy's destination
    assert _cow_waves(pkv, c, [(3, 5), (3, 6)]) == [0, 2]      # two reads of one block
    assert _cow_waves(pkv, c, []) == [0, 0]  # one empty wave
    rng = random.Random(7)
    for trial in range(3000):
        n = rng.randint(1, 14)
        pairs = [(rng.randrange(12), rng.randrange(12)) for _ in range(n)]
        pairs = [(a, b) for a, b in pairs if a != b] or [(0, 1)]
        st = _cow_waves(pkv, c, pairs)
        assert st[0] == 0 and st[-1] == len(pairs) and all(x < y for x, y in zip(st, st[1:]))
        blocks = list(range(12))
        for w in range(len(st) - 1):
            wave = pairs[st[w]:st[w + 1]]
            srcs, dsts = [a for a, _ in wave], [b for _, b in wave]
            assert len(set(dsts)) == len(dsts) and not set(dsts) & set(srcs), (pairs, st)
            if w + 1 < len(st) - 1:  # the next wave's first copy conflicts with this wave
                a, b = pairs[st[w + 1]]
                assert a in dsts or b in dsts or b in srcs, (pairs, st)
            # a conflict-free wave: reading everything first, then writing,
            # equals running its copies one by one
            new = blocks.copy()
            for a, b in wave:
                new[b] = blocks[a]
            seq = blocks.copy()
            for a, b in wave:
                seq[b] = seq[a]
            assert new == seq
            blocks = new


def _take_patches(pkv, c, queue=True):
    import ctypes
    cap = 1 << 16
    out = np.zeros(2 * cap, dtype=np.int32)
    n = ctypes.c_int32()
    pkv._abi.check(c.lib.pkv_test_take_patches(c._h, int(queue), out.ctypes.data, cap, ctypes.byref(n)))
    return out[: 2 * n.value].reshape(-1, 2)


@pytest.mark.parametrize("seed", range(6))
def test_table_patches_keep_the_device_table_equal_to_the_host_tables(pkv, seed):
    """The device block table is only ever changed by the queued patches.
    Replaying them in order into a model of it after every allocator call
    (adds, appends with copy-on-write, forks, frees, evictions, truncations,
    compactions, swaps) must give the host tables: a live sequence's row
    entry for entry up to its length and -1 past it; -1 everywhere in the
    rows of free or swapped-out ids.  A compaction queues at most one patch
    per entry (the library uploads them without collapsing)."""
    rng = random.Random(seed)
    S, MB = 12, 40
    c = pkv.PagedKVCache(300, 8, 2, 128, S, MB, kv_dtype="bf16", alloc_seed=seed + 1, host_only=True)
    c.swap_space(200)
    _take_patches(pkv, c)
    dev = np.full((S, MB), -1, dtype=np.int32)
    live = []
    for op in range(1500):
        r = rng.random()
        compacted = False
        try:
            if not live or r < 0.15:
                live.append(c.seq_add())
            elif r < 0.45:
                s = rng.choice(live)
                c.reserve_slots([s], rng.randint(1, 40))
            elif r < 0.58:
                live.append(c.seq_fork(rng.choice(live)))
            elif r < 0.68:
                s = rng.choice(live)
                c.seq_free(s)
                live.remove(s)
            elif r < 0.76:
                c.seq_evict(rng.choice(live), rng.randint(0, 20), rng.randint(1, 100))
            elif r < 0.84:
                s = rng.choice(live)
                c.seq_truncate(s, rng.randint(0, c.seq_len(s)))
            elif r < 0.90:
                group = rng.sample(live, rng.randint(1, min(3, len(live))))
                c.seq_compact(group, [rng.randint(0, c.seq_len(x)) for x in group])
                compacted = True
            else:
                s = rng.choice(live)
                (c.swap_in if c.swapped(s) else c.swap_out)([s])
        except pkv.PKVError:
            pass  # refused calls (out of blocks or ids, evicted last block, swapped-out sequence) change nothing
        patches = _take_patches(pkv, c)
        if compacted:
            assert len(set(patches[:, 0].tolist())) == len(patches)
        for idx, val in patches:
            dev.flat[idx] = val
        for s in range(S):
            want = np.full(MB, -1, dtype=np.int32)
            if s in live and not c.swapped(s):
                t = c.block_table(s)
                want[: t.size] = t
            assert np.array_equal(dev[s], want), (seed, op, s)
