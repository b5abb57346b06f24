"""The plan builder's work lists, checked on the host (no GPU): ``gva_plan_inspect``
returns the forward items, the backward dQ items and the dK / dV units a plan holds,
and each list is re-derived here from the segment geometry and compared.

What the lists must satisfy follows from the method: every used query row of every
(segment, KV head) is covered exactly once; an item's key blocks are the used keys of
its segment (block-causal: only those its last row can see, by the visibility rule of
"Problem and behavior" in the multiview causal replay); FLOPs count the score pairs
that are computed; and the kernels take the longest work first."""
import numpy as np
import pytest

from gapped_varlen_attention_gb300 import _lib, workloads as W
from oracle import gva_oracle as oracle

TILE_ROWS, BLOCK_KEYS, TILES_PER_ITEM, MERGE_ROWS = 128, 128, 2, 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    import gapped_varlen_attention_gb300 as gva
    gva.build()


SMS = 152


def inspect(g, causal_block=0, grid=SMS):
    return _lib.inspect_plan(g.cu_q, g.used_q, g.cu_k, g.used_k, g.num_heads_q, g.num_heads_kv, g.head_dim,
                             causal_block, grid=grid)


def item_index(r, c, grid):
    """The kernels' walk: CTA c takes entry r * grid + c in even rounds, the mirror in odd."""
    return r * grid + (grid - 1 - c if r & 1 else c)


def est_cost(it):
    """The plan's run-time estimate of a forward item, in key blocks of a two-tile item:
    1.6 us per block with two Q tiles, 1.38 us with one, about 3 us per item."""
    return 1.9 + (1.0 if it["n_tiles"] == 2 else 0.86) * it["nblk"]


def dq_cost(it):
    return 2.0 + it["nblk"]


def kv_cost(u):
    return 2.0 + u["n_tiles"]


MERGE_CTAS_PER_SM = 4


def merge_rows(uq, sms):
    """Rows per LSE-merge unit: 16 while 16-row units fit one wave of the merge's resident
    CTAs (4 per SM); else the used rows are spread over the waves those units need,
    keeping one unit per segment in reserve for the segments' last, shorter units (16
    rows if that leaves under half a wave)."""
    total = int(sum(int(q) for q in uq))
    resident = MERGE_CTAS_PER_SM * sms
    n16 = sum(-(-int(q) // MERGE_ROWS) for q in uq)
    if n16 <= resident:
        return MERGE_ROWS
    waves = -(-n16 // resident)
    slots = waves * resident - len(uq)
    if slots < resident // 2:
        return MERGE_ROWS
    return min(MERGE_ROWS, max(1, -(-total // slots)))


def check_walk(items, walk, grid, cost=est_cost):
    """Every item is walked exactly once, a CTA's padding comes after its items, and no
    CTA carries more than the average load plus one item."""
    n = len(items)
    if n == 0:
        assert len(walk) == 0
        return
    grid = min(grid, n)
    assert len(walk) % grid == 0
    seen = np.zeros(n, int)
    loads = []
    for c in range(grid):
        load, padded = 0.0, False
        for r in range(len(walk) // grid):
            e = int(walk[item_index(r, c, grid)])
            if e < 0:
                padded = True
                continue
            assert not padded, "an item after a CTA's padding"
            seen[e] += 1
            load += cost(items[e])
        loads.append(load)
    assert np.all(seen == 1)
    costs = [cost(it) for it in items]
    assert max(loads) <= sum(costs) / grid + max(costs) + 1e-9


def rec(a, fields):
    return [dict(zip(fields, map(int, r))) for r in a]


def limits(uq, uk, B):
    """Keys visible to each used row: all of them without masking, else the oracle's rule."""
    if B == 0:
        return np.full(uq, uk, np.int64)
    return oracle.causal_limits(uq, uk, B).astype(np.int64)


def kp_of(u):
    """Index of a unit's first key within its segment (block-causal units carry it)."""
    return u["key_pos0"]


def check_work(g, B=0):
    w = inspect(g, B)
    group = g.num_heads_q // g.num_heads_kv
    tpt = TILE_ROWS // group
    nseg = g.num_segments
    cu_q, uq = g.cu_q.astype(np.int64), g.used_q.astype(np.int64)
    cu_k, uk = g.cu_k.astype(np.int64), g.used_k.astype(np.int64)
    seg_of_row = {}
    for b in range(nseg):
        for r in range(int(cu_q[b]), int(cu_q[b] + uq[b])):
            seg_of_row[r] = b

    # ---- counts
    assert w["num_key_blocks"] == sum(-(-int(k) // BLOCK_KEYS) for k in uk)
    rows = merge_rows(uq, SMS)
    assert 1 <= rows <= MERGE_ROWS
    assert w["num_merge_units"] == sum(-(-int(q) // rows) for q in uq)
    # the units need no more waves of the merge's resident CTAs than 16-row units would,
    # and 16-row units that fit one wave stay as they are
    resident = MERGE_CTAS_PER_SM * SMS
    sixteen = sum(-(-int(q) // MERGE_ROWS) for q in uq)
    assert -(-w["num_merge_units"] // resident) <= max(1, -(-sixteen // resident))
    if sixteen <= resident:
        assert w["num_merge_units"] == sixteen
    pairs = sum(float(limits(int(uq[b]), int(uk[b]), B).sum()) for b in range(nseg))
    want = 4.0 * g.head_dim * g.num_heads_q * pairs
    assert w["used_flops"] == pytest.approx(want, rel=1e-12)
    if B == 0:
        assert w["used_flops"] == pytest.approx(oracle.used_flops(uq, uk, g.num_heads_q, g.head_dim), rel=1e-12)

    blk0 = np.concatenate([[0], np.cumsum([-(-int(k) // BLOCK_KEYS) for k in uk])]).astype(np.int64)

    def check_items(items, rows_per_item, tiles_per_item):
        cover = {}
        for it in items:
            b = seg_of_row.get(it["q_row0"])
            assert b is not None, it
            t0 = it["q_row0"] - int(cu_q[b])
            assert t0 % rows_per_item == 0
            assert it["q_rows"] == min(rows_per_item, int(uq[b]) - t0)
            assert it["n_tiles"] == min(tiles_per_item, -(-it["q_rows"] // tpt))
            assert it["blk0"] == blk0[b] and it["k_len"] == uk[b]
            assert 0 <= it["head_kv"] < g.num_heads_kv
            lim = limits(int(uq[b]), int(uk[b]), B)
            assert it["nblk"] == -(-int(lim[t0 + it["q_rows"] - 1]) // BLOCK_KEYS)
            if B > 0:
                assert it["q_pos0"] == t0 + int(uk[b]) - int(uq[b])
            for r in range(it["q_row0"], it["q_row0"] + it["q_rows"]):
                key = (r, it["head_kv"])
                assert key not in cover, f"row {r} head {it['head_kv']} covered twice"
                cover[key] = True
        assert len(cover) == int(uq.sum()) * g.num_heads_kv

    # ---- forward items: up to two Q tiles each, every used row once per KV head
    items = rec(w["items"], _lib.WORK_ITEM_FIELDS)
    assert len(items) == w["num_work_items"]
    check_items(items, tpt * TILES_PER_ITEM, TILES_PER_ITEM)
    cost = [est_cost(it) for it in items]
    assert cost == sorted(cost, reverse=True), "forward items not longest first"
    check_walk(items, w["walk"], SMS)

    # ---- dQ items: one Q tile each, sorted by key blocks
    bwd = rec(w["bwd_items"], _lib.WORK_ITEM_FIELDS)
    check_items(bwd, tpt, 1)
    nb = [it["nblk"] for it in bwd]
    assert nb == sorted(nb, reverse=True), "dQ items not longest first"
    check_walk(bwd, w["bwd_walk"], SMS, dq_cost)

    # ---- dK / dV units: one per (segment, KV head, key block), every used key once; each
    # lists its one segment (if that has rows) and runs over its Q tiles from tile0
    units = rec(w["kv_units"], _lib.KV_UNIT_FIELDS)
    segs = [tuple(int(x) for x in r) for r in w["kv_segs"]]
    want_units = []
    for b in range(nseg):
        n_tiles = -(-int(uq[b]) // tpt)
        lim = limits(int(uq[b]), int(uk[b]), B)
        for hk in range(g.num_heads_kv):
            for j in range(-(-int(uk[b]) // BLOCK_KEYS)):
                kp = j * BLOCK_KEYS
                sees = np.nonzero(lim > kp)[0]  # rows that see the block's first key
                if B == 0:
                    tile0 = 0
                else:
                    tile0 = int(sees[0]) // tpt if sees.size else None
                u = dict(key_row0=int(cu_k[b]) + kp, keys=min(BLOCK_KEYS, int(uk[b]) - kp), head_kv=hk,
                         key_pos0=kp if B else 0, pos_shift=int(uk[b]) - int(uq[b]) if B else 0)
                want_units.append((u, b, tile0, n_tiles, lim))
    assert len(units) == len(want_units)
    by_key = {(u["key_row0"], u["head_kv"]): u for u in units}
    assert len(by_key) == len(units), "a (key block, KV head) unit appears twice"
    for u, b, tile0, n_tiles, lim in want_units:
        got = by_key[(u["key_row0"], u["head_kv"])]
        assert {k: got[k] for k in u} == u
        if uq[b] == 0:
            assert got["n_tiles"] == 0  # no row attends the block: dK = dV = 0
            continue
        assert segs[got["seg0"]] == (int(cu_q[b]), int(uq[b]))
        assert got["n_tiles"] == n_tiles - got["tile0"]
        if tile0 is not None:
            assert got["tile0"] == tile0
        else:  # no row sees the block: the unit may skip every tile, and skips no row that would
            assert got["tile0"] <= n_tiles
            assert not np.any(lim[:got["tile0"] * tpt] > kp_of(u))
        # whatever the start tile, the rows it skips see no key of the block
        assert not np.any(lim[:min(got["tile0"] * tpt, len(lim))] > kp_of(u))
    tiles = [u["n_tiles"] for u in units]
    assert tiles == sorted(tiles, reverse=True), "dK / dV units not longest first"
    check_walk(units, w["kv_walk"], SMS, kv_cost)
    return w


def test_tiny():
    w = check_work(W.tiny())
    assert w["num_work_items"] == 3 * 2  # one item per segment and KV head


def test_cfg_text_cross():
    check_work(W.cfg_text_cross())


def test_multiview_causal_and_partitions():
    full, parts = W.multiview_causal()
    check_work(full)
    check_work(full, 64)
    for p in parts:
        check_work(p)


def test_long_replay_counts():
    g = W.long_replay()
    w = check_work(g)
    tpi = (TILE_ROWS // (g.num_heads_q // g.num_heads_kv)) * TILES_PER_ITEM
    assert w["num_work_items"] == g.num_heads_kv * sum(-(-int(q) // tpi) for q in g.used_q)


@pytest.mark.parametrize("grid", [1, 5, 152])
def test_walk_on_small_grids(grid):
    g = W.random_geometry(np.random.default_rng(40 + grid), 5, 900, 2000, 8, 2, 128)
    w = inspect(g, 0, grid)
    check_walk(rec(w["items"], _lib.WORK_ITEM_FIELDS), w["walk"], grid)


def test_walk_balances_the_text_video_forward():
    """960 items (720 of two tiles, 240 of one) on 152 CTAs: 48 CTAs must take 7 items.
    The snake order of the sorted list puts 5 long and 2 short items on some CTAs; the
    balanced walk's longest CTA carries at most the average plus one short item, and at
    least 5 % less than the snake's."""
    text, video, union, dead = W.lse_merge_union()
    w = inspect(video)
    items = rec(w["items"], _lib.WORK_ITEM_FIELDS)
    costs = np.array([est_cost(it) for it in items])
    snake = np.zeros(SMS)
    for i, c in enumerate(costs):
        r, k = divmod(i, SMS)
        snake[k if r % 2 == 0 else SMS - 1 - k] += c
    loads = np.zeros(SMS)
    for e in range(len(w["walk"])):
        if w["walk"][e] >= 0:
            r, k = divmod(e, SMS)
            loads[k if r % 2 == 0 else SMS - 1 - k] += costs[w["walk"][e]]
    assert loads.max() <= costs.sum() / SMS + costs.min() + 1e-9
    assert loads.max() < 0.95 * snake.max()


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("B", [0, 1, 7, 64, 128, 300])
def test_random_geometries(seed, B):
    rng = np.random.default_rng(7100 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([1, 2, 4, 8]))
    g = W.random_geometry(rng, int(rng.integers(1, 7)), 700, 900, hkv * group, hkv, int(rng.choice([64, 128])))
    check_work(g, B)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("B", [0, 5, 128])
def test_random_geometries_groups_not_dividing_128(seed, B):
    """GQA groups that do not divide the 128-row tile (g = 3 for 12 query heads over 4 KV
    heads, ...): a tile folds floor(128 / g) tokens of the g heads."""
    rng = np.random.default_rng(7200 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([3, 5, 6, 12, 24, 100]))
    g = W.random_geometry(rng, int(rng.integers(1, 7)), 700, 900, hkv * group, hkv, int(rng.choice([64, 128])))
    check_work(g, B)


def test_more_queries_than_keys_causal():
    """Rows whose key position is negative see nothing: they cost no key block."""
    cu = np.array([0, 300], np.int32)
    g = W._geom(cu, [300], np.array([0, 100], np.int32), [100], 8, 2, 64)
    w = check_work(g, 16)
    bwd = rec(w["bwd_items"], _lib.WORK_ITEM_FIELDS)
    assert min(it["nblk"] for it in bwd) == 0


def test_empty_geometry():
    z = np.zeros(1, np.int32)
    w = _lib.inspect_plan(z, np.zeros(0, np.int32), z, np.zeros(0, np.int32), 4, 2, 64)
    assert w["num_work_items"] == w["num_bwd_items"] == w["num_kv_units"] == 0
    assert w["used_flops"] == 0.0


def test_capacity_truncates_and_errors():
    import ctypes
    g = W.random_geometry(np.random.default_rng(3), 4, 600, 600, 8, 2, 128, allow_empty=False)
    full = inspect(g)
    lib = _lib.load_library()
    a = [np.ascontiguousarray(x, np.int32) for x in (g.cu_q, g.used_q, g.cu_k, g.used_k)]
    p = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    s = _lib.WorkSummary()
    one = np.full((2, 8), -5, np.int32)
    geo = [p(a[0]), p(a[1]), p(a[2]), p(a[3]), 4, None, None, None, 0]

    def call(block, hq, hkv, d, summ, items, cap, *rest, geometry=geo, grid=SMS, walk_list=0):
        return lib.gva_plan_inspect(*geometry, block, hq, hkv, d, grid, walk_list, summ, items, cap, None, 0, *rest,
                                    None, 0)
    assert call(0, 8, 2, 128, ctypes.byref(s), p(one), 1, None, 0, None, 0) == 0
    assert s.num_work_items == full["num_work_items"] and s.backward_ok == 1
    assert np.array_equal(one[0], full["items"][0]) and np.all(one[1] == -5)
    # NULL summary, negative block, bad geometry, unsupported head_dim
    assert call(0, 8, 2, 128, None, None, 0, None, 0, None, 0) == 1
    assert call(-1, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0) == 1
    bad = a[3].copy()
    bad[0] = a[2][1] - a[2][0] + 1  # used keys above the capacity
    assert call(0, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0,
                geometry=[p(a[0]), p(a[1]), p(a[2]), p(bad), 4, None, None, None, 0]) == 1
    assert call(0, 8, 2, 96, ctypes.byref(s), None, 0, None, 0, None, 0) == 2
    assert call(0, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0, grid=0) == 1
    assert call(0, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0, walk_list=3) == 1
    # ranges: a range past total_k, and ranges with a causal block, are refused
    off, st, ln = (np.ascontiguousarray(x, np.int32) for x in ([0, 1, 1, 1, 2], [0, 90], [50, 20]))
    rgeo = [p(a[0]), p(a[1]), None, None, 4, p(off), p(st), p(ln)]
    assert call(0, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0, geometry=rgeo + [110]) == 0
    assert call(0, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0, geometry=rgeo + [100]) == 1
    assert call(16, 8, 2, 128, ctypes.byref(s), None, 0, None, 0, None, 0, geometry=rgeo + [110]) == 1


def _random_ranges(rng, nseg, total_k, disjoint):
    if disjoint:
        cuts = np.sort(rng.choice(np.arange(1, total_k), size=8 * nseg, replace=False))
        pieces = [(int(cuts[2 * i]), int(cuts[2 * i + 1] - cuts[2 * i])) for i in range(4 * nseg)]
        rng.shuffle(pieces)
        out = []
        for _ in range(nseg):
            take = int(rng.integers(0, 5))
            out.append(pieces[:take])
            pieces = pieces[take:]
        return out
    out = []
    for _ in range(nseg):
        rr = []
        for _ in range(int(rng.integers(0, 5))):
            st = int(rng.integers(0, total_k))
            rr.append((st, int(rng.integers(0, min(700, total_k - st) + 1))))
        out.append(rr)
    return out


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("disjoint", [True, False])
def test_key_range_plans(seed, disjoint):
    """gva_plan_ranges' lists: each range cut into blocks of at most 128 keys in order;
    every item of a segment carries its segment's blocks and key count; FLOPs count the
    concatenated keys. dK / dV units, for disjoint and overlapping ranges alike: every
    K/V row some range covers lies in exactly one unit per KV head, no range boundary
    falls inside a unit, and a unit lists exactly the segments (with rows) whose ranges
    cover each of its rows, a segment once per covering range of its own."""
    from collections import Counter
    rng = np.random.default_rng(900 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = W.random_geometry(rng, int(rng.integers(1, 6)), 700, 10, hkv * int(rng.choice([1, 2, 8])), hkv, 128)
    total_k = 3000
    ranges = _random_ranges(rng, g.num_segments, total_k, disjoint)
    if not disjoint and g.num_segments > 0 and ranges[0]:
        ranges[0].append(ranges[0][0])  # one segment attends a range twice
    w = _lib.inspect_plan(g.cu_q, g.used_q, None, None, g.num_heads_q, g.num_heads_kv, g.head_dim,
                          key_ranges=ranges, total_k=total_k)
    assert w["backward_ok"]
    blocks, seg_blk0 = [], []
    for rr in ranges:
        seg_blk0.append(len(blocks))
        for st, n in rr:
            blocks += [(st + o, min(BLOCK_KEYS, n - o)) for o in range(0, n, BLOCK_KEYS)]
    assert w["num_key_blocks"] == len(blocks)
    keys = [sum(n for _, n in rr) for rr in ranges]
    assert w["used_flops"] == pytest.approx(
        4.0 * g.head_dim * g.num_heads_q * sum(int(q) * k for q, k in zip(g.used_q, keys)), rel=1e-12)
    seg_of = {}
    for b in range(g.num_segments):
        for r in range(int(g.cu_q[b]), int(g.cu_q[b] + g.used_q[b])):
            seg_of[r] = b
    covered = {}
    for it in rec(w["items"], _lib.WORK_ITEM_FIELDS):
        b = seg_of[it["q_row0"]]
        nb = (seg_blk0[b + 1] if b + 1 < len(seg_blk0) else len(blocks)) - seg_blk0[b]
        assert it["blk0"] == seg_blk0[b] and it["nblk"] == nb and it["k_len"] == keys[b]
        for r in range(it["q_row0"], it["q_row0"] + it["q_rows"]):
            assert (r, it["head_kv"]) not in covered
            covered[(r, it["head_kv"])] = True
    assert len(covered) == int(g.used_q.sum()) * g.num_heads_kv

    # ---- dK / dV units against a row-by-row count of the ranges covering each K/V row
    tpt = TILE_ROWS // (g.num_heads_q // g.num_heads_kv)
    cover = [Counter() for _ in range(total_k)]  # K/V row -> {segment: covering ranges}
    bounds = set()
    for b, rr in enumerate(ranges):
        for st, n in rr:
            if n > 0:
                bounds |= {st, st + n}
                for x in range(st, st + n):
                    cover[x][b] += 1
    seg_by_row0 = {int(g.cu_q[b]): b for b in range(g.num_segments) if g.used_q[b] > 0}
    units = rec(w["kv_units"], _lib.KV_UNIT_FIELDS)
    segs = [tuple(int(v) for v in r) for r in w["kv_segs"]]
    seen = Counter()
    for u in units:
        assert 1 <= u["keys"] <= BLOCK_KEYS and u["tile0"] == 0
        assert not any(u["key_row0"] < x < u["key_row0"] + u["keys"] for x in bounds), "a unit crosses a boundary"
        # the unit's segments: consecutive SegRefs whose tiles add up to n_tiles
        listed, tiles, i = Counter(), 0, u["seg0"]
        while tiles < u["n_tiles"]:
            q_row0, q_used = segs[i]
            listed[seg_by_row0[q_row0]] += 1
            assert q_used == int(g.used_q[seg_by_row0[q_row0]])
            tiles += -(-q_used // tpt)
            i += 1
        assert tiles == u["n_tiles"]
        for x in range(u["key_row0"], u["key_row0"] + u["keys"]):
            want = Counter({b: m for b, m in cover[x].items() if g.used_q[b] > 0})
            assert listed == want, (x, listed, want)
            seen[(x, u["head_kv"])] += 1
    rows = [x for x in range(total_k) if cover[x]]
    assert len(seen) == len(rows) * g.num_heads_kv and all(c == 1 for c in seen.values())
    tiles = [u["n_tiles"] for u in units]
    assert tiles == sorted(tiles, reverse=True)


def test_plan_building_stays_fast_on_a_large_geometry():
    """The host plan for half a million forward items (plus about a million dQ items and
    the dK / dV units) is built in well under a few seconds: the balancer's passes cost
    O(n log n) in the list lengths, not O(n^2)."""
    import ctypes
    import time
    rng = np.random.default_rng(0)
    b = 64
    uq = rng.integers(1, 262144, size=b)
    cu_q = np.concatenate([[0], np.cumsum(np.full(b, 262144))])
    uk = rng.integers(1, 4096, size=b)
    cu_k = np.concatenate([[0], np.cumsum(np.full(b, 4096))])
    a = [_lib._i32(x) for x in (cu_q, uq, cu_k, uk)]
    p = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    lib = _lib.load_library()
    summ = _lib.WorkSummary()
    t0 = time.perf_counter()
    st = lib.gva_plan_inspect(p(a[0]), p(a[1]), p(a[2]), p(a[3]), b, None, None, None, 0, 0, 16, 16, 128, SMS, 0,
                              ctypes.byref(summ), None, 0, None, 0, None, 0, None, 0, None, 0)
    took = time.perf_counter() - t0
    assert st == 0 and summ.num_work_items > 500_000
    assert took < 5.0, f"plan inspection took {took:.2f} s"
