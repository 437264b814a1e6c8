"""The tile schedulers (host logic, no GPU).  Forward: work items come in a
stable longest-first order of their segments (Zellige §IV-D orders the
coalesced call's segments stably; §IV-C fills in decreasing price), and
together they cover every (head, query row, key) of every sequence exactly
once, within each tile's ranges.  Backward: every sequence runs whole, stably
longest-first by query count, one item per (head, 128-key block)."""
import collections

import pytest
import torch

import synth
import mixed_length_dit_gb300 as zl


def _schedule(wl, tiles=None, dtype=torch.bfloat16, cu_q=None, cu_k=None):
    cu = wl.cu_seqlens()
    return zl.fwd_schedule(cu_q or cu, cu_k or cu, wl.num_heads, wl.head_dim, tiles=tiles, dtype=dtype)


def _segments(items):
    """Segments in the order their first item appears, with their items."""
    segs = collections.OrderedDict()
    for it in items:
        segs.setdefault((it[0], it[1], it[2]), []).append(it)
    return segs


def _check(wl, tiles, items, rows_per_item, cu_q=None, cu_k=None):
    cu_q = cu_q or wl.cu_seqlens()
    cu_k = cu_k or wl.cu_seqlens()
    H = wl.num_heads
    tiles = tiles or []
    split = {t[0] for t in tiles}
    segs = _segments(items)
    # longest first, ties in input order (sequence, then the tile's place in its grid)
    keyed = []
    for (launch, s, t), its in segs.items():
        k_len = its[0][7]
        assert all(i[7] == k_len for i in its)
        if t < 0:
            rank = (s, 0, 0, 0)
        else:
            tt = tuple(tiles[t]) + (0, 0, 0)[: max(0, 11 - len(tiles[t]))]
            rank = (s, tt[10], tt[5], tt[6])             # h_chunk, q_chunk, kv_chunk
        keyed.append((launch, -k_len, rank))
    assert keyed == sorted(keyed)
    # items of one segment: head-major, query block fastest, blocks of rows_per_item
    for (launch, s, t), its in segs.items():
        heads = [i[3] for i in its]
        assert heads == sorted(heads)
        for h in set(heads):
            q = [(i[4], i[5]) for i in its if i[3] == h]
            assert all(0 < ql <= rows_per_item for _, ql in q)
            assert all(q[j][0] + q[j][1] == q[j + 1][0] for j in range(len(q) - 1))
            assert all(ql == rows_per_item for _, ql in q[:-1])
    # coverage: every (head, query, key) of every sequence exactly once
    covered = collections.Counter()
    for it in items:
        _, s, t, h, q0, ql, k0, kl = it
        lq, lk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        assert 0 <= q0 and q0 + ql <= lq and 0 <= k0 and k0 + kl <= lk and 0 <= h < H
        if t < 0:
            assert s not in split and k0 == 0 and kl == lk
        else:
            tile = tiles[t]
            assert tile[0] == s
            assert tile[1] <= q0 and q0 + ql <= tile[1] + tile[2]
            assert (k0, kl) == (tile[3], tile[4])
            if len(tile) > 9 and tile[9] > 0:
                assert tile[8] <= h < tile[8] + tile[9]
        covered[(s, h)] += ql * kl
    for s in range(len(cu_q) - 1):
        lq, lk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        for h in range(H):
            assert covered.get((s, h), 0) == lq * lk, (s, h)
    # the same rectangle is never covered twice: count (head, query block, key range)
    keys = collections.Counter((i[1], i[3], i[4], i[6]) for i in items)
    assert max(keys.values()) == 1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9])
def test_schedule_of_each_workload(n):
    wl = synth.config(n)
    tiles = wl.tiles() or None
    items = _schedule(wl, tiles)
    _check(wl, tiles, items, 256)


def test_item_counts():
    """Item counts by hand: ceil(rows / 256) blocks per head of each segment."""
    wl = synth.config(4)                     # 131,072 as 4 x 4 tiles + 64 x 1,024
    assert len(_schedule(wl, wl.tiles())) == 16 * 40 * (32768 // 256) + 64 * 40 * 4
    wl = synth.config(2)                     # 16 x 256 + 8 x 1,024 + 4 x 4,096, 24 heads
    assert len(_schedule(wl)) == 24 * (16 * 1 + 8 * 4 + 4 * 16)


def test_float32_items_hold_128_rows():
    wl = synth.config(1)
    tiles = synth.grid_tiles(3, 256, 256, 2, 2)
    items = _schedule(wl, tiles, dtype=torch.float32)
    _check(wl, tiles, items, 128)
    assert len(items) == 2 * (1 + 1 + 1) + 4 * 2


def test_ragged_empty_and_cross_lengths():
    """Empty sequences get no items; query and key lengths may differ."""
    cu_q = [0, 5, 5, 200, 330, 330]
    cu_k = [0, 130, 140, 600, 601, 601]
    wl = synth.Workload("cross", [5, 0, 195, 130, 0], 3, 64)
    tiles = synth.grid_tiles(2, 195, 460, 2, 3)
    items = _schedule(wl, tiles, cu_q=cu_q, cu_k=cu_k)
    _check(wl, tiles, items, 256, cu_q=cu_q, cu_k=cu_k)
    assert not any(i[1] in (1, 4) for i in items)
    # longest first: the 130-key sequence 0 before the 1-key sequence 3
    order = list(_segments(items))
    assert order.index((0, 0, -1)) < order.index((0, 3, -1))


def test_stable_ties_keep_input_order():
    wl = synth.Workload("ties", [300, 50, 300, 300, 50], 2, 128)
    segs = list(_segments(_schedule(wl)))
    assert [s[1] for s in segs] == [0, 2, 3, 1, 4]


def test_schedule_rejects_what_the_forward_rejects():
    with pytest.raises(zl.ZlError):
        zl.fwd_schedule([1, 5], [0, 5], 2, 64)          # does not start at 0
    with pytest.raises(zl.ZlError):
        zl.fwd_schedule([0, 4], [0, 0], 2, 64)          # queries without keys
    with pytest.raises(zl.ZlError):
        zl.fwd_schedule([0, 5], [0, 5], 2, 96)          # unsupported head dim
    with pytest.raises(zl.ZlError):                      # an incomplete tile grid
        zl.fwd_schedule([0, 256], [0, 256], 2, 64, tiles=synth.grid_tiles(0, 256, 256, 2, 2)[:3])


def _check_bwd(wl, items, cu_q=None, cu_k=None):
    cu_q = cu_q or wl.cu_seqlens()
    cu_k = cu_k or wl.cu_seqlens()
    H = wl.num_heads
    # sequences stably longest-first by query count, each head-major, key block fastest
    order = []
    for it in items:
        if not order or order[-1] != (it[0], it[1]):
            order.append((it[0], it[1]))
    assert len(order) == len(set(order))
    lq = [cu_q[s + 1] - cu_q[s] for s in range(len(cu_q) - 1)]
    assert [(l, -lq[s], s) for l, s in order] == sorted((l, -lq[s], s) for l, s in order)
    covered = collections.Counter()
    for _, s, h, k0, kl, ql in items:
        lk = cu_k[s + 1] - cu_k[s]
        assert ql == lq[s] and 0 < kl <= 128 and k0 % 128 == 0 and k0 + kl <= lk and 0 <= h < H
        covered[(s, h)] += kl
    for s in range(len(cu_q) - 1):
        lk = cu_k[s + 1] - cu_k[s]
        want = lk if lq[s] > 0 else 0
        for h in range(H):
            assert covered.get((s, h), 0) == want, (s, h)
    assert max(collections.Counter((i[1], i[2], i[3]) for i in items).values()) == 1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8])
def test_backward_schedule_of_each_workload(n):
    """Every key block of every head of every sequence once; tiles change
    nothing (the backward runs every sequence whole)."""
    wl = synth.config(n)
    cu = wl.cu_seqlens()
    items = zl.bwd_schedule(cu, cu, wl.num_heads, wl.head_dim, tiles=wl.tiles() or None)
    _check_bwd(wl, items)
    assert items == zl.bwd_schedule(cu, cu, wl.num_heads, wl.head_dim)


def test_backward_schedule_ragged_and_keys_without_queries():
    cu_q = [0, 70, 70, 400, 400]
    cu_k = [0, 200, 330, 500, 501]
    wl = synth.Workload("bwd_cross", [70, 0, 330, 0], 2, 128)
    items = zl.bwd_schedule(cu_q, cu_k, 2, 128)
    _check_bwd(wl, items, cu_q=cu_q, cu_k=cu_k)
    assert [s for _, s in dict.fromkeys((i[0], i[1]) for i in items)] == [2, 0]
    assert len(items) == 2 * (2 + 2)          # sequence 0: 200 keys, sequence 2: 170 keys


def test_more_segments_than_one_launch_holds():
    """1,500 sequences exceed one launch's segment table (640): the items
    spread over three launches, each stably longest-first, all covered once;
    the backward splits the same way."""
    rng = __import__("numpy").random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 700, size=1500)]
    wl = synth.Workload("many", lens, 2, 64)
    items = _schedule(wl)
    _check(wl, None, items, 256)
    assert sorted({i[0] for i in items}) == [0, 1, 2]
    cu = wl.cu_seqlens()
    bitems = zl.bwd_schedule(cu, cu, 2, 64)
    _check_bwd(wl, bitems)
    assert sorted({i[0] for i in bitems}) == [0, 1, 2]


def test_key_count_bound():
    """Keys x heads x head dim is bounded as queries are (2^40 elements): a
    batch past it is rejected before any work, in both directions."""
    with pytest.raises(zl.ZlError):
        zl.fwd_schedule([0, 1], [0, 1 << 30], 2048, 128)
    with pytest.raises(zl.ZlError):
        zl.bwd_schedule([0, 1], [0, 1 << 30], 2048, 128)
    assert len(zl.bwd_schedule([0, 1], [0, 1 << 20], 2, 128)) == 2 * (1 << 20) // 128
