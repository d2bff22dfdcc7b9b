"""The balanced key-range cut of fa_fwd_ws (kv_chunk = 0), inspected on the host.

fa_fwd_split_segments reports the plan without a GPU.  Whatever the plan, the
segments of each row block must partition its K/V tiles exactly (no tile twice,
none missed, parts numbered in key order), every CTA must own one contiguous run,
and no CTA may cost more than the plan's own worst case; the worst case must sit
near the lower bound every cut has to pay (all tiles plus one fixed cost per row
block, shared by the SMs), and only row blocks too long for one CTA are cut.  A test that drops a tile, repeats one or leaves a CTA
over budget fails here before any kernel reads the table.
"""
import collections

import pytest

ITEM_COST = 6   # fixed cost of a segment, in K/V-tile steps
SMS = 152


@pytest.fixture(scope="module")
def fa():
    from exact_attention_26_gb300 import build as fb
    if fb.needs_build():
        fb.build()
    import exact_attention_26_gb300 as fa
    fa.load()
    return fa


def _row_tiles(N, d, causal):
    rows, bn = 128, (64 if d == 256 else 128)
    n_cb, n_kv = -(-N // rows), -(-N // bn)
    return {cb: (min(n_kv, (cb + 1) * rows // bn) if causal else n_kv) for cb in range(n_cb)}


SHAPES = [(1, 1, 16384, 128, True), (1, 1, 16384, 128, False), (1, 1, 8192, 128, False),
          (1, 1, 16384, 256, True), (1, 2, 6000, 128, True), (1, 1, 8192, 64, True),
          (1, 2, 8192, 96, True), (1, 2, 3000, 256, False)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_segments_partition_every_row_block(fa, shape):
    B, H, N, d, causal = shape
    segs = fa.fwd_split_segments(B, H, N, d, causal, SMS)
    assert segs, "these long few-head shapes are cut"
    tiles = _row_tiles(N, d, causal)
    parts = collections.defaultdict(list)
    for head, cb, lo, n, s, ns, cta in segs:
        assert 0 <= head < B * H and cb in tiles and n >= 1 and 1 <= ns <= 15
        parts[(head, cb)].append((lo, n, s, ns))
    assert set(parts) == {(h, cb) for h in range(B * H) for cb in tiles}
    for (head, cb), ps in parts.items():
        ps.sort()
        assert [p[2] for p in ps] == list(range(len(ps)))       # parts in key order
        assert {p[3] for p in ps} == {len(ps)}                  # one count per row block
        edge = 0
        for lo, n, _, _ in ps:
            assert lo == edge                                   # no gap, no overlap
            edge += n
        assert edge == tiles[cb]                                # every tile, once


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ctas_run_contiguously_and_are_balanced(fa, shape):
    B, H, N, d, causal = shape
    segs = fa.fwd_split_segments(B, H, N, d, causal, SMS)
    ctas = [s[6] for s in segs]
    assert ctas == sorted(ctas) and ctas[0] == 0 and set(ctas) == set(range(ctas[-1] + 1))
    assert ctas[-1] < SMS
    load = collections.Counter()
    for _, _, _, n, _, _, cta in segs:
        load[cta] += n + ITEM_COST
    tiles = _row_tiles(N, d, causal)
    bound = (B * H * (sum(tiles.values()) + ITEM_COST * len(tiles))) / SMS
    # each cut adds one fixed cost, and a run may stop short by up to two of the
    # shortest pieces the plan cuts (eight row blocks' worth of diagonal tiles);
    # even chunks with the snake schedule reach 88 steps on the first shape (bound 59.4)
    min_piece = 8 * (2 if d == 256 else 1)
    assert max(load.values()) <= bound + ITEM_COST + 2 * min_piece, (max(load.values()), bound)
    # only row blocks longer than a CTA's budget are cut; the others go whole
    budget = max(load.values())
    for head, cb, lo, n, part, parts, cta in segs:
        if parts > 1:
            assert tiles[cb] + ITEM_COST > budget, (cb, tiles[cb], budget)


def test_no_cut_when_the_row_blocks_fill_the_gpu(fa):
    assert fa.fwd_split_segments(1, 4, 16384, 128, True, SMS) == []   # 512 row blocks
    assert fa.fwd_split_segments(2, 16, 4096, 128, True, SMS) == []
    assert fa.fwd_split_segments(1, 1, 1024, 128, True, SMS) == []    # too little work


def test_plan_follows_the_sm_count(fa):
    a = fa.fwd_split_segments(1, 1, 16384, 128, True, 152)
    b = fa.fwd_split_segments(1, 1, 16384, 128, True, 132)
    assert max(s[6] for s in a) < 152 and max(s[6] for s in b) < 132
    assert a != b


def test_arguments_are_checked(fa):
    assert fa.fa_fwd_split_segments(1, 1, 16384, 128, 1, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_split_segments(1, 1, 16384, 100, 1, 152) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_split_segments(1, 1, 16384, 128, 1, 152, None, 4) == fa.FA_ERR_INVALID_ARG
    n = fa.fa_fwd_split_segments(1, 1, 16384, 128, 1, 152)
    assert n > 0
