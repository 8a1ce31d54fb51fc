"""Closed-form pins of the plain latency-model and eviction oracles
(oracle/costmodel.py, oracle/eviction.py).  Each pin takes the oracle module
as an argument (the real one, or a copy with a planted mistake) and checks it
against values worked out by hand here, on hand-built work lists: nothing in
these pins calls the library.

The model (MSA paper abstract; AsymCache explainer, "核心方法 2/3"): a work
item costs a fixed phase (decode: dec_item; prefill: pre_item + tile x
tiles x heads, tile = pre_tile x (1 - dfrac + dfrac x D / 128); plus box x
extra TMA boxes and, for a part of a split group, a merge constant) and,
for decode, a stream of tiles x 128 x D x 2 B x 2 (K and V) bytes at
min(per-CTA rate, shared rate / streaming CTAs); CTAs take items in queue
order as they free up.  The eviction score: alpha x hit + beta x
cost / max cost, lowest first, ties to the lower block; or hit x cost.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

PARAMS = dict(launch_us=6.5, dec_item_us=2.25, dec_gbs=6400.0, dec_cta_gbs=96.0, pre_item_us=3.5,
              pre_tile_us=0.875, box_us=0.0625, dec_merge_us=1.75, pre_merge_us=6.5)
TILE_BYTES = 2 * 128 * 128 * 2  # K and V of one 128-key tile, D = 128, bf16


def _item(kind, seq, heads, row0, kb, ke, part=0, head=0, nrows=1):
    return (kind, seq, head, heads, row0, nrows, kb, ke, part)


def _close(a, b, rel=1e-12):
    return math.isclose(a, b, rel_tol=rel, abs_tol=1e-12)


# ------------------------------------------------------------ latency model --

def pin_one_cta_mixed_items(oc):
    """One CTA runs a decode item (3 tiles), a prefill item (2 tiles x 2
    heads) and the two parts of a split decode group (2 tiles each) back to
    back: makespan = sum of fixed phases + all streamed bytes at min(per-CTA,
    shared) rate; time = launch + makespan."""
    tables = {0: list(range(0, 24)), 1: list(range(100, 116)), 2: list(range(200, 232))}
    lens = {0: 384, 1: 256, 2: 512}
    items = [_item(0, 0, 4, 0, 0, 384), _item(1, 1, 2, 1, 0, 256, nrows=128),
             _item(0, 2, 4, 129, 0, 256, part=0), _item(0, 2, 4, 129, 256, 512, part=1)]
    p = PARAMS
    fixed = (p["dec_item_us"] + (p["pre_item_us"] + p["pre_tile_us"] * 2 * 2)
             + 2 * (p["dec_item_us"] + p["dec_merge_us"]))
    stream = 7 * TILE_BYTES / (min(p["dec_cta_gbs"], p["dec_gbs"]) * 1e3)
    r = oc.estimate(items, [0, 1, 2, 3], tables, lens, 1, p, 128)
    assert r["n_items"] == 4 and r["n_split_items"] == 2
    assert r["decode_tiles"] == 7 and r["prefill_tile_heads"] == 4 and r["extra_boxes"] == 0
    assert r["stream_bytes"] == 7 * TILE_BYTES
    assert _close(r["fixed_us"], fixed)
    assert _close(r["makespan_us"], fixed + stream)
    assert _close(r["time_us"], p["launch_us"] + fixed + stream)


def pin_split_prefill_pays_its_merge(oc):
    """Two parts of a split prefill group (one head, 1 tile each) on two CTAs:
    each is pre_item + pre_tile + pre_merge, in parallel."""
    items = [_item(1, 0, 1, 0, 0, 128, part=0, nrows=128), _item(1, 0, 1, 0, 128, 256, part=1, nrows=128)]
    p = PARAMS
    r = oc.estimate(items, [0, 1], {0: list(range(16))}, {0: 256}, 2, p, 128)
    assert _close(r["makespan_us"], p["pre_item_us"] + p["pre_tile_us"] + p["pre_merge_us"])
    assert r["n_split_items"] == 2 and r["stream_bytes"] == 0


def pin_row_pair_prefill_counts_two_tiles(oc):
    """An odd Hq/Hkv prefill item: one head over 200 rows is two query tiles
    (128 + 72 rows) walking the same 3 key tiles: pre_item + pre_tile x 3 x 2;
    one head over 100 rows is one tile: pre_item + pre_tile x 3."""
    p = PARAMS
    items = [_item(1, 0, 1, 0, 0, 384, nrows=200), _item(1, 1, 1, 0, 0, 384, nrows=100)]
    tables = {0: list(range(24)), 1: list(range(100, 124))}
    r = oc.estimate(items, [0, 1], tables, {0: 384, 1: 384}, 1, p, 128)
    assert r["prefill_tile_heads"] == 3 * 2 + 3 * 1
    assert _close(r["fixed_us"], 2 * p["pre_item_us"] + p["pre_tile_us"] * (6 + 3))


def pin_tile_time_scales_with_head_dim(oc):
    """pre_tile_dfrac = 5/8 of a tile's D = 128 time scales with D: one
    prefill item of 3 key tiles x 2 heads costs pre_item + 6 x 0.875 = 8.75 us
    at D = 128 and pre_item + 6 x 0.875 x (3/8 + 5/8 x 1/2) = 3.5 + 3.609375 us
    at D = 64; a parameter set without the term prices D = 64 as D = 128."""
    items = [_item(1, 0, 2, 0, 0, 384, nrows=128)]
    tables, lens = {0: list(range(24))}, {0: 384}
    p = dict(PARAMS, pre_tile_dfrac=0.625)
    assert _close(oc.estimate(items, [0], tables, lens, 1, p, 128)["fixed_us"], 8.75)
    assert _close(oc.estimate(items, [0], tables, lens, 1, p, 64)["fixed_us"], 7.109375)
    assert _close(oc.estimate(items, [0], tables, lens, 1, PARAMS, 64)["fixed_us"], 8.75)
    assert _close(oc.tile_us(p, 64), 0.6015625) and _close(oc.tile_us(p, 128), 0.875)
    # all of a tile's time proportional to D halves it at D = 64; none of it, no change
    assert _close(oc.tile_us(dict(p, pre_tile_dfrac=1.0), 64), 0.4375)
    assert _close(oc.tile_us(dict(p, pre_tile_dfrac=0.0), 64), 0.875)


def pin_queue_order(oc):
    """Two CTAs, four prefill items of 4, 1, 2 and 6 tiles (one head) in that
    order: CTA 1 frees first and takes the third item, CTA 0 the fourth."""
    p = PARAMS
    cost = [p["pre_item_us"] + p["pre_tile_us"] * t for t in (4, 1, 2, 6)]
    items = [_item(1, s, 1, 0, 0, 128 * t, nrows=128) for s, t in enumerate((4, 1, 2, 6))]
    tables = {s: list(range(1000 * s, 1000 * s + 48)) for s in range(4)}
    lens = {s: 768 for s in range(4)}
    r = oc.estimate(items, [0, 1, 2, 3], tables, lens, 2, p, 128)
    want = max(cost[1] + cost[2], cost[0] + cost[3])
    assert _close(r["makespan_us"], want)


def pin_shared_bandwidth(oc):
    """Two CTAs stream at once with a shared rate below twice the per-CTA
    rate: each gets half of it."""
    p = dict(PARAMS, dec_gbs=100.0, dec_cta_gbs=96.0, box_us=0.0)
    items = [_item(0, s, 4, 0, 0, 384) for s in range(2)]
    tables = {0: list(range(24)), 1: list(range(100, 124))}
    r = oc.estimate(items, [0, 1], tables, {0: 384, 1: 384}, 2, p, 128)
    assert _close(r["makespan_us"], p["dec_item_us"] + 3 * TILE_BYTES / (50.0 * 1e3))


def pin_equal_items_in_rounds(oc):
    """N equal decode items (3 tiles) on C CTAs: rounds of k = min(C, left)
    items, each a fixed phase plus the stream at min(per-CTA, shared / k)."""
    for n, c, dec in ((6, 4, 6400.0), (20, 3, 6400.0), (9, 4, 150.0)):
        p = dict(PARAMS, box_us=0.0, dec_gbs=dec)
        items = [_item(0, s, 4, s, 0, 384) for s in range(n)]
        tables = {s: list(range(30 * s, 30 * s + 24)) for s in range(n)}
        r = oc.estimate(items, list(range(n)), tables, {s: 384 for s in range(n)}, c, p, 128)
        want, left = 0.0, n
        while left > 0:
            k = min(c, left)
            want += p["dec_item_us"] + 3 * TILE_BYTES / (min(p["dec_cta_gbs"], dec / k) * 1e3)
            left -= k
        assert _close(r["makespan_us"], want), (n, c, dec)


def pin_tma_boxes(oc):
    """Every block its own segment (physical blocks 0, 2, 4, ...): a full
    128-key tile needs 8 boxes (7 extra); the 40-key last tile 3 (2 extra).
    One segment: only the partial last tile (3 blocks) is cut, into a box of
    2 blocks and one of 1 (1 extra).  Segments of 7 and 1 blocks: the first
    tile is pieces of 7 blocks (4 + 2 + 1 blocks: 3 boxes) and 1 block."""
    L = 2 * 128 + 40
    nb = -(-L // 16)
    r = oc.estimate([_item(0, 0, 4, 0, 0, L)], [0], {0: [2 * b for b in range(nb)]}, {0: L}, 1, PARAMS, 128)
    assert r["extra_boxes"] == 2 * 7 + 2
    assert _close(r["fixed_us"], PARAMS["dec_item_us"] + PARAMS["box_us"] * 16)
    r1 = oc.estimate([_item(0, 0, 4, 0, 0, L)], [0], {0: list(range(nb))}, {0: L}, 1, PARAMS, 128)
    assert r1["extra_boxes"] == 1
    table = list(range(7)) + [20]  # blocks 0-6 contiguous, block 7 elsewhere
    r2 = oc.estimate([_item(0, 0, 4, 0, 0, 128)], [0], {0: table}, {0: 128}, 1, PARAMS, 128)
    assert r2["extra_boxes"] == (3 + 1) - 1


def pin_recompute_flops(oc):
    """4 D Hq sum_{p=a}^{b-1} min(p+1, L) by the arithmetic-series formula."""
    for a, b, L in ((0, 37, 400), (100, 228, 400), (380, 401, 400)):
        hi = min(b, L)
        s = hi * (hi + 1) // 2 - a * (a + 1) // 2 + (L if b == L + 1 else 0)
        assert oc.hole_recompute_flops(128, 8, a, b, L) == 4.0 * 128 * 8 * s


# ---------------------------------------------------------------- chunking --

def pin_chunk_candidates(oc):
    """Multiples of 128 up to the remainder, the remainder itself last; a cap
    cuts them; a remainder under one tile is the only candidate; 64
    multiples are thinned to every second (k = ceil(64 / 63) = 2), and the
    cap is added after 63 * 128 = 8064."""
    assert oc.chunk_candidates(1000) == [128, 256, 384, 512, 640, 768, 896, 1000]
    assert oc.chunk_candidates(1000, 128, 300) == [128, 256, 300]
    assert oc.chunk_candidates(100) == [100]
    assert oc.chunk_candidates(1024, 256) == [256, 512, 768, 1024]
    c = oc.chunk_candidates(8192)
    assert c == [128 * k for k in range(1, 64, 2)] + [8192] and len(c) == 33


def _closed_form_times(cands, F=32.0, a=1.0 / 1024.0, p0=4096):
    # one pending prefill at position p0: fixed step cost F plus attention
    # work a * sum over its c rows of (p0 + i), ~ a * c * (p0 + c / 2)
    return [F + a * c * (p0 + c / 2.0) for c in cands]


def pin_chunk_closed_form_optimum(oc):
    """T(c) = F + a c (p0 + c/2): T/c = F/c + a p0 + a c/2 is least at
    c* = sqrt(2F/a) = sqrt(2 * 32 * 1024) = 256 (per-token 4.25 against
    4.3125 at 128 and 4.2708 at 384)."""
    cands = [128 * k for k in range(1, 9)]
    t = _closed_form_times(cands)
    assert oc.choose_chunk(cands, t, cands, 0.0) == (256, True)


def pin_chunk_budget(oc):
    """T(256) = 32 + 0.25 * 4224 = 1088 and T(128) = 32 + 0.125 * 4160 = 552:
    a budget of 1000 leaves 128; a budget of 100 leaves nothing, and the
    smallest candidate comes back outside the budget."""
    cands = [128 * k for k in range(1, 9)]
    t = _closed_form_times(cands)
    assert t[0] == 552.0 and t[1] == 1088.0
    assert oc.choose_chunk(cands, t, cands, 1000.0) == (128, True)
    assert oc.choose_chunk(cands, t, cands, 100.0) == (128, False)


def pin_chunk_ties_to_the_larger(oc):
    """Time proportional to tokens (no fixed cost): every chunk costs the
    same per token, and the largest wins."""
    cands = [128, 256, 384]
    assert oc.choose_chunk(cands, [2.0 * c for c in cands], cands, 0.0) == (384, True)


def pin_chunk_batch(oc):
    """A pending sequence runs rows [start, start + min(c, end - start)) and
    holds start + that many tokens; the others keep their rows."""
    lens, indptr, ranges, tokens = oc.chunk_batch([100, 900, 50], [0, 1, 1, 2], [(100, 101), (49, 50)],
                                                  [(1, 300, 700)], 256)
    assert lens == [100, 556, 50] and indptr == [0, 1, 2, 3] and ranges == [(100, 101), (300, 556), (49, 50)]
    assert tokens == 256
    lens, _, ranges, tokens = oc.chunk_batch([100, 900, 50], [0, 1, 1, 2], [(100, 101), (49, 50)],
                                             [(1, 300, 700)], 1024)
    assert lens[1] == 700 and ranges[1] == (300, 700) and tokens == 400


COST_PINS = [pin_one_cta_mixed_items, pin_split_prefill_pays_its_merge, pin_row_pair_prefill_counts_two_tiles,
             pin_tile_time_scales_with_head_dim, pin_queue_order, pin_shared_bandwidth,
             pin_equal_items_in_rounds, pin_tma_boxes, pin_recompute_flops, pin_chunk_candidates,
             pin_chunk_closed_form_optimum, pin_chunk_budget, pin_chunk_ties_to_the_larger, pin_chunk_batch]


# ------------------------------------------------------------------ eviction --

def pin_block_cost(oe):
    """cost(b) = pre_tile * Hq * sum_{p in block b} (p + 1) / 128^2."""
    L, hq, pt = 1000, 32, 0.875
    cost = oe.recompute_cost_us(L, hq, pt)
    assert len(cost) == 63
    for b in (0, 10, 62):
        lo, hi = 16 * b, min(16 * b + 16, L)
        assert math.isclose(cost[b], pt * hq * ((hi * (hi + 1) - lo * (lo + 1)) // 2) / 16384, rel_tol=1e-15)


def pin_hit_only(oe):
    """alpha alone: the blocks least likely to be hit go first."""
    hit = np.linspace(1.0, 0.0, 40)
    ev, _ = oe.select_evictions(40 * 16, 32, hit, 1.0, 0.0, 0.875, 10)
    assert ev == list(range(30, 40))


def pin_cost_only(oe):
    """beta alone: recompute work grows with position, the first blocks go."""
    ev, cost = oe.select_evictions(40 * 16 + 5, 32, np.full(41, 0.5), 0.0, 1.0, 0.875, 7)
    assert ev == list(range(7))
    assert all(b > a for a, b in zip(cost[:-2], cost[1:-1]))


def pin_cost_on_the_keep_side(oe):
    """Equal hit probability except block 5 (slightly more likely to be hit):
    with the cost term added, the cheap early blocks still go before it, and
    a block dearer to recompute is kept over a cheaper one of equal hit."""
    hit = np.full(20, 0.5)
    hit[5] = 0.52
    ev, _ = oe.select_evictions(20 * 16, 32, hit, 1.0, 0.01, 0.875, 5)
    assert ev == [0, 1, 2, 3, 4]
    ev, _ = oe.select_evictions(20 * 16, 32, hit, 1.0, 0.01, 0.875, 6)
    assert ev == [0, 1, 2, 3, 4, 6]


def pin_ties_to_lower_block(oe):
    ev, _ = oe.select_evictions(20 * 16, 32, np.full(20, 0.3), 1.0, 0.0, 0.875, 5)
    assert ev == [0, 1, 2, 3, 4]


def pin_expected_cost_optimum(oe):
    """Brute force: no other n blocks have a lower sum of hit x cost."""
    rng = np.random.default_rng(3)
    L = 9 * 16 - 3
    hit = rng.random(9)
    for n in range(10):
        ev, cost = oe.select_evictions(L, 32, hit, 0.0, 0.0, 0.875, n, expected_cost=True)
        got = sum(hit[i] * cost[i] for i in ev)
        best = min(sum(hit[i] * cost[i] for i in c) for c in itertools.combinations(range(9), n))
        assert math.isclose(got, best, rel_tol=1e-12, abs_tol=1e-12) and len(ev) == n


def pin_prefix_cost_closed_form(oe):
    """Prefix reading: evicting block b leaves positions 16b .. L-1 to
    recompute, so cost(b) = pre_tile * Hq * sum_{p=16b}^{L-1} (p + 1) / 128^2
    = pre_tile * Hq * (L(L+1) - 16b(16b+1)) / 2 / 128^2, whatever the blocks
    after b look like (the last one partial here)."""
    L, hq, pt = 1000, 32, 0.875
    cost = oe.prefix_recompute_cost_us(L, hq, pt)
    assert len(cost) == 63
    for b in (0, 1, 31, 62):
        want = pt * hq * ((L * (L + 1) - 16 * b * (16 * b + 1)) // 2) / 16384
        assert math.isclose(cost[b], want, rel_tol=1e-13)


def pin_prefix_hand_worked(oe):
    """L = 48 (three full blocks), Hq = 1, pre_tile = 128^2 (cost in keys):
    hole costs 136, 392, 648; prefix costs 1176, 1040, 648.  With hit
    probabilities 0.9, 0.2, 0.5 the expected costs are 1058.4, 208, 324
    (prefix) against 122.4, 78.4, 324 (hole): one eviction takes block 1 in
    both readings, two take blocks 1 and 2 (prefix) but 0 and 1 (hole)."""
    assert oe.recompute_cost_us(48, 1, 16384.0) == [136.0, 392.0, 648.0]
    assert oe.prefix_recompute_cost_us(48, 1, 16384.0) == [1176.0, 1040.0, 648.0]
    hit = [0.9, 0.2, 0.5]
    assert oe.select_evictions(48, 1, hit, 0, 0, 16384.0, 1, expected_cost=True, prefix=True)[0] == [1]
    assert oe.select_evictions(48, 1, hit, 0, 0, 16384.0, 2, expected_cost=True, prefix=True)[0] == [1, 2]
    assert oe.select_evictions(48, 1, hit, 0, 0, 16384.0, 2, expected_cost=True)[0] == [0, 1]


def pin_prefix_cost_only_evicts_the_tail(oe):
    """beta alone in the prefix reading: cost falls strictly with position,
    so the last blocks go first (the cheap tail yields)."""
    ev, cost = oe.select_evictions(40 * 16 + 5, 32, np.full(41, 0.5), 0.0, 1.0, 0.875, 7, prefix=True)
    assert ev == list(range(34, 41))
    assert all(b < a for a, b in zip(cost[:-1], cost[1:]))


def pin_prefix_ties_to_lower_block(oe):
    """Equal scores evict the lower block first in the prefix reading too
    (alpha only, equal hits; and zero hit in expected-cost mode)."""
    ev, _ = oe.select_evictions(20 * 16, 32, np.full(20, 0.3), 1.0, 0.0, 0.875, 5, prefix=True)
    assert ev == [0, 1, 2, 3, 4]
    hit = np.full(20, 0.5)
    hit[[3, 9, 15]] = 0.0
    ev, _ = oe.select_evictions(20 * 16, 32, hit, 0.0, 0.0, 0.875, 2, expected_cost=True, prefix=True)
    assert ev == [3, 9]


EVICTION_PINS = [pin_block_cost, pin_hit_only, pin_cost_only, pin_cost_on_the_keep_side, pin_ties_to_lower_block,
                 pin_expected_cost_optimum, pin_prefix_cost_closed_form, pin_prefix_hand_worked,
                 pin_prefix_cost_only_evicts_the_tail, pin_prefix_ties_to_lower_block]
