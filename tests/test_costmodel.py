"""Attention-latency model (msa_plan_estimate): the library against the plain
Python restatement in oracle/costmodel.py, and both against closed forms."""
import math

import pytest

import oracle.costmodel as OC
from kv_cache_segment_gb300 import msa, workloads as W

PARAMS = dict(launch_us=6.5, dec_item_us=2.25, dec_gbs=6400.0, dec_cta_gbs=96.0, pre_item_us=3.5,
              pre_tile_us=0.875, box_us=0.0625, dec_merge_us=1.75, pre_merge_us=6.5)


def _plan(wl, num_sms=152):
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    return msa.msa_plan_create(dims, wl.block_table, wl.seq_lens, wl.q_range_indptr, wl.q_ranges_flat, num_sms)


def _both(wl, params=PARAMS, num_sms=152):
    plan = _plan(wl, num_sms)
    try:
        lib = msa.msa_plan_estimate(plan, params)
        items = msa.msa_plan_get_items(plan)
        order = msa.msa_plan_get_order(plan)
        grid = msa.msa_plan_get_info(plan)["grid"]
        ref = OC.estimate(items.tolist(), order.tolist(), wl.block_table, wl.seq_lens, grid, params, wl.head_dim)
        info = msa.msa_plan_get_info(plan)
    finally:
        msa.msa_plan_destroy(plan)
    return lib, ref, info


INT_KEYS = ("n_items", "n_split_items", "decode_tiles", "prefill_tile_heads", "extra_boxes", "stream_bytes")


def _odd_g(hq, hkv):
    return W.custom([700, 260, 90], [[4, 30, 10], [5, 12], [6]], [[(0, 300), (650, 701)], [(258, 261)], [(87, 91)]],
                    hq=hq, hkv=hkv, seed=11)


@pytest.mark.parametrize("wl_fn", [lambda: W.small_config(1), lambda: W.small_config(2), lambda: W.small_config(3),
                                   lambda: W.small_config(5), lambda: W.config(2), lambda: W.config(5),
                                   lambda: _odd_g(6, 2), lambda: _odd_g(4, 4)],
                         ids=["small1", "small2", "small3", "small5", "batched_decode", "mixed_batch", "G3", "G1"])
def test_library_matches_oracle(wl_fn):
    lib, ref, _ = _both(wl_fn())
    for k in INT_KEYS:
        assert lib[k] == ref[k], k
    for k in ("fixed_us", "makespan_us", "time_us"):
        assert lib[k] == pytest.approx(ref[k], rel=1e-9), k


@pytest.mark.parametrize("dfrac", [0.0, 0.4, 1.0])
@pytest.mark.parametrize("d", [64, 128])
def test_library_matches_oracle_head_dim_term(d, dfrac):
    """Prefill tiles priced at the plan's head dim (pre_tile_dfrac): library =
    oracle on a mixed decode + prefill + odd-G work list at D = 64 and 128."""
    wl = W.custom([700, 260, 90], [[4, 30, 10], [5, 12], [6]], [[(0, 300), (650, 701)], [(258, 261)], [(87, 91)]],
                  hq=6, hkv=2, d=d, seed=12)
    lib, ref, _ = _both(wl, dict(PARAMS, pre_tile_dfrac=dfrac))
    assert lib["prefill_tile_heads"] == ref["prefill_tile_heads"] > 0
    for k in ("fixed_us", "makespan_us", "time_us"):
        assert lib[k] == pytest.approx(ref[k], rel=1e-9), k
    if d == 128 or dfrac == 0.0:  # the term changes nothing there
        base, _, _ = _both(wl, PARAMS)
        assert lib["time_us"] == pytest.approx(base["time_us"], rel=1e-12)


@pytest.mark.parametrize("num_sms", [1, 7, 1500])
def test_library_matches_oracle_other_grids(num_sms):
    lib, ref, _ = _both(W.small_config(3), num_sms=num_sms)
    for k in INT_KEYS:
        assert lib[k] == ref[k], k
    assert lib["makespan_us"] == pytest.approx(ref["makespan_us"], rel=1e-9)


def test_one_cta_runs_items_back_to_back():
    """One CTA: every fixed phase plus every stream at min(per-CTA, shared)."""
    lib, ref, info = _both(W.small_config(5), num_sms=1)
    assert info["grid"] == 1
    rate = min(PARAMS["dec_cta_gbs"], PARAMS["dec_gbs"]) * 1e3
    want = lib["fixed_us"] + lib["stream_bytes"] / rate
    assert lib["makespan_us"] == pytest.approx(want, rel=1e-9)
    assert ref["makespan_us"] == pytest.approx(want, rel=1e-9)


@pytest.mark.parametrize("n_seqs,ctas,dec_gbs", [(6, 4, 6400.0), (8, 8, 6400.0), (20, 3, 6400.0), (6, 4, 200.0),
                                                 (9, 4, 150.0)])
def test_equal_items_fill_ctas_in_rounds(n_seqs, ctas, dec_gbs):
    """N identical decode groups (one segment, one query, 3 tiles, no split)
    on C CTAs run in rounds of k = min(C, items left) CTAs, each round one
    fixed phase plus the stream at min(per-CTA, shared / k)."""
    L = 3 * 128
    wl = W.custom([L] * n_seqs, [[L // 16]] * n_seqs, [[(L, L + 1)]] * n_seqs, hq=4, hkv=1)
    params = dict(PARAMS, box_us=0.0, dec_gbs=dec_gbs)
    lib, ref, info = _both(wl, params, num_sms=ctas)
    assert lib["n_items"] == n_seqs and lib["n_split_items"] == 0 and lib["decode_tiles"] == 3 * n_seqs
    C = info["grid"]
    tile_bytes = 2 * 128 * 128 * 2
    want, left = 0.0, n_seqs
    while left > 0:
        k = min(C, left)
        want += params["dec_item_us"] + 3 * tile_bytes / (min(params["dec_cta_gbs"], dec_gbs / k) * 1e3)
        left -= k
    assert lib["makespan_us"] == pytest.approx(want, rel=1e-9)
    assert ref["makespan_us"] == pytest.approx(want, rel=1e-9)


def test_single_block_segments_cost_seven_extra_boxes_per_full_tile():
    """Every block its own segment: a full tile touches 8 segments (8 boxes),
    a partial last tile of n keys ceil(n/16) boxes; in one segment the
    partial tile's 3 blocks take boxes of 2 and 1 blocks."""
    L = 2 * 128 + 40
    nb = -(-L // 16)
    wl = W.custom([L], [[1] * nb], [[(L, L + 1)]], hq=4, hkv=1)
    lib, ref, _ = _both(wl, num_sms=1)
    want = 2 * 7 + (math.ceil(40 / 16) - 1)
    assert lib["extra_boxes"] == want and ref["extra_boxes"] == want
    one = W.custom([L], [[nb]], [[(L, L + 1)]], hq=4, hkv=1)
    lib1, ref1, _ = _both(one, num_sms=1)
    assert lib1["extra_boxes"] == ref1["extra_boxes"] == 2 - 1  # only the partial tile: 3 blocks = 2 + 1


@pytest.mark.parametrize("a,b,L", [(0, 37, 400), (100, 228, 400), (380, 401, 400)])
def test_position_aware_recompute_flops(a, b, L):
    """Rows [a, b) of one sequence: 4 D Hq sum_p min(p+1, L); the closed form
    of the sum, the oracle and the plan agree."""
    hq, d = 8, 128
    closed = sum(p + 1 for p in range(a, min(b, L))) + (L if b == L + 1 else 0)
    arith = (min(b, L) * (min(b, L) + 1) // 2 - a * (a + 1) // 2) + (L if b == L + 1 else 0)
    assert closed == arith
    assert OC.hole_recompute_flops(d, hq, a, b, L) == 4.0 * d * hq * arith
    wl = W.custom([L], [[-(-L // 16)]], [[(a, b)]], hq=hq, hkv=2, d=d)
    _, _, info = _both(wl)
    dec_rows = 16 // (hq // 2)
    if b - a > dec_rows:
        n = b - a
        rem = n % 128
        if 0 < rem <= dec_rows:  # the trailing rows go to the decode path
            pre = 4.0 * d * hq * sum(min(p + 1, L) for p in range(a, b - rem))
        else:
            pre = 4.0 * d * hq * arith
        assert info["prefill_flops"] == pytest.approx(pre, rel=1e-12)


def test_estimate_rejects_null():
    with pytest.raises(msa.MsaError):
        msa._check(msa.load().msa_plan_estimate(None, None, None), "msa_plan_estimate")


# ------------------------------------------------- adaptive chunking (create_ex)

FITTED = dict(launch_us=31.0, dec_item_us=2.83, dec_gbs=7708.0, dec_cta_gbs=60.0, pre_item_us=4.58, pre_tile_us=0.884,
              box_us=0.0062, dec_merge_us=1.49, pre_merge_us=46.2)
DEC_CANDIDATES = (1.0, 1.5, 2.0, 3.0, 4.0)
PRE_CANDIDATES = (1.0, 2.0, 4.0)


def _args(wl):
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    return (dims, wl.block_table, wl.seq_lens, wl.q_range_indptr, wl.q_ranges_flat)


def _time(wl, d, p, params, num_sms=152):
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=num_sms, decode_split=d, prefill_split=p)
    try:
        return msa.msa_plan_estimate(plan, params)["time_us"]
    finally:
        msa.msa_plan_destroy(plan)


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_explicit_splits_are_used_and_reported(idx):
    wl = W.config(idx)
    counts = []
    for d, p in ((1.0, 1.0), (3.0, 4.0), (8.0, 8.0)):
        plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152, decode_split=d, prefill_split=p)
        try:
            info = msa.msa_plan_get_info(plan)
            assert (info["decode_split"], info["prefill_split"]) == (d, p)
            counts.append(info["num_items"])
        finally:
            msa.msa_plan_destroy(plan)
    assert counts[0] <= counts[1] <= counts[2]  # finer splits, no fewer items
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152)
    try:
        info = msa.msa_plan_get_info(plan)
        assert (info["decode_split"], info["prefill_split"]) == (3.0, 4.0)  # the defaults
    finally:
        msa.msa_plan_destroy(plan)


@pytest.mark.parametrize("wl_fn", [lambda: W.config(2), lambda: W.config(5), lambda: W.small_config(3),
                                   lambda: W.restrict_rows(W.config(4), "decode")],
                         ids=["batched_decode", "mixed_batch", "small3", "long_decode_rows"])
def test_chooser_picks_the_model_minimum(wl_fn):
    """Decode split first (prefill at its default), then prefill split, each
    the candidate with the lowest msa_plan_estimate time (first on ties)."""
    wl = wl_fn()
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152, choose_with=FITTED)
    try:
        info = msa.msa_plan_get_info(plan)
        kinds = set(msa.msa_plan_get_items(plan)[:, 0].tolist())
    finally:
        msa.msa_plan_destroy(plan)
    d, p, best = 3.0, 4.0, math.inf
    if 0 in kinds:
        for c in DEC_CANDIDATES:
            t = _time(wl, c, 4.0, FITTED)
            if t < best:
                best, d = t, c
    if 1 in kinds:
        for c in PRE_CANDIDATES:
            t = _time(wl, d, c, FITTED)
            if t < best:
                best, p = t, c
    assert (info["decode_split"], info["prefill_split"]) == (d, p)


@pytest.mark.parametrize("d,p", [(-1.0, 0.0), (0.0, float("nan")), (float("inf"), 1.0)])
def test_bad_split_options_are_rejected(d, p):
    with pytest.raises(msa.MsaError) as e:
        msa.msa_plan_create_ex(*_args(W.small_config(2)), num_sms=152, decode_split=d, prefill_split=p)
    assert e.value.status == msa.MSA_ERR_INVALID_ARG


def test_bad_cost_params_are_rejected():
    plan = msa.msa_plan_create_ex(*_args(W.small_config(2)), num_sms=152)
    try:
        with pytest.raises(msa.MsaError):
            msa.msa_plan_estimate(plan, dict(FITTED, dec_gbs=-1.0))
        with pytest.raises(msa.MsaError):
            msa.msa_plan_estimate(plan, dict(FITTED, pre_tile_us=float("nan")))
        for bad in (-0.1, 1.5, float("nan")):
            with pytest.raises(msa.MsaError):
                msa.msa_plan_estimate(plan, dict(FITTED, pre_tile_dfrac=bad))
    finally:
        msa.msa_plan_destroy(plan)


def test_fit_recovers_known_constants():
    """costfit.fit on launch times generated by the model itself from known
    constants (several workloads x split plans, one of them prefill at head
    dim 64) finds constants that predict those times to 1e-3; the ones the
    plans constrain well come back to 2 %."""
    from kv_cache_segment_gb300 import costfit
    truth = dict(launch_us=20.0, dec_item_us=3.0, dec_gbs=7000.0, dec_cta_gbs=55.0, pre_item_us=5.0,
                 pre_tile_us=0.9, box_us=0.01, dec_merge_us=1.5, pre_merge_us=40.0, pre_tile_dfrac=0.6)
    plans = []
    for wl in (W.small_config(2), W.small_config(3), W.small_config(5), W.config(2),
               W.batched_decode(seed=9, num_seqs=64, len_range=(512, 4096), pool_tokens=1 << 20),
               W.hole_recompute(seed=9, num_seqs=4, cached_blocks=128, evict_blocks=32, d=64)):
        dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
        for ds, ps in ((1.0, 1.0), (3.0, 4.0), (8.0, 8.0)):
            for sms in (152, 40):
                plans.append(msa.msa_plan_create_ex(dims, wl.block_table, wl.seq_lens, wl.q_range_indptr,
                                                    wl.q_ranges_flat, sms, ds, ps))
    try:
        records = [(p, msa.msa_plan_estimate(p, truth)["time_us"]) for p in plans]
        got = costfit.fit(records)
        err = costfit.errors(records, got)
        assert err["max_abs_rel_err"] < 1e-3, err
        for k in ("launch_us", "pre_tile_us", "dec_gbs", "pre_tile_dfrac"):
            assert got[k] == pytest.approx(truth[k], rel=0.02), (k, got[k])
        # without a prefill at another head dim the share is held at 0
        at128 = [r for r, p in zip(records, plans) if msa.msa_plan_estimate(p, dict(truth, pre_tile_dfrac=0.0))
                 ["time_us"] == r[1]]
        assert len(at128) < len(records) and costfit.fit(at128)["pre_tile_dfrac"] == 0.0
    finally:
        for p in plans:
            msa.msa_plan_destroy(p)


# ------------------------------------------------------- prefill chunk size --

def _pending_batch():
    """The small mixed batch: sequences 0-5 decode one row each; the prefills
    of sequences 6 and 7 are pending from positions 27 and 25 (500 and 1000
    positions still to run)."""
    wl = W.small_config(5)
    pending = [(6, 27, 527), (7, 25, 1025)]
    indptr, ranges = [0], []
    for s in range(wl.num_seqs):
        if s not in (6, 7):
            ranges.extend(wl.q_ranges[s])
        indptr.append(len(ranges))
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    return wl, dims, pending, indptr, ranges


@pytest.mark.parametrize("budget", ["none", "median", "tiny"])
def test_chunk_choice_matches_oracle(budget):
    """Candidates, each candidate's predicted step time (the oracle's latency
    model on the plan of that candidate's batch) and the choice."""
    wl, dims, pending, indptr, ranges = _pending_batch()
    lens = wl.seq_lens.tolist()
    choice, cands, times = msa.msa_choose_prefill_chunk(dims, wl.block_table, lens, indptr, ranges, pending, PARAMS,
                                                        num_sms=152)
    b = {"none": 0.0, "median": float(sorted(times)[len(times) // 2]), "tiny": 1.0}[budget]
    if b:
        choice, cands, times = msa.msa_choose_prefill_chunk(dims, wl.block_table, lens, indptr, ranges, pending,
                                                            PARAMS, budget_us=b, num_sms=152)
    assert cands.tolist() == OC.chunk_candidates(1000) == [128, 256, 384, 512, 640, 768, 896, 1000]
    tokens = []
    for c, t in zip(cands.tolist(), times.tolist()):
        lc, ic, rc, n = OC.chunk_batch(lens, indptr, ranges, pending, c)
        tokens.append(n)
        plan = msa.msa_plan_create(dims, wl.block_table, lc, ic, rc, 152)
        try:
            items = msa.msa_plan_get_items(plan).tolist()
            order = msa.msa_plan_get_order(plan).tolist()
            ref = OC.estimate(items, order, wl.block_table, lc, 152, PARAMS, wl.head_dim)
        finally:
            msa.msa_plan_destroy(plan)
        assert t == pytest.approx(ref["time_us"], rel=1e-9), c
    want = OC.choose_chunk(cands.tolist(), times.tolist(), tokens, b)
    assert (choice["chunk"], bool(choice["within_budget"])) == want
    i = cands.tolist().index(choice["chunk"])
    assert choice["tokens"] == tokens[i] and choice["time_us"] == times[i]
    assert choice["n_candidates"] == len(cands)
    if budget == "tiny":
        assert choice["chunk"] == 128 and not choice["within_budget"]


def test_chunk_choice_granularity_and_cap():
    wl, dims, pending, indptr, ranges = _pending_batch()
    _, cands, _ = msa.msa_choose_prefill_chunk(dims, wl.block_table, wl.seq_lens, indptr, ranges, pending, PARAMS,
                                               granularity=256, max_chunk=700, num_sms=152)
    assert cands.tolist() == OC.chunk_candidates(1000, 256, 700) == [256, 512, 700]


@pytest.mark.parametrize("bad", ["own_rows", "negative_start", "empty_range", "twice", "seq_out_of_range"])
def test_chunk_choice_rejects_bad_pending(bad):
    wl, dims, pending, indptr, ranges = _pending_batch()
    want = msa.MSA_ERR_INVALID_ARG
    if bad == "own_rows":
        pending = [(0, 10, 500)]  # sequence 0 already runs a decode row in the batch
    elif bad == "negative_start":
        pending, want = [(6, -1, 500)], msa.MSA_ERR_BAD_Q_RANGE
    elif bad == "empty_range":
        pending, want = [(6, 300, 300)], msa.MSA_ERR_BAD_Q_RANGE
    elif bad == "twice":
        pending = [(6, 27, 527), (6, 27, 527)]
    else:
        pending = [(8, 0, 100)]
    with pytest.raises(msa.MsaError) as e:
        msa.msa_choose_prefill_chunk(dims, wl.block_table, wl.seq_lens, indptr, ranges, pending, PARAMS,
                                     num_sms=152)
    assert e.value.status == want


# ----------------------------------------------- split chooser, by hand --

def _equal_decode_batch(n_seqs, length):
    """n_seqs sequences of `length` tokens in one segment each, one decode
    row per sequence, 32/8 heads, D = 128: 8 * n_seqs decode groups."""
    return W.custom([length] * n_seqs, [[length // 16]] * n_seqs, [[(length, length + 1)]] * n_seqs,
                    hq=32, hkv=8, seed=5)


TILE_US_AT_50 = 128 * 128 * 2 * 2 / 50e3  # one 128-key K+V tile (D = 128) at 50 GB/s: 1.31072 us


def test_split_chooser_by_hand_one_group_per_cta():
    """152 groups of 64 tiles on 152 CTAs: factor 1 gives each CTA one whole
    group, T = launch + item + 64 tiles = 5 + 2 + 83.886 = 90.886 us; any
    larger factor cuts each group in two or more parts, which adds items and
    merges on every CTA (factor 1.5 or 2: 5 + 2 x (2 + 2) + 83.886), so the
    chooser keeps factor 1."""
    p = dict(launch_us=5.0, dec_item_us=2.0, dec_gbs=1e7, dec_cta_gbs=50.0, pre_item_us=5.0, pre_tile_us=1.0,
             box_us=0.0, dec_merge_us=2.0, pre_merge_us=20.0)
    wl = _equal_decode_batch(19, 8192)
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152, choose_with=p)
    try:
        info = msa.msa_plan_get_info(plan)
        assert (info["decode_split"], info["num_items"]) == (1.0, 152)
        assert msa.msa_plan_estimate(plan, p)["time_us"] == pytest.approx(5.0 + 2.0 + 64 * TILE_US_AT_50, rel=1e-12)
    finally:
        msa.msa_plan_destroy(plan)
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152, decode_split=2.0, prefill_split=4.0)
    try:
        assert msa.msa_plan_estimate(plan, p)["time_us"] == pytest.approx(5.0 + 2 * 4.0 + 64 * TILE_US_AT_50,
                                                                          rel=1e-12)
    finally:
        msa.msa_plan_destroy(plan)


def test_split_chooser_by_hand_finer_parts_fill_the_rounds():
    """16 groups of 512 tiles on 152 CTAs, free items and merges, every CTA
    streaming at 50 GB/s.  The work per CTA is 16 x (512 x 1.1 + 0.5) / 152
    = 59.33 tile costs.  Factor 1: parts of ceil(59.33 / 1.1) = 54 tiles give
    10 parts a group (9 of 52, one of 44 once the range is cut evenly), 160
    items: the 8 left over run after the 44-tile ones, makespan 88 tiles.
    Factor 1.5 gives 15 parts a group, 240 items (makespan 35 + 35 = 70 tiles
    plus the uneven tail the model replays).  Factor 2: parts of
    ceil(29.67 / 1.1) = 27 tiles, 19 a group (18 of 27, one of 26), 304
    items = two full rounds of 152, makespan 54 tiles = 70.78 us + 5 us
    launch: the least, so the chooser takes 2 (3 ties it; the first minimum
    stands)."""
    p = dict(launch_us=5.0, dec_item_us=0.0, dec_gbs=1e7, dec_cta_gbs=50.0, pre_item_us=5.0, pre_tile_us=1.0,
             box_us=0.0, dec_merge_us=0.0, pre_merge_us=20.0)
    wl = _equal_decode_batch(2, 65536)
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152, choose_with=p)
    try:
        info = msa.msa_plan_get_info(plan)
        assert (info["decode_split"], info["num_items"]) == (2.0, 304)
        assert msa.msa_plan_estimate(plan, p)["time_us"] == pytest.approx(5.0 + 54 * TILE_US_AT_50, rel=1e-12)
    finally:
        msa.msa_plan_destroy(plan)
    plan = msa.msa_plan_create_ex(*_args(wl), num_sms=152, decode_split=1.0, prefill_split=4.0)
    try:
        assert msa.msa_plan_get_info(plan)["num_items"] == 160
        assert msa.msa_plan_estimate(plan, p)["time_us"] == pytest.approx(5.0 + 88 * TILE_US_AT_50, rel=1e-12)
    finally:
        msa.msa_plan_destroy(plan)
