"""Host planner behind msa_plan_create (CPU only): segments bit-exact against
the brute-force splitter, the work list covers every (row, head, key) once,
and bad inputs come back as status codes."""
import numpy as np
import pytest

from kv_cache_segment_gb300 import msa, workloads as W
from oracle import segments

NSM = 152


def _plan(wl, num_sms=NSM):
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    return msa.msa_plan_create(dims, wl.block_table, wl.seq_lens, wl.q_range_indptr, wl.q_ranges_flat, num_sms)


def _random_table(rng, n_seqs):
    lens = rng.integers(0, 400, size=n_seqs)
    maxb = max(1, int(-(-lens.max() // 16)))
    table = np.full((n_seqs, maxb + 2), -1, np.int32)
    free = list(rng.permutation(4000))
    for s in range(n_seqs):
        nb = -(-int(lens[s]) // 16)
        for b in range(nb):
            if b > 0 and rng.random() < 0.7 and table[s, b - 1] + 1 not in table:
                table[s, b] = table[s, b - 1] + 1
            else:
                table[s, b] = free.pop()
    return lens.astype(np.int32), table


def test_segments_match_brute_force():
    rng = np.random.default_rng(0)
    dims = msa.make_dims(8, 2, 128)
    for trial in range(300):
        S = int(rng.integers(1, 6))
        lens, table = _random_table(rng, S)
        indptr = np.arange(S + 1, dtype=np.int32)
        ranges = np.stack([lens, lens + 1], 1).astype(np.int32)
        plan = msa.msa_plan_create(dims, table, lens, indptr, ranges, NSM)
        try:
            for s in range(S):
                want = segments.split_into_contiguous_segments(table[s], lens[s], 16)
                got = msa.msa_plan_get_runs(plan, s)
                assert [tuple(w[:3]) for w in want] == [tuple(int(x) for x in g) for g in got], (trial, s)
        finally:
            msa.msa_plan_destroy(plan)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_workload_segments_and_coverage(idx):
    wl = W.small_config(idx)
    plan = _plan(wl)
    try:
        for s in range(wl.num_seqs):
            got = msa.msa_plan_get_runs(plan, s)
            assert len(got) == len(wl.runs_drawn[s])
            assert [tuple(int(x) for x in g) for g in got] == [tuple(r) for r in wl.runs_drawn[s]]
        _check_coverage(wl, plan)
    finally:
        msa.msa_plan_destroy(plan)


@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_full_size_coverage(idx):
    wl = W.config(idx)
    plan = _plan(wl)
    try:
        info = msa.msa_plan_get_info(plan)
        assert info["num_runs"] == sum(len(r) for r in wl.runs_drawn)
        _check_coverage(wl, plan, enumerate_keys=False)
    finally:
        msa.msa_plan_destroy(plan)


def _check_coverage(wl, plan, enumerate_keys=True):
    """Every (row, query head) is in exactly one group; a group's parts tile
    [0, min(p_max + 1, L)) in order without gaps or overlap."""
    items = msa.msa_plan_get_items(plan)
    G = wl.num_q_heads // wl.num_kv_heads
    q_pos = wl.q_pos
    q_indptr = wl.q_indptr
    owner = np.zeros((wl.num_q_rows, wl.num_q_heads), np.int32)
    groups = {}
    for kind, seq, head, nh, row0, nrows, kb, ke, part in items:
        groups.setdefault((kind, seq, head, nh, row0, nrows), []).append((part, kb, ke))
    for (kind, seq, head, nh, row0, nrows), parts in groups.items():
        assert q_indptr[seq] <= row0 and row0 + nrows <= q_indptr[seq + 1]
        if kind == 0:
            assert nh == G
            heads = range(head * G, head * G + G)
        else:
            assert nh in (1, 2) and (nh == 1 or head // G == (head + 1) // G)
            heads = range(head, head + nh)
        for h in heads:
            owner[row0:row0 + nrows, h] += 1
        parts.sort()
        assert [p[0] for p in parts] == list(range(len(parts)))
        L = int(wl.seq_lens[seq])
        want_end = min(int(q_pos[row0 + nrows - 1]) + 1, L)
        assert parts[0][1] == 0 and parts[-1][2] == want_end
        for a, b in zip(parts, parts[1:]):
            assert a[2] == b[1] and a[1] < a[2]
        if kind == 0:
            assert nrows * G <= 16
        elif nh == 2:
            # two heads of one kv head over one row tile; for odd G never the
            # kv head's last query head
            assert nrows <= 128 and (head % G) % 2 == 0 and (G % 2 == 0 or head % G <= G - 3)
        else:
            # odd G: the last query head of a kv head over one or two row tiles
            assert G % 2 == 1 and head % G == G - 1 and nrows <= 256
    assert np.all(owner == 1)
    if enumerate_keys:
        # every visible key of every row is inside exactly one part's range
        for (kind, seq, head, nh, row0, nrows), parts in groups.items():
            L = int(wl.seq_lens[seq])
            for r in range(row0, row0 + nrows):
                vis = min(int(q_pos[r]) + 1, L)
                cover = np.zeros(max(vis, 1), np.int32)
                for _, kb, ke in parts:
                    lo, hi = kb, min(ke, vis)
                    if hi > lo:
                        cover[lo:hi] += 1
                assert vis == 0 or np.all(cover[:vis] == 1)


def test_info_work_counts():
    wl = W.small_config(5)
    plan = _plan(wl)
    try:
        info = msa.msa_plan_get_info(plan)
        G = wl.num_q_heads // wl.num_kv_heads
        D = wl.head_dim
        dec_kv, flops = 0, 0.0
        for s in range(wl.num_seqs):
            L = int(wl.seq_lens[s])
            pos = wl.q_pos[wl.q_indptr[s]:wl.q_indptr[s + 1]]
            if len(pos) <= 16 // G:
                dec_kv += min(int(pos[-1]) + 1, L) * wl.num_kv_heads * D * 4
            else:
                flops += sum(4.0 * D * wl.num_q_heads * min(int(p) + 1, L) for p in pos)
        assert info["decode_kv_bytes"] == dec_kv
        assert info["prefill_flops"] == pytest.approx(flops, rel=1e-12)
        assert info["num_q_rows"] == wl.num_q_rows
    finally:
        msa.msa_plan_destroy(plan)


def _create(lens, table, indptr, ranges, dims=None):
    dims = dims or msa.make_dims(4, 2, 128)
    return msa.msa_plan_create(dims, np.asarray(table, np.int32), np.asarray(lens, np.int32),
                               np.asarray(indptr, np.int32), np.asarray(ranges, np.int32), NSM)


@pytest.mark.parametrize("lens,table,indptr,ranges,code", [
    ([40], [[3, -1, 5]], [0, 1], [[40, 41]], msa.MSA_ERR_MISSING_BLOCK),
    ([40], [[3, 4, 1 << 27]], [0, 1], [[40, 41]], msa.MSA_ERR_BAD_BLOCK_ID),
    ([40], [[3, 4, 5]], [0, 1], [[40, 42]], msa.MSA_ERR_BAD_Q_RANGE),          # p > L
    ([40], [[3, 4, 5]], [0, 1], [[-1, 3]], msa.MSA_ERR_BAD_Q_RANGE),           # p < 0
    ([40], [[3, 4, 5]], [0, 2], [[10, 20], [15, 25]], msa.MSA_ERR_BAD_Q_RANGE),  # overlap
    ([40], [[3, 4, 5]], [0, 2], [[20, 30], [0, 10]], msa.MSA_ERR_BAD_Q_RANGE),   # unsorted
    ([40], [[3, 4, 5]], [0, 1], [[5, 5]], msa.MSA_ERR_BAD_Q_RANGE),             # empty
    ([40], [[3, 4]], [0, 1], [[40, 41]], msa.MSA_ERR_INVALID_ARG),              # table too narrow
    ([-1], [[3, 4, 5]], [0, 1], [[0, 1]], msa.MSA_ERR_INVALID_ARG),
])
def test_bad_inputs_return_status(lens, table, indptr, ranges, code):
    with pytest.raises(msa.MsaError) as e:
        _create(lens, table, indptr, ranges)
    assert e.value.status == code


@pytest.mark.parametrize("dims", [
    (4, 2, 96, 16), (4, 2, 128, 32), (6, 4, 128, 16), (64, 2, 128, 16),
])
def test_unsupported_dims(dims):
    with pytest.raises(msa.MsaError) as e:
        _create([16], [[0]], [0, 1], [[16, 17]], msa.make_dims(*dims))
    assert e.value.status == msa.MSA_ERR_UNSUPPORTED_DIMS


def test_attention_before_upload_is_rejected():
    plan = _create([16], [[0]], [0, 1], [[16, 17]])
    try:
        with pytest.raises(msa.MsaError) as e:
            msa.msa_attention(16, 16, 16, 16, plan, 16)
        assert e.value.status == msa.MSA_ERR_NOT_UPLOADED
    finally:
        msa.msa_plan_destroy(plan)


def test_empty_sequence_and_split_groups():
    # an empty sequence queried at p = 0, and one long decode row split over parts
    lens = [0, 20000]
    nb = -(-20000 // 16)
    table = np.full((2, nb), -1, np.int32)
    table[1] = np.arange(nb) + 10
    plan = _create(lens, table, [0, 1, 2], [[0, 1], [20000, 20001]])
    try:
        items = msa.msa_plan_get_items(plan)
        empty = items[items[:, 1] == 0]
        assert len(empty) == 2 and np.all(empty[:, 6] == 0) and np.all(empty[:, 7] == 0)
        long = items[items[:, 1] == 1]
        assert long[:, 8].max() > 0  # split into several parts
    finally:
        msa.msa_plan_destroy(plan)


@pytest.mark.parametrize("idx", [4, 5])
def test_restricted_rows_partition_the_plan(idx):
    """Decode-only and prefill-only restrictions of a mixed workload (the
    bench's graded legs) split its rows, decode bytes and prefill flops
    exactly as the full plan classifies them."""
    wl = W.config(idx)
    dec, pre = W.restrict_rows(wl, "decode"), W.restrict_rows(wl, "prefill")
    assert dec.num_q_rows + pre.num_q_rows == wl.num_q_rows
    for s in range(wl.num_seqs):
        full = sorted(p for a, b in wl.q_ranges[s] for p in range(a, b))
        parts = sorted(p for r in (dec.q_ranges[s], pre.q_ranges[s]) for a, b in r for p in range(a, b))
        assert full == parts
    infos = []
    for w in (wl, dec, pre):
        plan = _plan(w)
        try:
            infos.append(msa.msa_plan_get_info(plan))
        finally:
            msa.msa_plan_destroy(plan)
    full, di, pi = infos
    assert di["decode_kv_bytes"] == full["decode_kv_bytes"] and di["prefill_flops"] == 0
    assert pi["decode_kv_bytes"] == 0 and pi["prefill_flops"] == pytest.approx(full["prefill_flops"], rel=1e-12)


def _plan_state(plan, n_seqs):
    info = msa.msa_plan_get_info(plan)
    info.pop("host_plan_us")
    return (info, msa.msa_plan_workspace_bytes(plan), msa.msa_plan_get_items(plan).tolist(),
            msa.msa_plan_get_order(plan).tolist(), [msa.msa_plan_get_runs(plan, s).tolist() for s in range(n_seqs)])


def test_recycled_plans_equal_fresh_ones():
    """msa_plan_destroy keeps freed plans' storage for the next create on the
    thread: a plan built on recycled storage (after a large plan, a small
    one, and a create that failed part-way) equals one built before."""
    small = W.small_config(5)
    want = []
    for wl in (small, W.small_config(3)):
        p = _plan(wl)
        want.append(_plan_state(p, wl.num_seqs))
        msa.msa_plan_destroy(p)
    big = _plan(W.config(3))
    big2 = _plan(W.config(5))
    msa.msa_plan_destroy(big)
    msa.msa_plan_destroy(big2)
    dims = msa.make_dims(8, 2, 128)
    with pytest.raises(msa.MsaError):  # fails after its runs were built
        msa.msa_plan_create(dims, np.array([[0, 1]], np.int32), np.array([20], np.int32), np.array([0, 1], np.int32),
                            np.array([5, 3], np.int32), NSM)
    for wl, w in zip((small, W.small_config(3)), want):
        p = _plan(wl)
        assert _plan_state(p, wl.num_seqs) == w
        msa.msa_plan_destroy(p)


@pytest.mark.parametrize("seed", range(48))
def test_random_workloads_coverage(seed):
    """The GPU parity test's seeded random shapes (GQA ratios 1-16, D 64/128,
    empty sequences, 1-8 segments, 1-3 query ranges, split options): runs
    equal the drawn layout and every (row, head, visible key) is covered
    exactly once, under the split factors the GPU test uses."""
    from gpu_harness import random_workload
    wl, opts = random_workload(seed)
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    plan = msa.msa_plan_create_ex(dims, wl.block_table, wl.seq_lens, wl.q_range_indptr, wl.q_ranges_flat, NSM,
                                  opts.get("decode_split", 0.0), opts.get("prefill_split", 0.0))
    try:
        for s in range(wl.num_seqs):
            got = msa.msa_plan_get_runs(plan, s)
            assert [tuple(int(x) for x in g) for g in got] == [tuple(r) for r in wl.runs_drawn[s]]
        _check_coverage(wl, plan)
    finally:
        msa.msa_plan_destroy(plan)
