"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerance (bf16 in, fp32 accumulate): every out element within
2e-3 + 1e-2*|ref|, lse within 1e-4 absolute; pool scatter bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from gpu_harness import compare, oracle_ref, random_workload, run_gpu
from kv_cache_segment_gb300 import msa, workloads as W
from kv_cache_segment_gb300.runner import MsaSession, append_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msa.load()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ------------------------------------------------------------------ append --

@pytest.mark.parametrize("hkv,d", [(8, 128), (4, 64), (1, 128)])
def test_append_kv_bit_exact(hkv, d):
    g = torch.Generator().manual_seed(5)
    pool_tokens, n = 4096, 700
    kp = torch.randn((pool_tokens, hkv, d), generator=g).to(torch.bfloat16).cuda()
    vp = torch.randn((pool_tokens, hkv, d), generator=g).to(torch.bfloat16).cuda()
    kn = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16).cuda()
    slot = torch.randperm(pool_tokens, generator=g)[:n].to(torch.int64)
    slot[::7] = -1
    want_k = oracle.scatter_rows(_bits(kn), slot.numpy(), _bits(kp).copy())
    want_v = oracle.scatter_rows(_bits(vn), slot.numpy(), _bits(vp).copy())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dims = msa.make_dims(hkv, hkv, d)
    append_kv(kn, vn, slot.cuda(), kp, vp, dims, error_word=err)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kp), want_k)
    assert np.array_equal(_bits(vp), want_v)
    assert int(err.item()) == 0
    # and against torch's own index_copy_
    keep = slot >= 0
    ref = torch.zeros_like(kp).copy_(kp)
    ref.index_copy_(0, slot[keep].cuda(), kn[keep.cuda()])
    assert torch.equal(ref.view(torch.int16), kp.view(torch.int16))


def test_append_kv_slot_past_pool_is_reported_not_written():
    kp = torch.zeros((64, 2, 64), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    kn = torch.ones((3, 2, 64), dtype=torch.bfloat16, device="cuda")
    slot = torch.tensor([1, 64, 5], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    append_kv(kn, kn, slot, kp, vp, msa.make_dims(2, 2, 64), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) != 0
    assert kp[1].float().sum().item() == 128 and kp[5].float().sum().item() == 128
    assert kp.float().sum().item() == 256


@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64)])
def test_gather_kv_bit_exact(hkv, d):
    """k_out[t] = k_pool[slot[t]] (and V) for slot >= 0; rows with slot -1
    keep what they held; against numpy indexing of the same bits."""
    g = torch.Generator().manual_seed(9)
    pool_tokens, n = 5000, 1500
    kp = torch.randn((pool_tokens, hkv, d), generator=g).to(torch.bfloat16).cuda()
    vp = torch.randn((pool_tokens, hkv, d), generator=g).to(torch.bfloat16).cuda()
    slot = torch.randint(0, pool_tokens, (n,), generator=g, dtype=torch.int64)
    slot[::5] = -1
    ko = torch.full((n, hkv, d), 3.0, dtype=torch.bfloat16, device="cuda")
    vo = torch.full((n, hkv, d), -3.0, dtype=torch.bfloat16, device="cuda")
    want_k, want_v = _bits(ko).copy(), _bits(vo).copy()
    keep = slot.numpy() >= 0
    want_k[keep] = _bits(kp)[slot.numpy()[keep]]
    want_v[keep] = _bits(vp)[slot.numpy()[keep]]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dims = msa.make_dims(hkv, hkv, d)
    msa.msa_gather_kv(kp, vp, pool_tokens, slot.cuda(), n, ko, vo, dims, err, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(ko), want_k) and np.array_equal(_bits(vo), want_v)
    assert int(err.item()) == 0
    sel = slot.cuda().clamp(min=0)
    assert torch.equal(kp.index_select(0, sel)[keep], ko[keep])


def test_gather_kv_slot_past_pool_is_reported_not_read():
    kp = torch.ones((64, 2, 64), dtype=torch.bfloat16, device="cuda")
    ko = torch.zeros((3, 2, 64), dtype=torch.bfloat16, device="cuda")
    slot = torch.tensor([1, 64, 5], dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msa.msa_gather_kv(kp, kp, 64, slot, 3, ko, ko.clone(), msa.make_dims(2, 2, 64), err,
                      torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert int(err.item()) == msa.MSA_DEVERR_SLOT
    assert ko[0].float().sum().item() == 128 and ko[1].float().sum().item() == 0 and ko[2].float().sum().item() == 128


# ------------------------------------------------------- attention, small --

@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_small_configs_match_oracle(idx):
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q)
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, wl.name)


@pytest.mark.parametrize("idx", [2, 3, 5])
def test_split_groups_merge(idx):
    """Many CTAs -> long groups split into parts merged by log-sum-exp."""
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q, num_sms=1500)
    assert info["num_items"] > info["num_groups"]
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, wl.name + "/split")


@pytest.mark.parametrize("idx", [2, 3, 5])
@pytest.mark.parametrize("opts", [dict(decode_split=1.0, prefill_split=1.0), dict(decode_split=12.0, prefill_split=16.0),
                                  "chooser"], ids=["coarse", "fine", "chooser"])
def test_plan_options_match_oracle(idx, opts):
    """Plans from msa_plan_create_ex (the bench's): few large items, many
    small split ones, and the latency model's choice."""
    from kv_cache_segment_gb300 import costfit
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    if opts == "chooser":
        params = costfit.load_params()
        if params is None:
            pytest.skip("no fitted latency-model constants")
        opts = dict(choose_with=params)
    out, lse, info = run_gpu(wl, k, v, q, num_sms=40, **opts)
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, f"{wl.name}/{opts}")


def test_fp32_output():
    wl = W.small_config(3)
    k, v, q = W.make_values(wl)
    out, lse, _ = run_gpu(wl, k, v, q, out_fp32=True)
    assert out.dtype == torch.float32
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, "fp32 out")


@pytest.mark.parametrize("idx", [3, 5])
def test_fp32_output_through_split_merges(idx):
    """fp32 out with split groups (many CTAs): the last-arriver merges write
    fp32 rows, within tolerance of the oracle."""
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q, out_fp32=True, num_sms=1000)
    assert out.dtype == torch.float32 and info["num_items"] > info["num_groups"]
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, "fp32 out, split")


def test_lse_null_gives_the_same_out():
    """lse is optional (NULL): out is bit-identical to a call that asks for it."""
    wl = W.small_config(5)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    sess = MsaSession.from_workload(wl, num_sms=400)
    try:
        qd = q.to(dev)
        lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
        a = sess.attention(qd, kp, vp, lse=lse).clone()
        b = sess.attention(qd, kp, vp)
        torch.cuda.synchronize()
        assert sess.check_device()[0] == 0
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    finally:
        sess.close()


def test_segmented_equals_contiguous_layout():
    """Losslessness: the same logical K/V laid out as one segment or as many
    gives the same result (both within tolerance of the oracle and of each
    other)."""
    lens = [1000, 777]
    many = [[5, 9, 3, 20, 12, 14], [7, 7, 7, 7, 7, 7, 7]]
    one = [[63], [49]]
    ranges = [[(100, 260), (1000, 1001)], [(0, 40), (500, 777)]]
    wl_a = W.custom(lens, many, ranges, hq=8, hkv=2, seed=3)
    wl_b = W.custom(lens, one, ranges, hq=8, hkv=2, seed=4)
    k, v, q = W.make_values(wl_a)
    oa, la, _ = run_gpu(wl_a, k, v, q)
    ob, lb, _ = run_gpu(wl_b, k, v, q)
    ro, rl = oracle_ref(wl_a, k, v, q)
    compare(oa, la, ro, rl, "segmented")
    compare(ob, lb, ro, rl, "contiguous")
    assert (oa.float() - ob.float()).abs().max().item() <= 4e-3


# ------------------------------------------------------------- edge cases --

@pytest.mark.parametrize("case", ["empty_seq", "mid_decode", "ragged", "gqa16", "d64_prefill", "one_key",
                                  "far_ranges", "single_block_runs"])
def test_edge_cases(case):
    if case == "empty_seq":       # L = 0 queried at p = 0 (no key visible) next to a normal one
        wl = W.custom([0, 50], [[], [4]], [[(0, 1)], [(50, 51)]], hq=4, hkv=2)
    elif case == "mid_decode":    # decode-path rows at p < L (they see keys <= p only)
        wl = W.custom([300], [[3, 5, 11]], [[(33, 35)]], hq=8, hkv=4)
    elif case == "ragged":        # partial last blocks, NaN past L, prefill tile + decode tail
        wl = W.custom([129, 1], [[2, 3, 4], [1]], [[(0, 129), (129, 130)], [(0, 2)]], hq=4, hkv=1)
    elif case == "gqa16":
        wl = W.custom([600, 90], [[10, 28], [6]], [[(600, 601)], [(20, 91)]], hq=16, hkv=1)
    elif case == "d64_prefill":
        wl = W.custom([700], [[4, 30, 10]], [[(0, 300), (650, 701)]], hq=8, hkv=2, d=64)
    elif case == "one_key":       # L = 1
        wl = W.custom([1, 1], [[1], [1]], [[(0, 2)], [(1, 2)]], hq=4, hkv=2)
    elif case == "far_ranges":    # one 128-row tile spanning distant ranges
        wl = W.custom([3000], [[40, 60, 88]], [[(10, 70), (1500, 1540), (2990, 3001)]], hq=4, hkv=2)
    else:                         # every block its own segment
        wl = W.custom([400], [[1] * 25], [[(0, 400), (400, 401)]], hq=8, hkv=2)
    k, v, q = W.make_values(wl)
    out, lse, _ = run_gpu(wl, k, v, q)
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, case)
    if case == "empty_seq":
        assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 128), (6, 2, 128), (10, 2, 128), (6, 2, 64)])
@pytest.mark.parametrize("opts", [dict(), dict(decode_split=12.0, prefill_split=16.0)])
def test_odd_gqa_ratios(hq, hkv, d, opts):
    """G = Hq/Hkv odd: a prefill item carries one query head over two
    consecutive 128-row tiles (over one, with the second softmax warpgroup
    idle, where the group is shorter), and a decode item packs floor(16 / G)
    rows.  Sequence 0
    has two full 128-row tiles and a ragged prefill tail; sequence 1 has 3
    decode rows; sequence 2 has 4 rows, which is a decode item for G <= 4
    and a 4-row prefill tile for G = 5.  The second plan splits groups, so
    one-head prefill parts go through the cross-CTA merge."""
    wl = W.custom([700, 260, 90], [[4, 30, 10], [5, 12], [6]], [[(0, 300), (650, 701)], [(258, 261)], [(87, 91)]],
                  hq=hq, hkv=hkv, d=d, seed=11)
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q, **opts)
    assert info["num_prefill_items"] > 0 and info["num_decode_items"] > 0
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, f"G={hq // hkv} d={d}")


@pytest.mark.parametrize("name", ["holes", "mixed", "long", "holes_g3"])
@pytest.mark.parametrize("opts", [dict(), dict(decode_split=12.0, prefill_split=16.0)])
def test_d64_prefill_workloads(name, opts):
    """Head dim 64 (the S MMAs rotate over three TMEM buffers, so a query
    tile's next S is computed while its softmax still works) on small
    hole-recompute, mixed and long-context shapes, with and without split
    groups; rows near a sequence start take the residual pass in S's
    columns."""
    if name == "holes":
        wl = W.hole_recompute(seed=41, num_seqs=2, cached_blocks=64, evict_blocks=16, hole_range=(2, 6),
                              turn_tokens=72, hq=8, hkv=2, d=64)
    elif name == "holes_g3":
        wl = W.hole_recompute(seed=42, num_seqs=2, cached_blocks=48, evict_blocks=12, hole_range=(2, 5),
                              turn_tokens=100, hq=6, hkv=2, d=64)
    elif name == "mixed":
        wl = W.mixed_batch(seed=43, num_decode=6, num_prefill=2, chunk=200, median=600, cap=3000, max_seg=8,
                           hq=16, hkv=2, d=64)
    else:
        wl = W.long_context(seed=44, num_seqs=1, length=4096 + 40, n_runs=12, p=1.0 / 16, chunk=300,
                            hq=8, hkv=2, d=64)
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q, **opts)
    assert info["num_prefill_items"] > 0
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, f"D=64 {name} {opts}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("num_sms", [1, 3])
@pytest.mark.parametrize("name", ["holes", "holes_g3", "mixed", "decode_split"])
def test_many_items_per_cta(name, num_sms, d):
    """One or three CTAs, so that every CTA walks many items and all state
    carried from item to item is exercised: at D = 64 the rotation of the
    three S buffers (slots counted across items), through one-query-tile
    items (G = 3, where warpgroup 1 sits items out) and, in the mixed batch,
    past decode items that the same CTAs run in between; at both head
    dimensions the O hand-over between items, the stage rings, and in the
    decode-only launch the merge warp's hand-offs and split groups merged by
    the last of their parts."""
    opts = {}
    if name == "holes":
        wl = W.hole_recompute(seed=45, num_seqs=2, cached_blocks=64, evict_blocks=16, hole_range=(2, 6),
                              turn_tokens=72, hq=8, hkv=2, d=d)
    elif name == "holes_g3":
        wl = W.hole_recompute(seed=46, num_seqs=2, cached_blocks=48, evict_blocks=12, hole_range=(2, 5),
                              turn_tokens=100, hq=6, hkv=2, d=d)
    elif name == "mixed":
        wl = W.mixed_batch(seed=47, num_decode=6, num_prefill=2, chunk=200, median=600, cap=3000, max_seg=8,
                           hq=16, hkv=2, d=d)
    else:
        wl = W.batched_decode(seed=48, num_seqs=6, len_range=(300, 2100), pool_tokens=1 << 16, hq=8, hkv=2, d=d)
        opts = dict(decode_split=12.0)
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q, num_sms=num_sms, **opts)
    assert info["grid"] == num_sms and info["num_items"] > 4 * num_sms
    if name == "decode_split":
        assert info["num_prefill_items"] == 0 and info["num_items"] > info["num_groups"]
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, f"D={d} {name} on {num_sms} CTAs")


def test_full_size_d64_hole_recompute_sampled():
    """The bench's head-dim-64 prefill shape (16 sequences of 8,192 cached
    tokens with 25 % recomputed in holes plus a 512-token turn, 32/8 heads)
    at full size, under the plan the bench times, checked on sampled rows:
    ~34 items per CTA through the rotating S buffers."""
    from kv_cache_segment_gb300 import costfit
    params = costfit.load_params()
    opts = dict(choose_with=params) if params is not None else {}
    wl = W.hole_recompute(seed=1003, hq=32, hkv=8, d=64)
    dev = torch.device("cuda")
    k, v, q = W.make_values(wl, device=dev)
    out, lse, info = run_gpu(wl, k, v, q, **opts)
    assert info["num_prefill_items"] > 20 * info["grid"]
    rng = np.random.default_rng(1003)
    rows = _sample_rows(wl, rng, per_seq=4)
    rows = rows[rng.permutation(len(rows))[:48]]
    rows.sort()
    ro, rl = oracle_ref(wl, k.cpu(), v.cpu(), q.cpu(), rows=rows)
    compare(out[torch.as_tensor(rows, device=dev)], lse[torch.as_tensor(rows, device=dev)], ro, rl, wl.name)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("shape", ["rising", "falling", "spikes"])
def test_running_max_moves(shape, d):
    """Scores far from N(0,1): keys whose scores rise along the sequence (the
    running max moves up by more than the lazy-rescale threshold many times,
    so O is rescaled in TMEM and in registers), fall (the first keys dominate
    and later probabilities underflow), or carry a few large outliers.  q is
    made positive and K[t] = a(t) + 0.25 N(0,1), so the score of key t is
    about a(t) * 0.8 * sqrt(D); a(t) stays <= 3.5 sqrt(128 / D), so the
    score stays <= ~32 (lse up to ~40), where fp32 accumulation in the MMA
    still meets the lse bound.  At D = 64 the O rescales wait for the PV of
    the previous tile, which can still be in flight there (the S MMAs rotate
    over three TMEM buffers)."""
    wl = W.custom([1500, 700], [[20, 44, 30], [10, 34]], [[(0, 260), (1490, 1501)], [(600, 700), (700, 701)]],
                  hq=8, hkv=2, d=d, seed=13)
    k, v, q = W.make_values(wl)
    g = torch.Generator().manual_seed(5)
    T = k.shape[0]
    t = torch.zeros(T)
    for s in range(wl.num_seqs):
        a, b = int(wl.kv_indptr[s]), int(wl.kv_indptr[s + 1])
        t[a:b] = torch.linspace(0.0, 1.0, b - a)
    top = 3.5 * (128.0 / d) ** 0.5
    if shape == "rising":
        amp = top * t
    elif shape == "falling":
        amp = top * (1.0 - t)
    else:
        amp = torch.zeros(T)
        amp[torch.randint(0, T, (40,), generator=g)] = top
    k = (amp[:, None, None] + 0.25 * torch.randn(k.shape, generator=g)).to(torch.bfloat16)
    q = q.float().abs().to(torch.bfloat16)
    out, lse, _ = run_gpu(wl, k, v, q)
    ro, rl = oracle_ref(wl, k, v, q)
    assert np.nanmax(rl) > 20.0  # the scores really are large
    compare(out, lse, ro, rl, shape)


def _sink_and_rival(wl, lens, d):
    """Values where key 0 of every sequence (an attention sink) takes most of
    a row's softmax mass and one rival key far into the sequence most of the
    rest (weights about 0.64 and 0.36), with V of the rival -1.8 times the
    sink's."""
    k, v, q = W.make_values(wl)
    q = q.float().abs().to(torch.bfloat16)  # positive q: a positive key gives a large score
    k = k.float()
    v = v.float()
    base = 0
    # scores ~ amp * 0.8 * sqrt(D); the rival sits 0.6 (natural log) below the sink
    amp = 14.0 / (0.8 * d ** 0.5)
    for s, L in enumerate(lens):
        rival = base + 600 + 37 * s
        k[base] = amp + 0.02 * k[base]
        k[rival] = amp - 0.6 / (0.8 * d ** 0.5) + 0.02 * k[rival]
        v[base] = 2.0 * v[base]
        v[rival] = -1.8 * v[base]
        base += L
    return k.to(torch.bfloat16), v.to(torch.bfloat16), q


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("opts", [dict(), dict(decode_split=12.0, prefill_split=16.0)])
def test_attention_sink_with_a_rival_key(d, opts):
    """Rows whose weight sits on two keys among more than a thousand: key 0
    of every sequence (an attention sink) takes most of the softmax mass and
    one rival key far into the sequence most of the rest (weights about
    0.64 and 0.36), with V of the rival -1.8 times the sink's, so the two
    products nearly cancel and the stated tolerance is almost all absolute.
    A single bf16 rounding of P is then not averaged away by the other keys;
    the output must still meet the stated tolerance with no allowance, for
    prefill rows before and after the rival, decode rows, and with the key
    range split into parts merged by log-sum-exp."""
    # sequences 0-1: prefill rows before and after the rival (and a decode
    # row in a prefill tile); 2-3: rows short enough for the GQA-packed
    # decode path (a lone decode row; three trailing rows)
    lens = [1500, 2100, 1800, 1301]
    wl = W.custom(lens, [[30, 40, 24], [50, 32, 30, 20], [40, 33, 40], [20, 21, 41]],
                  [[(0, 40), (560, 900), (1490, 1501)], [(1200, 1450), (2100, 2101)], [(1800, 1801)],
                   [(1298, 1301)]],
                  hq=8, hkv=2, d=d, seed=71)
    k, v, q = _sink_and_rival(wl, lens, d)
    out, lse, info = run_gpu(wl, k, v, q, **opts)
    assert info["num_prefill_items"] > 0 and info["num_decode_items"] > 0
    ro, rl = oracle_ref(wl, k, v, q)
    assert np.nanmax(rl) > 10.0  # the sink does dominate
    compare(out, lse, ro, rl, f"sink D={d} {opts}")


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (2, 2), (32, 2)])
@pytest.mark.parametrize("opts", [dict(), dict(decode_split=12.0)])
def test_attention_sink_decode_only(d, hq, hkv, opts):
    """The sink-and-rival values in a launch of decode rows only (the
    decode-only kernel): groups of at most 8 (query row x head) rows, whose
    padding rows carry the bf16 residual of P through the same MMAs (G = 4
    with one row, G = 1 with one and three rows), and groups of more (G = 4
    with three rows, G = 16 with one), which take a second MMA; with and
    without the key range split into parts."""
    lens = [1500, 2100, 1800, 1301]
    rows = 1 if hq // hkv == 16 else 3  # (query row x head) rows of a decode group: at most 16
    wl = W.custom(lens, [[30, 40, 24], [50, 32, 30, 20], [40, 33, 40], [20, 21, 41]],
                  [[(1499, 1500)], [(2101 - rows, 2101)], [(1799, 1800)], [(1301 - rows, 1301)]], hq=hq, hkv=hkv,
                  d=d, seed=72)
    k, v, q = _sink_and_rival(wl, lens, d)
    out, lse, info = run_gpu(wl, k, v, q, **opts)
    assert info["num_prefill_items"] == 0 and info["num_decode_items"] > 0
    ro, rl = oracle_ref(wl, k, v, q)
    assert np.nanmax(rl) > 10.0
    compare(out, lse, ro, rl, f"decode-only sink D={d} G={hq // hkv} {opts}")


@pytest.mark.parametrize("seed", range(48))
def test_random_workloads_match_oracle(seed):
    """Seeded random shapes, layouts, query ranges and split options
    (gpu_harness.random_workload) against the oracle."""
    wl, opts = random_workload(seed)
    k, v, q = W.make_values(wl)
    out, lse, _ = run_gpu(wl, k, v, q, **opts)
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, f"random {seed}: {wl.num_q_heads}/{wl.num_kv_heads} heads, D={wl.head_dim}, {opts}")


@pytest.mark.parametrize("seed", range(24))
def test_random_workloads_on_few_ctas(seed):
    """Seeded random workloads (as above, other seeds) on 1, 2 or 5 CTAs, so
    that every CTA runs many items of mixed kinds, query-tile counts and
    head dimensions back to back."""
    wl, opts = random_workload(1000 + seed)
    num_sms = (1, 2, 5)[seed % 3]
    k, v, q = W.make_values(wl)
    out, lse, info = run_gpu(wl, k, v, q, num_sms=num_sms, **opts)
    assert info["grid"] == num_sms or info["num_items"] == 0
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, f"random {1000 + seed} on {num_sms} CTAs: {wl.num_q_heads}/{wl.num_kv_heads} heads, "
                              f"D={wl.head_dim}, {opts}")


@pytest.mark.parametrize("idx", [2, 3, 5])
def test_cuda_graph_replay_equals_eager(idx):
    """append + attention captured once in a CUDA graph and replayed: the
    calls neither synchronise nor allocate, and the kernel resets its own
    queue and merge counters, so every replay gives the eager call's bits
    (split groups included: many CTAs force them).  The decode-only batch
    (2) captures the append -> attention programmatic dependency as well."""
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    sess = MsaSession.from_workload(wl, num_sms=1000)
    try:
        assert sess.info["num_items"] > sess.info["num_groups"]
        qd = q.to(dev)
        # re-append the first 8 cached rows of sequence 0 (same values: the result is unchanged)
        assert int(wl.seq_lens[0]) >= 8
        s0 = int(wl.kv_indptr[0])
        rows = torch.arange(8)
        slot = torch.as_tensor([int(wl.block_table[0][r // 16]) * 16 + r % 16 for r in rows.tolist()],
                               dtype=torch.int64, device=dev)
        kn, vn = k[s0:s0 + 8].to(dev).contiguous(), v[s0:s0 + 8].to(dev).contiguous()
        out = torch.empty((wl.num_q_rows, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
        side = torch.cuda.Stream()
        sess.stream = side
        with torch.cuda.stream(side):
            append_kv(kn, vn, slot, kp, vp, sess.dims, stream=side)
            sess.attention(qd, kp, vp, out=out, lse=lse)
        side.synchronize()
        want_o, want_l = out.clone(), lse.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            append_kv(kn, vn, slot, kp, vp, sess.dims, stream=side)
            sess.attention(qd, kp, vp, out=out, lse=lse)
        for _ in range(3):
            out.zero_()
            lse.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), want_o.view(torch.int16))
            assert torch.equal(lse, want_l)
        assert sess.check_device()[0] == 0
        ro, rl = oracle_ref(wl, k, v, q)
        compare(out, lse, ro, rl, "graph replay")
    finally:
        sess.close()


@pytest.mark.parametrize("d", [128, 64])
def test_append_then_decode_attention_back_to_back(d):
    """The serving step's order, issued back to back with no synchronisation:
    append a new last token into every sequence's pool rows, then a
    decode-only attention launch whose rows see it, four times over with
    different values for that token and an output buffer per step.  Both
    kernels are programmatic dependents of the kernel before them and wait
    for it before touching memory; every step's result must be the one of
    its own appended values (the new key is made to dominate its row's
    softmax, and its row held NaN before the first append).  This checks
    the results of the serving order, not the wait as such: an append of
    12 rows ends long before the attention's first K/V loads, so a kernel
    copy without the wait passed it too."""
    dev = torch.device("cuda")
    wl = W.batched_decode(seed=61, num_seqs=12, len_range=(300, 2500), max_seg=4, pool_tokens=1 << 16,
                          hq=16, hkv=4, d=d)
    k, v, q = W.make_values(wl)
    last = torch.as_tensor([int(wl.kv_indptr[s + 1]) - 1 for s in range(wl.num_seqs)])
    slot = torch.as_tensor([int(wl.block_table[s][(int(wl.seq_lens[s]) - 1) // 16]) * 16 +
                            (int(wl.seq_lens[s]) - 1) % 16 for s in range(wl.num_seqs)], dtype=torch.int64)
    k0, v0 = k.clone(), v.clone()
    k0[last] = float("nan")
    v0[last] = float("nan")
    kp, vp = W.make_pool(wl, k0.to(dev), v0.to(dev))
    sess = MsaSession.from_workload(wl)
    try:
        assert sess.info["num_prefill_items"] == 0
        g = torch.Generator().manual_seed(62)
        G = wl.num_q_heads // wl.num_kv_heads
        steps = []
        for i in range(4):
            # a key along the sum of the row's query heads of its kv head:
            # score about 10, so the new token carries most of the weight
            qs = q.float().view(wl.num_seqs, wl.num_kv_heads, G, d).sum(2)
            kn = (20.0 * qs / qs.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
            vn = torch.randn((wl.num_seqs, wl.num_kv_heads, d), generator=g).to(torch.bfloat16) * (i + 1)
            steps.append((kn, vn))
        outs = []
        qd, slot_d = q.to(dev), slot.to(dev)
        new = [(kn.to(dev).contiguous(), vn.to(dev).contiguous()) for kn, vn in steps]
        for kn, vn in new:
            append_kv(kn, vn, slot_d, kp, vp, sess.dims)
            out = torch.empty((wl.num_q_rows, wl.num_q_heads, d), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
            sess.attention(qd, kp, vp, out=out, lse=lse)
            outs.append((out, lse))
        torch.cuda.synchronize()
        assert sess.check_device()[0] == 0
        for i, ((kn, vn), (out, lse)) in enumerate(zip(steps, outs)):
            ki, vi = k.clone(), v.clone()
            ki[last] = kn
            vi[last] = vn
            ro, rl = oracle_ref(wl, ki, vi, q)
            compare(out, lse, ro, rl, f"append + attention step {i} D={d}")
    finally:
        sess.close()


def test_two_sessions_on_two_streams_at_once():
    """Plans with their own workspaces launched on two streams without
    ordering between them (a decode batch and a hole-recompute batch, split
    groups in both): each result equals the same plan run alone, bit for bit.
    The kernel keeps no state outside its plan's workspace."""
    dev = torch.device("cuda")
    runs = []
    for idx in (2, 3):
        wl = W.small_config(idx)
        k, v, q = W.make_values(wl)
        kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
        sess = MsaSession.from_workload(wl, num_sms=1000)
        runs.append((wl, sess, q.to(dev), kp, vp, k, v, q))
    try:
        alone = []
        for wl, sess, qd, kp, vp, *_ in runs:
            alone.append(sess.attention(qd, kp, vp).clone())
        torch.cuda.synchronize()
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        outs = [[], []]
        for _ in range(4):
            for i, (wl, sess, qd, kp, vp, *_rest) in enumerate(runs):
                sess.stream = streams[i]
                with torch.cuda.stream(streams[i]):
                    outs[i].append(sess.attention(qd, kp, vp))
        torch.cuda.synchronize()
        for i, (wl, sess, qd, kp, vp, k, v, q) in enumerate(runs):
            assert sess.check_device()[0] == 0
            for o in outs[i]:
                assert torch.equal(o.view(torch.int16), alone[i].view(torch.int16))
    finally:
        for r in runs:
            r[1].close()


def test_repeat_calls_are_identical():
    """Merge counters reset themselves: back-to-back calls give the same bits."""
    wl = W.small_config(2)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    sess = MsaSession.from_workload(wl, num_sms=1000)
    qd = q.to(dev)
    outs = [sess.attention(qd, kp, vp).clone() for _ in range(3)]
    assert sess.check_device()[0] == 0
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])
    sess.close()


# ---------------------------------------------------------- full size --

def _sample_rows(wl, rng, per_seq=2):
    rows = []
    for s in range(wl.num_seqs):
        a, b = int(wl.q_indptr[s]), int(wl.q_indptr[s + 1])
        if b - a <= per_seq:
            rows += list(range(a, b))
        else:
            rows += [a, b - 1] + list(rng.choice(np.arange(a + 1, b - 1), size=per_seq - 2 if per_seq > 2 else 0,
                                                 replace=False))
    return np.unique(np.asarray(rows, np.int64))


@pytest.mark.parametrize("plan", ["default", "chooser"])
@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_full_size_configs_sampled(idx, plan):
    """The full workloads, checked on sampled rows (first/last row of every
    sequence plus random ones), under the default plan and under the plan
    the bench times (split factors chosen by the latency model)."""
    from kv_cache_segment_gb300 import costfit
    opts = {}
    if plan == "chooser":
        params = costfit.load_params()
        if params is None:
            pytest.skip("no fitted latency-model constants")
        opts = dict(choose_with=params)
    wl = W.config(idx)
    dev = torch.device("cuda")
    k, v, q = W.make_values(wl, device=dev)
    out, lse, _ = run_gpu(wl, k, v, q, **opts)
    rng = np.random.default_rng(idx)
    rows = _sample_rows(wl, rng, per_seq=4 if idx != 4 else 6)
    if idx == 3:
        rows = rows[rng.permutation(len(rows))[:48]]
        rows.sort()
    ro, rl = oracle_ref(wl, k.cpu(), v.cpu(), q.cpu(), rows=rows)
    compare(out[torch.as_tensor(rows, device=dev)], lse[torch.as_tensor(rows, device=dev)], ro, rl, wl.name)


def test_million_token_sequence_sampled():
    """One sequence of 2^20 + 37 cached tokens in 40 segments (pools of 4 GiB
    each), queried by a 100-row recompute range at its end and a decode row:
    positions near 2^20, key ranges split over many CTAs and merged; checked
    on sampled rows."""
    L = (1 << 20) + 37
    nb = -(-L // 16)
    rng = np.random.default_rng(20)
    cuts = np.sort(rng.choice(np.arange(1, nb), size=39, replace=False))
    sizes = np.diff(np.concatenate([[0], cuts, [nb]])).tolist()
    wl = W.custom([L], [sizes], [[(L - 100, L + 1)]], hq=32, hkv=8, seed=21)
    dev = torch.device("cuda")
    k, v, q = W.make_values(wl, device=dev)
    out, lse, info = run_gpu(wl, k, v, q)
    assert info["num_items"] > info["num_groups"]  # split groups, merged by the last part
    rows = np.array([0, 1, 50, 98, 99, 100], np.int64)
    ro, rl = oracle_ref(wl, k.cpu(), v.cpu(), q.cpu(), rows=rows)
    sel = torch.as_tensor(rows, device=dev)
    compare(out[sel], lse[sel], ro, rl, "2^20-token sequence")


def test_misaligned_pointers_are_rejected_before_launch():
    """q and out must be 16-byte aligned (TMA, vector stores): a misaligned
    pointer comes back as MSA_ERR_INVALID_ARG and nothing is written."""
    wl = W.small_config(2)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    sess = MsaSession.from_workload(wl)
    try:
        qd = q.to(dev)
        n = qd.numel()
        big = torch.full((n + 8,), 7.0, dtype=torch.bfloat16, device=dev)
        out_bad = big[1:n + 1].view(qd.shape)  # 2 bytes past a 16-byte boundary
        with pytest.raises(msa.MsaError) as e:
            sess.attention(qd, kp, vp, out=out_bad)
        assert e.value.status == msa.MSA_ERR_INVALID_ARG
        torch.cuda.synchronize()
        assert torch.all(big == 7.0)
        qbig = torch.zeros((n + 8,), dtype=torch.bfloat16, device=dev)
        qbig[1:n + 1] = qd.reshape(-1)
        with pytest.raises(msa.MsaError) as e:
            sess.attention(qbig[1:n + 1].view(qd.shape), kp, vp)
        assert e.value.status == msa.MSA_ERR_INVALID_ARG
    finally:
        sess.close()


def test_wrong_tensors_are_refused_before_launch():
    """MsaSession.attention / append_kv check dtype, shape, contiguity and
    device of every tensor: a mis-shaped lse would otherwise be written past
    its end."""
    wl = W.small_config(2)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    sess = MsaSession.from_workload(wl)
    try:
        qd = q.to(dev)
        n_q, hq = qd.shape[0], qd.shape[1]
        with pytest.raises(TypeError):
            sess.attention(qd.half(), kp, vp)
        with pytest.raises(ValueError):
            sess.attention(qd, kp, vp, lse=torch.empty((n_q - 1, hq), dtype=torch.float32, device=dev))
        with pytest.raises(ValueError):
            sess.attention(qd[:-1], kp, vp)
        with pytest.raises(ValueError):
            sess.attention(qd, kp.transpose(1, 2).contiguous().transpose(1, 2), vp)
        with pytest.raises(ValueError):
            sess.attention(qd, kp, vp[:-1])
        with pytest.raises(ValueError):
            append_kv(kp[:4], vp[:4], torch.zeros(3, dtype=torch.int64, device=dev), kp, vp, sess.dims)
        torch.cuda.synchronize()
        assert sess.check_device()[0] == 0
    finally:
        sess.close()


def test_bounded_wait_runs_out_and_the_context_survives():
    """A wait on a barrier nothing arrives at gives up after its limit, the
    error bit reaches the host, a second waiter leaves on the abort flag, and
    the device keeps working (an attention call right after is exact)."""
    import time
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    msa.msa_selftest_wait_timeout(50_000_000, words, torch.cuda.current_stream())  # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert words[0].item() == msa.MSA_DEVERR_TIMEOUT_COMPUTE
    assert words[1].item() == 1
    assert 0.045 < dt < 2.0
    wl = W.small_config(1)
    k, v, q = W.make_values(wl)
    out, lse, _ = run_gpu(wl, k, v, q)
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out, lse, ro, rl, "after a timed-out wait")


@pytest.mark.parametrize("idx", [5, 3])
def test_device_check_clears_counters_left_by_an_aborted_launch(idx):
    """A launch that gave up can leave the merge counters of split groups (and
    the queue head) mid-count.  Stand in for one from the host: put nonzero
    counts there and set an error bit.  msa_plan_check_device reports the
    error and zeroes the counters with the word, so the next launch with the
    plan (split groups merged by the last part to arrive) is exact."""
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    sess = MsaSession.from_workload(wl, decode_split=12.0, prefill_split=16.0)
    try:
        info = sess.info
        a, nb = info["counters_offset"], info["counters_bytes"]
        assert nb > 0 and info["num_items"] > info["num_groups"]  # some groups are split
        sess.workspace[a:a + nb].fill_(1)            # every counter at 0x01010101
        sess.workspace[0:4].view(torch.int32).fill_(msa.MSA_DEVERR_TIMEOUT_COMPUTE)
        rc, word = sess.check_device()
        assert rc == msa.MSA_ERR_DEVICE_CHECK and word == msa.MSA_DEVERR_TIMEOUT_COMPUTE
        assert int(sess.workspace[a:a + nb].count_nonzero()) == 0
        assert int(sess.workspace[0:4].count_nonzero()) == 0
        lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
        out = sess.attention(q.to(dev), kp, vp, lse=lse)
        assert sess.check_device() == (0, 0)
        ro, rl = oracle_ref(wl, k, v, q)
        compare(out, lse, ro, rl, "after the counters were cleared")
    finally:
        sess.close()


@pytest.mark.parametrize("budget", [0.0, 31.0])
def test_chosen_prefill_chunk_step_matches_oracle(budget):
    """A serving step as msa_choose_prefill_chunk plans it: the small mixed
    batch's decode rows plus the chosen chunk of each pending prefill (the
    chunk's own K/V in the cache, rows [start, start + c)), run through the
    C ABI and compared with the oracle on the same step."""
    from kv_cache_segment_gb300 import costfit
    params = costfit.load_params()
    if params is None:
        pytest.skip("no fitted latency-model constants")
    wl = W.small_config(5)
    base, pending = W.pending_prefills(wl, remaining=500)
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    choice, cands, _ = msa.msa_choose_prefill_chunk(dims, base.block_table, base.seq_lens, base.q_range_indptr,
                                                    base.q_ranges_flat, pending, params, budget_us=budget,
                                                    granularity=64)
    assert choice["chunk"] in cands.tolist()
    step = W.with_prefill_chunk(base, pending, choice["chunk"])
    assert step.num_q_rows == sum(1 for rs in base.q_ranges for _ in rs) + choice["tokens"]
    k, v, q = W.make_values(step)
    out, lse, info = run_gpu(step, k, v, q)
    ro, rl = oracle_ref(step, k, v, q)
    compare(out, lse, ro, rl, f"chosen chunk {choice['chunk']}")


@pytest.mark.parametrize("name", ["decode", "holes", "mixed", "long", "holes_d64", "mixed_d64"])
def test_latency_model_predicts_measured_launches(name):
    """The shipped latency-model constants predict the measured launch time
    (back to back, as costfit measures and the bench times) of medium
    workloads it was not fitted on within 10 %, at head dims 128 and 64."""
    from kv_cache_segment_gb300 import costfit
    params = costfit.load_params()
    if params is None:
        pytest.skip("no fitted latency-model constants")
    wl = {"decode": lambda: W.batched_decode(seed=4001, num_seqs=40, len_range=(2048, 12288), max_seg=6,
                                             pool_tokens=1 << 20),
          "holes": lambda: W.hole_recompute(seed=4002, num_seqs=6, cached_blocks=448, evict_blocks=96),
          "mixed": lambda: W.mixed_batch(seed=4003, num_decode=48, num_prefill=2, chunk=1536),
          "long": lambda: W.long_context(seed=4004, num_seqs=1, length=40960, n_runs=24, chunk=1024),
          "holes_d64": lambda: W.hole_recompute(seed=4005, num_seqs=6, cached_blocks=448, evict_blocks=96, d=64),
          "mixed_d64": lambda: W.mixed_batch(seed=4006, num_decode=48, num_prefill=2, chunk=1536, d=64)}[name]()
    us, sess = costfit.measure(wl, torch.device("cuda"), reps=9, splits=((0.0, 0.0),))[0]
    try:
        pred = msa.msa_plan_estimate(sess.plan, params)["time_us"]
    finally:
        sess.close()
    assert abs(pred / us - 1.0) < 0.10, (name, pred, us)
