"""Kernel-aware eviction choice (msa_select_evictions) against the plain
restatement in oracle/eviction.py and closed forms."""
import numpy as np
import pytest

import oracle.costmodel as OC
import oracle.eviction as OE
from kv_cache_segment_gb300 import msa

PARAMS = dict(launch_us=17.3, dec_item_us=0.0, dec_gbs=7565.0, dec_cta_gbs=59.4, pre_item_us=30.1, pre_tile_us=0.787,
              box_us=0.0, dec_merge_us=8.43, pre_merge_us=20.0)


def _dims(hq=32, hkv=8, d=128):
    return msa.make_dims(hq, hkv, d)


@pytest.mark.parametrize("seed", range(24))
def test_library_matches_oracle(seed):
    """Random lengths, probabilities, weights and modes; every third case at
    head dim 64 with part of a tile's time proportional to D, where the
    costs take the latency model's tile time at that head dim."""
    rng = np.random.default_rng(seed)
    d = 64 if seed % 3 == 1 else 128
    params = dict(PARAMS, pre_tile_dfrac=0.55) if seed % 6 == 1 else PARAMS
    L = int(rng.integers(1, 5000))
    nb = -(-L // 16)
    hit = rng.random(nb).astype(np.float32)
    if seed % 2:
        hit = np.round(hit * 4) / 4  # many ties
    alpha, beta = float(rng.random() * 2), float(rng.random() * 2)
    n = int(rng.integers(0, nb + 1))
    expected, prefix = seed % 3 == 2, seed % 4 >= 2
    mode = (msa.MSA_EVICT_EXPECTED_COST if expected else 0) | (msa.MSA_EVICT_PREFIX_COST if prefix else 0)
    ev, cost = msa.msa_select_evictions(_dims(d=d), L, hit, alpha, beta, params, n, mode=mode)
    want, want_cost = OE.select_evictions(L, 32, hit, alpha, beta, OC.tile_us(params, d), n, expected_cost=expected,
                                          prefix=prefix)
    assert ev.tolist() == want
    # the suffix sums may add in another order: equal to the last few ulps
    assert np.allclose(cost, want_cost, rtol=1e-13 if prefix else 0, atol=0)


def test_hit_only_evicts_the_least_likely_blocks():
    L = 40 * 16
    hit = np.linspace(1.0, 0.0, 40).astype(np.float32)  # later blocks less likely to be hit
    ev, _ = msa.msa_select_evictions(_dims(), L, hit, 1.0, 0.0, PARAMS, 10)
    assert ev.tolist() == list(range(30, 40))


def test_cost_only_evicts_the_earliest_blocks():
    """Recompute work grows with position: with beta alone the first blocks go."""
    L = 40 * 16 + 5
    hit = np.full(41, 0.5, np.float32)
    ev, cost = msa.msa_select_evictions(_dims(), L, hit, 0.0, 1.0, PARAMS, 7)
    assert ev.tolist() == list(range(7))
    assert np.all(np.diff(cost[:-1]) > 0)


def test_prefix_reading_evicts_the_tail_first():
    """Prefix reading, beta alone: the cost of evicting block b is the
    recompute of b .. end, which falls with position, so the last blocks go."""
    L = 40 * 16 + 5
    hit = np.full(41, 0.5, np.float32)
    ev, cost = msa.msa_select_evictions(_dims(), L, hit, 0.0, 1.0, PARAMS, 7, mode=msa.MSA_EVICT_PREFIX_COST)
    assert ev.tolist() == list(range(34, 41))
    assert np.all(np.diff(cost) < 0)


@pytest.mark.parametrize("b", [0, 1, 31, 62])
def test_prefix_cost_closed_form(b):
    """prefix cost(b) = pre_tile_us * Hq * (L(L+1) - 16b(16b+1)) / 2 / 128^2."""
    L, hq = 1000, 32
    _, cost = msa.msa_select_evictions(_dims(hq), L, np.zeros(63, np.float32), 1.0, 1.0, PARAMS, 0,
                                       mode=msa.MSA_EVICT_PREFIX_COST)
    want = PARAMS["pre_tile_us"] * hq * ((L * (L + 1) - 16 * b * (16 * b + 1)) // 2) / 16384
    assert cost[b] == pytest.approx(want, rel=1e-13)


@pytest.mark.parametrize("b,L", [(0, 1000), (10, 1000), (62, 1000)])
def test_block_cost_closed_form(b, L):
    """cost = pre_tile_us * Hq * sum_{p in block} (p + 1) / 128^2."""
    hq = 32
    lo, hi = 16 * b, min(16 * b + 16, L)
    keys = (hi * (hi + 1) - lo * (lo + 1)) // 2
    _, cost = msa.msa_select_evictions(_dims(hq), L, np.zeros(-(-L // 16), np.float32), 1.0, 1.0, PARAMS, 0)
    assert cost[b] == pytest.approx(PARAMS["pre_tile_us"] * hq * keys / 16384, rel=1e-15)


def test_equal_scores_evict_lower_blocks_first():
    L = 20 * 16
    ev, _ = msa.msa_select_evictions(_dims(), L, np.full(20, 0.3, np.float32), 1.0, 0.0, PARAMS, 5)
    assert ev.tolist() == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("kw", [dict(n=-1), dict(n=99), dict(alpha=-1.0), dict(beta=float("nan")), dict(bad_p=True)])
def test_bad_arguments(kw):
    L = 10 * 16
    hit = np.full(10, 0.5, np.float32)
    if kw.get("bad_p"):
        hit[3] = 1.5
    with pytest.raises(msa.MsaError) as e:
        msa.msa_select_evictions(_dims(), L, hit, kw.get("alpha", 1.0), kw.get("beta", 1.0), PARAMS, kw.get("n", 2))
    assert e.value.status == msa.MSA_ERR_INVALID_ARG


def test_expected_cost_mode_minimises_expected_recompute():
    """Brute force on a tiny sequence: no other set of n blocks has a lower
    sum of hit * cost than the one chosen in expected-cost mode."""
    import itertools
    rng = np.random.default_rng(3)
    L = 9 * 16 - 3
    hit = rng.random(9).astype(np.float32)
    for n in range(0, 10):
        ev, cost = msa.msa_select_evictions(_dims(), L, hit, 0.0, 0.0, PARAMS, n, mode=msa.MSA_EVICT_EXPECTED_COST)
        got = float((hit[ev].astype(np.float64) * cost[ev]).sum())
        best = min(float(sum(hit[i] * cost[i] for i in c)) for c in itertools.combinations(range(9), n))
        assert got == pytest.approx(best, rel=1e-12, abs=1e-12)


def test_unknown_mode_is_rejected():
    with pytest.raises(msa.MsaError) as e:
        msa.msa_select_evictions(_dims(), 160, np.zeros(10, np.float32), 1.0, 1.0, PARAMS, 2, mode=4)
    assert e.value.status == msa.MSA_ERR_INVALID_ARG


def test_block_cost_scales_with_the_head_dim_term():
    """With pre_tile_dfrac = 0.5 a block's cost at D = 64 is 3/4 of its cost
    at D = 128; without the term the two are equal; a share outside [0, 1] is
    rejected."""
    L = 10 * 16
    hit = np.full(10, 0.5, np.float32)
    p = dict(PARAMS, pre_tile_dfrac=0.5)
    _, c128 = msa.msa_select_evictions(_dims(d=128), L, hit, 1.0, 1.0, p, 2)
    _, c64 = msa.msa_select_evictions(_dims(d=64), L, hit, 1.0, 1.0, p, 2)
    _, c64_flat = msa.msa_select_evictions(_dims(d=64), L, hit, 1.0, 1.0, PARAMS, 2)
    assert np.allclose(c64, 0.75 * c128, rtol=1e-15, atol=0)
    assert np.array_equal(c64_flat, c128)
    for bad in (-0.5, 2.0):
        with pytest.raises(msa.MsaError):
            msa.msa_select_evictions(_dims(d=64), L, hit, 1.0, 1.0, dict(PARAMS, pre_tile_dfrac=bad), 2)
