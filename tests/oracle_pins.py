"""Pins for the float64 oracle: checks against facts that do not come from
the oracle itself (hand-worked scores, closed forms, textbook library
routines, brute force, invariances the method's losslessness demands).

Each pin takes an optional `lib` (a bound build of oracle.c) so that the
same checks can be run against copies of the oracle with planted mistakes.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_bits(x):
    """Round float values to bf16 bit patterns (round-to-nearest-even via torch)."""
    import torch
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f64(b):
    b = np.asarray(b, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _dense(lib, k_bits, v_bits, q_bits, lens, q_counts, q_pos, hq, hkv, scale):
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q_indptr = np.concatenate([[0], np.cumsum(q_counts)]).astype(np.int64)
    return oracle.dense_attention(kv_indptr, k_bits, v_bits, q_indptr, q_pos, q_bits, hq, hkv, scale,
                                  num_threads=2, lib=lib)


def _paged(lens, k_log, v_log, runs_per_seq, order_seed, pool_factor=3, fill=np.nan, block=16):
    """Lay out logical K/V (float arrays) in a pool: runs_per_seq[s] = run sizes
    in blocks; runs placed in a shuffled order with one free block between
    them.  Returns (table, k_pool_bits, v_pool_bits)."""
    rng = np.random.default_rng(order_seed)
    items = [(s, i) for s, rs in enumerate(runs_per_seq) for i in range(len(rs))]
    rng.shuffle(items)
    starts = {}
    pos = 1
    for s, i in items:
        starts[(s, i)] = pos
        pos += runs_per_seq[s][i] + 1 + int(rng.integers(0, 3))
    pool_blocks = pos + 1
    hkv, d = k_log.shape[1], k_log.shape[2]
    kp = np.full((pool_blocks * block, hkv, d), fill, np.float32)
    vp = np.full((pool_blocks * block, hkv, d), fill, np.float32)
    max_blocks = max(sum(r) for r in runs_per_seq)
    table = np.full((len(lens), max_blocks), -1, np.int32)
    off = np.concatenate([[0], np.cumsum(lens)])
    for s, rs in enumerate(runs_per_seq):
        b = 0
        for i, n in enumerate(rs):
            table[s, b:b + n] = np.arange(starts[(s, i)], starts[(s, i)] + n)
            b += n
        for t in range(lens[s]):
            row = table[s, t // block] * block + t % block
            kp[row] = k_log[off[s] + t]
            vp[row] = v_log[off[s] + t]
    return table, bf16_bits(kp), bf16_bits(vp)


# ---------------------------------------------------------------- pins --

def pin_hand_cases(lib=None):
    """Hand-worked scores (tests/golden/hand_cases.json)."""
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        hq, hkv, d = c["num_q_heads"], c["num_kv_heads"], c["head_dim"]
        L = len(c["K"])
        k = bf16_bits(np.asarray(c["K"], np.float32).reshape(L, hkv, d))
        v = bf16_bits(np.asarray(c["V"], np.float32).reshape(L, hkv, d))
        q = bf16_bits(np.asarray(c["q"], np.float32))
        n = q.shape[0]
        out, lse = _dense(lib, k, v, q, [L], [n], np.asarray(c["q_pos"], np.int32), hq, hkv, c["scale"])
        vf = bits_to_f64(v)
        for i in range(n):
            for h in range(hq):
                vis = c["visible"][i][h]
                t = c["scores"][i][h]
                if not vis:
                    assert lse[i, h] == -math.inf, (c["name"], i, h, lse[i, h])
                    assert np.all(out[i, h] == 0.0)
                    continue
                z = sum(math.exp(x) for x in t)
                assert abs(lse[i, h] - math.log(z)) < 1e-13, (c["name"], i, h, lse[i, h], math.log(z))
                g = h // (hq // hkv)
                want = sum((math.exp(x) / z) * vf[j, g] for x, j in zip(t, vis))
                assert np.max(np.abs(out[i, h] - want)) < 1e-13, (c["name"], i, h, out[i, h], want)


def pin_uniform_when_q_zero(lib=None):
    """q = 0 makes every visible score equal: out = mean of the visible V rows
    and lse = ln(number of visible keys), for every causal row."""
    rng = np.random.default_rng(1)
    L, hkv, hq, d = 37, 2, 4, 8
    v = bf16_bits(rng.standard_normal((L, hkv, d)))
    k = bf16_bits(rng.standard_normal((L, hkv, d)))
    pos = np.array([0, 1, 5, 17, 36, 37, 40], np.int32)
    q = np.zeros((len(pos), hq, d), np.uint16)
    out, lse = _dense(lib, k, v, q, [L], [len(pos)], pos, hq, hkv, 0.3)
    vf = bits_to_f64(v)
    for i, p in enumerate(pos):
        n = min(p + 1, L)
        for h in range(hq):
            g = h // (hq // hkv)
            assert abs(lse[i, h] - math.log(n)) < 1e-13, (p, h, lse[i, h])
            assert np.max(np.abs(out[i, h] - vf[:n, g].mean(0))) < 1e-13


def pin_identical_keys(lib=None):
    """All keys equal: weights uniform whatever q is, out = mean of visible V."""
    rng = np.random.default_rng(2)
    L, d = 20, 4
    k = np.tile(bf16_bits(rng.standard_normal((1, 1, d))), (L, 1, 1))
    v = bf16_bits(rng.standard_normal((L, 1, d)))
    q = bf16_bits(rng.standard_normal((3, 1, d)))
    pos = np.array([3, 11, 25], np.int32)
    out, lse = _dense(lib, k, v, q, [L], [3], pos, 1, 1, 0.5)
    vf = bits_to_f64(v)
    kf = bits_to_f64(k)
    qf = bits_to_f64(q)
    for i, p in enumerate(pos):
        n = min(p + 1, L)
        t0 = 0.5 * float(np.dot(qf[i, 0], kf[0, 0]))
        assert abs(lse[i, 0] - (t0 + math.log(n))) < 1e-12
        assert np.max(np.abs(out[i, 0] - vf[:n, 0].mean(0))) < 1e-13


def pin_dominant_key(lib=None):
    """One key's score exceeds the others by > 50: out equals that key's V
    to within exp(-50)."""
    L, d = 9, 2
    kf = np.zeros((L, 1, d), np.float32)
    kf[4, 0] = [8.0, 0.0]
    vf = np.arange(L * d, dtype=np.float32).reshape(L, 1, d) - 5.0
    k, v = bf16_bits(kf), bf16_bits(vf)
    q = bf16_bits(np.array([[[8.0, 1.0]]], np.float32))
    out, lse = _dense(lib, k, v, q, [L], [1], np.array([8], np.int32), 1, 1, 1.0)
    assert np.max(np.abs(out[0, 0] - bits_to_f64(v)[4, 0])) < 1e-12
    # lse = 64 + ln(1 + 8 e^-64) ~ 64
    assert abs(lse[0, 0] - 64.0) < 1e-12


def pin_single_key(lib=None):
    """L = 1: out = V_0 and lse = scale * q.k_0 (pins the scale inside lse)."""
    rng = np.random.default_rng(3)
    d = 16
    k = bf16_bits(rng.standard_normal((1, 2, d)))
    v = bf16_bits(rng.standard_normal((1, 2, d)))
    q = bf16_bits(rng.standard_normal((2, 4, d)))
    pos = np.array([0, 7], np.int32)
    scale = 0.125
    out, lse = _dense(lib, k, v, q, [1], [2], pos, 4, 2, scale)
    kf, vf, qf = bits_to_f64(k), bits_to_f64(v), bits_to_f64(q)
    for i in range(2):
        for h in range(4):
            g = h // 2
            assert abs(lse[i, h] - scale * float(np.dot(qf[i, h], kf[0, g]))) < 1e-13
            assert np.max(np.abs(out[i, h] - vf[0, g])) < 1e-15


def pin_brute_force_tiny(lib=None):
    """Random tiny cases against the explicit-softmax loop version (brute.py)."""
    rng = np.random.default_rng(4)
    for trial in range(40):
        L = int(rng.integers(1, 9))
        d = int(rng.integers(1, 3))
        hkv = int(rng.integers(1, 3))
        hq = hkv * int(rng.integers(1, 3))
        n = int(rng.integers(1, 5))
        k = bf16_bits(rng.standard_normal((L, hkv, d)) * 2)
        v = bf16_bits(rng.standard_normal((L, hkv, d)))
        q = bf16_bits(rng.standard_normal((n, hq, d)) * 2)
        pos = np.sort(rng.choice(L + 1, size=n, replace=False)).astype(np.int32) if n <= L + 1 else \
            np.arange(n, dtype=np.int32)
        scale = float(rng.uniform(0.1, 1.5))
        out, lse = _dense(lib, k, v, q, [L], [n], pos, hq, hkv, scale)
        bo, bl = brute.attention_tiny(bits_to_f64(k), bits_to_f64(v), bits_to_f64(q), pos, hkv, scale)
        assert np.max(np.abs(out - bo)) < 1e-13, trial
        assert np.max(np.abs(lse - bl)) < 1e-13, trial


def pin_textbook_causal_attention(lib=None):
    """A whole sequence queried at every position (one segment, one range) is
    textbook causal attention: compare with torch's scaled_dot_product_attention
    in float64 (is_causal, default scale 1/sqrt(D), GQA by repeating each kv
    head over its consecutive query heads), and lse with scipy's logsumexp of
    the masked score matrix."""
    import torch
    from scipy.special import logsumexp
    rng = np.random.default_rng(5)
    L, hq, hkv, d = 70, 6, 2, 32
    k = bf16_bits(rng.standard_normal((L, hkv, d)))
    v = bf16_bits(rng.standard_normal((L, hkv, d)))
    q = bf16_bits(rng.standard_normal((L, hq, d)))
    scale = 1.0 / math.sqrt(d)
    out, lse = _dense(lib, k, v, q, [L], [L], np.arange(L, dtype=np.int32), hq, hkv, scale)
    G = hq // hkv
    kt = torch.from_numpy(bits_to_f64(k)).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(bits_to_f64(v)).permute(1, 0, 2).repeat_interleave(G, 0)
    qt = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    ref = ref.permute(1, 0, 2).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12
    scores = torch.matmul(qt, kt.transpose(1, 2)).numpy() * scale  # [hq, L, L]
    mask = np.tril(np.ones((L, L), bool))
    scores = np.where(mask[None], scores, -np.inf)
    ref_lse = logsumexp(scores, axis=-1).T  # [L, hq]
    assert np.max(np.abs(lse - ref_lse)) < 1e-12


def _segmented_case(lens, runs_per_seq, q_ranges, hq, hkv, d, seed, layout_seed, lib=None):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    kf = rng.standard_normal((T, hkv, d)).astype(np.float32)
    vf = rng.standard_normal((T, hkv, d)).astype(np.float32)
    q_pos = np.concatenate([np.arange(a, b) for rs in q_ranges for a, b in rs]).astype(np.int32)
    q_counts = [sum(b - a for a, b in rs) for rs in q_ranges]
    q = bf16_bits(rng.standard_normal((len(q_pos), hq, d)))
    k, v = bf16_bits(kf), bf16_bits(vf)
    dense = _dense(lib, k, v, q, lens, q_counts, q_pos, hq, hkv, 1.0 / math.sqrt(d))
    table, kp, vp = _paged(lens, bits_to_f64(k).astype(np.float32), bits_to_f64(v).astype(np.float32),
                           runs_per_seq, layout_seed)
    q_indptr = np.concatenate([[0], np.cumsum(q_counts)]).astype(np.int64)
    seg = oracle.segmented_attention(table, np.asarray(lens, np.int32), kp, vp, q_indptr, q_pos, q, hq,
                                     hkv, 16, 1.0 / math.sqrt(d), num_threads=2, lib=lib)
    return dense, seg


def pin_segment_merge_identity(lib=None):
    """Per-segment attention merged by log-sum-exp equals dense attention over
    the logical sequence (the exactness MSA claims), on ragged lengths,
    several segments, hole-like query ranges and a decode row; the pool's
    unused rows hold NaN, so any read outside the live rows shows."""
    lens = [100, 37, 256]
    runs = [[2, 3, 2], [3], [1, 4, 6, 5]]
    q_ranges = [[(0, 5), (40, 60), (100, 101)], [(37, 38)], [(16, 80), (200, 256)]]
    (do, dl), (so, sl) = _segmented_case(lens, runs, q_ranges, 4, 2, 16, 11, 12, lib)
    assert np.all(np.isfinite(so)) and np.all(np.isfinite(sl))
    assert np.max(np.abs(do - so)) < 1e-12
    assert np.max(np.abs(dl - sl)) < 1e-12


def pin_layout_invariance(lib=None):
    """Lossless management must not depend on where blocks live: the same
    logical K/V as one segment, as many segments, and with the pool order
    shuffled give the same result (within 1e-12)."""
    lens = [150]
    q_ranges = [[(0, 10), (60, 90), (149, 151)]]
    ref = None
    for runs, lseed in (([10], 1), ([1] * 10, 2), ([3, 3, 4], 3), ([2, 5, 1, 2], 4)):
        (_, _), (so, sl) = _segmented_case(lens, [runs], q_ranges, 2, 1, 8, 21, lseed, lib)
        if ref is None:
            ref = (so, sl)
        else:
            assert np.max(np.abs(ref[0] - so)) < 1e-12
            assert np.max(np.abs(ref[1] - sl)) < 1e-12


def pin_segment_splitter():
    """The C splitter matches the pure-Python brute-force scan (segments.py)
    on random tables, including partial last blocks."""
    from oracle import segments
    rng = np.random.default_rng(6)
    for _ in range(500):
        nb = int(rng.integers(1, 40))
        base = rng.permutation(200)[:nb]
        table = base.copy()
        # make some neighbours physically consecutive
        for b in range(1, nb):
            if rng.random() < 0.6:
                table[b] = table[b - 1] + 1
        L = (nb - 1) * 16 + int(rng.integers(1, 17))
        want = segments.split_into_contiguous_segments(table, L, 16)
        got = oracle.segment_runs(table.astype(np.int32), nb)
        assert [tuple(w[:3]) for w in want] == [tuple(int(x) for x in g) for g in got]


def pin_scatter():
    """Scatter reference equals numpy fancy assignment (slot -1 skipped)."""
    rng = np.random.default_rng(7)
    pool = rng.integers(0, 65535, size=(64, 2, 8)).astype(np.uint16)
    src = rng.integers(0, 65535, size=(10, 2, 8)).astype(np.uint16)
    slot = rng.choice(64, size=10, replace=False).astype(np.int64)
    slot[3] = -1
    want = pool.copy()
    keep = slot >= 0
    want[slot[keep]] = src[keep]
    got = oracle.scatter_rows(src, slot, pool.copy())
    assert np.array_equal(got, want)


ATTENTION_PINS = [pin_hand_cases, pin_uniform_when_q_zero, pin_identical_keys, pin_dominant_key,
                  pin_single_key, pin_brute_force_tiny, pin_textbook_causal_attention,
                  pin_segment_merge_identity, pin_layout_invariance]
