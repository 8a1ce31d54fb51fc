"""Seeded synthetic workloads for Multi-Segment Attention.

This module only draws inputs: sequence lengths, how each sequence's blocks
are scattered over the paged pool, which positions are queried, and the bf16
Q/K/V values.  It holds none of the method's arithmetic (no segment
splitting, no attention); both the CUDA path's tests/bench and the CPU oracle
consume what it draws.

Recipes follow the five workload shapes the MSA pages motivate (a cache with
eviction holes that are later recomputed, multi-turn dialogue, long context,
continuous batching):

  1 tiny_decode        1 seq, 4/4 heads, D=64, 256 tokens as 3 runs
                       (logical blocks 0-3, 4-9, 10-15) at shuffled
                       non-adjacent offsets of a 64-block pool; 1 query at 256.
  2 batched_decode     32 seqs, 32/8 heads, D=128, L ~ U{2048..16384}, each
                       split into U{1..8} runs at uniform interior block
                       boundaries, placed at random in a 4,194,304-token
                       pool; 1 query per seq at p = L.
  3 hole_recompute     16 seqs of 8192 cached tokens originally one run;
                       128 blocks (25 %) evicted in holes of U{2..32} blocks;
                       every hole's recomputed K/V lives in a fresh run
                       elsewhere; a 512-token new turn in another fresh run;
                       queries = every hole position + [8192, 8704).
  4 long_context       4 seqs of 131072 tokens in 64 runs with geometric
                       lengths (p = 1/128, rescaled to 8192 blocks by largest
                       remainder, min 1) in a 2x pool; queries
                       [129024, 131072) + one decode token at 131072.
  5 mixed_batch        64 decode + 4 prefill seqs, 64/8 heads, lengths
                       round(LogNormal(ln 4096, 1.0)) clipped to [16, 32768]
                       (prefill seqs redrawn until >= 2048), U{1..min(32,
                       blocks)} runs; prefill queries [L-2048, L).

Runs are always separated in the pool by at least one free block, so no two
runs of a sequence can touch physically and the drawn run count is exactly
the number of segments.  Values: fp32 N(0, 1) from a seeded torch generator,
rounded to bf16 (round-to-nearest-even).  Seeds default to 1000 + config id.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

BLOCK = 16


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seq_lens: np.ndarray          # int32 [S]
    block_table: np.ndarray       # int32 [S, max_blocks], -1 = no block
    pool_blocks: int
    q_ranges: List[List[Tuple[int, int]]]  # per seq, half-open [start, end)
    runs_drawn: List[List[Tuple[int, int, int]]]  # per seq (log block, phys block, n blocks)
    seed: int

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def pool_tokens(self) -> int:
        return self.pool_blocks * self.block_size

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def q_range_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum([len(r) for r in self.q_ranges])]).astype(np.int32)

    @property
    def q_ranges_flat(self) -> np.ndarray:
        flat = [list(r) for rs in self.q_ranges for r in rs]
        return np.asarray(flat, np.int32).reshape(-1, 2)

    @property
    def q_pos(self) -> np.ndarray:
        """Logical position of every packed query row, in (seq, range, position) order."""
        pos = [np.arange(a, b, dtype=np.int32) for rs in self.q_ranges for (a, b) in rs]
        return np.concatenate(pos).astype(np.int32) if pos else np.zeros(0, np.int32)

    @property
    def q_indptr(self) -> np.ndarray:
        counts = [sum(b - a for a, b in rs) for rs in self.q_ranges]
        return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)

    @property
    def kv_indptr(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens.astype(np.int64))]).astype(np.int64)

    @property
    def num_q_rows(self) -> int:
        return int(self.q_indptr[-1])

    def slot_mapping(self) -> np.ndarray:
        """Pool row of every logical token (all sequences, logical order), int64."""
        out = []
        for s in range(self.num_seqs):
            t = np.arange(int(self.seq_lens[s]), dtype=np.int64)
            out.append(self.block_table[s, t // self.block_size].astype(np.int64) * self.block_size
                       + t % self.block_size)
        return np.concatenate(out) if out else np.zeros(0, np.int64)


# ------------------------------------------------------------------ layout --

def _stars_and_bars(rng, total: int, bins: int) -> np.ndarray:
    """Uniformly random composition of `total` into `bins` non-negative parts."""
    if bins == 1:
        return np.array([total], np.int64)
    bars = np.sort(rng.choice(total + bins - 1, size=bins - 1, replace=False))
    edges = np.concatenate([[-1], bars, [total + bins - 1]])
    return (np.diff(edges) - 1).astype(np.int64)


def _place_extents(rng, sizes: Sequence[int], pool_blocks: int) -> np.ndarray:
    """Random non-overlapping placement of extents (sizes in blocks) with at
    least one free block between any two, in a random order."""
    n = len(sizes)
    need = int(sum(sizes)) + max(n - 1, 0)
    if need > pool_blocks:
        raise ValueError(f"pool of {pool_blocks} blocks cannot hold {need}")
    gaps = _stars_and_bars(rng, pool_blocks - need, n + 1)
    order = rng.permutation(n)
    starts = np.zeros(n, np.int64)
    pos = 0
    for i, idx in enumerate(order):
        pos += int(gaps[i]) + (1 if i > 0 else 0)
        starts[idx] = pos
        pos += int(sizes[idx])
    return starts


class _Layout:
    """Collects runs in logical order per sequence, grouped into extents
    (an extent is a stretch of pool placed as a unit; a run sits at a fixed
    offset inside its extent)."""

    def __init__(self, num_seqs: int):
        self.extents: List[int] = []
        self.runs: List[List[Tuple[int, int, int]]] = [[] for _ in range(num_seqs)]  # (n_blocks, extent, offset)

    def extent(self, size: int) -> int:
        self.extents.append(int(size))
        return len(self.extents) - 1

    def run(self, seq: int, n_blocks: int, extent: Optional[int] = None, offset: int = 0):
        if extent is None:
            extent = self.extent(n_blocks)
        self.runs[seq].append((int(n_blocks), extent, int(offset)))

    def realise(self, rng, seq_lens, pool_blocks):
        starts = _place_extents(rng, self.extents, pool_blocks)
        max_blocks = max(sum(r[0] for r in rs) for rs in self.runs)
        table = np.full((len(self.runs), max(max_blocks, 1)), -1, np.int32)
        drawn = []
        for s, rs in enumerate(self.runs):
            b = 0
            seq_runs = []
            for n_blocks, ext, off in rs:
                phys = int(starts[ext]) + off
                table[s, b:b + n_blocks] = np.arange(phys, phys + n_blocks, dtype=np.int32)
                seq_runs.append((b, phys, n_blocks))
                b += n_blocks
            assert b == -(-int(seq_lens[s]) // BLOCK), (s, b, seq_lens[s])
            drawn.append(seq_runs)
        return table, drawn


def _cut_sizes(rng, n_blocks: int, n_seg: int) -> List[int]:
    """Split n_blocks into n_seg runs at distinct uniform interior boundaries."""
    n_seg = max(1, min(n_seg, n_blocks))
    if n_seg == 1:
        return [n_blocks]
    cuts = np.sort(rng.choice(np.arange(1, n_blocks), size=n_seg - 1, replace=False))
    edges = np.concatenate([[0], cuts, [n_blocks]])
    return [int(x) for x in np.diff(edges)]


def _geometric_sizes(rng, total: int, n: int, p: float) -> List[int]:
    """n iid Geometric(p) draws rescaled to sum to `total` by largest remainder (min 1)."""
    x = rng.geometric(p, size=n).astype(np.float64)
    scaled = x * total / x.sum()
    base = np.maximum(1, np.floor(scaled)).astype(np.int64)
    frac = scaled - np.floor(scaled)
    diff = total - int(base.sum())
    order = np.argsort(-frac, kind="stable")
    i = 0
    while diff > 0:
        base[order[i % n]] += 1
        diff -= 1
        i += 1
    while diff < 0:
        j = int(np.argmax(base))
        base[j] -= 1
        diff += 1
    assert base.min() >= 1 and base.sum() == total
    return [int(v) for v in base]


def _finish(name, hq, hkv, d, seq_lens, layout, pool_blocks, q_ranges, rng, seed):
    seq_lens = np.asarray(seq_lens, np.int32)
    table, drawn = layout.realise(rng, seq_lens, pool_blocks)
    return Workload(name, hq, hkv, d, BLOCK, seq_lens, table, int(pool_blocks),
                    [list(map(tuple, r)) for r in q_ranges], drawn, seed)


def tiny_decode(seed: int = 1001) -> Workload:
    rng = np.random.default_rng(seed)
    lay = _Layout(1)
    for n in (4, 6, 6):
        lay.run(0, n)
    return _finish("tiny_decode", 4, 4, 64, [256], lay, 64, [[(256, 257)]], rng, seed)


def batched_decode(seed: int = 1002, num_seqs: int = 32, len_range=(2048, 16384), max_seg: int = 8,
                   pool_tokens: int = 4194304, hq: int = 32, hkv: int = 8, d: int = 128,
                   name: str = "batched_decode") -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_range[0], len_range[1] + 1, size=num_seqs)
    lay = _Layout(num_seqs)
    for s in range(num_seqs):
        nb = -(-int(lens[s]) // BLOCK)
        for n in _cut_sizes(rng, nb, int(rng.integers(1, max_seg + 1))):
            lay.run(s, n)
    ranges = [[(int(L), int(L) + 1)] for L in lens]
    return _finish(name, hq, hkv, d, lens, lay, pool_tokens // BLOCK, ranges, rng, seed)


def _draw_holes(rng, total_evict: int, lo: int, hi: int) -> List[int]:
    holes: List[int] = []
    left = total_evict
    while left > 0:
        h = min(int(rng.integers(lo, hi + 1)), left)
        if h == 1 and holes:
            holes[-1] += 1
        else:
            holes.append(h)
        left -= h
    return holes


def hole_recompute(seed: int = 1003, num_seqs: int = 16, cached_blocks: int = 512,
                   evict_blocks: int = 128, hole_range=(2, 32), turn_tokens: int = 512,
                   hq: int = 32, hkv: int = 8, d: int = 128, name: str = "hole_recompute") -> Workload:
    rng = np.random.default_rng(seed)
    lay = _Layout(num_seqs)
    lens, ranges = [], []
    for s in range(num_seqs):
        holes = _draw_holes(rng, evict_blocks, *hole_range)
        k = len(holes)
        live = cached_blocks - evict_blocks
        # gaps before / between / after the holes: interior gaps >= 1 live block
        gaps = _stars_and_bars(rng, live - (k - 1), k + 1)
        gaps[1:k] += 1
        original = lay.extent(cached_blocks)  # the sequence's original run, holes left empty
        b = 0
        seq_ranges = []
        for i in range(k + 1):
            if gaps[i] > 0:
                lay.run(s, int(gaps[i]), original, b)
                b += int(gaps[i])
            if i < k:
                lay.run(s, holes[i])  # recomputed hole K/V in a fresh run elsewhere
                seq_ranges.append((b * BLOCK, (b + holes[i]) * BLOCK))
                b += holes[i]
        assert b == cached_blocks
        turn_blocks = -(-turn_tokens // BLOCK)
        lay.run(s, turn_blocks)
        L = cached_blocks * BLOCK + turn_tokens
        seq_ranges.append((cached_blocks * BLOCK, L))
        lens.append(L)
        ranges.append(seq_ranges)
    total_blocks = sum(lay.extents)
    pool_blocks = 2 * total_blocks + len(lay.extents)
    return _finish(name, hq, hkv, d, lens, lay, pool_blocks, ranges, rng, seed)


def long_context(seed: int = 1004, num_seqs: int = 4, length: int = 131072, n_runs: int = 64,
                 p: float = 1.0 / 128, chunk: int = 2048, hq: int = 32, hkv: int = 8, d: int = 128,
                 name: str = "long_context") -> Workload:
    rng = np.random.default_rng(seed)
    lay = _Layout(num_seqs)
    nb = -(-length // BLOCK)
    for s in range(num_seqs):
        for n in _geometric_sizes(rng, nb, n_runs, p):
            lay.run(s, n)
    pool_blocks = 2 * num_seqs * nb
    ranges = [[(length - chunk, length), (length, length + 1)] for _ in range(num_seqs)]
    return _finish(name, hq, hkv, d, [length] * num_seqs, lay, pool_blocks, ranges, rng, seed)


def mixed_batch(seed: int = 1005, num_decode: int = 64, num_prefill: int = 4, chunk: int = 2048,
                median: float = 4096.0, sigma: float = 1.0, cap: int = 32768, max_seg: int = 32,
                hq: int = 64, hkv: int = 8, d: int = 128, name: str = "mixed_batch") -> Workload:
    rng = np.random.default_rng(seed)

    def draw_len(minimum):
        while True:
            L = int(np.clip(round(rng.lognormal(math.log(median), sigma)), 16, cap))
            if L >= minimum:
                return L

    lens = [draw_len(16) for _ in range(num_decode)] + [draw_len(chunk) for _ in range(num_prefill)]
    n = num_decode + num_prefill
    lay = _Layout(n)
    for s in range(n):
        nb = -(-lens[s] // BLOCK)
        for sz in _cut_sizes(rng, nb, int(rng.integers(1, min(max_seg, nb) + 1))):
            lay.run(s, sz)
    ranges = [[(L, L + 1)] for L in lens[:num_decode]] + [[(L - chunk, L)] for L in lens[num_decode:]]
    total_blocks = sum(lay.extents)
    pool_blocks = 2 * total_blocks + len(lay.extents)
    return _finish(name, hq, hkv, d, lens, lay, pool_blocks, ranges, rng, seed)


def custom(seq_lens, runs_per_seq, q_ranges, hq=8, hkv=2, d=128, seed=7, pool_factor=2,
           name="custom") -> Workload:
    """Explicit layout: runs_per_seq[s] = list of run sizes in blocks (logical order)."""
    rng = np.random.default_rng(seed)
    lay = _Layout(len(seq_lens))
    for s, sizes in enumerate(runs_per_seq):
        for n in sizes:
            lay.run(s, n)
    total = max(1, sum(lay.extents))
    pool_blocks = pool_factor * total + len(lay.extents) + 1
    return _finish(name, hq, hkv, d, seq_lens, lay, pool_blocks, q_ranges, rng, seed)


CONFIGS = {1: tiny_decode, 2: batched_decode, 3: hole_recompute, 4: long_context, 5: mixed_batch}


def config(index: int, seed: Optional[int] = None) -> Workload:
    fn = CONFIGS[index]
    return fn(seed=1000 + index if seed is None else seed)


def small_config(index: int, seed: Optional[int] = None) -> Workload:
    """Reduced versions of the five shapes that the float64 oracle finishes in
    seconds, still spanning several KV tiles, several query tiles and a
    ragged tail."""
    sd = 2000 + index if seed is None else seed
    if index == 1:
        return tiny_decode(seed=sd)
    if index == 2:
        return batched_decode(seed=sd, num_seqs=6, len_range=(300, 2100), pool_tokens=1 << 16,
                              name="batched_decode_small")
    if index == 3:
        return hole_recompute(seed=sd, num_seqs=2, cached_blocks=64, evict_blocks=16,
                              hole_range=(2, 6), turn_tokens=72, name="hole_recompute_small")
    if index == 4:
        return long_context(seed=sd, num_seqs=1, length=4096 + 40, n_runs=12, p=1.0 / 16,
                            chunk=300, name="long_context_small")
    if index == 5:
        return mixed_batch(seed=sd, num_decode=6, num_prefill=2, chunk=200, median=600, cap=3000,
                           max_seg=8, hq=16, hkv=2, name="mixed_batch_small")
    raise KeyError(index)


def restrict_rows(wl: Workload, kind: str) -> Workload:
    """The same sequences, block tables and pool with only part of the query
    rows: kind="decode" keeps the rows a plan serves as decode rows (a
    sequence's trailing rows when they number at most 16/G, the rest of its
    rows filling whole 128-row tiles or the sequence having no other rows),
    kind="prefill" keeps all the others.  The two together partition the rows;
    each keeps the tiling the full plan gives its rows."""
    assert kind in ("decode", "prefill")
    G = wl.num_q_heads // wl.num_kv_heads
    dec_rows = max(1, 16 // G)
    ranges = []
    for rs in wl.q_ranges:
        pos = [p for a, b in rs for p in range(a, b)]
        n = len(pos)
        if n == 0:
            n_dec = 0
        elif n <= dec_rows:
            n_dec = n
        else:
            rem = n % 128
            n_dec = rem if 0 < rem <= dec_rows else 0
        keep = pos[n - n_dec:] if kind == "decode" else pos[:n - n_dec]
        out = []
        for p in keep:
            if out and out[-1][1] == p:
                out[-1][1] = p + 1
            else:
                out.append([p, p + 1])
        ranges.append([tuple(r) for r in out])
    return dataclasses.replace(wl, q_ranges=ranges, name=f"{wl.name}/{kind}-rows")


def with_prefill_chunk(wl: Workload, pending, c: int) -> Workload:
    """The same pool and block tables for a serving step that runs the next
    min(c, end - start) positions of every pending prefill (seq, start, end):
    that sequence then holds start + n cached tokens (the chunk's own K/V is
    appended before attention) and queries rows [start, start + n); every
    other sequence keeps its length and rows."""
    lens = wl.seq_lens.copy()
    ranges = [list(r) for r in wl.q_ranges]
    for seq, start, end in pending:
        n = min(int(c), int(end) - int(start))
        lens[seq] = int(start) + n
        ranges[seq] = [(int(start), int(start) + n)]
    return dataclasses.replace(wl, seq_lens=lens.astype(np.int32), q_ranges=ranges, name=f"{wl.name}/chunk{c}")


def pending_prefills(wl: Workload, remaining: int = 8192):
    """The batch with its prefill sequences taken out as pending prefills:
    every sequence whose rows are not a lone decode row at p = L becomes a
    pending prefill of its last min(L, remaining) positions with no rows of
    its own; returns (batch workload, [(seq, start, end)])."""
    ranges, pending = [], []
    for s, rs in enumerate(wl.q_ranges):
        L = int(wl.seq_lens[s])
        if rs == [(L, L + 1)]:
            ranges.append(list(rs))
        else:
            pending.append((s, max(0, L - remaining), L))
            ranges.append([])
    return dataclasses.replace(wl, q_ranges=ranges, name=f"{wl.name}/pending"), pending


# ------------------------------------------------------------------ values --

def make_values(wl: Workload, device="cpu", seed: Optional[int] = None, dtype=None):
    """bf16 ~ N(0, 1) logical K, V [total_tokens, Hkv, D] and Q [n_q, Hq, D].

    Drawn as fp32 from a torch generator seeded with `seed` (default
    wl.seed) on `device`, then rounded to bf16.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed if seed is None else seed)
    dt = dtype or torch.bfloat16
    T = int(wl.seq_lens.sum())
    shape_kv = (T, wl.num_kv_heads, wl.head_dim)
    k = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(dt)
    v = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(dt)
    q = torch.randn((wl.num_q_rows, wl.num_q_heads, wl.head_dim), generator=g, device=device,
                    dtype=torch.float32).to(dt)
    return k, v, q


def make_pool(wl: Workload, k_logical, v_logical, fill: float = float("nan")):
    """Paged pools [pool_tokens, Hkv, D] holding the logical K/V at the rows the
    block table names; every other row is set to `fill` (NaN by default, so a
    kernel that reads outside the live rows shows it)."""
    import torch
    dev = k_logical.device
    shape = (wl.pool_tokens, wl.num_kv_heads, wl.head_dim)
    kp = torch.full(shape, fill, dtype=k_logical.dtype, device=dev)
    vp = torch.full(shape, fill, dtype=v_logical.dtype, device=dev)
    slots = torch.from_numpy(wl.slot_mapping()).to(dev)
    kp.index_copy_(0, slots, k_logical)
    vp.index_copy_(0, slots, v_logical)
    return kp, vp


def seq_kv(wl: Workload, k_logical, s: int):
    """Logical K (or V) rows of sequence s."""
    ind = wl.kv_indptr
    return k_logical[int(ind[s]):int(ind[s + 1])]
