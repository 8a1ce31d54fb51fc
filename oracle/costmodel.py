"""Plain Python restatement of the attention-latency model (test
infrastructure only: the library's msa_plan_estimate is checked against it).

AsymCache weighs a block's recompute cost and hit rate against the attention
kernel's expected latency (MSA paper abstract; AsymCache explainer, "核心方法
2" and "3").  The model prices each work item and replays the kernel's work
queue:

  fixed phase (us)   dec_item                                 (decode)
                   | pre_item + tile_us * tiles * qtiles      (prefill)
                     + box * extra_boxes
                     + dec_merge | pre_merge   [group split into parts]
  stream phase (B)   decode only: tiles * 128 * D * 2 * 2 (K and V, bf16),
                     at min(dec_cta, dec / n_streaming) GB/s per CTA
  tiles        128-key windows [kb + 128 i, min(kb + 128 (i+1), ke))
  qtiles       query tiles of 128 rows x one head: ceil(rows / 128) x heads
               (two heads over <= 128 rows, or one head over <= 256 rows)
  tile_us      pre_tile * ((1 - dfrac) + dfrac * D / 128): pre_tile is a
               tile's time at head dim 128, of which the share dfrac (MMAs,
               K/V loads) is proportional to D and the rest (the softmax of
               128 x 128 scores) is not
  extra_boxes  per tile, the TMA boxes beyond one: a full 128-key window
               inside one segment is one box; any other tile is fetched per
               segment piece, a piece of b whole 16-key blocks in boxes of 4,
               2 and 1 blocks (b // 4 + (b % 4) // 2 + b % 2 boxes)
  replay       CTAs 0..grid-1 take the first items of the plan's order; when
               a CTA's phases are done it takes the next item; between
               events every CTA advances at its phase's rate
  time         launch + the time the last CTA finishes

Segments come from oracle.segments (the brute-force splitter over the block
table), never from the library; the work list and its order are the plan's
(inputs here, not recomputed).  Pure Python loops: small and medium plans.
"""
from __future__ import annotations

from .segments import split_into_contiguous_segments

TILE = 128
BLOCK = 16


def _token_segments(table_row, seq_len):
    """[(first logical token, n_tokens)] of one sequence's segments."""
    return [(b0 * BLOCK, ntok) for (b0, _p, _nb, ntok) in split_into_contiguous_segments(table_row, seq_len, BLOCK)]


def _boxes(segs, t0, t1):
    """TMA boxes for the tile [t0, t1) of a sequence with segments `segs`."""
    boxes = 0
    for (a, n) in segs:
        lo, hi = max(a, t0), min(a + n, t1)
        if hi <= lo:
            continue
        if lo == t0 and hi - lo == TILE:
            boxes += 1
        else:
            b = -(-(hi - lo) // BLOCK)
            boxes += b // 4 + (b % 4) // 2 + b % 2
    return boxes


def tile_us(params, head_dim):
    """Time of one (128-key tile x 128-row query tile) at head dim D.  A
    parameter set without pre_tile_dfrac has no head-dim term (dfrac 0)."""
    dfrac = params.get("pre_tile_dfrac", 0.0)
    return params["pre_tile_us"] * ((1.0 - dfrac) + dfrac * head_dim / 128.0)


def estimate(items, order, block_table, seq_lens, grid, params, head_dim):
    """items: rows (kind, seq, head, heads, row0, nrows, kb, ke, part) as
    msa_plan_get_items returns them; order: msa_plan_get_order; params: dict
    of the msa_cost_params names.  Returns a dict like msa_plan_estimate."""
    segs = {}
    parts = {}
    for (kind, seq, head, heads, row0, nrows, kb, ke, part) in items:
        key = (kind, seq, head, row0)
        parts[key] = parts.get(key, 0) + 1
    fixed, stream = [], []
    out = {"n_items": len(items), "n_split_items": 0, "decode_tiles": 0, "prefill_tile_heads": 0,
           "extra_boxes": 0, "stream_bytes": 0, "fixed_us": 0.0}
    tile_bytes = 2.0 * TILE * head_dim * 2.0
    for (kind, seq, head, heads, row0, nrows, kb, ke, part) in items:
        if seq not in segs:
            segs[seq] = _token_segments(block_table[seq], int(seq_lens[seq]))
        tiles = 0
        extra = 0
        t0 = kb
        while t0 < ke:
            t1 = min(t0 + TILE, ke)
            tiles += 1
            extra += max(0, _boxes(segs[seq], t0, t1) - 1)
            t0 += TILE
        split = parts[(kind, seq, head, row0)] > 1
        if kind == 0:
            f = params["dec_item_us"]
            b = tile_bytes * tiles
            out["decode_tiles"] += tiles
        else:
            qtiles = -(-nrows // TILE) * heads
            f = params["pre_item_us"] + tile_us(params, head_dim) * tiles * qtiles
            b = 0.0
            out["prefill_tile_heads"] += tiles * qtiles
        merge = params["dec_merge_us"] if kind == 0 else params["pre_merge_us"]
        f += params["box_us"] * extra + (merge if split else 0.0)
        out["extra_boxes"] += extra
        out["n_split_items"] += 1 if split else 0
        out["stream_bytes"] += int(b)
        out["fixed_us"] += f
        fixed.append(f)
        stream.append(b)
    n_cta = max(1, int(grid))
    queue = list(order)
    cur = [None] * n_cta          # [item, phase, left] per CTA
    for c in range(n_cta):
        cur[c] = [queue.pop(0), 0, None] if queue else None
        if cur[c] is not None:
            cur[c][2] = fixed[cur[c][0]]
    t = 0.0
    while True:
        for c in range(n_cta):
            while cur[c] is not None and cur[c][2] <= 0.0:
                i, ph, _ = cur[c]
                if ph == 0 and stream[i] > 0.0:
                    cur[c] = [i, 1, stream[i]]
                elif queue:
                    j = queue.pop(0)
                    cur[c] = [j, 0, fixed[j]]
                else:
                    cur[c] = None
        busy = [c for c in range(n_cta) if cur[c] is not None]
        if not busy:
            break
        n_stream = sum(1 for c in busy if cur[c][1] == 1)
        rate = min(params["dec_cta_gbs"], params["dec_gbs"] / n_stream) * 1e3 if n_stream else 0.0
        ttf = {c: (cur[c][2] if cur[c][1] == 0 else cur[c][2] / rate) for c in busy}
        dt = min(ttf[c] for c in busy)
        t += dt
        for c in busy:
            if ttf[c] == dt:
                cur[c][2] = 0.0
            else:
                cur[c][2] -= dt if cur[c][1] == 0 else dt * rate
    out["makespan_us"] = t
    out["time_us"] = params["launch_us"] + t
    return out


def hole_recompute_flops(head_dim, num_q_heads, start, end, seq_len):
    """Attention flops of recomputing query rows [start, end) of a sequence
    holding seq_len tokens: 4 * D * Hq * sum over p of min(p + 1, seq_len),
    the position-aware recompute cost (a row at p attends to p + 1 keys)."""
    return 4.0 * head_dim * num_q_heads * sum(min(p + 1, seq_len) for p in range(start, end))


# --------------------------------------------------------- prefill chunking --
#
# AsymCache explainer, "核心方法 3" (adaptive chunking scheduler) and the MSA
# paper's methodology (a dynamic chunking scheduler that adapts prefill sizes
# to the hardware): a step runs the batch's other rows plus the next c
# positions of each pending prefill; the chunk size trades the step's fixed
# costs (launch, decode rows, per-item overheads), which a larger chunk
# spreads over more prefill tokens, against the step's latency.  The choice:
# the lowest predicted step time per prefill token among the candidates
# whose predicted time stays within the budget.

def chunk_candidates(max_remaining, granularity=0, max_chunk=0):
    """Multiples of the granularity (default 128) up to C = min(max_chunk,
    max_remaining) (no cap when max_chunk is 0), every k-th of them with
    k = ceil(multiples / 63) when there are more than 63, then C itself if
    it is not the last one."""
    g = granularity if granularity > 0 else TILE
    cap = max_remaining if max_chunk <= 0 else min(max_remaining, max_chunk)
    n_mult = cap // g
    step = max(1, -(-n_mult // 63))
    out = [k * g for k in range(1, n_mult + 1, step)]
    if not out or out[-1] != cap:
        out.append(cap)
    return out


def chunk_batch(seq_lens, q_range_indptr, q_ranges, pending, c):
    """The step's batch with chunk c: (seq_lens, indptr, ranges, prefill
    tokens).  A pending sequence (seq, start, end) runs rows [start, start +
    n) with n = min(c, end - start) and holds start + n cached tokens (the
    chunk's own K/V is appended first); every other sequence keeps its rows."""
    lens = [int(x) for x in seq_lens]
    pend = {int(s): (int(a), int(b)) for s, a, b in pending}
    indptr, ranges, tokens = [0], [], 0
    for s in range(len(lens)):
        if s in pend:
            a, b = pend[s]
            n = min(c, b - a)
            lens[s] = a + n
            ranges.append((a, a + n))
            tokens += n
        else:
            ranges.extend((int(q_ranges[r][0]), int(q_ranges[r][1]))
                          for r in range(q_range_indptr[s], q_range_indptr[s + 1]))
        indptr.append(len(ranges))
    return lens, indptr, ranges, tokens


def choose_chunk(cands, times_us, tokens, budget_us):
    """(chunk, within budget): the lowest times_us / tokens among candidates
    with times_us <= budget_us (budget_us <= 0: all), equal costs to the
    larger chunk; with none inside the budget, the smallest candidate."""
    ok = [(t / n, -c, c) for c, t, n in zip(cands, times_us, tokens) if budget_us <= 0 or t <= budget_us]
    if not ok:
        return min(cands), False
    return min(ok)[2], True
