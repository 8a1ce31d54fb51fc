"""Plain Python restatement of the kernel-aware eviction choice (test
infrastructure only: the library's msa_select_evictions is checked
against it).

AsymCache explainer, "核心方法 2": blocks are evicted lowest score first,
the score weighing a block's future hit probability (weight alpha) against
its position-aware recompute cost (weight beta).  The page gives the cost
two readings, and both are here:

* hole reading: only the evicted block is rebuilt; its cost is the
  attention work of recomputing its own rows.  Row p attends to min(p + 1, L)
  keys, so the work is the sum of min(p + 1, L) over the block's rows, here
  in units of a 128x128 tile of one head, times Hq heads, at `pre_tile_us`
  per tile and head (the latency model's tile time at the attention's head
  dim: oracle.costmodel.tile_us).  It grows with position (the page: the
  cost depends strongly on where the block sits).
* prefix reading: a block's cache is usable only with its whole prefix, so
  evicting block b leaves blocks b, b+1, ..., last to recompute; its cost is
  the sum of the hole costs of those blocks.  It falls with position, so the
  tail blocks are the cheap ones (the page: tail blocks are cheap and should
  yield first).

The cost enters normalised by its largest value over the sequence, on the
keep side (a block that is dear to recompute scores higher); equal scores
evict the lower block first.
"""
from __future__ import annotations

BLOCK = 16


def recompute_cost_us(seq_len, num_q_heads, pre_tile_us):
    """Hole reading, per block: pre_tile_us * Hq * (sum of min(p + 1, L) over its rows) / 128^2."""
    out = []
    n_blocks = -(-int(seq_len) // BLOCK)
    for b in range(n_blocks):
        keys = 0
        for p in range(b * BLOCK, min((b + 1) * BLOCK, seq_len)):
            keys += min(p + 1, seq_len)
        out.append(pre_tile_us * num_q_heads * keys / (128 * 128))
    return out


def prefix_recompute_cost_us(seq_len, num_q_heads, pre_tile_us):
    """Prefix reading, per block b: the hole costs of blocks b .. last, summed."""
    hole = recompute_cost_us(seq_len, num_q_heads, pre_tile_us)
    return [sum(hole[b:]) for b in range(len(hole))]


def select_evictions(seq_len, num_q_heads, hit_prob, alpha, beta, pre_tile_us, n_evict, expected_cost=False,
                     prefix=False):
    """Lowest scores first: alpha * hit + beta * cost / max cost, or (with
    expected_cost) hit * cost; cost in the hole reading, or the prefix
    reading with `prefix`."""
    if prefix:
        cost = prefix_recompute_cost_us(seq_len, num_q_heads, pre_tile_us)
    else:
        cost = recompute_cost_us(seq_len, num_q_heads, pre_tile_us)
    cmax = max(cost) if cost else 0.0
    scored = []
    for b, c in enumerate(cost):
        if expected_cost:
            s = float(hit_prob[b]) * c
        else:
            s = alpha * float(hit_prob[b]) + (beta * c / cmax if cmax > 0 else 0.0)
        scored.append((s, b))
    scored.sort(key=lambda x: (x[0], x[1]))
    return sorted(b for _, b in scored[:n_evict]), cost
