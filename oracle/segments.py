"""Brute-force segment splitter in pure Python (test infrastructure only).

Segments as the MSA explainer describes them (AsymCache explainer, "核心方法
1. Multi-Segment Attention": live blocks are regrouped by physical
contiguity in GPU memory, and eviction holes break a segment): a new segment
starts at logical block b whenever b == 0 or the physical id of b is not the
physical id of b-1 plus one.  Written as a direct scan over every block so it
shares nothing with the C oracle's run-walking loop or the library planner.
"""
from __future__ import annotations


def split_into_contiguous_segments(table_row, seq_len, block_size):
    """Return [(first_logical_block, first_physical_block, n_blocks, n_tokens)].

    n_tokens counts only tokens below seq_len (the last block may be partial).
    Raises ValueError for a missing block (negative id) inside [0, seq_len).
    """
    n_blocks = -(-int(seq_len) // block_size)
    starts = []
    for b in range(n_blocks):
        if table_row[b] < 0:
            raise ValueError(f"missing block at logical block {b}")
        if b == 0 or table_row[b] != table_row[b - 1] + 1:
            starts.append(b)
    segs = []
    for i, b0 in enumerate(starts):
        b1 = starts[i + 1] if i + 1 < len(starts) else n_blocks
        tokens = min(b1 * block_size, int(seq_len)) - b0 * block_size
        segs.append((b0, int(table_row[b0]), b1 - b0, tokens))
    return segs
