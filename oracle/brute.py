"""Tiny explicit-softmax float64 attention in numpy (test infrastructure only).

A second, independent restatement of the oracle's definition for tiny inputs
(pure-Python loops over rows and heads, numpy for the inner sums): for each
query row at position p and head h, take the keys j <= min(p, L-1) of kv head
h // G, form the scaled scores, the softmax weights exp(t - max) / sum, and
the weighted sum of the values.  lse is reported in natural log of the scaled
scores.  Used only to pin the C oracle on hand-sized cases.
"""
from __future__ import annotations

import math

import numpy as np


def attention_tiny(k, v, q, q_pos, num_kv_heads, scale):
    """k, v: float64 [L, Hkv, D]; q: float64 [n, Hq, D]; q_pos: [n] ints.

    Returns (out [n, Hq, D], lse [n, Hq]).
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q = np.asarray(q, np.float64)
    n, hq, d = q.shape
    length = k.shape[0]
    group = hq // num_kv_heads
    out = np.zeros((n, hq, d))
    lse = np.full((n, hq), -math.inf)
    for i in range(n):
        n_vis = min(int(q_pos[i]) + 1, length)
        if n_vis <= 0:
            continue
        for h in range(hq):
            g = h // group
            scores = [scale * sum(q[i, h, c] * k[j, g, c] for c in range(d)) for j in range(n_vis)]
            top = max(scores)
            weights = [math.exp(s - top) for s in scores]
            total = sum(weights)
            lse[i, h] = top + math.log(total)
            for j in range(n_vis):
                out[i, h] += (weights[j] / total) * v[j, g]
    return out, lse
