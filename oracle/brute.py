"""Pure-Python brute-force decode attention for tiny inputs (oracle side).

Nested loops with math.exp and no numpy arithmetic, written independently of
oracle.attention so the two can check one another: every key position is
looked up through the block table one token at a time (block = table[t // bs],
row = t % bs, as in the tutorial's PhysicalIndex, "10 — Paged Attention" §4),
scores are summed over head_dim element by element, and the softmax is formed
with an explicit running maximum.
"""
from __future__ import annotations

import math


def brute_decode_attention(q, k_pool, v_pool, block_tables, seq_lens, scale,
                           block_size):
    """q: nested lists [B][Hq][D] of floats; pools nested [NB][bs][Hkv][D].
    Returns nested lists [B][Hq][D]."""
    B = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(k_pool[0][0])
    G = Hq // Hkv
    out = []
    for b in range(B):
        L = int(seq_lens[b])
        rows = []
        for hq in range(Hq):
            h = hq // G
            if L == 0:
                rows.append([0.0] * D)
                continue
            scores = []
            for t in range(L):
                blk = int(block_tables[b][t // block_size])
                r = t % block_size
                acc = 0.0
                for d in range(D):
                    acc += q[b][hq][d] * k_pool[blk][r][h][d]
                scores.append(acc * scale)
            top = scores[0]
            for s in scores:
                if s > top:
                    top = s
            weights = [math.exp(s - top) for s in scores]
            total = 0.0
            for w in weights:
                total += w
            vec = [0.0] * D
            for t in range(L):
                blk = int(block_tables[b][t // block_size])
                r = t % block_size
                for d in range(D):
                    vec[d] += weights[t] * v_pool[blk][r][h][d]
            rows.append([x / total for x in vec])
        out.append(rows)
    return out
