"""fp64 multi-query attention over a paged KV pool with a causal mask (oracle
side; test infrastructure, imported only by the tests and the benchmark's CPU
legs).

Prefill computes the keys and values of every prompt token at once, and decode
then attends each new token to all tokens before it (subroutine-cs article,
introduction: the prefill and decode phases).  With the KV of a sequence's new
tokens already written to its blocks, the attention of those tokens is the
same paged gather as decode ("10 — Paged Attention" §4 PhysicalIndex, §5 "The
kernel side"), for many query tokens, each limited to the positions up to its
own.  Chunked prefill (a prompt processed in pieces, or the part of a prompt not
found in the prefix cache) and the verification of several drafted tokens are
the same computation with a shorter query range.

Definition (this library's reading, listed in the design notes): query rows
q_start[b] .. q_start[b+1]-1 of q belong to sequence b; with L = seq_lens[b] and
n = q_start[b+1] - q_start[b], row q_start[b] + i is the token at position
p = L - n + i (the last n tokens of the sequence) and, for query head hq with KV
head h = hq // G,

    s_t = sigma * sum_d q[row, hq, d] * K[slot_t, h, d]           t = 0 .. p
    out[row, hq] = sum_t softmax(s)_t * V[slot_t, h, :]

slot_t = block_tables[b][t // bs] * bs + t % bs.  Float64 over the exact
upcasts of the storage values; sigma is the fp32 scale, widened exactly.
"""
from __future__ import annotations

import numpy as np

from .attention import storage_to_f64, token_slots


def paged_prefill_attention(q, k_pool, v_pool, block_tables, seq_lens, q_start, scale,
                            dtype=None, rows=None) -> np.ndarray:
    """q [total_q, Hq, D]; pools [NB, bs, Hkv, D]; q_start [B + 1] non-decreasing,
    q_start[0] = 0, q_start[B] = total_q; seq_lens [B] >= the query counts.
    dtype None: float64 inputs, else uint16 storage bits of FLOAT16 / BFLOAT16.
    rows: optional subset of query rows to evaluate (others stay zero).
    Returns out [total_q, Hq, D] float64."""
    widen = (lambda a: np.asarray(a, dtype=np.float64)) if dtype is None else \
        (lambda a: storage_to_f64(a, dtype))
    qf = widen(q)
    total_q, Hq, D = qf.shape
    NB, bs, Hkv, Dk = k_pool.shape
    if Dk != D or Hq % Hkv:
        raise ValueError("shape mismatch")
    G = Hq // Hkv
    q_start = [int(x) for x in q_start]
    B = len(q_start) - 1
    if q_start[0] != 0 or q_start[B] != total_q:
        raise ValueError("q_start must run from 0 to total_q")
    sigma = float(np.float32(scale))
    k_rows = k_pool.reshape(NB * bs, Hkv, D)
    v_rows = v_pool.reshape(NB * bs, Hkv, D)
    out = np.zeros((total_q, Hq, D), dtype=np.float64)
    wanted = None if rows is None else set(int(r) for r in rows)
    for b in range(B):
        n = q_start[b + 1] - q_start[b]
        L = int(seq_lens[b])
        if n < 0 or n > L:
            raise ValueError(f"sequence {b}: {n} query tokens for a length of {L}")
        if n == 0:
            continue
        slots = token_slots(block_tables[b], L, bs)
        for h in range(Hkv):
            K = widen(k_rows[slots, h, :])              # [L, D]
            V = widen(v_rows[slots, h, :])
            for i in range(n):
                row = q_start[b] + i
                if wanted is not None and row not in wanted:
                    continue
                p = L - n + i
                for hq in range(h * G, (h + 1) * G):
                    s = (K[:p + 1] @ qf[row, hq]) * sigma
                    w = np.exp(s - s.max())
                    out[row, hq] = (w @ V[:p + 1]) / w.sum()
    return out


def causal_pairs(seq_lens, q_start) -> int:
    """Number of (query token, key token) pairs the causal mask allows: the
    per-head work unit of prefill (4 * head_dim flops each, q.k and p.v)."""
    total = 0
    for b in range(len(q_start) - 1):
        n = int(q_start[b + 1]) - int(q_start[b])
        L = int(seq_lens[b])
        # positions L-n .. L-1 see L-n+1 .. L keys
        total += n * (L - n) + n * (n + 1) // 2
    return total
