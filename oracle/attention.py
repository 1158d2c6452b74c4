"""fp64 decode attention over a paged KV pool (oracle side).

The method computes exact attention; paging only changes where the key and
value rows live ("PagedAttention" glossary entry, the kernel duties: read the
block table, gather from scattered blocks, handle a partly filled last block;
the same entry calls FlashAttention an exact attention algorithm that paging
complements).  The oracle is therefore the plain definition, written out:

  for sequence b and query head hq, with KV head h = hq // G (G = Hq / Hkv) and
  context length L = seq_lens[b]:
    slot_t = block_tables[b][t // bs] * bs + t % bs              for t < L
    s_t    = sigma * sum_d q[b, hq, d] * K[slot_t, h, d]
    out    = sum_t softmax(s)_t * V[slot_t, h, :]

The address translation is the tutorial's PhysicalIndex ("10 — Paged
Attention" §4 "Tiny example"); the pool layout [num_blocks, block_size, Hkv, D]
and the argument list (q [num_seqs, num_heads, head_dim], block_tables
[num_seqs, max_blocks_per_seq], context lengths) are those of the tutorial's
kernel sketch (§5 "The kernel side").  Everything is evaluated in float64 over
the exact upcasts of the fp16/bf16 storage values; sigma is the fp32 scale the
GPU receives, widened exactly.

Readings where the pages are silent: grouped-query heads map contiguously
(hq // G); a context length of zero yields a zero output row.
"""
from __future__ import annotations

import numpy as np

FLOAT16 = 0
BFLOAT16 = 1


def storage_to_f64(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact float64 values of fp16 / bf16 storage bits (uint16 arrays)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == FLOAT16:
        return bits.view(np.float16).astype(np.float64)
    if dtype == BFLOAT16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype code {dtype}")


def token_slots(block_table, length: int, block_size: int) -> np.ndarray:
    """Pool slots of tokens 0..length-1 of one sequence (PhysicalIndex)."""
    pos = np.arange(length, dtype=np.int64)
    table = np.asarray(block_table, dtype=np.int64)
    return table[pos // block_size] * block_size + pos % block_size


def paged_decode_attention(q, k_pool, v_pool, block_tables, seq_lens, scale,
                           sequences=None, heads=None, dtype=None) -> np.ndarray:
    """Exact decode attention in float64.

    q        [B, Hq, D]            float64
    k_pool   [NB, bs, Hkv, D]      float64 (v_pool the same)
    dtype    None: q and the pools hold float64 values.  FLOAT16 / BFLOAT16:
             they hold uint16 storage bits, widened exactly as rows are used.
    block_tables [B, max_blocks]   integer
    seq_lens [B]                   integer
    scale    python float (the fp32 scale passed to the kernel)
    sequences / heads: optional subsets of b and hq to evaluate (other rows of
      the result stay zero), for sampled checks of large workloads.
    Returns out [B, Hq, D] float64.
    """
    if dtype is None:
        widen = lambda a: np.asarray(a, dtype=np.float64)
    else:
        widen = lambda a: storage_to_f64(a, dtype)
    q = widen(q)
    B, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_pool.shape
    if Dk != D or Hq % Hkv:
        raise ValueError("shape mismatch")
    G = Hq // Hkv
    sigma = float(np.float32(scale))
    out = np.zeros((B, Hq, D), dtype=np.float64)
    k_rows = k_pool.reshape(NB * bs, Hkv, D)
    v_rows = v_pool.reshape(NB * bs, Hkv, D)
    seqs = range(B) if sequences is None else sequences
    head_list = list(range(Hq)) if heads is None else list(heads)
    for b in seqs:
        L = int(seq_lens[b])
        if L == 0:
            continue
        slots = token_slots(block_tables[b], L, bs)
        for hq in head_list:
            h = hq // G
            K = widen(k_rows[slots, h, :])              # [L, D]
            V = widen(v_rows[slots, h, :])              # [L, D]
            s = (K @ q[b, hq]) * sigma                  # [L]
            w = np.exp(s - s.max())
            out[b, hq] = (w @ V) / w.sum()
    return out


def within_tolerance(gpu: np.ndarray, ref: np.ndarray, atol=2e-3, rtol=1e-2) -> np.ndarray:
    """Elementwise acceptance |gpu - ref| <= atol + rtol * |ref|."""
    return np.abs(gpu - ref) <= atol + rtol * np.abs(ref)
