"""Pins of the oracle's paged prefill attention (CPU only): PyTorch's causal
scaled_dot_product_attention over contiguous K/V, the decode oracle for one
query per sequence, chunked prefill against the whole prompt, closed forms, and
the count of causal (query, key) pairs."""
import dataclasses

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from oracle.attention import paged_decode_attention, storage_to_f64
from oracle.prefill import causal_pairs, paged_prefill_attention

SMALL = dataclasses.replace(syn.PREFILL, name="prefill_small", num_seqs=3, length_kind="fixed",
                            lens=(37, 70, 16), num_q_heads=8, num_kv_heads=2, head_dim=32)


def _contiguous(pool, table, L, bs, h, dtype):
    """K or V of one head laid out token after token, block by block, without
    the slot formula: logical block i is physical block table[i], rows in order."""
    blocks = [storage_to_f64(pool[int(table[i]), :, h, :], dtype) for i in range(-(-L // bs))]
    return np.concatenate(blocks, axis=0)[:L]


@pytest.mark.parametrize("q_counts", [None, (5, 70, 1), (37, 1, 16)])
def test_matches_torch_causal_sdpa(q_counts):
    pb = scenarios.prefill_batch(SMALL, q_counts=q_counts)
    b = pb.batch
    got = scenarios.prefill_f64(pb)
    G = SMALL.num_q_heads // SMALL.num_kv_heads
    sigma = float(np.float32(SMALL.scale))
    for s in range(len(b.seq_lens)):
        L = int(b.seq_lens[s])
        r0, r1 = int(pb.q_start[s]), int(pb.q_start[s + 1])
        n = r1 - r0
        qf = storage_to_f64(pb.q[r0:r1], b.dtype)               # [n, Hq, D]
        for h in range(SMALL.num_kv_heads):
            K = torch.from_numpy(_contiguous(b.k_pool, b.block_tables[s], L, b.block_size, h, b.dtype))
            V = torch.from_numpy(_contiguous(b.v_pool, b.block_tables[s], L, b.block_size, h, b.dtype))
            Q = torch.from_numpy(qf[:, h * G:(h + 1) * G].transpose(1, 0, 2).copy())  # [G, n, D]
            # query i sits at position L - n + i: it may see keys 0 .. L - n + i
            mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                Q, K.expand(G, L, -1), V.expand(G, L, -1), attn_mask=mask, scale=sigma)
            np.testing.assert_allclose(got[r0:r1, h * G:(h + 1) * G].transpose(1, 0, 2),
                                       ref.numpy(), rtol=1e-12, atol=1e-13)


def test_one_query_per_sequence_is_decode():
    pb = scenarios.prefill_batch(SMALL, q_counts=(1, 1, 1))
    b = pb.batch
    dec = paged_decode_attention(pb.q, b.k_pool, b.v_pool, b.block_tables, b.seq_lens, b.scale,
                                 dtype=b.dtype)
    assert np.array_equal(scenarios.prefill_f64(pb), dec)


def test_chunk_equals_the_same_rows_of_the_whole_prompt():
    """The last 20 tokens as a chunk over the cached prefix give exactly the rows
    a whole-prompt prefill gives for those positions."""
    full = scenarios.prefill_batch(SMALL)
    b = full.batch
    out_full = scenarios.prefill_f64(full)
    n = np.minimum(b.seq_lens, 20)
    rows = np.concatenate([np.arange(full.q_start[s + 1] - n[s], full.q_start[s + 1])
                           for s in range(len(n))])
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    out_chunk = paged_prefill_attention(full.q[rows], b.k_pool, b.v_pool, b.block_tables,
                                        b.seq_lens, q_start, b.scale, dtype=b.dtype)
    assert np.array_equal(out_chunk, out_full[rows])


def test_first_position_returns_its_value_row_and_constant_values():
    pb = scenarios.prefill_batch(SMALL)
    b = pb.batch
    out = scenarios.prefill_f64(pb)
    G = SMALL.num_q_heads // SMALL.num_kv_heads
    for s in range(len(b.seq_lens)):
        slot0 = int(b.block_tables[s][0]) * b.block_size
        r0 = int(pb.q_start[s])
        for hq in range(SMALL.num_q_heads):
            v0 = storage_to_f64(b.v_pool.reshape(-1, SMALL.num_kv_heads, SMALL.head_dim)[slot0, hq // G],
                                b.dtype)
            assert np.array_equal(out[r0, hq], v0)
    # constant V rows give that constant at every position
    v_const = np.full_like(b.v_pool, syn.fp32_to_storage_bits(np.float32([0.75]), b.dtype)[0])
    out_c = paged_prefill_attention(pb.q, b.k_pool, v_const, b.block_tables, b.seq_lens,
                                    pb.q_start, b.scale, dtype=b.dtype)
    assert np.allclose(out_c, 0.75, rtol=0, atol=1e-15)


def test_rejects_more_queries_than_tokens():
    pb = scenarios.prefill_batch(SMALL)
    b = pb.batch
    with pytest.raises(ValueError):
        paged_prefill_attention(pb.q, b.k_pool, b.v_pool, b.block_tables,
                                np.array([10, 70, 16]), pb.q_start, b.scale, dtype=b.dtype)


def test_causal_pairs_count():
    lens, n = [37, 70, 16], [5, 70, 1]
    brute = sum(len(range(0, L - k + i + 1)) for L, k in zip(lens, n) for i in range(k))
    q_start = np.concatenate([[0], np.cumsum(n)])
    assert causal_pairs(lens, q_start) == brute
    assert causal_pairs([100], [0, 100]) == 5050          # L (L + 1) / 2
