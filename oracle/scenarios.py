"""Paged pool layouts of the decode workloads, built through the oracle's block
manager from a seed (oracle side).

Block ids come from a block manager whose free stack is a seeded permutation,
so that the tables point at scattered physical blocks, as in the tutorial's
picture of block tables over a physical pool ("10 — Paged Attention" §1
"What is it?").  Unused slots of every block, unused blocks and the block that
padding table entries point at are filled with NaN, so that reading any of
them changes the result.

Three flows:

fixed_batch    every sequence holds L_b tokens; one decode over the batch.
shared_prefix  P prompts of prefix+k_p tokens, each forked into S samples
               (refcount S on every prompt block); each sample then appends
               its own generated tokens one step at a time, with copy-on-write
               of a shared partly filled block ("10 — Paged Attention" §5
               "Copy-on-write sharing"; subroutine-cs article §3).
ragged_steps   continuous-batching steps ("PagedAttention" glossary entry,
               continuous batching): each sequence starts with L_b - 1 tokens;
               each step appends one token per sequence (a fresh block at a
               block boundary, tutorial §4 AppendToken), writes it, then the
               batch decodes with the grown lengths.
swap_round_trip  some sequences of a batch are evicted to a pool in CPU RAM
               (PagedAttention glossary entry, allocation and eviction: blocks
               moved to host memory), other work takes their GPU blocks, and the
               sequences come back into freshly allocated GPU blocks.

Readings (listed in the design notes): the decode after a write attends to the
token just written; the shared-prefix fork point is prefix + k_p with
k_p ~ U{0..15}, so the prompt's last block is partly filled and the first
append of each sample hits a shared block; within a step, samples append in
ascending index, so the last holder of a shared block writes in place.
"""
from __future__ import annotations

import copy
import dataclasses
import math
from typing import List, Optional

import numpy as np

import synthetic as syn
from .block_manager import BlockManager, Sequence, check_invariants
from .cache_ops import copy_blocks, reshape_and_cache, swap_blocks


@dataclasses.dataclass
class PagedBatch:
    workload: syn.Workload
    block_size: int
    num_blocks: int
    k_pool: np.ndarray          # [NB, bs, Hkv, D] uint16
    v_pool: np.ndarray
    q: np.ndarray               # [B, Hq, D] uint16
    block_tables: np.ndarray    # [B, max_blocks] int32
    seq_lens: np.ndarray        # [B] int32
    pad_block: int
    manager: BlockManager
    sequences: List[Sequence]

    @property
    def dtype(self) -> int:
        return self.workload.dtype

    @property
    def scale(self) -> float:
        return self.workload.scale

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]


@dataclasses.dataclass
class Step:
    """One decode step's writes: CoW copies first, then the new tokens."""
    cow_pairs: np.ndarray       # [n, 2] int32 (src, dst)
    slot_mapping: np.ndarray    # [T] int32
    key: np.ndarray             # [T, Hkv, D] uint16
    value: np.ndarray
    block_tables: np.ndarray    # tables after the step [B, max_blocks] int32
    seq_lens: np.ndarray        # lengths after the step [B] int32


def _tables(seqs: List[Sequence], pad: int, max_blocks: Optional[int] = None) -> np.ndarray:
    mb = max(1, max(len(s.block_table) for s in seqs))
    if max_blocks is not None:
        mb = max(mb, max_blocks)
    out = np.full((len(seqs), mb), pad, dtype=np.int32)
    for i, s in enumerate(seqs):
        out[i, :len(s.block_table)] = s.block_table
    return out


def _empty_pools(w: syn.Workload, nb: int, bs: int):
    shape = (nb, bs, w.num_kv_heads, w.head_dim)
    return syn.nan_bits(shape, w.dtype), syn.nan_bits(shape, w.dtype)


def _store_tokens(k_pool, v_pool, seq: Sequence, key, value, start: int = 0) -> None:
    slots = np.array([seq.physical_index(p) for p in range(start, start + key.shape[0])],
                     dtype=np.int64)
    reshape_and_cache(k_pool, v_pool, key, value, slots)


def fixed_batch(w: syn.Workload, lens=None, block_size: Optional[int] = None,
                fill_all: bool = False) -> PagedBatch:
    """Every sequence holds its tokens; tables padded with a NaN block.

    fill_all: fill every slot of the pool with random values instead of writing
    tokens one sequence at a time (large workloads checked on sampled rows)."""
    bs = block_size or w.block_size
    lens = syn.seq_lens(w) if lens is None else np.asarray(lens, dtype=np.int64)
    need = sum(-(-int(L) // bs) for L in lens)
    nb = w.num_blocks or int(math.ceil(w.pool_factor * need)) + 1
    mgr = BlockManager(nb, bs, syn.shuffled_free_order(nb, syn.rng(w, "free")))
    pad = mgr.allocate(1)[0]
    seqs = [Sequence(mgr, int(L)) for L in lens]
    if fill_all:
        wb = dataclasses.replace(w, block_size=bs)
        k_pool, v_pool = syn.pool_fill_bits(wb, nb)
        k_pool[pad] = syn.NAN_BITS[w.dtype]
        v_pool[pad] = syn.NAN_BITS[w.dtype]
    else:
        k_pool, v_pool = _empty_pools(w, nb, bs)
        for b, s in enumerate(seqs):
            key, value = syn.token_kv_bits(w, s.length, sub=b)
            _store_tokens(k_pool, v_pool, s, key, value)
    check_invariants(mgr, [[pad]] + [s.block_table for s in seqs])
    return PagedBatch(w, bs, nb, k_pool, v_pool, syn.query_bits(w, len(lens)),
                      _tables(seqs, pad), lens.astype(np.int32), pad, mgr, seqs)


def shared_prefix(w: syn.Workload, num_prompts: Optional[int] = None,
                  tail_cap: Optional[int] = None):
    """Returns (initial PagedBatch with the prompts written, list of Steps,
    final PagedBatch after applying every step on the oracle's pools)."""
    bs = w.block_size
    P = num_prompts or w.num_prompts
    S = w.samples_per_prompt
    extra = syn.prompt_extra_tokens(w)[:P]
    tails = syn.sample_tail_lens(w)[:P]
    if tail_cap is not None:
        tails = np.minimum(tails, tail_cap)
    prompt_lens = [w.prefix_tokens + int(k) for k in extra]
    # peak blocks: shared prompt blocks + each sample's private blocks (+1 CoW copy)
    peak = 0
    for p in range(P):
        nblk = -(-prompt_lens[p] // bs)
        peak += nblk
        for s in range(S):
            total = prompt_lens[p] + int(tails[p, s])
            peak += -(-total // bs) - nblk + 1
    nb = int(math.ceil(w.pool_factor * peak)) + 1
    mgr = BlockManager(nb, bs, syn.shuffled_free_order(nb, syn.rng(w, "free")))
    pad = mgr.allocate(1)[0]
    k_pool, v_pool = _empty_pools(w, nb, bs)
    samples: List[Sequence] = []
    for p in range(P):
        root = Sequence(mgr, prompt_lens[p])
        key, value = syn.token_kv_bits(w, prompt_lens[p], sub=p)
        _store_tokens(k_pool, v_pool, root, key, value)
        samples.append(root)
        for _ in range(S - 1):
            samples.append(root.fork())
    tail_flat = [int(tails[p, s]) for p in range(P) for s in range(S)]
    max_blocks = max(-(-(len_ + t) // bs) for len_, t in
                     zip([prompt_lens[i // S] for i in range(P * S)], tail_flat))
    initial = PagedBatch(w, bs, nb, k_pool.copy(), v_pool.copy(),
                         syn.query_bits(w, P * S), _tables(samples, pad, max_blocks),
                         np.array([s.length for s in samples], dtype=np.int32), pad,
                         mgr, samples)
    steps: List[Step] = []
    for t in range(max(tail_flat) if tail_flat else 0):
        active = [i for i in range(P * S) if tail_flat[i] > t]
        pairs, slots = [], []
        for i in active:
            slot, cow = samples[i].append_token()
            if cow is not None:
                pairs.append(cow)
            slots.append(slot)
        key, value = syn.token_kv_bits(w, len(active), sub=100_000 + t)
        pairs_arr = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
        slots_arr = np.asarray(slots, dtype=np.int32)
        copy_blocks(k_pool, v_pool, pairs_arr)
        reshape_and_cache(k_pool, v_pool, key, value, slots_arr)
        steps.append(Step(pairs_arr, slots_arr, key, value,
                          _tables(samples, pad, max_blocks),
                          np.array([s.length for s in samples], dtype=np.int32)))
    check_invariants(mgr, [[pad]] + [s.block_table for s in samples])
    final = PagedBatch(w, bs, nb, k_pool, v_pool, initial.q,
                       _tables(samples, pad, max_blocks),
                       np.array([s.length for s in samples], dtype=np.int32), pad,
                       mgr, samples)
    return initial, steps, final


def ragged_steps(w: syn.Workload, block_size: int, num_steps: int,
                 num_seqs: Optional[int] = None):
    """Returns (initial PagedBatch holding L_b - 1 tokens per sequence, Steps,
    final PagedBatch).  Each Step's tables/lengths are those its decode uses."""
    bs = block_size
    lens = syn.seq_lens(w)
    if num_seqs is not None:
        lens = lens[:num_seqs]
    B = len(lens)
    final_lens = lens + num_steps - 1
    need = sum(-(-int(L) // bs) for L in final_lens)
    nb = int(math.ceil(w.pool_factor * need)) + 1
    wb = dataclasses.replace(w, block_size=bs)
    mgr = BlockManager(nb, bs, syn.shuffled_free_order(nb, syn.rng(wb, "free", bs)))
    pad = mgr.allocate(1)[0]
    k_pool, v_pool = _empty_pools(w, nb, bs)
    seqs = []
    for b, L in enumerate(lens):
        s = Sequence(mgr, int(L) - 1)
        if s.length:
            key, value = syn.token_kv_bits(wb, s.length, sub=b)
            _store_tokens(k_pool, v_pool, s, key, value)
        seqs.append(s)
    max_blocks = max(-(-int(L) // bs) for L in final_lens)
    initial = PagedBatch(w, bs, nb, k_pool.copy(), v_pool.copy(), syn.query_bits(wb, B),
                         _tables(seqs, pad, max_blocks),
                         np.array([s.length for s in seqs], dtype=np.int32), pad, mgr, seqs)
    steps = []
    for t in range(num_steps):
        slots = []
        for s in seqs:
            slot, cow = s.append_token()
            assert cow is None
            slots.append(slot)
        key, value = syn.token_kv_bits(wb, B, sub=200_000 + t)
        slots_arr = np.asarray(slots, dtype=np.int32)
        reshape_and_cache(k_pool, v_pool, key, value, slots_arr)
        steps.append(Step(np.zeros((0, 2), np.int32), slots_arr, key, value,
                          _tables(seqs, pad, max_blocks),
                          np.array([s.length for s in seqs], dtype=np.int32)))
    check_invariants(mgr, [[pad]] + [s.block_table for s in seqs])
    final = PagedBatch(w, bs, nb, k_pool, v_pool, initial.q, _tables(seqs, pad, max_blocks),
                       np.array([s.length for s in seqs], dtype=np.int32), pad, mgr, seqs)
    return initial, steps, final


def decode_f64(batch: PagedBatch, sequences=None, heads=None) -> np.ndarray:
    """fp64 oracle output of a batch (convenience wrapper)."""
    from .attention import paged_decode_attention
    return paged_decode_attention(
        batch.q, batch.k_pool, batch.v_pool, batch.block_tables, batch.seq_lens,
        batch.scale, sequences=sequences, heads=heads, dtype=batch.dtype)


@dataclasses.dataclass
class SwapRoundTrip:
    before: PagedBatch           # the batch as given (not modified)
    after: PagedBatch            # after swap-out, reuse of the freed blocks, swap-in
    cpu_num_blocks: int
    out_pairs: np.ndarray        # [n, 2] (GPU block, CPU block)
    in_pairs: np.ndarray         # [n, 2] (CPU block, new GPU block)
    reused_blocks: np.ndarray    # GPU blocks another sequence took meanwhile (poisoned)
    cpu_k_pool: np.ndarray       # CPU pools right after the swap-out
    cpu_v_pool: np.ndarray


def swap_round_trip(batch: PagedBatch, swapped, cpu_num_blocks: int,
                    seed: int = 0) -> SwapRoundTrip:
    """Evict the sequences `swapped` to CPU pools, let another sequence take (and
    overwrite) the GPU blocks they freed, then bring them back.

    Swap-out: each evicted sequence gets CPU blocks from a CPU-side block manager
    (seeded free order), its blocks move GPU -> CPU, its GPU blocks are freed.
    Reuse: one new sequence allocates exactly the freed blocks (the free stack is
    last-in first-out) and fills them with NaN.  Swap-in: each evicted sequence
    allocates new GPU blocks, its blocks move CPU -> GPU, its CPU blocks are freed
    and its table points at the new blocks.  Attention over the result must be
    identical to attention over the batch as given."""
    after = copy.deepcopy(batch)
    mgr, seqs, bs = after.manager, after.sequences, after.block_size
    shape = after.k_pool.shape[1:]
    nan = syn.NAN_BITS[after.dtype]
    cpu_k = np.full((cpu_num_blocks,) + shape, nan, dtype=np.uint16)
    cpu_v = cpu_k.copy()
    cpu_mgr = BlockManager(cpu_num_blocks, bs,
                           syn.shuffled_free_order(cpu_num_blocks, np.random.default_rng(seed)))
    out_pairs, cpu_ids = [], {}
    for b in swapped:
        ids = cpu_mgr.allocate(len(seqs[b].block_table))
        cpu_ids[b] = ids
        out_pairs += list(zip(seqs[b].block_table, ids))
    out_arr = np.asarray(out_pairs, dtype=np.int32).reshape(-1, 2)
    swap_blocks([cpu_k, cpu_v], [after.k_pool, after.v_pool], out_arr)
    cpu_k_out, cpu_v_out = cpu_k.copy(), cpu_v.copy()
    freed = 0
    for b in swapped:
        freed += len(seqs[b].block_table)
        mgr.free_blocks(seqs[b].block_table)
        seqs[b].block_table = []
    reused = mgr.allocate(freed)
    after.k_pool[reused] = nan
    after.v_pool[reused] = nan
    in_pairs = []
    for b in swapped:
        new = mgr.allocate(len(cpu_ids[b]))
        in_pairs += list(zip(cpu_ids[b], new))
        seqs[b].block_table = new
    in_arr = np.asarray(in_pairs, dtype=np.int32).reshape(-1, 2)
    swap_blocks([after.k_pool, after.v_pool], [cpu_k, cpu_v], in_arr)
    for b in swapped:
        cpu_mgr.free_blocks(cpu_ids[b])
    check_invariants(mgr, [[after.pad_block], reused] + [s.block_table for s in seqs])
    check_invariants(cpu_mgr, [])
    after.block_tables = _tables(seqs, after.pad_block, batch.max_blocks)
    return SwapRoundTrip(batch, after, cpu_num_blocks, out_arr, in_arr,
                         np.asarray(reused, dtype=np.int32), cpu_k_out, cpu_v_out)


@dataclasses.dataclass
class PrefillBatch:
    batch: PagedBatch            # pools, tables, lengths (KV of every token written)
    q: np.ndarray                # [total_q, Hq, D] uint16 storage bits
    q_start: np.ndarray          # [B + 1] int32


def prefill_batch(w: syn.Workload, lens=None, q_counts=None, block_size: Optional[int] = None,
                  fill_all: bool = False) -> PrefillBatch:
    """A paged batch holding every token's KV plus queries for the last
    q_counts[b] tokens of each sequence (all of them for a whole-prompt
    prefill)."""
    batch = fixed_batch(w, lens=lens, block_size=block_size, fill_all=fill_all)
    n = syn.query_counts(w, batch.seq_lens) if q_counts is None else \
        np.asarray(q_counts, dtype=np.int64)
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = syn.prefill_query_bits(w, int(q_start[-1]))
    return PrefillBatch(batch, q, q_start)


def prefill_f64(pb: PrefillBatch, rows=None) -> np.ndarray:
    from .prefill import paged_prefill_attention
    b = pb.batch
    return paged_prefill_attention(pb.q, b.k_pool, b.v_pool, b.block_tables, b.seq_lens,
                                   pb.q_start, b.scale, dtype=b.dtype, rows=rows)
