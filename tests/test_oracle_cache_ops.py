"""Pins of the oracle's cache write, block copy and copy-on-write flows (CPU only)."""
import dataclasses

import numpy as np

import synthetic as syn
from oracle import scenarios
from oracle.block_manager import BlockManager, Sequence
from oracle.cache_ops import copy_blocks, copy_blocks_multi, reshape_and_cache, swap_blocks


def _pool(nb, bs, H, D, fill):
    return np.full((nb, bs, H, D), fill, dtype=np.uint16)


def test_reshape_and_cache_matches_blockwise_layout():
    """Writing a sequence token by token through its slots gives the layout in
    which logical block i occupies physical block table[i], rows in order."""
    bs, H, D = 4, 2, 8
    g = np.random.default_rng(1)
    mgr = BlockManager(12, bs, list(g.permutation(12)))
    s = Sequence(mgr, 0)
    L = 15
    key = g.integers(0, 2**16, size=(L, H, D), dtype=np.uint16)
    val = g.integers(0, 2**16, size=(L, H, D), dtype=np.uint16)
    kp, vp = _pool(12, bs, H, D, 0xAAAA), _pool(12, bs, H, D, 0x5555)
    for t in range(L):
        slot, _ = s.append_token()
        reshape_and_cache(kp, vp, key[t:t + 1], val[t:t + 1], [slot])
    expect_k, expect_v = _pool(12, bs, H, D, 0xAAAA), _pool(12, bs, H, D, 0x5555)
    for i, blk in enumerate(s.block_table):
        n = min(bs, L - i * bs)
        expect_k[blk, :n] = key[i * bs:i * bs + n]
        expect_v[blk, :n] = val[i * bs:i * bs + n]
    assert np.array_equal(kp, expect_k) and np.array_equal(vp, expect_v)


def test_negative_slots_are_skipped():
    kp, vp = _pool(4, 2, 1, 4, 7), _pool(4, 2, 1, 4, 9)
    key = np.ones((3, 1, 4), np.uint16)
    reshape_and_cache(kp, vp, key, key * 2, [-1, 5, -7])
    assert (kp[2, 1] == 1).all() and (vp[2, 1] == 2).all()
    kp[2, 1] = 7
    vp[2, 1] = 9
    assert (kp == 7).all() and (vp == 9).all()


def test_copy_blocks_copies_whole_blocks_only():
    g = np.random.default_rng(2)
    kp = g.integers(0, 2**16, size=(8, 4, 2, 8), dtype=np.uint16)
    vp = g.integers(0, 2**16, size=(8, 4, 2, 8), dtype=np.uint16)
    k0, v0 = kp.copy(), vp.copy()
    copy_blocks(kp, vp, [(1, 6), (3, 0)])
    assert np.array_equal(kp[6], k0[1]) and np.array_equal(vp[6], v0[1])
    assert np.array_equal(kp[0], k0[3]) and np.array_equal(vp[0], v0[3])
    rest = [1, 2, 3, 4, 5, 7]
    assert np.array_equal(kp[rest], k0[rest]) and np.array_equal(vp[rest], v0[rest])


def _logical(pool, seq, bs):
    return np.stack([pool[seq.block_table[p // bs], p % bs] for p in range(seq.length)])


def test_shared_prefix_flow_keeps_every_sample_consistent():
    """After forks, copy-on-write and per-sample appends, every sample reads
    back exactly the prompt followed by its own generated tokens."""
    w = syn.SHARED_PREFIX.__class__(**{**syn.SHARED_PREFIX.__dict__, "prefix_tokens": 40,
                                       "block_size": 8, "num_q_heads": 4, "num_kv_heads": 2,
                                       "head_dim": 16})
    P, cap = 3, 20
    initial, steps, final = scenarios.shared_prefix(w, num_prompts=P, tail_cap=cap)
    S = w.samples_per_prompt
    tails = np.minimum(syn.sample_tail_lens(w)[:P], cap).reshape(-1)
    extra = syn.prompt_extra_tokens(w)[:P]
    assert any(len(st.cow_pairs) for st in steps) == any(k % 8 for k in extra)
    # the generated keys of sample i: step t hands rows to active samples in order
    generated = {i: [] for i in range(P * S)}
    for t, st in enumerate(steps):
        active = [i for i in range(P * S) if tails[i] > t]
        assert len(active) == len(st.slot_mapping)
        for j, i in enumerate(active):
            generated[i].append(st.key[j])
    for p in range(P):
        Lp = 40 + int(extra[p])
        pk, _ = syn.token_kv_bits(w, Lp, sub=p)
        for s in range(S):
            i = p * S + s
            seq = final.sequences[i]
            assert seq.length == Lp + tails[i]
            got = _logical(final.k_pool, seq, w.block_size)
            assert np.array_equal(got[:Lp], pk)
            if tails[i]:
                assert np.array_equal(got[Lp:], np.stack(generated[i]))
    for st in steps:
        assert len(set(st.slot_mapping.tolist())) == len(st.slot_mapping)


def test_copy_on_write_fires_once_per_sharer():
    bs = 4
    w = syn.SHARED_PREFIX.__class__(**{**syn.SHARED_PREFIX.__dict__, "prefix_tokens": 8,
                                       "block_size": bs, "num_q_heads": 2, "num_kv_heads": 1,
                                       "head_dim": 8})
    initial, steps, final = scenarios.shared_prefix(w, num_prompts=4, tail_cap=6)
    extra = syn.prompt_extra_tokens(w)[:4]
    tails = np.minimum(syn.sample_tail_lens(w)[:4], 6)
    S = w.samples_per_prompt
    expect = 0
    for p in range(4):
        if extra[p] % bs:
            writers = int((tails[p] > 0).sum())
            expect += max(0, writers - 1) if writers == S else writers
    got = sum(len(st.cow_pairs) for st in steps)
    # sharers that append copy; the last remaining holder writes in place
    assert got == expect


def test_copy_blocks_multi_is_copy_blocks_on_every_layer():
    """Every layer's K and V pools get the same clones, and nothing else moves;
    checked element by element against the pools as they were."""
    g = np.random.default_rng(3)
    L, NB = 3, 9
    pools = [g.integers(0, 2**16, size=(NB, 2, 2, 4), dtype=np.uint16) for _ in range(2 * L)]
    before = [p.copy() for p in pools]
    pairs = [(4, 0), (7, 2), (1, 8)]
    copy_blocks_multi(pools, pairs)
    dst_of = {d: s for s, d in pairs}
    for p, p0 in zip(pools, before):
        for blk in range(NB):
            src = dst_of.get(blk, blk)
            for idx in np.ndindex(p.shape[1:]):
                assert p[(blk,) + idx] == p0[(src,) + idx]
    # one layer through the two-pool copy gives the same bytes
    k, v = before[0].copy(), before[1].copy()
    copy_blocks(k, v, pairs)
    assert np.array_equal(k, pools[0]) and np.array_equal(v, pools[1])


def test_swap_blocks_between_pools_of_different_sizes():
    g = np.random.default_rng(4)
    gpu = [g.integers(0, 2**16, size=(10, 4, 1, 8), dtype=np.uint16) for _ in range(2)]
    cpu = [np.zeros((3, 4, 1, 8), dtype=np.uint16) for _ in range(2)]
    swap_blocks(cpu, gpu, [(9, 0), (2, 2)])
    for c, gp in zip(cpu, gpu):
        assert np.array_equal(c[0], gp[9]) and np.array_equal(c[2], gp[2])
        assert not c[1].any()


def test_swap_round_trip_restores_attention_exactly():
    """Evict half the sequences to CPU RAM, let other work overwrite their GPU
    blocks, swap them back into different blocks: the fp64 attention is
    bit-identical (it depends on the logical token order only), the moved blocks
    hold the same bytes, and the freed blocks were really reused."""
    w = dataclasses.replace(syn.TINY, pool_factor=3.0)
    batch = scenarios.fixed_batch(w)
    want = scenarios.decode_f64(batch)
    rt = scenarios.swap_round_trip(batch, [0, 2], cpu_num_blocks=16, seed=5)
    got = scenarios.decode_f64(rt.after)
    assert np.array_equal(got, want)
    old = {int(gp): int(c) for gp, c in rt.out_pairs}
    new = {int(c): int(gp) for c, gp in rt.in_pairs}
    assert set(old.values()) == set(new)
    for gp, c in old.items():
        assert np.array_equal(rt.cpu_k_pool[c], batch.k_pool[gp])
        assert np.array_equal(rt.after.k_pool[new[c]], batch.k_pool[gp])
        assert np.array_equal(rt.after.v_pool[new[c]], batch.v_pool[gp])
    assert set(rt.reused_blocks.tolist()) == set(old)
    assert not set(new.values()) & set(old)        # the sequences moved
    assert np.array_equal(rt.before.k_pool, batch.k_pool)
    # a sequence that was not swapped kept its table
    assert np.array_equal(rt.after.block_tables[1], batch.block_tables[1])
