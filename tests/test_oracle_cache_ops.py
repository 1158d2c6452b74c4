"""Pins of the oracle's cache write, block copy and copy-on-write flows (CPU only)."""
import numpy as np

import synthetic as syn
from oracle import scenarios
from oracle.block_manager import BlockManager, Sequence
from oracle.cache_ops import copy_blocks, reshape_and_cache


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
