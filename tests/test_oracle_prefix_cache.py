"""Pins of the oracle's prefix cache (CPU only): the published FNV-1a-64 test
values, the sharing arithmetic of a common system prompt, the prefix-chained
keys, the eviction order, and the pool invariants under random traffic."""
import numpy as np
import pytest

from oracle.block_manager import OutOfBlocks, Sequence
from oracle.prefix_cache import (PrefixCachingBlockManager, block_key, check_cache_invariants,
                                 fnv1a64)


def test_fnv1a64_published_values():
    """Test values published with the Fowler-Noll-Vo hash definition."""
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_key_layout():
    """parent as 8 little-endian bytes, then each token as 4 little-endian bytes."""
    assert block_key(0, [1, -1]) == fnv1a64(bytes(8) + b"\x01\x00\x00\x00" + b"\xff\xff\xff\xff")
    assert block_key(0x0102030405060708, []) == fnv1a64(bytes([8, 7, 6, 5, 4, 3, 2, 1]))


@pytest.mark.parametrize("bs", [4, 16])
def test_shared_system_prompt_arithmetic(bs):
    """N requests = a P-token system prompt + private suffixes: the floor(P/bs)
    full prompt blocks exist once with refcount N; every request after the first
    skips exactly those tokens: shared blocks are referenced again, not
    recomputed (tutorial §5, the relationship to prefix caching)."""
    g = np.random.default_rng(bs)
    P, N = 5 * bs + bs // 2, 6
    prompt = list(g.integers(0, 1000, size=P))
    mgr = PrefixCachingBlockManager(200, bs, list(g.permutation(200)))
    seqs, cached = [], []
    for i in range(N):
        suffix = list(g.integers(0, 1000, size=int(g.integers(1, 3 * bs))))
        s, c = mgr.create_sequence(prompt + suffix)
        seqs.append(s)
        cached.append(c)
    full = P // bs
    assert cached == [0] + [full * bs] * (N - 1)
    shared = seqs[0].block_table[:full]
    for s in seqs:
        assert s.block_table[:full] == shared
    assert all(mgr.refcount[b] == N for b in shared)
    want_blocks = full + sum(s.mgr.blocks_needed(s.length) - full for s in seqs)
    assert mgr.num_used == want_blocks
    check_cache_invariants(mgr, [s.block_table for s in seqs])


def test_keys_cover_the_whole_prefix():
    """Equal block contents after different prefixes, or at another position,
    are different keys: only a common prefix is shared."""
    bs = 4
    mgr = PrefixCachingBlockManager(32, bs)
    a, _ = mgr.create_sequence([1, 2, 3, 4, 5, 6, 7, 8, 9, 9, 9, 9])
    b, cb = mgr.create_sequence([1, 2, 3, 4, 0, 0, 0, 0, 9, 9, 9, 9])
    c, cc = mgr.create_sequence([9, 9, 9, 9, 1, 2, 3, 4])
    assert cb == 4 and b.block_table[0] == a.block_table[0]
    assert b.block_table[2] != a.block_table[2]
    assert cc == 0 and not set(c.block_table) & set(a.block_table)
    # a partly filled last block is never shared
    d, cd = mgr.create_sequence([1, 2, 3, 4, 5, 6, 7, 8, 9, 9])
    assert cd == 8 and d.block_table[2] not in a.block_table
    check_cache_invariants(mgr, [s.block_table for s in (a, b, c, d)])


def test_released_prefix_stays_cached_until_evicted_tail_first():
    bs = 4
    mgr = PrefixCachingBlockManager(8, bs)
    prompt = list(range(12))
    a, _ = mgr.create_sequence(prompt)
    a0, a1, a2 = a.block_table
    a.release()
    assert mgr.num_free == 5 and mgr.evictable == [a2, a1, a0]
    again, c = mgr.create_sequence(prompt)            # all three come back
    assert c == 12 and again.block_table == [a0, a1, a2] and not mgr.evictable
    again.release()
    other = mgr.allocate(6)                           # 5 free + the queue's front (a2)
    assert a2 in other and mgr.evictable == [a1, a0]
    mgr.free_blocks([other.pop()])
    third, c3 = mgr.create_sequence(prompt)           # a0, a1 hit; block 2 recomputed
    assert c3 == 8 and third.block_table[:2] == [a0, a1]
    check_cache_invariants(mgr, [other, third.block_table])
    with pytest.raises(OutOfBlocks):
        mgr.create_sequence(list(range(100, 120)))


def test_shortage_counts_queued_hits_as_unavailable():
    """A request that hits queued blocks cannot also evict them for its own new
    blocks; when that leaves too few, nothing changes."""
    bs = 2
    mgr = PrefixCachingBlockManager(4, bs)
    a, _ = mgr.create_sequence([1, 2, 3, 4])
    a.release()                                       # 2 queued, 2 free
    before = (list(mgr.free), list(mgr.evictable), dict(mgr.refcount))
    with pytest.raises(OutOfBlocks):
        mgr.create_sequence([1, 2, 3, 4, 5, 6, 7, 8, 9])   # 2 hits + 3 new > 2 free
    assert (list(mgr.free), list(mgr.evictable), dict(mgr.refcount)) == before
    s, c = mgr.create_sequence([1, 2, 3, 4, 5, 6, 7])      # 2 hits + 2 new
    assert c == 4
    check_cache_invariants(mgr, [s.block_table])


@pytest.mark.parametrize("seed", range(4))
def test_random_traffic_keeps_invariants(seed):
    g = np.random.default_rng(seed)
    bs = [2, 4, 8, 16][seed]
    mgr = PrefixCachingBlockManager(64, bs, list(g.permutation(64)))
    prompts = [list(g.integers(0, 50, size=int(g.integers(1, 6 * bs)))) for _ in range(6)]
    live = []
    for _ in range(2000):
        op = g.integers(0, 5)
        try:
            if op <= 1 or not live:
                base = prompts[int(g.integers(0, len(prompts)))]
                cut = int(g.integers(0, len(base) + 1))
                toks = base[:cut] + list(g.integers(0, 50, size=int(g.integers(0, 2 * bs))))
                s, c = mgr.create_sequence(toks)
                assert c % bs == 0 and c <= len(toks)
                live.append(s)
            elif op == 2:
                live.pop(int(g.integers(0, len(live)))).release()
            elif op == 3:
                live[int(g.integers(0, len(live)))].append_token()
            else:
                live.append(live[int(g.integers(0, len(live)))].fork())
        except OutOfBlocks:
            pass
        check_cache_invariants(mgr, [s.block_table for s in live])
