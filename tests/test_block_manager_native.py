"""The library's C++ block manager (pa_bm_*) agrees exactly with the oracle's
block manager on the tutorial's worked example and on long random sequences of
create / fork / append / release operations (CPU only, host code)."""
import json
import os

import numpy as np
import pytest

from oracle.block_manager import BlockManager as OracleBM
from oracle.block_manager import OutOfBlocks, Sequence

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def native():
    from paged_kv_cache_301_gb300 import build
    build.build()
    import paged_kv_cache_301_gb300 as pa
    return pa


def test_go_tiny_example(native):
    g = json.load(open(os.path.join(GOLDEN, "go_tiny_example_trace.json")))
    bm = native.BlockManager(g["num_blocks"], g["block_size"])
    seqs = {n: bm.new_sequence(32) for n in "abcd"}
    tables, _ = bm.export([seqs[n] for n in "abcd"], 2, -1)
    assert tables.tolist() == [g["tables"][n] for n in "abcd"]
    bm.release(seqs["b"])
    bm.release(seqs["d"])
    assert bm.num_free == len(g["free_after_freeing_d"])
    e = bm.new_sequence(64)
    t, lens = bm.export([e], 4, -1)
    assert t.tolist()[0] == g["e_table"] and lens.tolist() == [64]
    # appended slots follow PhysicalIndex: token 64 opens a fifth block
    slot, cow = bm.append(e)
    t5, _ = bm.export([e], 5, -1)
    assert cow is None and slot == t5.tolist()[0][4] * g["block_size"]


def test_errors(native):
    bm = native.BlockManager(4, 16)
    ids = bm.allocate(3)
    with pytest.raises(native.PagedAttnError) as ei:
        bm.allocate(2)
    assert ei.value.status == 6 and bm.num_free == 1
    bm.free(ids)
    with pytest.raises(native.PagedAttnError) as ei:
        bm.free([ids[0]])
    assert ei.value.status == 7
    with pytest.raises(native.PagedAttnError):
        bm.fork_blocks([ids[0]])
    with pytest.raises(native.PagedAttnError):
        native.BlockManager(3, 16, free_stack=[0, 0, 1])
    # a request that would free a block twice in one call changes nothing
    a = bm.allocate(1)
    with pytest.raises(native.PagedAttnError):
        bm.free([a[0], a[0]])
    assert bm.refcount(a[0]) == 1


@pytest.mark.parametrize("seed", range(5))
def test_random_operations_match_oracle(native, seed):
    g = np.random.default_rng(seed)
    nb, bs = 96, [4, 8, 16, 2, 32][seed]
    order = [int(x) for x in g.permutation(nb)]
    ob = OracleBM(nb, bs, order)
    nbm = native.BlockManager(nb, bs, order)
    live = {}   # native id -> oracle Sequence
    for step in range(3000):
        op = g.integers(0, 10)
        if op == 0 or not live:
            L = int(g.integers(0, 3 * bs))
            try:
                o = Sequence(ob, L)
            except OutOfBlocks:
                with pytest.raises(native.PagedAttnError):
                    nbm.new_sequence(L)
                continue
            live[nbm.new_sequence(L)] = o
        elif op == 1:
            sid = list(live)[int(g.integers(0, len(live)))]
            live[nbm.fork(sid)] = live[sid].fork()
        elif op == 2 and len(live) > 3:
            sid = list(live)[int(g.integers(0, len(live)))]
            live.pop(sid).release()
            nbm.release(sid)
        else:
            sid = list(live)[int(g.integers(0, len(live)))]
            try:
                want = live[sid].append_token()
            except OutOfBlocks:
                with pytest.raises(native.PagedAttnError):
                    nbm.append(sid)
                continue
            assert nbm.append(sid) == want
        assert nbm.num_free == ob.num_free
    for b in range(nb):
        assert nbm.refcount(b) == ob.refcount.get(b, 0)
    ids = list(live)
    mb = max(1, max(len(live[i].block_table) for i in ids))
    tables, lens = nbm.export(ids, mb, -1)
    for row, L, i in zip(tables.tolist(), lens.tolist(), ids):
        t = live[i].block_table
        assert row[:len(t)] == t and L == live[i].length


@pytest.mark.parametrize("seed", range(4))
def test_prefix_cache_matches_oracle(native, seed):
    """Random traffic of cached prompts (drawn from a few shared prefixes, so
    that hits, revivals from the eviction queue and evictions all happen),
    releases, appends and forks: the native manager hands out the same blocks,
    reports the same cached prefixes and ends in the same state."""
    from oracle.prefix_cache import PrefixCachingBlockManager
    g = np.random.default_rng(100 + seed)
    nb, bs = 80, [2, 4, 8, 16][seed]
    order = [int(x) for x in g.permutation(nb)]
    ob = PrefixCachingBlockManager(nb, bs, order)
    nbm = native.BlockManager(nb, bs, order)
    prompts = [list(g.integers(-5, 40, size=int(g.integers(1, 5 * bs)))) for _ in range(5)]
    live = {}
    hits = 0
    for step in range(3000):
        op = g.integers(0, 6)
        if op <= 1 or not live:
            base = prompts[int(g.integers(0, len(prompts)))]
            toks = base[:int(g.integers(0, len(base) + 1))] + \
                list(g.integers(-5, 40, size=int(g.integers(0, 2 * bs))))
            try:
                o, c = ob.create_sequence(toks)
            except OutOfBlocks:
                with pytest.raises(native.PagedAttnError):
                    nbm.new_sequence_cached(toks)
                continue
            sid, nc = nbm.new_sequence_cached(toks)
            assert nc == c
            hits += c > 0
            live[sid] = o
        elif op == 2:
            sid = list(live)[int(g.integers(0, len(live)))]
            live.pop(sid).release()
            nbm.release(sid)
        elif op == 3:
            sid = list(live)[int(g.integers(0, len(live)))]
            live[nbm.fork(sid)] = live[sid].fork()
        else:
            sid = list(live)[int(g.integers(0, len(live)))]
            try:
                want = live[sid].append_token()
            except OutOfBlocks:
                with pytest.raises(native.PagedAttnError):
                    nbm.append(sid)
                continue
            assert nbm.append(sid) == want
        assert nbm.num_free == ob.num_free and nbm.num_evictable == ob.num_evictable
    assert hits > 10
    for b in range(nb):
        assert nbm.refcount(b) == ob.refcount.get(b, 0)
    if live:
        ids = list(live)
        mb = max(1, max(len(live[i].block_table) for i in ids))
        tables, lens = nbm.export(ids, mb, -1)
        for row, L, i in zip(tables.tolist(), lens.tolist(), ids):
            t = live[i].block_table
            assert row[:len(t)] == t and L == live[i].length
