"""Pins of the oracle's block manager against the pages' worked examples,
arithmetic and invariants (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import accounting
from oracle.block_manager import (BlockManager, BlockStateError, OutOfBlocks, Sequence,
                                  check_invariants)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_go_tiny_example_trace():
    """Tutorial §4 'Tiny example': scattered free blocks still satisfy a
    4-block request; token 40 of e lands in slot 120."""
    g = _load("go_tiny_example_trace.json")
    mgr = BlockManager(g["num_blocks"], g["block_size"])
    assert mgr.free == g["initial_free_stack_bottom_to_top"]
    seqs = {name: Sequence(mgr, 32) for name in "abcd"}
    for name, table in g["tables"].items():
        assert seqs[name].block_table == table
    assert mgr.free == g["free_after_four_allocations"]
    mgr.free_blocks(seqs["b"].block_table)
    assert mgr.free == g["free_after_freeing_b"]
    mgr.free_blocks(seqs["d"].block_table)
    assert mgr.free == g["free_after_freeing_d"]
    e = Sequence(mgr, 64)
    assert e.block_table == g["e_table"]
    assert mgr.free == g["free_after_e"]
    assert e.physical_index(40) == g["e_physical_index_of_token_40"]
    check_invariants(mgr, [seqs["a"].block_table, seqs["c"].block_table, e.block_table])


def test_physical_index_is_a_page_walk():
    """Slot = frame * page size + offset for every position (tutorial §4)."""
    mgr = BlockManager(64, 8, list(np.random.default_rng(5).permutation(64)))
    s = Sequence(mgr, 50)
    seen = set()
    for pos in range(50):
        slot = s.physical_index(pos)
        assert slot // 8 == s.block_table[pos // 8]
        assert slot % 8 == pos % 8
        seen.add(slot)
    assert len(seen) == 50
    with pytest.raises(IndexError):
        s.physical_index(56)


def test_allocate_shortage_leaves_state():
    mgr = BlockManager(4, 16)
    mgr.allocate(3)
    before = (list(mgr.free), dict(mgr.refcount))
    with pytest.raises(OutOfBlocks):
        mgr.allocate(2)
    assert (mgr.free, mgr.refcount) == before
    assert mgr.allocate(0) == []


def test_free_and_fork_errors():
    mgr = BlockManager(4, 16)
    (b,) = mgr.allocate(1)
    mgr.free_blocks([b])
    with pytest.raises(BlockStateError):
        mgr.free_blocks([b])
    with pytest.raises(BlockStateError):
        mgr.fork([b])


def test_refcount_frees_only_at_zero():
    mgr = BlockManager(8, 16)
    s = Sequence(mgr, 20)
    t = s.fork()
    assert all(mgr.refcount[b] == 2 for b in s.block_table)
    s.release()
    assert mgr.num_free == 6
    t.release()
    assert mgr.num_free == 8 and mgr.refcount == {}


def test_append_grows_one_block_at_boundary():
    mgr = BlockManager(16, 4)
    s = Sequence(mgr, 3)
    assert len(s.block_table) == 1
    slot, cow = s.append_token()          # position 3 fills block 0
    assert cow is None and len(s.block_table) == 1 and slot == s.block_table[0] * 4 + 3
    slot, cow = s.append_token()          # position 4 needs a second block
    assert cow is None and len(s.block_table) == 2 and slot == s.block_table[1] * 4
    empty = Sequence(mgr, 0)
    assert empty.block_table == []
    slot, _ = empty.append_token()
    assert len(empty.block_table) == 1 and slot == empty.block_table[0] * 4


def test_failed_append_leaves_sequence():
    mgr = BlockManager(1, 4)
    s = Sequence(mgr, 4)
    with pytest.raises(OutOfBlocks):
        s.append_token()
    assert s.length == 4 and len(s.block_table) == 1


def test_sharing_example_n4():
    """Tutorial §5 'Copy-on-write sharing': 3 shared prompt blocks + 1 private
    block per completion = 7 physical blocks instead of 16; refcount 4."""
    g = _load("kv_memory_accounting.json")["sharing_n4"]
    bs = 16
    mgr = BlockManager(32, bs, list(np.random.default_rng(0).permutation(32)))
    root = Sequence(mgr, g["prompt_blocks"] * bs)
    samples = [root] + [root.fork() for _ in range(g["samples"] - 1)]
    for s in samples:
        for _ in range(g["private_blocks"] * bs):
            _, cow = s.append_token()
            assert cow is None                 # block-aligned prompt: no CoW
    prompt = root.block_table[:g["prompt_blocks"]]
    assert all(mgr.refcount[b] == g["samples"] for b in prompt)
    assert mgr.num_used == g["with_sharing"]
    w, wo = accounting.shared_sampling_blocks(g["prompt_blocks"], g["samples"],
                                              g["private_blocks"])
    assert (w, wo) == (g["with_sharing"], g["without_sharing"])
    assert round(100 * (1 - w / wo)) == g["saved_percent_rounded"]
    check_invariants(mgr, [s.block_table for s in samples])


def test_beam_search_block_count():
    """subroutine-cs §3: beams over a shared prompt need about prompt blocks +
    K x generation blocks (exactly, when the prompt is block-aligned)."""
    bs, K, prompt_blocks, gen_blocks = 8, 4, 5, 3
    mgr = BlockManager(64, bs)
    root = Sequence(mgr, prompt_blocks * bs)
    beams = [root] + [root.fork() for _ in range(K - 1)]
    for s in beams:
        for _ in range(gen_blocks * bs):
            s.append_token()
    assert mgr.num_used == accounting.beam_search_blocks(prompt_blocks, K, gen_blocks)


def test_copy_on_write_of_partial_shared_block():
    """A token appended into a shared, partly filled block triggers a copy;
    the last holder writes in place."""
    bs = 4
    mgr = BlockManager(16, bs)
    root = Sequence(mgr, 6)                  # block 1 holds 2 of 4 slots
    kids = [root.fork(), root.fork()]
    shared_last = root.block_table[1]
    slot, cow = kids[0].append_token()
    assert cow[0] == shared_last and cow[1] == kids[0].block_table[1] != shared_last
    assert slot == cow[1] * bs + 2
    assert mgr.refcount[shared_last] == 2
    _, cow = kids[1].append_token()
    assert cow is not None and mgr.refcount[shared_last] == 1
    slot, cow = root.append_token()          # last holder: in place
    assert cow is None and slot == shared_last * bs + 2
    assert mgr.refcount[root.block_table[0]] == 3   # full prompt block stays shared
    check_invariants(mgr, [root.block_table] + [k.block_table for k in kids])


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_internal_fragmentation_is_half_a_block(bs):
    """Tutorial §5 'Block size': the last block wastes about bs/2 slots on average."""
    lens = np.random.default_rng(bs).integers(1, 100_000, size=200_000)
    waste = np.array([accounting.wasted_slots(int(L), bs) for L in lens])
    mgr = BlockManager(1, bs)
    assert all(mgr.blocks_needed(int(L)) * bs - int(L) == w for L, w in zip(lens[:2000], waste))
    assert abs(waste.mean() - (bs - 1) / 2) < 0.02 * bs


def test_memory_accounting():
    g = _load("kv_memory_accounting.json")
    m = g["llama3_8b"]
    per_tok = accounting.kv_bytes_per_token(m["layers"], m["kv_heads"], m["head_dim"],
                                            m["elem_bytes"])
    assert per_tok == m["bytes_per_token"]
    blk = accounting.kv_block_bytes(m["layers"], m["kv_heads"], m["head_dim"],
                                    m["block_size"], m["elem_bytes"])
    assert blk == m["block_bytes"]
    p = g["startup_pool"]
    nblk = accounting.pool_blocks(int(p["pool_gib"] * 2**30), blk)
    assert nblk == p["blocks"] and nblk * m["block_size"] == p["tokens"]
    x = g["llama3_70b_as_printed"]
    b70 = accounting.kv_bytes_per_token(x["layers"], x["heads"], x["head_dim"], x["elem_bytes"])
    assert b70 == x["bytes_per_token"]
    assert round(b70 / 1e6, 2) == x["bytes_per_token_mb_rounded"]
    assert round(b70 * x["context"] / 1e9, 1) == x["context_gb_rounded"]


def test_invariants_catch_a_leak():
    mgr = BlockManager(8, 4)
    s = Sequence(mgr, 8)
    mgr.refcount[s.block_table[0]] += 1      # a leaked reference
    with pytest.raises(AssertionError):
        check_invariants(mgr, [s.block_table])
