"""Prefix caching over the refcounted block manager (oracle side; test
infrastructure, imported only by the tests and the benchmark's CPU legs).

The "10 — Paged Attention" tutorial, §5 "The relationship to prefix caching":
once KV lives in shareable refcounted blocks, a prefix cache is a map from a
hash of each block's token ids to the block holding their KV; a new sequence
whose first blocks hash to cached blocks points its table at them and raises
their refcounts instead of computing them again.  Exercise A of §10 adds
eviction to the same manager.

Readings where the pages leave the details open (each listed in the design
notes):

* Key of a block.  The KV of a token depends on every token before it, so the
  key of full block i covers the whole prefix: key_i = FNV-1a-64 over
  (key_{i-1} as 8 little-endian bytes, then the block's token ids as 4-byte
  little-endian two's-complement integers), key_{-1} = 0.  FNV-1a-64 is the
  published Fowler-Noll-Vo hash (offset basis 0xcbf29ce484222325, prime
  0x100000001b3).  A hit also compares the stored parent key and token ids, so
  a false hit needs a 64-bit collision of the preceding prefix.
* Only full blocks are cached; a partly filled last block is private.  Blocks
  are registered when the sequence is created; the caller computes the KV of
  the tokens past the cached prefix before anything reads them.
* Lookup stops at the first miss: the KV of later blocks has to be recomputed
  anyway, because computing it needs the model state over the missed block.
  A key already cached (by a block that outlived the eviction of an earlier
  block of its prefix) is not registered a second time.
* A cached block whose refcount drops to zero is not freed: it waits on an
  eviction queue and can still be hit.  Blocks reaching zero in one release
  join the queue last block first, so the end of a prefix goes before its
  beginning.  Allocation takes free blocks first (the Go stack rule); when the
  stack is short, it evicts queue entries from the front (dropping their keys)
  and pushes them on the stack, then takes as usual.  A hit on a queued block
  takes it off the queue with refcount 1.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Sequence as Seq, Tuple

from .block_manager import BlockManager, BlockStateError, OutOfBlocks, Sequence

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
_MASK = (1 << 64) - 1


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & _MASK
    return h


def block_key(parent: int, tokens: Seq[int]) -> int:
    data = parent.to_bytes(8, "little") + b"".join(
        int(t).to_bytes(4, "little", signed=True) for t in tokens)
    return fnv1a64(data)


class PrefixCachingBlockManager(BlockManager):
    def __init__(self, num_blocks: int, block_size: int, free_stack=None):
        super().__init__(num_blocks, block_size, free_stack)
        self.entry: Dict[int, Tuple[int, int, Tuple[int, ...]]] = {}   # block -> (key, parent, tokens)
        self.block_of: Dict[int, int] = {}                              # key -> block
        self.evictable: List[int] = []                                  # front is evicted first

    # -- allocation with eviction -------------------------------------------
    def allocate(self, n: int) -> List[int]:
        if n < 0:
            raise ValueError("n must be >= 0")
        if len(self.free) + len(self.evictable) < n:
            raise OutOfBlocks(f"no free KV block left: need {n}, have "
                              f"{len(self.free)} free + {len(self.evictable)} evictable")
        while len(self.free) < n:
            b = self.evictable.pop(0)
            key = self.entry.pop(b)[0]
            del self.block_of[key]
            self.free.append(b)
        return super().allocate(n)

    def free_blocks(self, blocks: Iterable[int]) -> None:
        blocks = list(blocks)
        uses: Dict[int, int] = {}
        for b in blocks:
            uses[b] = uses.get(b, 0) + 1
            if uses[b] > self.refcount.get(b, 0):
                raise BlockStateError(f"block {b} freed while unreferenced")
        parked = []
        for b in blocks:
            count = self.refcount[b]
            if count == 1:
                del self.refcount[b]
                if b in self.entry:
                    parked.append(b)
                else:
                    self.free.append(b)
            else:
                self.refcount[b] = count - 1
        self.evictable.extend(reversed(parked))

    # -- the cache -----------------------------------------------------------
    def prompt_keys(self, tokens: Seq[int]) -> List[Tuple[int, int, Tuple[int, ...]]]:
        bs = self.block_size
        out, parent = [], 0
        for i in range(len(tokens) // bs):
            blk = tuple(int(t) for t in tokens[i * bs:(i + 1) * bs])
            k = block_key(parent, blk)
            out.append((k, parent, blk))
            parent = k
        return out

    def create_sequence(self, tokens: Seq[int]) -> Tuple[Sequence, int]:
        """A sequence holding `tokens`; returns it and the number of leading
        tokens whose KV is already in cached blocks (a multiple of block_size)."""
        keys = self.prompt_keys(tokens)
        hits: List[int] = []
        for k, parent, blk in keys:
            b = self.block_of.get(k)
            if b is None or self.entry[b][1:] != (parent, blk):
                break
            hits.append(b)
        need = self.blocks_needed(len(tokens)) - len(hits)
        queued = [b for b in hits if b not in self.refcount]
        if len(self.free) + len(self.evictable) - len(queued) < need:
            raise OutOfBlocks(f"no free KV block left: need {need} beyond the cached prefix")
        for b in hits:
            if b in self.refcount:
                self.refcount[b] += 1
            else:
                self.evictable.remove(b)
                self.refcount[b] = 1
        table = hits + self.allocate(need)
        for i in range(len(hits), len(keys)):
            k = keys[i][0]
            if k not in self.block_of:
                self.block_of[k] = table[i]
                self.entry[table[i]] = keys[i]
        return Sequence(self, len(tokens), table), len(hits) * self.block_size

    @property
    def num_evictable(self) -> int:
        return len(self.evictable)


def check_cache_invariants(mgr: PrefixCachingBlockManager, tables: Iterable[List[int]]) -> None:
    """Free, referenced and queued ids partition the pool; refcounts equal the
    table references; every queued block is cached; the key map and the block
    entries agree."""
    free, queued, used = set(mgr.free), set(mgr.evictable), set(mgr.refcount)
    if len(free) != len(mgr.free) or len(queued) != len(mgr.evictable):
        raise AssertionError("duplicate id on the free stack or the eviction queue")
    if free & queued or free & used or queued & used:
        raise AssertionError("a block is in two of free / queued / referenced")
    if free | queued | used != set(range(mgr.num_blocks)):
        raise AssertionError("free, queued and referenced blocks do not cover the pool")
    refs: Dict[int, int] = {}
    for t in tables:
        for b in t:
            refs[b] = refs.get(b, 0) + 1
    if refs != mgr.refcount:
        raise AssertionError(f"refcounts {mgr.refcount} != table references {refs}")
    if not queued <= set(mgr.entry):
        raise AssertionError("an uncached block waits for eviction")
    if free & set(mgr.entry):
        raise AssertionError("a free block still has a cache entry")
    for b, (k, _, _) in mgr.entry.items():
        if mgr.block_of.get(k) != b:
            raise AssertionError(f"key map and entry of block {b} disagree")
    if len(mgr.block_of) != len(mgr.entry):
        raise AssertionError("key map and entries differ in size")
