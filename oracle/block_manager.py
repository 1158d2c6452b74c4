"""Refcounted KV block manager (oracle side).

Semantics follow the Go block manager of the "10 — Paged Attention" tutorial,
§4 "Tiny example":

* the free list is a stack; a new manager pushes ids from num_blocks-1 down to
  0, so block 0 is on top;
* allocating n blocks takes the top n entries of the stack, in the order they
  sit in the stack (bottom-most of the n first), and gives each refcount 1; if
  fewer than n are free the call fails and nothing changes;
* freeing decrements each block's refcount and pushes the block back on the
  stack when the count reaches zero;
* forking increments the refcount of every block of a table and returns a copy
  of the table (same physical blocks, new logical sequence);
* blocks needed for t tokens is ceil(t / block_size);
* a sequence is a block table plus a length; appending a token grows the length
  and, when the length crosses a block boundary, allocates exactly one block;
* the physical slot of token `pos` is table[pos // bs] * bs + pos % bs.

Readings where the pages are silent (each listed in the design notes):

* freeing a block whose refcount is already zero, or forking a block that is not
  allocated, is an error (the Go listing would silently drive the count
  negative);
* a failed append leaves the sequence unchanged;
* copy-on-write, described in prose only (tutorial §5 "Copy-on-write sharing";
  subroutine-cs article §3 "Copy-on-Write and Parallel Sampling"): when the
  token being appended lands in a block whose refcount is above one, a fresh
  block is allocated, the pair (old, new) is recorded for a whole-block copy,
  the old block's refcount drops by one, the table entry is swapped, and only
  then is the token written.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Tuple


class OutOfBlocks(RuntimeError):
    """The free pool holds fewer blocks than requested (the Go ErrNoBlocks)."""


class BlockStateError(RuntimeError):
    """Free of an unreferenced block, or fork of a block that is not allocated."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int,
                 free_stack: Optional[Iterable[int]] = None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("num_blocks must be >= 0 and block_size > 0")
        self.num_blocks = num_blocks
        self.block_size = block_size
        if free_stack is None:
            # pushed from the highest id down, so id 0 ends on top
            stack = [num_blocks - 1 - i for i in range(num_blocks)]
        else:
            stack = [int(b) for b in free_stack]
            if sorted(stack) != list(range(num_blocks)):
                raise ValueError("free_stack must be a permutation of range(num_blocks)")
        self.free: List[int] = stack          # top of the stack is the end
        self.refcount: Dict[int, int] = {}

    # -- pool operations ---------------------------------------------------
    def allocate(self, n: int) -> List[int]:
        if n < 0:
            raise ValueError("n must be >= 0")
        have = len(self.free)
        if have < n:
            raise OutOfBlocks(f"no free KV block left: need {n}, have {have}")
        cut = have - n
        taken = self.free[cut:]
        self.free = self.free[:cut]
        for b in taken:
            self.refcount[b] = 1
        return taken

    def free_blocks(self, blocks: Iterable[int]) -> None:
        for b in blocks:
            count = self.refcount.get(b, 0)
            if count <= 0:
                raise BlockStateError(f"block {b} freed while unreferenced")
            if count == 1:
                del self.refcount[b]
                self.free.append(b)
            else:
                self.refcount[b] = count - 1

    def fork(self, blocks: Iterable[int]) -> List[int]:
        blocks = list(blocks)
        for b in blocks:
            if self.refcount.get(b, 0) <= 0:
                raise BlockStateError(f"block {b} forked while not allocated")
        for b in blocks:
            self.refcount[b] += 1
        return list(blocks)

    def blocks_needed(self, tokens: int) -> int:
        return -(-tokens // self.block_size)

    # -- statistics (pool utilisation is the signal to monitor, tutorial §8) --
    @property
    def num_free(self) -> int:
        return len(self.free)

    @property
    def num_used(self) -> int:
        return len(self.refcount)

    def utilisation(self) -> float:
        return self.num_used / self.num_blocks if self.num_blocks else 0.0


class Sequence:
    """Block table + length of one logical sequence."""

    def __init__(self, mgr: BlockManager, prompt_len: int,
                 table: Optional[List[int]] = None):
        self.mgr = mgr
        if table is None:
            table = mgr.allocate(mgr.blocks_needed(prompt_len))
        self.block_table: List[int] = table
        self.length = prompt_len

    def physical_index(self, pos: int) -> int:
        """Slot of token `pos` in the pool: a page-table walk, (page -> frame) *
        page size + offset (tutorial §4, PhysicalIndex)."""
        if not 0 <= pos < len(self.block_table) * self.mgr.block_size:
            raise IndexError(f"position {pos} outside the block table")
        bs = self.mgr.block_size
        return self.block_table[pos // bs] * bs + pos % bs

    def append_token(self) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Grow by one token.  Returns (slot of the new token, CoW pair or None).

        Allocates one block when the new length needs one more block; if instead
        the token lands in a shared block, performs copy-on-write first."""
        mgr = self.mgr
        pos = self.length
        new_len = pos + 1
        cow: Optional[Tuple[int, int]] = None
        if mgr.blocks_needed(new_len) > len(self.block_table):
            self.block_table.append(mgr.allocate(1)[0])
        else:
            idx = pos // mgr.block_size
            old = self.block_table[idx]
            if mgr.refcount[old] > 1:
                new = mgr.allocate(1)[0]
                mgr.free_blocks([old])
                self.block_table[idx] = new
                cow = (old, new)
        self.length = new_len
        return self.physical_index(pos), cow

    def fork(self) -> "Sequence":
        return Sequence(self.mgr, self.length, self.mgr.fork(self.block_table))

    def release(self) -> None:
        self.mgr.free_blocks(self.block_table)
        self.block_table = []
        self.length = 0


def check_invariants(mgr: BlockManager, tables: Iterable[List[int]]) -> None:
    """Pool invariants: free and used ids partition [0, NB); each used block's
    refcount equals the number of table entries that reference it."""
    free = mgr.free
    if len(set(free)) != len(free):
        raise AssertionError("duplicate id on the free stack")
    used = set(mgr.refcount)
    if used & set(free):
        raise AssertionError("block both free and referenced")
    if used | set(free) != set(range(mgr.num_blocks)):
        raise AssertionError("free and used blocks do not cover the pool")
    refs: Dict[int, int] = {}
    for t in tables:
        for b in t:
            refs[b] = refs.get(b, 0) + 1
    if refs != mgr.refcount:
        raise AssertionError(f"refcounts {mgr.refcount} != table references {refs}")
