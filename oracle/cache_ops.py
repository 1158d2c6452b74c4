"""Byte-exact cache write and block copy (oracle side).

reshape_and_cache: each new token's key and value rows ([Hkv, D] each) are
stored at pool slot slot_mapping[i]; the slot is the tutorial's PhysicalIndex of
the token's position ("10 — Paged Attention" §4 "Tiny example"), so slot s is
row s % bs of physical block s // bs.  A negative slot marks a padding token that
is skipped.

copy_blocks: the copy-on-write clone of a shared block — when a shared block
must be written, it is copied first ("10 — Paged Attention" §5 "Copy-on-write
sharing"; subroutine-cs article §3 "Copy-on-Write and Parallel Sampling").  Every
slot of the source block (all bs rows, all KV heads) is copied to the
destination block, for keys and for values.

copy_blocks_multi: the same clone in every pool a model keeps, one K and one V
pool per layer (subroutine-cs article §1, the bytes-per-token formula counts
2 x layers x heads x head_dim elements per token).

swap_blocks: blocks moved between two sets of pools, e.g. from the GPU pools to
pools in CPU RAM and back (PagedAttention glossary page, allocation and eviction:
evicted blocks can move to host memory).  Block dst of the destination pool i receives
block src of the source pool i.

All work on raw uint16 storage bits, so results are exact bit copies.
"""
from __future__ import annotations

import numpy as np


def reshape_and_cache(k_pool: np.ndarray, v_pool: np.ndarray, key: np.ndarray,
                      value: np.ndarray, slot_mapping) -> None:
    """In place.  k_pool/v_pool [NB, bs, Hkv, D] uint16; key/value [T, Hkv, D]."""
    NB, bs = k_pool.shape[:2]
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, row = divmod(int(slot), bs)
        if blk >= NB:
            raise IndexError(f"slot {slot} outside a pool of {NB} blocks")
        k_pool[blk, row] = key[i]
        v_pool[blk, row] = value[i]


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs) -> None:
    """In place.  pairs: iterable of (src, dst) block ids, applied in order."""
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        k_pool[dst] = k_pool[src]
        v_pool[dst] = v_pool[src]


def copy_blocks_multi(pools, pairs) -> None:
    """In place.  pools: sequence of [NB, ...] arrays (K and V of every layer);
    every (src, dst) pair is applied, in order, to every pool."""
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist()
    for pool in pools:
        for src, dst in pairs:
            pool[dst] = pool[src]


def swap_blocks(dst_pools, src_pools, pairs) -> None:
    """In place on dst_pools.  pairs: (src id in src_pools, dst id in dst_pools)."""
    if len(dst_pools) != len(src_pools):
        raise ValueError("one destination pool per source pool")
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist()
    for dst_pool, src_pool in zip(dst_pools, src_pools):
        if dst_pool.shape[1:] != src_pool.shape[1:]:
            raise ValueError("source and destination blocks differ in shape")
        for src, dst in pairs:
            dst_pool[dst] = src_pool[src]
