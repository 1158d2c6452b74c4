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

Both work on raw uint16 storage bits, so results are exact bit copies.
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
