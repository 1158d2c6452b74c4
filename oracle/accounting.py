"""KV-cache byte arithmetic (oracle side).

* Bytes per token of a model's KV cache: keys and values (factor 2), times the
  element size, layers, KV heads and head_dim (subroutine-cs article §1 "The GPU
  Memory Crisis", stated there for FP16 with the head count H; with grouped-query
  attention the count that is stored is the KV-head count).
* Block bytes: bytes per token times block_size ("10 — Paged Attention" §5, block
  size; §6 "Under the hood", the startup accounting).
* Sharing: n samples of one prompt keep one copy of the prompt blocks plus the
  private blocks of each sample (tutorial §5 "Copy-on-write sharing"); beam search
  needs about prompt blocks + K x generation blocks (subroutine-cs article §3).
* Expected internal fragmentation: with lengths spread evenly over block
  residues, the last block is on average half empty (tutorial §5 "Block size").
"""
from __future__ import annotations


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    return 2 * elem_bytes * layers * kv_heads * head_dim


def kv_block_bytes(layers: int, kv_heads: int, head_dim: int, block_size: int,
                   elem_bytes: int = 2) -> int:
    return kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes) * block_size


def pool_blocks(pool_bytes: int, block_bytes: int) -> int:
    """Whole blocks that fit in a pool of pool_bytes."""
    return pool_bytes // block_bytes


def shared_sampling_blocks(prompt_blocks: int, samples: int, private_blocks: int) -> tuple:
    """(blocks with sharing, blocks without sharing) for `samples` completions of
    one prompt, each adding `private_blocks` blocks of its own."""
    with_sharing = prompt_blocks + samples * private_blocks
    without = samples * (prompt_blocks + private_blocks)
    return with_sharing, without


def beam_search_blocks(prompt_blocks: int, beams: int, generation_blocks: int) -> int:
    return prompt_blocks + beams * generation_blocks


def wasted_slots(length: int, block_size: int) -> int:
    """Unused slots in the last block of a sequence of `length` tokens."""
    return (-length) % block_size
