"""Seeded synthetic inputs for paged decode attention.

This module is shared by the tests, the benchmark and the oracle's checks.  It
only draws random numbers and lays out raw storage bits: sequence lengths,
query/key/value values (drawn in fp32 from N(0, 1) and rounded to fp16 or bf16
storage bits), shuffled free-block orders and NaN poison patterns.  It holds
none of the attention, address-translation, cache-write or block-copy
arithmetic; those live, separately, in the CUDA library and in the oracle.

The workload shapes follow the five decode workloads this library is
measured on (tiny, Llama-3-8B-shaped, shared prefix, long context, ragged
continuous-batching step).  The sequence-length mixes follow the pages:
uniform ranges for the fixed-batch workloads, and a lognormal length mix for
the continuous-batching step (the simulator exercise of the Paged Attention
tutorial, §10 "Hands-on exercise", draws request lengths from a lognormal).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

# Storage dtype codes, identical to the C ABI's pa_dtype enumeration.
FLOAT16 = 0
BFLOAT16 = 1
DTYPE_NAMES = {FLOAT16: "f16", BFLOAT16: "bf16"}

# Quiet-NaN bit patterns used to poison unused slots and unused blocks.
NAN_BITS = {FLOAT16: 0x7E00, BFLOAT16: 0x7FC0}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and length distribution of one synthetic decode workload."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: int
    seed: int
    # length distribution: "fixed" (lens), "uniform" (lo..hi inclusive),
    # "lognormal" (median, sigma, clipped to lo..hi), "shared_prefix"
    length_kind: str
    lens: tuple = ()
    lo: int = 1
    hi: int = 1
    median: float = 0.0
    sigma: float = 0.0
    num_blocks: int = 0          # 0: pool_factor x the blocks the batch needs
    pool_factor: float = 1.25
    partition_tokens: int = 512
    # shared-prefix workload
    num_prompts: int = 0
    samples_per_prompt: int = 0
    prefix_tokens: int = 0
    prefix_jitter: int = 0       # extra prompt tokens drawn from U{0..jitter}
    tail_lo: int = 0
    tail_hi: int = 0
    # prefill workloads: query tokens per sequence, "" (decode: one), "full"
    # (the whole prompt) or "chunk" (the last min(L, chunk) tokens)
    prefill: str = ""
    chunk: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(head_dim), as the fp32 value a kernel receives."""
        return float(np.float32(1.0 / math.sqrt(self.head_dim)))

    @property
    def elem_bytes(self) -> int:
        return 2

    def with_block_size(self, bs: int) -> "Workload":
        return dataclasses.replace(self, block_size=bs, name=f"{self.name}_bs{bs}")


TINY = Workload(
    name="tiny", num_seqs=4, num_q_heads=4, num_kv_heads=4, head_dim=64,
    block_size=16, dtype=FLOAT16, seed=0, length_kind="fixed",
    lens=(5, 16, 37, 64), num_blocks=32)

LLAMA3_8B = Workload(
    name="llama3_8b", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=1, length_kind="uniform", lo=128, hi=4096)

SHARED_PREFIX = Workload(
    name="shared_prefix", num_seqs=128, num_q_heads=32, num_kv_heads=8,
    head_dim=128, block_size=16, dtype=BFLOAT16, seed=2, length_kind="shared_prefix",
    num_prompts=16, samples_per_prompt=8, prefix_tokens=2048, prefix_jitter=15,
    tail_lo=0, tail_hi=512)

LONG_CONTEXT = Workload(
    name="long_context", num_seqs=8, num_q_heads=64, num_kv_heads=8, head_dim=128,
    block_size=32, dtype=BFLOAT16, seed=3, length_kind="uniform", lo=32768, hi=131072)

RAGGED = Workload(
    name="ragged", num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=4, length_kind="lognormal",
    median=512.0, sigma=1.0, lo=1, hi=8192)

RAGGED_BLOCK_SIZES = (8, 16, 32, 64)

# Plain multi-head attention (Llama-2-7B-shaped: 32 query heads, 32 KV heads).
MHA_7B = Workload(
    name="mha_7b", num_seqs=64, num_q_heads=32, num_kv_heads=32, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=7, length_kind="uniform", lo=128, hi=4096)

# Llama-3-405B-shaped decode: 128 query heads over 8 KV heads (16 per group).
LLAMA3_405B = Workload(
    name="llama3_405b", num_seqs=64, num_q_heads=128, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=8, length_kind="uniform", lo=128, hi=4096)

# Five query heads per KV head (Qwen2.5-32B's 40 query / 8 KV heads), the
# Llama-3-8B-shaped lengths.
QWEN25_32B = Workload(
    name="qwen25_32b", num_seqs=64, num_q_heads=40, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=10, length_kind="uniform", lo=128, hi=4096)

# Continuous batching with many live requests: 2048 sequences of U[16, 1024] tokens.
MANY_SEQS = Workload(
    name="many_seqs", num_seqs=2048, num_q_heads=32, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=9, length_kind="uniform", lo=16, hi=1024)

# Prefill: whole prompts of U[512, 4096] tokens; chunked prefill: the last 512
# tokens of sequences of U[1024, 8192] tokens whose earlier tokens are cached.
PREFILL = Workload(
    name="prefill", num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=5, length_kind="uniform", lo=512, hi=4096,
    prefill="full")

# The whole-prompt batch with 40 query / 8 KV heads (Qwen2.5-32B-shaped).
PREFILL_QWEN = Workload(
    name="prefill_qwen25_32b", num_seqs=8, num_q_heads=40, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=5, length_kind="uniform", lo=512, hi=4096,
    prefill="full")

CHUNKED_PREFILL = Workload(
    name="chunked_prefill", num_seqs=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
    block_size=16, dtype=BFLOAT16, seed=6, length_kind="uniform", lo=1024, hi=8192,
    prefill="chunk", chunk=512)

WORKLOADS = {w.name: w for w in (TINY, LLAMA3_8B, SHARED_PREFIX, LONG_CONTEXT, RAGGED,
                                  PREFILL, CHUNKED_PREFILL, MHA_7B, LLAMA3_405B, MANY_SEQS,
                                  QWEN25_32B, PREFILL_QWEN)}


# ----------------------------------------------------------------------------
# random streams
# ----------------------------------------------------------------------------

_STREAMS = {"lens": 1, "values": 2, "free": 3, "query": 4, "new_kv": 5, "tails": 6,
            "prefill_query": 7}


def rng(w: Workload, stream: str, sub: int = 0) -> np.random.Generator:
    """Independent PCG64 stream per (workload seed, purpose, sub-index)."""
    return np.random.default_rng([w.seed, _STREAMS[stream], sub])


def seq_lens(w: Workload) -> np.ndarray:
    """Draw the per-sequence context lengths of a fixed-batch workload."""
    g = rng(w, "lens")
    if w.length_kind == "fixed":
        return np.asarray(w.lens, dtype=np.int64)
    if w.length_kind == "uniform":
        return g.integers(w.lo, w.hi + 1, size=w.num_seqs, dtype=np.int64)
    if w.length_kind == "lognormal":
        z = g.standard_normal(w.num_seqs)
        raw = np.rint(np.exp(math.log(w.median) + w.sigma * z))
        return np.clip(raw, w.lo, w.hi).astype(np.int64)
    raise ValueError(f"{w.name}: lengths of kind {w.length_kind!r} are drawn per prompt")


def prompt_extra_tokens(w: Workload) -> np.ndarray:
    """Shared-prefix workload: extra prompt tokens k_p ~ U{0..jitter} per prompt."""
    return rng(w, "lens").integers(0, w.prefix_jitter + 1, size=w.num_prompts, dtype=np.int64)


def sample_tail_lens(w: Workload) -> np.ndarray:
    """Shared-prefix workload: generated tokens per sample, U{tail_lo..tail_hi}."""
    return rng(w, "tails").integers(
        w.tail_lo, w.tail_hi + 1, size=(w.num_prompts, w.samples_per_prompt), dtype=np.int64)


def shuffled_free_order(num_blocks: int, g: np.random.Generator) -> list:
    """A seeded permutation of the block ids [0, num_blocks), used as the
    initial free stack so that allocations come out scattered."""
    return [int(x) for x in g.permutation(num_blocks)]


# ----------------------------------------------------------------------------
# storage bits
# ----------------------------------------------------------------------------

def fp32_to_storage_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp32 values to fp16/bf16 (round to nearest even) and return the
    raw 16-bit patterns as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == FLOAT16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BFLOAT16:
        u = x.view(np.uint32)
        nan = np.isnan(x)
        # finite values and infinities stay below 2^32 after the bias
        safe = np.where(nan, np.uint32(0), u)
        bits = ((safe + np.uint32(0x7FFF) + ((safe >> 16) & np.uint32(1))) >> 16).astype(np.uint16)
        if nan.any():
            bits[nan] = NAN_BITS[BFLOAT16]
        return bits
    raise ValueError(f"unknown dtype code {dtype}")


def normal_bits(g: np.random.Generator, shape: Sequence[int], dtype: int) -> np.ndarray:
    """N(0, 1) values drawn in fp32 and rounded to storage bits."""
    return fp32_to_storage_bits(g.standard_normal(size=tuple(shape), dtype=np.float32), dtype)


def nan_bits(shape: Sequence[int], dtype: int) -> np.ndarray:
    return np.full(tuple(shape), NAN_BITS[dtype], dtype=np.uint16)


def query_bits(w: Workload, num_seqs: Optional[int] = None, sub: int = 0) -> np.ndarray:
    b = w.num_seqs if num_seqs is None else num_seqs
    return normal_bits(rng(w, "query", sub), (b, w.num_q_heads, w.head_dim), w.dtype)


def token_kv_bits(w: Workload, num_tokens: int, sub: int) -> tuple:
    """K and V storage bits for `num_tokens` tokens: two [T, Hkv, D] uint16 arrays."""
    g = rng(w, "values", sub)
    shape = (num_tokens, w.num_kv_heads, w.head_dim)
    return normal_bits(g, shape, w.dtype), normal_bits(g, shape, w.dtype)


def pool_fill_bits(w: Workload, num_blocks: int, sub: int = 0, chunk_blocks: int = 4096) -> tuple:
    """A whole pool of random K and V bits, [NB, bs, Hkv, D] each (used where the
    values of every slot are random data rather than specific tokens).  Drawn in
    chunks of blocks to bound host memory."""
    g = rng(w, "values", 10_000 + sub)
    shape = (num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    k = np.empty(shape, dtype=np.uint16)
    v = np.empty(shape, dtype=np.uint16)
    for lo in range(0, num_blocks, chunk_blocks):
        hi = min(num_blocks, lo + chunk_blocks)
        k[lo:hi] = normal_bits(g, (hi - lo,) + shape[1:], w.dtype)
        v[lo:hi] = normal_bits(g, (hi - lo,) + shape[1:], w.dtype)
    return k, v


# ----------------------------------------------------------------------------
# request streams for the allocator simulator
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class RequestStream:
    """A serving request stream: Poisson arrivals (exponential gaps, counted in
    decode steps) and lognormal prompt and output lengths (the tutorial's
    simulator exercise, §10 B).  Lengths are clipped so that prompt + output
    never exceeds max_seq_len."""

    name: str
    seed: int
    num_requests: int
    rate: float                  # mean arrivals per decode step
    prompt_median: float
    prompt_sigma: float
    output_median: float
    output_sigma: float
    max_seq_len: int


SERVING_STREAM = RequestStream(
    name="serving", seed=11, num_requests=4000, rate=4.0, prompt_median=256.0,
    prompt_sigma=1.0, output_median=128.0, output_sigma=1.0, max_seq_len=2048)

SMALL_STREAM = RequestStream(
    name="small", seed=12, num_requests=300, rate=2.0, prompt_median=40.0, prompt_sigma=1.0,
    output_median=24.0, output_sigma=0.8, max_seq_len=256)


def request_arrays(s: RequestStream) -> tuple:
    """(arrival_step, prompt_len, output_len), int32 arrays of num_requests,
    arrival steps non-decreasing; prompt >= 1, output >= 1, sum <= max_seq_len."""
    g = np.random.default_rng([s.seed, 7])
    gaps = g.exponential(1.0 / s.rate, size=s.num_requests)
    arrival = np.floor(np.cumsum(gaps)).astype(np.int64)
    p = np.rint(np.exp(math.log(s.prompt_median) + s.prompt_sigma * g.standard_normal(s.num_requests)))
    o = np.rint(np.exp(math.log(s.output_median) + s.output_sigma * g.standard_normal(s.num_requests)))
    p = np.clip(p, 1, s.max_seq_len - 1).astype(np.int64)
    o = np.clip(o, 1, None).astype(np.int64)
    o = np.minimum(o, s.max_seq_len - p)
    return arrival.astype(np.int32), p.astype(np.int32), o.astype(np.int32)


def query_counts(w: Workload, lens) -> np.ndarray:
    """Query tokens per sequence of a prefill workload."""
    lens = np.asarray(lens, dtype=np.int64)
    if w.prefill == "full":
        return lens.copy()
    if w.prefill == "chunk":
        return np.minimum(lens, w.chunk)
    return np.minimum(lens, 1)


def prefill_query_bits(w: Workload, total_q: int, sub: int = 0) -> np.ndarray:
    """Queries of a prefill batch, [total_q, Hq, D] storage bits."""
    return normal_bits(rng(w, "prefill_query", sub), (total_q, w.num_q_heads, w.head_dim),
                       w.dtype)
