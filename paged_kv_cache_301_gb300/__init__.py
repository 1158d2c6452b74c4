"""PagedAttention decode for GB300 — thin Python binding over libpagedattn.

Argument marshalling only: every computation runs in the library's CUDA
kernels (or, for the block manager, its C++ host code).  Tensors are PyTorch
tensors used as device buffers; the current CUDA stream is passed through.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib

FLOAT16 = 0
BFLOAT16 = 1
_DTYPES = {torch.float16: FLOAT16, torch.bfloat16: BFLOAT16}

PA_OK = 0
DEFAULT_PARTITION_TOKENS = 512


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.load().pa_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libpagedattn must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}; use float16 or bfloat16") from None


def lib() -> ctypes.CDLL:
    return _lib.load()


def pa_decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int,
                              max_seq_len: int, partition_tokens: int = 0) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len,
                                               partition_tokens))


def alloc_workspace(num_seqs, num_q_heads, head_dim, max_seq_len, partition_tokens=0,
                    device="cuda") -> torch.Tensor:
    """A workspace large enough for any decode kernel (pa_decode_workspace_bytes)."""
    n = pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len, partition_tokens)
    if n == 0:
        raise ValueError("invalid workspace arguments")
    return torch.empty(n, dtype=torch.uint8, device=device)


def pa_decode_workspace_bytes_for(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                  head_dim: int, block_size: int, max_blocks: int,
                                  num_blocks: int, max_seq_len: int, dtype: int,
                                  partition_tokens: int = 0) -> int:
    """Bytes the decode kernel that serves these arguments needs (0: invalid)."""
    return int(lib().pa_decode_workspace_bytes_for(num_seqs, num_q_heads, num_kv_heads,
                                                   head_dim, block_size, max_blocks, num_blocks,
                                                   max_seq_len, dtype, partition_tokens))


def workspace_for(q: torch.Tensor, k_pool: torch.Tensor, block_tables: torch.Tensor,
                  max_seq_len: int, partition_tokens: int = 0,
                  strict: bool = True) -> torch.Tensor:
    """The workspace of exactly the size the decode kernel serving this call
    needs (pa_decode_workspace_bytes_for, under the current kernel selection).
    For arguments the library would reject: ValueError, or with strict=False an
    empty tensor, so that the decode call itself reports the library's status."""
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_pool.shape
    n = pa_decode_workspace_bytes_for(B, Hq, Hkv, D, bs, block_tables.shape[1], NB,
                                      int(max_seq_len), _dtype(q), partition_tokens)
    if n == 0 and strict:
        raise ValueError("invalid decode arguments")
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
              max_seq_len: Optional[int] = None, partition_tokens: int = 0,
              workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """Decode attention over a paged pool (see include/pagedattn.h, pa_decode).

    q, out [B, Hq, D]; k_pool, v_pool [NB, bs, Hkv, D]; block_tables [B, MB] int32;
    seq_lens [B] int32.  max_seq_len defaults to the table capacity MB * bs (no
    device read); workspace is allocated when not given."""
    B, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_pool.shape
    MB = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = MB * bs
    if workspace is None:
        workspace = workspace_for(q, k_pool, block_tables, max_seq_len, partition_tokens,
                                  strict=False)
    st = lib().pa_decode(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
        B, Hq, Hkv, D, bs, MB, NB, int(max_seq_len), float(scale), _dtype(q),
        int(partition_tokens), _ptr(workspace), workspace.numel(), _ptr(status),
        _stream(stream))
    _check(st, "pa_decode")
    return out


def pa_decode_append(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                     v_pool: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                     block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     max_seq_len: Optional[int] = None, partition_tokens: int = 0,
                     workspace: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step (see include/pagedattn.h, pa_decode_append): the newest
    token of every sequence (key/value [B, Hkv, D]) goes to its slot, then decode
    attention over the grown sequences, as pa_append_tokens + pa_decode."""
    B, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_pool.shape
    MB = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = MB * bs
    if workspace is None:
        workspace = workspace_for(q, k_pool, block_tables, max_seq_len, partition_tokens,
                                  strict=False)
    st = lib().pa_decode_append(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(key), _ptr(value),
        _ptr(block_tables), _ptr(seq_lens), B, Hq, Hkv, D, bs, MB, NB, int(max_seq_len),
        float(scale), _dtype(q), int(partition_tokens), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream(stream))
    _check(st, "pa_decode_append")
    return out


NOALLOC_SCRATCH_BYTES = 32 << 20


def pa_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                      v_pool: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      scale: float, max_seq_len: int, partition_tokens: int = 0,
                      status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_decode without a caller workspace, for callers that cannot allocate
    device memory when they call (see include/pagedattn.h, pa_decode_noalloc):
    the split-K scratch is a fixed 32 MiB array inside the library, shared by
    all calls, so calls must not overlap on the GPU."""
    B, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_pool.shape
    MB = block_tables.shape[1]
    st = lib().pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(seq_lens),
        B, Hq, Hkv, D, bs, MB, NB, int(max_seq_len), float(scale), _dtype(q),
        int(partition_tokens), _ptr(status), _stream(stream))
    _check(st, "pa_decode_noalloc")
    return out


DECODE_PATHS = {"auto": 0, "simt": 1, "tc": 2, "tc_head": 3}
DECODE_KERNELS = {0: "grouped", 1: "per_head", 2: "simt"}


def decode_kernel_for(q: torch.Tensor, k_pool: torch.Tensor, block_tables: torch.Tensor,
                      max_seq_len: int, partition_tokens: int = 0) -> Optional[str]:
    """Name of the decode kernel ("grouped", "per_head", "simt") that pa_decode
    runs for these arguments under the current selection; None if rejected."""
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_pool.shape
    k = lib().pa_decode_kernel_for(B, Hq, Hkv, D, bs, block_tables.shape[1], NB,
                                   int(max_seq_len), _dtype(q), partition_tokens)
    return DECODE_KERNELS.get(k)


def set_decode_path(name: str) -> None:
    """Select the decode kernel process-wide: "auto" (the grouped tensor-core
    kernel where it applies, else the per-head tensor-core kernel for head_dim
    128, else CUDA cores), "simt" (CUDA cores), "tc" (a tensor-core kernel) or
    "tc_head" (the per-head tensor-core kernel)."""
    _check(lib().pa_set_decode_path(DECODE_PATHS[name]), "pa_set_decode_path")


def pa_reshape_and_cache(k_pool: torch.Tensor, v_pool: torch.Tensor, key: torch.Tensor,
                         value: torch.Tensor, slot_mapping: torch.Tensor,
                         status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Store new tokens' K/V ([T, Hkv, D]) at pool slots slot_mapping[T] (int32)."""
    NB, bs, Hkv, D = k_pool.shape
    T = key.shape[0]
    st = lib().pa_reshape_and_cache(
        _ptr(k_pool), _ptr(v_pool), _ptr(key), _ptr(value), _ptr(slot_mapping), T, 0,
        Hkv, D, bs, NB, _dtype(k_pool), _ptr(status), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_copy_blocks(k_pool: torch.Tensor, v_pool: torch.Tensor, block_pairs: torch.Tensor,
                   status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy-on-write block clones; block_pairs [n, 2] int32 (src, dst)."""
    NB, bs, Hkv, D = k_pool.shape
    n = block_pairs.shape[0] if block_pairs.numel() else 0
    st = lib().pa_copy_blocks(
        _ptr(k_pool), _ptr(v_pool), _ptr(block_pairs) if n else None, n, Hkv, D, bs, NB,
        _dtype(k_pool), _ptr(status), _stream(stream))
    _check(st, "pa_copy_blocks")


def _pool_array(pools: Sequence[torch.Tensor], what: str):
    """(ctypes array of the pools' addresses, blocks per pool, bytes per block)."""
    if not pools:
        raise ValueError(f"{what}: no pools")
    first = pools[0]
    for t in pools:
        if t.shape != first.shape or t.dtype != first.dtype:
            raise ValueError(f"{what}: every pool needs the same shape and dtype")
    arr = (ctypes.c_void_p * len(pools))(*[_ptr(t) for t in pools])
    nb = first.shape[0]
    return arr, nb, first[0].numel() * first.element_size()


def pa_copy_blocks_multi(pools: Sequence[torch.Tensor], block_pairs: torch.Tensor,
                         status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy-on-write clones in every pool (the K and V pools of all layers) in
    one launch; block_pairs [n, 2] int32 (src, dst) on the device."""
    arr, nb, block_bytes = _pool_array(pools, "pa_copy_blocks_multi")
    n = block_pairs.shape[0] if block_pairs.numel() else 0
    st = lib().pa_copy_blocks_multi(
        ctypes.cast(arr, ctypes.c_void_p), len(pools), _ptr(block_pairs) if n else None, n,
        block_bytes, nb, _ptr(status), _stream(stream))
    _check(st, "pa_copy_blocks_multi")


def pa_swap_blocks(dst_pools: Sequence[torch.Tensor], src_pools: Sequence[torch.Tensor],
                   block_pairs: torch.Tensor, status: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Block dst of dst_pools[i] = block src of src_pools[i] for every (src, dst)
    pair and pool.  Pools live on the GPU or in pinned CPU memory
    (tensor.pin_memory()); block_pairs [n, 2] int32, on the GPU or pinned."""
    if len(dst_pools) != len(src_pools):
        raise ValueError("pa_swap_blocks: one destination pool per source pool")
    darr, dnb, dbytes = _pool_array(dst_pools, "pa_swap_blocks")
    sarr, snb, sbytes = _pool_array(src_pools, "pa_swap_blocks")
    if dbytes != sbytes or dst_pools[0].dtype != src_pools[0].dtype:
        raise ValueError("pa_swap_blocks: source and destination blocks differ")
    for t in list(dst_pools) + list(src_pools) + [block_pairs]:
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("pa_swap_blocks: CPU tensors must be pinned")
    n = block_pairs.shape[0] if block_pairs.numel() else 0
    st = lib().pa_swap_blocks(
        ctypes.cast(darr, ctypes.c_void_p), ctypes.cast(sarr, ctypes.c_void_p), len(dst_pools),
        _ptr(block_pairs) if n else None, n, dbytes, snb, dnb, _ptr(status), _stream(stream))
    _check(st, "pa_swap_blocks")


def pa_decode_slots(slot_mapping: torch.Tensor, block_tables: torch.Tensor,
                    seq_lens: torch.Tensor, block_size: int, num_blocks: int,
                    status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """slot_mapping[b] = pool slot of token seq_lens[b] - 1 (or -1 for an empty
    sequence, or, reported through `status`, a bad length or block id)."""
    B, MB = block_tables.shape
    st = lib().pa_decode_slots(_ptr(slot_mapping), _ptr(block_tables), _ptr(seq_lens), B, MB,
                               block_size, num_blocks, _ptr(status), _stream(stream))
    _check(st, "pa_decode_slots")
    return slot_mapping


PREFILL_PATHS = {"auto": 0, "simt": 1, "tc": 2}


def set_prefill_path(path: str) -> None:
    """Choose pa_prefill's kernel: "auto", "simt" (CUDA cores) or "tc"."""
    _check(lib().pa_set_prefill_path(PREFILL_PATHS[path]), "pa_set_prefill_path")


def pa_prefill(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
               block_tables: torch.Tensor, seq_lens: torch.Tensor, q_start: torch.Tensor,
               scale: float, max_q_len: Optional[int] = None,
               status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal attention of each sequence's last n_b tokens (q rows q_start[b] ..
    q_start[b+1]-1) over its paged K/V.  max_q_len: host bound of n_b (computed
    from q_start, with a device sync, when omitted)."""
    total_q, Hq, D = q.shape
    NB, bs, Hkv, _ = k_pool.shape
    B, MB = block_tables.shape
    if max_q_len is None:
        max_q_len = int((q_start[1:] - q_start[:-1]).max().item()) if B else 0
    st = lib().pa_prefill(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                          _ptr(seq_lens), _ptr(q_start), B, total_q, Hq, Hkv, D, bs, MB, NB,
                          max_q_len, float(scale), _dtype(q), _ptr(status), _stream(stream))
    _check(st, "pa_prefill")
    return out


def pa_append_tokens(k_pool: torch.Tensor, v_pool: torch.Tensor, key: torch.Tensor,
                     value: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                     slot_mapping: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Decode-step cache write: the newest token of every sequence (key/value
    [B, Hkv, D]) goes to its slot, computed from block_tables and seq_lens."""
    NB, bs, Hkv, D = k_pool.shape
    B, MB = block_tables.shape
    st = lib().pa_append_tokens(
        _ptr(k_pool), _ptr(v_pool), _ptr(key), _ptr(value), _ptr(block_tables), _ptr(seq_lens),
        _ptr(slot_mapping), B, 0, Hkv, D, bs, MB, NB, _dtype(k_pool), _ptr(status),
        _stream(stream))
    _check(st, "pa_append_tokens")


def pa_stream_read(buf: torch.Tensor, sink: Optional[torch.Tensor] = None, stream=None) -> None:
    """Read every byte of `buf` once (a plain contiguous read stream, see
    include/pagedattn.h, pa_stream_read): the read bandwidth measured beside the
    decode kernels.  sink: optional int64 device tensor of one element."""
    n = buf.numel() * buf.element_size()
    _check(lib().pa_stream_read(_ptr(buf), n, _ptr(sink), _stream(stream)), "pa_stream_read")


class _SimConfig(ctypes.Structure):
    _fields_ = [("allocator", ctypes.c_int), ("reserve", ctypes.c_int),
                ("block_size", ctypes.c_int), ("max_seq_len", ctypes.c_int),
                ("capacity_tokens", ctypes.c_int64), ("max_steps", ctypes.c_int64)]


_SIM_FIELDS = ("steps", "completed", "failed_allocations", "fragmentation_failures",
               "preemptions", "max_concurrency", "sum_concurrency", "busy_steps", "sum_stored",
               "sum_held", "peak_stored", "peak_held", "sum_table_len", "max_table_len")


class _SimResult(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in _SIM_FIELDS]


SIM_ALLOCATORS = {"contiguous": 0, "paged": 1}
SIM_RESERVE = {"max": 0, "pow2": 1, "exact": 2}


def simulate_allocator(arrival_step, prompt_len, output_len, allocator: str, capacity: int,
                       block_size: int = 16, reserve: str = "max", max_seq_len: int = 2048,
                       max_steps: int = 10_000_000) -> dict:
    """Contiguous or paged KV allocator over a request stream (pa_sim_run);
    returns the integer counters plus the derived ratios."""
    import numpy as np
    a = np.ascontiguousarray(arrival_step, dtype=np.int32)
    p = np.ascontiguousarray(prompt_len, dtype=np.int32)
    o = np.ascontiguousarray(output_len, dtype=np.int32)
    if not len(a) == len(p) == len(o):
        raise ValueError("one arrival, prompt and output length per request")
    cfg = _SimConfig(SIM_ALLOCATORS[allocator], SIM_RESERVE[reserve], block_size, max_seq_len,
                     capacity, max_steps)
    res = _SimResult()
    _check(lib().pa_sim_run(ctypes.byref(cfg), a.ctypes.data, p.ctypes.data, o.ctypes.data,
                            len(a), ctypes.byref(res)), "pa_sim_run")
    out = {f: int(getattr(res, f)) for f in _SIM_FIELDS}
    busy = max(out["busy_steps"], 1)
    out["utilisation_of_held"] = out["sum_stored"] / max(out["sum_held"], 1)
    out["utilisation_of_capacity"] = out["sum_stored"] / (busy * max(capacity, 1))
    out["mean_concurrency"] = out["sum_concurrency"] / busy
    if allocator == "paged":
        out["internal_fragmentation"] = 1.0 - out["utilisation_of_held"]
        out["mean_table_len"] = out["sum_table_len"] / max(out["sum_concurrency"], 1)
    return out


class BlockManager:
    """Host block manager of libpagedattn (pa_bm_*): allocate / free / fork and
    sequences that append one token at a time with copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int,
                 free_stack: Optional[Sequence[int]] = None):
        self._lib = lib()
        handle = ctypes.c_void_p()
        arr = None
        if free_stack is not None:
            arr = (ctypes.c_int32 * num_blocks)(*[int(x) for x in free_stack])
        _check(self._lib.pa_bm_create(num_blocks, block_size, arr, ctypes.byref(handle)),
               "pa_bm_create")
        self._h = handle
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.pa_bm_destroy(h)
            self._h = None

    @property
    def num_free(self) -> int:
        return self._lib.pa_bm_num_free(self._h)

    @property
    def num_evictable(self) -> int:
        """Cached blocks with refcount 0 waiting for eviction."""
        return self._lib.pa_bm_num_evictable(self._h)

    def refcount(self, block: int) -> int:
        return self._lib.pa_bm_refcount(self._h, block)

    def allocate(self, n: int) -> list:
        out = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pa_bm_allocate(self._h, n, out), "pa_bm_allocate")
        return list(out)[:n]

    def free(self, ids: Sequence[int]) -> None:
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(self._lib.pa_bm_free(self._h, arr, len(ids)), "pa_bm_free")

    def fork_blocks(self, ids: Sequence[int]) -> None:
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(self._lib.pa_bm_fork(self._h, arr, len(ids)), "pa_bm_fork")

    def new_sequence(self, prompt_len: int) -> int:
        sid = ctypes.c_int()
        _check(self._lib.pa_bm_seq_create(self._h, prompt_len, ctypes.byref(sid)),
               "pa_bm_seq_create")
        return sid.value

    def new_sequence_cached(self, token_ids: Sequence[int]):
        """Sequence holding token_ids, sharing the longest cached prefix of full
        blocks.  Returns (sequence id, tokens whose KV is already cached)."""
        n = len(token_ids)
        arr = (ctypes.c_int32 * max(n, 1))(*[int(t) for t in token_ids])
        sid, cached = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.pa_bm_seq_create_cached(self._h, arr, n, ctypes.byref(sid),
                                                 ctypes.byref(cached)),
               "pa_bm_seq_create_cached")
        return sid.value, cached.value

    def fork(self, seq: int) -> int:
        sid = ctypes.c_int()
        _check(self._lib.pa_bm_seq_fork(self._h, seq, ctypes.byref(sid)), "pa_bm_seq_fork")
        return sid.value

    def release(self, seq: int) -> None:
        _check(self._lib.pa_bm_seq_release(self._h, seq), "pa_bm_seq_release")

    def append(self, seq: int):
        """Returns (slot, (src, dst) copy-on-write pair or None)."""
        slot, src, dst = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pa_bm_seq_append(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                          ctypes.byref(dst)), "pa_bm_seq_append")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def seq_len(self, seq: int) -> int:
        return self._lib.pa_bm_seq_len(self._h, seq)

    def seq_num_blocks(self, seq: int) -> int:
        return self._lib.pa_bm_seq_num_blocks(self._h, seq)

    def export(self, seqs: Sequence[int], max_blocks: int, pad_id: int):
        """(block_tables [n, max_blocks] int32, seq_lens [n] int32) as CPU tensors."""
        n = len(seqs)
        ids = (ctypes.c_int * max(n, 1))(*seqs)
        tables = torch.empty((n, max_blocks), dtype=torch.int32)
        lens = torch.empty((n,), dtype=torch.int32)
        _check(self._lib.pa_bm_export(self._h, ids, n, max_blocks, pad_id, tables.data_ptr(),
                                      lens.data_ptr()), "pa_bm_export")
        return tables, lens


__all__ = [
    "FLOAT16", "BFLOAT16", "PagedAttnError", "pa_decode", "pa_decode_append",
    "pa_decode_workspace_bytes", "pa_decode_workspace_bytes_for", "workspace_for",
    "pa_decode_noalloc", "set_decode_path", "decode_kernel_for",
    "alloc_workspace", "pa_reshape_and_cache", "pa_append_tokens", "pa_prefill", "set_prefill_path",
    "pa_copy_blocks_multi", "pa_swap_blocks", "pa_copy_blocks", "pa_decode_slots",
    "BlockManager", "lib", "simulate_allocator", "pa_stream_read",
]
