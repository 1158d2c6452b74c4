"""Device marshalling shared by the GPU tests (numpy storage bits <-> torch)."""
import numpy as np
import torch

import synthetic as syn
from oracle.attention import within_tolerance

TORCH_DTYPE = {syn.FLOAT16: torch.float16, syn.BFLOAT16: torch.bfloat16}


def lib():
    from paged_kv_cache_301_gb300 import build
    build.build()
    import paged_kv_cache_301_gb300 as pa
    return pa


def to_dev(bits: np.ndarray, dtype: int) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DTYPE[dtype]).cuda()


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def widen(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "", atol=2e-3, rtol=1e-2):
    ok = within_tolerance(gpu, ref, atol, rtol)
    if not ok.all():
        err = np.abs(gpu - ref) - (atol + rtol * np.abs(ref))
        idx = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(
            f"{what}: {int((~ok).sum())} of {ok.size} elements outside |d| <= {atol} + "
            f"{rtol}|ref|; worst at {idx}: gpu={gpu[idx]!r} ref={ref[idx]!r}")


class DeviceBatch:
    """A PagedBatch uploaded to the GPU, pools with guard blocks on both sides."""

    GUARD = 2

    def __init__(self, batch, guard_bits=0x5A5A):
        self.batch = batch
        dt = batch.dtype
        g = self.GUARD
        shape = batch.k_pool.shape
        full = (shape[0] + 2 * g,) + shape[1:]
        kp = np.full(full, guard_bits, dtype=np.uint16)
        vp = np.full(full, guard_bits ^ 0xFFFF, dtype=np.uint16)
        kp[g:g + shape[0]] = batch.k_pool
        vp[g:g + shape[0]] = batch.v_pool
        self.k_full = to_dev(kp, dt)
        self.v_full = to_dev(vp, dt)
        self.k_pool = self.k_full[g:g + shape[0]]
        self.v_pool = self.v_full[g:g + shape[0]]
        self.q = to_dev(batch.q, dt)
        self.tables = i32(batch.block_tables)
        self.lens = i32(batch.seq_lens)
        self.guard_bits = guard_bits

    def guards_intact(self) -> bool:
        g = self.GUARD
        k = to_host_bits(self.k_full)
        v = to_host_bits(self.v_full)
        return bool((k[:g] == self.guard_bits).all() and (k[-g:] == self.guard_bits).all()
                    and (v[:g] == self.guard_bits ^ 0xFFFF).all()
                    and (v[-g:] == self.guard_bits ^ 0xFFFF).all())

    def decode(self, pa, tables=None, lens=None, max_seq_len=None, partition_tokens=0,
               status=None):
        tables = self.tables if tables is None else tables
        lens = self.lens if lens is None else lens
        if max_seq_len is None:
            max_seq_len = int(self.batch.seq_lens.max()) if lens is self.lens else None
        out = torch.empty_like(self.q)
        pa.pa_decode(out, self.q, self.k_pool, self.v_pool, tables, lens, self.batch.scale,
                     max_seq_len=max_seq_len, partition_tokens=partition_tokens,
                     status=status)
        return out
