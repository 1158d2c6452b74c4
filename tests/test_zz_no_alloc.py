"""pa_decode_noalloc: decode attention whose split-K scratch is a fixed array
inside the library, for callers that cannot allocate device memory when they
call (graph-recorded code without an allocator, plug-ins that only receive
pointers from a host application, allocator-free real-time loops).

Its output must match pa_decode (which uses a caller workspace) and the oracle
within the parity tolerance, on two calls in a row on every decode kernel (the
array keeps the first call's contents, which must not leak into the second),
and batches that need more scratch than the array holds must be rejected before
any device work.  This
file is collected last so a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from tests.gpu_helpers import DeviceBatch, assert_close, i32, lib, widen

pytestmark = pytest.mark.gpu


def _call(pa, dev, out, lens, max_seq_len, status=None):
    """Through the C ABI directly (no Python-side workspace at all)."""
    q, kp, vp, tables = dev.q, dev.k_pool, dev.v_pool, dev.tables
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = kp.shape
    return pa.lib().pa_decode_noalloc(
        out.data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(), tables.data_ptr(),
        lens.data_ptr(), B, Hq, Hkv, D, bs, tables.shape[1], NB, max_seq_len,
        ctypes.c_float(dev.batch.scale), 1 if q.dtype == torch.bfloat16 else 0, 0,
        None if status is None else status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("path", ["auto", "tc_head", "simt"])
def test_matches_pa_decode_on_two_calls_in_a_row(path):
    """Two different batches back to back on each decode kernel (the grouped
    tensor-core kernel by default, the per-head tensor-core kernel, the CUDA-core
    kernel: each uses a different part of the array).  The second batch has a
    different longest sequence, so its partial layout differs, and its call runs
    on scratch that still holds the first call's partials.  Each output is
    checked against pa_decode with a caller workspace and against the oracle."""
    pa = lib()
    w1 = syn.LLAMA3_8B.__class__(**{**syn.LLAMA3_8B.__dict__, "num_seqs": 24, "hi": 3000,
                                    "seed": 41})
    w2 = syn.LLAMA3_8B.__class__(**{**syn.LLAMA3_8B.__dict__, "num_seqs": 16, "lo": 1,
                                    "hi": 2100, "seed": 42})
    pa.set_decode_path(path)
    try:
        for w in (w1, w2):
            batch = scenarios.fixed_batch(w)
            dev = DeviceBatch(batch)
            max_len = int(batch.seq_lens.max())
            ref = dev.decode(pa, max_seq_len=max_len)          # caller-workspace path
            out = torch.full_like(dev.q, float("nan"))
            assert _call(pa, dev, out, dev.lens, max_len) == 0
            torch.cuda.synchronize()
            assert_close(widen(out), widen(ref), f"noalloc vs pa_decode ({path}, {w.num_seqs} seqs)")
            assert_close(widen(out), scenarios.decode_f64(batch),
                         f"noalloc vs oracle ({path}, {w.num_seqs} seqs)")
    finally:
        pa.set_decode_path("auto")


@pytest.mark.parametrize("path", ["tc_head", "simt"])
def test_oversized_batch_rejected_before_device_work(path):
    """8 sequences x 64 query heads up to 128K tokens: the partition kernels need
    about 65 MiB of partials, more than the array, so the call is refused before
    anything runs (the grouped kernel's need does not grow with the lengths)."""
    pa = lib()
    w = syn.LONG_CONTEXT.__class__(**{**syn.LONG_CONTEXT.__dict__, "length_kind": "fixed",
                                      "lens": (10,) * 8, "num_blocks": 16})
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    out = torch.zeros_like(dev.q)
    max_len = 131072
    tables = torch.zeros((8, max_len // w.block_size), dtype=torch.int32, device="cuda")
    tables[:, :1] = dev.tables[:, :1]
    pa.set_decode_path(path)
    try:
        need = pa.pa_decode_workspace_bytes_for(8, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                w.block_size, tables.shape[1], batch.num_blocks,
                                                max_len, 1)
        assert need > pa.NOALLOC_SCRATCH_BYTES
        st = pa.lib().pa_decode_noalloc(
            out.data_ptr(), dev.q.data_ptr(), dev.k_pool.data_ptr(), dev.v_pool.data_ptr(),
            tables.data_ptr(), dev.lens.data_ptr(), 8, w.num_q_heads, w.num_kv_heads,
            w.head_dim, w.block_size, tables.shape[1], batch.num_blocks, max_len,
            ctypes.c_float(w.scale), 1, 0, None, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        pa.set_decode_path("auto")
    assert st == 3
    assert not out.any()
