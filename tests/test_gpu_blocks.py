"""GPU parity of the multi-pool block moves: copy-on-write across every layer's
K and V pools in one launch, and block swaps between GPU pools and pools in
pinned CPU memory; bit-exact against the oracle over whole pools."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from oracle.cache_ops import copy_blocks_multi, swap_blocks
from tests.gpu_helpers import DeviceBatch, TORCH_DTYPE, assert_close, i32, lib, to_dev, \
    to_host_bits, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    return lib()


def _layer_pools(g, layers, nb, shape, dtype):
    """K and V pools of `layers` layers, random storage bits (compared as bits)."""
    return [g.integers(0, 2**16, size=(nb,) + shape, dtype=np.uint16) for _ in range(2 * layers)]


@pytest.mark.parametrize("layers,bs", [(1, 16), (4, 8), (32, 16), (3, 64)])
def test_copy_blocks_multi_bit_exact(pa, layers, bs):
    g = np.random.default_rng(layers * 100 + bs)
    nb, shape = 40, (bs, 8, 128)
    bits = _layer_pools(g, layers, nb, shape, syn.BFLOAT16)
    ids = g.permutation(nb)
    pairs = np.stack([ids[:12], ids[12:24]], axis=1).astype(np.int32)   # disjoint src / dst
    pools = [to_dev(b, syn.BFLOAT16) for b in bits]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks_multi(pools, i32(pairs), status=status)
    copy_blocks_multi(bits, pairs)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for p, b in zip(pools, bits):
        assert np.array_equal(to_host_bits(p), b)


def test_copy_blocks_multi_bad_id_reported_and_skipped(pa):
    g = np.random.default_rng(7)
    nb, shape = 12, (16, 8, 64)
    bits = _layer_pools(g, 2, nb, shape, syn.FLOAT16)
    pools = [to_dev(b, syn.FLOAT16) for b in bits]
    pairs = np.array([[1, 2], [3, nb], [-1, 4], [5, 6]], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks_multi(pools, i32(pairs), status=status)
    copy_blocks_multi(bits, pairs[[0, 3]])
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    for p, b in zip(pools, bits):
        assert np.array_equal(to_host_bits(p), b)
    pa.pa_copy_blocks_multi(pools, torch.empty((0, 2), dtype=torch.int32, device="cuda"))


def _pinned_like(bits, dtype):
    t = torch.from_numpy(bits.view(np.int16).copy()).view(TORCH_DTYPE[dtype]).pin_memory()
    return t


def _cpu_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("pairs_on", ["gpu", "pinned"])
def test_swap_out_and_in_bit_exact(pa, pairs_on):
    g = np.random.default_rng(11)
    layers, gnb, cnb, shape = 3, 30, 9, (16, 8, 128)
    gbits = _layer_pools(g, layers, gnb, shape, syn.BFLOAT16)
    cbits = _layer_pools(g, layers, cnb, shape, syn.BFLOAT16)
    gpu = [to_dev(b, syn.BFLOAT16) for b in gbits]
    cpu = [_pinned_like(b, syn.BFLOAT16) for b in cbits]
    out_pairs = np.array([[29, 0], [3, 8], [17, 4]], dtype=np.int32)
    in_pairs = np.array([[8, 0], [1, 28], [4, 10]], dtype=np.int32)

    def arr(p):
        t = torch.from_numpy(p)
        return t.cuda() if pairs_on == "gpu" else t.pin_memory()

    pa.pa_swap_blocks(cpu, gpu, arr(out_pairs))
    swap_blocks(cbits, gbits, out_pairs)
    torch.cuda.synchronize()
    for c, b in zip(cpu, cbits):
        assert np.array_equal(_cpu_bits(c), b)
    pa.pa_swap_blocks(gpu, cpu, arr(in_pairs))
    swap_blocks(gbits, cbits, in_pairs)
    torch.cuda.synchronize()
    for p, b in zip(gpu, gbits):
        assert np.array_equal(to_host_bits(p), b)


def test_swap_rejects_pageable_host_memory(pa):
    """Pageable memory is refused by the host-side check (nothing is launched)."""
    gpu = torch.zeros((4, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    host = np.zeros((4, 16, 8, 128), dtype=np.uint16)          # pageable
    pairs = i32(np.array([[0, 1]]))
    L = pa.lib()
    dst = (ctypes.c_void_p * 1)(host.ctypes.data)
    src = (ctypes.c_void_p * 1)(gpu.data_ptr())
    st = L.pa_swap_blocks(ctypes.cast(dst, ctypes.c_void_p), ctypes.cast(src, ctypes.c_void_p),
                          1, pairs.data_ptr(), 1, 16 * 8 * 128 * 2, 4, 4, None,
                          torch.cuda.current_stream().cuda_stream)
    assert st == 1
    with pytest.raises(ValueError):
        pa.pa_swap_blocks([torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16)], [gpu], pairs)


@pytest.mark.parametrize("bs", [16, 32])
def test_sequences_swapped_to_cpu_and_back_decode_identically(pa, bs):
    """Evict three sequences to pinned CPU pools, let another sequence overwrite
    their GPU blocks, swap them back into other blocks: pools bit-exact with the
    oracle's replay, decode bit-identical to the decode before the eviction and
    within tolerance of the fp64 oracle."""
    w = dataclasses.replace(syn.LLAMA3_8B, num_seqs=6, length_kind="fixed",
                            lens=(700, 33, 1500, 16, 260, 900), block_size=bs,
                            pool_factor=3.0)
    batch = scenarios.fixed_batch(w)
    swapped = [0, 2, 5]
    rt = scenarios.swap_round_trip(batch, swapped, cpu_num_blocks=300, seed=bs)
    dt = w.dtype
    dev = DeviceBatch(batch)
    before = dev.decode(pa)
    nan = syn.NAN_BITS[dt]
    shape = (rt.cpu_num_blocks,) + batch.k_pool.shape[1:]
    cpu_k = _pinned_like(np.full(shape, nan, np.uint16), dt)
    cpu_v = _pinned_like(np.full(shape, nan, np.uint16), dt)
    pa.pa_swap_blocks([cpu_k, cpu_v], [dev.k_pool, dev.v_pool], i32(rt.out_pairs))
    torch.cuda.synchronize()
    assert np.array_equal(_cpu_bits(cpu_k), rt.cpu_k_pool)
    assert np.array_equal(_cpu_bits(cpu_v), rt.cpu_v_pool)
    reused = torch.from_numpy(rt.reused_blocks.astype(np.int64)).cuda()
    poison = torch.tensor(np.array([nan], np.uint16).view(np.int16))
    dev.k_pool.view(torch.int16)[reused] = poison.cuda()
    dev.v_pool.view(torch.int16)[reused] = poison.cuda()
    pa.pa_swap_blocks([dev.k_pool, dev.v_pool], [cpu_k, cpu_v], i32(rt.in_pairs))
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(dev.k_pool), rt.after.k_pool)
    assert np.array_equal(to_host_bits(dev.v_pool), rt.after.v_pool)
    assert dev.guards_intact()
    after = dev.decode(pa, tables=i32(rt.after.block_tables), lens=dev.lens,
                       max_seq_len=int(batch.seq_lens.max()))
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    assert_close(widen(after), scenarios.decode_f64(rt.after), f"swap bs={bs}")


def test_swap_bad_ids_reported_and_skipped(pa):
    g = np.random.default_rng(12)
    gbits = _layer_pools(g, 1, 10, (16, 8, 128), syn.BFLOAT16)
    cbits = _layer_pools(g, 1, 4, (16, 8, 128), syn.BFLOAT16)
    gpu = [to_dev(b, syn.BFLOAT16) for b in gbits]
    cpu = [_pinned_like(b, syn.BFLOAT16) for b in cbits]
    pairs = np.array([[9, 0], [3, 4], [10, 1], [2, 3]], dtype=np.int32)   # dst 4 / src 10 invalid
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_swap_blocks(cpu, gpu, i32(pairs), status=status)
    swap_blocks(cbits, gbits, pairs[[0, 3]])
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    for c, b in zip(cpu, cbits):
        assert np.array_equal(_cpu_bits(c), b)


def test_stream_read_reads_every_byte():
    """pa_stream_read (the benchmark's read-stream context) counts, per thread,
    the words whose XOR equals 0x9E3779B9: in a zero buffer holding that word at
    the start, the middle and the end (and in the tail that does not fill a whole
    round of the grid), the sink counts three, so every region was read."""
    import torch
    from tests.gpu_helpers import lib
    pa = lib()
    n_words = (3 << 20) + 20                 # 12 MiB + 80 bytes: a ragged tail
    buf = torch.zeros(n_words, dtype=torch.int32, device="cuda")
    magic = 0x9E3779B9 - (1 << 32)           # as int32
    for i in (0, n_words // 2 + 4, n_words - 1):
        buf[i] = magic
    sink = torch.zeros(1, dtype=torch.int64, device="cuda")
    pa.pa_stream_read(buf, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == 3
