"""GPU parity of the cache writes (reshape_and_cache, copy_blocks, decode_slots)
and of whole decode steps, against the oracle, bit for bit over the whole pool
including guard blocks on both sides."""
import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from oracle.cache_ops import copy_blocks, reshape_and_cache
from tests.gpu_helpers import DeviceBatch, assert_close, i32, lib, to_dev, to_host_bits, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["simt", "tc_head", "tc"])
def pa(request):
    """Every test runs on each decode kernel: CUDA cores, the per-head
    tensor-core kernel and the grouped tensor-core kernel (for shapes it does
    not serve, "tc" runs the per-head one)."""
    m = lib()
    m.set_decode_path(request.param)
    m.decode_path = request.param
    yield m
    m.set_decode_path("auto")


def needs(pa, head_dim):
    if pa.decode_path != "simt" and head_dim != 128:
        pytest.skip("the tensor-core kernel serves head_dim 128")


def _pools_equal(dev, k_ref, v_ref):
    assert np.array_equal(to_host_bits(dev.k_pool), k_ref)
    assert np.array_equal(to_host_bits(dev.v_pool), v_ref)
    assert dev.guards_intact()


@pytest.mark.parametrize("dtype", [syn.FLOAT16, syn.BFLOAT16])
@pytest.mark.parametrize("head_dim,hkv", [(64, 4), (128, 8), (128, 1)])
def test_reshape_and_cache_bit_exact(pa, dtype, head_dim, hkv):
    w = syn.LLAMA3_8B.__class__(**{**syn.LLAMA3_8B.__dict__, "dtype": dtype,
                                   "head_dim": head_dim, "num_kv_heads": hkv,
                                   "num_q_heads": hkv, "length_kind": "fixed",
                                   "lens": (30, 200, 5), "num_seqs": 3})
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    g = np.random.default_rng(dtype * 7 + head_dim)
    T = 333
    nslots = batch.num_blocks * w.block_size
    slots = g.choice(nslots, size=T, replace=False).astype(np.int32)
    slots[::17] = -1                                  # padding tokens
    key, value = syn.token_kv_bits(w, T, sub=5)
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    reshape_and_cache(kp, vp, key, value, slots)
    pa.pa_reshape_and_cache(dev.k_pool, dev.v_pool, to_dev(key, dtype), to_dev(value, dtype),
                            i32(slots))
    torch.cuda.synchronize()
    _pools_equal(dev, kp, vp)


def test_reshape_and_cache_out_of_range_slot_reported(pa):
    batch = scenarios.fixed_batch(syn.TINY)
    dev = DeviceBatch(batch)
    key, value = syn.token_kv_bits(syn.TINY, 3, sub=9)
    slots = np.array([3, batch.num_blocks * 16 + 1, 40], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(dev.k_pool, dev.v_pool, to_dev(key, 0), to_dev(value, 0), i32(slots),
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    reshape_and_cache(kp, vp, key[[0, 2]], value[[0, 2]], slots[[0, 2]])
    _pools_equal(dev, kp, vp)


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_copy_blocks_bit_exact(pa, bs):
    w = syn.LLAMA3_8B.__class__(**{**syn.LLAMA3_8B.__dict__, "block_size": bs,
                                   "length_kind": "fixed", "lens": (900, 700), "num_seqs": 2})
    batch = scenarios.fixed_batch(w)
    batch.k_pool, batch.v_pool = syn.pool_fill_bits(w, batch.num_blocks, sub=bs)
    dev = DeviceBatch(batch)
    g = np.random.default_rng(bs)
    ids = g.permutation(batch.num_blocks)
    pairs = np.stack([ids[:6], ids[6:12]], axis=1).astype(np.int32)
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    copy_blocks(kp, vp, pairs)
    pa.pa_copy_blocks(dev.k_pool, dev.v_pool, i32(pairs))
    torch.cuda.synchronize()
    _pools_equal(dev, kp, vp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = np.array([[0, batch.num_blocks]], dtype=np.int32)
    pa.pa_copy_blocks(dev.k_pool, dev.v_pool, i32(bad), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    _pools_equal(dev, kp, vp)


def test_decode_slots_match_block_manager(pa):
    initial, steps, final = scenarios.ragged_steps(syn.RAGGED, 16, 3, num_seqs=64)
    nb = initial.num_blocks
    for st in steps:
        out = torch.empty(len(st.seq_lens), dtype=torch.int32, device="cuda")
        pa.pa_decode_slots(out, i32(st.block_tables), i32(st.seq_lens), 16, nb)
        assert np.array_equal(out.cpu().numpy(), st.slot_mapping)
    lens = steps[0].seq_lens.copy()
    lens[:5] = 0
    out = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_slots(out, i32(steps[0].block_tables), i32(lens), 16, nb, status=status)
    assert (out.cpu().numpy()[:5] == -1).all()
    assert int(status.item()) == 0              # empty sequences are not errors


def test_decode_slots_checked_mode_poisoned_table(pa):
    """A table entry outside the pool (negative, or num_blocks and beyond) where a
    newest token lands gives slot -1 and PA_ERR_BAD_BLOCK_ID; other slots are
    still those of the block manager."""
    initial, steps, final = scenarios.ragged_steps(syn.RAGGED, 16, 1, num_seqs=64)
    st = steps[0]
    nb = initial.num_blocks
    tables = st.block_tables.copy()
    last = (st.seq_lens.astype(np.int64) - 1) // 16
    bad = {3: -7, 10: nb, 20: nb + 1000}
    for b, v in bad.items():
        tables[b, last[b]] = v
    out = torch.empty(len(st.seq_lens), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_slots(out, i32(tables), i32(st.seq_lens), 16, nb, status=status)
    got = out.cpu().numpy()
    want = st.slot_mapping.copy()
    for b in bad:
        want[b] = -1
    assert np.array_equal(got, want)
    assert int(status.item()) == 5
    # a length past the table is reported the same way
    lens = st.seq_lens.copy()
    lens[7] = tables.shape[1] * 16 + 1
    status.zero_()
    pa.pa_decode_slots(out, i32(st.block_tables), i32(lens), 16, nb, status=status)
    assert int(out[7].item()) == -1 and int(status.item()) == 5


@pytest.mark.parametrize("bs", [8, 16, 64])
def test_append_tokens_matches_slots_then_write(pa, bs):
    """The fused decode-step write equals decode_slots + reshape_and_cache: same
    slots as the block manager, bit-exact pools, empty sequences skipped."""
    initial, steps, final = scenarios.ragged_steps(syn.RAGGED, bs, 2, num_seqs=48)
    dev = DeviceBatch(initial)
    dt = syn.RAGGED.dtype
    k_ref, v_ref = initial.k_pool.copy(), initial.v_pool.copy()
    for st in steps:
        lens = st.seq_lens.copy()
        lens[5] = 0                                   # an empty sequence writes nothing
        slots = torch.full((len(lens),), 7, dtype=torch.int32, device="cuda")
        pa.pa_append_tokens(dev.k_pool, dev.v_pool, to_dev(st.key, dt), to_dev(st.value, dt),
                            i32(st.block_tables), i32(lens), slot_mapping=slots)
        want = st.slot_mapping.copy()
        want[5] = -1
        assert np.array_equal(slots.cpu().numpy(), want)
        reshape_and_cache(k_ref, v_ref, st.key, st.value, want)
    torch.cuda.synchronize()
    _pools_equal(dev, k_ref, v_ref)


def test_shared_prefix_workload(pa):
    """16 prompts x 8 forked samples: every step's CoW copies then the new tokens,
    replayed on the GPU; pools bit-exact, then decode against the oracle."""
    initial, steps, final = scenarios.shared_prefix(syn.SHARED_PREFIX)
    dev = DeviceBatch(initial)
    dt = syn.SHARED_PREFIX.dtype
    ncow = 0
    for st in steps:
        if len(st.cow_pairs):
            ncow += len(st.cow_pairs)
            pa.pa_copy_blocks(dev.k_pool, dev.v_pool, i32(st.cow_pairs))
        pa.pa_reshape_and_cache(dev.k_pool, dev.v_pool, to_dev(st.key, dt), to_dev(st.value, dt),
                                i32(st.slot_mapping))
    torch.cuda.synchronize()
    assert ncow > 0
    _pools_equal(dev, final.k_pool, final.v_pool)
    out = dev.decode(pa, tables=i32(final.block_tables), lens=i32(final.seq_lens),
                     max_seq_len=int(final.seq_lens.max()))
    assert_close(widen(out), scenarios.decode_f64(final), "shared prefix")


@pytest.mark.parametrize("bs", syn.RAGGED_BLOCK_SIZES)
def test_ragged_continuous_batching_steps(pa, bs):
    """Each step: slots of the newest tokens (decode_slots), cache write, decode
    with the grown lengths.  8 steps so that block boundaries are crossed."""
    initial, steps, final = scenarios.ragged_steps(syn.RAGGED, bs, 8)
    dev = DeviceBatch(initial)
    dt = syn.RAGGED.dtype
    B = len(initial.seq_lens)
    k_ref, v_ref = initial.k_pool.copy(), initial.v_pool.copy()
    sample = list(range(0, B, 17))
    for i, st in enumerate(steps):
        tables, lens = i32(st.block_tables), i32(st.seq_lens)
        slots = torch.empty(B, dtype=torch.int32, device="cuda")
        pa.pa_decode_slots(slots, tables, lens, bs, initial.num_blocks)
        pa.pa_reshape_and_cache(dev.k_pool, dev.v_pool, to_dev(st.key, dt), to_dev(st.value, dt),
                                slots)
        out = dev.decode(pa, tables=tables, lens=lens, max_seq_len=int(st.seq_lens.max()))
        assert np.array_equal(slots.cpu().numpy(), st.slot_mapping)
        reshape_and_cache(k_ref, v_ref, st.key, st.value, st.slot_mapping)
        step_batch = scenarios.PagedBatch(initial.workload, bs, initial.num_blocks, k_ref, v_ref,
                                          initial.q, st.block_tables, st.seq_lens,
                                          initial.pad_block, None, [])
        last = i == len(steps) - 1
        ref = scenarios.decode_f64(step_batch, sequences=None if last else sample)
        got = widen(out)
        rows = slice(None) if last else sample
        assert_close(got[rows], ref[rows], f"bs={bs} step {i}")
    torch.cuda.synchronize()
    _pools_equal(dev, final.k_pool, final.v_pool)


def test_append_tokens_reports_bad_lengths_and_ids(pa):
    """Checked mode: a length past its table and a block id outside the pool are
    reported and skipped; every other sequence is written."""
    initial, steps, final = scenarios.ragged_steps(syn.RAGGED, 16, 1, num_seqs=12)
    st = steps[0]
    dev = DeviceBatch(initial)
    dt = syn.RAGGED.dtype
    lens = st.seq_lens.copy()
    tables = st.block_tables.copy()
    lens[2] = tables.shape[1] * 16 + 5                     # longer than its table
    row = (lens[7] - 1) // 16
    tables[7, row] = initial.num_blocks + 3                # the newest token's block: outside
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    pa.pa_append_tokens(dev.k_pool, dev.v_pool, to_dev(st.key, dt), to_dev(st.value, dt),
                        i32(tables), i32(lens), slot_mapping=slots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    got = slots.cpu().numpy()
    assert got[2] == -1 and got[7] == -1
    want = st.slot_mapping.copy()
    want[[2, 7]] = -1
    assert np.array_equal(got, want)
    k_ref, v_ref = initial.k_pool.copy(), initial.v_pool.copy()
    reshape_and_cache(k_ref, v_ref, st.key, st.value, want)
    _pools_equal(dev, k_ref, v_ref)
