"""GPU parity of pa_decode_append (one decode step: the newest token of every
sequence is written to its slot, then decode attention over the grown
sequences) against the oracle and against the two calls it stands for
(pa_append_tokens, then pa_decode).

Acceptance: pools bit-exact against the oracle's cache write; attention within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle|; and outputs bit-identical to the two
calls, since the same decode kernel reads the same pool contents.  The write is
fused into the grouped tensor-core kernel, so the cases span its tile shapes
(4 to 128 tokens per tile, tiles smaller and larger than a block) and batches
where a CTA's first tile is the last tile of a sequence."""
import dataclasses

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from oracle.cache_ops import reshape_and_cache
from tests.gpu_helpers import DeviceBatch, assert_close, i32, lib, to_dev, to_host_bits, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["auto", "simt"])
def pa(request):
    """The default kernel choice (the write runs inside the grouped tensor-core
    kernel where it serves the shape) and the CUDA-core kernel (two launches)."""
    m = lib()
    m.set_decode_path(request.param)
    yield m
    m.set_decode_path("auto")


def _pools_equal(dev, k_ref, v_ref):
    assert np.array_equal(to_host_bits(dev.k_pool), k_ref)
    assert np.array_equal(to_host_bits(dev.v_pool), v_ref)
    assert dev.guards_intact()


def _fused(pa, dev, key, value, tables, lens, scale, max_seq_len, status=None):
    out = torch.empty_like(dev.q)
    pa.pa_decode_append(out, dev.q, dev.k_pool, dev.v_pool, key, value, tables, lens, scale,
                        max_seq_len=max_seq_len, status=status)
    return out


def _two_calls(pa, dev, key, value, tables, lens, scale, max_seq_len, status=None):
    pa.pa_append_tokens(dev.k_pool, dev.v_pool, key, value, tables, lens, status=status)
    out = torch.empty_like(dev.q)
    pa.pa_decode(out, dev.q, dev.k_pool, dev.v_pool, tables, lens, scale,
                 max_seq_len=max_seq_len, status=status)
    return out


def _newest_slots(tables: np.ndarray, lens: np.ndarray, bs: int) -> np.ndarray:
    pos = lens.astype(np.int64) - 1
    return tables[np.arange(len(lens)), pos // bs].astype(np.int64) * bs + pos % bs


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16)


CASES = ([(32, 8, bs) for bs in syn.RAGGED_BLOCK_SIZES] +
         [(8, 1, 16), (16, 2, 64), (32, 32, 16), (32, 32, 64), (64, 8, 32), (16, 16, 8),
          (128, 8, 16), (128, 64, 16),      # head-group passes: each writes its own heads
          (40, 8, 16), (28, 4, 32)])        # 5 and 7 query heads per KV head


@pytest.mark.parametrize("hq,hkv,bs", CASES)
def test_continuous_batching_steps(pa, hq, hkv, bs):
    """Four decode steps over 64 lognormal-length sequences: every step's pools
    bit-exact, its outputs bit-identical to the two calls and within tolerance of
    the oracle (sampled rows; every row at the last step)."""
    w = dataclasses.replace(syn.RAGGED, num_q_heads=hq, num_kv_heads=hkv)
    initial, steps, final = scenarios.ragged_steps(w, bs, 4, num_seqs=64)
    fused_dev, split_dev = DeviceBatch(initial), DeviceBatch(initial)
    k_ref, v_ref = initial.k_pool.copy(), initial.v_pool.copy()
    sample = list(range(0, 64, 9))
    for i, st in enumerate(steps):
        tables, lens = i32(st.block_tables), i32(st.seq_lens)
        key, value = to_dev(st.key, w.dtype), to_dev(st.value, w.dtype)
        mx = int(st.seq_lens.max())
        got = _fused(pa, fused_dev, key, value, tables, lens, w.scale, mx)
        want = _two_calls(pa, split_dev, key, value, tables, lens, w.scale, mx)
        torch.cuda.synchronize()
        assert torch.equal(_bits(got), _bits(want)), f"step {i}: fused != two calls"
        reshape_and_cache(k_ref, v_ref, st.key, st.value, st.slot_mapping)
        step_batch = scenarios.PagedBatch(w, bs, initial.num_blocks, k_ref, v_ref, initial.q,
                                          st.block_tables, st.seq_lens, initial.pad_block,
                                          None, [])
        last = i == len(steps) - 1
        ref = scenarios.decode_f64(step_batch, sequences=None if last else sample)
        rows = slice(None) if last else sample
        assert_close(widen(got)[rows], ref[rows], f"Hq={hq} Hkv={hkv} bs={bs} step {i}")
    _pools_equal(fused_dev, final.k_pool, final.v_pool)
    _pools_equal(split_dev, final.k_pool, final.v_pool)


def test_many_short_sequences(pa):
    """1000 sequences of 1-40 tokens (1-3 tiles each): nearly every CTA range
    starts or ends on a sequence's last tile, the tile the write must precede."""
    g = np.random.default_rng(11)
    lens = g.integers(1, 41, size=1000)
    w = dataclasses.replace(syn.LLAMA3_8B, name="short", num_seqs=1000, length_kind="fixed",
                            lens=tuple(int(x) for x in lens))
    batch = scenarios.fixed_batch(w)
    key, value = syn.token_kv_bits(w, 1000, sub=300_000)
    slots = _newest_slots(batch.block_tables, batch.seq_lens, w.block_size)
    k_ref, v_ref = batch.k_pool.copy(), batch.v_pool.copy()
    reshape_and_cache(k_ref, v_ref, key, value, slots)
    dev = DeviceBatch(batch)
    out = _fused(pa, dev, to_dev(key, w.dtype), to_dev(value, w.dtype), dev.tables, dev.lens,
                 w.scale, 40)
    torch.cuda.synchronize()
    _pools_equal(dev, k_ref, v_ref)
    after = dataclasses.replace(batch, k_pool=k_ref, v_pool=v_ref)
    assert_close(widen(out), scenarios.decode_f64(after), "1000 short sequences")


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 2, 32), (8, 4, 8)])
def test_empty_sequences_between_segments(pa, hq, hkv, bs):
    """300 sequences of 0-200 tokens, every third one empty: segments follow each
    other across empty sequences (the next segment's inputs and Q are fetched
    ahead), finished segments stage their outputs in shared memory, and some
    CTA ranges hold many short sequences.  Empty sequences give zero rows and
    write nothing."""
    g = np.random.default_rng(21)
    lens = g.integers(1, 201, size=300)
    lens[::3] = 0
    w = dataclasses.replace(syn.LLAMA3_8B, name="gaps", num_seqs=300, length_kind="fixed",
                            lens=tuple(int(x) for x in np.maximum(lens, 1)),
                            num_q_heads=hq, num_kv_heads=hkv, block_size=bs)
    batch = scenarios.fixed_batch(w)
    key, value = syn.token_kv_bits(w, 300, sub=600_000)
    seq_lens = lens.astype(np.int32)
    live = seq_lens > 0
    slots = _newest_slots(batch.block_tables[live], seq_lens[live], bs)
    k_ref, v_ref = batch.k_pool.copy(), batch.v_pool.copy()
    reshape_and_cache(k_ref, v_ref, key[live], value[live], slots)
    dev = DeviceBatch(batch)
    out = _fused(pa, dev, to_dev(key, w.dtype), to_dev(value, w.dtype), dev.tables,
                 i32(seq_lens), w.scale, 200)
    torch.cuda.synchronize()
    _pools_equal(dev, k_ref, v_ref)
    after = dataclasses.replace(batch, k_pool=k_ref, v_pool=v_ref, seq_lens=seq_lens)
    got = widen(out)
    assert not got[~live].any()
    assert_close(got, scenarios.decode_f64(after), f"Hq={hq} Hkv={hkv} bs={bs} with gaps")


@pytest.mark.parametrize("w", [syn.LLAMA3_8B, syn.MHA_7B, syn.LONG_CONTEXT], ids=lambda w: w.name)
def test_benchmark_workloads(pa, w):
    """Full size, in the launch configuration the benchmark times: fused step
    bit-identical to the two calls; written slots bit-exact; sampled rows
    against the oracle."""
    batch = scenarios.fixed_batch(w, fill_all=True)
    B = len(batch.seq_lens)
    key, value = syn.token_kv_bits(w, B, sub=400_000)
    slots = _newest_slots(batch.block_tables, batch.seq_lens, w.block_size)
    fused_dev, split_dev = DeviceBatch(batch), DeviceBatch(batch)
    kd, vd = to_dev(key, w.dtype), to_dev(value, w.dtype)
    mx = int(batch.seq_lens.max())
    got = _fused(pa, fused_dev, kd, vd, fused_dev.tables, fused_dev.lens, w.scale, mx)
    want = _two_calls(pa, split_dev, kd, vd, split_dev.tables, split_dev.lens, w.scale, mx)
    torch.cuda.synchronize()
    assert torch.equal(_bits(got), _bits(want))
    bs, hkv = w.block_size, w.num_kv_heads
    for dev in (fused_dev, split_dev):
        k = to_host_bits(dev.k_pool.reshape(-1, hkv, w.head_dim)[torch.from_numpy(slots).cuda()])
        v = to_host_bits(dev.v_pool.reshape(-1, hkv, w.head_dim)[torch.from_numpy(slots).cuda()])
        assert np.array_equal(k, key) and np.array_equal(v, value)
        assert dev.guards_intact()
    k_ref, v_ref = batch.k_pool, batch.v_pool        # the batch's own arrays, updated in place
    reshape_and_cache(k_ref, v_ref, key, value, slots)
    seqs = sorted({0, B - 1, int(np.argmax(batch.seq_lens))})
    heads = [0, w.num_q_heads - 1] if w is syn.LONG_CONTEXT else None
    ref = scenarios.decode_f64(batch, sequences=seqs, heads=heads)
    h = slice(None) if heads is None else heads
    for s in seqs:
        assert_close(widen(got)[s, h], ref[s, h], f"{w.name} sequence {s}")


def test_bad_input_reported_like_the_two_calls(pa):
    """Checked mode: a newest-token block outside the pool, a length past the
    table, a negative length and an empty sequence.  Both forms report status 5,
    leave bit-identical pools (bad writes skipped) and give bit-identical rows."""
    w = dataclasses.replace(syn.RAGGED, num_q_heads=32, num_kv_heads=8)
    initial, steps, _ = scenarios.ragged_steps(w, 16, 1, num_seqs=24)
    st = steps[0]
    tables, lens = st.block_tables.copy(), st.seq_lens.copy()
    max_seq_len = tables.shape[1] * 16
    row = (lens[7] - 1) // 16
    tables[7, row] = initial.num_blocks + 3
    lens[2] = max_seq_len + 5
    lens[4] = -3
    lens[5] = 0
    key, value = to_dev(st.key, w.dtype), to_dev(st.value, w.dtype)
    results = []
    for form in (_fused, _two_calls):
        dev = DeviceBatch(initial)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = form(pa, dev, key, value, i32(tables), i32(lens), w.scale, max_seq_len, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 5, form.__name__
        results.append((out, to_host_bits(dev.k_pool), to_host_bits(dev.v_pool)))
        assert dev.guards_intact()
    (o1, k1, v1), (o2, k2, v2) = results
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    good = [b for b in range(24) if b not in (2, 4, 5, 7)]
    assert torch.equal(_bits(o1[good]), _bits(o2[good]))
    slots = st.slot_mapping.copy()
    slots[[2, 4, 5, 7]] = -1
    k_ref, v_ref = initial.k_pool.copy(), initial.v_pool.copy()
    reshape_and_cache(k_ref, v_ref, st.key, st.value, slots)
    assert np.array_equal(k1, k_ref) and np.array_equal(v1, v_ref)


def test_zero_max_seq_len_still_writes(pa):
    """max_seq_len 0 clamps every length to 0 (zero rows, reported); the cache
    write still stores every newest token, as pa_append_tokens does."""
    w = dataclasses.replace(syn.RAGGED, num_q_heads=32, num_kv_heads=8)
    initial, steps, final = scenarios.ragged_steps(w, 16, 1, num_seqs=20)
    st = steps[0]
    dev = DeviceBatch(initial)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _fused(pa, dev, to_dev(st.key, w.dtype), to_dev(st.value, w.dtype),
                 i32(st.block_tables), i32(st.seq_lens), w.scale, 0, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    assert not out.float().abs().sum().item()
    _pools_equal(dev, final.k_pool, final.v_pool)


def test_bad_arguments_raise(pa):
    w = dataclasses.replace(syn.RAGGED, num_q_heads=32, num_kv_heads=8)
    initial, steps, _ = scenarios.ragged_steps(w, 16, 1, num_seqs=4)
    st = steps[0]
    dev = DeviceBatch(initial)
    key, value = to_dev(st.key, w.dtype), to_dev(st.value, w.dtype)
    tables, lens = i32(st.block_tables), i32(st.seq_lens)
    out = torch.empty_like(dev.q)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.pa_decode_append(out, dev.q, dev.k_pool, dev.v_pool, None, value, tables, lens,
                            w.scale)
    assert ei.value.status == 1
    shifted = torch.empty(key.numel() + 8, dtype=key.dtype, device="cuda")[1:1 + key.numel()]
    shifted = shifted.view(key.shape).copy_(key)
    with pytest.raises(pa.PagedAttnError) as ei:
        pa.pa_decode_append(out, dev.q, dev.k_pool, dev.v_pool, shifted, value, tables, lens,
                            w.scale)
    assert ei.value.status == 1
    torch.cuda.synchronize()
    _pools_equal(dev, initial.k_pool, initial.v_pool)      # nothing ran


@pytest.mark.parametrize("w", [syn.LLAMA3_8B, syn.LLAMA3_405B, syn.TINY], ids=lambda w: w.name)
def test_step_captured_in_a_cuda_graph(pa, w):
    """A decode step with its workspace given allocates nothing, so it can be
    captured in a CUDA graph (launch-bound loops are replayed that way); the
    replayed step writes the same pools and outputs, bit for bit, as the eager
    call, and matches the oracle.  The 405B-shaped step (16 query heads per KV
    head) is two chained head-group passes and one combine."""
    if w is not syn.TINY:
        w = dataclasses.replace(w, name="graph_" + w.name, num_seqs=16)
    batch = scenarios.fixed_batch(w)
    B = len(batch.seq_lens)
    key_bits, val_bits = syn.token_kv_bits(w, B, sub=400_000)
    slots = _newest_slots(batch.block_tables, batch.seq_lens, w.block_size)
    k_ref, v_ref = batch.k_pool.copy(), batch.v_pool.copy()
    reshape_and_cache(k_ref, v_ref, key_bits, val_bits, slots)
    dev_e, dev_g = DeviceBatch(batch), DeviceBatch(batch)
    key, value = to_dev(key_bits, w.dtype), to_dev(val_bits, w.dtype)
    mx = int(batch.seq_lens.max())
    ws = pa.workspace_for(dev_g.q, dev_g.k_pool, dev_g.tables, mx)

    def step(dev, out):
        pa.pa_decode_append(out, dev.q, dev.k_pool, dev.v_pool, key, value, dev.tables, dev.lens,
                            w.scale, max_seq_len=mx, workspace=ws)

    eager = torch.empty_like(dev_e.q)
    step(dev_e, eager)
    torch.cuda.synchronize()
    out = torch.empty_like(dev_g.q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # warm-up outside the capture
        step(dev_g, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(dev_g, out)
    out.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    _pools_equal(dev_g, k_ref, v_ref)
    _pools_equal(dev_e, k_ref, v_ref)
    after = dataclasses.replace(batch, k_pool=k_ref, v_pool=v_ref)
    assert_close(widen(out), scenarios.decode_f64(after), f"graph replay {w.name}")
