"""GPU parity of pa_decode against the fp64 oracle, through the C ABI.

Acceptance: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise (fp32
accumulation, fp16/bf16 storage; the output's own rounding is at most 2^-9
relative for bf16, 2^-11 for fp16, well inside the relative term).  Closed forms
whose exact result is representable are checked bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from oracle.attention import paged_decode_attention, storage_to_f64
from oracle.brute import brute_decode_attention
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


def test_tiny_workload_matches_oracle_and_brute_force(pa):
    needs(pa, syn.TINY.head_dim)
    batch = scenarios.fixed_batch(syn.TINY)
    dev = DeviceBatch(batch)
    got = widen(dev.decode(pa))
    ref = scenarios.decode_f64(batch)
    assert_close(got, ref, "tiny")
    dt = batch.dtype
    brute = np.array(brute_decode_attention(
        storage_to_f64(batch.q, dt).tolist(), storage_to_f64(batch.k_pool, dt).tolist(),
        storage_to_f64(batch.v_pool, dt).tolist(), batch.block_tables.tolist(),
        batch.seq_lens.tolist(), float(np.float32(batch.scale)), batch.block_size))
    assert_close(got, brute, "tiny vs brute force")


def test_llama3_8b_workload_all_rows(pa):
    batch = scenarios.fixed_batch(syn.LLAMA3_8B)
    dev = DeviceBatch(batch)
    got = widen(dev.decode(pa))
    assert_close(got, scenarios.decode_f64(batch), "llama3_8b")


@pytest.fixture(scope="module")
def long_context():
    return scenarios.fixed_batch(syn.LONG_CONTEXT, fill_all=True)


def test_long_context_full_size_sampled_rows(pa, long_context):
    """Full-size long-context batch in the benchmark's launch configuration
    (split-K 512 + combine); sampled rows against the oracle, all rows finite."""
    batch = long_context
    dev = DeviceBatch(batch)
    out = dev.decode(pa, partition_tokens=512)
    got = widen(out)
    assert np.isfinite(got).all()
    seqs = [0, 3, 6]
    heads = [0, 7, 8, 33, 63]
    ref = scenarios.decode_f64(batch, sequences=seqs, heads=heads)
    for b in seqs:
        assert_close(got[b, heads], ref[b, heads], f"long_context b={b}")


def _small(name, **kw):
    base = syn.WORKLOADS[name] if name in syn.WORKLOADS else syn.LLAMA3_8B
    return dataclasses.replace(base, **kw)


@pytest.mark.parametrize("dtype", [syn.FLOAT16, syn.BFLOAT16])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_shapes_with_ragged_tails(pa, dtype, head_dim, bs):
    needs(pa, head_dim)
    lens = [1, 2, bs - 1, bs, bs + 1, 127, 128, 129, 511, 512, 513, 1000, 1024, 1025, 1537]
    w = _small("llama3_8b", num_seqs=len(lens), dtype=dtype, head_dim=head_dim, block_size=bs,
               seed=1000 + bs + head_dim + dtype, length_kind="fixed", lens=tuple(lens),
               num_q_heads=8, num_kv_heads=2)
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    got = widen(dev.decode(pa))
    assert_close(got, scenarios.decode_f64(batch), f"dt={dtype} D={head_dim} bs={bs}")


# groupings the grouped kernel does not serve: 5 query heads per KV head with
# 3 KV heads (odd groups are built for passes of 4 or 8 KV heads only)
PER_HEAD_GROUPINGS = {(15, 3)}


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 8), (64, 8), (32, 2), (24, 3),
                                    (16, 1), (8, 1), (2, 2), (16, 2), (32, 32), (64, 32),
                                    (16, 16), (64, 16), (48, 16), (64, 4), (128, 8), (128, 32),
                                    (256, 16), (128, 128),
                                    (40, 8), (28, 4), (56, 8), (24, 8), (48, 8), (20, 4),
                                    (12, 4), (80, 16), (15, 3)])
def test_query_groupings(pa, hq, hkv):
    """Every grouping the grouped kernel instantiates (1 to 32 KV heads per block:
    multi-query, grouped and plain multi-head attention; 16 query heads per KV
    head; 3, 5, 6 or 7 query heads per KV head (40/8 and 28/4 heads, as in
    Qwen2.5-32B and Qwen2-7B); more than 64 query heads, served as passes over
    groups of KV heads) and one it does not."""
    lens = [3, 70, 600, 1300]
    w = _small("llama3_8b", num_seqs=4, num_q_heads=hq, num_kv_heads=hkv, length_kind="fixed",
               lens=tuple(lens), seed=77 + hq + hkv)
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    if pa.decode_path == "tc":
        kernel = pa.decode_kernel_for(dev.q, dev.k_pool, dev.tables, int(batch.seq_lens.max()))
        want = "per_head" if (hq, hkv) in PER_HEAD_GROUPINGS else "grouped"
        assert kernel == want, (hq, hkv, kernel)
    got = widen(dev.decode(pa))
    assert_close(got, scenarios.decode_f64(batch), f"Hq={hq} Hkv={hkv}")


@pytest.mark.parametrize("hq,hkv,bs", [(40, 8, 16), (28, 4, 64), (24, 8, 8), (48, 8, 32)])
def test_odd_query_groups_fp16(pa, hq, hkv, bs):
    """3, 5, 6 and 7 query heads per KV head in fp16 (the grouped kernel's other
    storage type), ragged lengths across block and tile edges."""
    lens = (1, bs - 1, bs + 1, 129, 700, 2049)
    w = _small("llama3_8b", num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv,
               block_size=bs, dtype=syn.FLOAT16, length_kind="fixed", lens=lens,
               seed=300 + hq + bs)
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    if pa.decode_path == "tc":
        assert pa.decode_kernel_for(dev.q, dev.k_pool, dev.tables, 2049) == "grouped"
    got = widen(dev.decode(pa))
    assert_close(got, scenarios.decode_f64(batch), f"fp16 Hq={hq} Hkv={hkv} bs={bs}")


@pytest.mark.parametrize("hkv,hq,bs,lens", [
    (8, 32, 16, (100,)),                 # fewer tiles than SMs: most CTAs idle
    (4, 16, 32, (128, 300)),
    (4, 4, 64, (513, 77)),
    (8, 64, 8, (1, 2, 3)),
    (8, 32, 16, tuple(range(1, 400, 7))),  # many short sequences per CTA
])
def test_small_and_many_short_batches(pa, hkv, hq, bs, lens):
    """Batches with fewer token tiles than SMs, and CTAs spanning many short
    sequences: the work split must still cover every token exactly once."""
    w = _small("llama3_8b", num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv, block_size=bs,
               length_kind="fixed", lens=tuple(lens), seed=31 + hq + bs)
    batch = scenarios.fixed_batch(w)
    got = widen(DeviceBatch(batch).decode(pa))
    assert_close(got, scenarios.decode_f64(batch), f"Hkv={hkv} Hq={hq} bs={bs} B={len(lens)}")


@pytest.mark.parametrize("pt", [128, 256, 512, 1024])
def test_partition_sizes(pa, pt):
    lens = [1, 127, 128, 129, 1024, 2049, 3000]
    w = _small("llama3_8b", num_seqs=len(lens), length_kind="fixed", lens=tuple(lens), seed=5 + pt)
    batch = scenarios.fixed_batch(w)
    got = widen(DeviceBatch(batch).decode(pa, partition_tokens=pt))
    assert_close(got, scenarios.decode_f64(batch), f"partition {pt}")


def test_zero_length_sequences_give_zero_rows(pa):
    w = _small("llama3_8b", num_seqs=4, length_kind="fixed", lens=(5, 1, 700, 3), seed=9)
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    lens = batch.seq_lens.copy()
    lens[1] = 0
    lens[3] = 0
    out = dev.decode(pa, lens=i32(lens), max_seq_len=int(lens.max()))
    got = widen(out)
    assert not got[1].any() and not got[3].any()
    ref = paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.block_tables, lens,
                                 batch.scale, dtype=batch.dtype)
    assert_close(got, ref, "zero-length rows")


def test_length_one_is_exact(pa):
    w = _small("llama3_8b", num_seqs=16, length_kind="fixed", lens=(1,) * 16, seed=11)
    batch = scenarios.fixed_batch(w)
    out = to_host_bits(DeviceBatch(batch).decode(pa))
    G = w.group
    for b in range(16):
        blk = batch.block_tables[b, 0]
        for hq in range(w.num_q_heads):
            assert np.array_equal(out[b, hq], batch.v_pool[blk, 0, hq // G])


def test_constant_values_and_equal_keys(pa):
    w = _small("llama3_8b", num_seqs=6, length_kind="fixed", lens=(9, 100, 513, 1024, 2000, 1),
               seed=12)
    batch = scenarios.fixed_batch(w)
    c = syn.fp32_to_storage_bits(np.float32(0.8125), w.dtype)
    batch.v_pool[...] = c
    out = widen(DeviceBatch(batch).decode(pa))
    assert np.all(out == 0.8125)
    batch = scenarios.fixed_batch(w)
    batch.k_pool[...] = syn.fp32_to_storage_bits(np.float32(0.5), w.dtype)
    got = widen(DeviceBatch(batch).decode(pa))
    assert_close(got, scenarios.decode_f64(batch), "equal keys (mean of V)")


def test_relabelled_blocks_give_identical_bits(pa):
    """Permuting physical block ids (pool and tables together) leaves the output
    bit-identical: no atomics, the reduction order depends on logical positions only."""
    w = _small("llama3_8b", num_seqs=8, length_kind="fixed",
               lens=(17, 300, 512, 777, 1500, 2048, 2600, 4096), seed=13)
    batch = scenarios.fixed_batch(w)
    out1 = to_host_bits(DeviceBatch(batch).decode(pa))
    out1b = to_host_bits(DeviceBatch(batch).decode(pa))
    assert np.array_equal(out1, out1b)
    perm = np.random.default_rng(3).permutation(batch.num_blocks)
    kp = np.empty_like(batch.k_pool)
    vp = np.empty_like(batch.v_pool)
    kp[perm] = batch.k_pool
    vp[perm] = batch.v_pool
    batch.k_pool, batch.v_pool = kp, vp
    batch.block_tables = perm[batch.block_tables].astype(np.int32)
    out2 = to_host_bits(DeviceBatch(batch).decode(pa))
    assert np.array_equal(out1, out2)


def test_forked_tables_give_identical_rows(pa):
    w = _small("llama3_8b", num_seqs=4, length_kind="fixed", lens=(1000, 1000, 40, 40), seed=14)
    batch = scenarios.fixed_batch(w)
    batch.block_tables[1] = batch.block_tables[0]
    batch.block_tables[3] = batch.block_tables[2]
    batch.q[1] = batch.q[0]
    batch.q[3] = batch.q[2]
    out = to_host_bits(DeviceBatch(batch).decode(pa))
    assert np.array_equal(out[0], out[1]) and np.array_equal(out[2], out[3])


def test_checked_mode_reports_bad_block_ids(pa):
    w = _small("llama3_8b", num_seqs=3, length_kind="fixed", lens=(40, 600, 33), seed=15)
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev.decode(pa, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tables = batch.block_tables.copy()
    tables[1, 3] = batch.num_blocks + 5          # outside the pool
    tables[2, 0] = -2
    dev.decode(pa, tables=i32(tables), max_seq_len=600, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    assert dev.guards_intact()


def test_too_long_sequence_is_reported_in_checked_mode(pa):
    w = _small("llama3_8b", num_seqs=2, length_kind="fixed", lens=(40, 60), seed=16)
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    lens = batch.seq_lens.copy()
    lens[0] = batch.block_tables.shape[1] * w.block_size + 7
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = dev.decode(pa, lens=i32(lens), max_seq_len=batch.block_tables.shape[1] * w.block_size,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    assert np.isfinite(widen(out)[1]).all()


def test_bad_arguments_raise(pa):
    needs(pa, syn.TINY.head_dim)
    batch = scenarios.fixed_batch(syn.TINY)
    dev = DeviceBatch(batch)
    with pytest.raises(pa.PagedAttnError):
        pa.pa_decode(torch.empty_like(dev.q), dev.q, dev.k_pool, dev.v_pool, dev.tables,
                     dev.lens, 0.125, max_seq_len=10_000)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError):
        pa.pa_decode(torch.empty_like(dev.q), dev.q, dev.k_pool, dev.v_pool, dev.tables,
                     dev.lens, 0.125, max_seq_len=64, workspace=ws)


def test_one_workspace_serves_a_sequence_of_batches(pa):
    """One workspace reused by consecutive decodes of different batches (many
    short sequences, then few long ones): nothing a call leaves in it affects the
    next, and a repeated batch gives identical bits."""
    w1 = dataclasses.replace(syn.LLAMA3_8B, num_seqs=64, lo=100, hi=1500)
    w2 = dataclasses.replace(syn.LLAMA3_8B, num_seqs=40, lo=500, hi=3000, seed=9)
    w3 = dataclasses.replace(syn.LLAMA3_8B, num_seqs=4, lo=3000, hi=9000, seed=10)
    batches = [scenarios.fixed_batch(w, fill_all=True) for w in (w1, w2, w3)]
    ws = pa.alloc_workspace(64, 32, 128, 9000)
    outs = []
    for batch in batches + batches[:1]:
        dev = DeviceBatch(batch)
        out = torch.empty_like(dev.q)
        pa.pa_decode(out, dev.q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, batch.scale,
                     max_seq_len=int(batch.seq_lens.max()), workspace=ws)
        torch.cuda.synchronize()
        rows = list(range(0, len(batch.seq_lens), 7))
        assert_close(widen(out)[rows], scenarios.decode_f64(batch, sequences=rows)[rows],
                     f"batch of {len(batch.seq_lens)}")
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[3].view(torch.int16))


@pytest.mark.parametrize("B,hi", [(1100, 300), (4000, 64)])
def test_large_batches(pa, B, hi):
    """Thousands of short sequences (continuous batching with many live
    requests): the grouped kernel serves them (each CTA's range meets dozens of
    sequences, most of them whole); checked on sampled rows and on every row of
    the sequences around CTA range boundaries' typical spacing."""
    w = _small("llama3_8b", num_seqs=B, length_kind="uniform", lo=1, hi=hi, seed=77 + B)
    batch = scenarios.fixed_batch(w, fill_all=True)
    dev = DeviceBatch(batch)
    if pa.decode_path == "tc":
        assert pa.decode_kernel_for(dev.q, dev.k_pool, dev.tables,
                                    int(batch.seq_lens.max())) == "grouped"
    got = widen(dev.decode(pa))
    rows = sorted(set(list(range(0, B, 37)) + list(range(B // 2, B // 2 + 40)) + [B - 1]))
    assert_close(got[rows], scenarios.decode_f64(batch, sequences=rows)[rows], f"B={B}")


@pytest.mark.parametrize("hq,hkv,bs", [(32, 32, 16), (32, 32, 8), (8, 1, 32), (64, 16, 64)])
def test_more_kv_heads_per_block_ragged(pa, hq, hkv, bs):
    """Many KV heads per block mean few tokens per 128-row tile (4 for 32 heads),
    so tiles split blocks; one KV head means a tile spans up to 16 blocks."""
    w = _small("llama3_8b", num_seqs=6, num_q_heads=hq, num_kv_heads=hkv, block_size=bs,
               length_kind="fixed", lens=(1, 5, 129, 700, 2049, 33), seed=5 + hq + bs)
    batch = scenarios.fixed_batch(w)
    got = widen(DeviceBatch(batch).decode(pa))
    assert_close(got, scenarios.decode_f64(batch), f"Hq={hq} Hkv={hkv} bs={bs}")


def test_workspace_of_exactly_the_grouped_kernels_size(pa):
    """The grouped kernel's workspace is its stream-K area only (tile and weight
    prefixes, the start weight, per-CTA (max, sum) and accumulators of up to 160
    CTAs x 2 segments), whatever the lengths: pa_decode runs with exactly that
    many bytes and refuses one fewer; the result matches the oracle."""
    if pa.decode_path != "tc":
        pytest.skip("the grouped kernel's layout")
    w = syn.LLAMA3_8B.__class__(**{**syn.LLAMA3_8B.__dict__, "num_seqs": 12, "hi": 1500,
                                   "seed": 77})
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    B, Hq, D = dev.q.shape
    max_len = int(batch.seq_lens.max())
    n = pa.pa_decode_workspace_bytes_for(B, Hq, w.num_kv_heads, D, w.block_size,
                                         dev.tables.shape[1], batch.num_blocks, max_len, 1)
    parts = 160 * 2 * Hq
    assert n == (-(-4 * (B + 1) // 256) * 256) + (-(-4 * (B + 2) // 256) * 256) + \
        2 * (-(-4 * parts // 256) * 256) + (-(-4 * parts * D // 256) * 256)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev.q)
    pa.pa_decode(out, dev.q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, batch.scale,
                 max_seq_len=max_len, workspace=ws)
    torch.cuda.synchronize()
    assert_close(widen(out), scenarios.decode_f64(batch), "exact grouped workspace")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode(out, dev.q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, batch.scale,
                     max_seq_len=max_len, workspace=ws[:n - 256])
    assert e.value.status == 3


@pytest.mark.parametrize("B", [10000, 20000])
def test_ten_thousands_of_tiny_sequences(pa, B):
    """10,000 and 20,000 sequences of 1-8 tokens: each CTA's range meets ~66 or
    ~130 sequences (the grouped kernel's shared-memory window), most CTA
    boundaries fall between sequences; sampled rows against the oracle, every
    row finite."""
    if pa.decode_path == "simt":
        pytest.skip("the grouped kernel's window; the CUDA-core kernel is covered elsewhere")
    w = _small("llama3_8b", num_seqs=B, length_kind="uniform", lo=1, hi=8, seed=4242 + B)
    batch = scenarios.fixed_batch(w, fill_all=True)
    dev = DeviceBatch(batch)
    if pa.decode_path == "tc":
        assert pa.decode_kernel_for(dev.q, dev.k_pool, dev.tables, 8) == "grouped"
    got = widen(dev.decode(pa, max_seq_len=8))
    assert np.isfinite(got).all()
    mid = B // 2
    rows = sorted(set(list(range(0, B, 97)) + list(range(mid - 10, mid + 30)) + [B - 1]))
    assert_close(got[rows], scenarios.decode_f64(batch, sequences=rows)[rows], f"B={B}")


@pytest.mark.parametrize("hq,hkv,lens", [
    (32, 8, (60000,)),                    # one sequence over every CTA
    (32, 8, (20000, 100, 9000)),          # two sequences over dozens of CTAs each
    (128, 8, (30000, 7)),                 # 16 query heads per KV head: two passes
    (64, 8, (3000,) * 40),                # parts of up to 5 CTAs, most CTAs cut two
])
def test_sequences_cut_into_many_parts(pa, hq, hkv, lens):
    """Sequences cut into many parts by the grouped kernel's split (a CTA's
    share is ~W / 152 tiles), merged by the combine kernel: every row against
    the oracle, and a second call with the same workspace gives identical bits."""
    w = _small("llama3_8b", num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv,
               length_kind="fixed", lens=tuple(lens), seed=900 + hq + len(lens))
    batch = scenarios.fixed_batch(w)
    dev = DeviceBatch(batch)
    max_len = int(batch.seq_lens.max())
    ws = pa.workspace_for(dev.q, dev.k_pool, dev.tables, max_len)
    outs = []
    for _ in range(2):
        out = torch.empty_like(dev.q)
        pa.pa_decode(out, dev.q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, batch.scale,
                     max_seq_len=max_len, workspace=ws)
        torch.cuda.synchronize()
        outs.append(out)
    assert_close(widen(outs[0]), scenarios.decode_f64(batch), f"Hq={hq} lens={lens[:3]}")
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_one_workspace_serves_every_kernel_in_turn():
    """One workspace passed to every decode kernel in turn, over batches with
    different cuts: nothing a call leaves in it affects the next call, whichever
    kernel either runs."""
    pa = lib()
    w1 = dataclasses.replace(syn.LLAMA3_8B, num_seqs=24, lo=100, hi=4000, seed=61)
    w2 = dataclasses.replace(syn.LLAMA3_8B, num_seqs=7, lo=2000, hi=9000, seed=62)
    batches = [scenarios.fixed_batch(w) for w in (w1, w2)]
    ws = pa.alloc_workspace(24, 32, 128, 9000)
    try:
        for path in ("tc", "simt", "tc", "tc_head", "tc", "tc"):
            pa.set_decode_path(path)
            for batch in batches:
                dev = DeviceBatch(batch)
                out = torch.empty_like(dev.q)
                pa.pa_decode(out, dev.q, dev.k_pool, dev.v_pool, dev.tables, dev.lens,
                             batch.scale, max_seq_len=int(batch.seq_lens.max()), workspace=ws)
                torch.cuda.synchronize()
                assert_close(widen(out), scenarios.decode_f64(batch),
                             f"{path}, batch of {len(batch.seq_lens)}")
    finally:
        pa.set_decode_path("auto")


def test_short_sequences_beside_one_very_long_sequence():
    """700 one-token sequences ahead of one 3.2M-token sequence (32/8 heads, bs
    16): with one unit of weight per sequence start, the first CTA's equal share
    of the grouped kernel's split would meet ~660 sequences, more than the 640
    its window holds; the kernel raises the start weight for such batches.
    Closed forms check the result: a one-token sequence's output is its V row,
    bit for bit; with every key zero the long sequence's weights are uniform, so
    its output is the mean of its V rows (fp64, on the CPU)."""
    pa = lib()
    n_short, L, Hq, Hkv, D, bs = 700, 3_200_000, 32, 8, 128, 16
    nb_long = L // bs
    NB = nb_long + n_short + 1
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = nb_long + n_short                 # 16 tokens per 128-row tile
    assert (-(-(tiles + n_short + 1) // min(grid, 160))) // 2 > 640
    rng = np.random.default_rng(4711)
    tables = np.full((n_short + 1, nb_long), NB - 1, np.int32)
    tables[:n_short, 0] = nb_long + rng.permutation(n_short)
    tables[n_short] = rng.permutation(nb_long)
    lens = np.array([1] * n_short + [L], np.int32)
    g = torch.Generator(device="cuda")
    g.manual_seed(4711)
    k_pool = torch.zeros((NB, bs, Hkv, D), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.empty((NB, bs, Hkv, D), dtype=torch.bfloat16, device="cuda")
    for i in range(0, NB, 20000):
        n = min(20000, NB - i)
        v_pool[i:i + n] = torch.randn((n, bs, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((n_short + 1, Hq, D), generator=g, device="cuda").to(torch.bfloat16)
    t_dev, l_dev = i32(tables), i32(lens)
    pa.set_decode_path("tc")
    try:
        assert pa.decode_kernel_for(q, k_pool, t_dev, L) == "grouped"
        out = torch.empty_like(q)
        pa.pa_decode(out, q, k_pool, v_pool, t_dev, l_dev, D ** -0.5, max_seq_len=L)
        torch.cuda.synchronize()
    finally:
        pa.set_decode_path("auto")
    got = to_host_bits(out)
    rows = to_host_bits(v_pool[nb_long:nb_long + n_short, 0])        # [n_short, Hkv, D]
    want = rows[tables[:n_short, 0] - nb_long].repeat(Hq // Hkv, axis=1)
    assert np.array_equal(got[:n_short], want)
    total = torch.zeros((Hkv, D), dtype=torch.float64)
    for i in range(0, nb_long, 20000):
        total += v_pool[i:min(nb_long, i + 20000)].cpu().double().sum(dim=(0, 1))
    mean = (total / L).numpy().repeat(Hq // Hkv, axis=0)
    assert_close(widen(out)[n_short], mean, "long sequence: mean of its V rows")
