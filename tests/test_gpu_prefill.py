"""GPU parity of pa_prefill (causal multi-query attention over the paged pool)
against the fp64 oracle: every row on small batches that span several query and
key tiles with ragged tails, sampled rows at the benchmark sizes, and the
properties that hold at any size (causality, determinism, one query = decode)."""
import dataclasses

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from tests.gpu_helpers import DeviceBatch, assert_close, i32, lib, to_dev, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["auto", "simt"])
def pa(request):
    """Every test runs on the default choice (the tensor-core kernel where it
    serves the shape) and on the CUDA-core kernel."""
    m = lib()
    m.set_prefill_path(request.param)
    m.prefill_path = request.param
    yield m
    m.set_prefill_path("auto")


def _run(pa, pb, dev=None, status=None, max_q_len=None):
    b = pb.batch
    dev = dev or DeviceBatch(b)
    q = to_dev(pb.q, b.dtype)
    out = torch.full_like(q, float("nan"))
    n = np.diff(pb.q_start)
    pa.pa_prefill(out, q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, i32(pb.q_start),
                  b.scale, max_q_len=int(n.max()) if max_q_len is None else max_q_len,
                  status=status)
    return out, dev


def _small(G, bs, dtype, lens, hkv=2):
    return dataclasses.replace(syn.PREFILL, name=f"pf_g{G}_bs{bs}", num_seqs=len(lens),
                               length_kind="fixed", lens=tuple(lens), num_kv_heads=hkv,
                               num_q_heads=hkv * G, block_size=bs, dtype=dtype)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8, 16])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_whole_prompts_every_row(pa, G, bs):
    """Lengths that end mid-block, mid-tile and exactly on tile edges; every query
    group the tensor-core kernel serves (with 3, 5, 6 or 7 query heads per KV
    head a 128-row tile holds 42, 25, 21 or 18 query tokens)."""
    w = _small(G, bs, syn.BFLOAT16, [1, 127, 128, 300, 37])
    pb = scenarios.prefill_batch(w)
    out, dev = _run(pa, pb)
    torch.cuda.synchronize()
    assert_close(widen(out), scenarios.prefill_f64(pb), f"G={G} bs={bs}")
    assert dev.guards_intact()


@pytest.mark.parametrize("dtype", [syn.FLOAT16, syn.BFLOAT16])
@pytest.mark.parametrize("q_counts", [(5, 1, 200, 0, 64), (1, 1, 1, 1, 1), (17, 33, 129, 3, 70)])
def test_chunks_over_cached_prefix_every_row(pa, dtype, q_counts):
    """The last n tokens of each sequence attend to the whole cached prefix plus
    themselves; n = 0 leaves a sequence out, n = 1 is a decode step."""
    w = _small(4, 16, dtype, [700, 33, 1000, 90, 70], hkv=4)
    pb = scenarios.prefill_batch(w, q_counts=q_counts)
    out, _ = _run(pa, pb)
    torch.cuda.synchronize()
    assert_close(widen(out), scenarios.prefill_f64(pb), f"chunks {q_counts}")


def test_one_query_matches_decode(pa):
    w = _small(4, 16, syn.BFLOAT16, [700, 33, 1000, 90, 1], hkv=8)
    pb = scenarios.prefill_batch(w, q_counts=(1, 1, 1, 1, 1))
    out, dev = _run(pa, pb)
    dec = torch.empty_like(out)
    pa.pa_decode(dec, to_dev(pb.q, w.dtype), dev.k_pool, dev.v_pool, dev.tables, dev.lens,
                 w.scale, max_seq_len=1000)
    torch.cuda.synchronize()
    ref = scenarios.prefill_f64(pb)
    assert_close(widen(out), ref, "prefill n=1")
    assert_close(widen(dec), ref, "decode")


def test_causal_mask_ignores_later_tokens(pa):
    """Overwriting the K/V of each sequence's last token with a large value
    changes only the last row of that sequence; every earlier row, for which the
    token lies past its position, stays bit-identical (masked keys weigh exactly
    zero)."""
    w = _small(4, 16, syn.BFLOAT16, [300, 129, 64], hkv=2)
    pb = scenarios.prefill_batch(w)
    out1, dev = _run(pa, pb)
    b = pb.batch
    for s, L in enumerate(b.seq_lens):
        slot = int(b.block_tables[s][(L - 1) // b.block_size]) * b.block_size + (L - 1) % b.block_size
        dev.k_pool.view(-1, w.num_kv_heads, w.head_dim)[slot] = 3.0e4
        dev.v_pool.view(-1, w.num_kv_heads, w.head_dim)[slot] = 3.0e4
    out2, _ = _run(pa, pb, dev=dev)
    torch.cuda.synchronize()
    last = sorted(int(x) - 1 for x in pb.q_start[1:])
    keep = [r for r in range(out1.shape[0]) if r not in set(last)]
    assert torch.equal(out1[keep].view(torch.int16), out2[keep].view(torch.int16))
    assert not torch.equal(out1[last].view(torch.int16), out2[last].view(torch.int16))


def test_deterministic_and_bad_input_reported(pa):
    w = _small(8, 32, syn.BFLOAT16, [500, 260], hkv=4)
    pb = scenarios.prefill_batch(w)
    a, dev = _run(pa, pb)
    c, _ = _run(pa, pb, dev=dev)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    # more queries than tokens in sequence 1: reported, its rows untouched (NaN)
    bad = dataclasses.replace(pb, q_start=np.array([0, 500, 761], dtype=np.int32),
                              q=np.concatenate([pb.q, pb.q[:1]]))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(pa, bad, dev=dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    assert torch.isnan(out[500:].float()).all()
    assert torch.equal(out[:500].view(torch.int16), a[:500].view(torch.int16))


@pytest.mark.parametrize("dtype", [syn.FLOAT16, syn.BFLOAT16])
@pytest.mark.parametrize("head_dim,hq,hkv", [(64, 4, 4), (64, 12, 4), (128, 24, 2), (128, 40, 4),
                                             (128, 6, 2), (128, 40, 8)])
def test_other_shapes_every_row(pa, dtype, head_dim, hq, hkv):
    """head_dim 64, query groups of 10 and 12 (the CUDA-core kernel), and groups of
    3 and 5 in fp16 and bf16."""
    w = dataclasses.replace(syn.PREFILL, name="pf_other", num_seqs=4, length_kind="fixed",
                            lens=(1, 70, 200, 33), num_q_heads=hq, num_kv_heads=hkv,
                            head_dim=head_dim, block_size=16, dtype=dtype)
    pb = scenarios.prefill_batch(w, q_counts=(1, 70, 50, 10))
    out, dev = _run(pa, pb)
    torch.cuda.synchronize()
    assert_close(widen(out), scenarios.prefill_f64(pb), f"D={head_dim} Hq={hq} Hkv={hkv}")
    assert dev.guards_intact()


def test_forcing_tensor_cores_on_other_shapes_is_refused(pa):
    w = dataclasses.replace(syn.PREFILL, name="pf_d64", num_seqs=1, length_kind="fixed",
                            lens=(10,), num_q_heads=4, num_kv_heads=2, head_dim=64)
    pb = scenarios.prefill_batch(w)
    dev = DeviceBatch(pb.batch)
    q = to_dev(pb.q, w.dtype)
    out = torch.empty_like(q)
    pa.set_prefill_path("tc")
    try:
        with pytest.raises(pa.PagedAttnError) as ei:
            pa.pa_prefill(out, q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, i32(pb.q_start),
                          w.scale, max_q_len=10)
        assert ei.value.status == 2
    finally:
        pa.set_prefill_path(pa.prefill_path)


@pytest.mark.parametrize("w", [syn.PREFILL, syn.CHUNKED_PREFILL], ids=lambda w: w.name)
def test_benchmark_workloads_sampled_rows(pa, w):
    """Full size, in the launch configuration the benchmark times; the oracle
    checks 48 rows spread over every sequence, first and last rows included."""
    pb = scenarios.prefill_batch(w)
    out, dev = _run(pa, pb)
    torch.cuda.synchronize()
    g = np.random.default_rng(9)
    rows = set(int(x) for x in pb.q_start[:-1]) | set(int(x) - 1 for x in pb.q_start[1:])
    rows |= set(int(x) for x in g.integers(0, int(pb.q_start[-1]), size=48 - len(rows)))
    rows = sorted(rows)
    ref = scenarios.prefill_f64(pb, rows=rows)
    assert_close(widen(out)[rows], ref[rows], w.name)
    assert dev.guards_intact()


@pytest.mark.parametrize("scale", [0.25, 1.0])
def test_sharp_attention_every_row(pa, scale):
    """Large softmax scales concentrate each row's weight on a few keys anywhere
    in the sequence (logit spread 2.8 and 11): the rows where a single rounding
    of P would break the tolerance."""
    w = dataclasses.replace(_small(4, 16, syn.BFLOAT16, [700, 300, 129], hkv=2))
    pb = scenarios.prefill_batch(w)
    b = pb.batch
    dev = DeviceBatch(b)
    q = to_dev(pb.q, w.dtype)
    out = torch.empty_like(q)
    pa.pa_prefill(out, q, dev.k_pool, dev.v_pool, dev.tables, dev.lens, i32(pb.q_start), scale,
                  max_q_len=700)
    torch.cuda.synchronize()
    from oracle.prefill import paged_prefill_attention
    ref = paged_prefill_attention(pb.q, b.k_pool, b.v_pool, b.block_tables, b.seq_lens,
                                  pb.q_start, scale, dtype=b.dtype)
    assert_close(widen(out), ref, f"scale {scale}")


def test_bad_block_id_reported_and_read_as_zeros(pa):
    """Checked mode: a table entry outside the pool is reported; the kernel reads
    zeros there (never outside the pool), so the other sequences are unaffected."""
    w = _small(4, 16, syn.BFLOAT16, [200, 90], hkv=2)
    pb = scenarios.prefill_batch(w)
    b = pb.batch
    good, dev = _run(pa, pb)
    tables = b.block_tables.copy()
    tables[0, 3] = b.num_blocks + 100
    bad = dataclasses.replace(pb, batch=dataclasses.replace(b, block_tables=tables))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev.tables = i32(tables)
    out, _ = _run(pa, bad, dev=dev, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    assert torch.equal(out[200:].view(torch.int16), good[200:].view(torch.int16))
    assert torch.isfinite(out[:200].float()).all()


def test_many_sequences(pa):
    """300 sequences with 1-40 query tokens each over contexts of up to 600."""
    g = np.random.default_rng(5)
    lens = tuple(int(x) for x in g.integers(1, 600, size=300))
    w = dataclasses.replace(syn.PREFILL, name="pf_many", num_seqs=300, length_kind="fixed",
                            lens=lens, num_q_heads=32, num_kv_heads=8)
    q_counts = tuple(int(min(L, c)) for L, c in zip(lens, g.integers(1, 41, size=300)))
    pb = scenarios.prefill_batch(w, q_counts=q_counts)
    out, _ = _run(pa, pb)
    torch.cuda.synchronize()
    rows = sorted(set(int(x) for x in g.integers(0, int(pb.q_start[-1]), size=60)))
    assert_close(widen(out)[rows], scenarios.prefill_f64(pb, rows=rows)[rows], "B=300")
