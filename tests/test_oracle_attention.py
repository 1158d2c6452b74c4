"""Pins of the oracle's fp64 decode attention (CPU only).

The oracle is checked against things other than itself: PyTorch's
scaled_dot_product_attention over contiguous (unpaged) keys and values laid out
block by block without the oracle's address translation, a pure-Python brute
force, closed forms, and invariances under relabelling physical blocks and
forking."""
import math

import numpy as np
import pytest
import torch

import synthetic as syn
from oracle import scenarios
from oracle.attention import paged_decode_attention, storage_to_f64, token_slots
from oracle.brute import brute_decode_attention


def _blockwise_pool(tokens_k, tokens_v, tables, nb, bs, fill=np.nan):
    """Lay logical tokens out block by block: logical block i of a sequence
    occupies physical block table[i], rows 0.. in order (the page-table picture
    of the tutorial §1), without any per-token slot formula."""
    Hkv, D = tokens_k[0].shape[1:]
    kp = np.full((nb, bs, Hkv, D), fill)
    vp = np.full((nb, bs, Hkv, D), fill)
    for K, V, table in zip(tokens_k, tokens_v, tables):
        for i, blk in enumerate(table):
            chunk_k = K[i * bs:(i + 1) * bs]
            if len(chunk_k) == 0:
                break
            kp[blk, :len(chunk_k)] = chunk_k
            vp[blk, :len(chunk_k)] = V[i * bs:(i + 1) * bs]
    return kp, vp


def _random_case(seed, B=3, Hq=8, Hkv=2, D=16, bs=4, max_len=23):
    g = np.random.default_rng(seed)
    lens = g.integers(1, max_len + 1, size=B)
    nblk = [-(-int(L) // bs) for L in lens]
    nb = sum(nblk) + 3
    perm = g.permutation(nb)
    tables, at = [], 0
    mb = max(nblk) + 2
    pad = int(perm[-1])
    padded = np.full((B, mb), pad, dtype=np.int64)
    for b, n in enumerate(nblk):
        t = [int(x) for x in perm[at:at + n]]
        at += n
        tables.append(t)
        padded[b, :n] = t
    K = [g.standard_normal((int(L), Hkv, D)) for L in lens]
    V = [g.standard_normal((int(L), Hkv, D)) for L in lens]
    q = g.standard_normal((B, Hq, D))
    kp, vp = _blockwise_pool(K, V, tables, nb, bs)
    return dict(q=q, K=K, V=V, kp=kp, vp=vp, tables=padded, lens=lens, bs=bs,
                scale=1 / math.sqrt(D))


@pytest.mark.parametrize("seed", range(6))
def test_matches_library_attention_on_contiguous_kv(seed):
    c = _random_case(seed, Hq=8, Hkv=2 if seed % 2 else 8, D=16 if seed < 3 else 64)
    out = paged_decode_attention(c["q"], c["kp"], c["vp"], c["tables"], c["lens"], c["scale"])
    Hq = c["q"].shape[1]
    for b, L in enumerate(c["lens"]):
        G = Hq // c["K"][b].shape[1]
        k = torch.from_numpy(c["K"][b]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        v = torch.from_numpy(c["V"][b]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        q = torch.from_numpy(c["q"][b]).unsqueeze(1)           # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0),
            scale=float(np.float32(c["scale"])))[0, :, 0, :].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)


def test_brute_force_on_tiny_workload():
    batch = scenarios.fixed_batch(syn.TINY)
    out = scenarios.decode_f64(batch)
    dt = batch.dtype
    q = storage_to_f64(batch.q, dt).tolist()
    kp = storage_to_f64(batch.k_pool, dt).tolist()
    vp = storage_to_f64(batch.v_pool, dt).tolist()
    ref = np.array(brute_decode_attention(q, kp, vp, batch.block_tables.tolist(),
                                          batch.seq_lens.tolist(), float(np.float32(batch.scale)),
                                          batch.block_size))
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_random_gqa(seed):
    c = _random_case(100 + seed, B=2, Hq=6, Hkv=3, D=8, bs=2, max_len=9)
    out = paged_decode_attention(c["q"], c["kp"], c["vp"], c["tables"], c["lens"], c["scale"])
    ref = np.array(brute_decode_attention(c["q"].tolist(), c["kp"].tolist(), c["vp"].tolist(),
                                          c["tables"].tolist(), c["lens"].tolist(),
                                          float(np.float32(c["scale"])), c["bs"]))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_invariant_under_relabelling_physical_blocks():
    c = _random_case(7)
    out = paged_decode_attention(c["q"], c["kp"], c["vp"], c["tables"], c["lens"], c["scale"])
    nb = c["kp"].shape[0]
    perm = np.random.default_rng(99).permutation(nb)
    kp2 = np.empty_like(c["kp"])
    vp2 = np.empty_like(c["vp"])
    kp2[perm] = c["kp"]
    vp2[perm] = c["vp"]
    out2 = paged_decode_attention(c["q"], kp2, vp2, perm[c["tables"]], c["lens"], c["scale"])
    assert np.array_equal(out, out2)


def test_forked_sequences_share_blocks_and_outputs():
    c = _random_case(8, B=2)
    tables = c["tables"].copy()
    tables[1] = tables[0]                       # a fork: same physical blocks
    lens = c["lens"].copy()
    lens[1] = lens[0]
    q = c["q"].copy()
    q[1] = q[0]
    out = paged_decode_attention(q, c["kp"], c["vp"], tables, lens, c["scale"])
    assert np.array_equal(out[0], out[1])


def test_unused_slots_and_padding_are_not_read():
    c = _random_case(9)
    out_nan = paged_decode_attention(c["q"], c["kp"], c["vp"], c["tables"], c["lens"], c["scale"])
    kp = np.nan_to_num(c["kp"], nan=0.0)
    vp = np.nan_to_num(c["vp"], nan=0.0)
    out_zero = paged_decode_attention(c["q"], kp, vp, c["tables"], c["lens"], c["scale"])
    assert np.isfinite(out_nan).all()
    assert np.array_equal(out_nan, out_zero)


def test_length_one_returns_the_value_row():
    c = _random_case(10)
    lens = np.ones_like(c["lens"])
    out = paged_decode_attention(c["q"], c["kp"], c["vp"], c["tables"], lens, c["scale"])
    G = c["q"].shape[1] // c["kp"].shape[2]
    for b in range(len(lens)):
        for hq in range(c["q"].shape[1]):
            assert np.array_equal(out[b, hq], c["vp"][c["tables"][b, 0], 0, hq // G])


def test_constant_values_and_equal_keys():
    c = _random_case(11)
    G = c["q"].shape[1] // c["kp"].shape[2]
    vp = np.full_like(c["vp"], 0.375)
    out = paged_decode_attention(c["q"], c["kp"], vp, c["tables"], c["lens"], c["scale"])
    np.testing.assert_allclose(out, 0.375, rtol=1e-14)
    kp = np.ones_like(c["kp"])
    out = paged_decode_attention(c["q"], kp, c["vp"], c["tables"], c["lens"], c["scale"])
    for b, L in enumerate(c["lens"]):
        mean = c["V"][b].mean(axis=0)               # [Hkv, D], logical order
        for hq in range(c["q"].shape[1]):
            np.testing.assert_allclose(out[b, hq], mean[hq // G], rtol=1e-12, atol=1e-14)


def test_gqa_head_mapping_is_contiguous():
    """KV head h serves query heads h*G .. h*G+G-1 (the Llama grouping)."""
    c = _random_case(12, Hq=8, Hkv=2)
    vp = np.empty_like(c["vp"])
    vp[:, :, 0, :] = -1.0
    vp[:, :, 1, :] = 2.0
    out = paged_decode_attention(c["q"], c["kp"], vp, c["tables"], c["lens"], c["scale"])
    np.testing.assert_allclose(out[:, :4], -1.0, rtol=1e-14)
    np.testing.assert_allclose(out[:, 4:], 2.0, rtol=1e-14)


def test_two_keys_logistic_closed_form():
    """Two tokens: out = v0 * sigmoid(d) + v1 * (1 - sigmoid(d)), d = scale*(q.k0 - q.k1)."""
    D, bs = 8, 2
    g = np.random.default_rng(13)
    q = g.standard_normal((1, 1, D))
    K = g.standard_normal((2, 1, D))
    V = g.standard_normal((2, 1, D))
    kp, vp = _blockwise_pool([K], [V], [[1]], 3, bs)
    scale = 0.3
    sig = float(np.float32(scale))
    out = paged_decode_attention(q, kp, vp, np.array([[1]]), np.array([2]), scale)
    d = sig * (q[0, 0] @ K[0, 0] - q[0, 0] @ K[1, 0])
    w0 = 1.0 / (1.0 + math.exp(-d))
    np.testing.assert_allclose(out[0, 0], w0 * V[0, 0] + (1 - w0) * V[1, 0], rtol=1e-12)


def test_dominant_key_selects_its_value():
    c = _random_case(14, B=1, Hq=2, Hkv=2)
    L = int(c["lens"][0])
    j = L // 2
    kp = c["kp"].copy()
    slot = token_slots(c["tables"][0], L, c["bs"])[j]
    blk, row = divmod(int(slot), c["bs"])
    kp[blk, row] = c["q"][0] * 1e3              # q.k_j dominates by far more than 100
    out = paged_decode_attention(c["q"], kp, c["vp"], c["tables"], c["lens"], c["scale"])
    np.testing.assert_allclose(out[0], c["vp"][blk, row], rtol=1e-12, atol=1e-12)


def test_zero_length_gives_zero_row():
    c = _random_case(15)
    lens = c["lens"].copy()
    lens[1] = 0
    out = paged_decode_attention(c["q"], c["kp"], c["vp"], c["tables"], lens, c["scale"])
    assert not out[1].any()


def test_storage_widening_is_exact():
    vals = np.array([1.0, -2.5, 0.1, 65504.0, 1e-7], dtype=np.float32)
    h = vals.astype(np.float16)
    assert np.array_equal(storage_to_f64(h.view(np.uint16), syn.FLOAT16), h.astype(np.float64))
    bits = syn.fp32_to_storage_bits(vals, syn.BFLOAT16)
    back = storage_to_f64(bits, syn.BFLOAT16)
    # bf16 keeps 8 significant bits: relative rounding error at most 2^-9
    assert np.all(np.abs(back - vals) <= np.abs(vals) * 2.0 ** -9)
    assert storage_to_f64(np.array([0x3F80], np.uint16), syn.BFLOAT16)[0] == 1.0
