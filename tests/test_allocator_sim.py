"""Allocator simulator: the oracle's rules pinned by hand-worked traces and
closed forms, the native simulator (pa_sim_run) equal to the oracle on every
counter, and the tutorial's utilisation finding reproduced (CPU only)."""
import dataclasses

import numpy as np
import pytest

import synthetic as syn
from oracle.allocator_sim import (CONTIGUOUS, PAGED, RESERVE_EXACT, RESERVE_MAX, RESERVE_POW2,
                                  SimResult, simulate)


def _r(**kw):
    return dataclasses.replace(SimResult(), **kw)


def test_single_paged_request_by_hand():
    """P=5, O=3, block 4: admitted at t=0 with 2 blocks (5 stored, 8 held), then
    6, 7, 8 tokens in the same 2 blocks; finishes after step 3."""
    got = simulate([0], [5], [3], PAGED, capacity=16, block_size=4, max_seq_len=32)
    assert got == _r(steps=4, completed=1, max_concurrency=1, sum_concurrency=4, busy_steps=4,
                     sum_stored=5 + 6 + 7 + 8, sum_held=4 * 8, peak_stored=8, peak_held=8,
                     sum_table_len=8, max_table_len=2)


def test_contiguous_external_fragmentation_by_hand():
    """A(3+1), B(2+3), C(2+1) fill 12 slots as [0,4) [4,9) [9,12).  D(5+1)
    arrives at t=1: no room (t=1), then 7 free slots in two holes of 4 and 3
    (t=2, t=3: fragmentation failures), admitted at t=4 when B's extent merges
    the holes."""
    got = simulate([0, 0, 0, 1], [3, 2, 2, 5], [1, 3, 1, 1], CONTIGUOUS, capacity=12,
                   reserve=RESERVE_EXACT, max_seq_len=12)
    assert got == _r(steps=6, completed=4, failed_allocations=3, fragmentation_failures=2,
                     max_concurrency=3, sum_concurrency=3 + 3 + 1 + 1 + 1 + 1, busy_steps=6,
                     sum_stored=7 + 10 + 4 + 5 + 5 + 6, sum_held=12 + 12 + 5 + 5 + 6 + 6,
                     peak_stored=10, peak_held=12)


def test_paged_preemption_by_hand():
    """Two blocks of 4.  A(4+2) and B(4+1) take one each; at t=1 A needs a block
    first and finds none: preempted (its block goes to B, which finishes); A is
    readmitted at t=2 with one block, grows into a second at t=3, done at t=4."""
    got = simulate([0, 0], [4, 4], [2, 1], PAGED, capacity=8, block_size=4, max_seq_len=8)
    assert got == _r(steps=5, completed=2, failed_allocations=1, preemptions=1,
                     max_concurrency=2, sum_concurrency=2 + 1 + 1 + 1 + 1, busy_steps=5,
                     sum_stored=8 + 5 + 4 + 5 + 6, sum_held=8 + 8 + 4 + 8 + 8, peak_stored=8,
                     peak_held=8, sum_table_len=2 + 2 + 1 + 2 + 2, max_table_len=2)


def test_reservations_and_block_size_one():
    """Closed forms on a random stream: block size 1 wastes nothing (held ==
    stored); with unlimited memory the contiguous reservations are exactly
    max_seq_len / next power of two / prompt + output per running request."""
    a, p, o = syn.request_arrays(syn.SMALL_STREAM)
    s = syn.SMALL_STREAM
    r1 = simulate(a, p, o, PAGED, capacity=10**6, block_size=1, max_seq_len=s.max_seq_len)
    assert r1.sum_held == r1.sum_stored and r1.failed_allocations == 0
    assert r1.sum_table_len == r1.sum_stored
    big = 10**7
    for rule, size in ((RESERVE_MAX, lambda t: s.max_seq_len),
                       (RESERVE_POW2, lambda t: 1 << (int(t) - 1).bit_length()),
                       (RESERVE_EXACT, lambda t: int(t))):
        r = simulate(a, p, o, CONTIGUOUS, capacity=big, reserve=rule, max_seq_len=s.max_seq_len)
        # without memory pressure request i runs steps arrival_i .. arrival_i + o_i
        assert r.failed_allocations == 0 and r.completed == len(a)
        assert r.sum_held == sum(size(pi + oi) * (oi + 1) for pi, oi in zip(p, o))
        assert r.sum_stored == sum(sum(pi + k for k in range(oi + 1)) for pi, oi in zip(p, o))


def test_reproduces_the_utilisation_gap():
    """The tutorial's §7 table: contiguous KV memory utilisation 20-38%, paged
    96%+, and 2.5-4x the concurrent sequences, on a saturated serving stream."""
    a, p, o = syn.request_arrays(syn.SERVING_STREAM)
    cap = 26777 * 16          # the tutorial's §6 pool: 26,777 blocks of 16 tokens
    c = simulate(a, p, o, CONTIGUOUS, capacity=cap, reserve=RESERVE_MAX, max_seq_len=2048)
    g = simulate(a, p, o, PAGED, capacity=cap, block_size=16, max_seq_len=2048)
    assert 0.20 <= c.sum_stored / c.sum_held <= 0.38
    assert g.sum_stored / g.sum_held >= 0.96
    assert 2.5 <= g.max_concurrency / c.max_concurrency <= 4.0


def test_invalid_requests_rejected():
    with pytest.raises(ValueError):
        simulate([0], [0], [3], PAGED, capacity=16, block_size=4)
    with pytest.raises(ValueError):
        simulate([1, 0], [2, 2], [1, 1], PAGED, capacity=16, block_size=4)
    with pytest.raises(ValueError):
        simulate([0], [10], [10], PAGED, capacity=16, block_size=4, max_seq_len=32)


@pytest.fixture(scope="module")
def native():
    from paged_kv_cache_301_gb300 import build
    build.build()
    import paged_kv_cache_301_gb300 as pa
    return pa


CASES = [("contiguous", "max", 16), ("contiguous", "pow2", 16), ("contiguous", "exact", 16)] + \
    [("paged", "max", bs) for bs in (1, 8, 16, 32, 64, 128)]


@pytest.mark.parametrize("allocator,reserve,bs", CASES)
@pytest.mark.parametrize("stream,cap", [(syn.SMALL_STREAM, 2048), (syn.SMALL_STREAM, 9000),
                                        (syn.SERVING_STREAM, 26777 * 16)])
def test_native_simulator_matches_oracle(native, allocator, reserve, bs, stream, cap):
    if stream is syn.SERVING_STREAM and bs not in (16, 128) and allocator == "paged":
        pytest.skip("the full sweep runs in the benchmark")
    a, p, o = syn.request_arrays(stream)
    want = simulate(a, p, o, CONTIGUOUS if allocator == "contiguous" else PAGED, capacity=cap,
                    block_size=bs, max_seq_len=stream.max_seq_len,
                    reserve={"max": RESERVE_MAX, "pow2": RESERVE_POW2, "exact": RESERVE_EXACT}[reserve])
    got = native.simulate_allocator(a, p, o, allocator, cap, block_size=bs, reserve=reserve,
                                    max_seq_len=stream.max_seq_len)
    assert {k: got[k] for k in dataclasses.asdict(want)} == dataclasses.asdict(want)


def test_native_simulator_rejects_bad_input(native):
    with pytest.raises(native.PagedAttnError):
        native.simulate_allocator([0], [0], [3], "paged", 16, block_size=4)
    with pytest.raises(native.PagedAttnError):
        native.simulate_allocator([0], [30], [3], "contiguous", 16, reserve="exact",
                                  max_seq_len=64)
    r = native.simulate_allocator([0, 0], [4, 4], [2, 1], "paged", 8, block_size=4,
                                  max_seq_len=8, max_steps=2)
    assert r["steps"] == 2 and r["completed"] == 1
