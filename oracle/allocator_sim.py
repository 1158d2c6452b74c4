"""KV-cache allocator simulator (oracle side; test infrastructure, imported only
by the tests and the benchmark's CPU legs).

The tutorial's exercises §10 B and C ("10 — Paged Attention"): a contiguous
allocator and a paged allocator serve the same request stream (Poisson
arrivals, lognormal lengths); measure memory utilisation, allocation failures,
concurrency, internal fragmentation and block-table length, and sweep the block
size.  The pages give the goal, not the rules; the rules below are this
library's reading (each listed in the design notes), and the library's native
simulator follows the same rules.

Time advances in decode steps t = 0, 1, 2, ...  Each step:

1. arrivals: requests with arrival_step <= t join the back of the waiting queue;
2. admission: the head of the queue is admitted while its allocation succeeds
   (first come first served; the first failure ends admission for the step and
   counts one failed allocation).  An admitted request holds `len` tokens: its
   prompt, or after a preemption everything it had (the KV is recomputed);
3. growth: every request admitted in an earlier step, in admission order,
   appends one token.  Paged: when its blocks are full it needs one more block;
   if none is free, the request is preempted (one failed allocation, one
   preemption): its blocks are freed and it returns to the front of the waiting
   queue (requests preempted in the same step keep their admission order);
4. measurement: tokens stored (sum of len), memory held (contiguous: the sum of
   the reservations; paged: blocks held x block_size), running requests, and
   (paged) blocks per request;
5. completion: requests with len == prompt + output release their memory.

Contiguous allocator: one extent of `reserve` tokens in a linear space of
`capacity` token slots, taken first-fit (lowest address); freed extents merge
with free neighbours.  `reserve` is max_seq_len ("max"), the next power of two
of prompt + output ("pow2"), or exactly prompt + output ("exact").  Growth never
fails.  A failed admission while the free total would have covered the request
is counted as a fragmentation failure (external fragmentation).

Paged allocator: capacity // block_size blocks; admission needs
ceil(len / block_size) free blocks.  Any free block serves, so a fragmentation
failure cannot happen.

All results are integers (sums over steps), so two implementations of these
rules agree exactly.
"""
from __future__ import annotations

import dataclasses
from collections import deque
from typing import List, Tuple

CONTIGUOUS, PAGED = 0, 1
RESERVE_MAX, RESERVE_POW2, RESERVE_EXACT = 0, 1, 2


@dataclasses.dataclass
class SimResult:
    steps: int = 0
    completed: int = 0
    failed_allocations: int = 0
    fragmentation_failures: int = 0
    preemptions: int = 0
    max_concurrency: int = 0
    sum_concurrency: int = 0
    busy_steps: int = 0
    sum_stored: int = 0
    sum_held: int = 0
    peak_stored: int = 0
    peak_held: int = 0
    sum_table_len: int = 0
    max_table_len: int = 0


def next_pow2(x: int) -> int:
    p = 1
    while p < x:
        p *= 2
    return p


class FirstFit:
    """Free extents of a linear space, kept sorted by start address."""

    def __init__(self, capacity: int):
        self.free: List[Tuple[int, int]] = [(0, capacity)] if capacity > 0 else []

    def total_free(self) -> int:
        return sum(size for _, size in self.free)

    def allocate(self, size: int):
        for i, (start, length) in enumerate(self.free):
            if length >= size:
                if length == size:
                    del self.free[i]
                else:
                    self.free[i] = (start + size, length - size)
                return start
        return None

    def release(self, start: int, size: int) -> None:
        self.free.append((start, size))
        self.free.sort()
        merged: List[Tuple[int, int]] = []
        for s, n in self.free:
            if merged and merged[-1][0] + merged[-1][1] == s:
                merged[-1] = (merged[-1][0], merged[-1][1] + n)
            else:
                merged.append((s, n))
        self.free = merged


def simulate(arrival, prompt, output, allocator: int, capacity: int, block_size: int = 16,
             reserve: int = RESERVE_MAX, max_seq_len: int = 2048,
             max_steps: int = 10_000_000) -> SimResult:
    if allocator not in (CONTIGUOUS, PAGED) or reserve not in (RESERVE_MAX, RESERVE_POW2,
                                                                RESERVE_EXACT):
        raise ValueError("unknown allocator or reservation rule")
    if capacity < 0 or max_seq_len < 2 or max_steps < 0 or (allocator == PAGED and block_size <= 0):
        raise ValueError("invalid simulator configuration")
    n = len(arrival)
    arrival = [int(x) for x in arrival]
    prompt = [int(x) for x in prompt]
    output = [int(x) for x in output]
    for i in range(n):
        if prompt[i] < 1 or output[i] < 1 or prompt[i] + output[i] > max_seq_len:
            raise ValueError(f"request {i}: lengths outside [1, max_seq_len]")
        if i and arrival[i] < arrival[i - 1]:
            raise ValueError("arrival steps must not decrease")
    if allocator == PAGED:
        if max((-(-(p + o) // block_size) for p, o in zip(prompt, output)), default=0) > \
                capacity // block_size:
            raise ValueError("a request needs more blocks than the pool holds")
    elif n:
        total = [p + o for p, o in zip(prompt, output)]
        size = {RESERVE_MAX: [max_seq_len] * n, RESERVE_POW2: [next_pow2(x) for x in total],
                RESERVE_EXACT: total}[reserve]
        if max(size) > capacity:
            raise ValueError("a reservation exceeds the capacity")
    cur = list(prompt)                      # tokens held (or to hold) per request
    admitted = [-1] * n
    extent = [None] * n                     # contiguous: (start, size)
    blocks = [0] * n                        # paged: blocks held
    ff = FirstFit(capacity)
    free_blocks = capacity // block_size if allocator == PAGED else 0
    waiting: deque = deque()
    running: List[int] = []
    res = SimResult()
    nxt = 0
    t = 0

    def need_of(r: int) -> int:
        if allocator == PAGED:
            return -(-cur[r] // block_size)
        total = prompt[r] + output[r]
        return {RESERVE_MAX: max_seq_len, RESERVE_POW2: next_pow2(total),
                RESERVE_EXACT: total}[reserve]

    while res.completed < n:
        if t >= max_steps:
            break
        while nxt < n and arrival[nxt] <= t:
            waiting.append(nxt)
            nxt += 1
        # admission
        while waiting:
            r = waiting[0]
            need = need_of(r)
            if allocator == PAGED:
                ok = free_blocks >= need
                if ok:
                    free_blocks -= need
                    blocks[r] = need
            else:
                start = ff.allocate(need)
                ok = start is not None
                if ok:
                    extent[r] = (start, need)
                elif ff.total_free() >= need:
                    res.fragmentation_failures += 1
            if not ok:
                res.failed_allocations += 1
                break
            waiting.popleft()
            running.append(r)
            admitted[r] = t
        # growth
        preempted = []
        for r in list(running):
            if admitted[r] == t:
                continue
            if allocator == PAGED and cur[r] % block_size == 0:
                if free_blocks == 0:
                    res.failed_allocations += 1
                    res.preemptions += 1
                    free_blocks += blocks[r]
                    blocks[r] = 0
                    running.remove(r)
                    preempted.append(r)
                    continue
                free_blocks -= 1
                blocks[r] += 1
            cur[r] += 1
        for r in reversed(preempted):
            waiting.appendleft(r)
        # measurement
        if running:
            stored = sum(cur[r] for r in running)
            if allocator == PAGED:
                held = sum(blocks[r] for r in running) * block_size
                tl = [blocks[r] for r in running]
                res.sum_table_len += sum(tl)
                res.max_table_len = max(res.max_table_len, max(tl))
            else:
                held = sum(extent[r][1] for r in running)
            res.busy_steps += 1
            res.sum_stored += stored
            res.sum_held += held
            res.peak_stored = max(res.peak_stored, stored)
            res.peak_held = max(res.peak_held, held)
            res.sum_concurrency += len(running)
            res.max_concurrency = max(res.max_concurrency, len(running))
        # completion
        for r in list(running):
            if cur[r] == prompt[r] + output[r]:
                if allocator == PAGED:
                    free_blocks += blocks[r]
                    blocks[r] = 0
                else:
                    ff.release(*extent[r])
                    extent[r] = None
                running.remove(r)
                res.completed += 1
        t += 1
    res.steps = t
    return res
