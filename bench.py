"""Benchmark: one decode step of paged attention per timed step, on GB300.

A step is the whole hot path over one batch: copy-on-write block copies when
the workload shares blocks (pa_copy_blocks), the cache write of each sequence's
newest token at the slot its block table gives (pa_append_tokens: the slot
translation and reshape_and_cache in one launch), and decode attention over the
paged pool (pa_decode: split-K main kernel + combine).  Inputs are synthetic and seeded; the pool is
resident in HBM before timing starts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (the path has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and decode tokens/s, 1 GPU"
L2_BYTES = 126 * 2**20
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------
# workload description shared by both arms
# ----------------------------------------------------------------------------

def workload(name: str, block_size: int | None):
    w = syn.WORKLOADS[name]
    if block_size:
        w = w.with_block_size(block_size)
    return w


def kv_bytes(lens, w) -> int:
    """Algorithmic K+V bytes one decode reads: every token once per KV head."""
    return int(np.sum(lens)) * w.num_kv_heads * w.head_dim * 2 * w.elem_bytes


def decode_bytes(lens, w, max_blocks) -> int:
    """Algorithmic bytes of one pa_decode launch: K/V once per KV head, q read,
    out written, the table entries of every block used, seq_lens."""
    B = len(lens)
    qo = 2 * B * w.num_q_heads * w.head_dim * w.elem_bytes
    blocks = int(np.sum([-(-int(L) // w.block_size) for L in lens]))
    return kv_bytes(lens, w) + qo + 4 * blocks + 4 * B


def slowest_rank(times_ms, world, device):
    """Max over ranks of each timing (every rank replicates the workload, so the
    job takes as long as its slowest rank)."""
    if world <= 1:
        return list(times_ms)
    import torch
    t = torch.tensor(times_ms, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_rank_step, world, ms_per_step):
    """Whole-job throughput: the K/V bytes all ranks processed per step over the
    (slowest-rank) step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_uuid(torch, dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ----------------------------------------------------------------------------
# native arm
# ----------------------------------------------------------------------------

# The device code of the grouped decode kernel: its template, the parameter
# struct it reads, and the device headers it includes (host-side launch code is
# left out, so a change there keeps the recorded counters).
DECODE_KERNEL_TEXT = (
    ("pa_decode_tcg.cu", "__device__ __forceinline__ int clamp_len", "// Merge the partials"),
    ("pa_internal.h", "struct DecodeParams {", "};"),
    ("pa_common.cuh", None, None),
    ("pa_sm100.cuh", None, None),
)


def kernel_sources_sha() -> str:
    csrc = os.path.join(ROOT, "paged_kv_cache_301_gb300", "csrc")
    h = hashlib.sha256()
    for f, start, end in DECODE_KERNEL_TEXT:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        if start is not None:
            i = text.index(start)
            text = text[i:text.index(end, i) + len(end)]
        h.update(text.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str, kernel: str):
    """DRAM bytes per launch of the grouped decode kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if kernel != "tcg" or not os.path.exists(p):
        return None
    sha = kernel_sources_sha()
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == workload_name and parts[1] == sha:
            return int(parts[2])
    return None


def decode_kernel_for(w, kernel: str) -> str:
    """Which decode kernel runs (mirrors the library's selection)."""
    grouped = (w.head_dim == 128 and w.num_kv_heads in (1, 2, 4, 8, 16, 32)
               and w.group in (1, 2, 4, 8) and w.num_q_heads <= 64 and w.num_seqs <= 1023)
    if kernel in ("auto", "tc"):
        if grouped:
            return "tcg"
        return "tc_head" if w.head_dim == 128 else "simt"
    return kernel


class NativeStep:
    """Device state of one replica: pool, tables, inputs; run() = one step."""

    def __init__(self, pa, torch, w, dev, partition_tokens: int, kernel: str,
                 fused: bool = True):
        self.pa, self.torch, self.w, self.dev = pa, torch, w, dev
        self.fused = fused
        bs = w.block_size
        pairs = []
        if w.length_kind == "shared_prefix":
            # P prompts, each forked into S samples that share every prompt block
            # (refcount S); the step appends one token per sample, so each sample
            # that writes into the shared, partly filled last block first copies
            # it (copy-on-write), the last holder writes in place.
            prompt_lens = [w.prefix_tokens + int(k) for k in syn.prompt_extra_tokens(w)]
            blocks = sum(-(-L // bs) for L in prompt_lens) + w.num_prompts * w.samples_per_prompt
            nb = int(math.ceil(w.pool_factor * blocks)) + 1
            bm = pa.BlockManager(nb, bs, syn.shuffled_free_order(nb, syn.rng(w, "free")))
            pad = bm.allocate(1)[0]
            seqs = []
            for L in prompt_lens:
                root = bm.new_sequence(L)
                seqs += [root] + [bm.fork(root) for _ in range(w.samples_per_prompt - 1)]
            for sq in seqs:
                _, cow = bm.append(sq)
                if cow is not None:
                    pairs.append(cow)
            lens = np.array([bm.seq_len(sq) for sq in seqs], dtype=np.int64)
            self.unique_tokens = sum(prompt_lens) + len(seqs)
        else:
            lens = syn.seq_lens(w)
            blocks = sum(-(-int(L) // bs) for L in lens)
            nb = int(math.ceil(w.pool_factor * blocks)) + 1
            bm = pa.BlockManager(nb, bs, syn.shuffled_free_order(nb, syn.rng(w, "free")))
            pad = bm.allocate(1)[0]
            seqs = []
            for L in lens:
                s = bm.new_sequence(int(L) - 1)     # context before this step
                bm.append(s)                        # the step's token: opens a block at a boundary
                seqs.append(s)
            self.unique_tokens = int(np.sum(lens))
        B = len(lens)
        mb = max(bm.seq_num_blocks(s) for s in seqs)
        tables, seq_lens = bm.export(seqs, mb, pad)
        self.pairs = (torch.tensor(pairs, dtype=torch.int32, device=dev).reshape(-1, 2)
                      if pairs else None)
        self.lens = lens
        self.max_blocks = mb
        self.num_blocks = nb
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        tdt = torch.bfloat16 if w.dtype == syn.BFLOAT16 else torch.float16
        shape = (nb, bs, w.num_kv_heads, w.head_dim)
        self.k_pool = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(tdt)
        self.v_pool = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(tdt)
        self.q = torch.randn((B, w.num_q_heads, w.head_dim), generator=g, device=dev).to(tdt)
        self.key = torch.randn((B, w.num_kv_heads, w.head_dim), generator=g, device=dev).to(tdt)
        self.value = torch.randn_like(self.key)
        self.tables = tables.to(dev)
        self.seq_lens = seq_lens.to(dev)
        self.slots = torch.empty(B, dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.max_seq_len = int(lens.max())
        self.pt = partition_tokens
        self.ws = pa.alloc_workspace(B, w.num_q_heads, w.head_dim, self.max_seq_len,
                                     partition_tokens, dev)
        P = -(-self.max_seq_len // (partition_tokens or 512))
        # decode_slots + reshape_and_cache + decode (+ plan on the tensor-core
        # path) + combine when a sequence spans several partitions
        self.kernel = decode_kernel_for(w, kernel)
        # append_tokens, then decode: main + combine (grouped), plan + main
        # (+ combine) (per-head), main (+ combine) (CUDA cores).  The fused step
        # (pa_decode_append) writes the new tokens inside the grouped main kernel.
        if self.kernel == "tcg":
            self.launches_per_step = (0 if fused else 1) + 2
        elif self.kernel == "tc_head":
            self.launches_per_step = 1 + 2 + (1 if P > 1 else 0)
        else:
            self.launches_per_step = 1 + 1 + (1 if P > 1 else 0)
        if self.pairs is not None:      # copy-on-write block copies
            self.launches_per_step += 1
        # End-to-end measurement: every step's inputs (q, the new tokens' K/V,
        # tables, lengths, copy-on-write pairs) live packed in one pinned host
        # buffer mirrored by one device buffer, whose views the step uses, so a
        # step moves them with one host-to-device copy; the output comes back
        # with one device-to-host copy.
        parts = [("q", self.q), ("key", self.key), ("value", self.value),
                 ("tables", self.tables), ("seq_lens", self.seq_lens)]
        if self.pairs is not None:
            parts.append(("pairs", self.pairs))
        offs, total = [], 0
        for _, t in parts:
            offs.append(total)
            total += -(-t.numel() * t.element_size() // 256) * 256
        self.d_in = torch.empty(total, dtype=torch.uint8, device=dev)
        self.h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        for (name, t), off in zip(parts, offs):
            n = t.numel() * t.element_size()
            dview = self.d_in[off:off + n].view(t.dtype).view(t.shape)
            dview.copy_(t)
            self.h_in[off:off + n].view(t.dtype).view(t.shape).copy_(t.cpu())
            setattr(self, name, dview)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for _, t in parts)
        self.d2h_bytes = self.h_out.numel() * self.h_out.element_size()

    def write_step(self):
        pa = self.pa
        if self.pairs is not None:
            pa.pa_copy_blocks(self.k_pool, self.v_pool, self.pairs)
        if not self.fused:
            pa.pa_append_tokens(self.k_pool, self.v_pool, self.key, self.value, self.tables,
                                self.seq_lens)

    def decode(self):
        """The decode call; with `fused`, pa_decode_append, which also writes the
        step's new tokens (inside the grouped kernel, else as a launch before it)."""
        if self.fused:
            self.pa.pa_decode_append(self.out, self.q, self.k_pool, self.v_pool, self.key,
                                     self.value, self.tables, self.seq_lens, self.w.scale,
                                     max_seq_len=self.max_seq_len, partition_tokens=self.pt,
                                     workspace=self.ws)
        else:
            self.pa.pa_decode(self.out, self.q, self.k_pool, self.v_pool, self.tables,
                              self.seq_lens, self.w.scale, max_seq_len=self.max_seq_len,
                              partition_tokens=self.pt, workspace=self.ws)

    def run(self):
        self.write_step()
        self.decode()

    def run_e2e(self):
        # the step's inputs from pinned host memory (one copy), the result back
        self.d_in.copy_(self.h_in, non_blocking=True)
        self.run()
        self.h_out.copy_(self.out, non_blocking=True)


def run_native(args, dist_info):
    import torch
    import paged_kv_cache_301_gb300 as pa
    from paged_kv_cache_301_gb300 import build as _build

    rank, world, local = dist_info
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args.workload, args.block_size)
    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline and w.length_kind != "shared_prefix":
        # before the first GPU call: the oracle's pool is a spawn pool anyway
        cpu_baseline = cpu_oracle_baseline(w, budget_s=args.cpu_budget)
    pa.set_decode_path(args.kernel)
    step = NativeStep(pa, torch, w, dev, args.partition_tokens, args.kernel,
                      fused=not args.split_step)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(torch, dev))
    clocks.start()
    time.sleep(0.25)           # let the sampler take its first reading
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    # the K steps back to back (events between the steps would break the
    # programmatic-dependent-launch chain from one step's last kernel to the
    # next step's first)
    t_start.record(stream)
    for i in range(args.steps):
        step.run()
    t_end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    # then K more with events around each decode call, for its own duration
    for i in range(args.steps):
        step.write_step()
        ev[i][0].record(stream)
        step.decode()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    decode_ms = [a.elapsed_time(b) for a, b in ev]

    # end to end: host buffers in, host result out, every step
    for _ in range(max(3, args.warmup // 4)):
        step.run_e2e()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step.run_e2e()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    total_ms, e2e_ms = slowest_rank([total_ms, e2e_ms], world, dev)
    if rank != 0:
        return None

    ms_step = total_ms / args.steps
    kvb = kv_bytes(step.lens, w)
    B = len(step.lens)
    value = whole_job_gbs(kvb, world, ms_step)
    dec_avg_ms = sum(decode_ms) / len(decode_ms)
    dec_bytes = decode_bytes(step.lens, w, step.max_blocks)
    if step.fused:     # the new tokens' K/V read once and written to the pool
        dec_bytes += 4 * B * w.num_kv_heads * w.head_dim * w.elem_bytes
    peak, peak_kind = measured_peaks()
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = recorded_traffic(w.name, step.kernel)
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": syn.DTYPE_NAMES[w.dtype],
        "data": "synthetic (seeded N(0,1) q/K/V; block ids a seeded permutation)",
        "config": {
            "workload": w.name, "num_seqs": B, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "seq_lens": {
                "fixed": list(w.lens), "uniform": f"uniform [{w.lo},{w.hi}]",
                "lognormal": f"lognormal median {w.median:g} sigma {w.sigma:g} clipped [{w.lo},{w.hi}]",
                "shared_prefix": f"{w.num_prompts} prompts x {w.samples_per_prompt} samples, "
                                 f"prefix {w.prefix_tokens}+U{{0..{w.prefix_jitter}}}, +1 token"}[w.length_kind],
            "total_tokens": int(np.sum(step.lens)), "num_blocks": step.num_blocks,
            "partition_tokens": args.partition_tokens or 512,
            "kv_bytes_per_step": kvb,
            "l2": f"inputs larger than L2: {kvb / 2**20:.0f} MiB of K/V read per step vs "
                  f"{L2_BYTES / 2**20:.0f} MiB L2; no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "decode_kernel": {"tcg": "tcgen05 + TMA, whole-block (decode_tcg_kernel)",
                              "tc_head": "tcgen05 + TMA, per KV head (decode_tc_kernel)",
                              "simt": "CUDA cores (decode_simt_kernel)"}[step.kernel],
            "step": ("pa_decode_append: new tokens' cache write + decode in one call"
                     if step.fused else "pa_append_tokens, then pa_decode"),
        },
        "tokens_per_s": round(world * B / (ms_step * 1e-3), 1),
        "unique_kv_gbs": round(whole_job_gbs(step.unique_tokens * w.num_kv_heads * w.head_dim * 4,
                                             world, ms_step), 1),
        "cow_block_copies_per_step": 0 if step.pairs is None else int(step.pairs.shape[0]),
        "kv_frac_of_peak": round(value / world / peak, 4),
        "wall_s": round(wall, 4),
        "e2e": {
            "value": round(world * kvb / (e2e_ms / args.steps * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms / args.steps, 5),
            "h2d_bytes_per_step": step.h2d_bytes,
            "d2h_bytes_per_step": step.d2h_bytes,
        },
        "gpu_launches": step.launches_per_step * args.steps,
        "roofline": {
            "kernel": ("pa_decode_append" if step.fused else "pa_decode") + " " +
                      {"tcg": "(stream-K main + combine)" + (
                          ", cache write inside the main kernel" if step.fused else ""),
                       "tc_head": "(plan + split-K main + combine)" + (
                           ", after the cache write" if step.fused else ""),
                       "simt": "(split-K main + combine)" + (
                           ", after the cache write" if step.fused else "")}[step.kernel],
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "traffic_unit": "bytes per decode_tcg_kernel launch (ncu dram read + write)",
            "algorithmic_bytes": dec_bytes,
            "avg_launch_ms": round(dec_avg_ms, 5),
        },
        "clocks": clk,
        "cpu_baseline": cpu_baseline,
    }
    return result


# ----------------------------------------------------------------------------
# whole-block moves across a model's layers (not the decode step)
# ----------------------------------------------------------------------------

def run_blocks(args):
    """--op swap: blocks of every layer's K and V pool between the GPU and pinned
    CPU memory (pa_swap_blocks, both directions), against a contiguous
    copy-engine transfer of the same byte count (the link's ceiling).
    --op cow_layers: copy-on-write clones in every layer's pools in one launch
    (pa_copy_blocks_multi), against the measured HBM copy peak."""
    import torch
    import paged_kv_cache_301_gb300 as pa
    from paged_kv_cache_301_gb300 import build as _build

    _build.build()
    torch.cuda.set_device(0)
    layers, bs, hkv, d = 32, 16, 8, 128            # Llama-3-8B: 32 layers, 8 KV heads
    pools_n = 2 * layers
    block_bytes = bs * hkv * d * 2
    gpu_nb = 1024
    n = args.pairs
    g = np.random.default_rng(1234)
    gpu = [torch.empty((gpu_nb, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
           for _ in range(pools_n)]
    for t in gpu:
        t.normal_()
    src_ids = g.permutation(gpu_nb)[:n].astype(np.int32)
    stream = torch.cuda.current_stream()

    def time_it(fn, steps, warmup):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    peak, peak_kind = measured_peaks()
    moved = n * pools_n * block_bytes
    if args.op == "swap":
        cpu_nb = n
        cpu = [torch.empty((cpu_nb, bs, hkv, d), dtype=torch.bfloat16, pin_memory=True)
               for _ in range(pools_n)]
        cpu_ids = g.permutation(cpu_nb).astype(np.int32)
        out_pairs = torch.from_numpy(np.stack([src_ids, cpu_ids], 1)).cuda()
        in_pairs = torch.from_numpy(np.stack([cpu_ids, src_ids], 1)).cuda()
        out_ms = time_it(lambda: pa.pa_swap_blocks(cpu, gpu, out_pairs), args.steps, args.warmup)
        in_ms = time_it(lambda: pa.pa_swap_blocks(gpu, cpu, in_pairs), args.steps, args.warmup)
        flat_dev = torch.empty(moved // 2, dtype=torch.bfloat16, device="cuda")
        flat_host = torch.empty(moved // 2, dtype=torch.bfloat16, pin_memory=True)
        d2h_ms = time_it(lambda: flat_host.copy_(flat_dev, non_blocking=True), args.steps,
                         args.warmup)
        h2d_ms = time_it(lambda: flat_dev.copy_(flat_host, non_blocking=True), args.steps,
                         args.warmup)
        gbs = lambda ms: round(moved / (ms * 1e-3) / 1e9, 1)
        return {
            "metric": "KV block swap GB/s, GPU pools <-> pinned CPU pools (every layer, one launch)",
            "value": gbs(out_ms), "unit": "GB/s", "op": "swap", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic N(0,1) pools; seeded block permutation",
            "config": {"workload": "llama3_8b_layers", "layers": layers, "pools": pools_n,
                       "block_size": bs, "num_kv_heads": hkv, "head_dim": d,
                       "block_bytes": block_bytes, "blocks_per_pool": n,
                       "bytes_per_swap": moved},
            "swap_out": {"gbs": gbs(out_ms), "ms": round(out_ms, 4),
                         "frac_of_contiguous_copy": round(d2h_ms / out_ms, 4)},
            "swap_in": {"gbs": gbs(in_ms), "ms": round(in_ms, 4),
                        "frac_of_contiguous_copy": round(h2d_ms / in_ms, 4)},
            "contiguous_copy_engine": {"d2h_gbs": gbs(d2h_ms), "h2d_gbs": gbs(h2d_ms),
                                       "what": "one cudaMemcpyAsync of the same byte count"},
            "gpu_launches": 2 * args.steps,
        }
    # cow_layers
    ids = g.permutation(gpu_nb)
    pairs = torch.from_numpy(np.stack([ids[:n], ids[n:2 * n]], 1).astype(np.int32)).cuda()
    ms = time_it(lambda: pa.pa_copy_blocks_multi(gpu, pairs), args.steps, args.warmup)
    gbs = 2 * moved / (ms * 1e-3) / 1e9                # read + write
    return {
        "metric": "copy-on-write block copies across all layers, GB/s (read + write)",
        "value": round(gbs, 1), "unit": "GB/s", "op": "cow_layers", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic N(0,1) pools; seeded block permutation",
        "config": {"workload": "llama3_8b_layers", "layers": layers, "pools": pools_n,
                   "block_size": bs, "block_bytes": block_bytes, "pairs": n,
                   "bytes_copied": moved},
        "ms": round(ms, 4),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(gbs / peak, 4)},
        "gpu_launches": args.steps,
    }


def run_prefill(args):
    """--op prefill: causal multi-query attention over the paged pool (pa_prefill)
    on the whole-prompt or the chunked-prefill workload; FLOP/s of the causal
    (query, key) pairs against the measured bf16 tensor peak."""
    import torch
    import paged_kv_cache_301_gb300 as pa
    from paged_kv_cache_301_gb300 import build as _build
    from oracle import scenarios
    from oracle.prefill import causal_pairs

    _build.build()
    name = args.workload if args.workload in ("prefill", "chunked_prefill") else "prefill"
    w = syn.WORKLOADS[name]
    pb = scenarios.prefill_batch(w, fill_all=True)
    b = pb.batch
    torch.cuda.set_device(0)
    dt = {syn.FLOAT16: torch.float16, syn.BFLOAT16: torch.bfloat16}[w.dtype]

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(dt)

    pa.set_prefill_path("simt" if args.kernel == "simt" else "auto")
    kp, vp, q = dev(b.k_pool), dev(b.v_pool), dev(pb.q)
    tables = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    qst = torch.from_numpy(pb.q_start).cuda()
    out = torch.empty_like(q)
    max_q = int(np.diff(pb.q_start).max())
    stream = torch.cuda.current_stream()

    def step():
        pa.pa_prefill(out, q, kp, vp, tables, lens, qst, w.scale, max_q_len=max_q)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_uuid(torch, torch.device("cuda", 0)))
    clocks.start()
    time.sleep(0.25)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    pairs = causal_pairs(b.seq_lens, pb.q_start)
    flops = 4.0 * w.head_dim * w.num_q_heads * pairs          # q.k and p.v per pair and head
    tflops = flops / (ms * 1e-3) / 1e12
    total_q = int(pb.q_start[-1])
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    peak = peaks.get("bf16_tflops") or 1900.0
    peak_kind = "measured (cuBLAS bf16, burst)" if "bf16_tflops" in peaks else "fallback"
    cpu = None
    if not args.no_cpu_baseline:
        g = np.random.default_rng(3)
        rows = sorted(set(int(x) for x in g.integers(0, total_q, size=16)))
        t0 = time.perf_counter()
        scenarios.prefill_f64(pb, rows=rows)
        el = time.perf_counter() - t0
        # flops of the sampled rows: each row sees position + 1 keys, all heads
        pos = []
        for r in rows:
            s_ = int(np.searchsorted(pb.q_start, r, side="right")) - 1
            n_ = int(pb.q_start[s_ + 1] - pb.q_start[s_])
            pos.append(int(b.seq_lens[s_]) - n_ + (r - int(pb.q_start[s_])))
        f_rows = 4.0 * w.head_dim * w.num_q_heads * sum(p_ + 1 for p_ in pos)
        cpu = {"value": round(f_rows / el / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
               "kind": "oracle", "sample": f"{len(rows)} query rows (all heads) of the {name} "
                                           f"workload, fp64 oracle, {el:.1f} s"}
    return {
        "metric": "paged prefill attention TFLOP/s (causal pairs x 4 x head_dim x heads)",
        "value": round(tflops, 1), "unit": "TFLOP/s", "op": "prefill", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "dtype": syn.DTYPE_NAMES[w.dtype],
        "data": "synthetic (seeded N(0,1) q/K/V; block ids a seeded permutation)",
        "config": {"workload": name, "num_seqs": len(b.seq_lens), "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "total_tokens": int(b.seq_lens.sum()),
                   "query_tokens": total_q, "causal_pairs_per_head": pairs},
        "tokens_per_s": round(total_q / (ms * 1e-3), 1),
        "roofline": {"kernel": "prefill_simt_kernel" if args.kernel == "simt" else "prefill_tc_kernel",
                     "bound": "tensor",
                     "achieved": round(tflops, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "algorithmic_flops": flops, "avg_launch_ms": round(ms, 5)},
        "clocks": clk, "cpu_baseline": cpu, "gpu_launches": args.steps,
    }


def run_allocsim(args):
    """--op allocsim: contiguous vs paged KV allocation on a saturated serving
    stream (Poisson arrivals, lognormal lengths), block-size sweep; host code
    (pa_sim_run), the oracle's simulator timed beside it."""
    import paged_kv_cache_301_gb300 as pa
    from paged_kv_cache_301_gb300 import build as _build

    _build.build()
    s = syn.SERVING_STREAM
    a, p, o = syn.request_arrays(s)
    cap = 26777 * 16
    runs = [("contiguous", r, 16) for r in ("max", "pow2", "exact")] + \
        [("paged", "max", bs) for bs in (1, 8, 16, 32, 64, 128)]
    rows = []
    t0 = time.perf_counter()
    for alloc, rule, bs in runs:
        r = pa.simulate_allocator(a, p, o, alloc, cap, block_size=bs, reserve=rule,
                                  max_seq_len=s.max_seq_len)
        row = {"allocator": alloc if alloc == "paged" else f"contiguous/{rule}",
               "block_size": bs if alloc == "paged" else None,
               "kv_utilisation": round(r["utilisation_of_held"], 4),
               "utilisation_of_pool": round(r["utilisation_of_capacity"], 4),
               "max_concurrency": r["max_concurrency"],
               "mean_concurrency": round(r["mean_concurrency"], 1),
               "failed_allocations": r["failed_allocations"],
               "fragmentation_failures": r["fragmentation_failures"],
               "preemptions": r["preemptions"], "steps": r["steps"]}
        if alloc == "paged":
            row["internal_fragmentation"] = round(r["internal_fragmentation"], 4)
            row["mean_block_table_len"] = round(r["mean_table_len"], 2)
            row["max_block_table_len"] = r["max_table_len"]
        rows.append(row)
    native_s = time.perf_counter() - t0
    oracle_s = None
    if not args.no_cpu_baseline:
        from oracle.allocator_sim import simulate, CONTIGUOUS, PAGED, RESERVE_MAX
        t0 = time.perf_counter()
        simulate(a, p, o, PAGED, capacity=cap, block_size=16, max_seq_len=s.max_seq_len)
        simulate(a, p, o, CONTIGUOUS, capacity=cap, reserve=RESERVE_MAX,
                 max_seq_len=s.max_seq_len)
        oracle_s = time.perf_counter() - t0
    paged16 = next(r for r in rows if r["block_size"] == 16)
    contig = rows[0]
    return {
        "metric": "KV memory utilisation, paged (block 16) vs contiguous (max reservation)",
        "value": paged16["kv_utilisation"], "unit": "fraction", "op": "allocsim",
        "higher_is_better": True, "data": "synthetic request stream (seeded)",
        "config": {"workload": "serving_stream", "requests": s.num_requests,
                   "arrivals_per_step": s.rate, "prompt": f"lognormal median {s.prompt_median:g} "
                   f"sigma {s.prompt_sigma:g}", "output": f"lognormal median {s.output_median:g} "
                   f"sigma {s.output_sigma:g}", "max_seq_len": s.max_seq_len,
                   "capacity_tokens": cap},
        "contiguous_max_utilisation": contig["kv_utilisation"],
        "concurrency_gain": round(paged16["max_concurrency"] / contig["max_concurrency"], 2),
        "sweep": rows,
        "native_s_for_sweep": round(native_s, 3),
        "oracle_s_for_two_runs": None if oracle_s is None else round(oracle_s, 3),
        "gpu_launches": 0,
    }


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ----------------------------------------------------------------------------

_shared = {}


def _pool_init(spec):
    from multiprocessing import shared_memory
    for key, (name, shape, dtype) in spec.items():
        shm = shared_memory.SharedMemory(name=name)
        _shared[key] = (shm, np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf))


def _pool_task(args):
    b, scale, dtype, heads = args
    from oracle.attention import paged_decode_attention
    out = paged_decode_attention(_shared["q"][1], _shared["k"][1], _shared["v"][1],
                                 _shared["tables"][1], _shared["lens"][1], scale,
                                 sequences=[b], heads=heads, dtype=dtype)
    return float(out[b].sum())


class OraclePool:
    """The fp64 oracle over a host copy of the workload, run on a spawn pool with
    one single-threaded worker per host core."""

    def __init__(self, w, cores=None):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        from oracle import scenarios
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.batch = scenarios.fixed_batch(w)
        b = self.batch
        arrays = {"q": b.q, "k": b.k_pool, "v": b.v_pool,
                  "tables": b.block_tables.astype(np.int32),
                  "lens": b.seq_lens.astype(np.int32)}
        self.shms = []
        spec = {}
        for key, arr in arrays.items():
            shm = shared_memory.SharedMemory(create=True, size=max(arr.nbytes, 1))
            view = np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)
            view[...] = arr
            self.shms.append(shm)
            spec[key] = (shm.name, arr.shape, arr.dtype.str)
        self.cores = cores or len(os.sched_getaffinity(0))
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(self.cores, initializer=_pool_init, initargs=(spec,))
        self.pool.map(_pool_task, [(0, b.scale, b.dtype, [0])] * self.cores)   # warm the workers
        self.w = w

    def run(self, units):
        """units: list of (b, heads); returns seconds."""
        t0 = time.perf_counter()
        self.pool.map(_pool_task, [(b, self.batch.scale, self.batch.dtype, heads)
                                   for b, heads in units], chunksize=1)
        return time.perf_counter() - t0

    def unit_bytes(self, units):
        w = self.w
        G = w.group
        lens = self.batch.seq_lens
        # K/V bytes the oracle reads: per query head it gathers its KV head's rows
        return sum(int(lens[b]) * w.head_dim * 2 * w.elem_bytes * len(heads) / G
                   for b, heads in units)

    def close(self):
        self.pool.terminate()
        for s in self.shms:
            s.close()
            s.unlink()


def cpu_oracle_baseline(w, budget_s=15.0):
    """Oracle throughput on the host cores: whole passes over the batch until
    about budget_s of CPU work (wall time x worker processes) is spent."""
    op = OraclePool(w)
    try:
        B = len(op.batch.seq_lens)
        all_heads = list(range(w.num_q_heads))
        units = [(b, all_heads) for b in range(B)]
        passes, secs = 0, 0.0
        while passes == 0 or secs * op.cores < budget_s:
            secs += op.run(units)
            passes += 1
        kvb = passes * kv_bytes(op.batch.seq_lens, w)
        return {"value": round(kvb / secs / 1e9, 4), "unit": "GB/s", "cores": op.cores,
                "kind": "oracle",
                "sample": f"fp64 oracle, {passes} full pass(es) over the {B} sequences x "
                          f"{w.num_q_heads} query heads of the {w.name} workload, {secs:.2f} s "
                          f"wall on {op.cores} single-threaded worker processes",
                "tokens_per_s": round(passes * B / secs, 3)}
    finally:
        op.close()


def run_reference(args, dist_info):
    rank, world, _ = dist_info
    if rank != 0:
        return None
    w = workload(args.workload, args.block_size)
    op = OraclePool(w)
    try:
        B = len(op.batch.seq_lens)
        G = w.group
        # unit = one (sequence, KV head): its G query heads
        units = [(b, list(range(h * G, (h + 1) * G))) for b in range(B)
                 for h in range(w.num_kv_heads)]
        probe = units[:op.cores]
        t = op.run(probe)
        per_unit = t / len(probe)
        total_steps = args.steps + args.warmup
        budget = args.cpu_budget * 8          # whole reference run: a few minutes at most
        n = max(1, min(len(units), int(budget / total_steps / max(per_unit, 1e-9))))
        sample = units[:n]
        for _ in range(args.warmup):
            op.run(sample)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            op.run(sample)
        secs = time.perf_counter() - t0
        kvb = op.unit_bytes(sample) * args.steps
        value = kvb / secs / 1e9
        line = {
            "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) q/K/V; block ids a seeded permutation)",
            "config": {"workload": w.name, "num_seqs": B, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                       "block_size": w.block_size},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": op.cores,
                             "kind": "oracle",
                             "sample": f"each step: {n} (sequence, KV head) units of "
                                       f"{len(units)} of the {w.name} workload, fp64 oracle"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        return line
    finally:
        op.close()


# ----------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "native":
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    return rank, world, local


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="llama3_8b",
                    choices=["llama3_8b", "long_context", "shared_prefix", "ragged", "tiny",
                             "mha_7b", "prefill", "chunked_prefill"])
    ap.add_argument("--block-size", type=int, default=None)
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--kernel", choices=["auto", "simt", "tc", "tc_head"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--split-step", action="store_true",
                    help="decode step as pa_append_tokens + pa_decode instead of the one "
                         "pa_decode_append call")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--op", choices=["decode", "swap", "cow_layers", "allocsim", "prefill"],
                    default="decode",
                    help="decode: the decode step (default); swap / cow_layers: whole-block "
                         "moves over a 32-layer model's pools; allocsim: contiguous vs paged "
                         "allocator simulation (host only); prefill: paged causal "
                         "multi-query attention (--workload prefill | chunked_prefill)")
    ap.add_argument("--pairs", type=int, default=512, help="blocks per pool moved (--op swap, "
                                                           "cow_layers)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.op == "decode" and args.workload in ("prefill", "chunked_prefill"):
        ap.error("the prefill workloads run with --op prefill")
    if args.op != "decode":
        if args.impl == "reference":
            why = {"prefill": "the prefill line carries its oracle timing in cpu_baseline",
                   "allocsim": "the allocator line times the oracle simulator itself"}.get(
                       args.op, "no CPU arm for block moves")
            print(json.dumps({"impl": "reference", "op": args.op, "unavailable": why}), flush=True)
        elif args.op == "allocsim":
            print(json.dumps(run_allocsim(args)), flush=True)
        elif args.op == "prefill":
            print(json.dumps(run_prefill(args)), flush=True)
        else:
            print(json.dumps(run_blocks(args)), flush=True)
        return
    dist_info = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, dist_info)
    else:
        res = run_native(args, dist_info)
    if res is not None:
        print(json.dumps(res), flush=True)
    if dist_info[1] > 1 and args.impl == "native":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
