"""Benchmark: one decode step of paged attention per timed step, on GB300.

A step is the whole hot path over one batch: copy-on-write block copies when
the workload shares blocks (pa_copy_blocks), then one pa_decode_append call: the
cache write of each sequence's newest token at the slot its block table gives,
and decode attention over the paged pool (split-K main kernel + combine).
Inputs are synthetic and seeded; the pool is resident in HBM before timing
starts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the host cores

Timing: after W warm-up steps, blocks of K steps run back to back between CUDA
events (synchronize on both sides of each block), repeated at least
--min-repeats times and for about --timed-seconds; the median block gives
`value`.  Each decode call is then timed alone (events around it) for the
roofline, after an L2 flush as well, and end to end with the inputs copied in
from pinned host memory and the output copied back every step.  The default run
(Llama-3-8B-shaped headline) also measures the long-context, shared-prefix and
ragged decode workloads, whole-prompt prefill and a plain read stream, each in
the `workloads` / `stream_read` objects of the same line.

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

# The device code of the grouped decode kernel: its constants and tile
# geometry, its template, the parameter structs it reads, and the device headers
# it includes (host-side launch code is left out, so a change there keeps the
# recorded counters).
DECODE_KERNEL_TEXT = (
    ("pa_decode_tcg.cu", "constexpr int kD = 128;", "// Merge the partials"),
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
            nb = pool_blocks(w, lens)
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
        self.lens = lens
        self.max_blocks = mb
        self.num_blocks = nb
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        tdt = torch.bfloat16 if w.dtype == syn.BFLOAT16 else torch.float16
        shape = (nb, bs, w.num_kv_heads, w.head_dim)
        self.k_pool = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(tdt)
        self.v_pool = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(tdt)
        q = torch.randn((B, w.num_q_heads, w.head_dim), generator=g, device=dev).to(tdt)
        key = torch.randn((B, w.num_kv_heads, w.head_dim), generator=g, device=dev).to(tdt)
        value = torch.randn_like(key)
        self.max_seq_len = int(lens.max())
        self.pt = partition_tokens
        pa.set_decode_path(kernel)
        self.ws = pa.workspace_for(q, self.k_pool, tables, self.max_seq_len, partition_tokens)
        P = -(-self.max_seq_len // (partition_tokens or 512))
        # the kernel the library runs for this call (its own selection)
        self.kernel = {"grouped": "tcg", "per_head": "tc_head", "simt": "simt"}[
            pa.decode_kernel_for(q, self.k_pool, tables, self.max_seq_len, partition_tokens)]
        # append_tokens, then decode: main + combine (grouped), plan + main
        # (+ combine) (per-head), main (+ combine) (CUDA cores).  The fused step
        # (pa_decode_append) writes the new tokens inside the grouped and the
        # CUDA-core main kernels.
        if self.kernel == "tcg":
            self.launches_per_step = (0 if fused else 1) + 2
        elif self.kernel == "tc_head":
            self.launches_per_step = 1 + 2 + (1 if P > 1 else 0)
        else:
            self.launches_per_step = (0 if fused else 1) + 1 + (1 if P > 1 else 0)
        if pairs:                       # copy-on-write block copies
            self.launches_per_step += 1
        # Every step's inputs (q, the new tokens' K/V, tables, lengths,
        # copy-on-write pairs) live packed in one pinned host buffer; two device
        # buffers mirror it, so that the end-to-end step can copy step i+1's
        # inputs in while step i computes.  A step moves its inputs with one
        # host-to-device copy and its output with one device-to-host copy.
        parts = [("q", q), ("key", key), ("value", value), ("tables", tables),
                 ("seq_lens", seq_lens)]
        if pairs:
            parts.append(("pairs", torch.tensor(pairs, dtype=torch.int32).reshape(-1, 2)))
        offs, total = [], 0
        for _, t in parts:
            offs.append(total)
            total += -(-t.numel() * t.element_size() // 256) * 256
        self.h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.bufs = []
        for _ in range(2):
            d_in = torch.empty(total, dtype=torch.uint8, device=dev)
            views = {"d_in": d_in, "out": torch.empty_like(q),
                     "h_out": torch.empty(q.shape, dtype=q.dtype).pin_memory()}
            for (name, t), off in zip(parts, offs):
                n = t.numel() * t.element_size()
                dview = d_in[off:off + n].view(t.dtype).view(t.shape)
                dview.copy_(t)
                views[name] = dview
            views.setdefault("pairs", None)
            self.bufs.append(views)
        for (name, t), off in zip(parts, offs):
            n = t.numel() * t.element_size()
            self.h_in[off:off + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        self.num_pairs = len(pairs)
        self.h2d_bytes = sum(t.numel() * t.element_size() for _, t in parts)
        self.d2h_bytes = q.numel() * q.element_size()
        self.streams = None

    def write_step(self, s: int = 0):
        pa, v = self.pa, self.bufs[s]
        if v["pairs"] is not None:
            pa.pa_copy_blocks(self.k_pool, self.v_pool, v["pairs"])
        if not self.fused:
            pa.pa_append_tokens(self.k_pool, self.v_pool, v["key"], v["value"], v["tables"],
                                v["seq_lens"])

    def decode(self, s: int = 0):
        """The decode call; with `fused`, pa_decode_append, which also writes the
        step's new tokens (inside the grouped and CUDA-core kernels, else as a launch
        before it)."""
        v = self.bufs[s]
        if self.fused:
            self.pa.pa_decode_append(v["out"], v["q"], self.k_pool, self.v_pool, v["key"],
                                     v["value"], v["tables"], v["seq_lens"], self.w.scale,
                                     max_seq_len=self.max_seq_len, partition_tokens=self.pt,
                                     workspace=self.ws)
        else:
            self.pa.pa_decode(v["out"], v["q"], self.k_pool, self.v_pool, v["tables"],
                              v["seq_lens"], self.w.scale, max_seq_len=self.max_seq_len,
                              partition_tokens=self.pt, workspace=self.ws)

    def run(self, s: int = 0):
        self.write_step(s)
        self.decode(s)

    def run_e2e_serial(self):
        """One step with its copies in line: inputs in, the step, the output back."""
        v = self.bufs[0]
        v["d_in"].copy_(self.h_in, non_blocking=True)
        self.run(0)
        v["h_out"].copy_(v["out"], non_blocking=True)

    def e2e_block(self, K: int, start_event):
        """K end-to-end steps with the copies pipelined: step i+1's inputs are
        copied in (its own stream) while step i computes, and step i's output is
        copied back (a third stream) while step i+1 computes.  Two device buffer
        sets alternate; events order every reuse.  Every step still moves its
        whole input in and its whole output out; the block ends when the last
        output is in host memory."""
        torch = self.torch
        if self.streams is None:
            self.streams = (torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev))
            E = lambda: [torch.cuda.Event(), torch.cuda.Event()]
            self.ev_ready, self.ev_computed, self.ev_drained = E(), E(), E()
        h2d, d2h = self.streams
        main = torch.cuda.current_stream()

        def copy_in(i):
            s = i % 2
            h2d.wait_event(start_event)
            if i >= 2:          # step i-2 has finished reading buffer s
                h2d.wait_event(self.ev_computed[s])
            with torch.cuda.stream(h2d):
                self.bufs[s]["d_in"].copy_(self.h_in, non_blocking=True)
            self.ev_ready[s].record(h2d)

        copy_in(0)
        for i in range(K):
            s = i % 2
            if i + 1 < K:
                copy_in(i + 1)
            main.wait_event(self.ev_ready[s])
            if i >= 2:          # step i-2's output has left buffer s
                main.wait_event(self.ev_drained[s])
            self.run(s)
            self.ev_computed[s].record(main)
            d2h.wait_event(self.ev_computed[s])
            with torch.cuda.stream(d2h):
                self.bufs[s]["h_out"].copy_(self.bufs[s]["out"], non_blocking=True)
            self.ev_drained[s].record(d2h)
        for s in range(min(K, 2)):
            main.wait_event(self.ev_drained[s])


def pool_blocks(w, lens) -> int:
    """Physical blocks of a fixed-batch workload's pool: 1.25 x the blocks the
    batch needs, plus the padding block table entries past a sequence point at."""
    need = sum(-(-int(L) // w.block_size) for L in lens)
    return int(math.ceil(w.pool_factor * need)) + 1


def workload_config(w, lens, num_blocks, args) -> dict:
    """The `config` object of a decode line; both arms emit the same one."""
    kvb = kv_bytes(lens, w)
    return {
        "workload": w.name, "num_seqs": int(len(lens)), "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
        "block_size": w.block_size, "seq_lens": {
            "fixed": list(w.lens), "uniform": f"uniform [{w.lo},{w.hi}]",
            "lognormal": f"lognormal median {w.median:g} sigma {w.sigma:g} clipped [{w.lo},{w.hi}]",
            "shared_prefix": f"{w.num_prompts} prompts x {w.samples_per_prompt} samples, "
                             f"prefix {w.prefix_tokens}+U{{0..{w.prefix_jitter}}}, +1 token"}[w.length_kind],
        "total_tokens": int(np.sum(lens)), "num_blocks": int(num_blocks),
        "partition_tokens": args.partition_tokens or 512,
        "kv_bytes_per_step": kvb,
        "l2": (f"inputs larger than L2: {kvb / 2**20:.0f} MiB of K/V read per step vs "
               f"{L2_BYTES / 2**20:.0f} MiB L2; no flush between steps (the l2_flushed "
               f"figure flushes before each call)") if kvb > L2_BYTES else
              (f"{kvb / 2**10:.0f} KiB of K/V per step, resident in L2: a latency-bound "
               f"step (no roofline target), no flush"),
        "parallelism": f"replicas x{args.world}" if args.world > 1 else "1 GPU",
    }


def agree_max(n: int, world: int, device) -> int:
    """The largest of the ranks' values of n (every rank runs the same loop)."""
    if world <= 1:
        return n
    import torch
    t = torch.tensor([n], dtype=torch.int64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return int(t.item())


def barrier(world):
    if world > 1:
        import torch
        torch.distributed.barrier()


def repeat_count(block_ms: float, args) -> int:
    """Repeats of the K-step block: at least --min-repeats, and enough for about
    --timed-seconds of timed work (so the clock sampler sees the load)."""
    want = int(math.ceil(args.timed_seconds * 1e3 / max(block_ms, 1e-3)))
    return max(args.min_repeats, min(want, args.max_repeats))


def measure_decode(torch, step, args, world, dev, flushed: bool):
    """Time one workload's decode step.  Returns per-repeat figures (max over
    ranks): ms per step of each K-step block run back to back, ms of each decode
    call with events around it, ms of calls after an L2 flush, and ms per step of
    end-to-end blocks (pipelined and serial copies)."""
    K = args.steps
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def block(fn):
        torch.cuda.synchronize()
        barrier(world)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    reps = agree_max(repeat_count(block(step.run), args), world, dev)
    clocks = ClockSampler(gpu_uuid(torch, dev))
    clocks.start()
    time.sleep(0.25)           # let the sampler take its first reading
    wall0 = time.perf_counter()
    # the K steps of a block back to back (events between the steps would break
    # the programmatic-dependent-launch chain from one step's last kernel to the
    # next step's first)
    step_ms = [block(step.run) / K for _ in range(reps)]
    wall = time.perf_counter() - wall0
    # then each decode call with events around it, for its own duration
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    call_ms = []
    for _ in range(reps):
        torch.cuda.synchronize()
        barrier(world)
        for i in range(K):
            step.write_step()
            ev[i][0].record(stream)
            step.decode()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        call_ms += [x.elapsed_time(y) for x, y in ev]
    clk = clocks.stop()
    flushed_ms = []
    if flushed:
        # L2 flush before each call: write one buffer of twice the L2, then read
        # another, so that the L2 holds clean lines of neither the workload nor
        # the first buffer (dirty lines would be written back inside the call)
        fw = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        fr = torch.zeros(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        for _ in range(max(args.min_repeats, 25)):
            step.write_step()
            fw.zero_()
            fr.sum()
            a.record(stream)
            step.decode()
            b.record(stream)
            torch.cuda.synchronize()
            flushed_ms.append(a.elapsed_time(b))
        del fw, fr
    # end to end: host buffers in, host result out, every step
    for _ in range(3):
        step.run_e2e_serial()
    torch.cuda.synchronize()
    e2e_ms, e2e_serial_ms = [], []
    for _ in range(reps):
        torch.cuda.synchronize()
        barrier(world)
        a.record(stream)
        step.e2e_block(K, a)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(a.elapsed_time(b) / K)
    for _ in range(reps):
        e2e_serial_ms.append(block(step.run_e2e_serial) / K)
    out = {"reps": reps, "step_ms": step_ms, "call_ms": call_ms, "flushed_ms": flushed_ms,
           "e2e_ms": e2e_ms, "e2e_serial_ms": e2e_serial_ms, "clocks": clk, "wall_s": wall}
    for key in ("step_ms", "call_ms", "flushed_ms", "e2e_ms", "e2e_serial_ms"):
        if out[key]:
            out[key] = slowest_rank(out[key], world, dev)
    return out


def med(xs):
    return statistics.median(xs) if xs else None


def measure_graph(torch, step, args, dev, reps: int = 25):
    """The K-step block captured once in a CUDA graph and replayed: the step's
    device time without the host's per-call launch cost (which bounds the
    latency-bound tiny workload when it is called from Python).  The library
    allocates nothing during a call given its workspace, so the calls capture
    as they are.  Returns a dict for the line, or one with the reason the
    capture failed."""
    K = args.steps
    main = torch.cuda.current_stream()
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(main)
        with torch.cuda.stream(side):
            for _ in range(3):
                step.run()
        main.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(K):
                step.run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            a.record(main)
            g.replay()
            b.record(main)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b) / K)
        del g
        return {"ms_per_step": round(med(ms), 5), "repeats": reps,
                "how": f"the K = {K} steps captured once in a CUDA graph, replayed between "
                       f"CUDA events; median over {reps} replays / K"}
    except Exception as e:       # report, never fail the line
        torch.cuda.synchronize()
        return {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}


def decode_entry(step, m, w, world, peak, peak_kind, args) -> dict:
    """Figures of one decode workload from its measurements."""
    K = args.steps
    B = len(step.lens)
    kvb = kv_bytes(step.lens, w)
    ms_step = med(m["step_ms"])
    call = med(m["call_ms"])
    dec_bytes = decode_bytes(step.lens, w, step.max_blocks)
    if step.fused:     # the new tokens' K/V read once and written to the pool
        dec_bytes += 4 * B * w.num_kv_heads * w.head_dim * w.elem_bytes
    # the decode call's average duration over the timed region: the step time
    # (one call per step; with copy-on-write pairs the step's block copies count
    # against it too)
    achieved = dec_bytes / (ms_step * 1e-3) / 1e9
    iso = dec_bytes / (call * 1e-3) / 1e9
    gbs = lambda ms: round(whole_job_gbs(kvb, world, ms), 1)
    e = {
        "value": gbs(ms_step), "unit": "GB/s",
        "ms_per_step": round(ms_step, 5),
        "ms_per_step_mean": round(statistics.fmean(m["step_ms"]), 5),
        "repeats": m["reps"], "steps_per_repeat": K,
        "tokens_per_s": round(world * B / (ms_step * 1e-3), 1),
        "kv_frac_of_peak": round(whole_job_gbs(kvb, 1, ms_step) / peak, 4),
        "config": workload_config(w, step.lens, step.num_blocks, args),
        "decode_kernel": {"tcg": "tcgen05 + TMA, whole-block (decode_tcg_kernel)",
                          "tc_head": "tcgen05 + TMA, per KV head (decode_tc_kernel)",
                          "simt": "CUDA cores (decode_simt_kernel)"}[step.kernel],
        "step": ("pa_decode_append: new tokens' cache write + decode in one call"
                 if step.fused else "pa_append_tokens, then pa_decode")
                + (f"; pa_copy_blocks of {step.num_pairs} copy-on-write pairs first"
                   if step.num_pairs else ""),
        "gpu_launches_per_step": step.launches_per_step,
        "roofline": {
            "kernel": ("pa_decode_append" if step.fused else "pa_decode") + " " +
                      {"tcg": "(stream-K main + combine)" + (
                          ", cache write inside the main kernel" if step.fused else ""),
                       "tc_head": "(plan + split-K main + combine)" + (
                           ", after the cache write" if step.fused else ""),
                       "simt": "(split-K main + combine)" + (
                           ", cache write inside the main kernel" if step.fused else "")}[step.kernel],
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(w.name, step.kernel),
            "traffic_unit": "bytes per decode_tcg_kernel launch (ncu dram read + write)",
            "algorithmic_bytes": dec_bytes,
            "avg_launch_ms": round(ms_step, 5),
            "launch_timing": f"median over {m['reps']} repeats of the timed region's K = {K} "
                             f"back-to-back calls (CUDA events on the launching stream) / K",
            "isolated_call": {
                "avg_launch_ms": round(call, 5),
                "launch_ms_mean": round(statistics.fmean(m["call_ms"]), 5),
                "achieved": round(iso, 1),
                "frac": round(iso / peak, 4),
                "how": f"median of {len(m['call_ms'])} calls with CUDA events around each "
                       f"call: no overlap with the previous call's end, its launch latency "
                       f"included",
            },
        },
        "e2e": {
            "value": gbs(med(m["e2e_ms"])), "unit": "GB/s",
            "ms_per_step": round(med(m["e2e_ms"]), 5),
            "h2d_bytes_per_step": step.h2d_bytes,
            "d2h_bytes_per_step": step.d2h_bytes,
            "copies": "pinned host inputs in and the output back every step; step i+1's "
                      "input copy and step i-1's output copy overlap step i (two device "
                      "buffer sets)",
            "serial": {"value": gbs(med(m["e2e_serial_ms"])),
                       "ms_per_step": round(med(m["e2e_serial_ms"]), 5),
                       "copies": "in, step, out, in line on one stream"},
        },
        "clocks": m["clocks"],
        "wall_s": round(m["wall_s"], 4),
    }
    if w.length_kind == "shared_prefix":
        e["unique_kv_gbs"] = round(whole_job_gbs(step.unique_tokens * w.num_kv_heads *
                                                 w.head_dim * 4, world, ms_step), 1)
        e["cow_block_copies_per_step"] = step.num_pairs
        e["roofline"]["note"] = ("logical bytes: the samples of a prompt read its shared "
                                 "prefix blocks, which stay in L2 between them; "
                                 "unique_kv_gbs counts each physical token once")
    if m["flushed_ms"]:
        fl = med(m["flushed_ms"])
        e["l2_flushed"] = {"avg_launch_ms": round(fl, 5),
                           "achieved": round(dec_bytes / (fl * 1e-3) / 1e9, 1),
                           "frac": round(dec_bytes / (fl * 1e-3) / 1e9 / peak, 4),
                           "calls": len(m["flushed_ms"]),
                           "how": "before each call: write a 2x L2 buffer, then read "
                                  "another; median of the calls"}
        e["warm"] = {"avg_launch_ms": round(call, 5), "achieved": round(iso, 1),
                     "frac": round(iso / peak, 4),
                     "how": "calls timed alone with events, no flush in between (the previous "
                            "call's data may sit in L2)"}
    return e


class PrefillStep:
    """Device state of one prefill workload: every token's K/V in a pool reached
    through block tables (the library's block manager over a shuffled free
    stack), queries for the last n_b tokens of each sequence."""

    def __init__(self, pa, torch, w, dev):
        self.pa, self.torch, self.w = pa, torch, w
        lens = syn.seq_lens(w)
        qn = syn.query_counts(w, lens)
        bs = w.block_size
        nb = pool_blocks(w, lens)
        bm = pa.BlockManager(nb, bs, syn.shuffled_free_order(nb, syn.rng(w, "free")))
        pad = bm.allocate(1)[0]
        seqs = [bm.new_sequence(int(L)) for L in lens]
        mb = max(bm.seq_num_blocks(s) for s in seqs)
        tables, seq_lens = bm.export(seqs, mb, pad)
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        tdt = torch.bfloat16 if w.dtype == syn.BFLOAT16 else torch.float16
        shape = (nb, bs, w.num_kv_heads, w.head_dim)
        self.k_pool = torch.randn(shape, generator=g, device=dev).to(tdt)
        self.v_pool = torch.randn(shape, generator=g, device=dev).to(tdt)
        q_start = np.concatenate([[0], np.cumsum(qn)]).astype(np.int32)
        self.total_q = int(q_start[-1])
        self.q = torch.randn((self.total_q, w.num_q_heads, w.head_dim), generator=g,
                             device=dev).to(tdt)
        self.out = torch.empty_like(self.q)
        self.tables = tables.to(dev)
        self.seq_lens = seq_lens.to(dev)
        self.q_start = torch.from_numpy(q_start).to(dev)
        self.max_q = int(qn.max())
        self.lens, self.qn = lens, qn
        # causal (query, key) pairs per head: query i of n attends to L - n + i + 1 keys
        self.pairs = int(sum(int(n) * (int(L) - int(n)) + int(n) * (int(n) + 1) // 2
                             for L, n in zip(lens, qn)))

    def run(self):
        self.pa.pa_prefill(self.out, self.q, self.k_pool, self.v_pool, self.tables,
                           self.seq_lens, self.q_start, self.w.scale, max_q_len=self.max_q)


def tensor_peak():
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    if "bf16_tflops" in peaks:
        return float(peaks["bf16_tflops"]), "measured (cuBLAS bf16, burst)"
    return 1900.0, "fallback"


def measure_prefill(torch, pa, name, args, dev, kernel="auto") -> dict:
    """Prefill TFLOP/s on one workload: median over repeats of K back-to-back calls."""
    w = syn.WORKLOADS[name]
    pa.set_prefill_path("simt" if kernel == "simt" else "auto")
    ps = PrefillStep(pa, torch, w, dev)
    stream = torch.cuda.current_stream()
    K = args.steps
    for _ in range(args.warmup):
        ps.run()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def block():
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(K):
            ps.run()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K

    reps = repeat_count(block() * K, args)
    clocks = ClockSampler(gpu_uuid(torch, dev))
    clocks.start()
    time.sleep(0.25)
    ms_list = [block() for _ in range(reps)]
    clk = clocks.stop()
    ms = med(ms_list)
    flops = 4.0 * w.head_dim * w.num_q_heads * ps.pairs     # q.k and p.v per pair and head
    tflops = flops / (ms * 1e-3) / 1e12
    peak, peak_kind = tensor_peak()
    res = {
        "value": round(tflops, 1), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
        "ms_per_step_mean": round(statistics.fmean(ms_list), 5), "repeats": reps,
        "steps_per_repeat": K,
        "config": {"workload": name, "num_seqs": len(ps.lens), "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "total_tokens": int(np.sum(ps.lens)),
                   "query_tokens": ps.total_q, "causal_pairs_per_head": ps.pairs},
        "tokens_per_s": round(ps.total_q / (ms * 1e-3), 1),
        "roofline": {"kernel": "prefill_simt_kernel" if kernel == "simt" else "prefill_tc_kernel",
                     "bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "algorithmic_flops": flops, "avg_launch_ms": round(ms, 5)},
        "clocks": clk, "gpu_launches_per_step": 1,
    }
    pa.set_prefill_path("auto")
    return res


def measure_stream_read(torch, pa, dev, args) -> dict:
    """The library's plain read stream over a 4 GiB buffer (context for the
    decode kernels' bandwidth): median of repeated passes."""
    nbytes = 4 << 30
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.random_(0, 256)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        pa.pa_stream_read(buf)
    ms = []
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max(args.min_repeats, 25)):
        a.record(stream)
        pa.pa_stream_read(buf)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    del buf
    m = med(ms)
    return {"gbs": round(nbytes / (m * 1e-3) / 1e9, 1), "bytes": nbytes, "passes": len(ms),
            "ms": round(m, 5), "kernel": "stream_read_kernel (pa_stream_read): contiguous "
            "16-byte loads, 8 in flight per thread, 4 x 512 threads per SM",
            "what": "read-only HBM bandwidth reached without a gather, same run; the "
                    "roofline peak is the copy (read + write) figure"}


# Workloads measured beside the headline one in a default run.
# The other workloads of the default line: (entry, workload, block size or None
# for the workload's own); the ragged step at every block size it sweeps.
PREFILL_WORKLOADS = ("prefill", "chunked_prefill", "prefill_qwen25_32b")

EXTRA_WORKLOADS = (("long_context", "long_context", None), ("shared_prefix", "shared_prefix", None),
                   ("ragged", "ragged", None), ("ragged_bs8", "ragged", 8),
                   ("ragged_bs32", "ragged", 32), ("ragged_bs64", "ragged", 64),
                   ("many_seqs", "many_seqs", None), ("mha_7b", "mha_7b", None),
                   ("qwen25_32b", "qwen25_32b", None), ("llama3_405b", "llama3_405b", None),
                   ("tiny", "tiny", None))


def run_native(args, dist_info):
    import torch
    import paged_kv_cache_301_gb300 as pa
    from paged_kv_cache_301_gb300 import build as _build

    rank, world, local = dist_info
    args.world = world
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args.workload, args.block_size)
    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline and w.length_kind != "shared_prefix":
        # before the first GPU call: the oracle's pool is a spawn pool anyway
        cpu_baseline = cpu_oracle_baseline(w, budget_s=args.cpu_budget)
    peak, peak_kind = measured_peaks()
    pa.set_decode_path(args.kernel)
    step = NativeStep(pa, torch, w, dev, args.partition_tokens, args.kernel,
                      fused=not args.split_step)
    m = measure_decode(torch, step, args, world, dev, flushed=True)
    head = decode_entry(step, m, w, world, peak, peak_kind, args)
    head["graph"] = measure_graph(torch, step, args, dev)
    del step
    torch.cuda.empty_cache()
    workloads = {}
    stream_read = None
    if args.workload == "llama3_8b" and not args.single_workload:
        for name, wname, wbs in EXTRA_WORKLOADS:
            wx = workload(wname, wbs)
            st = NativeStep(pa, torch, wx, dev, args.partition_tokens, args.kernel,
                            fused=not args.split_step)
            workloads[name] = decode_entry(st, measure_decode(torch, st, args, world, dev,
                                                              flushed=False),
                                           wx, world, peak, peak_kind, args)
            workloads[name]["graph"] = measure_graph(torch, st, args, dev)
            del st
            torch.cuda.empty_cache()
        if args.kernel in ("auto", "tc"):
            workloads["prefill"] = measure_prefill(torch, pa, "prefill", args, dev)
            torch.cuda.empty_cache()
        stream_read = measure_stream_read(torch, pa, dev, args)
    if rank != 0:
        return None
    reps = head["repeats"]
    result = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": syn.DTYPE_NAMES[w.dtype],
        "data": "synthetic (seeded N(0,1) q/K/V; block ids a seeded permutation)",
        "config": head.pop("config"),
        "timing": (f"value and ms_per_step: median over {reps} repeats of the K = {args.steps} "
                   f"steps timed back to back between CUDA events (synchronize on both "
                   f"sides of each repeat; ms_per_step_mean is the mean)"),
    }
    result.update(head)
    result["gpu_launches"] = head["gpu_launches_per_step"] * args.steps * reps
    result["cpu_baseline"] = cpu_baseline
    if workloads:
        result["workloads"] = workloads
    if stream_read is not None:
        result["stream_read"] = stream_read
        result["roofline"]["frac_of_stream_read"] = round(
            result["roofline"]["achieved"] / stream_read["gbs"], 4)
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


def prefill_cpu_baseline(name: str) -> dict:
    """The fp64 oracle on 16 sampled query rows (all heads) of a prefill
    workload, one host thread, on the oracle's own copy of the inputs."""
    from oracle import scenarios
    w = syn.WORKLOADS[name]
    pb = scenarios.prefill_batch(w, fill_all=True)
    b = pb.batch
    total_q = int(pb.q_start[-1])
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
    return {"value": round(f_rows / el / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle", "sample": f"{len(rows)} query rows (all heads) of the {name} "
                                        f"workload, fp64 oracle, {el:.1f} s"}


def run_prefill(args):
    """--op prefill: causal multi-query attention over the paged pool (pa_prefill)
    on the whole-prompt or the chunked-prefill workload; FLOP/s of the causal
    (query, key) pairs against the measured bf16 tensor peak."""
    import torch
    import paged_kv_cache_301_gb300 as pa
    from paged_kv_cache_301_gb300 import build as _build

    _build.build()
    name = args.workload if args.workload in PREFILL_WORKLOADS else "prefill"
    w = syn.WORKLOADS[name]
    cpu = None if args.no_cpu_baseline else prefill_cpu_baseline(name)
    torch.cuda.set_device(0)
    r = measure_prefill(torch, pa, name, args, torch.device("cuda", 0),
                        kernel="simt" if args.kernel == "simt" else "auto")
    out = {
        "metric": "paged prefill attention TFLOP/s (causal pairs x 4 x head_dim x heads)",
        "value": r["value"], "unit": "TFLOP/s", "op": "prefill", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "dtype": syn.DTYPE_NAMES[w.dtype],
        "data": "synthetic (seeded N(0,1) q/K/V; block ids a seeded permutation)",
    }
    out.update(r)
    out["cpu_baseline"] = cpu
    out["gpu_launches"] = args.steps * r["repeats"]
    return out


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


def _pool_task_timed(args):
    """Run the units (b, heads) `repeats` times in this worker; the seconds are
    measured here, so no inter-process traffic is counted."""
    units, scale, dtype, repeats = args
    from oracle.attention import paged_decode_attention
    t0 = time.perf_counter()
    for _ in range(repeats):
        for b, heads in units:
            paged_decode_attention(_shared["q"][1], _shared["k"][1], _shared["v"][1],
                                   _shared["tables"][1], _shared["lens"][1], scale,
                                   sequences=[b], heads=heads, dtype=dtype)
    return time.perf_counter() - t0


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

    def run_single(self, units, repeats=1):
        """One worker (one host thread) runs the units `repeats` times in turn;
        returns its seconds."""
        return self.pool.apply(_pool_task_timed,
                               ((units, self.batch.scale, self.batch.dtype, repeats),))

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


def single_thread_baseline(op, units_all, budget_s: float) -> dict:
    """The oracle on one host thread: whole (sequence, all heads) units in turn,
    as many as fit about budget_s (at least one), repeated for short workloads."""
    w = op.w
    t1 = op.run_single(units_all[:1])
    n = max(1, min(len(units_all), int(budget_s / max(t1, 1e-6))))
    units = units_all[:n]
    repeats = 1
    if n == len(units_all):
        t_all = op.run_single(units)
        repeats = max(1, int(budget_s / max(t_all, 1e-6)))
    secs = op.run_single(units, repeats)
    lens = op.batch.seq_lens
    kvb = repeats * sum(int(lens[b]) for b, _ in units) * w.num_kv_heads * w.head_dim * 2 * \
        w.elem_bytes
    return {"workload": w.name, "value": round(kvb / secs / 1e9, 5), "unit": "GB/s",
            "cores": 1, "tokens_per_s": round(repeats * len(units) / secs, 3),
            "sample": f"{len(units)} of {len(units_all)} sequences (all {w.num_q_heads} query "
                      f"heads) x {repeats} pass(es), {secs:.2f} s on one single-threaded "
                      f"worker process"}


def cpu_oracle_baseline(w, budget_s=15.0):
    """Oracle throughput on the host cores: whole passes over the batch until
    about budget_s of CPU work (wall time x worker processes) is spent; then the
    same oracle on one host thread, on this workload and on the tiny one."""
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
        res = {"value": round(kvb / secs / 1e9, 4), "unit": "GB/s", "cores": op.cores,
               "kind": "oracle",
               "sample": f"fp64 oracle, {passes} full pass(es) over the {B} sequences x "
                         f"{w.num_q_heads} query heads of the {w.name} workload, {secs:.2f} s "
                         f"wall on {op.cores} single-threaded worker processes",
               "tokens_per_s": round(passes * B / secs, 3)}
        single = [single_thread_baseline(op, units, budget_s / 5)]
    finally:
        op.close()
    if w.name != "tiny":
        tiny = syn.WORKLOADS["tiny"]
        op = OraclePool(tiny, cores=1)
        try:
            tu = [(b, list(range(tiny.num_q_heads))) for b in range(len(op.batch.seq_lens))]
            single.append(single_thread_baseline(op, tu, budget_s / 15))
        finally:
            op.close()
    res["single_thread"] = single
    return res


def run_reference(args, dist_info):
    rank, world, _ = dist_info
    args.world = world
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
            "config": workload_config(w, op.batch.seq_lens, pool_blocks(w, op.batch.seq_lens),
                                      args),
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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--min-repeats", type=int, default=25,
                    help="repeats of the K-step timed block at least (the median is reported)")
    ap.add_argument("--max-repeats", type=int, default=1000)
    ap.add_argument("--timed-seconds", type=float, default=0.6,
                    help="aim for about this much timed work per loop and workload")
    ap.add_argument("--single-workload", action="store_true",
                    help="measure only --workload (the default run adds the other decode "
                         "workloads, prefill and the read stream)")
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="llama3_8b",
                    choices=["llama3_8b", "long_context", "shared_prefix", "ragged", "tiny",
                             "mha_7b", "llama3_405b", "many_seqs", "qwen25_32b", "prefill",
                             "chunked_prefill", "prefill_qwen25_32b"])
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
    if args.op == "decode" and args.workload in PREFILL_WORKLOADS:
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
