"""The benchmark's one-line JSON contract, for both arms: the keys the line
must carry and the values that must hold whatever the machine (the reference arm
is the fp64 oracle on the host cores; the native arm needs the GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e"}


def _run(*args, timeout=600):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert BASE_KEYS <= set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3
    assert d["config"]["workload"] == "llama3_8b" and d["value"] > 0
    # the same workload description as the native arm's line
    assert {"num_seqs", "seq_lens", "total_tokens", "num_blocks", "kv_bytes_per_step"} <= \
        set(d["config"])
    assert d["config"]["num_seqs"] == 64 and d["config"]["total_tokens"] == 149573
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]


@pytest.mark.gpu
def test_native_arm_line():
    d = _run("--steps", "20", "--warmup", "5", "--no-cpu-baseline")
    assert BASE_KEYS <= set(d) and {"roofline", "clocks", "gpu_launches", "cpu_baseline"} <= set(d)
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 5
    assert d["scaling"] == "weak" and d["higher_is_better"] is True and d["dtype"] == "bf16"
    assert d["config"]["workload"] == "llama3_8b" and d["value"] > 0
    # the step is one pa_decode_append call: main + combine on the grouped kernel;
    # the value is the median over the repeats of the 20-step block
    assert d["gpu_launches_per_step"] == 2 and d["repeats"] >= 25
    assert d["gpu_launches"] == 2 * 20 * d["repeats"]
    # every other decode workload, prefill and the read stream in the same line
    assert {"long_context", "shared_prefix", "ragged", "ragged_bs8", "ragged_bs32", "ragged_bs64",
            "many_seqs", "mha_7b", "qwen25_32b", "llama3_405b", "tiny", "prefill"} <= \
        set(d["workloads"])
    assert d["workloads"]["tiny"]["ms_per_step"] > 0         # latency-bound: no roofline target
    # the same steps replayed from a CUDA graph (the host's launch cost left out)
    assert d["graph"]["ms_per_step"] > 0 and d["workloads"]["tiny"]["graph"]["ms_per_step"] > 0
    for name in ("long_context", "shared_prefix", "ragged", "ragged_bs8", "ragged_bs32", "ragged_bs64",
                 "many_seqs", "mha_7b", "qwen25_32b", "llama3_405b"):
        x = d["workloads"][name]
        assert x["config"]["workload"] == name and x["value"] > 0 and x["tokens_per_s"] > 0
        assert x["roofline"]["bound"] == "hbm" and 0 < x["roofline"]["frac"] < 1.5
    assert d["workloads"]["prefill"]["roofline"]["bound"] == "tensor"
    assert d["stream_read"]["gbs"] > 0
    assert d["l2_flushed"]["avg_launch_ms"] > 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    # achieved over the timed region's average call; the isolated call beside it
    assert abs(r["avg_launch_ms"] - d["ms_per_step"]) < 1e-9
    assert 0 < r["isolated_call"]["frac"] <= r["frac"] + 0.05
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
