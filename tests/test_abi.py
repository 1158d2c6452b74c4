"""The C-ABI library builds, loads, exports every declared symbol, and rejects
bad arguments on the host before any launch (CPU only: no kernel runs)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_301_gb300 import build
    build.build()
    from paged_kv_cache_301_gb300 import _lib
    return _lib.load()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\*?\s+\*?(pa_\w+)\s*\(", text,
                             flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert {"pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode_slots",
            "pa_decode_workspace_bytes", "pa_status_string", "pa_bm_create"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_binding_signatures_cover_the_header(lib):
    from paged_kv_cache_301_gb300 import _lib
    assert _declared_symbols() == set(_lib.SIGNATURES)


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"ok"
    assert b"unsupported" in lib.pa_status_string(2)
    assert lib.pa_version() >= 100


def _decode(lib, **kw):
    a = dict(out=16, q=16, k=16, v=16, tables=16, lens=16, B=2, Hq=8, Hkv=2, D=128, bs=16,
             MB=4, NB=8, max_len=64, scale=0.1, dtype=1, pt=0, ws=256, ws_bytes=1 << 20,
             status=None, stream=None)
    a.update(kw)
    return lib.pa_decode(a["out"], a["q"], a["k"], a["v"], a["tables"], a["lens"], a["B"],
                         a["Hq"], a["Hkv"], a["D"], a["bs"], a["MB"], a["NB"], a["max_len"],
                         a["scale"], a["dtype"], a["pt"], a["ws"], a["ws_bytes"], a["status"],
                         a["stream"])


def test_decode_argument_checks(lib):
    assert _decode(lib, D=96) == 2                 # head_dim not built
    assert _decode(lib, bs=12) == 2                # block size not built
    assert _decode(lib, dtype=5) == 2
    assert _decode(lib, Hq=6, Hkv=4) == 1          # Hq not a multiple of Hkv
    assert _decode(lib, max_len=65) == 1           # longer than the table can hold
    assert _decode(lib, pt=100) == 1               # partition not a multiple of 128
    assert _decode(lib, out=None) == 1
    assert _decode(lib, q=8) == 1                  # misaligned
    assert _decode(lib, ws_bytes=16) == 3          # workspace too small
    assert _decode(lib, ws=None) == 3
    assert _decode(lib, ws=16) == 3                # workspace not 256-byte aligned
    assert _decode(lib, scale=float("nan")) == 1
    assert _decode(lib, B=0) == 0                  # nothing to do, no launch


def _decode_append(lib, **kw):
    a = dict(out=16, q=16, k=16, v=16, key=16, value=16, tables=16, lens=16, B=2, Hq=8, Hkv=2,
             D=128, bs=16, MB=4, NB=8, max_len=64, scale=0.1, dtype=1, pt=0, ws=256,
             ws_bytes=1 << 20, status=None, stream=None)
    a.update(kw)
    return lib.pa_decode_append(a["out"], a["q"], a["k"], a["v"], a["key"], a["value"],
                                a["tables"], a["lens"], a["B"], a["Hq"], a["Hkv"], a["D"],
                                a["bs"], a["MB"], a["NB"], a["max_len"], a["scale"],
                                a["dtype"], a["pt"], a["ws"], a["ws_bytes"], a["status"],
                                a["stream"])


def test_decode_append_argument_checks(lib):
    """Every case returns before any launch: the step's new K/V must be given
    and 16-byte aligned; the other checks are pa_decode's."""
    assert _decode_append(lib, key=None) == 1
    assert _decode_append(lib, value=None) == 1
    assert _decode_append(lib, key=8) == 1         # misaligned
    assert _decode_append(lib, value=24) == 1
    assert _decode_append(lib, D=96) == 2          # head_dim not built
    assert _decode_append(lib, Hq=6, Hkv=4) == 1
    assert _decode_append(lib, ws_bytes=16) == 3   # workspace too small
    assert _decode_append(lib, B=0, key=None, value=None) == 0   # nothing to do


def test_workspace_size(lib):
    # m and l: B*Hq*P floats each; acc: B*Hq*P*D floats; 256-byte aligned parts
    n = lib.pa_decode_workspace_bytes(64, 32, 128, 4096, 0)
    P = 4096 // 512
    rows = 64 * 32 * P
    a = lambda x: (x + 255) // 256 * 256
    # per-head path: queue counters, (sequence, partition) list, m, l, acc;
    # grouped path: tile prefixes, weight prefixes and the start weight, and the
    # partials of up to 160 CTAs x 2 segments x Hq heads
    per_head = 256 + a(64 * P * 8) + 2 * a(rows * 4) + a(rows * 128 * 4)
    parts = 160 * 2 * 32
    grouped = a(65 * 4) + a(66 * 4) + 2 * a(parts * 4) + a(parts * 128 * 4)
    # enough for whichever kernel runs (each lays out its own parts from 0)
    assert n == max(per_head, grouped)
    assert lib.pa_decode_workspace_bytes(64, 32, 128, 4096, 100) == 0
    assert lib.pa_decode_workspace_bytes(-1, 32, 128, 4096, 0) == 0


def test_cache_argument_checks(lib):
    f = lib.pa_reshape_and_cache
    assert f(16, 16, 16, 16, 16, 4, 0, 8, 96, 16, 8, 1, None, None) == 2
    assert f(16, 16, 16, 16, 16, 4, 12, 8, 128, 16, 8, 1, None, None) == 1   # stride < row
    assert f(16, 16, 16, 16, 16, 0, 0, 8, 128, 16, 8, 1, None, None) == 0    # no tokens
    assert f(None, 16, 16, 16, 16, 4, 0, 8, 128, 16, 8, 1, None, None) == 1
    g = lib.pa_copy_blocks
    assert g(16, 16, 16, 2, 8, 128, 16, 8, 3, None, None) == 2
    assert g(16, 16, 16, 0, 8, 128, 16, 8, 1, None, None) == 0
    assert g(16, 16, None, 2, 8, 128, 16, 8, 1, None, None) == 1
    s = lib.pa_decode_slots
    assert s(16, 16, 16, 0, 4, 16, 8, None, None) == 0
    assert s(None, 16, 16, 3, 4, 16, 8, None, None) == 1
    assert s(16, 16, 16, 3, 4, 16, 0, None, None) == 1            # no pool
    assert s(16, 16, 16, 3, 4, 64, 1 << 26, None, None) == 1      # slots overflow int32


def _align(x):
    return (x + 255) // 256 * 256


def test_workspace_size_of_the_cuda_core_kernel(lib):
    """pa_decode_workspace_bytes_for sizes the kernel that runs: with the CUDA-core
    kernel selected, [B, Hq, P] maxima and sums plus [B, Hq, P, D] accumulators
    (P = 512-token partitions of the longest sequence); never above the
    kernel-independent bound; 0 for arguments pa_decode would reject."""
    assert lib.pa_set_decode_path(1) == 0
    try:
        f = lib.pa_decode_workspace_bytes_for
        for B, Hq, Hkv, D, bs, mx in ((64, 32, 8, 128, 16, 4096), (8, 64, 8, 128, 32, 131072),
                                      (3, 4, 4, 64, 8, 1)):
            P = -(-mx // 512)
            rows = B * Hq * P
            want = 2 * _align(4 * rows) + _align(4 * rows * D)
            got = f(B, Hq, Hkv, D, bs, -(-mx // bs), 1000, mx, 1, 0)
            assert got == want
            assert got <= lib.pa_decode_workspace_bytes(B, Hq, D, mx, 0)
        assert f(4, 6, 4, 128, 16, 8, 100, 128, 1, 0) == 0           # Hq % Hkv
        assert f(4, 8, 4, 96, 16, 8, 100, 128, 1, 0) == 0            # head_dim
        assert f(4, 8, 4, 128, 16, 8, 100, 129, 1, 0) == 0           # longer than the table
        assert f(4, 8, 4, 128, 16, 8, 100, 128, 1, 100) == 0         # partition size
    finally:
        lib.pa_set_decode_path(0)
