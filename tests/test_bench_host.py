"""Host-side pieces of the benchmark and of the GPU tests' checkers (no GPU):
the needed-bytes accounting against a hand count, the L2 flush, the comment-insensitive
code hash that keys committed DRAM captures, the FP8 interval check used by the
fused-decode parity tests, and the JSON line of the reference arm."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
import workloads as W
from helpers import assert_fp8_codes
from oracle import formats as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_needed_bytes_counts_shared_pages_once():
    # two sequences share their first 64-token page; 100 + 64 and 64 + 30 tokens otherwise
    wl = W.make_shared_prefix("acct", 1, 2, 8, 128, [164, 94], 2, 64, append=False)
    total, tokens = bench.needed_bytes(wl)
    assert tokens == 64 + 100 + 30
    kv = 2 * (64 + 8)                      # K and V: d/2 code bytes + d/16 scale bytes at d = 128
    pt = (3 + 2) * 4                       # page-table entries read: 3 + 2 pages
    win = 2 * 128 * 128 * 2                # FP8 K and V windows of both sequences
    q = 2 * 8 * 128 * 2                    # bf16 queries
    o = 2 * 8 * 129 * 4                    # FP32 O and LSE
    assert total == tokens * kv + pt + win + q + o
    # fused decode: E4M3 O, FP32 LSE, each row's position and cos/sin row
    total_f, _ = bench.needed_bytes(wl, fused=True)
    assert total_f == tokens * kv + pt + win + q + 2 * 8 * 128 + 2 * 8 * 4 + 2 * (4 + W.ROPE_DIM * 4)


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) {  // add one\n  return x + 1;\n}\n/* block\n comment */\n")
    b = tmp_path / "b.cu"
    b.write_text("int f(int x) {\n\n  return x + 1;   // changed comment\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_sha(str(a)) == bench.code_sha(str(b))
    assert bench.code_sha(str(a)) != bench.code_sha(str(c))


def test_fp8_interval_check_accepts_rounding_and_rejects_wrong_codes():
    r = np.random.default_rng(3)
    Or = r.standard_normal((4, 64)) * 0.05
    codes = F.fp8_quantize(Or, W.OUT_SCALE)
    assert_fp8_codes(codes, Or, W.OUT_SCALE, "exact")
    # a value whose tolerance band holds no rounding midpoint: its code is forced
    bad = codes.copy()
    x = np.abs(Or / W.OUT_SCALE)
    i = np.unravel_index(np.argmax(x), x.shape)
    bad[i] = (int(bad[i]) & 0x80) | ((int(bad[i]) & 0x7F) - 3)     # three steps smaller in magnitude
    with pytest.raises(AssertionError):
        assert_fp8_codes(bad, Or, W.OUT_SCALE, "planted")


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "c1",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] >= 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["metric"] == "decode-attention KV GB/s (needed bytes / step time)"


def test_every_bench_workload_builds_and_is_described():
    names = sorted(bench.WORKLOADS) + sorted(bench.SWEEP) + sorted(bench.SCORE_SWEEP)
    for name in names:
        wl = bench._wl_cache(name)
        assert wl.B >= 1 and wl.page_table.shape[0] == wl.B, name
        assert (wl.page_table[wl.page_table >= 0] < wl.num_pages).all(), name
        desc = bench.workload_desc(name) if name not in bench.SCORE_SWEEP else wl.name
        assert isinstance(desc, str) and desc, name
        total, tokens = bench.needed_bytes(wl, fused=name in bench.FUSED)
        assert total > 0 and tokens >= 0, name
        bench._WL.pop(name, None)
    assert set(bench.FUSED) <= set(bench.WORKLOADS)


def test_l2_flush_writes_then_reads_twice_the_l2():
    """The flush before a timed step writes one buffer and then reads another, each
    at least twice the 129 MB L2, so no line of the step stays resident and the
    lines left behind are clean; the config string says so."""
    import torch
    f = bench.L2Flush(torch.device("cpu"))
    assert f.w.numel() * f.w.element_size() >= 2 * bench.L2_BYTES
    assert f.r.numel() * f.r.element_size() >= 2 * bench.L2_BYTES
    assert f.w.data_ptr() != f.r.data_ptr()
    f()
    assert int(f.w[0]) == 1 and int(f.w[-1]) == 1
    assert "written" in bench.L2Flush.DESC and "read" in bench.L2Flush.DESC
