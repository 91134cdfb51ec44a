"""The C-ABI library loads and exports every entry point include/pkv.h declares
(no compute calls: runs without a GPU)."""
import os
import re
import subprocess

import pytest

from conftest import ROOT


def declared_symbols():
    with open(os.path.join(ROOT, "include", "pkv.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ["pkv_init", "pkv_destroy", "pkv_append_kv", "pkv_score_topk", "pkv_decode_attn",
              "pkv_replay_attn", "pkv_merge", "pkv_get_error", "pkv_workspace_bytes"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    import precision_kv_cache_gb300 as P
    if not os.path.exists(P.LIB_PATH):
        from precision_kv_cache_gb300 import build
        build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", P.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    L = P.lib()
    for n in declared_symbols():
        assert hasattr(L, n)
    assert L.pkv_status_str(0) == b"ok"


def test_host_validation_without_gpu():
    import ctypes
    import precision_kv_cache_gb300 as P
    L = P.lib()
    # null config / null out pointer are rejected before any CUDA call
    assert L.pkv_init(None, 0, None) == P.ERR_INVALID_ARG
    cfg = P._Config(500, 64, 64, 128, 128, 64)
    h = ctypes.c_void_p()
    assert L.pkv_init(ctypes.byref(cfg), 0, ctypes.byref(h)) == P.ERR_UNSUPPORTED
    assert L.pkv_merge(None, None, None, None, None, None, 4, 8, None) == P.ERR_INVALID_ARG
    assert L.pkv_quantize_fp8(None, 16, ctypes.c_float(1.0), None, None) == P.ERR_INVALID_ARG
    assert L.pkv_workspace_bytes(None, 1, 1, 1) == 0
