"""pkv_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers may not call cudaMalloc (code running during a global-mode CUDA
graph capture, plugins inside a framework that owns the device memory, loops
that cannot afford an allocator synchronization).  The no-alloc entry point
takes its split-K scratch from a fixed array inside the library instead of a
caller buffer.  This file checks, through the C ABI, that it returns what
pkv_decode_attn returns with a caller-provided workspace and what the oracle
computes, on two calls in a row (the second with other queries, so stale
scratch from the first would show), for dense decode and for decode over
selected positions (whose gather scratch sits in the same array), and that
requests larger than the array or with an oversized page table are refused.
It is named so pytest collects it last.
"""
import math

import numpy as np
import pytest

import workloads as W
from helpers import assert_close, i32, q_tensor, torch_dev, upload_cache, window_tensors
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("noalloc", 40, 4, 64, 512, [1500, 700, 64, 2000])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    wlen = [128, 17, 0, 128]
    win, kw, vw = window_tensors(wl, tw, tw, wlen)
    ctx = P.Context(512, 64)
    dev = torch_dev()
    pt, sl = i32(wl.page_table), i32(wl.seq_len)
    scale = 1 / math.sqrt(512)
    g = np.random.default_rng(41)
    for call in range(2):
        bits = W.to_bf16_bits(g.standard_normal((4, 64, 512)).astype(np.float32))
        q = q_tensor(bits)
        ref_o = torch.empty(4, 64, 512, device=dev)
        ref_l = torch.empty(4, 64, device=dev)
        ctx.pkv_decode_attn(q, cache, pt, sl, win, scale, ref_o, ref_l)
        o = torch.full((4, 64, 512), float("nan"), device=dev)
        l = torch.full((4, 64), float("nan"), device=dev)
        ctx.pkv_decode_attn_noalloc(q, cache, pt, sl, win, scale, o, l)
        torch.cuda.synchronize()
        assert ctx.pkv_get_error() == P.OK
        go, gl = o.cpu().numpy(), l.cpu().numpy()
        assert_close(go, ref_o.cpu().numpy(), f"O call {call}")
        assert_close(gl, ref_l.cpu().numpy(), f"LSE call {call}")
        for b in range(4):
            L = int(wl.seq_len[b])
            K = C.dequant_seq(wl, Kp, ts, b, L)
            V = C.dequant_seq(wl, Vp, ts, b, L)
            n = wlen[b]
            Or, Lr = A.decode(F.bf16_to_f64(bits[b]), K, V, F.fp8_dequantize(kw[b][:n], tw),
                              F.fp8_dequantize(vw[b][:n], tw), scale)
            assert_close(go[b], Or, f"O vs oracle, call {call} seq {b}")
            assert_close(gl[b], Lr, f"LSE vs oracle, call {call} seq {b}")


def test_noalloc_selected_positions_twice():
    # decode over selected positions: the gathered compact pages live in the same array
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("noalloc_sel", 42, 2, 64, 512, [5000, 3000])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, kw, vw = window_tensors(wl, tw, tw)
    ctx = P.Context(512, 64)
    dev = torch_dev()
    pt, sl = i32(wl.page_table), i32(wl.seq_len)
    scale = 1 / math.sqrt(512)
    g = np.random.default_rng(43)
    k = 256
    for call in range(2):
        sel = np.full((2, k), -1, np.int32)
        for b in range(2):
            n = k - 40 * b                          # the second row is -1 padded
            sel[b, :n] = np.sort(g.choice(int(wl.seq_len[b]), n, replace=False))
        bits = W.to_bf16_bits(g.standard_normal((2, 64, 512)).astype(np.float32))
        q = q_tensor(bits)
        ref_o = torch.empty(2, 64, 512, device=dev)
        ref_l = torch.empty(2, 64, device=dev)
        ctx.pkv_decode_attn(q, cache, pt, sl, win, scale, ref_o, ref_l, sel_idx=i32(sel))
        o = torch.full((2, 64, 512), float("nan"), device=dev)
        l = torch.full((2, 64), float("nan"), device=dev)
        ctx.pkv_decode_attn_noalloc(q, cache, pt, sl, win, scale, o, l, sel_idx=i32(sel))
        torch.cuda.synchronize()
        assert ctx.pkv_get_error() == P.OK
        go, gl = o.cpu().numpy(), l.cpu().numpy()
        assert_close(go, ref_o.cpu().numpy(), f"selected O call {call}")
        assert_close(gl, ref_l.cpu().numpy(), f"selected LSE call {call}")
        for b in range(2):
            idx = [int(t) for t in sel[b] if t >= 0]
            K = C.dequant_tokens(wl, Kp, ts, b, idx)
            V = C.dequant_tokens(wl, Vp, ts, b, idx)
            Or, Lr = A.decode(F.bf16_to_f64(bits[b]), K, V, F.fp8_dequantize(kw[b], tw), F.fp8_dequantize(vw[b], tw),
                              scale)
            assert_close(go[b], Or, f"selected O vs oracle, call {call} seq {b}")
            assert_close(gl[b], Lr, f"selected LSE vs oracle, call {call} seq {b}")


def test_noalloc_refuses_requests_beyond_its_array():
    import torch
    import precision_kv_cache_gb300 as P
    ctx = P.Context(512, 64)
    dev = torch_dev()
    B, max_pages = 64, 512                      # 64 sequences of up to 32K tokens
    need = ctx.pkv_workspace_bytes(P.OP_DECODE, B, max_pages * 64)
    assert need > (16 << 20)
    cache = P.KVCache.empty(4, 512, 0.01, 0.01)
    z8 = torch.zeros(B, 128, 512, dtype=torch.uint8, device=dev)
    win = P.Window(z8, z8, 0.1, 0.1)
    q = torch.zeros(B, 64, 512, dtype=torch.bfloat16, device=dev)
    out = torch.empty(B, 64, 512, device=dev)
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_decode_attn_noalloc(q, cache, torch.zeros(B, max_pages, dtype=torch.int32, device=dev),
                                    torch.zeros(B, dtype=torch.int32, device=dev), win, 0.1, out)
    assert e.value.status == P.ERR_WORKSPACE


def test_noalloc_refuses_an_oversized_page_table_before_any_work():
    # max_pages * 64 beyond 2^30 positions is refused on the host, as pkv_decode_attn does
    import ctypes
    import torch
    import precision_kv_cache_gb300 as P
    ctx = P.Context(512, 64)
    dev = torch_dev()
    cache = P.KVCache.empty(4, 512, 0.01, 0.01)
    z8 = torch.zeros(1, 128, 512, dtype=torch.uint8, device=dev)
    win = P.Window(z8, z8, 0.1, 0.1)
    q = torch.zeros(1, 64, 512, dtype=torch.bfloat16, device=dev)
    out = torch.empty(1, 64, 512, device=dev)
    small = torch.zeros(1, 4, dtype=torch.int32, device=dev)
    c, w = cache._c(), win._c()
    for max_pages in ((1 << 24) + 1, (1 << 30) + 5):
        st = P.lib().pkv_decode_attn_noalloc(ctx.h, ctypes.c_void_p(q.data_ptr()), ctypes.byref(c),
                                              ctypes.c_void_p(small.data_ptr()), max_pages,
                                              ctypes.c_void_p(small.data_ptr()), 1, None, 0, ctypes.byref(w),
                                              ctypes.c_float(0.1), ctypes.c_void_p(out.data_ptr()), None, None)
        assert st == P.ERR_UNSUPPORTED, max_pages
