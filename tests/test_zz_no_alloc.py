"""pkv_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers may not call cudaMalloc (code running during a global-mode CUDA
graph capture, plugins inside a framework that owns the device memory, loops
that cannot afford an allocator synchronization).  The no-alloc entry point
takes its split-K scratch from a fixed array inside the library instead of a
caller buffer.  This file checks, through the C ABI, that it returns what
pkv_decode_attn returns with a caller-provided workspace, on two calls in a row
(the second with other queries, so stale scratch from the first would show),
and that a request larger than the array is refused.  It is named so pytest
collects it last.
"""
import math

import numpy as np
import pytest

import workloads as W
from helpers import assert_close, i32, q_tensor, torch_dev, upload_cache, window_tensors
from oracle import cache as C

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("noalloc", 40, 4, 64, 512, [1500, 700, 64, 2000])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw, [128, 17, 0, 128])
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
        assert_close(o.cpu().numpy(), ref_o.cpu().numpy(), f"O call {call}")
        assert_close(l.cpu().numpy(), ref_l.cpu().numpy(), f"LSE call {call}")


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
