"""GPU parity of the fused decode (vLLM blog, "MegaAttention avec KV compressé
NVFP4": query RoPE, attention, inverse RoPE on the output and FP8 conversion in
one pass) against the oracle's float64 fused decode.

O' (float32) and LSE within |gpu - oracle| <= 2e-3 + 1e-2 |oracle|; the E4M3
codes checked by interval (helpers.assert_fp8_codes).
"""
import math

import numpy as np
import pytest

import workloads as W
from helpers import assert_close, assert_fp8_codes, i32, q_tensor, torch_dev, upload_cache, window_tensors
from oracle import cache as C

pytestmark = pytest.mark.gpu


def _fused_case(wl, rope_dim=W.ROPE_DIM, sel=None, table=None, pos=None, bad_rows=()):
    import torch
    import precision_kv_cache_gb300 as P
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, kw, vw = window_tensors(wl, tw, tw, wl.win_len)
    ctx = P.Context(wl.d, wl.H)
    dev = torch_dev()
    q = q_tensor(wl.q_bits())
    pos = wl.rope_pos() if pos is None else np.asarray(pos, np.int32)
    if table is None:
        table = W.rope_table(wl.seed, int(max(pos.max(), 0)) + 1, rope_dim)
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    o8 = torch.empty(wl.B, wl.H, wl.d, dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(wl.d)
    sel_t = None if sel is None else i32(sel)
    ctx.pkv_decode_attn_fused(q, cache, i32(wl.page_table), i32(wl.seq_len), win, scale, i32(pos),
                              torch.from_numpy(table).to(dev), rope_dim, W.OUT_SCALE, o8, out, lse, sel_idx=sel_t)
    torch.cuda.synchronize()
    err = ctx.pkv_get_error()
    assert err == (P.ERR_BAD_PAGE if len(bad_rows) else P.OK)
    assert ctx.pkv_attn_path() == 2
    go, gl, g8 = out.cpu().numpy(), lse.cpu().numpy(), o8.cpu().numpy()
    for b in range(wl.B):
        s = None if sel is None else sel[b]
        if b in bad_rows:      # position outside the table: the row is not rotated
            assert s is None
            O, Lr = C.expected_decode(wl, Kp, Vp, ts, ts, tw, tw, b, scale=scale)
            assert_close(go[b], O, f"unrotated O seq {b}")
            assert_close(gl[b], Lr, f"unrotated LSE seq {b}")
            assert_fp8_codes(g8[b], O, W.OUT_SCALE, f"unrotated FP8 seq {b}")
            continue
        Or, Lr, _ = C.expected_decode_fused(wl, Kp, Vp, ts, ts, tw, tw, b, table, rope_dim, W.OUT_SCALE,
                                            pos=pos[b], sel=s, scale=scale)
        assert_close(go[b], Or, f"O' seq {b}")
        assert_close(gl[b], Lr, f"LSE seq {b}")
        assert_fp8_codes(g8[b], Or, W.OUT_SCALE, f"FP8 O' seq {b}")
    return ctx, go, g8


def test_fused_tiny_config():
    """The tiny decode shape (B=1, 8 heads, d=128, 1024 tokens + window), last 64 channels rotated."""
    _fused_case(W.config(0))


@pytest.mark.parametrize("d,H,rd", [(512, 64, 64), (128, 8, 8), (256, 32, 256), (512, 16, 128)])
def test_fused_ragged(d, H, rd):
    # several tiles plus partial tails, a single token, an empty prefix, short windows
    wl = W.make_dense("fused_ragged", 11, 4, H, d, [1000, 1, 300, 129], win=[128, 5, 0, 1])
    _fused_case(wl, rope_dim=rd)


def test_fused_sparse_selected_positions():
    g = np.random.default_rng(12)
    wl = W.make_dense("fused_sparse", 13, 3, 64, 512, [5000, 3000, 40])
    k = 96
    sel = np.full((3, k), -1, np.int32)
    for b, L in enumerate(wl.seq_len):
        n = min(k, int(L))
        sel[b, :n] = np.sort(g.choice(int(L), n, replace=False))
    _fused_case(wl, sel=sel)


def test_fused_identity_table_equals_plain_decode():
    """cos = 1, sin = 0: the fused call's FP32 output is the plain decode's, bit for bit."""
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("fused_ident", 14, 3, 64, 512, [700, 129, 2000])
    table = np.concatenate([np.ones((2000, 32)), np.zeros((2000, 32))], 1).astype(np.float32)
    ctx, go, g8 = _fused_case(wl, table=table)
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    dev = torch_dev()
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win,
                        1.0 / math.sqrt(wl.d), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), go)


def test_fused_position_outside_table_is_reported():
    wl = W.make_dense("fused_badpos", 15, 3, 64, 512, [300, 400, 500])
    table = W.rope_table(wl.seed, 450, W.ROPE_DIM)
    # rows 0 and 2 outside [0, 450): reported, not rotated; row 1 rotated
    _fused_case(wl, table=table, pos=[-1, 399, 450], bad_rows=(0, 2))


def test_fused_fp8_only_output():
    """out (float32) may be NULL: the FP8 buffer alone is written."""
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("fused_fp8only", 16, 2, 64, 512, [900, 64])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    ctx = P.Context(wl.d, wl.H)
    dev = torch_dev()
    table = W.rope_table(wl.seed, 1000, W.ROPE_DIM)
    o8 = torch.zeros(wl.B, wl.H, wl.d, dtype=torch.uint8, device=dev)
    ctx.pkv_decode_attn_fused(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win,
                              1.0 / math.sqrt(wl.d), i32(wl.rope_pos()), torch.from_numpy(table).to(dev),
                              W.ROPE_DIM, W.OUT_SCALE, o8)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    g8 = o8.cpu().numpy()
    for b in range(wl.B):
        Or, _, _ = C.expected_decode_fused(wl, Kp, Vp, ts, ts, tw, tw, b, table, W.ROPE_DIM, W.OUT_SCALE)
        assert_fp8_codes(g8[b], Or, W.OUT_SCALE, f"FP8 seq {b}")


def test_fused_host_validation():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("fused_val", 17, 1, 64, 512, [128])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    ctx = P.Context(wl.d, wl.H)
    dev = torch_dev()
    table = torch.from_numpy(W.rope_table(wl.seed, 200, 64)).to(dev)
    o8 = torch.empty(1, 64, 512, dtype=torch.uint8, device=dev)
    args = (q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win, 0.04, i32([5]))
    for rd, sc, want in [(60, 1.0, P.ERR_INVALID_ARG), (0, 1.0, P.ERR_INVALID_ARG), (520, 1.0, P.ERR_INVALID_ARG),
                         (64, 0.0, P.ERR_INVALID_ARG), (64, float("inf"), P.ERR_INVALID_ARG)]:
        with pytest.raises(P.PkvError) as e:
            ctx.pkv_decode_attn_fused(*args, table, rd, sc, o8)
        assert e.value.status == want, (rd, sc)
    # a window V scale far from the cache's: the tensor-core kernel (which holds the fusion) declines
    win2 = P.Window(win.k, win.v, tw, float(ts) * 1000.0)
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_decode_attn_fused(args[0], cache, args[2], args[3], win2, 0.04, args[6], table, 64, 1.0, o8)
    assert e.value.status == P.ERR_UNSUPPORTED
