"""GPU parity of decode attention (dense, sparse), bounded replay and the LSE merge.

The GPU consumes the oracle's cache bytes; outputs are compared element by
element with |gpu - oracle| <= 2e-3 + 1e-2 |oracle| (O and LSE).
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


def _decode_case(wl, win_len=None, sel=None, seed_scale=None):
    import torch
    import precision_kv_cache_gb300 as P
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, kw, vw = window_tensors(wl, tw, tw, win_len)
    ctx = P.Context(wl.d, wl.H)
    q = q_tensor(wl.q_bits())
    out = torch.empty(wl.B, wl.H, wl.d, device=torch_dev())
    lse = torch.empty(wl.B, wl.H, device=torch_dev())
    scale = 1.0 / math.sqrt(wl.d)
    sel_t = None if sel is None else i32(sel)
    ctx.pkv_decode_attn(q, cache, i32(wl.page_table), i32(wl.seq_len), win, scale, out, lse, sel_idx=sel_t)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(wl.B):
        L = int(wl.seq_len[b])
        n = 128 if win_len is None else int(win_len[b])
        if sel is None:
            K = C.dequant_seq(wl, Kp, ts, b, L)
            V = C.dequant_seq(wl, Vp, ts, b, L)
        else:
            idx = [int(t) for t in sel[b] if t >= 0]
            K = C.dequant_tokens(wl, Kp, ts, b, idx)
            V = C.dequant_tokens(wl, Vp, ts, b, idx)
        Kw = F.fp8_dequantize(kw[b, :n], tw)
        Vw = F.fp8_dequantize(vw[b, :n], tw)
        O, Lr = A.decode(F.bf16_to_f64(wl.q_bits_seq(b)), K, V, Kw, Vw, scale)
        assert_close(go[b], O, f"O seq {b}")
        assert_close(gl[b], Lr, f"LSE seq {b}")


def test_decode_tiny_dense_config():
    """The tiny dense decode configuration at full size: B=1, 8 heads, d=128, 1024 tokens + window."""
    _decode_case(W.config(0))


@pytest.mark.parametrize("d,H", [(512, 64), (128, 8), (256, 32), (512, 16)])
def test_decode_ragged(d, H):
    # ragged lengths: several 128-token tiles plus a partial tail, a single token, an empty prefix
    wl = W.make_dense("ragged", 5, 4, H, d, [1000, 1, 300, 129])
    _decode_case(wl, win_len=[128, 5, 0, 1])


@pytest.mark.parametrize("d,H", [(512, 64), (256, 16)])
def test_decode_many_short_rows(d, H):
    """Many short ragged rows: most CTA ranges hold several row ends (window tiles
    read through the V ring), some hold planning units only, windows of every
    length from empty to full."""
    rs = np.random.default_rng(11)
    B = 40
    lens = rs.integers(0, 400, size=B)
    lens[:4] = [0, 1, 64, 129]
    wins = rs.integers(0, 129, size=B)
    wins[:4] = [0, 128, 1, 31]
    wl = W.make_dense("short_rows", 12, B, H, d, lens)
    _decode_case(wl, win_len=list(int(w) for w in wins))


def test_decode_empty_everything():
    import torch
    wl = W.make_dense("empty", 6, 2, 64, 512, [0, 64])
    _decode_case(wl, win_len=[0, 0])


def test_decode_shared_prefix_with_append():
    """Ragged paged decode with shared prefix pages; the appended token is attended."""
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_shared_prefix("shared", 7, 6, 64, 512, [700, 640, 900, 500, 513, 450], 3, 384)
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    knew, vnew = wl.new_rows(W.T_KNEW), wl.new_rows(W.T_VNEW)
    pos = (wl.seq_len - 1).astype(np.int32)
    C.append_tokens(wl, Kp, Vp, knew, vnew, np.arange(wl.B), pos, ts, ts)
    # GPU: oracle bytes of the fill, then the GPU appends the new token
    Kf, Vf = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kf, Vf, ts, ts)
    ctx = P.Context(wl.d, wl.H)
    dev = torch_dev()
    ctx.pkv_append_kv(torch.from_numpy(knew).to(dev), torch.from_numpy(vnew).to(dev), i32(np.arange(wl.B)),
                      i32(pos), cache, i32(wl.page_table))
    torch.cuda.synchronize()
    assert (cache.k_data.cpu().numpy() == Kp.data).all() and (cache.v_data.cpu().numpy() == Vp.data).all()
    win, kw, vw = window_tensors(wl, tw, tw)
    q = q_tensor(wl.q_bits())
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    scale = 1.0 / math.sqrt(wl.d)
    ctx.pkv_decode_attn(q, cache, i32(wl.page_table), i32(wl.seq_len), win, scale, out, lse)
    torch.cuda.synchronize()
    for b in range(wl.B):
        O, Lr = C.expected_decode(wl, Kp, Vp, ts, ts, tw, tw, b, scale=scale)
        assert_close(out[b].cpu().numpy(), O, f"O seq {b}")
        assert_close(lse[b].cpu().numpy(), Lr, f"LSE seq {b}")


def test_decode_sparse_selected_positions():
    g = np.random.default_rng(9)
    wl = W.make_dense("sparse", 8, 3, 64, 512, [5000, 3000, 40])
    k = 96
    sel = np.full((3, k), -1, np.int32)
    for b, L in enumerate(wl.seq_len):
        n = min(k, int(L))
        sel[b, :n] = np.sort(g.choice(int(L), n, replace=False))
    _decode_case(wl, sel=sel)


def test_single_position_returns_v_exactly():
    """One global token and no window: O equals the dequantized V row (P = 1)."""
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("one", 10, 2, 64, 512, [1, 1])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw, [0, 0])
    ctx = P.Context(512, 64)
    out = torch.empty(2, 64, 512, device=torch_dev())
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win,
                        1 / math.sqrt(512), out)
    torch.cuda.synchronize()
    for b in range(2):
        V = C.dequant_seq(wl, Vp, ts, b, 1)[0]
        assert np.allclose(out[b].cpu().numpy(), np.broadcast_to(V, (64, 512)), rtol=2e-7, atol=0)


def test_replay_rows_match_oracle():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_replay("replay", 11, 2, 64, 512, [128, 128 + 333])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, kw, vw = window_tensors(wl, tw, tw)
    ctx = P.Context(512, 64)
    dev = torch_dev()
    q = np.stack([wl.replay_q_bits(b) for b in range(wl.B)])       # [B][128][H][d]
    out = torch.empty(wl.B, 128, 64, 512, device=dev)
    lse = torch.empty(wl.B, 128, 64, device=dev)
    scale = 1 / math.sqrt(512)
    ctx.pkv_replay_attn(q_tensor(q), cache, i32(wl.page_table), i32(wl.prefix_len), win, scale, out, lse)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(wl.B):
        s = int(wl.prefix_len[b]) - 128
        K = C.dequant_seq(wl, Kp, ts, b, s)
        V = C.dequant_seq(wl, Vp, ts, b, s)
        Kw = F.fp8_dequantize(kw[b], tw)
        Vw = F.fp8_dequantize(vw[b], tw)
        rows = [0, 1, 63, 64, 127] + list(np.random.default_rng(b).choice(128, 6, replace=False))
        O, Lr = A.replay(F.bf16_to_f64(q[b]), K, V, Kw, Vw, scale, rows=rows)
        for r in rows:
            assert_close(go[b, r], O[r], f"O seq {b} row {r}")
            assert_close(gl[b, r], Lr[r], f"LSE seq {b} row {r}")
    # H = 128: row 0 sees exactly one window entry
    V0 = F.fp8_dequantize(vw[0, 0], tw)
    assert np.allclose(go[0, 0], np.broadcast_to(V0, (64, 512)), rtol=2e-7, atol=0)


def test_merge_matches_oracle():
    import torch
    import precision_kv_cache_gb300 as P
    g = np.random.default_rng(12)
    rows, dv = 300, 512
    oa, ob = g.standard_normal((rows, dv)), g.standard_normal((rows, dv))
    la, lb = g.standard_normal(rows) * 5, g.standard_normal(rows) * 5
    la[:5] = -np.inf
    lb[3:8] = -np.inf
    dev = torch_dev()
    t = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(dev)
    o, l = torch.empty(rows, dv, device=dev), torch.empty(rows, device=dev)
    P.pkv_merge(t(oa), t(la), t(ob), t(lb), o, l)
    torch.cuda.synchronize()
    Or, Lr = A.merge(oa, la, ob, lb)
    assert_close(o.cpu().numpy(), Or, "merge O", atol=1e-5, rtol=1e-5)
    assert_close(l.cpu().numpy(), Lr, "merge LSE", atol=1e-5, rtol=1e-5)
    # in place (o, lse alias a)
    oa_t, la_t = t(oa), t(la)
    P.pkv_merge(oa_t, la_t, t(ob), t(lb), oa_t, la_t)
    torch.cuda.synchronize()
    assert_close(oa_t.cpu().numpy(), Or, "merge O in place", atol=1e-5, rtol=1e-5)
