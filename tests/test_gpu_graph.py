"""The decode and sparse-selection calls capture into a CUDA graph: replays give
the same bytes as eager calls (the calls allocate nothing and never synchronize)."""
import math

import numpy as np
import pytest

import workloads as W
from helpers import i32, torch_dev, upload_cache, window_tensors, q_tensor
from oracle import cache as C
from oracle import formats as F

pytestmark = pytest.mark.gpu


def _capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                   # warm-up on the side stream
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_graph_replay_matches_eager():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("graph", 40, 3, 64, 512, [3000, 700, 1500])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    ctx = P.Context(wl.d, wl.H)
    q = q_tensor(wl.q_bits())
    pt, sl = i32(wl.page_table), i32(wl.seq_len)
    ws = ctx.workspace(P.OP_DECODE, wl.B, wl.page_table.shape[1] * 64)
    dev = torch_dev()
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    scale = 1.0 / math.sqrt(wl.d)
    call = lambda: ctx.pkv_decode_attn(q, cache, pt, sl, win, scale, out, lse, ws=ws)
    call()
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    g = _capture(call)
    out.zero_()
    lse.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_sparse_step_graph_replay_matches_eager():
    """Candidate scoring + top-k + sparse decode, captured as one graph."""
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    wl = W.make_dense("graph_sparse", 41, 2, 64, 512, [5000, 2600])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    pool = C.Pools(wl.num_pages, 128, "i")
    for p in range(wl.num_pages):
        c, s = F.nvfp4_quantize(wl.index_rows(p), ts)
        pool.store(p, np.arange(64), c, s)
    ic = P.IdxCache(torch.from_numpy(pool.data).to(dev), torch.from_numpy(pool.scale).to(dev), float(ts))
    qf = wl.index_q()
    tq = F.tensor_scale_fp8(qf)
    qc = torch.from_numpy(F.fp8_quantize(qf, tq)).to(dev)
    w = torch.from_numpy(wl.index_w()).to(dev)
    cand = i32(wl.cand_lists(1000))
    k = 256
    ctx = P.Context(wl.d, wl.H)
    q = q_tensor(wl.q_bits())
    pt, sl = i32(wl.page_table), i32(wl.seq_len)
    ws_s = ctx.workspace(P.OP_SCORE_CAND, wl.B, 1000)
    ws_d = ctx.workspace(P.OP_DECODE_SPARSE, wl.B, k)
    sel = torch.empty(wl.B, k, dtype=torch.int32, device=dev)
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    scale = 1.0 / math.sqrt(wl.d)

    def step():
        ctx.pkv_score_topk_cand(qc, float(tq), w, ic, pt, cand, k, sel, ws=ws_s)
        ctx.pkv_decode_attn(q, cache, pt, sl, win, scale, out, lse, ws=ws_d, sel_idx=sel)
    step()
    torch.cuda.synchronize()
    ref = (sel.clone(), out.clone(), lse.clone())
    g = _capture(step)
    sel.fill_(-7)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    assert torch.equal(sel, ref[0]) and torch.equal(out, ref[1]) and torch.equal(lse, ref[2])
