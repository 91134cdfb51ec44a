"""Parity at the full sizes of the five bench configurations, in the launch
configuration bench.py times, on sampled outputs the oracle computes one by one.

The cache is filled through the product path (NVFP4 append of the seeded
rows), exactly as the benchmark does; the oracle rebuilds the bytes of the
sampled sequences from the same seeded rows (append parity is bit-exact, pinned
in test_gpu_append.py) and computes their outputs in float64.
"""
import concurrent.futures as cf
import math
import multiprocessing as mp
import os

import numpy as np
import pytest

import workloads as W
from helpers import assert_close, assert_scores_close, i32, torch_dev
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    n = max(1, min(16, len(os.sched_getaffinity(0)) - 1))
    ex = cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn"))
    yield ex
    ex.shutdown()


def _setup(name, pool):
    import torch
    import bench
    import precision_kv_cache_gb300 as P
    wl = bench._wl_cache(name)
    ts, tw = bench.tensor_scales()
    ctx = P.Context(wl.d, wl.H)
    cache, pt = bench.fill_cache(ctx, P, torch, wl, name, ts, ts, pool)
    dev = torch_dev()
    wk = bench.window_codes_gpu(P, torch, wl, tw, dev, lambda b: wl.window_rows(W.T_KW, b))
    wv = bench.window_codes_gpu(P, torch, wl, tw, dev, lambda b: wl.window_rows(W.T_VW, b))
    return wl, ctx, cache, pt, P.Window(wk, wv, tw, tw), np.float32(ts), np.float32(tw)


def _oracle_seq(wl, b, n_tok, ts):
    """Oracle pools holding the pages of tokens [0, n_tok) of sequence b."""
    pages = {int(wl.page_table[b, j]) for j in range((n_tok + 63) // 64)}
    return C.fill_pages(wl, ts, ts, pages=pages)


def test_fullsize_dense_decode_8k(pool):
    import torch
    wl, ctx, cache, pt, win, ts, tw = _setup("c1", pool)
    dev = torch_dev()
    q = torch.from_numpy(wl.q_bits().view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    scale = 1 / math.sqrt(wl.d)
    ctx.pkv_decode_attn(q, cache, pt, torch.from_numpy(wl.seq_len).to(dev), win, scale, out, lse)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == 0 and ctx.pkv_attn_path() == 2
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b in (0, 17, 31):
        Kp, Vp = _oracle_seq(wl, b, int(wl.seq_len[b]), ts)
        O, L = C.expected_decode(wl, Kp, Vp, ts, ts, tw, tw, b, scale=scale)
        assert_close(go[b], O, f"c1 O seq {b}")
        assert_close(gl[b], L, f"c1 LSE seq {b}")


def test_fullsize_fused_dense_decode_8k(pool):
    """Fused decode (query RoPE, inverse RoPE on O, FP8 output) at the 8K dense decode size."""
    import torch
    from helpers import assert_fp8_codes
    wl, ctx, cache, pt, win, ts, tw = _setup("c1", pool)
    dev = torch_dev()
    q = torch.from_numpy(wl.q_bits().view(np.int16)).to(dev).view(torch.bfloat16)
    pos = wl.rope_pos()
    table = W.rope_table(wl.seed, int(pos.max()) + 1, W.ROPE_DIM)
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    o8 = torch.empty(wl.B, wl.H, wl.d, dtype=torch.uint8, device=dev)
    scale = 1 / math.sqrt(wl.d)
    ctx.pkv_decode_attn_fused(q, cache, pt, torch.from_numpy(wl.seq_len).to(dev), win, scale, i32(pos),
                              torch.from_numpy(table).to(dev), W.ROPE_DIM, W.OUT_SCALE, o8, out, lse)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == 0 and ctx.pkv_attn_path() == 2
    go, gl, g8 = out.cpu().numpy(), lse.cpu().numpy(), o8.cpu().numpy()
    for b in (0, 31):
        Kp, Vp = _oracle_seq(wl, b, int(wl.seq_len[b]), ts)
        Or, L, _ = C.expected_decode_fused(wl, Kp, Vp, ts, ts, tw, tw, b, table, W.ROPE_DIM, W.OUT_SCALE,
                                           scale=scale)
        assert_close(go[b], Or, f"c1 fused O' seq {b}")
        assert_close(gl[b], L, f"c1 fused LSE seq {b}")
        assert_fp8_codes(g8[b], Or, W.OUT_SCALE, f"c1 fused FP8 seq {b}")


def test_fullsize_ragged_paged_decode_with_append(pool):
    import torch
    wl, ctx, cache, pt, win, ts, tw = _setup("c2", pool)
    dev = torch_dev()
    knew, vnew = wl.new_rows(W.T_KNEW), wl.new_rows(W.T_VNEW)
    pos = (wl.seq_len - 1).astype(np.int32)
    ctx.pkv_append_kv(torch.from_numpy(knew).to(dev), torch.from_numpy(vnew).to(dev), i32(np.arange(wl.B)), i32(pos),
                      cache, pt)
    q = torch.from_numpy(wl.q_bits().view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    scale = 1 / math.sqrt(wl.d)
    ctx.pkv_decode_attn(q, cache, pt, torch.from_numpy(wl.seq_len).to(dev), win, scale, out, lse)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == 0 and ctx.pkv_attn_path() == 2
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b in (0, 9, 63):            # group leaders and a member reading shared prefix pages
        L = int(wl.seq_len[b])
        pages = {int(wl.page_table[b, j]) for j in range((L + 63) // 64)}
        Kp, Vp = C.fill_pages(wl, ts, ts, pages=pages)
        C.append_tokens(wl, Kp, Vp, knew[b:b + 1], vnew[b:b + 1], [b], [L - 1], ts, ts)
        O, Lr = C.expected_decode(wl, Kp, Vp, ts, ts, tw, tw, b, scale=scale)
        assert_close(go[b], O, f"c2 O seq {b}")
        assert_close(gl[b], Lr, f"c2 LSE seq {b}")


def test_fullsize_sparse_scoring_topk_and_decode(pool):
    import torch
    import bench
    import precision_kv_cache_gb300 as P
    wl, ctx, cache, pt, win, ts, tw = _setup("c3", pool)
    dev = torch_dev()
    # index keys through the product append, as the bench does
    ic = P.IdxCache.empty(wl.num_pages, float(ts), device=dev)
    owner = {int(wl.page_table[b, j]): (b, j) for b in range(wl.B) for j in range(wl.page_table.shape[1])}
    pages = list(range(wl.num_pages))
    for pg, rows in pool.map(bench._gen_index, [("c3", pages[i:i + 512]) for i in range(0, len(pages), 512)]):
        bs = np.repeat([owner[p][0] for p in pg], 64).astype(np.int32)
        ps = np.concatenate([64 * owner[p][1] + np.arange(64) for p in pg]).astype(np.int32)
        ctx.pkv_append_index(torch.from_numpy(rows.reshape(-1, 128)).to(dev), i32(bs), i32(ps), ic, pt)
    qf = wl.index_q()
    tq = F.tensor_scale_fp8(qf)
    qc = F.fp8_quantize(qf, tq)
    w = wl.index_w()
    k = wl.topk
    Lmax = pt.shape[1] * 64
    sel = torch.empty(wl.B, k, dtype=torch.int32, device=dev)
    scores = torch.empty(wl.B, Lmax, device=dev)
    ctx.pkv_score_topk(torch.from_numpy(qc).to(dev), float(tq), torch.from_numpy(w).to(dev), ic, pt,
                       torch.from_numpy(wl.seq_len).to(dev), k, sel, scores)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == 0
    gsel, gsc = sel.cpu().numpy(), scores.cpu().numpy()
    for b in range(wl.B):
        assert (np.diff(gsel[b]) > 0).all() and gsel[b, 0] >= 0
    ref_sel = {}
    for b in (0, 3):                   # two sequences scored by the oracle (8192 pages each)
        L = int(wl.seq_len[b])
        khat = np.empty((L, 128))
        for j in range(L // 64):
            p = int(wl.page_table[b, j])
            c, s = F.nvfp4_quantize(wl.index_rows(p), ts)
            khat[64 * j:64 * j + 64] = F.nvfp4_dequantize(c, s, ts)
        qhat = F.fp8_dequantize(qc[b], tq)
        ref = A.index_score(qhat, w[b].astype(np.float64), khat)
        assert_scores_close(gsc[b, :L], qhat, w[b], khat, f"c3 scores seq {b}")
        ok, why = A.topk_matches(gsel[b], ref, k)
        assert ok, f"c3 top-k seq {b}: {why}"
        ref_sel[b] = A.topk(ref, k)
    # sparse decode over the oracle's selection (oracle -> GPU direction only)
    q = torch.from_numpy(wl.q_bits().view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty(wl.B, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, wl.H, device=dev)
    scale = 1 / math.sqrt(wl.d)
    sel_in = gsel.copy()
    for b, r in ref_sel.items():
        sel_in[b] = r
    ctx.pkv_decode_attn(q, cache, pt, torch.from_numpy(wl.seq_len).to(dev), win, scale, out, lse,
                        sel_idx=i32(sel_in))
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == 0 and ctx.pkv_attn_path() == 2
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    for b in (0, 3):
        idx = [int(t) for t in ref_sel[b]]
        rowsK = np.stack([wl.token_rows(W.T_K, b, t, t + 1)[0] for t in idx])
        rowsV = np.stack([wl.token_rows(W.T_V, b, t, t + 1)[0] for t in idx])
        K = F.nvfp4_dequantize(*F.nvfp4_quantize(rowsK, ts), ts)
        V = F.nvfp4_dequantize(*F.nvfp4_quantize(rowsV, ts), ts)
        kw, vw = C.window_codes(wl, tw, tw, b)
        O, Lr = A.decode(F.bf16_to_f64(wl.q_bits_seq(b)), K, V, F.fp8_dequantize(kw, tw), F.fp8_dequantize(vw, tw),
                         scale)
        assert_close(go[b], O, f"c3 O seq {b}")
        assert_close(gl[b], Lr, f"c3 LSE seq {b}")


def test_fullsize_bounded_replay(pool):
    import torch
    wl, ctx, cache, pt, win, ts, tw = _setup("c4", pool)
    dev = torch_dev()
    qh = np.stack([wl.replay_q_bits(b) for b in range(wl.B)])
    q = torch.from_numpy(qh.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty(wl.B, 128, wl.H, wl.d, device=dev)
    lse = torch.empty(wl.B, 128, wl.H, device=dev)
    scale = 1 / math.sqrt(wl.d)
    ctx.pkv_replay_attn(q, cache, pt, torch.from_numpy(wl.prefix_len).to(dev), win, scale, out, lse)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == 0 and ctx.pkv_attn_path() == 2
    for b in (0, 11):
        s = int(wl.prefix_len[b]) - 128
        Kp, Vp = _oracle_seq(wl, b, s, ts)
        K = C.dequant_seq(wl, Kp, ts, b, s)
        V = C.dequant_seq(wl, Vp, ts, b, s)
        kw, vw = C.window_codes(wl, tw, tw, b)
        rows = [0, 77, 127]
        O, Lr = A.replay(F.bf16_to_f64(qh[b]), K, V, F.fp8_dequantize(kw, tw), F.fp8_dequantize(vw, tw), scale,
                         rows=rows)
        go = out[b].cpu().numpy()
        gl = lse[b].cpu().numpy()
        for r in rows:
            assert_close(go[r], O[r], f"c4 O seq {b} row {r}")
            assert_close(gl[r], Lr[r], f"c4 LSE seq {b} row {r}")
