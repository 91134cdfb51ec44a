"""GPU parity of the NVFP4 append and FP8 encode: bytes must match the oracle bit for bit."""
import numpy as np
import pytest

import workloads as W
from helpers import i32, torch_dev
from oracle import cache as C
from oracle import formats as F

pytestmark = pytest.mark.gpu


def _gpu_fill(ctx, wl, ts_k, ts_v, order_seed=0, chunk=4096):
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    cache = P.KVCache.empty(wl.num_pages, wl.d, float(ts_k), float(ts_v))
    pt = i32(wl.page_table)
    segs = []
    for (b, t0, t1) in wl.fill_segments():
        segs += [(b, t) for t in range(t0, t1)]
    order = np.random.default_rng(order_seed).permutation(len(segs))   # arbitrary order, many per page
    for s in range(0, len(order), chunk):
        idx = order[s:s + chunk]
        bs = np.array([segs[i][0] for i in idx], np.int32)
        ts = np.array([segs[i][1] for i in idx], np.int32)
        kr = np.stack([wl.token_rows(W.T_K, int(b), int(t), int(t) + 1)[0] for b, t in zip(bs, ts)])
        vr = np.stack([wl.token_rows(W.T_V, int(b), int(t), int(t) + 1)[0] for b, t in zip(bs, ts)])
        ctx.pkv_append_kv(torch.from_numpy(kr).to(dev), torch.from_numpy(vr).to(dev), i32(bs), i32(ts), cache, pt)
    torch.cuda.synchronize()
    return cache


@pytest.mark.parametrize("d,H", [(512, 64), (128, 8), (256, 16)])
def test_append_bytes_match_oracle(d, H):
    import precision_kv_cache_gb300 as P
    wl = W.make_shared_prefix("append", 3, 4, H, d, [333, 200, 130, 129], 2, 128, append=False)
    ts_k, _ = C.tensor_scales(wl)
    ts_v = np.float32(ts_k * np.float32(0.5))       # a second scale exercises saturation
    Kp, Vp = C.fill_pages(wl, ts_k, ts_v)
    ctx = P.Context(d, H)
    cache = _gpu_fill(ctx, wl, ts_k, ts_v)
    assert ctx.pkv_get_error() == P.OK
    for name, g, r in (("k_data", cache.k_data, Kp.data), ("k_scale", cache.k_scale, Kp.scale),
                       ("v_data", cache.v_data, Vp.data), ("v_scale", cache.v_scale, Vp.scale)):
        g = g.cpu().numpy()
        bad = np.argwhere(g != r)
        assert bad.size == 0, f"{name}: {len(bad)} bytes differ, first at {bad[:3]}"


def test_append_overwrites_and_edge_values():
    """Overwriting a token replaces its nibbles only; ties, saturation, zero blocks, tiny values."""
    import torch
    import precision_kv_cache_gb300 as P
    d, dev = 128, torch_dev()
    wl = W.make_dense("edge", 0, 1, 8, d, [64])
    ts = np.float32(0.01)
    g = np.random.default_rng(0)
    rows = (g.standard_normal((64, d)) * g.choice([1e-6, 0.05, 1, 30, 500], (64, 1))).astype(np.float32)
    rows[3] = 0.0
    rows[4, :16] = np.float32(6 * 448 * 0.01) * np.array([1, -1, .5, .25, .125, .75, -.75, 1.25, 2.5 / 6, 3.5 / 6,
                                                          5 / 6, 1.75 / 6, .01, -.01, 0, 1], np.float32)
    rows[5] = -1e-30
    cache = P.KVCache.empty(1, d, float(ts), float(ts))
    ctx = P.Context(d, 8)
    pt = i32(wl.page_table)
    # write garbage first, then the real rows in reverse order (overwrite path)
    junk = torch.randn(64, d, device=dev) * 10
    ctx.pkv_append_kv(junk, junk, i32(np.zeros(64)), i32(np.arange(64)), cache, pt)
    ctx.pkv_append_kv(torch.from_numpy(rows[::-1].copy()).to(dev), torch.from_numpy(rows[::-1].copy()).to(dev),
                      i32(np.zeros(64)), i32(np.arange(63, -1, -1)), cache, pt)
    torch.cuda.synchronize()
    Kp = C.Pools(1, d, "k"); Vp = C.Pools(1, d, "v")
    c, s = F.nvfp4_quantize(rows, ts)
    Kp.store(0, np.arange(64), c, s)
    Vp.store(0, np.arange(64), c, s)
    assert (cache.k_data.cpu().numpy() == Kp.data).all()
    assert (cache.k_scale.cpu().numpy() == Kp.scale).all()
    assert (cache.v_data.cpu().numpy() == Vp.data).all()
    assert (cache.v_scale.cpu().numpy() == Vp.scale).all()


def test_index_append_and_fp8_encode_match_oracle():
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    wl = W.make_dense("idx", 1, 2, 64, 512, [200, 70])
    ts = np.float32(48 / 2688)
    ic = P.IdxCache.empty(wl.num_pages, float(ts))
    ctx = P.Context(512, 64)
    ref = C.Pools(wl.num_pages, 128, "i")
    bs, ps, rows = [], [], []
    for b in range(wl.B):
        for j in range((int(wl.seq_len[b]) + 63) // 64):
            p = int(wl.page_table[b, j])
            n = min(64, int(wl.seq_len[b]) - 64 * j)
            r = wl.index_rows(p)[:n]
            c, s = F.nvfp4_quantize(r, ts)
            ref.store(p, np.arange(n), c, s)
            bs += [b] * n; ps += list(range(64 * j, 64 * j + n)); rows.append(r)
    ctx.pkv_append_index(torch.from_numpy(np.concatenate(rows)).to(dev), i32(bs), i32(ps), ic, i32(wl.page_table))
    torch.cuda.synchronize()
    assert (ic.data.cpu().numpy() == ref.data).all() and (ic.scale.cpu().numpy() == ref.scale).all()
    # FP8 encode: random values plus ties, saturation, tiny and negative-zero cases
    g = np.random.default_rng(2)
    x = np.concatenate([(g.standard_normal(100001) * 40).astype(np.float32),
                        np.array([1.0625, 1.1875, 460, -500, 2 ** -10, 1.5 * 2 ** -10, 1.5 * 2 ** -9, -1e-9, 0.0,
                                  232, 1e30, -0.0], np.float32)])
    tw = np.float32(1.0)
    out = torch.empty(x.size, dtype=torch.uint8, device=dev)
    P.pkv_quantize_fp8(torch.from_numpy(x).to(dev), float(tw), out)
    torch.cuda.synchronize()
    ref8 = F.fp8_quantize(x, tw)
    g8 = out.cpu().numpy()
    assert (g8 == ref8).all(), np.argwhere(g8 != ref8)[:5]
