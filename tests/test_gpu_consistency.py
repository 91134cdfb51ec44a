"""GPU self-consistency of decode and bounded replay: properties the outputs
must have whatever their values (GPU against GPU; the oracle parity of each
call is in test_gpu_attention.py).

* Where a page sits in the pool does not matter: moving every page (and the
  page table with it) gives bit-identical outputs.
* Two sequences that read the same pages and window with the same queries
  give the same outputs, up to the rounding of different split points.
* Bounded replay ("SWA bounded replay", vLLM blog): row r equals a decode of
  the same query over the global tokens [0, s) and the window entries [0, r].
"""
import math

import numpy as np
import pytest

import workloads as W
from helpers import assert_close, i32, q_tensor, torch_dev, upload_cache, window_tensors
from oracle import cache as C

pytestmark = pytest.mark.gpu

# The compared calls split a row at different points, so the P operand (rounded
# to f16 against the running maximum of the rows it has seen) can round
# differently: up to 2^-11 relative each way, hence 2^-10 on O.  The LSE sums
# FP32 probabilities and differs by FP32 rounding only.
TIGHT_O = dict(atol=1e-5, rtol=2.0 ** -10)
TIGHT_LSE = dict(atol=1e-5, rtol=1e-5)
# Replay against decode: the window tile's probabilities are scaled into f16
# against maxima that differ between the two calls, and small probabilities
# fall into f16's subnormal range differently (measured: 1 % on a 0.04 element
# of O).  Each call is within the oracle tolerance (2e-3 + 1e-2 |r|), so the two
# differ by at most twice it; a wrong window clip or global range differs by
# far more.
TWICE_ORACLE = dict(atol=4e-3, rtol=2e-2)


def _decode(ctx, wl, cache, pt, seq_len, win, q):
    import torch
    B = len(seq_len)
    out = torch.empty(B, wl.H, wl.d, device=torch_dev())
    lse = torch.empty(B, wl.H, device=torch_dev())
    ctx.pkv_decode_attn(q, cache, i32(pt), i32(seq_len), win, 1 / math.sqrt(wl.d), out, lse)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy()


def test_page_placement_does_not_change_outputs():
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("placement", 31, 3, 64, 512, [1000, 333, 2050])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    ctx = P.Context(wl.d, wl.H)
    q = q_tensor(wl.q_bits())
    o1, l1 = _decode(ctx, wl, upload_cache(Kp, Vp, ts, ts), wl.page_table, wl.seq_len, win, q)
    # physical page p moves to perm[p]
    perm = np.random.default_rng(5).permutation(wl.num_pages)
    K2, V2 = C.Pools(wl.num_pages, wl.d, "k"), C.Pools(wl.num_pages, wl.d, "v")
    K2.data[perm], K2.scale[perm] = Kp.data, Kp.scale
    V2.data[perm], V2.scale[perm] = Vp.data, Vp.scale
    pt2 = np.where(wl.page_table >= 0, perm[np.maximum(wl.page_table, 0)], -1).astype(np.int32)
    o2, l2 = _decode(ctx, wl, upload_cache(K2, V2, ts, ts), pt2, wl.seq_len, win, q)
    assert ctx.pkv_get_error() == P.OK
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sequences_reading_the_same_pages_agree():
    import precision_kv_cache_gb300 as P
    # three sequences, all pages shared (prefix = whole length), queries and windows copied from sequence 0
    wl = W.make_shared_prefix("same_pages", 32, 3, 64, 512, [1280, 1280, 1280], 3, 1280, append=False)
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    win.k[1:] = win.k[0]
    win.v[1:] = win.v[0]
    qb = wl.q_bits()
    qb[1:] = qb[0]
    ctx = P.Context(wl.d, wl.H)
    o, l = _decode(ctx, wl, upload_cache(Kp, Vp, ts, ts), wl.page_table, wl.seq_len, win, q_tensor(qb))
    assert ctx.pkv_get_error() == P.OK
    for b in (1, 2):
        assert_close(o[b], o[0], f"O seq {b} vs 0", **TIGHT_O)
        assert_close(l[b], l[0], f"LSE seq {b} vs 0", **TIGHT_LSE)


def test_replay_row_equals_decode_over_its_entries():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_replay("replay_vs_decode", 33, 1, 64, 512, [128 + 700])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)       # the chunk window: FP8 K/V of positions s .. H-1
    ctx = P.Context(512, 64)
    dev = torch_dev()
    q = wl.replay_q_bits(0)                      # [128][H][d]
    out = torch.empty(1, 128, 64, 512, device=dev)
    lse = torch.empty(1, 128, 64, device=dev)
    scale = 1 / math.sqrt(512)
    ctx.pkv_replay_attn(q_tensor(q[None]), cache, i32(wl.page_table), i32(wl.prefix_len), win, scale, out, lse)
    torch.cuda.synchronize()
    go, gl = out.cpu().numpy()[0], lse.cpu().numpy()[0]
    # the same rows as decodes: global [0, s), window entries [0, r]
    rows = [0, 5, 64, 127]
    s = int(wl.prefix_len[0]) - 128
    Bd = len(rows)
    wd = P.Window(win.k.repeat(Bd, 1, 1), win.v.repeat(Bd, 1, 1), win.tw_k, win.tw_v, i32([r + 1 for r in rows]))
    od, ld = _decode(ctx, wl, cache, np.repeat(wl.page_table[:1], Bd, 0), np.full(Bd, s, np.int32), wd,
                     q_tensor(np.ascontiguousarray(q[rows])))
    assert ctx.pkv_get_error() == P.OK
    for i, r in enumerate(rows):
        assert_close(go[r], od[i], f"replay row {r} vs decode", **TWICE_ORACLE)
        assert_close(gl[r], ld[i], f"replay LSE row {r} vs decode", **TIGHT_LSE)
