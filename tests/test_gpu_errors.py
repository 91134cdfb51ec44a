"""Failure reporting without a GPU fault: bad inputs are rejected on the host or
caught by the kernels' own bounds checks (skip the access, set the context's
error word), and the context stays usable afterwards."""
import math

import numpy as np
import pytest

import workloads as W
from helpers import i32, q_tensor, torch_dev, upload_cache, window_tensors
from oracle import cache as C

pytestmark = pytest.mark.gpu


def test_bad_page_ids_are_reported_not_faulted():
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("bad", 30, 2, 64, 512, [200, 100])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    ctx = P.Context(512, 64)
    pt = wl.page_table.copy()
    pt[0, 1] = wl.num_pages + 5          # out of the pool
    pt[1, 0] = -7
    dev = torch_dev()
    out = torch.empty(2, 64, 512, device=dev)
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(pt), i32(wl.seq_len), win, 1 / math.sqrt(512), out)
    assert ctx.pkv_get_error() == P.ERR_BAD_PAGE
    assert torch.isfinite(out).all()
    # a sequence longer than its page table is clamped and reported
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32([10 ** 6, 5]), win,
                        1 / math.sqrt(512), out)
    assert ctx.pkv_get_error() == P.ERR_BAD_PAGE
    # append through a bad page id
    x = torch.zeros(1, 512, device=dev)
    ctx.pkv_append_kv(x, x, i32([0]), i32([64]), cache, i32(pt))
    assert ctx.pkv_get_error() == P.ERR_BAD_PAGE
    # the context still works and the error word was cleared
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win,
                        1 / math.sqrt(512), out)
    assert ctx.pkv_get_error() == P.OK


def test_host_validation_rejects_before_launch():
    import torch
    import precision_kv_cache_gb300 as P
    ctx = P.Context(512, 64)
    dev = torch_dev()
    ic = P.IdxCache.empty(4, 0.01)
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_score_topk(torch.zeros(1, 64, 128, dtype=torch.uint8, device=dev), 1.0,
                           torch.zeros(1, 64, device=dev), ic, i32(np.zeros((1, 4))), i32([10]), 5000,
                           torch.empty(1, 5000, dtype=torch.int32, device=dev))
    assert e.value.status == P.ERR_INVALID_ARG
    small = torch.empty(8, dtype=torch.uint8, device=dev)
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_score_topk(torch.zeros(1, 64, 128, dtype=torch.uint8, device=dev), 1.0,
                           torch.zeros(1, 64, device=dev), ic, i32(np.zeros((1, 4))), i32([10]), 5,
                           torch.empty(1, 5, dtype=torch.int32, device=dev), ws=small)
    assert e.value.status == P.ERR_WORKSPACE
    with pytest.raises(P.PkvError) as e:
        P.Context(100, 64)
    assert e.value.status == P.ERR_UNSUPPORTED


def test_bounded_wait_gives_up_reports_timeout_and_recovers():
    """A wait that runs out, in the form the failure path is built for: CTA 0 never
    issues one K-tile copy (testing hook), so the MMA warp's bounded wait for it
    ends after a short limit (2e6 SM cycles, about a millisecond); the kernel sets
    the error word, the other roles leave their loops, every CTA drains the copies
    and MMAs it issued and frees its tensor memory.  The call reports
    PKV_ERR_TIMEOUT, and the next call on the same context is correct."""
    import torch
    import precision_kv_cache_gb300 as P
    from helpers import assert_close
    wl = W.make_dense("timeout", 31, 1, 64, 512, [1024])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, _, _ = window_tensors(wl, tw, tw)
    ctx = P.Context(512, 64)
    dev = torch_dev()
    out = torch.empty(1, 64, 512, device=dev)
    lse = torch.empty(1, 64, device=dev)
    scale = 1 / math.sqrt(512)
    ctx.pkv_set_test_hooks(2_000_000, 0)          # CTA 0's first K-tile copy is never issued
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win, scale, out, lse)
    assert ctx.pkv_get_error() == P.ERR_TIMEOUT
    ctx.pkv_set_test_hooks()                      # defaults: a long limit, no skipped copy
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), win, scale, out, lse)
    assert ctx.pkv_get_error() == P.OK
    O, L = C.expected_decode(wl, Kp, Vp, ts, ts, tw, tw, 0, scale=scale)
    assert_close(out.cpu().numpy()[0], O, "O after the timed-out call")
    assert_close(lse.cpu().numpy()[0], L, "LSE after the timed-out call")
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_set_test_hooks(10, -1)            # a limit below 1000 cycles is refused
    assert e.value.status == P.ERR_INVALID_ARG


def test_window_scale_ratio_outside_the_kernel_range_is_refused():
    """The window's V scale is folded into the f16 softmax weights, so tw_v / ts_v
    must lie in [2^-7, 2^7]: outside it every attention call returns
    PKV_ERR_UNSUPPORTED before launching anything (there is no second kernel)."""
    import torch
    import precision_kv_cache_gb300 as P
    wl = W.make_dense("ratio", 32, 2, 64, 512, [300, 200])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    cache = upload_cache(Kp, Vp, ts, ts)
    win, kw, vw = window_tensors(wl, tw, tw)
    bad = P.Window(win.k, win.v, float(tw), float(ts) * 2.0 ** -9)
    ctx = P.Context(512, 64)
    dev = torch_dev()
    out = torch.empty(2, 64, 512, device=dev)
    n0 = ctx.pkv_launch_count()
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), bad,
                            1 / math.sqrt(512), out)
    assert e.value.status == P.ERR_UNSUPPORTED
    with pytest.raises(P.PkvError) as e:
        ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), bad,
                            1 / math.sqrt(512), out, sel_idx=i32([[0, 1, 2, 3], [5, 6, 7, -1]]))
    assert e.value.status == P.ERR_UNSUPPORTED
    assert ctx.pkv_launch_count() == n0
    # inside the range the same call runs
    ok = P.Window(win.k, win.v, float(tw), float(ts) * 2.0 ** -7)
    ctx.pkv_decode_attn(q_tensor(wl.q_bits()), cache, i32(wl.page_table), i32(wl.seq_len), ok,
                        1 / math.sqrt(512), out)
    assert ctx.pkv_get_error() == P.OK
