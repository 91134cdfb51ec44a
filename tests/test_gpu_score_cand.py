"""GPU parity of candidate-list index scoring (only a fixed candidate set per
sequence is scored, then top-k among the candidates).

Scores of the valid candidates are compared element-wise (relative 1e-5 of the
score scale); the selected positions must be the oracle's candidate top-k,
except members within 1e-5 relative of the k-th score; -1 padded when a row
has fewer than k candidates.
"""
import numpy as np
import pytest

import workloads as W
from helpers import assert_scores_close, i32, torch_dev
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F

pytestmark = pytest.mark.gpu


def _cand_lists(wl, n, seed):
    """Ascending candidate positions per sequence (min(n, L) of them), -1 padded to n."""
    rng = np.random.default_rng(seed)
    out = np.full((wl.B, n), -1, np.int32)
    for b in range(wl.B):
        L = int(wl.seq_len[b])
        m = min(n, L)
        out[b, :m] = np.sort(rng.choice(L, size=m, replace=False))
    return out


def _cand_case(wl, cand, k, keys_override=None):
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    ts = np.float32(48 / 2688)
    pool = C.Pools(wl.num_pages, 128, "i")
    for p in range(wl.num_pages):
        rows = wl.index_rows(p) if keys_override is None else keys_override(p)
        c, s = F.nvfp4_quantize(rows, ts)
        pool.store(p, np.arange(64), c, s)
    qf = wl.index_q()
    tq = F.tensor_scale_fp8(qf)
    qc = F.fp8_quantize(qf, tq)
    w = wl.index_w()
    ic = P.IdxCache(torch.from_numpy(pool.data).to(dev), torch.from_numpy(pool.scale).to(dev), float(ts))
    ctx = P.Context(512, 64)
    B, n = cand.shape
    out_idx = torch.empty(B, k, dtype=torch.int32, device=dev)
    out_score = torch.empty(B, n, device=dev)
    ctx.pkv_score_topk_cand(torch.from_numpy(qc).to(dev), float(tq), torch.from_numpy(w).to(dev), ic,
                            i32(wl.page_table), i32(cand), k, out_idx, out_score)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    gi, gs = out_idx.cpu().numpy(), out_score.cpu().numpy()
    for b in range(B):
        valid = cand[b][cand[b] >= 0].astype(np.int64)
        rows = []
        for t in valid:
            codes, scales = pool.load(int(wl.page_table[b, t >> 6]))
            rows.append(F.nvfp4_dequantize(codes, scales, ts)[t & 63])
        khat = np.stack(rows)
        qhat = F.fp8_dequantize(qc[b], tq)
        ref = A.index_score(qhat, w[b].astype(np.float64), khat)
        assert_scores_close(gs[b, :len(valid)], qhat, w[b], khat, f"candidate scores seq {b}")
        # positions -> candidate indices, then the same set check as the dense path
        sel = gi[b]
        assert np.isin(sel[sel >= 0], valid).all(), f"seq {b}: a selected position is not a candidate"
        as_idx = np.where(sel >= 0, np.searchsorted(valid, np.maximum(sel, 0)), -1)
        ok, why = A.topk_matches(as_idx, ref, k)
        assert ok, f"candidate top-k seq {b}: {why}"
        want = A.topk_cand(ref, valid, k)
        assert (sel[:len(valid)] >= 0).sum() == (want >= 0).sum()
    return gi


def test_cand_scoring_ragged():
    wl = W.make_dense("cand", 30, 3, 64, 512, [9000, 3000, 500])
    _cand_case(wl, _cand_lists(wl, 1200, 31), 256)


def test_cand_fewer_than_k_pads():
    wl = W.make_dense("cand_small", 32, 2, 64, 512, [4000, 70])
    cand = _cand_lists(wl, 40, 33)
    cand[1, 10:] = -1                                    # 10 candidates only
    gi = _cand_case(wl, cand, 64)
    assert (gi[0, :40] == cand[0]).all() and (gi[0, 40:] == -1).all()
    assert (gi[1, :10] == cand[1, :10]).all() and (gi[1, 10:] == -1).all()


def test_cand_ties_take_lowest_positions():
    """Identical keys: every candidate scores the same; the k lowest candidate positions win."""
    wl = W.make_dense("cand_ties", 34, 1, 64, 512, [20000])
    row = W.normal_rows(0, 97, (0,), 1, 128)
    cand = _cand_lists(wl, 3000, 35)
    gi = _cand_case(wl, cand, 100, keys_override=lambda p: np.repeat(row, 64, axis=0))
    assert (gi[0] == cand[0, :100]).all()


def test_cand_unmapped_page_is_reported():
    """A candidate whose page is not in the page table sets the error word (no fault)."""
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    wl = W.make_dense("cand_bad", 36, 1, 64, 512, [1000])
    ic = P.IdxCache.empty(wl.num_pages, 48 / 2688, device=dev)
    pt = wl.page_table.copy()
    pt[0, 3] = -1
    cand = np.array([[1, 2, 200, 999]], np.int32)           # 200 lies in page 3
    ctx = P.Context(512, 64)
    out_idx = torch.empty(1, 4, dtype=torch.int32, device=dev)
    q = torch.zeros(1, 64, 128, dtype=torch.uint8, device=dev)
    w = torch.ones(1, 64, device=dev)
    ctx.pkv_score_topk_cand(q, 1.0, w, ic, i32(pt), i32(cand), 4, out_idx)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.ERR_BAD_PAGE
