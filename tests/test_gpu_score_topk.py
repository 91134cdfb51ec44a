"""GPU parity of the sparse index scoring and exact top-k.

Scores are compared position by position against an FP32-accumulation error
bound (helpers.assert_scores_close); the top-k set must equal the oracle's,
except for members within 1e-5 relative of the k-th score; positions must be
ascending, unique, -1 padded when L < k.
"""
import numpy as np
import pytest

import workloads as W
from helpers import assert_scores_close, i32, torch_dev
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F

pytestmark = pytest.mark.gpu


def _index_case(wl, k, keys_override=None, w_override=None, qc_override=None, quantize_on_device=False):
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    ts = np.float32(48 / 2688)
    pool = C.Pools(wl.num_pages, 128, "i")
    for p in range(wl.num_pages):
        rows = wl.index_rows(p) if keys_override is None else keys_override(p)
        c, s = F.nvfp4_quantize(rows, ts)
        pool.store(p, np.arange(64), c, s)
    if qc_override is None:
        qf = wl.index_q()
        tq = F.tensor_scale_fp8(qf)
        qc = F.fp8_quantize(qf, tq)
    else:
        qc, tq = qc_override
    w = wl.index_w() if w_override is None else w_override
    ic = P.IdxCache(torch.from_numpy(pool.data).to(dev), torch.from_numpy(pool.scale).to(dev), float(ts))
    ctx = P.Context(512, 64)
    Lmax = wl.page_table.shape[1] * 64
    out_idx = torch.empty(wl.B, k, dtype=torch.int32, device=dev)
    out_score = torch.empty(wl.B, Lmax, device=dev)
    wd, pt, sl = torch.from_numpy(w).to(dev), i32(wl.page_table), i32(wl.seq_len)
    if quantize_on_device:
        # the library's FP8 encode feeds the scoring launch directly: same stream,
        # no synchronization in between (dependent launch keeps the order)
        qf_dev = torch.from_numpy(np.ascontiguousarray(qf, np.float32)).to(dev)
        torch.cuda.synchronize()
        q_dev = torch.empty(qc.shape, dtype=torch.uint8, device=dev)
        P.pkv_quantize_fp8(qf_dev, float(tq), q_dev)
    else:
        q_dev = torch.from_numpy(qc).to(dev)
    ctx.pkv_score_topk(q_dev, float(tq), wd, ic, pt, sl, k, out_idx, out_score)
    torch.cuda.synchronize()
    assert ctx.pkv_get_error() == P.OK
    if quantize_on_device:
        assert np.array_equal(q_dev.cpu().numpy(), qc), "device FP8 encode differs from the oracle's"
    gi, gs = out_idx.cpu().numpy(), out_score.cpu().numpy()
    for b in range(wl.B):
        L = int(wl.seq_len[b])
        khat = np.concatenate([F.nvfp4_dequantize(*pool.load(int(wl.page_table[b, j])), ts)
                               for j in range((L + 63) // 64)])[:L]
        qhat = F.fp8_dequantize(qc[b], tq)
        ref = A.index_score(qhat, w[b].astype(np.float64), khat)
        assert_scores_close(gs[b, :L], qhat, w[b], khat, f"scores seq {b}")
        ok, why = A.topk_matches(gi[b], ref, k)
        assert ok, f"top-k seq {b}: {why}"
    return gi


def test_score_topk_ragged():
    wl = W.make_dense("score", 20, 3, 64, 512, [9000, 2500, 100])
    _index_case(wl, 256)


def test_topk_larger_than_length_pads():
    wl = W.make_dense("score_small", 21, 2, 64, 512, [50, 1])
    gi = _index_case(wl, 64)
    assert (gi[0, :50] == np.arange(50)).all() and (gi[0, 50:] == -1).all()
    assert gi[1, 0] == 0 and (gi[1, 1:] == -1).all()


def test_topk_all_ties_take_lowest_positions():
    """Identical keys give identical scores: the k lowest positions win (candidate overflow path)."""
    wl = W.make_dense("ties", 22, 1, 64, 512, [20000])
    row = W.normal_rows(0, 99, (0,), 1, 128)
    gi = _index_case(wl, 100, keys_override=lambda p: np.repeat(row, 64, axis=0))
    assert (gi[0] == np.arange(100)).all()


def test_topk_many_near_ties():
    """Keys drawn from a handful of distinct rows: large tie groups at the boundary."""
    wl = W.make_dense("near_ties", 23, 2, 64, 512, [6000, 7000])
    rows = W.normal_rows(0, 98, (0,), 5, 128)
    pick = lambda p: rows[np.random.default_rng(p).integers(0, 5, 64)]
    gi = _index_case(wl, 1000, keys_override=pick)
    for b in range(2):
        assert (np.diff(gi[b]) > 0).all()


def test_planted_tokens_selected():
    wl = W.make_dense("plant", 24, 1, 64, 512, [4096])
    qf = wl.index_q()[0]
    w = wl.index_w()
    planted = {(3, 7), (40, 0), (63, 63)}

    def keys(p):
        r = wl.index_rows(p)
        for (pp, s) in planted:
            if p == int(wl.page_table[0, pp]):
                r[s] = 4 * qf[0] / np.linalg.norm(qf[0]) * 10
        return r
    gi = _index_case(wl, 16, keys_override=keys)
    for (pp, s) in planted:
        assert 64 * pp + s in set(gi[0].tolist())


def test_score_queries_of_every_magnitude():
    """FP8 query codes over the whole E4M3 range (448 down to the 2^-9 subnormal, both
    signs) in every 16-channel block, blocks mixing the largest and smallest
    magnitudes, a head of zeros and an all-zero query: the largest number of FP4
    query terms the kernel builds, each score within the FP32 bound (exactly 0 for
    the zero query)."""
    wl = W.make_dense("qmag", 23, 3, 64, 512, [3000, 1500, 700])
    rng = np.random.default_rng(23)
    valid = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    qc = rng.choice(valid, size=(3, 64, 128)).astype(np.uint8)
    qc[0, 0, :] = 0x7E                     # 448 everywhere
    qc[0, 1, :] = 0x01                     # 2^-9 everywhere
    qc[0, 2, 0::2], qc[0, 2, 1::2] = 0x7E, 0x81     # 448 and -2^-9 side by side
    qc[0, 3, :] = 0x00
    qc[1, :, :16] = 0xFE                   # -448 in block 0 of every head
    qc[2] = 0                              # zero query: every score is exactly 0
    _index_case(wl, 200, qc_override=(qc, np.float32(0.0125)))


def test_score_reads_queries_encoded_just_before_on_the_stream():
    """FP8 index queries encoded by the library on the device and scored by the
    next call on the same stream without a synchronization: the codes equal the
    oracle's bit for bit and the scores and top-k match the oracle."""
    wl = W.make_dense("qdev", 24, 3, 64, 512, [5000, 2100, 900])
    _index_case(wl, 300, quantize_on_device=True)
