"""Pins of the oracle's page layout, attention, replay, merge, scoring and top-k.

Checks use hand-worked addresses (tests/golden), closed forms (single entry,
identical keys, zero scale), brute force in pure Python with math.fsum on tiny
inputs, and structural truths of bounded replay.
"""
import math

import numpy as np
import pytest

import workloads as W
from conftest import golden_lines
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F
from oracle import layout as LY


# ---------------------------------------------------------------- layout
def test_layout_golden_addresses():
    for line in golden_lines("layout_addresses.txt"):
        f = line.split()
        kind, d, t, j = f[0], int(f[1]), int(f[2]), int(f[3])
        if kind == "kdata":
            assert LY.k_data_index(d)[t, j] == int(f[4]), line
            assert LY._k_data_addr(t, j, d) == int(f[4]), line
        elif kind == "idata":
            assert LY.i_data_index()[t, j] == int(f[4]), line
            assert LY._i_data_addr(t, j) == int(f[4]), line
        elif kind == "kscale":
            assert LY.k_scale_index(d)[t, j] == int(f[4]), line
        elif kind == "vdata":
            a, hi = LY.v_data_index(d)
            assert a[t, j] == int(f[4]) and int(hi[t, j]) == int(f[5]), line
        elif kind == "vscale":
            assert LY.v_scale_index(d)[t, j] == int(f[4]), line


@pytest.mark.parametrize("d", [128, 256, 512])
def test_layout_is_a_bijection_and_roundtrips(d):
    # every byte of a page is used exactly once (K: one pair per byte; V: two nibbles per byte)
    kd = LY.k_data_index(d).ravel()
    assert np.array_equal(np.sort(kd), np.arange(LY.k_data_bytes(d)))
    if d == 128:
        idd = LY.i_data_index().ravel()
        assert np.array_equal(np.sort(idd), np.arange(LY.k_data_bytes(d)))
    ks = LY.k_scale_index(d).ravel()
    assert np.array_equal(np.sort(ks), np.arange(LY.k_scale_bytes(d)))
    va, vh = LY.v_data_index(d)
    key = va.ravel() * 2 + vh.ravel()
    assert np.array_equal(np.sort(key), np.arange(2 * LY.v_data_bytes(d)))
    g = np.random.default_rng(5)
    codes = g.integers(0, 16, (64, d)).astype(np.uint8)
    sc = g.integers(0, 127, (64, d // 16)).astype(np.uint8)
    for kind in (("k", "v", "i") if d == 128 else ("k", "v")):
        p = C.Pools(3, d, kind)
        # write odd then even slots in two calls, then all again: same bytes
        p.store(1, np.arange(1, 64, 2), codes[1::2], sc[1::2])
        p.store(1, np.arange(0, 64, 2), codes[0::2], sc[0::2])
        c2, s2 = p.load(1)
        assert (c2 == codes).all() and (s2 == sc).all()
        assert not p.data[0].any() and not p.data[2].any()
        # the per-token (loop) form reads the same values
        if kind == "v":
            c3, s3 = LY.load_v_token(p.data, p.scale, 1, 37, d)
        else:
            c3, s3 = LY.load_k_token(p.data, p.scale, 1, 37, d, index_keys=kind == "i")
        assert (c3 == codes[37]).all() and (s3 == sc[37]).all()


def test_v_layout_octet_words():
    # channel ch of the 8 tokens 8o..8o+7 form one little-endian 32-bit word
    d = 128
    p = C.Pools(1, d, "v")
    codes = np.zeros((64, d), np.uint8)
    codes[8:16, 5] = np.arange(1, 9)          # tokens 8..15, channel 5
    p.store(0, np.arange(64), codes, np.zeros((64, 8), np.uint8))
    word = int(p.data[0, 4 * (1 * d + 5):4 * (1 * d + 5) + 4].view("<u4")[0])
    assert word == 0x87654321


# ---------------------------------------------------------------- attention
def brute_attention(q, K, V, scale):
    """Pure-Python softmax attention of one head with math.fsum."""
    z = [scale * math.fsum(qi * ki for qi, ki in zip(q, k)) for k in K]
    m = max(z)
    p = [math.exp(zi - m) for zi in z]
    l = math.fsum(p)
    o = [math.fsum(pi * v[c] for pi, v in zip(p, V)) / l for c in range(len(V[0]))]
    return o, m + math.log(l)


def test_segment_matches_brute_force():
    g = np.random.default_rng(6)
    q = g.standard_normal((3, 8))
    K = g.standard_normal((11, 8)) * 2
    V = g.standard_normal((11, 5))
    O, L = A.segment(q, K, V, 0.7)
    for h in range(3):
        o, lse = brute_attention(q[h].tolist(), K.tolist(), V.tolist(), 0.7)
        assert np.allclose(O[h], o, rtol=1e-13, atol=1e-14)
        assert abs(L[h] - lse) < 1e-12


def test_single_entry_returns_v_exactly():
    g = np.random.default_rng(7)
    q = g.standard_normal((4, 16))
    K = g.standard_normal((1, 16))
    V = g.standard_normal((1, 16))
    O, L = A.segment(q, K, V, 0.25)
    assert (O == V[0]).all()
    assert np.allclose(L, 0.25 * q @ K[0], rtol=0, atol=1e-15)


def test_identical_keys_give_mean_of_v():
    g = np.random.default_rng(8)
    q = g.standard_normal((2, 16))
    K = np.repeat(g.standard_normal((1, 16)), 9, axis=0)
    V = g.standard_normal((9, 16))
    O, L = A.segment(q, K, V, 1.0)
    assert np.allclose(O, V.mean(0), rtol=1e-14, atol=1e-15)
    assert np.allclose(L, q @ K[0] + math.log(9), atol=1e-13)


def test_zero_scale_is_uniform_average():
    g = np.random.default_rng(9)
    O, L = A.segment(g.standard_normal((2, 4)), g.standard_normal((7, 4)),
                     np.arange(21.0).reshape(7, 3), 0.0)
    assert np.allclose(O, np.arange(21.0).reshape(7, 3).mean(0), atol=1e-14)
    assert np.allclose(L, math.log(7))


def test_empty_segment_and_merge_weight_zero():
    O, L = A.segment(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 3)), 1.0)
    assert (O == 0).all() and np.isneginf(L).all()
    g = np.random.default_rng(10)
    Ob = g.standard_normal((2, 3))
    Lb = g.standard_normal(2)
    Om, Lm = A.merge(O, L, Ob, Lb)
    assert np.allclose(Om, Ob) and np.allclose(Lm, Lb)
    Om, Lm = A.merge(O, L, O, L)
    assert (Om == 0).all() and np.isneginf(Lm).all()


def test_split_merge_equals_full_softmax():
    g = np.random.default_rng(11)
    q = g.standard_normal((5, 32))
    K = g.standard_normal((200, 32)) * 3
    V = g.standard_normal((200, 16))
    Of, Lf = A.segment(q, K, V, 1 / math.sqrt(32))
    cuts = [0, 17, 64, 130, 200]
    O, L = None, None
    for a, b in zip(cuts[:-1], cuts[1:]):
        Oi, Li = A.segment(q, K[a:b], V[a:b], 1 / math.sqrt(32))
        O, L = (Oi, Li) if O is None else A.merge(O, L, Oi, Li)
    assert np.allclose(O, Of, rtol=1e-13, atol=1e-14)
    assert np.allclose(L, Lf, rtol=1e-14, atol=1e-13)


def test_decode_is_softmax_over_global_then_window():
    g = np.random.default_rng(12)
    q = g.standard_normal((2, 8))
    K, V = g.standard_normal((6, 8)), g.standard_normal((6, 8))
    Kw, Vw = g.standard_normal((3, 8)), g.standard_normal((3, 8))
    O, L = A.decode(q, K, V, Kw, Vw, 0.5)
    for h in range(2):
        o, lse = brute_attention(q[h].tolist(), K.tolist() + Kw.tolist(), V.tolist() + Vw.tolist(), 0.5)
        assert np.allclose(O[h], o, atol=1e-13) and abs(L[h] - lse) < 1e-12


# ---------------------------------------------------------------- replay
def test_replay_structure():
    g = np.random.default_rng(13)
    R, H, d = 6, 2, 8
    q = g.standard_normal((R, H, d))
    K, V = g.standard_normal((10, d)), g.standard_normal((10, d))
    Kw, Vw = g.standard_normal((R, d)), g.standard_normal((R, d))
    O, L = A.replay(q, K, V, Kw, Vw, 0.3)
    for r in range(R):
        # row r == decode with the window clipped to entries [0, r]
        Od, Ld = A.decode(q[r], K, V, Kw[:r + 1], Vw[:r + 1], 0.3)
        assert np.allclose(O[r], Od, atol=1e-14) and np.allclose(L[r], Ld)
        # and is independent of later window entries (causality)
        Kw2 = Kw.copy(); Kw2[r + 1:] += 100.0
        O2, _ = A.replay(q, K, V, Kw2, Vw, 0.3, rows=[r])
        assert np.allclose(O2[r], O[r], atol=1e-14)
    # H = 128: the prefix is empty (s = 0); row 0 sees only window entry 0 -> V exactly
    O, L = A.replay(q, K[:0], V[:0], Kw, Vw, 0.3)
    assert (O[0] == Vw[0]).all()
    o, lse = brute_attention(q[3, 1].tolist(), Kw[:4].tolist(), Vw[:4].tolist(), 0.3)
    assert np.allclose(O[3][1], o, atol=1e-13)


# ---------------------------------------------------------------- scoring / top-k
def test_index_score_brute_force_and_single_head():
    g = np.random.default_rng(14)
    qh = g.standard_normal((4, 6))
    w = g.random(4)
    k = g.standard_normal((9, 6))
    s = A.index_score(qh, w, k)
    for t in range(9):
        ref = math.fsum(w[h] * max(0.0, math.fsum(qh[h, i] * k[t, i] for i in range(6))) for h in range(4))
        assert abs(s[t] - ref) < 1e-13
    s1 = A.index_score(qh[:1], np.ones(1), k)
    assert np.allclose(s1, np.maximum(k @ qh[0], 0), atol=1e-14)
    # negative weights are allowed by the definition
    s2 = A.index_score(qh, -w, k)
    assert np.allclose(s2, -s, atol=1e-14)


def test_topk_brute_force_ties_and_padding():
    s = np.array([3.0, 1.0, 3.0, 5.0, 3.0, 0.0, 3.0])
    assert A.topk(s, 3).tolist() == [0, 2, 3]        # 5, then the two lowest-index 3s
    assert A.topk(s, 1).tolist() == [3]
    assert A.topk(s, 9).tolist() == [0, 1, 2, 3, 4, 5, 6, -1, -1]
    g = np.random.default_rng(15)
    for _ in range(20):
        x = g.integers(0, 6, 50).astype(np.float64)
        k = int(g.integers(1, 50))
        ref = sorted(sorted(range(50), key=lambda i: (-x[i], i))[:k])
        assert A.topk(x, k).tolist() == ref


def test_topk_matches_accepts_only_boundary_swaps():
    s = np.array([10.0, 9.0, 8.0, 8.0 * (1 + 5e-6), 1.0])
    ok, _ = A.topk_matches(np.array([0, 1, 3]), s, 3)
    assert ok
    ok, _ = A.topk_matches(np.array([0, 1, 2]), s, 3)      # 8.0 within 1e-5 of S_k
    assert ok
    ok, _ = A.topk_matches(np.array([0, 2, 3]), s, 3)      # drops 9.0: not a near-tie
    assert not ok
    ok, _ = A.topk_matches(np.array([1, 0, 3]), s, 3)      # not ascending
    assert not ok


def test_planted_tokens_are_selected():
    g = np.random.default_rng(16)
    qh = g.standard_normal((8, 16))
    w = g.random(8)
    k = g.standard_normal((300, 16))
    plant = [5, 77, 200]
    for t in plant:
        k[t] = 20 * qh[0] / np.linalg.norm(qh[0])
    s = A.index_score(qh, w, k)
    assert set(plant) <= set(A.topk(s, 3).tolist())


# ---------------------------------------------------------------- cache build / read
def test_cache_fill_and_dequant_match_direct_quantization():
    wl = W.make_shared_prefix("t", 0, 4, 8, 128, [200, 260, 130, 199], 2, 128, append=True)
    ts, _ = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    for b in range(4):
        n = int(wl.fill_end[b])
        K = C.dequant_seq(wl, Kp, ts, b, n)
        rows = wl.token_rows(W.T_K, b, 0, n)
        c, s = F.nvfp4_quantize(rows, ts)
        assert (K == F.nvfp4_dequantize(c, s, ts)).all()
        V = C.dequant_seq(wl, Vp, ts, b, n)
        c, s = F.nvfp4_quantize(wl.token_rows(W.T_V, b, 0, n), ts)
        assert (V == F.nvfp4_dequantize(c, s, ts)).all()
    # groups share their first 2 pages physically
    assert (wl.page_table[0, :2] == wl.page_table[1, :2]).all()
    assert (wl.page_table[2, :2] == wl.page_table[3, :2]).all()
    assert wl.page_table[0, 0] != wl.page_table[2, 0]


def test_topk_cand_all_positions_is_dense_topk():
    """Candidate list = every position: the candidate top-k is the dense top-k."""
    rng = np.random.default_rng(7)
    s = rng.normal(size=300)
    s[[5, 17, 200]] = s.max() + 1.0               # planted maxima
    assert (A.topk_cand(s, np.arange(300), 40) == A.topk(s, 40)).all()


def test_topk_cand_brute_force_small():
    """Tiny cases against enumeration: positions of the k best candidates, ties to the lower position."""
    rng = np.random.default_rng(8)
    for _ in range(200):
        n = int(rng.integers(1, 9))
        cand = np.sort(rng.choice(50, size=n, replace=False))
        sc = rng.integers(0, 4, size=n).astype(np.float64)      # many ties
        k = int(rng.integers(1, 10))
        best = sorted(range(n), key=lambda i: (-sc[i], cand[i]))[:k]
        want = sorted(int(cand[i]) for i in best) + [-1] * (k - min(k, n))
        assert list(A.topk_cand(sc, cand, k)) == want


@pytest.mark.parametrize("d", [128, 256, 512])
def test_k_layout_rows_are_swizzled_operand_rows(d):
    # Read back by the rule of a K-major swizzled operand: the 16-byte chunk at
    # position p of row t in column block b holds logical chunk p XOR w(t), and a
    # row's column blocks are 64*R bytes apart; each column block of a page is a
    # [64][R] array of rows.  (A second formulation, by chunk position instead of
    # by channel, of the same byte map.)
    R = min(128, d // 2)
    g = np.random.default_rng(8)
    codes = g.integers(0, 16, (64, d)).astype(np.uint8)
    p = C.Pools(1, d, "k")
    p.store(0, np.arange(64), codes, np.zeros((64, d // 16), np.uint8))
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)        # [64][d/2]
    page = p.data[0]
    for t in range(64):
        w = t % 8 if R == 128 else (t // 2) % 4
        for b in range(d // 2 // R):
            row = page[b * 64 * R + t * R: b * 64 * R + (t + 1) * R]
            for pos in range(R // 16):
                logical = b * (R // 16) + (pos ^ w)
                assert (row[16 * pos:16 * pos + 16] == packed[t, 16 * logical:16 * logical + 16]).all()


def test_v_layout_chunks_are_contiguous_runs():
    # d = 512: the words of channels 128c .. 128c+127 of all 64 tokens form one
    # contiguous 4 KB run (chunk c), octet-major inside it
    d = 512
    p = C.Pools(1, d, "v")
    codes = np.zeros((64, d), np.uint8)
    codes[8:16, 300] = np.arange(1, 9)        # tokens 8..15 (octet 1), channel 300 (chunk 2, lane 44)
    codes[0:8, 511] = 15                      # octet 0, last channel
    p.store(0, np.arange(64), codes, np.zeros((64, 32), np.uint8))
    w = p.data[0].view("<u4")
    assert int(w[(2 * 8 + 1) * 128 + 44]) == 0x87654321
    assert int(w[(3 * 8 + 0) * 128 + 127]) == 0xFFFFFFFF
    assert np.count_nonzero(w) == 2


def test_append_tokens_and_dequant_tokens():
    """append_tokens writes the new token's own NVFP4 codes at slot pos % 64 of page
    page_table[b][pos // 64] and nothing else; dequant_tokens returns the same rows as
    the whole-sequence dequantization at the asked positions."""
    wl = W.make_shared_prefix("app", 3, 4, 8, 128, [200, 260, 130, 199], 2, 128, append=True)
    ts, _ = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    before = [(C.dequant_seq(wl, Kp, ts, b, int(wl.fill_end[b])), C.dequant_seq(wl, Vp, ts, b, int(wl.fill_end[b])))
              for b in range(wl.B)]
    kd0, vd0 = Kp.data.copy(), Vp.data.copy()
    knew, vnew = wl.new_rows(W.T_KNEW), wl.new_rows(W.T_VNEW)
    pos = (wl.seq_len - 1).astype(np.int32)
    C.append_tokens(wl, Kp, Vp, knew, vnew, np.arange(wl.B), pos, ts, ts)
    touched = set()
    for b in range(wl.B):
        L = int(wl.seq_len[b])
        K = C.dequant_seq(wl, Kp, ts, b, L)
        V = C.dequant_seq(wl, Vp, ts, b, L)
        assert (K[:L - 1] == before[b][0][:L - 1]).all() and (V[:L - 1] == before[b][1][:L - 1]).all()
        c, s = F.nvfp4_quantize(knew[b:b + 1], ts)
        assert (K[L - 1] == F.nvfp4_dequantize(c, s, ts)[0]).all()
        c, s = F.nvfp4_quantize(vnew[b:b + 1], ts)
        assert (V[L - 1] == F.nvfp4_dequantize(c, s, ts)[0]).all()
        touched.add(int(wl.page_table[b, (L - 1) // W.PAGE]))
        idx = np.random.default_rng(b).choice(L, size=min(L, 37), replace=False)
        assert (C.dequant_tokens(wl, Kp, ts, b, idx) == K[idx]).all()
        assert (C.dequant_tokens(wl, Vp, ts, b, idx) == V[idx]).all()
    # pages no append landed on keep their bytes
    for p in range(Kp.data.shape[0]):
        if p not in touched:
            assert (Kp.data[p] == kd0[p]).all() and (Vp.data[p] == vd0[p]).all()
