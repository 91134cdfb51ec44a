"""Pins of the oracle's rotary embedding and fused decode (query RoPE, attention,
inverse RoPE on the output, FP8 output; vLLM blog, "MegaAttention avec KV
compressé NVFP4").

The rotation is checked against basis vectors turned by a quarter turn,
against complex multiplication by e^{i theta} (a second formulation), for
inversion, length preservation and the relative-position property of angles
linear in the position; the fused decode against the plain decode with an
identity table and against a second route that turns the keys the other way
instead of the query.
"""
import numpy as np
import pytest

import workloads as W
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F


def _complex_rotate(x, theta, rope_dim, sign=1.0):
    """Second formulation: pair (x0, x1) as x0 + i x1, multiplied by e^{i sign theta}."""
    x = np.array(x, np.float64)
    d = x.shape[-1]
    z = x[..., d - rope_dim::2] + 1j * x[..., d - rope_dim + 1::2]
    z = z * np.exp(1j * sign * np.asarray(theta))
    y = x.copy()
    y[..., d - rope_dim::2] = z.real
    y[..., d - rope_dim + 1::2] = z.imag
    return y


@pytest.mark.parametrize("d,rd", [(16, 8), (128, 64), (64, 64)])
def test_quarter_turn_moves_basis_vectors(d, rd):
    # cos = 0, sin = 1: e_{2i} -> e_{2i+1}, e_{2i+1} -> -e_{2i} inside the rotated part
    cos, sin = np.zeros(rd // 2), np.ones(rd // 2)
    for i in range(rd // 2):
        c0 = d - rd + 2 * i
        e = np.zeros(d); e[c0] = 1.0
        y = A.rope(e, cos, sin, rd)
        want = np.zeros(d); want[c0 + 1] = 1.0
        assert np.array_equal(y, want)
        e = np.zeros(d); e[c0 + 1] = 1.0
        y = A.rope(e, cos, sin, rd)
        want = np.zeros(d); want[c0] = -1.0
        assert np.array_equal(y, want)
        # the inverse turns the other way
        y = A.rope(e, cos, sin, rd, inverse=True)
        want = np.zeros(d); want[c0] = 1.0
        assert np.array_equal(y, want)


def test_channels_outside_the_rotated_part_pass_through():
    r = np.random.default_rng(1)
    x = r.standard_normal((3, 5, 96))
    th = r.random(16) * 6.28
    y = A.rope(x, np.cos(th), np.sin(th), 32)
    assert np.array_equal(y[..., :64], x[..., :64])
    assert np.array_equal(A.rope(x, [], [], 0), x)


@pytest.mark.parametrize("inverse", [False, True])
def test_matches_complex_multiplication(inverse):
    r = np.random.default_rng(2)
    x = r.standard_normal((7, 128))
    th = r.random(32) * 2 * np.pi
    y = A.rope(x, np.cos(th), np.sin(th), 64, inverse=inverse)
    z = _complex_rotate(x, th, 64, sign=-1.0 if inverse else 1.0)
    np.testing.assert_allclose(y, z, rtol=0, atol=1e-13)


def test_inverse_undoes_and_lengths_are_kept():
    r = np.random.default_rng(3)
    x = r.standard_normal((4, 256))
    th = r.random(32) * 2 * np.pi
    c, s = np.cos(th), np.sin(th)
    y = A.rope(x, c, s, 64)
    np.testing.assert_allclose(A.rope(y, c, s, 64, inverse=True), x, rtol=0, atol=1e-13)
    # every pair keeps its length
    p0 = x[:, 192::2] ** 2 + x[:, 193::2] ** 2
    p1 = y[:, 192::2] ** 2 + y[:, 193::2] ** 2
    np.testing.assert_allclose(p1, p0, rtol=1e-13)


def test_relative_position_property():
    # angles linear in the position (theta_i(m) = m f_i): <R(m) q, R(n) k> = <R(m - n) q, k>
    r = np.random.default_rng(4)
    f = 10000.0 ** (-np.arange(32) / 32.0)
    q, k = r.standard_normal(128), r.standard_normal(128)
    rot = lambda x, m: A.rope(x, np.cos(m * f), np.sin(m * f), 64)
    for m, n in [(5, 3), (100, 7), (1000, 999), (17, 40)]:
        assert abs(rot(q, m) @ rot(k, n) - rot(q, m - n) @ k) < 1e-9


def _small_workload():
    wl = W.make_dense("fused_small", 3, 2, 4, 128, [300, 77])
    ts, tw = C.tensor_scales(wl)
    Kp, Vp = C.fill_pages(wl, ts, ts)
    return wl, Kp, Vp, ts, ts, tw, tw


def test_fused_with_identity_table_is_the_plain_decode():
    wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v = _small_workload()
    table = np.concatenate([np.ones((400, 32)), np.zeros((400, 32))], 1).astype(np.float32)
    for b in range(wl.B):
        O, L = C.expected_decode(wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v, b)
        Of, Lf, codes = C.expected_decode_fused(wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v, b, table, 64, W.OUT_SCALE)
        assert np.array_equal(Of, O) and np.array_equal(Lf, L)
        assert np.array_equal(codes, F.fp8_quantize(O, W.OUT_SCALE))


def test_fused_equals_keys_turned_the_other_way():
    # <q', k> = <R^-1 q', R^-1 k>: the rotated query q' (float32 rotation rounded to
    # bf16) turned back by the exact inverse, attending over inversely turned keys
    # (complex formulation), then the output turned back
    wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v = _small_workload()
    table = W.rope_table(wl.seed, 400, 64)
    for b in range(wl.B):
        pos = int(wl.rope_pos()[b])
        th = np.arctan2(table[pos, 32:].astype(np.float64), table[pos, :32].astype(np.float64))
        rad = np.hypot(table[pos, 32:].astype(np.float64), table[pos, :32].astype(np.float64))
        L = int(wl.seq_len[b])
        K = C.dequant_seq(wl, Kp, ts_k, b, L)
        V = C.dequant_seq(wl, Vp, ts_v, b, L)
        kw, vw = C.window_codes(wl, tw_k, tw_v, b)
        Kw, Vw = F.fp8_dequantize(kw, tw_k), F.fp8_dequantize(vw, tw_v)
        Kall = np.concatenate([K, Kw], 0)
        Vall = np.concatenate([V, Vw], 0)
        q = F.bf16_to_f64(wl.q_bits_seq(b))
        qp = A.rope_query_bf16(q, table[pos, :32], table[pos, 32:], 64)
        qs = _complex_rotate(qp, th, 64, sign=-1.0)
        Kinv = _complex_rotate(Kall, th, 64, sign=-1.0)
        z = (qs @ Kinv.T) / np.sqrt(128)
        m = z.max(1, keepdims=True)
        p = np.exp(z - m)
        O = (p @ Vall) / p.sum(1, keepdims=True)
        lse = (m + np.log(p.sum(1, keepdims=True)))[:, 0]
        O = _complex_rotate(O, th, 64, sign=-1.0)
        O[:, 64::2] *= rad
        O[:, 65::2] *= rad
        Of, Lf, codes = C.expected_decode_fused(wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v, b, table, 64, W.OUT_SCALE)
        np.testing.assert_allclose(Of, O, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(Lf, lse, rtol=1e-12)


def test_fused_codes_are_the_fp8_encoding_of_the_output():
    wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v = _small_workload()
    table = W.rope_table(wl.seed, 400, 64)
    Of, _, codes = C.expected_decode_fused(wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v, 0, table, 64, W.OUT_SCALE)
    assert codes.dtype == np.uint8 and codes.shape == Of.shape
    # decoded codes within half an E4M3 step of the scaled output (no saturation here)
    x = Of / W.OUT_SCALE
    assert np.abs(x).max() < 448
    dec = F.fp8_dequantize(codes, W.OUT_SCALE) / W.OUT_SCALE
    step = np.where(np.abs(x) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6))) - 3))
    assert np.all(np.abs(dec - x) <= step / 2 + 1e-12)


def test_fused_sparse_selection_matches_dense_on_all_positions():
    wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v = _small_workload()
    table = W.rope_table(wl.seed, 400, 64)
    b = 1
    sel = np.arange(int(wl.seq_len[b]))
    a = C.expected_decode_fused(wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v, b, table, 64, W.OUT_SCALE)
    s = C.expected_decode_fused(wl, Kp, Vp, ts_k, ts_v, tw_k, tw_v, b, table, 64, W.OUT_SCALE, sel=sel)
    assert all(np.array_equal(x, y) for x, y in zip(s, a))


def _f32_round(fr):
    """Nearest float32 (ties to even) of an exact rational, by comparing neighbours."""
    from fractions import Fraction
    c = np.float32(float(fr))
    best = None
    for v in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        dv = abs(Fraction(float(v)) - fr)
        if best is None or dv < best[0] or (dv == best[0] and (int(np.float32(v).view(np.uint32)) & 1) == 0):
            best = (dv, v)
    return np.float32(best[1])


def _bf16_round(v32):
    """Nearest bf16 value of a float32 (ties to even), by comparing the two bf16 neighbours exactly."""
    from fractions import Fraction
    u = int(np.array([v32], np.float32).view(np.uint32)[0])
    lo = u & 0xFFFF0000
    cands = [lo, lo + 0x10000]
    fv = Fraction(float(v32))
    best = None
    for cb in cands:
        val = Fraction(float(np.array([cb & 0xFFFFFFFF], np.uint32).view(np.float32)[0]))
        dv = abs(val - fv)
        if best is None or dv < best[0] or (dv == best[0] and ((cb >> 16) & 1) == 0):
            best = (dv, float(val))
    return best[1]


def test_rope_query_bf16_by_exact_rationals():
    # second formulation: products and difference / sum as exact rationals, each
    # rounded to float32 by neighbour comparison, then to bf16 the same way
    from fractions import Fraction
    r = np.random.default_rng(9)
    d, rd = 32, 16
    q = F.bf16_to_f64(W.to_bf16_bits(r.standard_normal((3, d)).astype(np.float32)))
    th = r.random(rd // 2) * 2 * np.pi
    cos, sin = np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)
    got = A.rope_query_bf16(q, cos, sin, rd)
    for h in range(3):
        for c in range(d):
            if c < d - rd:
                assert got[h, c] == q[h, c]
                continue
            i = (c - (d - rd)) // 2
            x0, x1 = Fraction(float(q[h, c - (c - (d - rd)) % 2])), Fraction(float(q[h, c - (c - (d - rd)) % 2 + 1]))
            cc, ss = Fraction(float(cos[i])), Fraction(float(sin[i]))
            if (c - (d - rd)) % 2 == 0:
                y = _f32_round(Fraction(float(_f32_round(x0 * cc))) - Fraction(float(_f32_round(x1 * ss))))
            else:
                y = _f32_round(Fraction(float(_f32_round(x0 * ss))) + Fraction(float(_f32_round(x1 * cc))))
            assert got[h, c] == _bf16_round(y), (h, c)


def test_rope_query_bf16_is_the_rotation_to_bf16_precision():
    r = np.random.default_rng(10)
    q = F.bf16_to_f64(W.to_bf16_bits(r.standard_normal((8, 128)).astype(np.float32)))
    th = r.random(32) * 2 * np.pi
    cos, sin = np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)
    exact = A.rope(q, cos.astype(np.float64), sin.astype(np.float64), 64)
    got = A.rope_query_bf16(q, cos, sin, 64)
    # within half a bf16 ulp (2^-9 relative) plus the float32 rotation's own rounding
    assert (np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-30).all()
    assert np.array_equal(got[:, :64], q[:, :64])
