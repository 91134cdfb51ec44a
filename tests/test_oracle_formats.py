"""Pins of the oracle's E2M1 / E4M3 tables and NVFP4 / FP8 encoders.

Each check is independent of the oracle's own code: literal value lists typed
from the OCP definitions, hand-worked blocks under tests/golden, an
independent library (ml_dtypes, when installed), closed-form error bounds and
idempotence.
"""
import math

import numpy as np
import pytest

from conftest import golden_lines
from oracle import formats as F

# OCP MX v1.0, FP4 E2M1 element values for codes 0..15 (sign bit = bit 3)
E2M1_OCP = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
            -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_table_matches_ocp_list():
    for c in range(16):
        assert F.E2M1[c] == E2M1_OCP[c]
        assert math.copysign(1.0, F.E2M1[c]) == math.copysign(1.0, E2M1_OCP[c])


def test_e4m3_table_landmarks():
    # OCP OFP8 E4M3: a few values every implementation must agree on
    landmarks = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
                 0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0,
                 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0, 0x77: 240.0, 0x30: 0.5}
    for c, v in landmarks.items():
        assert F.E4M3[c] == v, hex(c)
    assert math.isnan(F.E4M3[0x7F]) and math.isnan(F.E4M3[0xFF])
    assert np.isfinite(F.E4M3[np.r_[0:0x7F, 0x80:0xFF]]).all()
    # monotone in code on the positive half, symmetric in sign
    pos = F.E4M3[:0x7F]
    assert (np.diff(pos) > 0).all()
    assert (F.E4M3[0x80:0xFF] == -pos).all()


def test_tables_match_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    e4 = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    fin = np.isfinite(e4)
    assert (fin == np.isfinite(F.E4M3)).all()
    assert (e4[fin] == F.E4M3[fin]).all()
    e2 = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    assert (e2 == F.E2M1).all()


def test_e2m1_tie_table():
    # magnitude -> code under ties-to-even (worked from the grid)
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             0.26: 1, 0.74: 1, 0.76: 2, 4.9: 6, 5.1: 7, 6.0: 7, 7.0: 7, 1e9: 7,
             0.0: 0, 0.24: 0}
    for v, c in cases.items():
        assert int(F.e2m1_encode(np.float32(v))) == c, v
        assert int(F.e2m1_encode(np.float32(-v))) == c | 8, -v


def test_e4m3_rounding_golden():
    for line in golden_lines("e4m3_rounding_cases.txt"):
        x, code = line.split()
        assert int(F.e4m3_encode(np.float32(float(x)))) == int(code, 16), line


def test_encoders_match_ml_dtypes_in_range():
    ml = pytest.importorskip("ml_dtypes")
    g = np.random.default_rng(1)
    x = np.concatenate([g.standard_normal(20000).astype(np.float32) * 50,
                        g.standard_normal(2000).astype(np.float32) * 1e-3])
    x = x[np.abs(x) <= 448]
    ref = x.astype(ml.float8_e4m3fn).view(np.uint8)
    assert (F.e4m3_encode(x) == ref).all()
    v = (g.standard_normal(20000) * 2).astype(np.float32)
    v = v[np.abs(v) <= 6]
    ref4 = v.astype(ml.float4_e2m1fn).astype(np.float64)
    assert (F.E2M1[F.e2m1_encode(v)] == ref4).all()


def test_nvfp4_worked_blocks():
    for line in golden_lines("nvfp4_worked_blocks.txt"):
        ts, xs, sc, cs = [p.strip() for p in line.split(";")]
        x = np.array([float(v) for v in xs.split()], np.float32)
        c, s = F.nvfp4_quantize(x, np.float32(float(ts)))
        assert int(s[0]) == int(sc, 16), line
        assert [int(v) for v in c] == [int(v, 16) for v in cs.split()], line


def test_nvfp4_error_bound_and_zero_blocks():
    g = np.random.default_rng(2)
    x = (g.standard_normal((4000, 64)) * g.choice([0.01, 1, 8, 40], (4000, 1))).astype(np.float32)
    x[7] = 0.0
    ts = np.float32(48.0 / 2688.0)
    c, s = F.nvfp4_quantize(x, ts)
    xh = F.nvfp4_dequantize(c, s, ts)
    assert (c[7] == 0).all() and (s[7] == 0).all()
    blk = x.reshape(4000, 4, 16).astype(np.float64)
    den = (F.E4M3[s] * np.float64(ts))[..., None]
    v = np.abs(blk) / np.where(den > 0, den, 1)
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    bound = np.where(v < 6, 0.5 * step * den, np.abs(blk) - 6 * den) + 1e-6 * np.abs(blk) + 1e-30
    err = np.abs(blk - xh.reshape(blk.shape))
    assert (err <= bound).all()
    # the block scale makes the largest element land near the top of the grid
    # (E4M3 keeps 3 mantissa bits: relative rounding <= 1/16 when the scale is normal)
    amax = np.abs(blk).max(-1)
    nz = (F.E4M3[s] >= 2.0 ** -6) & (amax <= 6 * 448 * np.float64(ts))   # normal, unsaturated scale
    assert (np.abs(amax[nz] / (F.E4M3[s][nz] * np.float64(ts)) - 6) <= 6 / (1 - 1 / 16) - 6 + 1e-9).all()


def test_nvfp4_idempotent_on_grid_values():
    # dequantized values re-quantize to the same bytes (same tensor scale)
    g = np.random.default_rng(3)
    x = (g.standard_normal((500, 32)) * 3).astype(np.float32)
    ts = np.float32(0.01)
    c, s = F.nvfp4_quantize(x, ts)
    xh = F.nvfp4_dequantize(c, s, ts).astype(np.float32)
    c2, s2 = F.nvfp4_quantize(xh, ts)
    # -0 codes of elements that dequantize to 0 may lose their sign: compare magnitudes there
    same = (c2 == c) | ((c & 7) == 0) & ((c2 & 7) == 0)
    assert same.all() and (s2 == s).all()


def test_fp8_quantize_roundtrip():
    g = np.random.default_rng(4)
    x = (g.standard_normal(10000) * 4).astype(np.float32)
    tw = np.float32(np.abs(x).max() / np.float32(448))
    c = F.fp8_quantize(x, tw)
    xh = F.fp8_dequantize(c, tw)
    rel = np.abs(xh - x) / np.maximum(np.abs(x), 2.0 ** -6 * float(tw))
    assert rel.max() <= 2.0 ** -4 + 1e-6      # half an ulp of a 3-bit mantissa


def test_rejects_nonfinite():
    with pytest.raises(ValueError):
        F.e4m3_encode(np.float32(np.inf))
    with pytest.raises(ValueError):
        F.nvfp4_quantize(np.zeros(16, np.float32), np.float32(0.0))


# ---------------------------------------------------------------- bf16 queries
def _bf16_by_definition(b: int) -> float:
    """bf16 bit pattern -> value from the format's fields: sign bit 15, exponent
    bits 14..7 (bias 127), mantissa bits 6..0 (7 bits, implicit leading 1 for
    normal numbers); exponent 0 = subnormal (2^-126 * m/128), 255 = inf / NaN."""
    s = -1.0 if b & 0x8000 else 1.0
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    if e == 0xFF:
        return s * math.inf if m == 0 else math.nan
    if e == 0:
        return s * math.ldexp(m, -126 - 7)
    return s * math.ldexp(128 + m, e - 127 - 7)


def test_bf16_to_f64_hand_worked_patterns():
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3FC0: 1.5, 0xBF00: -0.5, 0x4049: 3.140625,
             0x0080: 2.0 ** -126,                       # smallest normal
             0x0001: 2.0 ** -133,                       # smallest subnormal
             0x7F7F: (2.0 - 2.0 ** -7) * 2.0 ** 127,    # largest finite
             0x7F80: math.inf, 0xFF80: -math.inf, 0x0000: 0.0}
    got = F.bf16_to_f64(np.array(list(cases), np.uint16))
    for (b, v), g in zip(cases.items(), got):
        assert g == v, hex(b)
    neg0 = F.bf16_to_f64(np.array([0x8000], np.uint16))[0]
    assert neg0 == 0.0 and math.copysign(1.0, neg0) == -1.0
    assert math.isnan(F.bf16_to_f64(np.array([0x7FC0], np.uint16))[0])


def test_bf16_to_f64_every_pattern_by_field_decomposition():
    got = F.bf16_to_f64(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    ref = np.array([_bf16_by_definition(b) for b in range(65536)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def test_bf16_to_f64_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = b.view(ml.bfloat16).astype(np.float64)
    got = F.bf16_to_f64(b)
    fin = np.isfinite(ref)
    assert (np.isfinite(got) == fin).all()
    assert (got[fin] == ref[fin]).all()


# ---------------------------------------------------------------- FP8 tensor scale
def _f32_nearest(fr) -> np.float32:
    """The float32 nearest to the rational fr (ties to the even significand),
    found by comparing exact rationals against the neighbouring float32 values."""
    from fractions import Fraction
    c = np.float32(float(fr))
    best = None
    for v in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        d = abs(Fraction(float(v)) - fr)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(v).view(np.uint32)) & 1) == 0):
            best = (d, v)
    return np.float32(best[1])


def test_tensor_scale_fp8_worked_and_rounded():
    from fractions import Fraction
    assert F.tensor_scale_fp8(np.array([448.0, -3.0], np.float32)) == np.float32(1.0)
    assert F.tensor_scale_fp8(np.array([-896.0, 5.0], np.float32)) == np.float32(2.0)
    # amax is taken over magnitudes, then divided by 448 with one float32 rounding
    for xs in ([-48.0, 3.0, 0.5], [100.0, -7.25], [1e-3, -2.5e-3], [3.0e4, 1.0]):
        x = np.array(xs, np.float32)
        amax = max(abs(Fraction(float(v))) for v in x)
        assert F.tensor_scale_fp8(x) == _f32_nearest(amax / 448), xs
    # every value of the tensor then encodes without saturation
    g = np.random.default_rng(5)
    x = (g.standard_normal(4096) * 7).astype(np.float32)
    tw = F.tensor_scale_fp8(x)
    assert np.abs(F.fp8_dequantize(F.fp8_quantize(x, tw), tw)).max() <= 448 * float(tw)


# ---------------------------------------------------------------- float32 -> bf16
def test_f32_to_bf16_hand_worked_ties():
    def f(bits):
        return np.array([bits], np.uint32).view(np.float32)
    def b(bits16):
        return float(np.array([bits16 << 16], np.uint32).view(np.float32)[0])
    cases = [(0x3F800000, 0x3F80), (0x3F808000, 0x3F80),   # exact half between 1.0 and the next: even (down)
             (0x3F818000, 0x3F82),                          # half between 0x3F81 and 0x3F82: even (up)
             (0x3F808001, 0x3F81), (0x3F807FFF, 0x3F80),    # just above / below the half
             (0xBF818000, 0xBF82), (0x00000000, 0x0000), (0x80000000, 0x8000),
             (0x7F7F7FFF, 0x7F7F)]                          # below the half under the largest finite
    for src, want in cases:
        got = F.f32_to_bf16(f(src))[0]
        assert got == b(want) and np.signbit(got) == bool(want & 0x8000), hex(src)


def test_f32_to_bf16_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    g = np.random.default_rng(6)
    x = np.concatenate([g.standard_normal(50000).astype(np.float32) * np.float32(3),
                        (g.standard_normal(1000) * 1e-30).astype(np.float32)])
    assert (F.f32_to_bf16(x) == x.astype(ml.bfloat16).astype(np.float64)).all()
