"""E2M1 / E4M3 tables and the NVFP4 / FP8 encoders (oracle; test infrastructure).

Format sources: OCP Microscaling Formats (MX) v1.0, "FP4 (E2M1)" element
format; OCP 8-bit Floating Point (OFP8) "E4M3" (the FN variant: no infinities,
S.1111.111 is NaN, largest finite 448).  NVFP4 = E2M1 elements, one E4M3 scale
per 16 consecutive elements, one FP32 scale per tensor.  The pages ([blog]
"MegaAttention avec KV compressé NVFP4"; [news] "Les particularités du modèle
lui-même") fix the cache to FP4 with FP8 for the window and nothing finer; the
rounding contract below is this library's (ties to the even code, saturating).

All decisions that turn a float into a code are taken in float32, the
precision the kernels use, so both sides take the same integer decision.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * (m / 2.0)                  # subnormal: 2^(1-1) * m/2
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


def e4m3_value(code: int) -> float:
    """Value of an 8-bit E4M3 (FN) code: sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6      # subnormal
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3 = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)

# non-negative finite magnitudes in code order (codes are monotone in value)
_E2M1_POS = E2M1[:8]                    # codes 0..7
_E4M3_POS = E4M3[:0x7F]                 # codes 0x00..0x7E (0x7F is NaN)
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _nearest_even_code(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to each a >= 0 (a <= grid[-1]); exact
    midpoints go to the even index.  The midpoints of these short grids are
    exact in float64, and so are the comparisons against float32 inputs."""
    mid = (grid[:-1] + grid[1:]) / 2.0
    i = np.searchsorted(mid, a, side="left")        # first midpoint >= a
    # a == mid[i] exactly: a tie between codes i and i+1 -> pick the even one
    idx = np.clip(i, 0, len(mid) - 1)
    tie = (i < len(mid)) & (a == mid[idx])
    i = np.where(tie & (i % 2 == 1), i + 1, i)
    return i.astype(np.int64)


def e4m3_encode(x) -> np.ndarray:
    """float32 -> E4M3 code: nearest finite value, ties to the even code,
    magnitudes above 448 saturate to 448 (0x7E), sign bit = sign of x.
    NaN / inf inputs are an error."""
    x = np.asarray(x, dtype=F32)
    if not np.isfinite(x).all():
        raise ValueError("E4M3 encode of a non-finite value")
    a = np.abs(x).astype(np.float64)
    a = np.minimum(a, E4M3_MAX)
    code = _nearest_even_code(a, _E4M3_POS)
    sign = np.signbit(x).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """float32 -> E2M1 code: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the
    even code, |v| >= 6 -> 6, sign bit = sign of v (small negatives give -0)."""
    v = np.asarray(v, dtype=F32)
    if not np.isfinite(v).all():
        raise ValueError("E2M1 encode of a non-finite value")
    a = np.minimum(np.abs(v).astype(np.float64), E2M1_MAX)
    code = _nearest_even_code(a, _E2M1_POS)
    sign = np.signbit(v).astype(np.int64) << 3
    return (code | sign).astype(np.uint8)


def nvfp4_quantize(x, ts) -> tuple:
    """NVFP4 encode of float32 rows ``x[..., n*16]`` with the FP32 tensor scale ``ts``.

    Per block of 16 consecutive elements (the contract of this library):
      1. amax = max |x_i|
      2. s = fp32(amax / fp32(6 * ts))            (two float32 RN operations)
      3. S = E4M3 code of s (nearest, ties even, saturating)
      4. S == 0: all element codes are 0
      5. den = fp32(E4M3[S] * ts); v_i = fp32(x_i / den)   (true division)
      6. c_i = E2M1 code of v_i (nearest, ties even, |v| >= 6 -> 6, sign of x_i)
    Returns (codes uint8 [..., n*16] in 0..15, scales uint8 [..., n]).
    """
    x = np.asarray(x, dtype=F32)
    ts = F32(ts)
    if not (np.isfinite(ts) and ts > 0):
        raise ValueError("tensor scale must be finite and > 0")
    shp = x.shape
    assert shp[-1] % 16 == 0
    blk = x.reshape(shp[:-1] + (shp[-1] // 16, 16))
    amax = np.abs(blk).max(axis=-1)                                # float32, exact
    t = F32(F32(6.0) * ts)
    s = (amax / t).astype(F32)                                     # float32 RN division
    S = e4m3_encode(s)
    sval = E4M3[S].astype(F32)                                     # exact in float32
    den = (sval * ts).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (blk / den[..., None]).astype(F32)
    v = np.where((S == 0)[..., None], F32(0.0), v)
    c = e2m1_encode(v)
    c = np.where((S == 0)[..., None], np.uint8(0), c)
    return c.reshape(shp).astype(np.uint8), S.astype(np.uint8)


def nvfp4_dequantize(codes, scales, ts) -> np.ndarray:
    """x_hat = E2M1[c] * E4M3[S] * ts, exactly, in float64."""
    codes = np.asarray(codes)
    scales = np.asarray(scales)
    shp = codes.shape
    c = codes.reshape(shp[:-1] + (shp[-1] // 16, 16))
    return (E2M1[c] * E4M3[scales][..., None] * np.float64(F32(ts))).reshape(shp)


def fp8_quantize(x, tw) -> np.ndarray:
    """FP8 (E4M3) encode with one FP32 tensor scale: code = E4M3(fp32(x / tw))."""
    x = np.asarray(x, dtype=F32)
    tw = F32(tw)
    if not (np.isfinite(tw) and tw > 0):
        raise ValueError("tensor scale must be finite and > 0")
    return e4m3_encode((x / tw).astype(F32))


def fp8_dequantize(codes, tw) -> np.ndarray:
    return E4M3[np.asarray(codes)] * np.float64(F32(tw))


def tensor_scale_fp8(x) -> np.float32:
    """FP32 tensor scale of an FP8 tensor: fp32(amax / 448)."""
    return F32(F32(np.abs(np.asarray(x, F32)).max()) / F32(448.0))


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact): a bf16 value is the
    float32 whose upper 16 bits are the pattern and whose lower 16 bits are 0."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> nearest bf16 value (ties to the even significand), returned as
    float64: keep the upper 16 bits of the float32 pattern after adding half of
    the dropped range (0x7FFF) plus the lowest kept bit (finite inputs)."""
    u = np.ascontiguousarray(np.asarray(x, dtype=F32)).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)
