"""Shared helpers of the GPU parity tests: oracle-built inputs uploaded to the device.

Inputs flow one way only: seeded rows (workloads) -> oracle quantization ->
bytes copied to the GPU.  Nothing the CUDA path writes is fed back to the oracle.
"""
import math

import numpy as np

import workloads as W
from oracle import attention as A
from oracle import cache as C
from oracle import formats as F

# attention tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle|, element-wise
ATOL = 2e-3
RTOL = 1e-2


def assert_close(g, r, what, atol=ATOL, rtol=RTOL):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    both_inf = np.isneginf(g) & np.isneginf(r)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(g - r))
    lim = atol + rtol * np.where(both_inf, 0.0, np.abs(r))
    bad = ~(err <= lim)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - lim, -np.inf)), g.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {g.size} outside tolerance; worst at {i}: "
                             f"gpu={g[i]} oracle={r[i]} (max abs err {np.nanmax(err):.3e})")


def torch_dev():
    import torch
    return torch.device("cuda:0")


def upload_cache(Kp, Vp, ts_k, ts_v):
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return P.KVCache(t(Kp.data), t(Kp.scale), t(Vp.data), t(Vp.scale), float(ts_k), float(ts_v))


def window_tensors(wl, tw_k, tw_v, win_len=None):
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch_dev()
    kw = np.stack([C.window_codes(wl, tw_k, tw_v, b)[0] for b in range(wl.B)])
    vw = np.stack([C.window_codes(wl, tw_k, tw_v, b)[1] for b in range(wl.B)])
    wlen = None if win_len is None else torch.tensor(np.asarray(win_len, np.int32), device=dev)
    return P.Window(torch.from_numpy(kw).to(dev), torch.from_numpy(vw).to(dev), float(tw_k), float(tw_v), wlen), kw, vw


def q_tensor(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(torch_dev()).view(torch.bfloat16)


def i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).to(torch_dev())


def assert_fp8_codes(gc, Or, out_scale, what, atol=ATOL, rtol=RTOL):
    """E4M3 codes the GPU encoded from its own FP32 output, against the oracle's
    float64 output Or.  The GPU's value lies within the attention tolerance of
    Or and E4M3 rounding is monotone, so each code must decode between the
    oracle's encodings of Or - tol and Or + tol: it equals the oracle's code
    wherever no rounding midpoint lies within the tolerance."""
    Or = np.asarray(Or, np.float64)
    tol = atol + rtol * np.abs(Or)
    lo = F.fp8_dequantize(F.fp8_quantize(Or - tol, out_scale), out_scale)
    hi = F.fp8_dequantize(F.fp8_quantize(Or + tol, out_scale), out_scale)
    g = F.fp8_dequantize(np.asarray(gc, np.uint8), out_scale)
    bad = ~((g >= lo) & (g <= hi))
    if bad.any():
        i = np.unravel_index(np.argmax(bad), g.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {g.size} FP8 codes outside [{lo[i]}, {hi[i]}] at {i}: "
                             f"gpu={g[i]} oracle value={Or[i]}")
    # where the interval holds one value, the code is the oracle's exactly
    one = lo == hi
    rc = F.fp8_quantize(Or, out_scale)
    assert np.array_equal(g[one], F.fp8_dequantize(rc, out_scale)[one]), what


def assert_scores_close(g, qhat, w, khat, what):
    """Element-wise bound on index scores sum_h w_h ReLU(qhat_h . k_t): each head's
    128-term dot product is accumulated in FP32 from exact products (a tensor-core
    contraction on f16 operands that hold the FP8 / NVFP4 values exactly), so its
    error is at most 128 * 2^-23 * sum_i |q_hi k_ti| even with truncating adds; the
    epilogue adds at most 66 roundings of 2^-24 (tensor scales, weight, ReLU'd sum of
    64 non-negative terms).  Bound per position t: 2^-23 * (128 + 66) * R_t, with
    R_t = sum_h |w_h| sum_i |qhat_hi khat_ti|."""
    qhat = np.asarray(qhat, np.float64)
    khat = np.asarray(khat, np.float64)
    w = np.asarray(w, np.float64)
    ref = np.maximum(khat @ qhat.T, 0.0) @ w
    R = (np.abs(khat) @ np.abs(qhat).T) @ np.abs(w)
    lim = 2.0 ** -23 * (128 + 66) * R
    err = np.abs(np.asarray(g, np.float64) - ref)
    bad = err > lim
    if bad.any():
        i = int(np.argmax(np.where(bad, err / np.maximum(lim, 1e-300), 0)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {len(ref)} scores outside the bound; worst at {i}: "
                             f"gpu={g[i]} oracle={ref[i]} bound={lim[i]:.3e}")
    return float((err / np.maximum(lim, 1e-300)).max())
