"""Float64 attention, replay, merge, index scoring and top-k (oracle; test infrastructure).

Each function is the plain definition, with no blocking, fusion or reordering:

* ``segment`` / ``decode``: softmax attention of one query head over a set of
  entries, z = scale * q.k, O = sum_i exp(z_i - m) v_i / sum_i exp(z_i - m),
  LSE = m + ln sum_i exp(z_i - m).  All query heads read the same K/V (MQA over
  one shared latent: [blog] "Performances agentiques", DP attention paragraph).
  In decode the entries are the global tokens [0, L) followed by the FP8
  sliding-window entries ([news] "Les particularités du modèle lui-même": a
  compressed FP4 global KV plus an uncompressed FP8 window of the last 128
  positions); the two sets are disjoint.
* ``replay``: bounded replay after a prefix hit of length H ([blog] "SWA
  bounded replay" and "Côté encodeur : reconstruire la fenêtre lors d'un hit de
  cache"): the 128 tokens at positions s + r, r = 0..127, s = H - 128, are re-run;
  query r attends the global tokens [0, s) and, causally, the window entries of
  positions s..s+r (window clipped at s).
* ``merge``: the log-sum-exp combination of two partial results of disjoint
  entry sets.
* ``index_score``: the sparse indexer score score_t = sum_h w_h ReLU(q_h . k_t)
  ([blog] "Kernels", "Logits MQA creux": late indexer layers pick their top-k
  positions from scores).
* ``topk``: the k highest scores, ties to the lower index, returned ascending.
* ``rope``: the rotary position embedding that the fused decode of [blog]
  "MegaAttention avec KV compressé NVFP4" applies to the queries before QK and,
  inverted, to the output after the attention.  The pages name the step but
  not its layout; the reading taken: the last ``rope_dim`` channels of a head
  rotate, as interleaved pairs (2i, 2i+1), each pair by its own angle, given
  by a caller table of cosines and sines (the rotary cache a serving engine
  keeps), the other channels pass through.
"""
from __future__ import annotations

import numpy as np


def segment(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """q [H][d], K [n][d], V [n][dv] (float64) -> (O [H][dv], LSE [H]).
    An empty entry set gives O = 0 and LSE = -inf."""
    q = np.asarray(q, np.float64)
    H = q.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, V.shape[1])), np.full(H, -np.inf)
    z = scale * (q @ np.asarray(K, np.float64).T)          # [H][n]
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    O = (p @ np.asarray(V, np.float64)) / l
    return O, (m + np.log(l))[:, 0]


def decode(q, K, V, Kw, Vw, scale):
    """One decode step of one sequence: global entries K/V [L] plus window Kw/Vw [W]."""
    return segment(q, np.concatenate([K, Kw], 0), np.concatenate([V, Vw], 0), scale)


def replay(q, K, V, Kw, Vw, scale, rows=None):
    """q [R][H][d]; global K/V [s]; window Kw/Vw [R] of positions s..s+R-1.
    Query r attends K/V[0:s] and Kw/Vw[0:r+1].  ``rows`` restricts to a subset of r."""
    R = q.shape[0]
    rows = range(R) if rows is None else rows
    O = {}
    L = {}
    for r in rows:
        O[r], L[r] = segment(q[r], np.concatenate([K, Kw[:r + 1]], 0),
                             np.concatenate([V, Vw[:r + 1]], 0), scale)
    return O, L


def rope(x, cos, sin, rope_dim: int, inverse: bool = False):
    """x [..., d] (float64) with pair i = channels (d - rope_dim + 2i, d - rope_dim + 2i + 1)
    turned by the angle whose cosine and sine are cos[i], sin[i] (by minus that
    angle when ``inverse``):  y0 = x0 cos - x1 sin,  y1 = x0 sin + x1 cos.
    cos / sin broadcast against x[..., rope_dim // 2]."""
    y = np.array(x, dtype=np.float64, copy=True)
    if rope_dim == 0:
        return y
    d = y.shape[-1]
    c = np.asarray(cos, np.float64)
    s = np.asarray(sin, np.float64)
    if inverse:
        s = -s
    x0 = y[..., d - rope_dim::2].copy()
    x1 = y[..., d - rope_dim + 1::2].copy()
    y[..., d - rope_dim::2] = x0 * c - x1 * s
    y[..., d - rope_dim + 1::2] = x0 * s + x1 * c
    return y


def rope_query_bf16(q, cos, sin, rope_dim: int):
    """The rotated query of a fused decode as the contraction receives it: the
    rotation of ``rope`` computed in float32, each product and the difference /
    sum rounded separately (y0 = fp32(fp32(x0 c) - fp32(x1 s)), y1 =
    fp32(fp32(x0 s) + fp32(x1 c)), c and s the table's float32 values), then
    rounded to bf16 (nearest, ties to even): the rotated query is a bf16 tensor
    like the query itself.  q [..., d] holds float32-exact values; returns
    float64."""
    F32 = np.float32
    y = np.array(q, dtype=F32, copy=True)
    if rope_dim:
        d = y.shape[-1]
        c = np.asarray(cos, F32)
        s = np.asarray(sin, F32)
        x0 = y[..., d - rope_dim::2].copy()
        x1 = y[..., d - rope_dim + 1::2].copy()
        y[..., d - rope_dim::2] = (x0 * c).astype(F32) - (x1 * s).astype(F32)
        y[..., d - rope_dim + 1::2] = (x0 * s).astype(F32) + (x1 * c).astype(F32)
    from . import formats
    return formats.f32_to_bf16(y)


def merge(Oa, La, Ob, Lb):
    """LSE merge: lse = ln(e^La + e^Lb), O = e^(La-lse) Oa + e^(Lb-lse) Ob.
    A part with LSE = -inf has weight 0; both empty gives O = 0, LSE = -inf."""
    La = np.asarray(La, np.float64)
    Lb = np.asarray(Lb, np.float64)
    m = np.maximum(La, Lb)
    both_empty = np.isneginf(m)
    ms = np.where(both_empty, 0.0, m)
    wa = np.exp(La - ms)
    wb = np.exp(Lb - ms)
    s = wa + wb
    lse = np.where(both_empty, -np.inf, ms + np.log(np.where(both_empty, 1.0, s)))
    sd = np.where(both_empty, 1.0, s)
    O = (wa[..., None] * Oa + wb[..., None] * Ob) / sd[..., None]
    O = np.where(both_empty[..., None], 0.0, O)
    return O, lse


def index_score(qhat, w, khat):
    """qhat [Hi][di], w [Hi], khat [L][di] (float64) -> score [L] = sum_h w_h max(0, qhat_h . k_t)."""
    dots = np.asarray(khat, np.float64) @ np.asarray(qhat, np.float64).T   # [L][Hi]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def topk(scores, k):
    """Indices of the k highest scores (ties: lower index first), returned in
    ascending index order; fewer than k scores -> all indices then -1 padding."""
    s = np.asarray(scores, np.float64)
    L = s.shape[0]
    order = np.lexsort((np.arange(L), -s))     # primary: -score, secondary: index
    sel = np.sort(order[:min(k, L)])
    out = np.full(k, -1, np.int64)
    out[:len(sel)] = sel
    return out


def topk_cand(cand_scores, cand, k):
    """Top-k restricted to a candidate list ("Logits MQA creux", vLLM blog
    "Kernels": only a fixed candidate set is scored): ``cand`` holds ascending
    positions, ``cand_scores[i]`` the score of position cand[i].  Returns the
    selected positions in ascending order (ties: lower position first, which is
    the lower candidate index because the list is ascending), -1 padded."""
    cand = np.asarray(cand, np.int64)
    sel = topk(cand_scores, k)
    return np.where(sel >= 0, cand[np.maximum(sel, 0)], -1)


def topk_matches(gpu_idx, scores, k, rel=1e-5):
    """Set check of a top-k answer against float64 scores: exactly the oracle's
    set, except members whose score lies within ``rel`` * |S_k| of the k-th
    score S_k (near-ties at the boundary may go either way).  ``gpu_idx`` must
    also be ascending, unique, and padded with -1 exactly when L < k."""
    s = np.asarray(scores, np.float64)
    L = len(s)
    g = np.asarray(gpu_idx, np.int64)
    ref = topk(s, k)
    n = min(k, L)
    if (g[n:] != -1).any() or (g[:n] < 0).any() or (g[:n] >= L).any():
        return False, "bad padding or range"
    gv = g[:n]
    if n > 1 and not (np.diff(gv) > 0).all():
        return False, "not ascending/unique"
    if n == 0:
        return True, "empty"
    Sk = np.sort(s)[::-1][n - 1]
    tol = rel * abs(Sk)
    a = set(gv.tolist())
    b = set(ref[:n].tolist())
    for i in a ^ b:
        if abs(s[i] - Sk) > tol:
            return False, f"index {i} score {s[i]} differs from boundary {Sk}"
    return True, f"{len(a ^ b)} boundary swaps"
