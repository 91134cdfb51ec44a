"""Seeded synthetic inputs for the decode-attention path (shared input side only).

This module is the one piece that both the float64 oracle (``oracle/``, test
infrastructure) and the CUDA path's tests and benchmark draw from.  It holds
none of the method's arithmetic: no quantization, no scoring, no attention.
It only draws random numbers, builds page tables and lengths, and names which
physical page holds which token.

Workload shapes follow the five configurations of the decode-attention bench
(see ``CONFIGS``): values are N(0, 1) float32 with 2 % of the channels scaled by
8, queries are rounded to bf16, the index-head weights are U(0, 1).  Every page
of every tensor is drawn from its own ``numpy.random.SeedSequence`` substream
keyed by (seed, tensor, page key), so any page can be regenerated alone - that
is what lets the oracle check sampled outputs of a full-size run without
holding the whole cache.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Tuple

import numpy as np

PAGE = 64          # tokens per page of the global cache
WINDOW = 128       # sliding-window (SWA) entries per sequence
D_INDEX = 128      # index-key / index-query width
H_INDEX = 64       # index heads

# tensor ids of the substreams
T_K, T_V, T_Q, T_KW, T_VW, T_IK, T_IQ, T_W, T_KNEW, T_VNEW, T_RQ, T_OUTL, T_CAND, T_ROPE = range(1, 15)

ROPE_DIM = 64      # channels of each head a fused decode rotates (the last ROPE_DIM of d)
OUT_SCALE = 1.0 / 64.0   # FP8 output scale of a fused decode: O/OUT_SCALE in E4M3's normal range
                         # for softmax averages of N(0,1) rows; |O| > 7 saturates at 448


def rng(seed: int, *key: int) -> np.random.Generator:
    """A counter-free PCG64 stream for one (seed, key...) tuple."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed)] + [int(k) for k in key])))


def outlier_channels(seed: int, tensor: int, d: int) -> np.ndarray:
    """round(2 % of d) channel ids, drawn without replacement, fixed over tokens."""
    n = int(round(0.02 * d))
    return np.sort(rng(seed, T_OUTL, tensor, d).choice(d, size=n, replace=False))


def normal_rows(seed: int, tensor: int, key: Tuple[int, ...], n: int, d: int,
                outliers: bool = True, outlier_tensor: Optional[int] = None) -> np.ndarray:
    """float32 [n][d] ~ N(0, 1); the outlier channels of ``outlier_tensor`` x8."""
    x = rng(seed, tensor, *key).standard_normal((n, d), dtype=np.float32)
    if outliers:
        ch = outlier_channels(seed, tensor if outlier_tensor is None else outlier_tensor, d)
        x[:, ch] *= np.float32(8.0)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@dataclasses.dataclass
class Workload:
    """One decode-attention workload: shapes, page tables and the page keys.

    ``page_table[b][j]`` is the physical page that holds tokens [64j, 64j+64) of
    sequence b.  ``page_key[p]`` is the substream key of physical page p;
    pages shared by a group of sequences have one key.  Tokens [fill_start[b],
    fill_end[b]) of sequence b are the ones a cache fill writes through b's page
    table (shared pages are written once, through the group's first sequence).
    """
    name: str
    seed: int
    B: int
    H: int
    d: int
    seq_len: np.ndarray            # int32 [B]: global tokens attended (after any append)
    win_len: np.ndarray            # int32 [B]: window entries (decode)
    page_table: np.ndarray         # int32 [B][max_pages]
    num_pages: int
    page_key: Dict[int, Tuple[int, ...]]
    fill_start: np.ndarray
    fill_end: np.ndarray
    append: bool = False           # one new token per sequence at position seq_len-1
    topk: int = 0                  # >0: sparse path (index scoring + top-k)
    replay: bool = False           # bounded replay: 128 queries at [H-128, H)
    prefix_len: Optional[np.ndarray] = None   # H per sequence (replay)
    n_cand: int = 0                # >0: candidate-list scoring of that many positions per sequence

    def rope_pos(self) -> np.ndarray:
        """int32 [B]: position of each sequence's query token (its newest, seq_len - 1)."""
        return np.maximum(self.seq_len.astype(np.int64) - 1, 0).astype(np.int32)

    def cand_lists(self, n: int) -> np.ndarray:
        """int32 [B][n]: min(n, L) distinct positions per sequence, ascending, -1 padded."""
        out = np.full((self.B, n), -1, np.int32)
        for b in range(self.B):
            L = int(self.seq_len[b])
            m = min(n, L)
            out[b, :m] = np.sort(rng(self.seed, T_CAND, b).choice(L, size=m, replace=False))
        return out

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    # ---- value rows -------------------------------------------------
    def page_rows(self, tensor: int, page: int, d: Optional[int] = None) -> np.ndarray:
        """float32 [64][d] fp32 values of physical page ``page`` for K/V/index keys."""
        d = self.d if d is None else d
        return normal_rows(self.seed, tensor, self.page_key[page], PAGE, d)

    def token_rows(self, tensor: int, b: int, t0: int, t1: int, d: Optional[int] = None) -> np.ndarray:
        """float32 [t1-t0][d] values of tokens [t0, t1) of sequence b (assembled from pages)."""
        d = self.d if d is None else d
        out = np.empty((max(t1 - t0, 0), d), np.float32)
        t = t0
        while t < t1:
            j, s = divmod(t, PAGE)
            n = min(PAGE - s, t1 - t)
            out[t - t0:t - t0 + n] = self.page_rows(tensor, int(self.page_table[b, j]), d)[s:s + n]
            t += n
        return out

    def new_rows(self, tensor: int) -> np.ndarray:
        """float32 [B][d]: the token appended to each sequence in the step."""
        return normal_rows(self.seed, tensor, (0,), self.B, self.d,
                           outlier_tensor=T_K if tensor == T_KNEW else T_V)

    def window_rows(self, tensor: int, b: int) -> np.ndarray:
        """float32 [128][d] window K (T_KW) or V (T_VW) values of sequence b."""
        return normal_rows(self.seed, tensor, (b,), WINDOW, self.d,
                           outlier_tensor=T_K if tensor == T_KW else T_V)

    def q_bits(self) -> np.ndarray:
        """bf16 bits [B][H][d] of the decode queries."""
        return to_bf16_bits(normal_rows(self.seed, T_Q, (0,), self.B * self.H, self.d,
                                        outliers=False)).reshape(self.B, self.H, self.d)

    def q_bits_seq(self, b: int) -> np.ndarray:
        return self.q_bits()[b]

    def replay_q_bits(self, b: int) -> np.ndarray:
        """bf16 bits [128][H][d] of the replayed queries of sequence b."""
        return to_bf16_bits(normal_rows(self.seed, T_RQ, (b,), WINDOW * self.H, self.d,
                                        outliers=False)).reshape(WINDOW, self.H, self.d)

    def index_q(self) -> np.ndarray:
        """float32 [B][64][128] index queries (to be FP8-quantized)."""
        return normal_rows(self.seed, T_IQ, (0,), self.B * H_INDEX, D_INDEX,
                           outliers=False).reshape(self.B, H_INDEX, D_INDEX)

    def index_w(self) -> np.ndarray:
        """float32 [B][64] index-head weights ~ U(0, 1)."""
        return rng(self.seed, T_W, 0).random((self.B, H_INDEX), dtype=np.float32)

    def index_rows(self, page: int) -> np.ndarray:
        """float32 [64][128] index keys of physical page ``page``."""
        return normal_rows(self.seed, T_IK, self.page_key[page], PAGE, D_INDEX)

    def fill_segments(self) -> List[Tuple[int, int, int]]:
        """(b, t0, t1) token ranges a cache fill writes, shared pages once."""
        return [(b, int(self.fill_start[b]), int(self.fill_end[b])) for b in range(self.B)
                if self.fill_end[b] > self.fill_start[b]]


def rope_table(seed: int, max_pos: int, rope_dim: int = ROPE_DIM) -> np.ndarray:
    """float32 [max_pos][rope_dim] rotary table in the layout a serving engine
    keeps: per position, the cosines of its rope_dim/2 pair angles, then their
    sines.  The angles are drawn uniformly on [0, 2 pi) (seeded), so the table
    exercises arbitrary rotations; the attention path takes any table."""
    th = rng(seed, T_ROPE, max_pos, rope_dim).random((max_pos, rope_dim // 2)) * (2.0 * np.pi)
    return np.concatenate([np.cos(th), np.sin(th)], axis=1).astype(np.float32)


def _pages_for(lengths: np.ndarray) -> np.ndarray:
    return (lengths + PAGE - 1) // PAGE


def make_dense(name: str, seed: int, B: int, H: int, d: int, lens, win=WINDOW,
               perm_seed_key: int = 0) -> Workload:
    """Private pages only; the page table is a random permutation of the pool."""
    lens = np.asarray(lens, np.int32).reshape(B)
    npg = _pages_for(lens)
    num_pages = int(npg.sum())
    perm = rng(seed, 100, perm_seed_key).permutation(num_pages).astype(np.int32)
    maxp = max(int(npg.max()), 1)
    pt = np.full((B, maxp), -1, np.int32)
    key: Dict[int, Tuple[int, ...]] = {}
    o = 0
    for b in range(B):
        for j in range(int(npg[b])):
            p = int(perm[o]); o += 1
            pt[b, j] = p
            key[p] = (1, b, j)
    winl = np.full(B, win, np.int32) if np.isscalar(win) else np.asarray(win, np.int32)
    return Workload(name, seed, B, H, d, lens, winl, pt, num_pages, key,
                    np.zeros(B, np.int32), lens.copy())


def make_shared_prefix(name: str, seed: int, B: int, H: int, d: int, lens, group: int,
                       shared_tokens: int, append: bool = True) -> Workload:
    """Groups of ``group`` sequences share the physical pages of their first
    ``shared_tokens`` tokens; the pool is shuffled."""
    lens = np.asarray(lens, np.int32).reshape(B)
    assert shared_tokens % PAGE == 0 and (lens >= shared_tokens).all()
    ngroups = (B + group - 1) // group
    nshared = shared_tokens // PAGE
    npg = _pages_for(lens)
    num_pages = ngroups * nshared + int((npg - nshared).sum())
    perm = rng(seed, 101, 0).permutation(num_pages).astype(np.int32)
    maxp = int(npg.max())
    pt = np.full((B, maxp), -1, np.int32)
    key: Dict[int, Tuple[int, ...]] = {}
    o = 0
    shared_ids = np.empty((ngroups, nshared), np.int32)
    for g in range(ngroups):
        for j in range(nshared):
            p = int(perm[o]); o += 1
            shared_ids[g, j] = p
            key[p] = (2, g, j)
    for b in range(B):
        pt[b, :nshared] = shared_ids[b // group]
        for j in range(nshared, int(npg[b])):
            p = int(perm[o]); o += 1
            pt[b, j] = p
            key[p] = (1, b, j)
    fs = np.where(np.arange(B) % group == 0, 0, shared_tokens).astype(np.int32)
    fe = (lens - 1 if append else lens).astype(np.int32)
    return Workload(name, seed, B, H, d, lens, np.full(B, WINDOW, np.int32), pt, num_pages,
                    key, fs, fe, append=append)


def make_replay(name: str, seed: int, B: int, H: int, d: int, prefix_lens) -> Workload:
    """Bounded replay: global pages hold [0, H-128); queries sit at [H-128, H)."""
    hl = np.asarray(prefix_lens, np.int32).reshape(B)
    assert (hl >= WINDOW).all()
    w = make_dense(name, seed, B, H, d, hl - WINDOW, win=WINDOW, perm_seed_key=7)
    w.replay = True
    w.prefix_len = hl
    return w


def uniform_lengths(seed: int, key: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Integer lengths uniform on [lo, hi] inclusive."""
    return rng(seed, 200, key).integers(lo, hi + 1, size=B).astype(np.int32)


# The five configurations of the decode-attention bench (full size).
def config(i: int, seed: int = 0) -> Workload:
    if i == 0:   # tiny dense decode
        return make_dense("c0_tiny_dense_decode", seed, 1, 8, 128, [1024])
    if i == 1:   # dense decode at 8K
        return make_dense("c1_dense_decode_8k", seed, 32, 64, 512, [8192] * 32)
    if i == 2:   # ragged paged decode, shared 4K prefixes, 1-token append
        lens = uniform_lengths(seed, 2, 64, 16384, 32768)
        return make_shared_prefix("c2_ragged_paged_decode", seed, 64, 64, 512, lens, 8, 4096)
    if i == 3:   # long-context sparse path
        w = make_dense("c3_sparse_512k", seed, 4, 64, 512, [524288] * 4)
        w.topk = 2048
        return w
    if i == 4:   # bounded replay after a prefix hit
        hl = uniform_lengths(seed, 4, 16, 32768, 131072)
        return make_replay("c4_bounded_replay", seed, 16, 64, 512, hl)
    raise ValueError(i)


# Profiling cases: smaller runs of the c2 and c4 kernels for multi-pass ncu
# captures (a few hundred MB on the device, launches of milliseconds at most).
def profile_case(name: str, seed: int = 0) -> Workload:
    if name == "p2":   # c2's shape at 16 sequences (two prefix groups of 8)
        lens = uniform_lengths(seed, 12, 16, 16384, 32768)
        return make_shared_prefix("p2_ragged_paged_decode_small", seed, 16, 64, 512, lens, 8, 4096)
    if name == "p4":   # c4's shape at 2 sequences
        hl = uniform_lengths(seed, 14, 2, 32768, 65536)
        return make_replay("p4_bounded_replay_small", seed, 2, 64, 512, hl)
    raise ValueError(name)


# Long-context decode sweep: the dense 64-head d=512 decode shape at one length
# L, with the batch sized so that the NVFP4 K/V read per step is at least 1 GiB.
LONG_CONTEXT = (32768, 65536, 131072, 262144, 524288)


def long_context(L: int, seed: int = 0) -> Workload:
    B = -(-(1 << 30) // (L * 576))
    return make_dense(f"sweep_decode_{L // 1024}k", seed, B, 64, 512, [L] * B, perm_seed_key=L)


CONFIGS = {
    0: "batch 1, 8 heads, d=128, 1024 global tokens + 128-entry FP8 window",
    1: "batch 32, 64 heads, d=512, 8192 global tokens each + window",
    2: "batch 64, 64 heads, d=512, lengths U[16K,32K], 8 groups share 4K-token prefixes, 1-token append",
    3: "batch 4, 524288 tokens, index scoring 64x128 FP8 q / NVFP4 keys, top-2048, 64-head attention",
    4: "batch 16, prefix H U[32K,128K], 128 replayed queries x 64 heads, d=512",
}
