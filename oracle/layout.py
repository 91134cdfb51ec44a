"""Byte layout of one 64-token page of the NVFP4 cache (oracle; test infrastructure).

The pages fix only that the global KV is stored in FP4 and paged ([blog]
"SWA bounded replay": compressed, shared across layers, FP4); the byte layout is
this library's definition, chosen so that a 64-token page is a few contiguous
runs of bytes.  Written out here address by address:

K-layout (the K cache), d channels: a token's d/2 code bytes are cut into
  column blocks of R = min(128, d/2) bytes, stored [d/(2R) blocks][64 tokens][R
  bytes]; inside a block the 16-byte chunk c of token t is stored at chunk
  position c XOR w(t), w(t) = t mod 8 when R = 128 and (t div 2) mod 4 when
  R = 64 (the K-major operand layouts with the 128- and 64-byte swizzle of a
  block-scaled FP4 tensor-core contraction, so that a page is read as is):
  data  channel pair (2j, 2j+1) of token t sits in byte
        (q div (R/16))*64*R + t*R + 16*((q mod (R/16)) XOR w(t)) + (j mod 16),
        q = j div 16, channel 2j in the low nibble, 2j+1 in the high nibble.
  scale [d/128 groups][64 tokens][8 bytes]: the scale of block j (channels
        16j..16j+15) of token t sits in byte ((j div 8)*64 + t)*8 + (j mod 8).
Index-key layout (the 128-wide index keys): data [64 tokens][64 bytes], channel
  pair j of token t in byte t*64 + 16*((j div 16) XOR (t AND 3)) + (j mod 16);
  scales as the K-layout.
V-layout (V), d channels: 32-bit words grouped by 128-channel chunk,
  data  [d/128 chunks][8 octets][128 channels][4 bytes]: channel ch of token t
        is nibble (t mod 8) of the little-endian 32-bit word
        ((ch div 128)*8 + (t div 8))*128 + (ch mod 128), i.e. byte
        4*(that word) + (t mod 8) div 2, low nibble for even t (one 128-channel
        chunk of a page is one contiguous run of 4 KB).
  scale [d/16 blocks][64 tokens]: block j of token t sits in byte j*64 + t.
Each pool is an array [num_pages][bytes per page] of uint8.
"""
from __future__ import annotations

import numpy as np

PAGE = 64


def k_data_bytes(d: int) -> int:
    return PAGE * d // 2


def k_scale_bytes(d: int) -> int:
    return PAGE * d // 16


v_data_bytes = k_data_bytes
v_scale_bytes = k_scale_bytes


def _k_data_addr(t: int, j: int, d: int) -> int:
    R = min(128, d // 2)
    w = t % 8 if R == 128 else (t // 2) % 4
    q = j // 16
    return (q // (R // 16)) * PAGE * R + t * R + 16 * ((q % (R // 16)) ^ w) + (j % 16)


def _i_data_addr(t: int, j: int) -> int:
    return t * 64 + 16 * ((j // 16) ^ (t & 3)) + (j % 16)


def _k_scale_addr(t: int, j: int) -> int:
    return ((j // 8) * PAGE + t) * 8 + (j % 8)


def _v_data_addr(t: int, ch: int, d: int) -> tuple:
    return 4 * (((ch // 128) * 8 + t // 8) * 128 + ch % 128) + (t % 8) // 2, (t % 2)


def _v_scale_addr(t: int, j: int) -> int:
    return j * PAGE + t


def _data_addr(t: int, j: int, d: int, index_keys: bool) -> int:
    return _i_data_addr(t, j) if index_keys else _k_data_addr(t, j, d)


def store_k_token(data_pool, scale_pool, page, t, codes, scales, index_keys=False):
    """Write one token's NVFP4 codes [d] (0..15) and scale bytes [d/16] into page
    ``page``, slot ``t`` (K-layout, or the index-key layout when ``index_keys``)."""
    d = len(codes)
    for j in range(d // 2):
        data_pool[page, _data_addr(t, j, d, index_keys)] = (int(codes[2 * j]) & 0xF) | ((int(codes[2 * j + 1]) & 0xF) << 4)
    for j in range(d // 16):
        scale_pool[page, _k_scale_addr(t, j)] = scales[j]


def load_k_token(data_pool, scale_pool, page, t, d, index_keys=False):
    codes = np.empty(d, np.uint8)
    for j in range(d // 2):
        b = int(data_pool[page, _data_addr(t, j, d, index_keys)])
        codes[2 * j] = b & 0xF
        codes[2 * j + 1] = b >> 4
    scales = np.array([scale_pool[page, _k_scale_addr(t, j)] for j in range(d // 16)], np.uint8)
    return codes, scales


def store_v_token(data_pool, scale_pool, page, t, codes, scales):
    d = len(codes)
    for ch in range(d):
        a, hi = _v_data_addr(t, ch, d)
        old = int(data_pool[page, a])
        c = int(codes[ch]) & 0xF
        data_pool[page, a] = (old & 0x0F) | (c << 4) if hi else (old & 0xF0) | c
    for j in range(d // 16):
        scale_pool[page, _v_scale_addr(t, j)] = scales[j]


def load_v_token(data_pool, scale_pool, page, t, d):
    codes = np.empty(d, np.uint8)
    for ch in range(d):
        a, hi = _v_data_addr(t, ch, d)
        b = int(data_pool[page, a])
        codes[ch] = (b >> 4) if hi else (b & 0xF)
    scales = np.array([scale_pool[page, _v_scale_addr(t, j)] for j in range(d // 16)], np.uint8)
    return codes, scales


# ---- vectorized forms of the same formulas (used on whole pages) -------------

def k_data_index(d: int) -> np.ndarray:
    """[64][d/2] byte address of channel pair j of token t (K-layout formula above)."""
    t = np.arange(PAGE)[:, None]
    j = np.arange(d // 2)[None, :]
    R = min(128, d // 2)
    w = t % 8 if R == 128 else (t // 2) % 4
    q = j // 16
    return (q // (R // 16)) * PAGE * R + t * R + 16 * ((q % (R // 16)) ^ w) + (j % 16)


def i_data_index() -> np.ndarray:
    """[64][64] byte address of channel pair j of token t of a 128-wide index key."""
    t = np.arange(PAGE)[:, None]
    j = np.arange(64)[None, :]
    return t * 64 + 16 * ((j // 16) ^ (t & 3)) + (j % 16)


def k_scale_index(d: int) -> np.ndarray:
    t = np.arange(PAGE)[:, None]
    j = np.arange(d // 16)[None, :]
    return ((j // 8) * PAGE + t) * 8 + (j % 8)


def v_data_index(d: int) -> tuple:
    """([64][d] byte address, [64][d] high-nibble flag) of channel ch of token t."""
    t = np.arange(PAGE)[:, None]
    ch = np.arange(d)[None, :]
    return 4 * (((ch // 128) * 8 + t // 8) * 128 + ch % 128) + (t % 8) // 2, np.broadcast_to(t % 2 == 1, (PAGE, d))


def v_scale_index(d: int) -> np.ndarray:
    t = np.arange(PAGE)[:, None]
    j = np.arange(d // 16)[None, :]
    return j * PAGE + t


def store_k_page(data_pool, scale_pool, page, slots, codes, scales, index_keys=False):
    """Write tokens at ``slots`` of page ``page``: codes [n][d], scales [n][d/16]
    (K-layout, or the index-key layout when ``index_keys``)."""
    d = codes.shape[1]
    slots = np.asarray(slots)
    packed = (codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)
    idx = i_data_index() if index_keys else k_data_index(d)
    data_pool[page, idx[slots]] = packed.astype(np.uint8)
    scale_pool[page, k_scale_index(d)[slots]] = scales


def load_k_page(data_pool, scale_pool, page, d, index_keys=False):
    """codes [64][d], scales [64][d/16] of a whole page."""
    b = data_pool[page][i_data_index() if index_keys else k_data_index(d)]
    codes = np.empty((PAGE, d), np.uint8)
    codes[:, 0::2] = b & 0xF
    codes[:, 1::2] = b >> 4
    return codes, scale_pool[page][k_scale_index(d)]


def store_v_page(data_pool, scale_pool, page, slots, codes, scales):
    d = codes.shape[1]
    slots = np.asarray(slots)
    addr, hi = v_data_index(d)
    a = addr[slots]
    h = hi[slots]
    c = (codes & 0xF).astype(np.uint8)
    # the two tokens of one byte (slots 2i, 2i+1) may arrive in one call:
    # write even slots, then odd slots, so no byte is read-modify-written twice at once
    ev = (slots % 2 == 0)
    for sel in (ev, ~ev):
        if sel.any():
            aa = a[sel]
            oo = data_pool[page, aa]
            cc = c[sel]
            hh = h[sel]
            data_pool[page, aa] = np.where(hh, (oo & 0x0F) | (cc << 4), (oo & 0xF0) | cc).astype(np.uint8)
    scale_pool[page, v_scale_index(d)[slots]] = scales


def load_v_page(data_pool, scale_pool, page, d):
    addr, hi = v_data_index(d)
    b = data_pool[page][addr]
    codes = np.where(hi, b >> 4, b & 0xF).astype(np.uint8)
    return codes, scale_pool[page][v_scale_index(d)]
