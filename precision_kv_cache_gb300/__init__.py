"""Python binding of the GB300 NVFP4-KV decode-attention library (libpkv.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/pkv.h``.  The functions keep the C
names (``pkv_append_kv``, ``pkv_decode_attn`` ...) and take torch CUDA tensors,
whose device pointers are passed through unchanged; torch is used for device
memory and streams only.  If the shared library has not been built
(``python -m precision_kv_cache_gb300.build`` or ``__graft_entry__.build()``)
importing the kernels raises - there is no CPU fallback.

A decode step (d = 512, 64 query heads; every tensor on the context's GPU):

    import precision_kv_cache_gb300 as P
    ctx = P.Context(512, 64)
    cache = P.KVCache.empty(num_pages, 512, ts_k, ts_v)     # paged NVFP4 K/V pools
    win = P.Window(k_fp8, v_fp8, tw_k, tw_v)                # E4M3 window, [B][128][512]
    ctx.pkv_append_kv(k_new, v_new, seq_idx, pos, cache, page_table)
    ctx.pkv_decode_attn(q_bf16, cache, page_table, seq_len, win, 512 ** -0.5, out, lse)
    assert ctx.pkv_get_error() == P.OK                      # synchronizes the stream

A sparse step selects positions with ``pkv_score_topk`` (all positions) or
``pkv_score_topk_cand`` (a candidate list) and passes them as ``sel_idx``;
``pkv_decode_attn_fused`` adds query RoPE, inverse RoPE on the output and an
E4M3 output; ``pkv_replay_attn`` re-runs the last 128 positions after a
prefix hit.  Workspaces are sized by ``Context.workspace`` (or passed in).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

PAGE = 64
WINDOW = 128
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_BAD_PAGE, ERR_TIMEOUT, ERR_WORKSPACE = range(7)
OP_DECODE, OP_SCORE_TOPK, OP_REPLAY, OP_DECODE_SPARSE, OP_SCORE_CAND = 1, 2, 3, 4, 5


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_status_str(status)} ({status})")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("n_heads", ctypes.c_int), ("page_size", ctypes.c_int),
                ("window", ctypes.c_int), ("d_index", ctypes.c_int), ("n_index_heads", ctypes.c_int)]


class _KVCache(ctypes.Structure):
    _fields_ = [("k_data", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_data", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("num_pages", ctypes.c_int), ("ts_k", ctypes.c_float),
                ("ts_v", ctypes.c_float)]


class _IdxCache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("ts", ctypes.c_float)]


class _Window(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("tw_k", ctypes.c_float),
                ("tw_v", ctypes.c_float), ("win_len", ctypes.c_void_p)]


class _RopeFp8(ctypes.Structure):
    _fields_ = [("pos", ctypes.c_void_p), ("cos_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int),
                ("rope_dim", ctypes.c_int), ("out_scale", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpkv.so (raises if it is missing: the kernels are the only path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run precision_kv_cache_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "pkv_init": (i, [ctypes.POINTER(_Config), i, ctypes.POINTER(vp)]),
            "pkv_destroy": (None, [vp]),
            "pkv_workspace_bytes": (sz, [vp, i, i, i]),
            "pkv_append_kv": (i, [vp, vp, vp, vp, vp, i, ctypes.POINTER(_KVCache), vp, i, vp]),
            "pkv_append_index": (i, [vp, vp, vp, vp, i, ctypes.POINTER(_IdxCache), vp, i, vp]),
            "pkv_quantize_fp8": (i, [vp, sz, f, vp, vp]),
            "pkv_score_topk": (i, [vp, vp, f, vp, ctypes.POINTER(_IdxCache), vp, i, vp, i, i, vp, vp, vp, sz, vp]),
            "pkv_score_topk_cand": (i, [vp, vp, f, vp, ctypes.POINTER(_IdxCache), vp, i, vp, i, i, i, vp, vp, vp, sz,
                                        vp]),
            "pkv_decode_attn": (i, [vp, vp, ctypes.POINTER(_KVCache), vp, i, vp, i, vp, i,
                                    ctypes.POINTER(_Window), f, vp, vp, vp, sz, vp]),
            "pkv_decode_attn_fused": (i, [vp, vp, ctypes.POINTER(_KVCache), vp, i, vp, i, vp, i,
                                          ctypes.POINTER(_Window), f, ctypes.POINTER(_RopeFp8), vp, vp, vp, vp, sz,
                                          vp]),
            "pkv_replay_attn": (i, [vp, vp, ctypes.POINTER(_KVCache), vp, i, vp, i, ctypes.POINTER(_Window),
                                    f, vp, vp, vp, sz, vp]),
            "pkv_merge": (i, [vp, vp, vp, vp, vp, vp, i, i, vp]),
            "pkv_get_error": (i, [vp, vp]),
            "pkv_status_str": (ctypes.c_char_p, [i]),
            "pkv_set_profile_events": (i, [vp, vp, vp]),
            "pkv_decode_attn_noalloc": (i, [vp, vp, ctypes.POINTER(_KVCache), vp, i, vp, i, vp, i,
                                            ctypes.POINTER(_Window), f, vp, vp, vp]),
            "pkv_set_test_hooks": (i, [vp, ctypes.c_longlong, i]),
            "pkv_launch_count": (ctypes.c_longlong, [vp]),
            "pkv_attn_path": (i, [vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _status_str(s: int) -> str:
    try:
        return lib().pkv_status_str(s).decode()
    except Exception:  # pragma: no cover - library missing
        return "status"


def _check(s: int, what: str):
    if s != OK:
        raise PkvError(s, what)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclasses.dataclass
class KVCache:
    """Device pools of one paged NVFP4 K/V cache (uint8 [num_pages][bytes per page])."""
    k_data: torch.Tensor
    k_scale: torch.Tensor
    v_data: torch.Tensor
    v_scale: torch.Tensor
    ts_k: float
    ts_v: float

    @staticmethod
    def empty(num_pages: int, d: int, ts_k: float, ts_v: float, device="cuda") -> "KVCache":
        z = lambda n: torch.zeros((num_pages, n), dtype=torch.uint8, device=device)
        return KVCache(z(PAGE * d // 2), z(PAGE * d // 16), z(PAGE * d // 2), z(PAGE * d // 16), ts_k, ts_v)

    @property
    def num_pages(self) -> int:
        return self.k_data.shape[0]

    def _c(self) -> _KVCache:
        return _KVCache(self.k_data.data_ptr(), self.k_scale.data_ptr(), self.v_data.data_ptr(),
                        self.v_scale.data_ptr(), self.num_pages, self.ts_k, self.ts_v)


@dataclasses.dataclass
class IdxCache:
    data: torch.Tensor
    scale: torch.Tensor
    ts: float

    @staticmethod
    def empty(num_pages: int, ts: float, d_index: int = 128, device="cuda") -> "IdxCache":
        return IdxCache(torch.zeros((num_pages, PAGE * d_index // 2), dtype=torch.uint8, device=device),
                        torch.zeros((num_pages, PAGE * d_index // 16), dtype=torch.uint8, device=device), ts)

    def _c(self) -> _IdxCache:
        return _IdxCache(self.data.data_ptr(), self.scale.data_ptr(), self.data.shape[0], self.ts)


@dataclasses.dataclass
class Window:
    """FP8 window K/V codes uint8 [B][128][d] with their tensor scales."""
    k: torch.Tensor
    v: torch.Tensor
    tw_k: float
    tw_v: float
    win_len: Optional[torch.Tensor] = None

    def _c(self) -> _Window:
        return _Window(self.k.data_ptr(), self.v.data_ptr(), self.tw_k, self.tw_v,
                       None if self.win_len is None else self.win_len.data_ptr())


class Context:
    """A pkv_ctx: fixed shapes (d, heads) on one device."""

    def __init__(self, d: int, n_heads: int, n_index_heads: int = 64, device: int = 0):
        cfg = _Config(d, n_heads, PAGE, WINDOW, 128, n_index_heads)
        h = ctypes.c_void_p()
        _check(lib().pkv_init(ctypes.byref(cfg), device, ctypes.byref(h)), "pkv_init")
        self.h = h
        self.d, self.n_heads, self.n_index_heads, self.device = d, n_heads, n_index_heads, device

    def close(self):
        if getattr(self, "h", None):
            lib().pkv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- calls
    def pkv_workspace_bytes(self, op: int, batch: int, max_len: int) -> int:
        return int(lib().pkv_workspace_bytes(self.h, op, batch, max_len))

    def pkv_append_kv(self, k_new, v_new, seq_idx, pos, cache: KVCache, page_table, stream=None):
        n = k_new.shape[0]
        c = cache._c()
        _check(lib().pkv_append_kv(self.h, _p(k_new), _p(v_new), _p(seq_idx), _p(pos), n, ctypes.byref(c),
                                   _p(page_table), page_table.shape[1], _stream(stream)), "pkv_append_kv")

    def pkv_append_index(self, k_idx, seq_idx, pos, icache: IdxCache, page_table, stream=None):
        c = icache._c()
        _check(lib().pkv_append_index(self.h, _p(k_idx), _p(seq_idx), _p(pos), k_idx.shape[0], ctypes.byref(c),
                                      _p(page_table), page_table.shape[1], _stream(stream)), "pkv_append_index")

    def pkv_score_topk(self, q_idx, tq, w, icache: IdxCache, page_table, seq_len, k, out_idx,
                       out_score=None, ws=None, stream=None):
        B = seq_len.shape[0]
        if ws is None:
            ws = self.workspace(OP_SCORE_TOPK, B, page_table.shape[1] * PAGE)
        c = icache._c()
        _check(lib().pkv_score_topk(self.h, _p(q_idx), tq, _p(w), ctypes.byref(c), _p(page_table),
                                    page_table.shape[1], _p(seq_len), B, k, _p(out_idx), _p(out_score),
                                    _p(ws), ws.numel(), _stream(stream)), "pkv_score_topk")

    def pkv_score_topk_cand(self, q_idx, tq, w, icache: IdxCache, page_table, cand, k, out_idx, out_score=None,
                            ws=None, stream=None):
        B, n = cand.shape
        if ws is None:
            ws = self.workspace(OP_SCORE_CAND, B, n)
        c = icache._c()
        _check(lib().pkv_score_topk_cand(self.h, _p(q_idx), tq, _p(w), ctypes.byref(c), _p(page_table),
                                         page_table.shape[1], _p(cand), n, B, k, _p(out_idx), _p(out_score),
                                         _p(ws), ws.numel(), _stream(stream)), "pkv_score_topk_cand")

    def pkv_decode_attn(self, q, cache: KVCache, page_table, seq_len, win: Window, scale, out, out_lse=None,
                        ws=None, sel_idx=None, stream=None):
        B = seq_len.shape[0]
        k = sel_idx.shape[1] if sel_idx is not None else 0
        if ws is None:
            ws = (self.workspace(OP_DECODE_SPARSE, B, k) if sel_idx is not None
                  else self.workspace(OP_DECODE, B, page_table.shape[1] * PAGE))
        c = cache._c()
        w = win._c()
        _check(lib().pkv_decode_attn(self.h, _p(q), ctypes.byref(c), _p(page_table), page_table.shape[1],
                                     _p(seq_len), B, _p(sel_idx), k, ctypes.byref(w), scale, _p(out),
                                     _p(out_lse), _p(ws), ws.numel(), _stream(stream)), "pkv_decode_attn")

    def pkv_decode_attn_fused(self, q, cache: KVCache, page_table, seq_len, win: Window, scale, pos, cos_sin,
                              rope_dim, out_scale, out_fp8, out=None, out_lse=None, ws=None, sel_idx=None,
                              stream=None):
        """Decode with query RoPE, inverse RoPE on O and E4M3 output (cos_sin float32 [max_pos][rope_dim])."""
        B = seq_len.shape[0]
        k = sel_idx.shape[1] if sel_idx is not None else 0
        if ws is None:
            ws = (self.workspace(OP_DECODE_SPARSE, B, k) if sel_idx is not None
                  else self.workspace(OP_DECODE, B, page_table.shape[1] * PAGE))
        c = cache._c()
        w = win._c()
        fz = _RopeFp8(pos.data_ptr(), cos_sin.data_ptr(), cos_sin.shape[0], rope_dim, out_scale)
        _check(lib().pkv_decode_attn_fused(self.h, _p(q), ctypes.byref(c), _p(page_table), page_table.shape[1],
                                           _p(seq_len), B, _p(sel_idx), k, ctypes.byref(w), scale, ctypes.byref(fz),
                                           _p(out_fp8), _p(out), _p(out_lse), _p(ws), ws.numel(), _stream(stream)),
               "pkv_decode_attn_fused")

    def pkv_decode_attn_noalloc(self, q, cache: KVCache, page_table, seq_len, win: Window, scale, out,
                                out_lse=None, sel_idx=None, stream=None):
        """pkv_decode_attn with the library's built-in scratch array instead of a caller buffer."""
        B = seq_len.shape[0]
        k = sel_idx.shape[1] if sel_idx is not None else 0
        c = cache._c()
        w = win._c()
        _check(lib().pkv_decode_attn_noalloc(self.h, _p(q), ctypes.byref(c), _p(page_table), page_table.shape[1],
                                             _p(seq_len), B, _p(sel_idx), k, ctypes.byref(w), scale, _p(out),
                                             _p(out_lse), _stream(stream)), "pkv_decode_attn_noalloc")

    def pkv_replay_attn(self, q, cache: KVCache, page_table, prefix_len, chunk_win: Window, scale, out,
                        out_lse=None, ws=None, stream=None):
        B = prefix_len.shape[0]
        if ws is None:
            ws = self.workspace(OP_REPLAY, B, page_table.shape[1] * PAGE)
        c = cache._c()
        w = chunk_win._c()
        _check(lib().pkv_replay_attn(self.h, _p(q), ctypes.byref(c), _p(page_table), page_table.shape[1],
                                     _p(prefix_len), B, ctypes.byref(w), scale, _p(out), _p(out_lse), _p(ws),
                                     ws.numel(), _stream(stream)), "pkv_replay_attn")

    def pkv_get_error(self, stream=None) -> int:
        return int(lib().pkv_get_error(self.h, _stream(stream)))

    def pkv_set_profile_events(self, start: "torch.cuda.Event", stop: "torch.cuda.Event"):
        """Record start/stop around the main kernel of the next attention call."""
        for ev in (start, stop):
            if not ev.cuda_event:       # torch creates the CUDA event on first record
                ev.record()
        _check(lib().pkv_set_profile_events(self.h, ctypes.c_void_p(start.cuda_event),
                                            ctypes.c_void_p(stop.cuda_event)), "pkv_set_profile_events")

    def pkv_set_test_hooks(self, wait_limit_cycles: int = 1 << 31, skip_copy: int = -1):
        """Testing aid: bounded-wait limit (SM cycles) and a K-tile copy CTA 0 leaves out (-1 = none)."""
        _check(lib().pkv_set_test_hooks(self.h, wait_limit_cycles, skip_copy), "pkv_set_test_hooks")

    def pkv_launch_count(self) -> int:
        return int(lib().pkv_launch_count(self.h))

    def pkv_attn_path(self) -> int:
        """2 once an attention call has launched the tensor-core kernels, 0 before."""
        return int(lib().pkv_attn_path(self.h))

    def workspace(self, op: int, batch: int, max_len: int) -> torch.Tensor:
        n = self.pkv_workspace_bytes(op, batch, max_len)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=f"cuda:{self.device}")


def pkv_quantize_fp8(x: torch.Tensor, tw: float, out: torch.Tensor, stream=None):
    _check(lib().pkv_quantize_fp8(_p(x), x.numel(), tw, _p(out), _stream(stream)), "pkv_quantize_fp8")


def pkv_merge(o_a, lse_a, o_b, lse_b, o, lse, stream=None):
    rows = lse_a.numel()
    _check(lib().pkv_merge(_p(o_a), _p(lse_a), _p(o_b), _p(lse_b), _p(o), _p(lse), rows,
                           o_a.numel() // max(rows, 1), _stream(stream)), "pkv_merge")
