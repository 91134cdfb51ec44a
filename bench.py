#!/usr/bin/env python
"""Benchmark of the NVFP4-KV decode-attention path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload c1|c2|c3|c4|c3c|c1f|c3f]

A step is one pass of the decode path over one batch held in HBM.  Default
workload (c2): 64 sequences of 16K-32K tokens (uniform), 64 query heads sharing
one NVFP4 KV (d=512), 8 groups of 8 sequences sharing the physical pages of
their first 4096 tokens, an FP8 window of 128 entries per sequence; the step
appends one NVFP4 token per sequence and then runs decode attention (split-K
over the global pages, window segment, LSE merge).  Other workloads: c1 (dense
8K decode, B=32), c3 (index scoring + top-2048 + sparse decode, B=4 at 512K),
c4 (bounded replay of 128 tokens, B=16, H in [32K,128K]); c3c (c3 scoring a
fixed 16K candidate set per sequence); c1f / c3f (c1 / c3 with the decode as
one fused call: query RoPE, attention, inverse RoPE on O, E4M3 output).

Metric: decode-attention KV GB/s = needed bytes / step time, where needed bytes
count the NVFP4 K/V bytes (codes + scales) of every distinct token the step
reads (shared pages once), the page-table entries, the FP8 window, Q, O/LSE
and the appended tokens.  One JSON line on rank 0.  Synthetic data (seeded
generators of ``workloads``).  A step whose bytes are under 4x the 129 MB L2
(c1, the sparse workloads) is preceded by an L2 flush (256 MB written, then
another 256 MB read, before the step's start event); the larger ones run
without one.

--impl reference times the float64 CPU oracle (the only reference that exists
for this path) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

WORKLOADS = {"c1": 1, "c2": 2, "c3": 3, "c4": 4, "c3c": 3, "c1f": 1, "c3f": 3}
CAND_C3C = 16384                   # c3c: the sparse workload scoring a fixed candidate set per sequence
FUSED = ("c1f", "c3f")             # the decode as one fused call: query RoPE, attention, inverse RoPE, FP8 O
SWEEP = {f"s{L // 1024}k": L for L in W.LONG_CONTEXT}     # long-context decode sweep (--sweep)
PROFILE = ("p2", "p4")              # smaller c2 / c4 runs for multi-pass ncu captures (not bench lines)
SCORE_SWEEP = {f"x{L // 1024}k": L for L in W.LONG_CONTEXT}   # index-scoring sweep (--score-sweep)
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 << 20
NOMINAL_HBM_GBS = 8000.0


# ----------------------------------------------------------------------------- helpers
def _gen_rows(args):
    """(worker) float32 K and V rows of tokens [t0, t1) of sequence b."""
    name, b, t0, t1 = args
    wl = _wl_cache(name)
    return b, t0, t1, wl.token_rows(W.T_K, b, t0, t1), wl.token_rows(W.T_V, b, t0, t1)


def _gen_index(args):
    name, pages = args
    wl = _wl_cache(name)
    return pages, np.stack([wl.index_rows(p) for p in pages])


_WL = {}


def _wl_cache(name):
    if name not in _WL:
        if name in SCORE_SWEEP:     # the sparse shape (4 sequences, top-2048) at length L
            L = SCORE_SWEEP[name]
            _WL[name] = W.make_dense(f"sweep_scoring_{L // 1024}k", 0, 4, 64, 512, [L] * 4, perm_seed_key=L + 1)
            _WL[name].topk = 2048
        else:
            if name in SWEEP:
                _WL[name] = W.long_context(SWEEP[name])
            elif name in PROFILE:
                _WL[name] = W.profile_case(name)
            else:
                _WL[name] = W.config(WORKLOADS[name])
        if name == "c3c":
            _WL[name].n_cand = CAND_C3C
        if name in FUSED:
            _WL[name].name += "_fused"
    return _WL[name]


def workload_desc(name):
    if name in SWEEP:
        wl = _wl_cache(name)
        return f"long-context decode sweep: batch {wl.B}, 64 heads, d=512, {SWEEP[name]} global tokens each + window"
    if name == "c3c":
        return W.CONFIGS[3] + f", scoring only a fixed {CAND_C3C}-position candidate set per sequence"
    if name == "p2":
        return "profiling case: c2's shape at batch 16 (two 8-sequence prefix groups), 1-token append"
    if name == "p4":
        return "profiling case: c4's shape at batch 2, prefix H U[32K,64K]"
    if name in FUSED:
        return (W.CONFIGS[WORKLOADS[name]] + f"; fused decode: query RoPE on the last {W.ROPE_DIM} channels, "
                "inverse RoPE on O, E4M3 output")
    return W.CONFIGS[WORKLOADS[name]]


def tensor_scales():
    """FP32 tensor scales fixed at cache creation: NVFP4 fp32(48/2688), FP8 fp32(48/448)
    (48 = 8 x 6 sigma bounds the synthetic N(0,1) values with x8 outlier channels)."""
    return float(np.float32(np.float32(48.0) / np.float32(2688.0))), float(np.float32(np.float32(48.0) / np.float32(448.0)))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.dev = device_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(self.dev)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1])); smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "sampled_s": round(self.t1 - self.t0 + 0.25, 3)}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(values, world, device):
    """The element-wise maximum over all ranks (the slowest rank times the job); identity at world = 1."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbs(step_bytes_per_rank, ms_step_max, world):
    """Whole-job throughput: every rank processes its own copy of the workload (weak
    scaling, no data-path collective); the job takes as long as its slowest rank."""
    return step_bytes_per_rank * world / (ms_step_max * 1e-3) / 1e9


def tensor_peak():
    """Dense bf16 (= f16) tensor peak: the measured sustained figure (a long kernel), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (bf16 dense, sustained)"
    except Exception:
        return 1700.0, "fallback (bf16 dense, sustained)"


def code_sha(path: str) -> str:
    """Hash of a C/CUDA source without its comments and blank lines (a capture stays
    valid across comment edits, not across code edits)."""
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    code = "\n".join(ln for ln in lines if ln.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel code."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d[kernel][workload]
        src = os.path.join(ROOT, "precision_kv_cache_gb300", "csrc", e["source"])
        return float(e["dram_bytes_per_launch"]) if code_sha(src) == e["code_sha"] else None
    except Exception:
        return None


# ----------------------------------------------------------------------------- accounting
def kv_token_bytes(d):
    return 2 * (d // 2 + d // 16)          # K and V: codes + E4M3 scales


def needed_bytes(wl, sel_counts=None, fused=False):
    """Algorithmic bytes of one decode-attention launch over ``wl`` (see module doc)."""
    d, H, B = wl.d, wl.H, wl.B
    if sel_counts is not None:
        tokens = int(np.sum(sel_counts))
        pt = tokens * 4
    elif wl.replay:
        tokens = 0
        used = {}
        for b in range(B):
            s = int(wl.prefix_len[b]) - 128
            for j in range((s + 63) // 64):
                used[int(wl.page_table[b, j])] = max(used.get(int(wl.page_table[b, j]), 0), min(64, s - 64 * j))
        tokens = sum(used.values())
        pt = sum((int(wl.prefix_len[b]) - 128 + 63) // 64 for b in range(B)) * 4
    else:
        used = {}
        for b in range(B):
            L = int(wl.seq_len[b])
            for j in range((L + 63) // 64):
                p = int(wl.page_table[b, j])
                used[p] = max(used.get(p, 0), min(64, L - 64 * j))
        tokens = sum(used.values())
        pt = sum((int(wl.seq_len[b]) + 63) // 64 for b in range(B)) * 4
    rows = B * (128 if wl.replay else 1)
    win = B * 128 * d * 2
    q = rows * H * d * 2
    o = rows * H * (d + 1) * 4
    if fused:     # E4M3 O + LSE, plus each row's position and cos/sin row
        o = rows * H * d + rows * H * 4 + rows * (4 + W.ROPE_DIM * 4)
    return tokens * kv_token_bytes(d) + pt + win + q + o, tokens


# ----------------------------------------------------------------------------- GPU arm
def fill_cache(ctx, P, torch, wl, name, ts_k, ts_v, pool):
    dev = torch.device(f"cuda:{ctx.device}")
    cache = P.KVCache.empty(wl.num_pages, wl.d, ts_k, ts_v, device=dev)
    pt = torch.from_numpy(wl.page_table).to(dev)
    jobs = []
    for (b, t0, t1) in wl.fill_segments():
        for s in range(t0, t1, 8192):
            jobs.append((name, b, s, min(t1, s + 8192)))
    it = pool.map(_gen_rows, jobs) if pool else map(_gen_rows, jobs)
    for (b, t0, t1, kr, vr) in it:
        n = t1 - t0
        ctx.pkv_append_kv(torch.from_numpy(kr).to(dev), torch.from_numpy(vr).to(dev),
                          torch.full((n,), b, dtype=torch.int32, device=dev),
                          torch.arange(t0, t1, dtype=torch.int32, device=dev), cache, pt)
    torch.cuda.synchronize()
    return cache, pt


def fill_index(ctx, P, torch, wl, name, ts, pool, pt):
    """NVFP4 index keys of every page through the product append (each page written via its owner)."""
    dev = torch.device(f"cuda:{ctx.device}")
    ic = P.IdxCache.empty(wl.num_pages, ts, device=dev)
    pages = list(range(wl.num_pages))
    chunks = [(name, pages[i:i + 512]) for i in range(0, len(pages), 512)]
    it = pool.map(_gen_index, chunks) if pool else map(_gen_index, chunks)
    owner = {int(wl.page_table[b, j]): (b, j) for b in range(wl.B) for j in range(wl.page_table.shape[1])
             if wl.page_table[b, j] >= 0}
    for (pg, rows) in it:
        bs = np.repeat([owner[p][0] for p in pg], 64).astype(np.int32)
        ps = np.concatenate([64 * owner[p][1] + np.arange(64) for p in pg]).astype(np.int32)
        ctx.pkv_append_index(torch.from_numpy(rows.reshape(-1, 128)).to(dev), torch.from_numpy(bs).to(dev),
                             torch.from_numpy(ps).to(dev), ic, pt)
    torch.cuda.synchronize()
    return ic


def score_kernel_bytes(wl, positions, pages):
    """Algorithmic bytes of one index-scoring launch: 72 B of NVFP4 key + 4 B of score per
    position, the page-table entries, the FP8 queries and the head weights."""
    return positions * (64 + 8 + 4) + pages * 4 + wl.B * 64 * 128 + wl.B * 64 * 4


def window_codes_gpu(P, torch, wl, tw, dev, rows_fn):
    x = torch.from_numpy(np.stack([rows_fn(b) for b in range(wl.B)])).to(dev)
    out = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    P.pkv_quantize_fp8(x, tw, out)
    return out


def run_gpu(args, rank, world, pool):
    import torch
    import precision_kv_cache_gb300 as P

    dev = torch.device(f"cuda:{int(os.environ.get('LOCAL_RANK', 0))}")
    torch.cuda.set_device(dev)
    name = args.workload
    wl = _wl_cache(name)
    ts, tw = tensor_scales()
    ctx = P.Context(wl.d, wl.H, device=dev.index)
    t_setup = time.time()
    cache, pt = fill_cache(ctx, P, torch, wl, name, ts, ts, pool)
    wk = window_codes_gpu(P, torch, wl, tw, dev, lambda b: wl.window_rows(W.T_KW, b))
    wv = window_codes_gpu(P, torch, wl, tw, dev, lambda b: wl.window_rows(W.T_VW, b))
    win = P.Window(wk, wv, tw, tw)
    scale = 1.0 / math.sqrt(wl.d)
    seq_len = torch.from_numpy(wl.seq_len).to(dev)
    B, H, d = wl.B, wl.H, wl.d
    extra = {}
    if wl.replay:
        q_host = np.stack([wl.replay_q_bits(b) for b in range(B)])
        out = torch.empty(B, 128, H, d, device=dev)
        lse = torch.empty(B, 128, H, device=dev)
        plen = torch.from_numpy(wl.prefix_len).to(dev)
        ws = ctx.workspace(P.OP_REPLAY, B, pt.shape[1] * 64)
    else:
        q_host = wl.q_bits()
        out = torch.empty(B, H, d, device=dev)
        lse = torch.empty(B, H, device=dev)
    q = torch.from_numpy(q_host.view(np.int16)).to(dev).view(torch.bfloat16)
    sel = None
    if wl.topk:
        ic = fill_index(ctx, P, torch, wl, name, ts, pool, pt)
        qf = wl.index_q()
        tq = float(np.float32(np.float32(np.abs(qf).max()) / np.float32(448.0)))
        qidx = torch.empty(qf.shape, dtype=torch.uint8, device=dev)
        P.pkv_quantize_fp8(torch.from_numpy(qf).to(dev), tq, qidx)
        wts = torch.from_numpy(wl.index_w()).to(dev)
        sel = torch.empty(B, wl.topk, dtype=torch.int32, device=dev)
        if wl.n_cand:
            cand = torch.from_numpy(wl.cand_lists(wl.n_cand)).to(dev)
            ws_s = ctx.workspace(P.OP_SCORE_CAND, B, wl.n_cand)
        else:
            ws_s = ctx.workspace(P.OP_SCORE_TOPK, B, pt.shape[1] * 64)
        ws = ctx.workspace(P.OP_DECODE_SPARSE, B, wl.topk)
    elif not wl.replay:
        ws = ctx.workspace(P.OP_DECODE, B, pt.shape[1] * 64)
    fused = name in FUSED
    if fused:
        rpos = torch.from_numpy(wl.rope_pos()).to(dev)
        table = torch.from_numpy(W.rope_table(wl.seed, int(wl.rope_pos().max()) + 1, W.ROPE_DIM)).to(dev)
        out8 = torch.empty(B, H, d, dtype=torch.uint8, device=dev)
    if wl.append:
        knew = torch.from_numpy(wl.new_rows(W.T_KNEW)).to(dev)
        vnew = torch.from_numpy(wl.new_rows(W.T_VNEW)).to(dev)
        bidx = torch.arange(B, dtype=torch.int32, device=dev)
        pos = (seq_len - 1).to(torch.int32)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup
    # L2 flush between timed steps when the step's bytes would largely fit the 129 MB L2
    ws_bytes = needed_bytes(wl, fused=fused)[0] if not wl.topk else 0
    flush_l2 = args.flush_l2 == "on" or (args.flush_l2 == "auto" and (wl.topk or ws_bytes < 4 * L2_BYTES))
    flush_l2_fn = L2Flush(dev) if flush_l2 else None

    def flush():
        if flush_l2_fn is not None:
            flush_l2_fn()

    def step(ev=None):
        if wl.append:
            ctx.pkv_append_kv(knew, vnew, bidx, pos, cache, pt)
        if ev is not None:
            # the dominant kernel: index scoring on the sparse workloads, attention otherwise
            ctx.pkv_set_profile_events(ev[0], ev[1])
        if wl.topk:
            if wl.n_cand:
                ctx.pkv_score_topk_cand(qidx, tq, wts, ic, pt, cand, wl.topk, sel, ws=ws_s)
            else:
                ctx.pkv_score_topk(qidx, tq, wts, ic, pt, seq_len, wl.topk, sel, ws=ws_s)
        if wl.replay:
            ctx.pkv_replay_attn(q, cache, pt, plen, win, scale, out, lse, ws=ws)
        elif fused:
            ctx.pkv_decode_attn_fused(q, cache, pt, seq_len, win, scale, rpos, table, W.ROPE_DIM, W.OUT_SCALE, out8,
                                      None, lse, ws=ws, sel_idx=sel)
        else:
            ctx.pkv_decode_attn(q, cache, pt, seq_len, win, scale, out, lse, ws=ws, sel_idx=sel)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ctx.pkv_get_error() != P.OK:
        raise RuntimeError("device error during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    n0 = ctx.pkv_launch_count()
    if args.profile_region:
        torch.cuda.profiler.start()
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0e.record()
    for i in range(args.steps):
        flush()
        step_evs[i][0].record()
        step(evs[i])
        step_evs[i][1].record()
    t1e.record()
    torch.cuda.synchronize()
    if args.profile_region:
        torch.cuda.profiler.stop()
    n1 = ctx.pkv_launch_count()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    # medians over the timed steps (each step between its own pair of events)
    ms_step = statistics.median(a.elapsed_time(b) for a, b in step_evs)
    kern_ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    ms_step, kern_ms = max_over_ranks([ms_step, kern_ms], world, dev)
    ms_eager = ms_step
    graph = getattr(args, "graph", False)
    if graph:
        # the whole step captured once as a CUDA graph, then replayed: same kernels, no
        # per-launch host work (kern_ms above stays the eager per-launch measurement)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            gev[i][0].record()
            g.replay()
            gev[i][1].record()
        torch.cuda.synchronize()
        ms_step = max_over_ranks([statistics.median(a.elapsed_time(b) for a, b in gev)], world, dev)[0]
    if ctx.pkv_get_error() != P.OK:
        raise RuntimeError("device error in the timed region")

    # ---- accounting
    if wl.topk:
        cnt = (sel >= 0).sum(1).cpu().numpy()
        attn_bytes, tokens = needed_bytes(wl, sel_counts=cnt, fused=fused)
        if wl.n_cand:     # candidate list + the candidates' index keys
            score_bytes = B * wl.n_cand * (4 + 64 + 8) + B * 64 * 128 + B * 64 * 4 + B * wl.topk * 4
        else:
            score_bytes = sum((int(L) + 63) // 64 for L in wl.seq_len) * 64 * (64 + 8) + B * 64 * 128 + B * 64 * 4 + B * wl.topk * 4
        step_bytes = attn_bytes + score_bytes
    else:
        attn_bytes, tokens = needed_bytes(wl, fused=fused)
        step_bytes = attn_bytes + (B * (2 * d * 4 + 8 + kv_token_bytes(d)) if wl.append else 0)
    gbs = job_gbs(step_bytes, ms_step, world)
    peak, peak_kind = measured_peak()
    achieved = attn_bytes / (kern_ms * 1e-3) / 1e9
    roofline = {"kernel": "attention (global + window segments)", "bound": "hbm",
                "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "bytes_per_launch": int(attn_bytes), "launch_ms": round(kern_ms, 5),
                "traffic": committed_traffic("attention", name)}
    if wl.topk:
        if wl.n_cand:
            positions, pages = B * wl.n_cand, B * ((wl.n_cand + 63) // 64)
        else:
            pages = sum((int(L) + 63) // 64 for L in wl.seq_len)
            positions = int(np.sum(wl.seq_len))
        sbytes = score_kernel_bytes(wl, positions, pages)
        sach = sbytes / (kern_ms * 1e-3) / 1e9
        roofline = {"kernel": "index scoring (score_tc_kernel)", "bound": "hbm", "achieved": round(sach, 2),
                    "peak": peak, "unit": "GB/s", "frac": round(sach / peak, 4), "peak_kind": peak_kind,
                    "bytes_per_launch": int(sbytes), "launch_ms": round(kern_ms, 5),
                    "traffic": committed_traffic("score", name)}
    if wl.replay:
        # bounded replay is a dense contraction: QK^T and P.V, 2 flops per multiply-add,
        # for every (replayed row, head, entry it attends) = 4*H*d flops per (row, entry)
        entries = sum(128 * (int(wl.prefix_len[b]) - 128) + 128 * 129 // 2 for b in range(B))
        flops = 4.0 * H * d * entries
        tpeak, tkind = tensor_peak()
        tf = flops / (kern_ms * 1e-3) / 1e12
        roofline = {"kernel": "attention (replay)", "bound": "tensor", "achieved": round(tf, 1), "peak": tpeak,
                    "unit": "TFLOP/s", "frac": round(tf / tpeak, 4), "peak_kind": tkind,
                    "flops_per_launch": flops, "launch_ms": round(kern_ms, 5),
                    "traffic": committed_traffic("attention", name), "hbm_gbs": round(achieved, 2)}
    launches_per_step = (n1 - n0) / args.steps

    # ---- end to end through the public API with host buffers: every step copies its
    # inputs in from pinned host memory (the bf16 query, the appended K/V rows, for
    # the sparse path the float32 index query, quantized to FP8 on the device) and
    # its results out (O or its FP8 form, LSE, the selected positions)
    qh = torch.from_numpy(q_host.view(np.int16)).pin_memory()
    o_dev = out8 if fused else out
    oh = torch.empty(o_dev.shape, dtype=o_dev.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    kh = vh = None
    if wl.append:
        kh = torch.from_numpy(wl.new_rows(W.T_KNEW)).pin_memory()
        vh = torch.from_numpy(wl.new_rows(W.T_VNEW)).pin_memory()
    qfh = qf_dev = selh = None
    if wl.topk:
        qfh = torch.from_numpy(np.ascontiguousarray(qf)).pin_memory()
        qf_dev = torch.empty(qfh.shape, dtype=torch.float32, device=dev)
        selh = torch.empty(sel.shape, dtype=torch.int32).pin_memory()
    n_e2e = max(3, min(args.steps, 50))

    def e2e_step():
        q.view(torch.int16).copy_(qh, non_blocking=True)
        if wl.append:
            knew.copy_(kh, non_blocking=True)
            vnew.copy_(vh, non_blocking=True)
        if wl.topk:
            qf_dev.copy_(qfh, non_blocking=True)
            P.pkv_quantize_fp8(qf_dev, tq, qidx)
        step()
        oh.copy_(o_dev, non_blocking=True)
        lh.copy_(lse, non_blocking=True)
        if wl.topk:
            selh.copy_(sel, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_e2e)]
    for i in range(n_e2e):
        flush()
        e2e_evs[i][0].record()
        e2e_step()
        e2e_evs[i][1].record()
    torch.cuda.synchronize()
    e2e_ms = statistics.median(a.elapsed_time(b) for a, b in e2e_evs)
    bi = qh.numel() * 2 + (kh.numel() * 4 * 2 if wl.append else 0) + (qfh.numel() * 4 if wl.topk else 0)
    bo = oh.numel() * oh.element_size() + lh.numel() * 4 + (selh.numel() * 4 if wl.topk else 0)
    e2e = {"value": round(step_bytes / (e2e_ms * 1e-3) / 1e9 * world, 2), "unit": "GB/s",
           "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo)}

    res = {
        "metric": "decode-attention KV GB/s (needed bytes / step time)",
        "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvf4 block-scaled QK^T (5 FP4 query terms), e4m3 window QK^T, f16 PV; f32 accumulate and softmax",
        "attention_path": {2: "tcgen05 tensor-core"}.get(ctx.pkv_attn_path(), "none"),
        "data": "synthetic (seeded N(0,1), 2% channels x8, bf16 Q; no trained weights)",
        "config": {"workload": workload_desc(name), "name": wl.name, "batch": B, "heads": H, "d": d,
                   "tokens_read": int(tokens), "needed_bytes_per_step": int(step_bytes),
                   "l2": (L2Flush.DESC if flush_l2 else "working set > 4x the 129 MB L2; no flush between steps"),
                   "timing": "median over the timed steps"},
        "pct_of_hbm_peak": round(100 * gbs / world / peak, 2), "hbm_peak_kind": peak_kind,
        "pct_of_8TBps_nominal": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "seq_per_s": round(B * world / (ms_step * 1e-3), 1),
        "roofline": roofline,
        "clocks": clk, "gpu_launches": int(n1 - n0), "launches_per_step": launches_per_step,
        "setup_s": round(setup_s, 1),
        "step_mode": "cuda graph replay" if graph else "eager", "ms_per_step_eager": round(ms_eager, 4),
    }
    res["e2e"] = e2e
    return res, wl


class L2Flush:
    """Evicts the step's data from the 129 MB L2 before a timed step: writes a
    256 MB buffer, then reads another 256 MB one.  The read leaves the L2 full of
    clean lines, so the timed step does not pay for writing back the flush's own
    dirty lines (measured: 6-8 us of DRAM time inside the next launch after a
    write-only flush).  Both passes run before the step's start event."""
    DESC = "L2 flushed before every timed step: 256 MB written, then another 256 MB read (clean lines left)"

    def __init__(self, dev):
        import torch
        self.w = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def run_score_sweep(args, name, pool):
    """Index scoring + top-2048 of the sparse shape (4 sequences) at one length, the L2
    flushed before every step (256 MB written, then 256 MB read), so the index keys come from HBM: one
    line with the scoring kernel's roofline."""
    import torch
    import precision_kv_cache_gb300 as P
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = _wl_cache(name)
    ts, _ = tensor_scales()
    ctx = P.Context(wl.d, wl.H, device=0)
    pt = torch.from_numpy(wl.page_table).to(dev)
    ic = fill_index(ctx, P, torch, wl, name, ts, pool, pt)
    qf = wl.index_q()
    tq = float(np.float32(np.float32(np.abs(qf).max()) / np.float32(448.0)))
    qidx = torch.empty(qf.shape, dtype=torch.uint8, device=dev)
    P.pkv_quantize_fp8(torch.from_numpy(qf).to(dev), tq, qidx)
    wts = torch.from_numpy(wl.index_w()).to(dev)
    seq_len = torch.from_numpy(wl.seq_len).to(dev)
    sel = torch.empty(wl.B, wl.topk, dtype=torch.int32, device=dev)
    ws = ctx.workspace(P.OP_SCORE_TOPK, wl.B, pt.shape[1] * 64)
    flush = L2Flush(dev)

    def call():
        ctx.pkv_score_topk(qidx, tq, wts, ic, pt, seq_len, wl.topk, sel, ws=ws)

    for _ in range(max(3, args.warmup)):
        flush()
        call()
    torch.cuda.synchronize()
    if ctx.pkv_get_error() != P.OK:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(dev.index)
    clocks.start()
    # the scoring kernel alone: eager calls, the library's events around that kernel
    n0 = ctx.pkv_launch_count()
    kern_t = []
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        flush()
        ctx.pkv_set_profile_events(k0, k1)
        call()
        torch.cuda.synchronize()
        kern_t.append(k0.elapsed_time(k1))
    n_call = (ctx.pkv_launch_count() - n0) // args.steps
    # the whole call (scoring + top-k) captured once as a CUDA graph; each step flushes
    # the L2, then replays it between two events
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(g):
        call()
    for _ in range(3):
        flush()
        g.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    call_t = []
    for _ in range(args.steps):
        flush()
        a0.record()
        g.replay()
        a1.record()
        torch.cuda.synchronize()
        call_t.append(a0.elapsed_time(a1))
    clk = clocks.stop()
    if ctx.pkv_get_error() != P.OK:
        raise RuntimeError("device error in the timed region")
    n0, n1 = 0, n_call * args.steps
    call_ms = statistics.mean(call_t)
    kern_ms = statistics.mean(kern_t)
    pages = sum((int(L) + 63) // 64 for L in wl.seq_len)
    positions = int(np.sum(wl.seq_len))
    sbytes = score_kernel_bytes(wl, positions, pages)
    needed = positions * (64 + 8) + pages * 4 + wl.B * 64 * (128 + 4) + wl.B * wl.topk * 4
    peak, peak_kind = measured_peak()
    ach = sbytes / (kern_ms * 1e-3) / 1e9
    return {"metric": "index scoring + top-k GB/s (needed bytes / call time)",
            "value": round(needed / (call_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(call_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 tensor-core MMA (f32 accumulate)",
            "data": "synthetic (seeded N(0,1) index keys with 2% channels x8, FP8 queries, U(0,1) weights)",
            "config": {"workload": f"index scoring sweep: batch {wl.B}, 64 FP8 index heads x 128, NVFP4 keys, "
                                   f"{SCORE_SWEEP[name]} positions each, top-{wl.topk}",
                       "name": wl.name, "batch": wl.B, "positions": positions, "needed_bytes_per_step": int(needed),
                       "l2": L2Flush.DESC},
            "roofline": {"kernel": "index scoring (score_tc_kernel)", "bound": "hbm", "achieved": round(ach, 2),
                         "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4), "peak_kind": peak_kind,
                         "bytes_per_launch": int(sbytes), "launch_ms": round(kern_ms, 5), "traffic": None},
            "clocks": clk, "gpu_launches": int(n1 - n0), "launches_per_step": (n1 - n0) / args.steps,
            "plan_topk_ms": round(call_ms - kern_ms, 4), "step_mode": "call: cuda graph replay; scoring kernel: eager calls; L2 flushed before each"}


# ----------------------------------------------------------------------------- oracle (CPU) arm
_TABLE = {}


def _oracle_decode(name, wl, b, q, K, V, Kw, Vw, scale):
    """The oracle's decode of one sequence; for a fused workload with the query
    rotated, the output turned back and encoded as E4M3."""
    from oracle import attention as A
    from oracle import formats as F
    if name not in FUSED:
        return A.decode(q, K, V, Kw, Vw, scale)
    if name not in _TABLE:
        _TABLE[name] = W.rope_table(wl.seed, int(wl.rope_pos().max()) + 1, W.ROPE_DIM)
    row = _TABLE[name][int(wl.rope_pos()[b])].astype(np.float64)
    c, sn = row[:W.ROPE_DIM // 2], row[W.ROPE_DIM // 2:]
    O, lse = A.decode(A.rope(q, c, sn, W.ROPE_DIM), K, V, Kw, Vw, scale)
    return F.fp8_quantize(A.rope(O, c, sn, W.ROPE_DIM, inverse=True), W.OUT_SCALE), lse


def oracle_sample(name, budget_s=15.0, max_seqs=None):
    """Time the float64 oracle's decode step on a bounded sample of the workload:
    sequences in order until ~budget_s seconds of timed CPU work."""
    from oracle import attention as A
    from oracle import cache as C
    from oracle import formats as F
    wl = _wl_cache(name)
    ts, tw = tensor_scales()
    ts, tw = np.float32(ts), np.float32(tw)
    spent, nbytes, seqs = 0.0, 0, 0
    scale = 1.0 / math.sqrt(wl.d)
    if name in FUSED and name not in _TABLE:
        _TABLE[name] = W.rope_table(wl.seed, int(wl.rope_pos().max()) + 1, W.ROPE_DIM)
    order = range(wl.B) if max_seqs is None else range(min(wl.B, max_seqs))
    for b in order:
        if wl.replay:
            L = int(wl.prefix_len[b]) - 128
        else:
            L = int(wl.seq_len[b])
        pages = {int(wl.page_table[b, j]) for j in range((L + 63) // 64)}
        Kp, Vp = C.fill_pages(wl, ts, ts, pages=pages)
        kw, vw = C.window_codes(wl, tw, tw, b)
        t0 = time.perf_counter()
        K = C.dequant_seq(wl, Kp, ts, b, L)
        V = C.dequant_seq(wl, Vp, ts, b, L)
        Kw, Vw = F.fp8_dequantize(kw, tw), F.fp8_dequantize(vw, tw)
        if wl.replay:
            q = F.bf16_to_f64(wl.replay_q_bits(b))
            A.replay(q, K, V, Kw, Vw, scale, rows=[0, 127])
            rows = 2
        else:
            _oracle_decode(name, wl, b, F.bf16_to_f64(wl.q_bits_seq(b)), K, V, Kw, Vw, scale)
            rows = 1
        spent += time.perf_counter() - t0
        nbytes += L * kv_token_bytes(wl.d) + 128 * wl.d * 2 + rows * wl.H * wl.d * (2 + 4)
        seqs += 1
        if spent >= budget_s:
            break
    cores = len(os.sched_getaffinity(0))
    return {"value": round(nbytes / spent / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{seqs} of {wl.B} sequences of {wl.name} ({'2 replay rows each, ' if wl.replay else ''}"
                      f"dequantize + float64 attention, numpy BLAS threads)",
            "seconds": round(spent, 2)}


def run_reference(args):
    """--impl reference: the oracle as it stands, each step one sampled sequence."""
    from oracle import attention as A
    from oracle import cache as C
    from oracle import formats as F
    name = args.workload
    wl = _wl_cache(name)
    ts, tw = tensor_scales()
    ts, tw = np.float32(ts), np.float32(tw)
    scale = 1.0 / math.sqrt(wl.d)
    prepared = []
    nprep = min(wl.B, 4)
    if name in FUSED and name not in _TABLE:
        _TABLE[name] = W.rope_table(wl.seed, int(wl.rope_pos().max()) + 1, W.ROPE_DIM)
    for b in range(nprep):
        L = int(wl.prefix_len[b]) - 128 if wl.replay else int(wl.seq_len[b])
        pages = {int(wl.page_table[b, j]) for j in range((L + 63) // 64)}
        Kp, Vp = C.fill_pages(wl, ts, ts, pages=pages)
        prepared.append((b, L, Kp, Vp, C.window_codes(wl, tw, tw, b)))

    def step(i):
        b, L, Kp, Vp, (kw, vw) = prepared[i % nprep]
        L = min(L, 8192)          # bounded sample: the first 8192 global tokens of the sequence
        K = C.dequant_seq(wl, Kp, ts, b, L)
        V = C.dequant_seq(wl, Vp, ts, b, L)
        Kw, Vw = F.fp8_dequantize(kw, tw), F.fp8_dequantize(vw, tw)
        if wl.replay:
            A.replay(F.bf16_to_f64(wl.replay_q_bits(b)), K, V, Kw, Vw, scale, rows=[0])
            return L * kv_token_bytes(wl.d) + 128 * wl.d * 2 + wl.H * wl.d * 6
        _oracle_decode(name, wl, b, F.bf16_to_f64(wl.q_bits_seq(b)), K, V, Kw, Vw, scale)
        return L * kv_token_bytes(wl.d) + 128 * wl.d * 2 + wl.H * wl.d * 6

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    nb = 0
    for i in range(args.steps):
        nb += step(i)
    dt = time.perf_counter() - t0
    v = nb / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    return {"impl": "reference", "metric": "decode-attention KV GB/s (needed bytes / step time)", "value": round(v, 4),
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(name), "name": wl.name,
                       "sample": f"each step: the first <=8192 global tokens + window of one of the first {nprep} "
                                 f"sequences (dequantize + float64 decode)"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"one sequence of {wl.name} per step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(SWEEP) + list(PROFILE), default="c2",
                    help="c1-c4 (and c3c, c1f, c3f): the bench workloads; s32k..s512k: one sweep length; "
                         "p2, p4: smaller c2 / c4 runs used as ncu capture cases")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time eager calls instead of the step captured as one CUDA graph (the default)")
    ap.add_argument("--score-sweep", action="store_true",
                    help="index-scoring sweep (4 sequences of 32K-512K positions, L2 flushed per step): one line per length")
    ap.add_argument("--sweep", action="store_true",
                    help="long-context decode sweep (32K-512K tokens, >= 1 GiB of KV per step): one line per length")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flush-l2", choices=["auto", "on", "off"], default="auto",
                    help="write 256 MB before every timed step (auto: when the step's bytes are < 4x the L2)")
    ap.add_argument("--profile-region", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    # spawn the generator pool before any CUDA call
    import concurrent.futures as cf
    import multiprocessing as mp
    nproc = max(1, min(16, len(os.sched_getaffinity(0)) - 1))
    pool = cf.ProcessPoolExecutor(nproc, mp_context=mp.get_context("spawn")) if nproc > 1 else None
    try:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group("nccl")
        if args.score_sweep:
            if rank == 0:
                for name in sorted(SCORE_SWEEP, key=SCORE_SWEEP.get):
                    print(json.dumps(run_score_sweep(args, name, pool)), flush=True)
                    _WL.pop(name, None)
            return
        if args.sweep:
            for name in sorted(SWEEP, key=SWEEP.get):
                args.workload = name
                res, wl = run_gpu(args, rank, world, pool)
                if rank == 0:
                    print(json.dumps(res), flush=True)
                _WL.pop(name, None)
            return
        res, wl = run_gpu(args, rank, world, pool)
    finally:
        if pool:
            pool.shutdown()
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = oracle_sample(args.workload, args.cpu_budget)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
