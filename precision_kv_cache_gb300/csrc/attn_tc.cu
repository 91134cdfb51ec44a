// Tensor-core decode / replay attention over the paged NVFP4 global KV and the
// FP8 window, for sm_103a (tcgen05 MMA, block-scaled FP4 for QK^T, TMEM).
//
// What it computes: for every query row g (a decode sequence, or one replayed
// token), all H <= 64 query heads attend the same K/V (MQA over one shared
// latent - vLLM blog "Performances agentiques"): the global tokens of the
// sequence, stored in NVFP4 64-token pages ("MegaAttention avec KV compressé
// NVFP4"), then the FP8 window entries (cocoloop summary of the same blog,
// "Les particularités du modèle lui-même"; replay: causal, clipped at
// s = H-128, "SWA bounded replay").
// Output: a normalized partial (O, LSE) per (CTA, query row) segment, merged
// by merge_tc_kernel ("flash-decoding": split along the sequence + LSE merge).
//
// Design (one persistent CTA per SM, 768 threads, warp-specialized):
//   * work = 128-token tiles; each query row has ceil(L/128) NVFP4 tiles plus
//     one window tile; the concatenated tile list, with ROW_END empty planning
//     units after every row (the cost of a row's end), is cut into one
//     contiguous range per CTA.
//   * S^T = K Q^T (M = 128 tokens, N = 64 heads) runs on the block-scaled FP4
//     tensor-core contraction: A = the two K pages of a tile as stored (E2M1
//     codes, K-major with the 128/64-byte swizzle; copied from shared memory
//     into TMEM once per tile with tcgen05.cp), their E4M3 block scales in
//     TMEM (written by warps 12-15, thread = tile row), B = the query written as a
//     sum of NQT FP4 terms, q ~ sigma_h * sum_t c_t 8^-t (c_t E2M1 codes, one
//     factor sigma_h per head applied to the logits; the term weights 8^-t are
//     the constant B block scales).  No K dequantization.
//   * the window tile's S^T runs on the FP8 contraction: A = the window K codes
//     (E4M3, copied by TMA with the 128-byte swizzle), B = the query as two E4M3
//     terms with a power-of-two factor per head (exact for a bf16 query).
//   * warp 22 streams V pages (and the window V, 32 entries per ring slot, by
//     TMA) into a shared-memory ring; warps 0-11, three
//     groups of four, dequantize V^T to f16 into TMEM (thread = channel, 128
//     channels x 64 tokens at a time: the A operand of O^T = V^T P, M = 128
//     channels, N = 64 heads); warp 23 issues the PV MMAs (P f16 in shared
//     memory, B operand).
//   * warps 12-19 run the online softmax on S (FP32, exp2, lazy max update with
//     threshold 2^8), write P (f16), normalize O and write the partial result.
//     The query terms of each row are split ahead by qsplit_kernel; warp 21
//     copies them into shared memory at the row's first tile (and its window
//     tile) and issues the QK MMAs.
//   * fused decode ("MegaAttention avec KV compressé NVFP4": query RoPE,
//     attention, inverse RoPE on the output, FP8 output in one pass): the query
//     is turned before it is split into terms, and the merge turns the final O
//     back and encodes it as E4M3 - no extra kernel and no extra pass over O.
// Every wait is bounded; on a timeout the CTA sets the error word, stops all
// roles, drains its own copies / MMAs and frees its TMEM before returning.
#include <cstddef>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_tc.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace tcattn {

constexpr int TILE = 128;
constexpr int NH = 64;                 // MMA N: query heads (zero-padded)
constexpr int NQT = 5;                 // FP4 terms of the query
constexpr int NTHREADS = 768;          // 24 warps
// warp roles
constexpr int W_VDEQ = 0;              // 12 warps: V dequantizers, NVG groups of four
constexpr int W_SMAX = 12;             // 8 warps: softmax + epilogue; warps 12-15 also the K block scales
constexpr int W_KPROD = 20;            // K tile producer
constexpr int W_QK = 21;               // QK MMA issuer, TMEM owner
constexpr int W_VPROD = 22;            // V page producer
constexpr int W_PV = 23;               // PV MMA issuer
constexpr uint32_t NGRP = 4;           // arrivals per V ring slot release / V chunk: one per warp of a group
constexpr int NVG = 3;                 // V dequant groups (chunk i of the CTA to group i % NVG)
// Planning units per query row beyond its tiles: the CTA ranges are cut over
// tiles + ROW_END units per row, so a range that holds a row's end (window tile,
// partial write, the next row's start: measured at about four to five tiles of
// time) gets that many fewer tiles.  The extra units hold no work.
constexpr int ROW_END = 5;
constexpr float TAU = 8.f;             // lazy rescale threshold (log2 units)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// TMEM columns (512 allocated)
constexpr int NVS = 2;                 // V chunk slots (chunk i of the CTA in slot i % NVS)
constexpr uint32_t COL_S = 0;          // S^T tile: 64 columns (fp32)
constexpr uint32_t COL_SFA = 64;       // K block scales of a tile: 32 columns (4 per 64-channel K step)
constexpr uint32_t COL_SFB = 96;       // query term weights: 4 columns per term
constexpr uint32_t COL_KA = 128;       // the tile's K codes, A operand of S^T: 8 columns per 64-channel K step
constexpr uint32_t COL_V = 192;        // V^T chunk slots: NVS x 32 columns (128 channels x 64 tokens, f16 pairs)
constexpr uint32_t COL_O = 256;        // O^T: 4 chunks x 64 columns
static_assert(COL_SFA + 32 <= COL_SFB && COL_SFB + 32 <= COL_KA && COL_KA + 64 <= COL_V && COL_V + 32 * NVS <= COL_O,
              "TMEM map");

constexpr int NKS = 2;                 // K tile slots (two pages each, or window chunks)
constexpr int NVR = 9;                 // V ring: slots of one 128-channel chunk of one page
constexpr int VGRP = 4;                // V ring slots filled by one warp instruction (one lane each)
constexpr int VCODES = 8 * 128 * 4;    // V codes of a 128-channel chunk of a page (8 octets x 128 words)
constexpr int VSCALES = 8 * PKV_PAGE;  // its block scales (8 blocks x 64 tokens)
constexpr int VSLOT = VCODES + VSCALES;
constexpr int WCHUNK = 128 * 128;      // window K chunk: 128 entries x 128 channels of E4M3
constexpr int WVROWS = 32;             // window V chunk: 32 entries x 128 channels of E4M3, one V ring slot
constexpr int WVQ = PKV_WINDOW / WVROWS;   // window V chunks per 128-channel chunk
static_assert(WVROWS * 128 <= VCODES, "a window V chunk fits a ring slot");

template <int D>
struct Cfg {
  static constexpr int RB = D / 2 < 128 ? D / 2 : 128;       // K code bytes of a row per column block
  static constexpr int NCB = D / 2 / RB;                     // column blocks of a K row
  static constexpr int KS = D / 64;                          // K steps of the FP4 contraction
  static constexpr int PAGE_DATA = PKV_PAGE * D / 2;
  static constexpr int PAGE_SCALE = PKV_PAGE * D / 16;
  static constexpr int QT_BYTES = NH * D / 2;                // one FP4 query term [NCB][64][RB]
  static constexpr int QW_BYTES = NH * D;                    // one E4M3 query term [D/128][64][128]
  static constexpr int Q_BYTES = NQT * QT_BYTES > 2 * QW_BYTES ? NQT * QT_BYTES : 2 * QW_BYTES;
  static constexpr int P_BYTES = TILE * NH * 2;
  static constexpr int KSLOT = TILE * D / 2 > WCHUNK ? TILE * D / 2 : WCHUNK;
  static constexpr int NWC = D / 128;                        // window K chunks
  static constexpr int CPS = KSLOT / WCHUNK;                 // window chunks per K slot
  static constexpr int NWS = (NWC + CPS - 1) / CPS;          // K slots one window tile uses
  static constexpr int NVCH = D / 128;                       // V chunks of 128 channels
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = OFF_Q + Q_BYTES;              // 2 P buffers
  static constexpr int OFF_K = OFF_P + 2 * P_BYTES;          // K tile slots
  static constexpr int OFF_V = OFF_K + NKS * KSLOT;          // V ring
  static constexpr int DYN = OFF_V + NVR * VSLOT + 1024;     // + alignment slack
  // a query row split ahead of the attention (qsplit_kernel), in global memory:
  // the FP4 terms, the E4M3 terms, then the two logit-factor vectors
  static constexpr int QS_E4M3 = NQT * QT_BYTES;
  static constexpr int QS_ZSG = QS_E4M3 + 2 * QW_BYTES;
  static constexpr int QS_ZSW = QS_ZSG + NH * 4;
  static constexpr int QS_ROW = (QS_ZSW + NH * 4 + 1023) / 1024 * 1024;
  static_assert(QT_BYTES % 1024 == 0 && OFF_P % 1024 == 0 && OFF_K % 1024 == 0 && KSLOT % 1024 == 0 &&
                OFF_V % 16 == 0, "operand tiles stay 1024-aligned");
  static_assert(KS * 4 <= 32, "K scales of a tile fit one 32-column buffer");
};

struct Shared {
  uint64_t kr_full[NKS], kr_empty[NKS], vr_full[NVR], vr_empty[NVR];
  uint64_t sfa_full;
  uint64_t vfull[NVS];     // slot s holds chunk i (i % NVS == s): its four V warps stored it
  uint64_t vempty[NVG];    // barrier i % NVG: the P.V of chunk i is complete
  uint64_t s_full, s_empty, p_full[2], p_empty[2], q_full, q_empty, o_empty, drain, drain2;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float m[NH];     // running max per head (log2 units)
  alignas(16) float alpha[NH];
  alignas(16) float zsg[NH];   // logit factor per head of the global tiles (log2 units)
  alignas(16) float zsw[NH];   // logit factor per head of the window tile (log2 units)
  float red[4][NH];            // cross-warp reductions
  alignas(16) uint32_t vsc[4 * NVG][64];   // per V warp: f16x2 block-scale pairs of its current chunk (2 blocks x 32)
  alignas(16) uint32_t sfs[TILE][8];       // K block-scale words of the next tile, row m = token m (staged by cp.async)
};
static_assert(offsetof(Shared, m) % 16 == 0 && offsetof(Shared, alpha) % 16 == 0 && offsetof(Shared, zsg) % 16 == 0 &&
                  offsetof(Shared, zsw) % 16 == 0 && offsetof(Shared, vsc) % 16 == 0 && offsetof(Shared, sfs) % 16 == 0,
              "16-byte shared-memory vector accesses");

// ---------------------------------------------------------------- schedule
__device__ __forceinline__ long long cta_start(long long T, int G, int c) { return (T * c) / G; }

// first group whose tiles reach past x
__device__ __forceinline__ int group_of(const int* ts, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)ts[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Unit {            // what a query row sees
  int b, n_glob, n_win, row;
  const uint8_t* wk;
  const uint8_t* wv;
};

__device__ __forceinline__ Unit unit_of(const AttnArgs& a, int g) {
  Unit u;
  int b, ng, nw;
  const uint8_t *wk, *wv;
  unit_extent(a, g, &b, &ng, &nw, &wk, &wv);
  u.b = b; u.n_glob = ng; u.n_win = nw; u.row = g; u.wk = wk; u.wv = wv;
  return u;
}

// ---------------------------------------------------------------- plan
// tile_start[g] = sum over g' < g of (ceil(n_glob(g')/128) + 1 + ROW_END); tile_start[n] =
// total; then tile_start[n + 1 + c] = the query row where CTA c (of G) starts
// (run by one block of the query-split launch, whose other blocks do not read it)
__device__ __noinline__ void plan_tiles(const AttnArgs& a, int* tile_start, int G) {
  __shared__ int wsum[32];
  __shared__ int carry;
  const int NT = blockDim.x;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.n_groups; base += NT) {
    const int g = base + threadIdx.x;
    int n = 0;
    if (g < a.n_groups) {
      int b, ng, nw;
      const uint8_t *wk, *wv;
      unit_extent(a, g, &b, &ng, &nw, &wk, &wv);
      n = (ng + TILE - 1) / TILE + 1 + ROW_END;
    }
    int incl = n;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int pre = carry;
    for (int i = 0; i < w; ++i) pre += wsum[i];
    if (g < a.n_groups) tile_start[g] = pre + incl - n;
    __syncthreads();
    if (threadIdx.x == NT - 1) carry = pre + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_start[a.n_groups] = carry;
  __syncthreads();
  const long long T = carry;
  for (int c = threadIdx.x; c < G; c += NT) tile_start[a.n_groups + 1 + c] = group_of(tile_start, a.n_groups, cta_start(T, G, c));
}

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

__device__ __forceinline__ void fail(Shared& sh, int* err) {
  sh.abort_flag = 1;
  report(err, PKV_DEVERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t f32_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^x, one approximate-unit instruction (relative error ~2^-22; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sum of v[i] over the 32 lanes of the warp, by reduce-scatter: lane l returns
// the total of entry (l >> 1) & 15 (the two lanes of a pair hold the same sum).
__device__ __forceinline__ float warp_sum16(const float* v, int lane) {
  float a[8], b[4], c[2];
  const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    a[i] = (u4 ? v[i + 8] : v[i]) + __shfl_xor_sync(0xffffffffu, u4 ? v[i] : v[i + 8], 16);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = (u3 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xffffffffu, u3 ? a[i] : a[i + 4], 8);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    c[i] = (u2 ? b[i + 2] : b[i]) + __shfl_xor_sync(0xffffffffu, u2 ? b[i] : b[i + 2], 4);
  const float d = (u1 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, u1 ? c[0] : c[1], 2);
  return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// The same reduce-scatter with max instead of sum.
__device__ __forceinline__ float warp_max16(const float* v, int lane) {
  float a[8], b[4], c[2];
  const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    a[i] = fmaxf(u4 ? v[i + 8] : v[i], __shfl_xor_sync(0xffffffffu, u4 ? v[i] : v[i + 8], 16));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = fmaxf(u3 ? a[i + 4] : a[i], __shfl_xor_sync(0xffffffffu, u3 ? a[i] : a[i + 4], 8));
#pragma unroll
  for (int i = 0; i < 2; ++i)
    c[i] = fmaxf(u2 ? b[i + 2] : b[i], __shfl_xor_sync(0xffffffffu, u2 ? b[i] : b[i + 2], 4));
  const float d = fmaxf(u1 ? c[1] : c[0], __shfl_xor_sync(0xffffffffu, u1 ? c[0] : c[1], 2));
  return fmaxf(d, __shfl_xor_sync(0xffffffffu, d, 1));
}

// E4M3 code of 8 * 8^-t: the B-side block scale of query term t
__host__ __device__ constexpr uint32_t term_scale_code(int t) {
  return t == 0 ? 0x50u : t == 1 ? 0x38u : t == 2 ? 0x20u : t == 3 ? 0x08u : 0x01u;   // 8, 1, 1/8, 1/64, 1/512
}
static_assert(NQT <= 5 && 4 * NQT <= 32, "term_scale_code covers five terms; one 32-column store writes them");

// channels c .. c+7 of query head h of row g as float (bf16 -> f32, exact); in the
// rotated part of a fused decode, turned by the row's angles in FP32 (every
// product, difference and sum rounded separately: no fused multiply-add) and
// rounded back to bf16 (nearest, ties to even) - the rotated query is a bf16
// tensor like the query itself
template <int D>
__device__ __forceinline__ void cvt_q8(const AttnArgs& a, uint4 v, int c, int pos, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  if (pos >= 0 && c >= D - a.rope_dim) {
    const int i0 = (c - (D - a.rope_dim)) / 2;
    const float* row = a.cos_sin + (size_t)pos * a.rope_dim;
    const float4 cr = __ldg(reinterpret_cast<const float4*>(row + i0));
    const float4 sr = __ldg(reinterpret_cast<const float4*>(row + a.rope_dim / 2 + i0));
    const float cc[4] = {cr.x, cr.y, cr.z, cr.w}, ss[4] = {sr.x, sr.y, sr.z, sr.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float x0 = x[2 * i], x1 = x[2 * i + 1];
      const float y0 = __fsub_rn(__fmul_rn(x0, cc[i]), __fmul_rn(x1, ss[i]));
      const float y1 = __fadd_rn(__fmul_rn(x0, ss[i]), __fmul_rn(x1, cc[i]));
      x[2 * i] = __bfloat162float(__float2bfloat16_rn(y0));
      x[2 * i + 1] = __bfloat162float(__float2bfloat16_rn(y1));
    }
  }
}


// ---------------------------------------------------------------- query split
// Both forms of a query row as the B operand of S^T = K Q^T, written once per
// row to global memory (the attention CTAs of the row copy them in):
//   fp4 form (global tiles): per head, x = q * 4/amax_h in [-4, 4];
//     c_0 = E2M1(x), c_t = E2M1(8 (r_{t-1} ...)): x ~ sum_t c_t 8^-t, the codes
//     stored as NQT K-major FP4 terms [NCB][64 heads][RB] (swizzle as the K
//     pages); the B block scales 8^(1-t) are constants in TMEM, so the
//     contraction gives 8x and the logit factor is scale * ts_k * amax_h / 32.
//   e4m3 form (window tile): x = q * 2^-k_h (k_h: the least power of two with
//     |x| <= 448), t1 = E4M3(x), t2 = E4M3(x - t1) (exact for a bf16 q), two
//     K-major E4M3 terms [D/128][64 heads][128] (128-byte swizzle); the logit
//     factor is scale * tw_k * 2^k_h.
// plus the per-head logit factors (log2 units) of each form.  Grid: (row,
// group of 256 / (D/32) heads); thread st takes head st / (D/32) of the group
// and its 32 channels 32 * (st % (D/32)) ..; heads >= H are written as zero.
// One more block (x = n_groups, y = 0) computes the attention launch's tile
// plan, beside the splits rather than before one of them.
template <int D>
__global__ void __launch_bounds__(256) qsplit_kernel(AttnArgs a, uint8_t* __restrict__ qs, int* tile_start, int G) {
  pkv::dep_wait();
  pkv::dep_trigger();
  if ((int)blockIdx.x == a.n_groups) {
    if (blockIdx.y == 0) plan_tiles(a, tile_start, G);   // the attention launch's tile plan
    return;
  }
  using C = Cfg<D>;
  using KL = KLayout<D>;
  constexpr int PARTS = D / 32;              // threads per head
  constexpr int HPB = 256 / PARTS;           // heads per block
  const int g = blockIdx.x, st = threadIdx.x;
  const int h = blockIdx.y * HPB + st / PARTS, part = st % PARTS;
  const int c0 = 32 * part;
  const bool live = h < a.H;
  int pos = -1;
  if (a.rope_dim > 0) {
    pos = a.rope_pos[g];
    if (pos < 0 || pos >= a.max_pos) {
      if (st == 0 && blockIdx.y == 0) report(a.err, PKV_DEVERR_BAD_PAGE);
      pos = -1;
    }
  }
  // the thread's 32 channels (turned in a fused decode), all loads in flight at once
  float x[32];
  if (live) {
    const uint16_t* qh = a.q + ((size_t)g * a.H + h) * D + c0;
    uint4 raw[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) raw[v] = __ldg(reinterpret_cast<const uint4*>(qh) + v);
#pragma unroll
    for (int v = 0; v < 4; ++v) cvt_q8<D>(a, raw[v], c0 + 8 * v, pos, x + 8 * v);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = 0.f;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < PARTS; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  uint8_t* dst = qs + (size_t)g * C::QS_ROW;
  {
    // FP4 terms: one 16-byte chunk of each term
    const float inv = amax > 0.f ? 4.f / amax : 0.f;
    if (part == 0)
      reinterpret_cast<float*>(dst + C::QS_ZSG)[h] = amax > 0.f ? a.scale * a.cache.ts_k * LOG2E / (8.f * inv) : 0.f;
    uint32_t w[NQT][4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = x[8 * v + i] * inv;
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        uint32_t word = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t b = tc::f32x2_to_e2m1x2(y[2 * i], y[2 * i + 1]);
          word |= b << (8 * i);
          if (t + 1 < NQT) {
            const uint32_t v2 = tc::e2m1x2_to_f16x2(b);
            y[2 * i] = 8.f * (y[2 * i] - tc::f16_lo_to_f32(v2));
            y[2 * i + 1] = 8.f * (y[2 * i + 1] - tc::f16_hi_to_f32(v2));
          }
        }
        w[t][v] = word;
      }
    }
    const int off = KL::chunk(h, part);            // head row h of a term, as token row h of a page
#pragma unroll
    for (int t = 0; t < NQT; ++t)
      *reinterpret_cast<uint4*>(dst + t * C::QT_BYTES + off) = make_uint4(w[t][0], w[t][1], w[t][2], w[t][3]);
  }
  {
    // E4M3 terms: two 16-channel chunks of each term
    int k = 0;
    if (amax > 0.f) {
      const uint32_t u = __float_as_uint(amax / 448.f);
      k = (int)((u >> 23) & 0xFFu) - 127 + ((u & 0x7FFFFFu) ? 1 : 0);
      k = k < -126 ? -126 : (k > 126 ? 126 : k);
    }
    const float down = __uint_as_float((uint32_t)(127 - k) << 23);   // 2^-k
    const float up = __uint_as_float((uint32_t)(127 + k) << 23);     // 2^k
    if (part == 0) reinterpret_cast<float*>(dst + C::QS_ZSW)[h] = amax > 0.f ? a.scale * a.tw_k * up * LOG2E : 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int c = c0 + 16 * half;
      uint32_t w1[4], w2[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const float* y = x + 16 * half + 2 * i;
        const float y0 = y[0] * down, y1 = y[1] * down, y2 = y[2] * down, y3 = y[3] * down;
        const uint32_t b0 = tc::f32x2_to_e4m3x2(y0, y1);
        const uint32_t b1 = tc::f32x2_to_e4m3x2(y2, y3);
        const uint32_t v0 = tc::e4m3x2_to_f16x2(b0), v1 = tc::e4m3x2_to_f16x2(b1);
        const uint32_t r0 = tc::f32x2_to_e4m3x2(y0 - tc::f16_lo_to_f32(v0), y1 - tc::f16_hi_to_f32(v0));
        const uint32_t r1 = tc::f32x2_to_e4m3x2(y2 - tc::f16_lo_to_f32(v1), y3 - tc::f16_hi_to_f32(v1));
        w1[i / 2] = b0 | (b1 << 16);
        w2[i / 2] = r0 | (r1 << 16);
      }
      const int ch = c / 128, sub = (c % 128) / 16;
      const int off = ch * (NH * 128) + h * 128 + 16 * (sub ^ (h & 7));
      *reinterpret_cast<uint4*>(dst + C::QS_E4M3 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
      *reinterpret_cast<uint4*>(dst + C::QS_E4M3 + C::QW_BYTES + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
    }
  }
}

// ---------------------------------------------------------------- K block scales
// The block-scaled MMA of a global tile reads row m's E4M3 scales of K step k
// from TMEM lane m, column COL_SFA + 4k + m/32.  Thread m of warps 12-15 stages
// the scale words of its token (row m) of the CTA's next global tile in shared
// memory (cp.async, issued a tile ahead) and stores them into TMEM once the MMAs
// of the global tile before it are complete - which the softmax learns from that
// tile's S.  The cursor walks the CTA's global tiles in order (a row's window
// tile has no block scales).
struct SfCursor {
  int g, j, jend;        // query row, tile, end of the row's global tiles in range
  int b, n_glob;         // the row's sequence and global length
  bool live;
};

__device__ __forceinline__ void sf_settle(const AttnArgs& a, const int* tile_start, long long x1, SfCursor& c) {
  while (c.live && c.j >= c.jend) {
    ++c.g;
    if (c.g >= a.n_groups || tile_start[c.g] >= x1) {
      c.live = false;
      break;
    }
    const int nt = tile_start[c.g + 1] - tile_start[c.g] - ROW_END;
    c.j = 0;
    c.jend = (int)min((long long)(nt - 1), x1 - tile_start[c.g]);
    int nw;
    const uint8_t *wk, *wv;
    unit_extent(a, c.g, &c.b, &c.n_glob, &nw, &wk, &wv);
  }
}

__device__ __forceinline__ SfCursor sf_first(const AttnArgs& a, const int* tile_start, long long x0, long long x1, int g0) {
  SfCursor c;
  const int nt = tile_start[g0 + 1] - tile_start[g0] - ROW_END;
  c.g = g0;
  c.j = (int)(x0 - tile_start[g0]);
  c.jend = (int)min((long long)(nt - 1), x1 - tile_start[g0]);
  c.live = x0 < x1;
  int nw;
  const uint8_t *wk, *wv;
  unit_extent(a, g0, &c.b, &c.n_glob, &nw, &wk, &wv);
  sf_settle(a, tile_start, x1, c);
  return c;
}

// row m's scale words of the cursor's tile -> shared memory (zero past the end)
template <int D>
__device__ __forceinline__ void sf_stage(const AttnArgs& a, const SfCursor& c, int m, uint32_t dst) {
  using C = Cfg<D>;
  const int pos = TILE * c.j + m;
  if (pos < c.n_glob) {
    int pid = a.page_table[(size_t)c.b * a.max_pages + (pos >> 6)];
    if (pid < 0 || pid >= a.cache.num_pages) pid = 0;      // the K producer reports it
    const uint8_t* sp = a.cache.k_scale + (size_t)pid * C::PAGE_SCALE + (pos & 63) * 8;
#pragma unroll
    for (int q = 0; q < C::KS / 2; ++q) tc::cp_async8(dst + 8 * q, sp + q * (PKV_PAGE * 8));
  } else {
#pragma unroll
    for (int k = 0; k < C::KS; ++k) tc::sts32(dst + 4 * k, 0u);
  }
  tc::cp_async_commit();
}

// the staged words -> TMEM: only the column the lane quarter's rows are read from
template <int D>
__device__ __forceinline__ void sf_store(uint32_t taddr, uint32_t src) {
  using C = Cfg<D>;
  tc::cp_async_wait_all();
#pragma unroll
  for (int k = 0; k < C::KS; ++k) tc::tmem_st1(taddr + 4 * k, tc::lds32(src + 4 * k));
  tc::tc_wait_st();
}

// ---------------------------------------------------------------- the kernel
template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) attn_tc_kernel(AttnArgs a, const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap vmap,
                                                              const int* __restrict__ tile_start,
                                                              float* __restrict__ part_o,
                                                              float* __restrict__ part_lse) {
  using C = Cfg<D>;
  extern __shared__ uint8_t dyn_raw[];
  uint8_t* dyn = (uint8_t*)(((uintptr_t)dyn_raw + 1023) & ~(uintptr_t)1023);
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int G = gridDim.x, cta = blockIdx.x;
  const long long lim = a.wait_limit;

  if (tid == 0) {
    for (int i = 0; i < NKS; ++i) {
      tc::mbar_init(&sh.kr_full[i], 1);
      tc::mbar_init(&sh.kr_empty[i], 1);
    }
    for (int i = 0; i < NVR; ++i) {
      tc::mbar_init(&sh.vr_full[i], 1);
      tc::mbar_init(&sh.vr_empty[i], NGRP);
    }
    tc::mbar_init(&sh.sfa_full, 4);
    for (int i = 0; i < NVS; ++i) tc::mbar_init(&sh.vfull[i], NGRP);
    for (int i = 0; i < NVG; ++i) tc::mbar_init(&sh.vempty[i], 1);
    tc::mbar_init(&sh.s_full, 1);
    tc::mbar_init(&sh.s_empty, 8);
    tc::mbar_init(&sh.p_full[0], 8);
    tc::mbar_init(&sh.p_full[1], 8);
    tc::mbar_init(&sh.p_empty[0], 1);
    tc::mbar_init(&sh.p_empty[1], 1);
    tc::mbar_init(&sh.q_full, 1);
    tc::mbar_init(&sh.q_empty, 1);
    tc::mbar_init(&sh.o_empty, 8);
    tc::mbar_init(&sh.drain, 1);
    tc::mbar_init(&sh.drain2, 1);
    sh.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == W_QK) {
    tc::tmem_alloc(&sh.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;
  // the set-up above may overlap the end of the query split; from here on the
  // plan, the query terms and the cache it saw are read
  pkv::dep_wait();
  pkv::dep_trigger();
  const long long T = tile_start[a.n_groups];
  const long long x0 = cta_start(T, G, cta), x1 = cta_start(T, G, cta + 1);
  const int g0 = tile_start[a.n_groups + 1 + cta];     // query row of tile x0 (from the plan)

  volatile int* abort_p = &sh.abort_flag;

  uint8_t* sQ = dyn + C::OFF_Q;
  uint8_t* sP = dyn + C::OFF_P;
  uint8_t* sK = dyn + C::OFF_K;
  uint8_t* sV = dyn + C::OFF_V;
  const size_t pdb = (size_t)C::PAGE_DATA, psb = (size_t)C::PAGE_SCALE;

  if (x0 < x1) {
    // ======================================================== K tile producer
    // Tile j of a row: its two pages, each column block of a page one 1-D bulk
    // copy into the tile slot ([column block][128 rows][RB]: rows 0-63 the first
    // page, 64-127 the second); the window tile: its E4M3 K rows by TMA, 128
    // channels (one 16 KB chunk, 128-byte swizzle) per copy.
    if (warp == W_KPROD) {
      int kt = 0;               // slot uses issued
      int skipped = -1;         // copy left out by the testing hook
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g] - ROW_END;   // tiles of the row
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        const int npr = (u.n_glob + PKV_PAGE - 1) / PKV_PAGE;       // pages of the row
        int pbase = -1, pl = -1;            // lane i holds page id pbase + i of the row
        for (int j = j0; j < j1 && ok; ++j) {
          const bool win = (j == nt - 1);
          if (!win) {
            const int p0 = 2 * j, npg = (TILE * j + PKV_PAGE < u.n_glob) ? 2 : 1;
            if (pbase < 0 || p0 + 1 >= pbase + 32) {
              pbase = p0;
              pl = (pbase + lane < npr) ? a.page_table[(size_t)u.b * a.max_pages + pbase + lane] : -1;
            }
            const int pid0 = __shfl_sync(0xffffffffu, pl, p0 - pbase);
            const int pid1 = __shfl_sync(0xffffffffu, pl, p0 + 1 - pbase);
            const int slot = kt % NKS, use = kt / NKS;
            if (lane == 0 && !tc::mbar_wait(&sh.kr_empty[slot], (use & 1) ^ 1, abort_p, lim)) {
              fail(sh, a.err);
              ok = false;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) {
              if (a.hook_skip_copy == kt && cta == 0) {
                skipped = kt;
              } else {
                if (lane == 0) tc::mbar_arrive_expect_tx(&sh.kr_full[slot], (uint32_t)(npg * C::PAGE_DATA));
                __syncwarp();
                // one lane per (page, column block): the tile's copies leave in one instruction
                if (lane < npg * C::NCB) {
                  const int p = lane / C::NCB, cb = lane % C::NCB;
                  int pid = p ? pid1 : pid0;
                  if (pid < 0 || pid >= a.cache.num_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); pid = 0; }
                  tc::bulk_g2s(sK + slot * C::KSLOT + cb * (TILE * C::RB) + p * (PKV_PAGE * C::RB),
                               a.cache.k_data + (size_t)pid * pdb + cb * (PKV_PAGE * C::RB),
                               (uint32_t)(PKV_PAGE * C::RB), &sh.kr_full[slot]);
                }
              }
            }
            ++kt;
          } else {
            for (int s = 0; s < C::NWS && ok; ++s) {
              if (lane == 0) {
                const int slot = kt % NKS, use = kt / NKS;
                if (!tc::mbar_wait(&sh.kr_empty[slot], (use & 1) ^ 1, abort_p, lim)) { fail(sh, a.err); ok = false; }
                if (ok) {
                  const int c0 = s * C::CPS, nc = min(C::CPS, C::NWC - c0);
                  tc::mbar_arrive_expect_tx(&sh.kr_full[slot], (uint32_t)(nc * WCHUNK));
                  for (int c = 0; c < nc; ++c)
                    tc::tma_load_2d(sK + slot * C::KSLOT + c * WCHUNK, &wmap, (c0 + c) * 128, u.b * PKV_WINDOW,
                                    &sh.kr_full[slot]);
                }
              }
              ok = __shfl_sync(0xffffffffu, ok, 0);
              ++kt;
            }
          }
        }
        x = min((long long)tile_start[g + 1], x1);
        ++g;
      }
      // drain: every copy issued must have landed before this CTA may exit
      // (the last use of each slot; earlier uses were waited for by the MMA warp)
      if (lane == 0)
        for (int k = (kt > NKS ? kt - NKS : 0); k < kt; ++k)
          if (k != skipped && !tc::mbar_drain(&sh.kr_full[k % NKS], (k / NKS) & 1, lim)) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    // ======================================================== V page producer
    // For every global tile, every 128-channel chunk c, both pages: chunk c of the
    // page (4 KB of codes, contiguous in the V layout) and its 512 bytes of block
    // scales into one ring slot, in the order the dequantizers consume them.
    else if (warp == W_VPROD) {
      int vi = 0;     // ring slots issued
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g] - ROW_END;   // tiles of the row
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        const int npr = (u.n_glob + PKV_PAGE - 1) / PKV_PAGE;
        int pbase = -1, pl = -1;            // lane i holds page id pbase + i of the row
        for (int j = j0; j < j1 && j < nt - 1 && ok; ++j) {
          const int p0 = 2 * j, npg = (TILE * j + PKV_PAGE < u.n_glob) ? 2 : 1;
          if (pbase < 0 || p0 + 1 >= pbase + 32) {
            pbase = p0;
            pl = (pbase + lane < npr) ? a.page_table[(size_t)u.b * a.max_pages + pbase + lane] : -1;
          }
          const int pid0 = __shfl_sync(0xffffffffu, pl, p0 - pbase);
          const int pid1 = __shfl_sync(0xffffffffu, pl, p0 + 1 - pbase);
          // the tile's chunk-pages (chunk c of page p is number c * npg + p) in groups
          // of VGRP: lane i waits for the ring slot of chunk-page k + i and issues its
          // two copies, so the copies of a group leave in one warp instruction
          const int n = C::NVCH * npg;
          for (int k = 0; k < n && ok; k += VGRP) {
            const int ni = min(VGRP, n - k);
            const int cp = k + lane, c = cp / npg, p = cp % npg;
            const int slot = (vi + lane) % NVR, use = (vi + lane) / NVR;
            bool w_ok = true;
            if (lane < ni) w_ok = tc::mbar_wait(&sh.vr_empty[slot], (use & 1) ^ 1, abort_p, lim);
            if (!__all_sync(0xffffffffu, w_ok)) {
              if (lane == 0) fail(sh, a.err);
              ok = false;
              break;
            }
            if (lane < ni) {
              int pid = p ? pid1 : pid0;
              if (pid < 0 || pid >= a.cache.num_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); pid = 0; }
              tc::mbar_arrive_expect_tx(&sh.vr_full[slot], VSLOT);
              uint8_t* dst = sV + slot * VSLOT;
              tc::bulk_g2s(dst, a.cache.v_data + (size_t)pid * pdb + c * VCODES, VCODES, &sh.vr_full[slot]);
              tc::bulk_g2s(dst + VCODES, a.cache.v_scale + (size_t)pid * psb + c * VSCALES, VSCALES, &sh.vr_full[slot]);
            }
            vi += ni;
          }
        }
        // the window tile: NVCH x WVQ chunks of WVROWS entries x 128 channels (E4M3),
        // one ring slot each, by TMA in the same groups of VGRP
        if (ok && j0 < j1 && j1 == nt) {
          const int n = C::NVCH * WVQ;
          for (int k = 0; k < n && ok; k += VGRP) {
            const int ni = min(VGRP, n - k);
            const int cq = k + lane, c = cq / WVQ, q = cq % WVQ;
            const int slot = (vi + lane) % NVR, use = (vi + lane) / NVR;
            bool w_ok = true;
            if (lane < ni) w_ok = tc::mbar_wait(&sh.vr_empty[slot], (use & 1) ^ 1, abort_p, lim);
            if (!__all_sync(0xffffffffu, w_ok)) {
              if (lane == 0) fail(sh, a.err);
              ok = false;
              break;
            }
            if (lane < ni) {
              tc::mbar_arrive_expect_tx(&sh.vr_full[slot], WVROWS * 128);
              tc::tma_load_2d(sV + slot * VSLOT, &vmap, 128 * c, u.b * PKV_WINDOW + WVROWS * q, &sh.vr_full[slot]);
            }
            vi += ni;
          }
        }
        x = min((long long)tile_start[g + 1], x1);
        ++g;
      }
      if (lane == 0)
        for (int k = (vi > NVR ? vi - NVR : 0); k < vi; ++k)
          if (!tc::mbar_drain(&sh.vr_full[k % NVR], (k / NVR) & 1, lim)) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    // ======================================================== QK MMA issuer
    // Global tile: NQT x KS block-scaled FP4 MMAs (M128 N64 K64) into S; window
    // tile: 2 terms x D/32 FP8 MMAs (M128 N64 K32).  The whole warp runs the
    // schedule and one elected lane issues (operands stay warp-uniform).
    else if (warp == W_QK) {
      const uint32_t idq = tc::idesc_nvf4(128, NH), idw = tc::idesc_e4m3(128, NH);
      const uint32_t sk = tc::smem_u32(sK), sq = tc::smem_u32(sQ);
      const uint64_t dK = tc::sdesc_kmajor(sk, C::RB), dQ = tc::sdesc_kmajor(sq, C::RB);
      const uint64_t dKw = tc::sdesc_kmajor(sk, 128), dQw = tc::sdesc_kmajor(sq, 128);
      int kt = 0, gt = 0, nq = 0, iq = 0;
      bool q_landed = true;      // the last query copy issued has been seen complete
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int nt = tile_start[g + 1] - tile_start[g] - ROW_END;   // tiles of the row
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        for (int j = j0; j < j1 && ok; ++j) {
          const bool win = (j == nt - 1);
          // the query form this tile reads (FP4 terms from the row's first global
          // tile in range on, E4M3 terms for the window tile), copied from the
          // rows split ahead once the previous form's MMAs are complete
          if (win || j == j0) {
            if (iq > 0) ok = tc::mbar_wait(&sh.q_empty, (iq - 1) & 1, abort_p, lim);
            if (!ok) break;
            const uint32_t nb = win ? 2 * C::QW_BYTES : NQT * C::QT_BYTES;
            const uint8_t* src = a.qs + (size_t)g * C::QS_ROW + (win ? C::QS_E4M3 : 0);
            if (lane == 0) tc::mbar_arrive_expect_tx(&sh.q_full, nb);
            __syncwarp();
            if (lane < 16) tc::bulk_g2s(sQ + lane * (nb / 16), src + lane * (nb / 16), nb / 16, &sh.q_full);
            ok = tc::mbar_wait(&sh.q_full, iq & 1, abort_p, lim);
            ++iq;
            q_landed = ok;
          }
          // S free (the previous tile copied out by the softmax)
          ok = ok && tc::mbar_wait(&sh.s_empty, (nq & 1) ^ 1, abort_p, lim);
          if (!win) {
            const int slot = kt % NKS;
            ok = ok && tc::mbar_wait(&sh.kr_full[slot], (kt / NKS) & 1, abort_p, lim);
            ok = ok && tc::mbar_wait(&sh.sfa_full, gt & 1, abort_p, lim);
            tc::compiler_fence();          // issue strictly after the waits
            if (!ok) break;
            tc::tc_fence_after();
            if (tc::elect_one()) {
              // the tile's K codes into TMEM (read from shared memory once: the
              // contraction then reads only the query terms from shared memory);
              // the slot is released as soon as the copies are done
#pragma unroll
              for (int k = 0; k < C::KS; ++k) {
                const int cb = (32 * k) / C::RB, kk = (32 * k) % C::RB;
                tc::tmem_cp_128x256b(tbase + COL_KA + 8 * k,
                                     dK + (uint64_t)((slot * C::KSLOT + cb * TILE * C::RB + kk) >> 4));
              }
              tc::mma_commit(&sh.kr_empty[slot]);
#pragma unroll 1
              for (int t = 0; t < NQT; ++t) {
#pragma unroll
                for (int k = 0; k < C::KS; ++k) {
                  const int cb = (32 * k) / C::RB, kk = (32 * k) % C::RB;
                  const uint64_t bd = dQ + (uint64_t)((t * C::QT_BYTES + cb * NH * C::RB + kk) >> 4);
                  tc::mma_nvf4_ts(tbase + COL_S, tbase + COL_KA + 8 * k, bd, idq, tbase + COL_SFA + 4 * k,
                                  tbase + COL_SFB + 4 * t, (t | k) != 0);
                }
              }
              tc::mma_commit(&sh.s_full);
              // the row's last global tile in range: its FP4 query terms are free
              if (j == min(j1, nt - 1) - 1) tc::mma_commit(&sh.q_empty);
            }
            __syncwarp();
            ++kt;
            ++gt;
          } else {
            for (int s = 0; s < C::NWS && ok; ++s) {
              const int slot = kt % NKS;
              ok = ok && tc::mbar_wait(&sh.kr_full[slot], (kt / NKS) & 1, abort_p, lim);
              tc::compiler_fence();
              if (!ok) break;
              tc::tc_fence_after();
              if (tc::elect_one()) {
                const int c0 = s * C::CPS, nc = min(C::CPS, C::NWC - c0);
                for (int c = 0; c < nc; ++c)
#pragma unroll
                  for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                      const uint64_t ad = dKw + (uint64_t)((slot * C::KSLOT + c * WCHUNK + 32 * kk) >> 4);
                      const uint64_t bd = dQw + (uint64_t)((t * C::QW_BYTES + (c0 + c) * NH * 128 + 32 * kk) >> 4);
                      tc::mma_f8_ss(tbase + COL_S, ad, bd, idw, !(s == 0 && c == 0 && t == 0 && kk == 0));
                    }
                tc::mma_commit(&sh.kr_empty[slot]);
                if (s == C::NWS - 1) {
                  tc::mma_commit(&sh.s_full);
                  tc::mma_commit(&sh.q_empty);       // the E4M3 query terms are free
                }
              }
              __syncwarp();
              ++kt;
            }
          }
          ++nq;
        }
        x = min((long long)tile_start[g + 1], x1);
        ++g;
      }
      if (!ok && lane == 0) fail(sh, a.err);
      // a query copy whose wait gave up must still land before the CTA exits
      if (!q_landed && lane == 0 && !tc::mbar_drain(&sh.q_full, (iq - 1) & 1, lim)) report(a.err, PKV_DEVERR_TIMEOUT);
      // drain outstanding MMAs before TMEM is freed
      if (tc::elect_one()) tc::mma_commit(&sh.drain);
      __syncwarp();
      if (!tc::mbar_drain(&sh.drain, 0, lim) && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    // ======================================================== PV MMA issuer
    // Per V chunk (128 channels x the 64 tokens of one page): O^T[chunk] += V^T P,
    // 4 MMAs (M128 N64 K16); chunk i of the CTA comes from dequant group i % 2
    // in TMEM slot i % NVS.
    else if (warp == W_PV) {
      const uint32_t idV = tc::idesc_f16(128, NH, false, true);    // B = P, MN-major
      const uint64_t dp0 = tc::sdesc_sw128(tc::smem_u32(sP), 8192, 1024);
      int ci = 0, np = 0, ip = 0;   // chunks consumed, P tiles consumed, rows done
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g] - ROW_END;   // tiles of the row
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        // O of the previous item read out by the epilogue (a row whose part of the
        // range is planning units only is no item)
        if (j0 < j1) {
          ok = tc::mbar_wait(&sh.o_empty, (ip & 1) ^ 1, abort_p, lim);
          ++ip;
        }
        for (int j = j0; j < j1 && ok; ++j) {
          ok = tc::mbar_wait(&sh.p_full[np & 1], (np >> 1) & 1, abort_p, lim);
          const uint64_t bpn = dp0 + (uint64_t)(((np & 1) * C::P_BYTES) >> 4);
          // global tile: chunk k = 128 channels (k / halves) x the 64 tokens of page
          // half k % halves, 4 MMAs; window tile: 128 channels (k / WVQ) x WVROWS
          // entries, WVROWS / 16 MMAs
          const bool win = (j == nt - 1);
          const int halves = (TILE * j + PKV_PAGE < u.n_glob) ? 2 : 1;
          const int nk = win ? C::NVCH * WVQ : C::NVCH * halves;
          const int nmma = win ? WVROWS / 16 : 4;
          for (int k = 0; k < nk && ok; ++k) {
            const int slot = ci % NVS;
            const int c = win ? k / WVQ : k >> (halves - 1);                     // halves is 1 or 2
            const int t0 = win ? WVROWS * (k % WVQ) : 64 * (k & (halves - 1));   // the chunk's first token
            ok = tc::mbar_wait(&sh.vfull[slot], (ci / NVS) & 1, abort_p, lim);
            tc::compiler_fence();
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t dO = tbase + COL_O + 64 * c, aV = tbase + COL_V + 32 * slot;
            const uint64_t bp = bpn + (uint64_t)(((t0 / 8) * 1024) >> 4);       // P rows: 8 tokens per 1 KB
            if (tc::elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                if (kk < nmma)
                  tc::mma_ts(dO, aV + 8 * kk, bp + (uint64_t)(kk * (2048 >> 4)), idV, !(j == j0 && t0 == 0 && kk == 0));
              tc::mma_commit(&sh.vempty[ci % NVG]);
              if (k == nk - 1) tc::mma_commit(&sh.p_empty[np & 1]);
            }
            __syncwarp();
            ++ci;
          }
          ++np;
        }
        x = min((long long)tile_start[g + 1], x1);
        ++g;
      }
      if (!ok && lane == 0) fail(sh, a.err);
      if (tc::elect_one()) tc::mma_commit(&sh.drain2);
      __syncwarp();
      if (!tc::mbar_drain(&sh.drain2, 0, lim) && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    // ======================================================== V dequantizer (thread = channel)
    // NVG groups of four warps (one warp per TMEM lane quarter) take the chunks of
    // the tiles in turn: chunk k of a tile is 128 channels (k / halves) x the 64
    // tokens of page half (k % halves), one V ring slot; group vg takes the chunk
    // numbers i (counted over the CTA's tiles) with i % NVG == vg, into the
    // 32-column TMEM slot i % NVS once the P.V of chunk i - NVS is complete
    // (barrier (i - NVS) % NVG: with one barrier per group, a group waits at most
    // one phase ahead - its previous chunk's wait saw the phase before).  Each warp converts the E4M3 block scales it needs once per chunk
    // (two per lane) and shares them through shared memory; the ring slot is
    // released as soon as its codes are read.
    else if (warp >= W_VDEQ && warp < W_VDEQ + 4 * NVG) {
      const int vw = warp - W_VDEQ;                  // 0 .. 4 NVG - 1
      const int dl = 32 * (vw & 3) + lane;           // channel lane 0..127 within a chunk
      const int vg = vw >> 2;                        // group: chunks i with i % NVG == vg
      const uint32_t lb = lane_base(warp);
      const uint32_t vsc_s = tc::smem_u32(sh.vsc[vw]);
      const uint32_t sv0 = tc::smem_u32(sV);
      int vbase = 0;            // ring slots of the tiles before this one
      int ci0 = 0;              // chunks of all groups before this tile
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g] - ROW_END;   // tiles of the row
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        for (int j = j0; j < j1 && ok; ++j) {
          const bool win = (j == nt - 1);
          const int halves = (TILE * j + PKV_PAGE < u.n_glob) ? 2 : 1;
          const int nvalid = win ? u.n_win : min(TILE, u.n_glob - TILE * j);
          // global tile: NVCH x halves chunks of 64 tokens; window tile: NVCH x WVQ
          // chunks of WVROWS entries; one ring slot each
          const int nk = win ? C::NVCH * WVQ : C::NVCH * halves;
          // this group's chunks of the tile: numbers ci = ci0 + k with ci % NVG == vg
#pragma unroll 1
          for (int k = (vg + NVG - ci0 % NVG) % NVG; k < nk && ok; k += NVG) {
            const int ci = ci0 + k;
            const int ri = vbase + k, rs = ri % NVR;
            const int vs = ci % NVS, pc = ci - NVS;
            if (win) {
              // WVROWS entries x this lane's channel of the ring slot (row-major
              // [entry][128 channels] E4M3), pairs of entries -> f16x2
              const bool w_ok = tc::mbar_wait(&sh.vr_full[rs], (ri / NVR) & 1, abort_p, lim);
              if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
              const uint32_t wb = sv0 + rs * VSLOT + dl;
              uint32_t r[WVROWS / 2];
#pragma unroll
              for (int i = 0; i < WVROWS / 2; ++i)
                r[i] = tc::e4m3x2_to_f16x2(tc::lds8(wb + 256 * i) | (tc::lds8(wb + 256 * i + 128) << 8));
              tc::reg_fence16(r);
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.vr_empty[rs]);
              // entries beyond the window's count are zero
              const int t0 = WVROWS * (k % WVQ);
              if (t0 + WVROWS > nvalid) {
#pragma unroll
                for (int i = 0; i < WVROWS / 2; ++i) {
                  const int tt = t0 + 2 * i;
                  if (tt >= nvalid) r[i] = 0u;
                  else if (tt + 1 >= nvalid) r[i] &= 0xFFFFu;
                }
              }
              tc::reg_fence16(r);
              const bool s_ok = pc < 0 || tc::mbar_wait(&sh.vempty[pc % NVG], (pc / NVG) & 1, abort_p, lim);
              if (!__all_sync(0xffffffffu, s_ok)) { fail(sh, a.err); ok = false; break; }
              tc::tc_fence_after();
              tc::tmem_st16(tbase + lb + COL_V + 32 * vs, r);
              tc::tc_wait_st();
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.vfull[vs]);
              continue;
            }
            const int h = k & (halves - 1);           // page half (halves is 1 or 2)
            uint32_t r[32];
            {
              const bool w_ok = tc::mbar_wait(&sh.vr_full[rs], (ri / NVR) & 1, abort_p, lim);
              if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
              const uint32_t base = sv0 + rs * VSLOT;
              // block scales of this warp's two channel blocks x 64 tokens: lane
              // converts token pairs (lane & 15) and 16 + (lane & 15) of block (lane >> 4)
              const uint32_t sb = base + VCODES + (2 * (vw & 3) + (lane >> 4)) * PKV_PAGE + 2 * (lane & 15);
              const uint32_t s2a = tc::e4m3x2_to_f16x2(tc::lds16(sb));
              const uint32_t s2b = tc::e4m3x2_to_f16x2(tc::lds16(sb + 32));
              __syncwarp();                            // previous readers of vsc are done
              tc::sts32(vsc_s + 4 * (lane >> 4) * 32 + 4 * (lane & 15), s2a);
              tc::sts32(vsc_s + 4 * (lane >> 4) * 32 + 64 + 4 * (lane & 15), s2b);
              __syncwarp();
              const uint32_t sp = vsc_s + 128 * (lane >> 4);   // this channel's block: 32 pairs
              const uint32_t wd = base + 4 * dl;               // word (octet o, channel dl): o*512 + 4*dl
#pragma unroll
              for (int o = 0; o < 8; ++o) {              // octet o of the page: tokens 8o .. 8o+7
                const uint32_t w = tc::lds32(wd + 512 * o);
                const uint4 s4 = tc::lds128(sp + 16 * o);
                const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
                uint32_t e[4];
                tc::e2m1x8_to_f16x2x4(w, e);
#pragma unroll
                for (int i = 0; i < 4; ++i) r[4 * o + i] = tc::hmul2(e[i], sv[i]);
              }
              tc::reg_fence32(r);                      // the slot's codes are in registers: release it
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.vr_empty[rs]);
            }
            // zero the tokens beyond the valid count
            const int t0 = 64 * h;
            if (t0 + 64 > nvalid) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int tt = t0 + 2 * i;
                if (tt >= nvalid) r[i] = 0u;
                else if (tt + 1 >= nvalid) r[i] &= 0xFFFFu;
              }
            }
            tc::reg_fence32(r);             // conversion done before the (blocking) slot wait
            // the PV of the chunk NVS before this one has read the TMEM slot
            const bool s_ok = pc < 0 || tc::mbar_wait(&sh.vempty[pc % NVG], (pc / NVG) & 1, abort_p, lim);
            if (!__all_sync(0xffffffffu, s_ok)) { fail(sh, a.err); ok = false; break; }
            tc::tc_fence_after();
            tc::tmem_st32(tbase + lb + COL_V + 32 * vs, r);
            tc::tc_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sh.vfull[vs]);
          }
          ci0 += nk;
          vbase += nk;
        }
        x = min((long long)tile_start[g + 1], x1);
        ++g;
      }
    }
    // ======================================================== softmax + epilogue
    else if (warp >= W_SMAX && warp < W_SMAX + 8) {
      const int st = tid - 32 * W_SMAX;         // 0..255
      const int hh = (warp - W_SMAX) >> 2;      // head half: heads 32*hh .. 32*hh+31
      const int q4 = warp & 3;                  // TMEM lane quarter
      const int t = 32 * q4 + lane;             // token lane (S) / channel lane (O)
      const uint32_t lb = lane_base(warp);
      const float ratio = a.tw_v / a.cache.ts_v;
      const uint32_t m_s = tc::smem_u32(sh.m);
      // the partial results stay in L2 for the merge that follows (the K/V stream
      // would evict them otherwise)
      const uint64_t pol = tc::l2_evict_last();
      // warps 12-15: the query terms' constant B-side block scales, then the K
      // block scales of the CTA's first global tile (staged and stored at once)
      // and, staged a tile ahead, those of each next one
      const bool sfw = hh == 0;
      const uint32_t sf_t = tbase + lb + COL_SFA + q4;     // this quarter's column of K step 0
      const uint32_t sf_s = tc::smem_u32(sh.sfs[t]);
      SfCursor sfc{};
      if (sfw) {
        sfc = sf_first(a, tile_start, x0, x1, g0);
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = i < 4 * NQT ? term_scale_code(i / 4) * 0x01010101u : 0u;
        tc::tmem_st32(tbase + lb + COL_SFB, r);
        tc::tc_wait_st();
        if (sfc.live) {
          sf_stage<D>(a, sfc, t, sf_s);
          sf_store<D>(sf_t, sf_s);
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sh.sfa_full);
          ++sfc.j;
          sf_settle(a, tile_start, x1, sfc);
          if (sfc.live) sf_stage<D>(a, sfc, t, sf_s);
        }
      }
      int ntile = 0;
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g] - ROW_END;   // tiles of the row
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        if (j0 >= j1) {                     // planning units only: no item
          x = min((long long)tile_start[g + 1], x1);
          ++g;
          continue;
        }
        // the running max and the logit factors of the row's two query forms
        // (split ahead, in global memory); every thread passed the previous
        // row's closing barrier, so nobody reads the old ones any more
        if (st < NH) {
          const float* zr = reinterpret_cast<const float*>(a.qs + (size_t)g * C::QS_ROW);
          sh.m[st] = -INFINITY;
          sh.zsg[st] = __ldg(zr + C::QS_ZSG / 4 + st);
          sh.zsw[st] = __ldg(zr + C::QS_ZSW / 4 + st);
        }
        tc::named_bar(1, 256);
        // l of head 32*hh + 16*hq + hs over this warp's 32 tokens (both lanes of a pair hold it)
        const int hs = (lane >> 1) & 15;
        float l[2] = {0.f, 0.f};
        for (int j = j0; j < j1; ++j) {
          const bool win = (j == nt - 1);
          const int nvalid = win ? u.n_win : min(TILE, u.n_glob - TILE * j);
          const uint32_t zs_s = tc::smem_u32(win ? sh.zsw : sh.zsg);
          const float pr = win ? ratio : 1.f;
          const bool valid = t < nvalid;
          // ---- S tile ready?  Copy this token's 32 logits out of TMEM at once and
          // free S for the next tile's QK.
          bool w_ok = tc::mbar_wait(&sh.s_full, ntile & 1, abort_p, lim);
          if (tc::named_bar_or(3, 256, !w_ok)) { fail(sh, a.err); ok = false; break; }
          tc::tc_fence_after();
          float sa[32];
          {
            uint32_t r[32];
            tc::tmem_ld32(tbase + lb + COL_S + 32 * hh, r);
            tc::tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) sa[i] = __uint_as_float(r[i]);
          }
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sh.s_empty);
          // a global tile's S is complete, so are its MMAs: the next global
          // tile's K block scales may replace its own
          if (sfw && !win && sfc.live) {
            sf_store<D>(sf_t, sf_s);
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sh.sfa_full);
            ++sfc.j;
            sf_settle(a, tile_start, x1, sfc);
            if (sfc.live) sf_stage<D>(a, sfc, t, sf_s);
          }
          // two passes of 16 heads; the f16 P values of both wait in registers
          // until the P buffer is free
          const int pb = ntile & 1;
          const uint32_t prow = tc::smem_u32(sP) + pb * C::P_BYTES + (t >> 3) * 1024 + (t & 7) * 128;
          uint32_t pk2[2][8];
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            const int h0 = 32 * hh + 16 * hq;            // first head of this pass
            // logits of this token for heads h0 .. h0+15, log2 units: S * zs_h (in place)
            float* sv = sa + 16 * hq;
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const uint4 zb = tc::lds128(zs_s + 4 * (h0 + 4 * i4));
              sv[4 * i4] *= __uint_as_float(zb.x);
              sv[4 * i4 + 1] *= __uint_as_float(zb.y);
              sv[4 * i4 + 2] *= __uint_as_float(zb.z);
              sv[4 * i4 + 3] *= __uint_as_float(zb.w);
            }
            // does any logit exceed its running max by more than TAU?
            bool need = false;
            if (valid) {
#pragma unroll
              for (int i4 = 0; i4 < 4; ++i4) {
                const uint4 mb = tc::lds128(m_s + 4 * (h0 + 4 * i4));
                need |= (sv[4 * i4] - __uint_as_float(mb.x) > TAU) | (sv[4 * i4 + 1] - __uint_as_float(mb.y) > TAU) |
                        (sv[4 * i4 + 2] - __uint_as_float(mb.z) > TAU) | (sv[4 * i4 + 3] - __uint_as_float(mb.w) > TAU);
              }
            }
            if (tc::named_bar_or(2, 256, need)) {
              // tile max per head: over the 32 tokens of the warp (reduce-scatter:
              // lanes 2i, 2i+1 end with head h0 + i), then the 4 lane quarters
              {
                float mv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) mv[i] = valid ? sv[i] : -INFINITY;
                const float v = warp_max16(mv, lane);
                if ((lane & 1) == 0) sh.red[q4][h0 + hs] = v;
              }
              tc::named_bar(1, 256);
              if (q4 == 0 && lane < 16) {
                const int h = h0 + lane;
                const float tm = fmaxf(fmaxf(sh.red[0][h], sh.red[1][h]), fmaxf(sh.red[2][h], sh.red[3][h]));
                const float mo = sh.m[h];
                const float mn = fmaxf(mo, tm);
                sh.alpha[h] = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                sh.m[h] = mn;
              }
              tc::named_bar(1, 256);
              l[hq] *= sh.alpha[h0 + hs];
              if (j > j0) {
                // every P.V into O so far (tile ntile-1 and earlier) must be complete
                const int kp = ntile - 1;
                const bool pv_ok = tc::mbar_wait(&sh.p_empty[kp & 1], (kp >> 1) & 1, abort_p, lim);
                if (tc::named_bar_or(3, 256, !pv_ok)) { fail(sh, a.err); ok = false; break; }
                tc::tc_fence_after();
                // O^T columns of these 16 heads, every channel chunk, times alpha
#pragma unroll 1
                for (int c8 = 0; c8 < 2 * C::NVCH; ++c8) {
                  uint32_t o[8];
                  const int hb = h0 + 8 * (c8 & 1);
                  const uint32_t ta = tbase + lb + COL_O + 64 * (c8 >> 1) + hb;
                  tc::tmem_ld8(ta, o);
                  tc::tc_wait_ld();
#pragma unroll
                  for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * sh.alpha[hb + i]);
                  tc::tmem_st8(ta, o);
                }
                tc::tc_wait_st();
              }
            }
            // ---- P = exp2(S * zs - m) (f16); l sums the FP32 values.  The
            // arguments are <= TAU, so the approximate exp2 stays in range.
            uint32_t* pk = pk2[hq];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint4 ma = tc::lds128(m_s + 4 * (h0 + 8 * k));
              const uint4 mb = tc::lds128(m_s + 4 * (h0 + 8 * k + 4));
              const float mk[8] = {__uint_as_float(ma.x), __uint_as_float(ma.y), __uint_as_float(ma.z),
                                   __uint_as_float(ma.w), __uint_as_float(mb.x), __uint_as_float(mb.y),
                                   __uint_as_float(mb.z), __uint_as_float(mb.w)};
#pragma unroll
              for (int i2 = 0; i2 < 4; ++i2) {
                const int i = 4 * k + i2;        // head pair index within the pass
                const float p0 = ex2_approx(valid ? sv[2 * i] - mk[2 * i2] : -INFINITY);
                const float p1 = ex2_approx(valid ? sv[2 * i + 1] - mk[2 * i2 + 1] : -INFINITY);
                sv[2 * i] = p0;
                sv[2 * i + 1] = p1;
                pk[i] = f32_to_f16x2(p0 * pr, p1 * pr);
              }
            }
            l[hq] += warp_sum16(sv, lane);
          }
          if (!ok) break;
          // P buffer ntile&1 is free once the P.V of tile ntile-2 is done; both
          // passes' f16 P values wait in registers until then
          w_ok = tc::mbar_wait(&sh.p_empty[pb], ((ntile >> 1) & 1) ^ 1, abort_p, lim);
          if (tc::named_bar_or(3, 256, !w_ok)) { fail(sh, a.err); ok = false; break; }
          // row t of P (MN-major, 128-byte swizzle): heads 8c .. 8c+7 = 16-byte chunk c
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            tc::sts128(prow + 16 * ((4 * hh + 2 * hq) ^ (t & 7)), make_uint4(pk2[hq][0], pk2[hq][1], pk2[hq][2], pk2[hq][3]));
            tc::sts128(prow + 16 * ((4 * hh + 2 * hq + 1) ^ (t & 7)), make_uint4(pk2[hq][4], pk2[hq][5], pk2[hq][6], pk2[hq][7]));
          }
          tc::fence_proxy_async_smem();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sh.p_full[pb]);
          ++ntile;
        }
        if (!ok) break;
        // ---- end of the item: wait for its last P.V, then write the partial
        const int klast = ntile - 1;       // P.V of the item's last tile done -> O complete
        bool w_ok = tc::mbar_wait(&sh.p_empty[klast & 1], (klast >> 1) & 1, abort_p, lim);
        if (tc::named_bar_or(3, 256, !w_ok)) { fail(sh, a.err); ok = false; break; }
        tc::tc_fence_after();
        // l over all 128 token lanes: the four lane quarters are summed below
        if ((lane & 1) == 0) {
          sh.red[q4][32 * hh + hs] = l[0];
          sh.red[q4][32 * hh + 16 + hs] = l[1];
        }
        tc::named_bar(1, 256);
        const size_t prow_i = (size_t)cta + (size_t)g;          // partial row of this segment
        // per head: output factor ts_v / l (0 when l = 0) and the partial LSE
        if (st < NH) {
          const float lh = sh.red[0][st] + sh.red[1][st] + sh.red[2][st] + sh.red[3][st];
          sh.alpha[st] = lh > 0.f ? a.cache.ts_v / lh : 0.f;
          if (st < a.H) tc::st_f32_l2(part_lse + prow_i * a.H + st, lh > 0.f ? (sh.m[st] + log2f(lh)) * LN2 : -INFINITY, pol);
        }
        tc::named_bar(1, 256);
        float* po = part_o + prow_i * a.H * D;
        const uint32_t al_s = tc::smem_u32(sh.alpha);
#pragma unroll 1
        for (int c = 0; c < C::NVCH; ++c) {
          const int d = 128 * c + t;
#pragma unroll 1
          for (int hq = 0; hq < 2; ++hq) {
            const int hb = 32 * hh + 16 * hq;
            uint32_t o[16];
            tc::tmem_ld16(tbase + lb + COL_O + 64 * c + hb, o);
            tc::tc_wait_ld();
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const uint4 f = tc::lds128(al_s + 4 * (hb + 4 * i4));
              const float fv[4] = {__uint_as_float(f.x), __uint_as_float(f.y), __uint_as_float(f.z), __uint_as_float(f.w)};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int h = hb + 4 * i4 + i;
                if (h < a.H) tc::st_f32_l2(po + (size_t)h * D + d, __uint_as_float(o[4 * i4 + i]) * fv[i], pol);
              }
            }
          }
        }
        tc::tc_fence_before();
        tc::named_bar(1, 256);                 // sh.red / sh.m / zs reads done before the next item resets them
        if (lane == 0) tc::mbar_arrive(&sh.o_empty);
        x = min((long long)tile_start[g + 1], x1);
        ++g;
      }
      if (sfw) tc::cp_async_wait_all();      // a staging copy of a role that gave up lands before exit
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == W_QK) tc::tmem_dealloc(tbase, 512);
}

// Output side of a fused decode, applied by the merge to the final O.
struct Epilogue {
  const int32_t* rope_pos;    // NULL: no rotation
  const float* cos_sin;
  int max_pos, rope_dim;
  float out_scale;
  uint8_t* out_fp8;           // NULL: no FP8 output
  int* err;
};

// Merge the segment partials of each query row: rows cta+g for every CTA whose
// (non-empty) tile range meets g's tiles.  One block of D/4 threads per (g, h):
// warp 0 computes the LSE weights once, every thread combines one float4.
// Fused decode: the merged O is turned back by the row's rotary angles and
// encoded as E4M3 of O / out_scale.
__global__ void merge_tc_kernel(const int* __restrict__ tile_start, int n_groups, int G, int H, int D,
                                const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                float* __restrict__ out, float* __restrict__ out_lse, Epilogue ep) {
  pkv::dep_wait();
  pkv::dep_trigger();
  __shared__ float wts[1024];
  __shared__ int nseg_s, cl_s, pos_s;
  __shared__ float lse_s;
  const int g = blockIdx.x / H, h = blockIdx.x % H;
  const long long T = tile_start[n_groups];
  if (threadIdx.x < 32) {
    const long long first = tile_start[g], last = tile_start[g + 1] - 1 - ROW_END;   // the window tile
    const int c_lo = (int)(((first + 1) * G - 1) / T), c_hi = (int)(((last + 1) * G - 1) / T);
    const int n = min(c_hi - c_lo + 1, 1024);
    float m = -INFINITY;
    for (int i = threadIdx.x; i < n; i += 32) {
      const int c = c_lo + i;
      const bool live = cta_start(T, G, c) != cta_start(T, G, c + 1);
      const float ls = live ? part_lse[((size_t)c + g) * H + h] : -INFINITY;
      wts[i] = ls;
      m = fmaxf(m, ls);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
    for (int i = threadIdx.x; i < n; i += 32) {
      const float w = (m == -INFINITY || wts[i] == -INFINITY) ? 0.f : exp2f((wts[i] - m) * LOG2E);
      wts[i] = w;
      sum += w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncwarp();
    if (threadIdx.x == 0) {
      nseg_s = n;
      cl_s = c_lo;
      lse_s = m == -INFINITY ? -INFINITY : m + logf(sum);
      int p = -1;
      if (ep.rope_pos) {
        p = ep.rope_pos[g];
        if (p < 0 || p >= ep.max_pos) {
          if (h == 0) report(ep.err, PKV_DEVERR_BAD_PAGE);
          p = -1;
        }
      }
      pos_s = p;
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int i = threadIdx.x; i < n; i += 32) wts[i] *= inv;
  }
  __syncthreads();
  const int n = nseg_s, c_lo = cl_s;
  for (int d4 = threadIdx.x; d4 < D / 4; d4 += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // four segments per round, loads issued before use (segments are L2 round trips)
    for (int i0 = 0; i0 < n; i0 += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u;
        v[u] = (i < n && wts[i] != 0.f)
                   ? __ldg(reinterpret_cast<const float4*>(part_o + (((size_t)(c_lo + i) + g) * H + h) * D) + d4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float w = i0 + u < n ? wts[i0 + u] : 0.f;
        acc.x = fmaf(w, v[u].x, acc.x); acc.y = fmaf(w, v[u].y, acc.y);
        acc.z = fmaf(w, v[u].z, acc.z); acc.w = fmaf(w, v[u].w, acc.w);
      }
    }
    if (pos_s >= 0 && 4 * d4 >= D - ep.rope_dim) {
      // pairs i0, i0+1 of the rotated part: turn back by the row's angles
      const int i0 = 2 * d4 - (D - ep.rope_dim) / 2;
      const float* row = ep.cos_sin + (size_t)pos_s * ep.rope_dim;
      const float2 c = __ldg(reinterpret_cast<const float2*>(row + i0));
      const float2 sn = __ldg(reinterpret_cast<const float2*>(row + ep.rope_dim / 2 + i0));
      const float4 o = acc;
      acc.x = o.x * c.x + o.y * sn.x;
      acc.y = o.y * c.x - o.x * sn.x;
      acc.z = o.z * c.y + o.w * sn.y;
      acc.w = o.w * c.y - o.z * sn.y;
    }
    if (out) reinterpret_cast<float4*>(out + ((size_t)g * H + h) * D)[d4] = acc;
    if (ep.out_fp8) {
      const float sc = ep.out_scale;
      const uint32_t code = e4m3_code(__fdiv_rn(acc.x, sc)) | (e4m3_code(__fdiv_rn(acc.y, sc)) << 8) |
                            (e4m3_code(__fdiv_rn(acc.z, sc)) << 16) | (e4m3_code(__fdiv_rn(acc.w, sc)) << 24);
      reinterpret_cast<uint32_t*>(ep.out_fp8 + ((size_t)g * H + h) * D)[d4] = code;
    }
  }
  if (threadIdx.x == 0 && out_lse) out_lse[(size_t)g * H + h] = lse_s;
}

}  // namespace tcattn
}  // namespace pkv

// ---------------------------------------------------------------- host side
namespace {
template <int D>
cudaError_t set_attrs() {
  return cudaFuncSetAttribute(pkv::tcattn::attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              pkv::tcattn::Cfg<D>::DYN);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// tensor map of a window K buffer [rows][d] (uint8): boxes of 128 rows x 128 bytes, 128-byte swizzle
// window K (128 x 128 boxes, 128-byte swizzle: the MMA's A operand) or window V
// (128 channels x WVROWS entries, no swizzle: read byte by byte by the V warps)
cudaError_t window_map(const uint8_t* w, int d, int rows, int box_rows, bool swz, CUtensorMap* map) {
  if (!g_encode) return cudaErrorInitializationError;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d};
  const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t pkv_attn_tc_init(int) {
  cudaError_t e = set_attrs<128>();
  if (e == cudaSuccess) e = set_attrs<256>();
  if (e == cudaSuccess) e = set_attrs<512>();
  if (e == cudaSuccess && !g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn)) e = cudaErrorNotSupported;
    if (e == cudaSuccess) g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  }
  return e;
}

bool pkv_attn_tc_supported(const pkv::AttnArgs& a, int d) {
  if (a.sel) return false;
  if (d != 128 && d != 256 && d != 512) return false;
  if (a.H < 1 || a.H > pkv::tcattn::NH) return false;
  // the window's V scale is folded into P (f16): keep tw_v / ts_v within 2^+-7
  const float r = a.tw_v / a.cache.ts_v;
  if (!(r >= 1.f / 128.f && r <= 128.f)) return false;
  return true;
}

// persistent grid: one CTA per SM, or fewer when there are fewer tiles than SMs
static int tc_grid(int num_sms, int n_groups, int max_entries) {
  const long long glob = max_entries > PKV_WINDOW ? max_entries - PKV_WINDOW : 0;
  const long long tmax = (long long)n_groups * ((glob + 127) / 128 + 1);
  return (int)(tmax < num_sms ? tmax : num_sms);
}

static size_t qs_row_bytes(int D) {
  using namespace pkv::tcattn;
  return D == 128 ? Cfg<128>::QS_ROW : D == 256 ? Cfg<256>::QS_ROW : Cfg<512>::QS_ROW;
}

// [plan][partial O][partial LSE][split query rows (1024-aligned)]
size_t pkv_attn_tc_ws_bytes(int num_sms, int H, int D, int n_groups, int max_entries) {
  const size_t rows = (size_t)tc_grid(num_sms, n_groups, max_entries) + n_groups;
  const size_t plan = (size_t)(n_groups + 1 + tc_grid(num_sms, n_groups, max_entries)) * 4;
  const size_t head = (plan + 255) / 256 * 256 + rows * H * D * 4 + rows * H * 4;
  return 256 + (head + 1023) / 1024 * 1024 + (size_t)n_groups * qs_row_bytes(D) + 1024;
}

cudaError_t pkv_launch_attn_tc(pkv::AttnArgs& a, int num_sms, int max_entries, float* out, float* out_lse,
                               void* ws, cudaStream_t st, cudaEvent_t e0, cudaEvent_t e1, int* n_launches) {
  using namespace pkv::tcattn;
  uint8_t* p = (uint8_t*)ws;
  int* tile_start = (int*)p;
  const int G = tc_grid(num_sms, a.n_groups, max_entries);
  p += ((size_t)(a.n_groups + 1 + G) * 4 + 255) / 256 * 256;
  const size_t rows = (size_t)G + a.n_groups;
  float* part_o = (float*)p;
  p += rows * a.H * a.D * 4;
  float* part_lse = (float*)p;
  p += rows * a.H * 4;
  p = (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
  a.qs = p;
  CUtensorMap wmap, vmap;
  const int nseq = a.replay ? a.n_groups / PKV_WINDOW : a.n_groups;
  cudaError_t e = window_map(a.wk, a.D, nseq * PKV_WINDOW, 128, true, &wmap);
  if (e == cudaSuccess) e = window_map(a.wv, a.D, nseq * PKV_WINDOW, WVROWS, false, &vmap);
  if (e != cudaSuccess) return e;
  switch (a.D) {
    case 128: e = pkv::launch_pdl(qsplit_kernel<128>, dim3(a.n_groups + 1, 1), 256, 0, st, a, p, tile_start, G); break;
    case 256: e = pkv::launch_pdl(qsplit_kernel<256>, dim3(a.n_groups + 1, 2), 256, 0, st, a, p, tile_start, G); break;
    case 512: e = pkv::launch_pdl(qsplit_kernel<512>, dim3(a.n_groups + 1, 4), 256, 0, st, a, p, tile_start, G); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if (e0 && e1) cudaEventRecord(e0, st);
  switch (a.D) {
    case 128: e = pkv::launch_pdl(attn_tc_kernel<128>, G, NTHREADS, Cfg<128>::DYN, st, a, wmap, vmap, tile_start, part_o, part_lse); break;
    case 256: e = pkv::launch_pdl(attn_tc_kernel<256>, G, NTHREADS, Cfg<256>::DYN, st, a, wmap, vmap, tile_start, part_o, part_lse); break;
    case 512: e = pkv::launch_pdl(attn_tc_kernel<512>, G, NTHREADS, Cfg<512>::DYN, st, a, wmap, vmap, tile_start, part_o, part_lse); break;
    default: return cudaErrorInvalidValue;
  }
  if (e0 && e1) cudaEventRecord(e1, st);
  if (e != cudaSuccess) return e;
  Epilogue ep{};
  if (a.rope_dim > 0) {
    ep.rope_pos = a.rope_pos;
    ep.cos_sin = a.cos_sin;
    ep.max_pos = a.max_pos;
    ep.rope_dim = a.rope_dim;
  }
  ep.out_scale = a.out_scale;
  ep.out_fp8 = a.out_fp8;
  ep.err = a.err;
  *n_launches = 3;
  return pkv::launch_pdl(merge_tc_kernel, a.n_groups * a.H, a.D / 4, 0, st, (const int*)tile_start, a.n_groups, G,
                         a.H, a.D, (const float*)part_o, (const float*)part_lse, out, out_lse, ep);
}
