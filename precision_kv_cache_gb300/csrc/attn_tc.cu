// Tensor-core decode / replay attention over the paged NVFP4 global KV and the
// FP8 window, for sm_103a (tcgen05 MMA with TMEM operands and accumulators).
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
// Design (one persistent CTA per SM, 896 threads, warp-specialized):
//   * work = 128-token tiles; each query row has ceil(L/128) NVFP4 tiles plus
//     one window tile; the concatenated tile list is cut into one contiguous
//     range per CTA (balanced to one tile).
//   * warps 24 (K) and 26 (V) stream the raw pages of each tile (codes +
//     scales) into two shared-memory page rings with 1-D bulk copies (TMA).
//   * warps 0-7 (thread = token) dequantize K to f16 (exact: E2M1 x E4M3 has
//     <= 6 significant bits) into TMEM, 64 channels at a time: the A operand
//     of S^T = K Q^T  (M = 128 tokens, N = 64 heads, K = d).  Two groups of
//     four warps (one per TMEM lane quarter) take alternate chunks.
//   * warps 8-15 (thread = channel) dequantize V^T to f16 into TMEM, 128
//     channels x 64 tokens at a time: the A operand of O^T = V^T P (M = 128
//     channels, N = 64 heads, K = tokens); two groups of four warps take
//     alternate chunks.  Each warp converts the E4M3 block scales of its
//     chunk once (two per lane) and shares them through shared memory.
//   * warp 25 issues the QK MMAs, warp 27 the PV MMAs (Q and P are the
//     shared-memory B operands).
//   * warps 16-23 run the online softmax on S (FP32, exp2, lazy max update
//     with threshold 2^8), write P (f16, shared memory) and finally normalize
//     O and write the partial result.
//   * fused decode ("MegaAttention avec KV compressé NVFP4": query RoPE,
//     attention, inverse RoPE on the output, FP8 output in one pass): the Q
//     load turns the rotary pairs of each query before its f16 rounding, and
//     the merge turns the final O back and encodes it as E4M3 - no extra
//     kernel and no extra pass over O.
// Every wait is bounded; on a timeout the CTA sets the error word, stops all
// roles, drains its own copies / MMAs and frees its TMEM before returning.
#include <cstddef>
#include "attn_tc.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace tcattn {

constexpr int TILE = 128;
constexpr int NH = 64;                 // MMA N: query heads (zero-padded)
constexpr int NTHREADS = 896;       // 28 warps
// warp roles
constexpr int W_KDEQ = 0;              // 8 warps: K dequantizers
constexpr int W_VDEQ = 8;              // 8 warps: V dequantizers
constexpr int W_SMAX = 16;             // 8 warps: softmax + epilogue
constexpr int W_KPROD = 24;            // K page producer
constexpr int W_MMA = 25;              // QK MMA issuer, TMEM owner
constexpr int W_VPROD = 26;            // V page producer
constexpr int W_MMA2 = 27;             // PV MMA issuer
constexpr uint32_t NDEQ = 8;           // arrivals per K (V) page release: one per dequant warp
constexpr uint32_t NGRP = 4;           // arrivals per K (V) chunk: one per warp of a group
constexpr float TAU = 8.f;             // lazy rescale threshold (log2 units)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// TMEM columns (512 allocated)
constexpr int NKS = 3;                 // K chunk slots
constexpr int NVS = 3;                 // V chunk slots
constexpr uint32_t COL_S = 0;          // S^T tile: 64 columns (fp32); the softmax copies it out at once
constexpr uint32_t COL_K = 64;         // K chunk slots: NKS x 32 columns (64 channels, f16 pairs)
constexpr uint32_t COL_V = 160;        // V^T chunk slots: NVS x 32 columns (64 tokens, f16 pairs)
constexpr uint32_t COL_O = 256;        // O^T: 4 chunks x 64 columns
static_assert(COL_K == COL_S + 64 && COL_V == COL_K + 32 * NKS && COL_O >= COL_V + 32 * NVS, "TMEM map");

constexpr int NKR = 4;                 // K ring: page slots (a tile holds two for its whole duration)
constexpr int NVR = 3;                 // V ring: page slots (released page by page)

template <int D>
struct Cfg {
  static constexpr int PAGE_DATA = PKV_PAGE * D / 2;
  static constexpr int PAGE_SCALE = PKV_PAGE * D / 16;
  static constexpr int PSLOT = PAGE_DATA + PAGE_SCALE;            // one page of K (or V): codes + scales
  static constexpr int Q_BYTES = NH * D * 2;
  static constexpr int P_BYTES = TILE * NH * 2;
  static constexpr int NKCH = D / 64;                             // K chunks of 64 channels
  static constexpr int NVCH = D / 128;                            // V chunks of 128 channels
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = OFF_Q + Q_BYTES;                   // 2 P buffers
  static constexpr int OFF_K = OFF_P + 2 * P_BYTES;               // K ring
  static constexpr int OFF_V = OFF_K + NKR * PSLOT;               // V ring
  static constexpr int DYN = OFF_V + NVR * PSLOT + 1024;          // + alignment slack
  static_assert(OFF_K % 1024 == 0, "operand tiles stay 1024-aligned");
};

struct Shared {
  uint64_t kr_full[NKR], kr_empty[NKR], vr_full[NVR], vr_empty[NVR];
  uint64_t kfull[NKS], kempty[NKS], vfull[NVS], vempty[NVS];
  uint64_t s_full, s_empty, p_full[2], p_empty[2], q_full, o_empty, drain, drain2;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float m[NH];     // running max per head (log2 units)
  float alpha[NH];             // rescale factor of the current tile
  float red[4][NH];            // cross-warp reductions
  alignas(16) uint32_t vsc[8][64];   // per V warp: f16x2 block-scale pairs of its current chunk (2 blocks x 32)
};
static_assert(offsetof(Shared, m) % 16 == 0 && offsetof(Shared, alpha) % 16 == 0 && offsetof(Shared, vsc) % 16 == 0,
              "16-byte shared-memory vector accesses");

// ---------------------------------------------------------------- schedule
struct Sched {
  const int* tile_start;       // [n_groups + 1]
  int n_groups, G;
  long long T;
};

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

// ---------------------------------------------------------------- plan kernel
// tile_start[g] = sum over g' < g of (ceil(n_glob(g')/128) + 1); tile_start[n] = total;
// then tile_start[n + 1 + c] = the query row where CTA c (of G) starts.
__global__ void __launch_bounds__(1024) plan_kernel(AttnArgs a, int* tile_start, int G) {
  __shared__ int wsum[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.n_groups; base += 1024) {
    const int g = base + threadIdx.x;
    int n = 0;
    if (g < a.n_groups) {
      int b, ng, nw;
      const uint8_t *wk, *wv;
      unit_extent(a, g, &b, &ng, &nw, &wk, &wv);
      n = (ng + TILE - 1) / TILE + 1;
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
    if (threadIdx.x == 1023) carry = pre + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_start[a.n_groups] = carry;
  __syncthreads();
  const long long T = carry;
  for (int c = threadIdx.x; c < G; c += 1024) tile_start[a.n_groups + 1 + c] = group_of(tile_start, a.n_groups, cta_start(T, G, c));
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
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
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

// Q of query row g -> shared memory: f16 (from bf16; exact for |q| in [2^-14, 65504]),
// K-major with the 128-byte swizzle, heads >= H zero.  Called by the 256 softmax threads.
// Fused decode: the pairs (2i, 2i+1) of the last rope_dim channels are first turned
// by the row's rotary angles (FP32, then rounded to f16).
template <int D>
__device__ __noinline__ void load_q(const AttnArgs& a, int g, uint8_t* sQ, int st) {
  constexpr int NV = NH * D / 8 / 256;                // 16-byte vectors per thread
  constexpr int NB = 4;                               // loads in flight per thread
  static_assert(NV % NB == 0, "Q vectors per thread");
  static_assert(256 % (D / 8) == 0, "a thread sees the same 8 channels in every vector");
  const uint16_t* qg = a.q + (size_t)g * a.H * D;
  const uint32_t sq = tc::smem_u32(sQ);
  // rotary factors of this thread's 4 channel pairs (if they lie in the rotated part)
  bool rot = false;
  float4 cr = make_float4(1.f, 1.f, 1.f, 1.f), sr = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.rope_dim > 0 && 8 * (st % (D / 8)) >= D - a.rope_dim) {
    const int p = a.rope_pos[g];
    if (p >= 0 && p < a.max_pos) {
      const int i0 = 4 * (st % (D / 8)) - (D - a.rope_dim) / 2;
      const float* row = a.cos_sin + (size_t)p * a.rope_dim;
      cr = __ldg(reinterpret_cast<const float4*>(row + i0));
      sr = __ldg(reinterpret_cast<const float4*>(row + a.rope_dim / 2 + i0));
      rot = true;
    } else {
      report(a.err, PKV_DEVERR_BAD_PAGE);
    }
  }
#pragma unroll 1
  for (int b0 = 0; b0 < NV; b0 += NB) {
    uint4 in[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int v = st + 256 * (b0 + k);
      const int h = v / (D / 8), c8 = v % (D / 8);    // 8 channels per vector
      in[k] = h < a.H ? __ldg(reinterpret_cast<const uint4*>(qg + (size_t)h * D + 8 * c8)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int v = st + 256 * (b0 + k);
      const int h = v / (D / 8), c8 = v % (D / 8);
      const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
      uint32_t r[4];
      if (rot) {
        const float c[4] = {cr.x, cr.y, cr.z, cr.w}, sn[4] = {sr.x, sr.y, sr.z, sr.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xFFFF0000u);
          r[i] = f32_to_f16x2(x0 * c[i] - x1 * sn[i], x0 * sn[i] + x1 * c[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          r[i] = f32_to_f16x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
      }
      const int atom = c8 >> 3, ch = c8 & 7;
      tc::sts128(sq + atom * (NH * 128) + h * 128 + 16 * (ch ^ (h & 7)), make_uint4(r[0], r[1], r[2], r[3]));
    }
  }
  tc::fence_proxy_async_smem();
}

// ---------------------------------------------------------------- the kernel
template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) attn_tc_kernel(AttnArgs a, const int* __restrict__ tile_start,
                                                              float* __restrict__ part_o,
                                                              float* __restrict__ part_lse) {
  using C = Cfg<D>;
  extern __shared__ uint8_t dyn_raw[];
  uint8_t* dyn = (uint8_t*)(((uintptr_t)dyn_raw + 1023) & ~(uintptr_t)1023);
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int G = gridDim.x, cta = blockIdx.x;
  const long long T = tile_start[a.n_groups];
  const long long x0 = cta_start(T, G, cta), x1 = cta_start(T, G, cta + 1);
  const int g0 = tile_start[a.n_groups + 1 + cta];     // query row of tile x0 (from the plan)

  if (tid == 0) {
    for (int i = 0; i < NKR; ++i) {
      tc::mbar_init(&sh.kr_full[i], 1);
      tc::mbar_init(&sh.kr_empty[i], NDEQ);
    }
    for (int i = 0; i < NVR; ++i) {
      tc::mbar_init(&sh.vr_full[i], 1);
      tc::mbar_init(&sh.vr_empty[i], NDEQ);
    }
    for (int i = 0; i < NKS; ++i) {
      tc::mbar_init(&sh.kfull[i], NGRP);
      tc::mbar_init(&sh.kempty[i], 1);
    }
    for (int i = 0; i < NVS; ++i) {
      tc::mbar_init(&sh.vfull[i], NGRP);
      tc::mbar_init(&sh.vempty[i], 1);
    }
    tc::mbar_init(&sh.s_full, 1);
    tc::mbar_init(&sh.s_empty, 8);
    tc::mbar_init(&sh.p_full[0], 8);
    tc::mbar_init(&sh.p_full[1], 8);
    tc::mbar_init(&sh.p_empty[0], 1);
    tc::mbar_init(&sh.p_empty[1], 1);
    tc::mbar_init(&sh.q_full, 8);
    tc::mbar_init(&sh.o_empty, 8);
    tc::mbar_init(&sh.drain, 1);
    tc::mbar_init(&sh.drain2, 1);
    sh.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == W_MMA) {
    tc::tmem_alloc(&sh.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;

  volatile int* abort_p = &sh.abort_flag;

  uint8_t* sQ = dyn + C::OFF_Q;
  uint8_t* sP = dyn + C::OFF_P;
  uint8_t* sK = dyn + C::OFF_K;
  uint8_t* sV = dyn + C::OFF_V;
  const size_t pdb = (size_t)C::PAGE_DATA, psb = (size_t)C::PAGE_SCALE;

  if (x0 < x1) {
    // ======================================================== producers
    // one warp streams K pages (codes + scales) into the K ring, another V pages
    // into the V ring, one page per slot, with 1-D bulk copies.
    if (warp == W_KPROD || warp == W_VPROD) {
      // The whole warp walks the pages; page-table entries are read 32 at a time
      // (one per lane, coalesced) and lane 0 issues the copies.
      const bool isK = (warp == W_KPROD);
      const int nslot = isK ? NKR : NVR;
      uint64_t* fullb = isK ? sh.kr_full : sh.vr_full;
      uint64_t* emptyb = isK ? sh.kr_empty : sh.vr_empty;
      uint8_t* ring = isK ? sK : sV;
      const uint8_t* gdata = isK ? a.cache.k_data : a.cache.v_data;
      const uint8_t* gscale = isK ? a.cache.k_scale : a.cache.v_scale;
      int pi = 0;     // pages issued
      bool ok = true;
      long long x = x0;
      int g = g0;
      const uint8_t* last_win = nullptr;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        if (lane == 0) {
          // the next query row's Q (loaded by the softmax at this row's end): warm L2
          if (isK && j0 == 0 && x1 > tile_start[g + 1] && g + 1 < a.n_groups && ((uintptr_t)a.q & 15u) == 0)
            tc::bulk_prefetch_l2(a.q + (size_t)(g + 1) * a.H * D, (uint32_t)(a.H * D * 2));
          // the window tile (last of the row) is read from global memory by the
          // dequant warps: warm L2 with it while the paged tiles stream
          if (isK && j1 == nt && u.wk != last_win && (((uintptr_t)u.wk | (uintptr_t)u.wv) & 15u) == 0) {
            tc::bulk_prefetch_l2(u.wk, (uint32_t)(PKV_WINDOW * D));    // window buffers are [B][128][d]
            tc::bulk_prefetch_l2(u.wv, (uint32_t)(PKV_WINDOW * D));
            last_win = u.wk;
          }
        }
        // pages [2*j0, pend) of the row: those of its NVFP4 tiles in this CTA's range
        const int jp = min(j1, nt - 1);
        const int pend = min(2 * jp, (u.n_glob + PKV_PAGE - 1) / PKV_PAGE);
        for (int pb = 2 * j0; pb < pend && ok; pb += 32) {
          int pl = -1;
          if (pb + lane < pend) pl = a.page_table[(size_t)u.b * a.max_pages + pb + lane];
          const int cnt = min(32, pend - pb);
          for (int q = 0; q < cnt; ++q) {
            int p = __shfl_sync(0xffffffffu, pl, q);
            if (lane == 0) {
              if (p < 0 || p >= a.cache.num_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); p = 0; }
              const int slot = pi % nslot, use = pi / nslot;
              if (!tc::mbar_wait(&emptyb[slot], (use & 1) ^ 1, abort_p)) { fail(sh, a.err); ok = false; }
              if (ok) {
                tc::mbar_arrive_expect_tx(&fullb[slot], C::PSLOT);
                uint8_t* dst = ring + slot * C::PSLOT;
                tc::bulk_g2s(dst, gdata + (size_t)p * pdb, C::PAGE_DATA, &fullb[slot]);
                tc::bulk_g2s(dst + C::PAGE_DATA, gscale + (size_t)p * psb, C::PAGE_SCALE, &fullb[slot]);
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ++pi;
          }
        }
        x = tile_start[g] + j1;
        ++g;
      }
      // drain: every copy issued must have landed before this CTA may exit
      // (the last use of each slot; earlier uses were waited for by the consumers)
      if (lane == 0)
        for (int k = (pi > nslot ? pi - nslot : 0); k < pi; ++k)
          if (!tc::mbar_drain(&fullb[k % nslot], (k / nslot) & 1)) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    // ======================================================== MMA issuers
    // One warp issues S^T = K Q^T (per 64-channel K chunk: 4 MMAs), another
    // O^T += V^T P (per 128-channel x 64-token V chunk: 4 MMAs), each in the
    // fixed order of its inputs with blocking waits.  The whole warp runs the
    // schedule and one elected lane issues (operands stay warp-uniform).
    else if (warp == W_MMA) {
      const uint32_t idK = tc::idesc_f16(128, NH, false, false);   // B = Q, K-major
      // descriptor base; the start-address field (bits 0-13, address >> 4) is advanced by addition
      const uint64_t dq0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);
      int ks = 0, nq = 0, iq = 0;
      uint32_t kph = 0;          // K slot ring: slot, phase
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int j1 = (int)min((long long)(tile_start[g + 1] - tile_start[g]), x1 - tile_start[g]);
        // Q of this item in shared memory
        ok = tc::mbar_wait(&sh.q_full, iq & 1, abort_p);
        ++iq;
        for (int j = (int)(x - tile_start[g]); j < j1 && ok; ++j) {
          // S free (the previous tile copied out by the softmax)
          ok = tc::mbar_wait(&sh.s_empty, (nq & 1) ^ 1, abort_p);
          const uint32_t dS = tbase + COL_S;
          for (int c = 0; c < C::NKCH && ok; ++c) {
            const int slot = ks;
            ok = tc::mbar_wait(&sh.kfull[slot], kph, abort_p);
            tc::compiler_fence();          // issue strictly after the wait (measured: large effect)
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t aK = tbase + COL_K + 32 * slot;
            const uint64_t bq = dq0 + (uint64_t)(c * (NH * 128 / 16));
            if (tc::elect_one()) {
#pragma unroll
              for (int k = 0; k < 4; ++k) tc::mma_ts(dS, aK + 8 * k, bq + 2 * k, idK, (c | k) != 0);
              tc::mma_commit(&sh.kempty[slot]);
              if (c == C::NKCH - 1) tc::mma_commit(&sh.s_full);
            }
            __syncwarp();
            if (++ks == NKS) { ks = 0; kph ^= 1; }
          }
          ++nq;
        }
        x = tile_start[g] + j1;
        ++g;
      }
      if (!ok && lane == 0) fail(sh, a.err);
      // drain outstanding MMAs before TMEM is freed
      if (tc::elect_one()) tc::mma_commit(&sh.drain);
      __syncwarp();
      if (!tc::mbar_drain(&sh.drain, 0) && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    else if (warp == W_MMA2) {
      const uint32_t idV = tc::idesc_f16(128, NH, false, true);    // B = P, MN-major
      const uint64_t dp0 = tc::sdesc_sw128(tc::smem_u32(sP), 8192, 1024);
      int vs = 0, np = 0, ip = 0;
      uint32_t vph = 0;          // V slot ring: slot, phase
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)(tile_start[g + 1] - tile_start[g]), x1 - tile_start[g]);
        // O of the previous item read out by the epilogue
        ok = tc::mbar_wait(&sh.o_empty, (ip & 1) ^ 1, abort_p);
        ++ip;
        for (int j = j0; j < j1 && ok; ++j) {
          ok = tc::mbar_wait(&sh.p_full[np & 1], (np >> 1) & 1, abort_p);
          const uint64_t bpn = dp0 + (uint64_t)(((np & 1) * C::P_BYTES) >> 4);
          // chunk order: page half 0 for every channel chunk, then page half 1
          for (int cp = 0; cp < 2 * C::NVCH && ok; ++cp) {
            const int slot = vs, half = cp / C::NVCH, c = cp % C::NVCH;
            ok = tc::mbar_wait(&sh.vfull[slot], vph, abort_p);
            tc::compiler_fence();
            if (!ok) break;
            tc::tc_fence_after();
            const uint32_t dO = tbase + COL_O + 64 * c, aV = tbase + COL_V + 32 * slot;
            const uint64_t bp = bpn + (uint64_t)((half * 8192) >> 4);
            if (tc::elect_one()) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc::mma_ts(dO, aV + 8 * k, bp + (uint64_t)(k * (2048 >> 4)), idV, !(j == j0 && half == 0 && k == 0));
              tc::mma_commit(&sh.vempty[slot]);
              if (cp == 2 * C::NVCH - 1) tc::mma_commit(&sh.p_empty[np & 1]);
            }
            __syncwarp();
            if (++vs == NVS) { vs = 0; vph ^= 1; }
          }
          ++np;
        }
        x = tile_start[g] + j1;
        ++g;
      }
      if (!ok && lane == 0) fail(sh, a.err);
      if (tc::elect_one()) tc::mma_commit(&sh.drain2);
      __syncwarp();
      if (!tc::mbar_drain(&sh.drain2, 0) && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    }
    // ======================================================== K dequantizer (thread = token)
    // Two groups of four warps (one warp per TMEM lane quarter); group kg
    // converts the 64-channel chunks c = kg, kg+2, ... of every tile, a full
    // 32-column slot per chunk.  Chunks are numbered across tiles and use the
    // slot ring in order; a group advances two chunks at a time.
    else if (warp < W_VDEQ) {
      const int t = 32 * (warp & 3) + lane;          // token lane 0..127
      const int kg = (warp - W_KDEQ) >> 2;           // chunk parity of this group
      const uint32_t lb = lane_base(warp);
      int kp = 0;               // pages consumed
      int ks = kg;              // slot of this group's next chunk (chunk number kg, kg+2, ...)
      uint32_t kph = 0;         // its phase
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        for (int j = j0; j < j1 && ok; ++j) {
          const bool win = (j == nt - 1);
          int npg = 0;
          bool valid;
          const uint8_t* row = nullptr;
          uint32_t srow_s = 0, ssc_s = 0;     // shared addresses: token row, its scale bytes
          int slot = 0;
          if (!win) {
            npg = (TILE * j + PKV_PAGE < u.n_glob) ? 2 : 1;
            bool w_ok = true;
            for (int q = 0; q < npg; ++q)
              w_ok = w_ok && tc::mbar_wait(&sh.kr_full[(kp + q) % NKR], ((kp + q) / NKR) & 1, abort_p);
            if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
            valid = (TILE * j + t) < u.n_glob;
            const uint32_t page = tc::smem_u32(sK) + ((kp + (t >> 6)) % NKR) * C::PSLOT;
            slot = t & 63;
            srow_s = page + slot * (D / 2);
            ssc_s = page + C::PAGE_DATA + slot * 8;
          } else {
            valid = t < u.n_win;
            row = u.wk + (size_t)t * D;
          }
#pragma unroll 1
          for (int c = kg; c < C::NKCH; c += 2) {
            uint32_t r[32];
            if (!valid) {
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = 0u;
            } else if (!win) {
              constexpr int SW = (D / 32 < 8 ? D / 32 : 8) - 1;
              // channels 64c .. 64c+63: two 16-byte pieces, four scale blocks
              const uint4 v0 = tc::lds128(srow_s + 16 * ((2 * c) ^ (slot & SW)));
              const uint4 v1 = tc::lds128(srow_s + 16 * ((2 * c + 1) ^ (slot & SW)));
              const uint32_t sc = tc::lds32(ssc_s + (c >> 1) * (PKV_PAGE * 8) + 4 * (c & 1));
              const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
              uint32_t s4[2];                            // f16 scales: (s0, s1), (s2, s3)
              tc::e4m3x4_to_f16x2x2(sc, s4);
#pragma unroll
              for (int q = 0; q < 8; ++q) {              // word q: channels 8q .. 8q+7 of the chunk (block q/2)
                uint32_t e[4];
                tc::e2m1x8_to_f16x2x4(w[q], e);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  r[4 * q + i] = (q & 2) ? tc::hmul2_hi(e[i], s4[q >> 2]) : tc::hmul2_lo(e[i], s4[q >> 2]);
              }
            } else {
              const uint4* p4 = reinterpret_cast<const uint4*>(row + 64 * c);
#pragma unroll
              for (int h4 = 0; h4 < 4; ++h4) {
                const uint4 v = __ldg(p4 + h4);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) tc::e4m3x4_to_f16x2x2(w[i], &r[8 * h4 + 2 * i]);
              }
            }
            tc::reg_fence32(r);               // conversion done before the (blocking) slot wait
            const bool w_ok = tc::mbar_wait(&sh.kempty[ks], kph ^ 1, abort_p);
            if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
            tc::tmem_st32(tbase + lb + COL_K + 32 * ks, r);
            tc::tc_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sh.kfull[ks]);
            ks += 2;
            if (ks >= NKS) { ks -= NKS; kph ^= 1; }
          }
          if (!ok) break;
          if (!win) {
            __syncwarp();
            if (lane == 0)
              for (int q = 0; q < npg; ++q) tc::mbar_arrive(&sh.kr_empty[(kp + q) % NKR]);
            kp += npg;
          }
        }
        x = tile_start[g] + j1;
        ++g;
      }
    }
    // ======================================================== V dequantizer (thread = channel)
    // Two groups of four warps (one warp per TMEM lane quarter); the V^T chunks
    // of a tile (128 channels x 64 tokens) are taken page-major - every channel
    // chunk of page half 0, then of half 1 - and group vg converts the chunks of
    // parity vg, a full 32-column slot each.  Each warp converts the E4M3 block
    // scales it needs once (two per lane) and shares them through shared memory.
    else if (warp < W_SMAX) {
      const int vw = warp - W_VDEQ;                  // 0..7
      const int dl = 32 * (vw & 3) + lane;           // channel lane 0..127 within a chunk
      const int vg = vw >> 2;                        // chunk parity of this group
      const uint32_t lb = lane_base(warp);
      const uint32_t vsc_s = tc::smem_u32(sh.vsc[vw]);
      int vp = 0;               // pages consumed
      int vs = vg;              // slot of this group's next chunk
      uint32_t vph = 0;         // its phase
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        for (int j = j0; j < j1 && ok; ++j) {
          const bool win = (j == nt - 1);
          const int npg = win ? 0 : ((TILE * j + PKV_PAGE < u.n_glob) ? 2 : 1);
          const int nvalid = win ? u.n_win : min(TILE, u.n_glob - TILE * j);
#pragma unroll 1
          for (int half = 0; half < 2 && ok; ++half) {       // tokens 64*half .. 64*half+63
            const bool paged = half < npg;
            if (paged) {
              const bool w_ok = tc::mbar_wait(&sh.vr_full[(vp + half) % NVR], ((vp + half) / NVR) & 1, abort_p);
              if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
            }
            const uint32_t base = tc::smem_u32(sV) + ((vp + half) % NVR) * C::PSLOT;
            // chunk cp = half * NVCH + c belongs to group cp & 1
#pragma unroll 1
            for (int c = (vg ^ (half * C::NVCH)) & 1; c < C::NVCH; c += 2) {
              const int d = 128 * c + dl;
              uint32_t r[32];
              if (paged) {
                // block scales of this warp's two channel blocks x 64 tokens: lane
                // converts token pairs (lane & 15) and 16 + (lane & 15) of block (lane >> 4)
                const int blk = ((128 * c + 32 * (vw & 3)) >> 4) + (lane >> 4);
                const uint32_t sb = base + C::PAGE_DATA + blk * PKV_PAGE + 2 * (lane & 15);
                const uint32_t s2a = tc::e4m3x2_to_f16x2(tc::lds16(sb));
                const uint32_t s2b = tc::e4m3x2_to_f16x2(tc::lds16(sb + 32));
                __syncwarp();                            // previous readers of vsc are done
                tc::sts32(vsc_s + 4 * (lane >> 4) * 32 + 4 * (lane & 15), s2a);
                tc::sts32(vsc_s + 4 * (lane >> 4) * 32 + 64 + 4 * (lane & 15), s2b);
                __syncwarp();
                const uint32_t sp = vsc_s + 128 * (lane >> 4);   // this channel's block: 32 pairs
                const uint32_t wd = base + 4 * d;
#pragma unroll
                for (int o = 0; o < 8; ++o) {              // octet o of the page: tokens 8o .. 8o+7
                  const uint32_t w = tc::lds32(wd + 4 * o * D);
                  const uint4 s4 = tc::lds128(sp + 16 * o);
                  const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
                  uint32_t e[4];
                  tc::e2m1x8_to_f16x2x4(w, e);
#pragma unroll
                  for (int i = 0; i < 4; ++i) r[4 * o + i] = tc::hmul2(e[i], sv[i]);
                }
              } else if (win) {
                const uint8_t* col = u.wv + d;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const int e = 64 * half + 2 * i;
                  const uint32_t b0 = __ldg(col + (size_t)e * D), b1 = __ldg(col + (size_t)(e + 1) * D);
                  r[i] = tc::e4m3x2_to_f16x2(b0 | (b1 << 8));
                }
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = 0u;      // second page absent: no valid token
              }
              // zero the tokens beyond the valid count (their K rows are zero too)
              const int t0 = 64 * half;
              if (t0 + 64 > nvalid) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const int tt = t0 + 2 * i;
                  if (tt >= nvalid) r[i] = 0u;
                  else if (tt + 1 >= nvalid) r[i] &= 0xFFFFu;
                }
              }
              tc::reg_fence32(r);             // conversion done before the (blocking) slot wait
              const bool w_ok = tc::mbar_wait(&sh.vempty[vs], vph ^ 1, abort_p);
              if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
              tc::tmem_st32(tbase + lb + COL_V + 32 * vs, r);
              tc::tc_wait_st();
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.vfull[vs]);
              vs += 2;
              if (vs >= NVS) { vs -= NVS; vph ^= 1; }
            }
            if (!ok) break;
            if (paged) {
              // every code of this page this warp needs is in TMEM now: release it
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.vr_empty[(vp + half) % NVR]);
            }
          }
          if (!ok) break;
          vp += npg;
        }
        x = tile_start[g] + j1;
        ++g;
      }
    }
    // ======================================================== softmax + epilogue
    else if (warp < W_KPROD) {
      const int st = tid - 32 * W_SMAX;         // 0..255
      const int hh = (warp - W_SMAX) >> 2;      // head half: heads 32*hh .. 32*hh+31
      const int q4 = warp & 3;                  // TMEM lane quarter
      const int t = 32 * q4 + lane;             // token lane (S) / channel lane (O)
      const uint32_t lb = lane_base(warp);
      const float ratio = a.tw_v / a.cache.ts_v;
      const uint32_t m_s = tc::smem_u32(sh.m);
      int ntile = 0;
      bool ok = true;
      long long x = x0;
      int g = g0;
      load_q<D>(a, g, sQ, st);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh.q_full);
      while (x < x1 && ok) {
        const Unit u = unit_of(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        const long long xn = tile_start[g] + j1;
        if (st < NH) sh.m[st] = -INFINITY;
        tc::named_bar(1, 256);
        // l of head 32*hh + 16*hq + hs over this warp's 32 tokens (both lanes of a pair hold it)
        const int hs = (lane >> 1) & 15;
        float l[2] = {0.f, 0.f};
        for (int j = j0; j < j1; ++j) {
          const bool win = (j == nt - 1);
          const int nvalid = win ? u.n_win : min(TILE, u.n_glob - TILE * j);
          const float zs = a.scale * (win ? a.tw_k : a.cache.ts_k) * LOG2E;
          const float pr = win ? ratio : 1.f;
          const bool valid = t < nvalid;
          // ---- S tile ready?  Copy this token's 32 logits out of TMEM at once and
          // free S for the next tile's QK.
          bool w_ok = tc::mbar_wait(&sh.s_full, ntile & 1, abort_p);
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
          // P buffer ntile&1 is free once the P.V of tile ntile-2 is done
          const int pb = ntile & 1;
          w_ok = tc::mbar_wait(&sh.p_empty[pb], ((ntile >> 1) & 1) ^ 1, abort_p);
          if (tc::named_bar_or(3, 256, !w_ok)) { fail(sh, a.err); ok = false; break; }
          const uint32_t prow = tc::smem_u32(sP) + pb * C::P_BYTES + (t >> 3) * 1024 + (t & 7) * 128;
          // two passes of 16 heads (keeps 16 logits live instead of 32)
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            const int h0 = 32 * hh + 16 * hq;            // first head of this pass
            // raw S^T of this token for heads h0 .. h0+15 (scaled below: d = S * zs - m)
            float sv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[i] = sa[16 * hq + i];
            // does any logit exceed its running max by more than TAU?
            bool need = false;
            if (valid) {
#pragma unroll
              for (int i4 = 0; i4 < 4; ++i4) {
                const uint4 mb = tc::lds128(m_s + 4 * (h0 + 4 * i4));
                need |= (fmaf(sv[4 * i4], zs, -__uint_as_float(mb.x)) > TAU) |
                        (fmaf(sv[4 * i4 + 1], zs, -__uint_as_float(mb.y)) > TAU) |
                        (fmaf(sv[4 * i4 + 2], zs, -__uint_as_float(mb.z)) > TAU) |
                        (fmaf(sv[4 * i4 + 3], zs, -__uint_as_float(mb.w)) > TAU);
              }
            }
            if (tc::named_bar_or(2, 256, need)) {
              // tile max per head: over the 32 tokens of the warp, then the 4 lane quarters
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float v = valid ? sv[i] * zs : -INFINITY;
#pragma unroll
                for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                if (lane == 0) sh.red[q4][h0 + i] = v;
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
                const bool pv_ok = tc::mbar_wait(&sh.p_empty[kp & 1], (kp >> 1) & 1, abort_p);
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
            // ---- P = exp2(S * zs - m) (f16): row t of P (MN-major, 128-byte swizzle),
            // heads h0 .. h0+15 = two 16-byte chunks; l sums the FP32 values.  The
            // arguments are <= TAU, so the approximate exp2 stays in range.
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint32_t pk[4];
              const uint4 ma = tc::lds128(m_s + 4 * (h0 + 8 * k));
              const uint4 mb = tc::lds128(m_s + 4 * (h0 + 8 * k + 4));
              const float mk[8] = {__uint_as_float(ma.x), __uint_as_float(ma.y), __uint_as_float(ma.z),
                                   __uint_as_float(ma.w), __uint_as_float(mb.x), __uint_as_float(mb.y),
                                   __uint_as_float(mb.z), __uint_as_float(mb.w)};
#pragma unroll
              for (int i2 = 0; i2 < 4; ++i2) {
                const int i = 4 * k + i2;        // head pair index within the pass
                const float p0 = ex2_approx(valid ? fmaf(sv[2 * i], zs, -mk[2 * i2]) : -INFINITY);
                const float p1 = ex2_approx(valid ? fmaf(sv[2 * i + 1], zs, -mk[2 * i2 + 1]) : -INFINITY);
                sv[2 * i] = p0;
                sv[2 * i + 1] = p1;
                pk[i2] = f32_to_f16x2(p0 * pr, p1 * pr);
              }
              tc::sts128(prow + 16 * (((h0 >> 3) + k) ^ (t & 7)), make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
            l[hq] += warp_sum16(sv, lane);
          }
          if (!ok) break;
          tc::fence_proxy_async_smem();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sh.p_full[pb]);
          ++ntile;
          // all S of this item consumed: Q of the next item may replace this one
          // (done here, where few registers are live across the call)
          if (j == j1 - 1 && xn < x1) {
            load_q<D>(a, g + 1, sQ, st);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sh.q_full);
          }
        }
        if (!ok) break;
        // ---- end of the item: wait for its last P.V, then write the partial
        const int klast = ntile - 1;       // P.V of the item's last tile done -> O complete
        bool w_ok = tc::mbar_wait(&sh.p_empty[klast & 1], (klast >> 1) & 1, abort_p);
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
          if (st < a.H) part_lse[prow_i * a.H + st] = lh > 0.f ? (sh.m[st] + log2f(lh)) * LN2 : -INFINITY;
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
                if (h < a.H) po[(size_t)h * D + d] = __uint_as_float(o[4 * i4 + i]) * fv[i];
              }
            }
          }
        }
        tc::tc_fence_before();
        tc::named_bar(1, 256);                 // sh.red / sh.m reads done before the next item resets them
        if (lane == 0) tc::mbar_arrive(&sh.o_empty);
        x = xn;
        ++g;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == W_MMA) tc::tmem_dealloc(tbase, 512);
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
  __shared__ float wts[1024];
  __shared__ int nseg_s, cl_s, pos_s;
  __shared__ float lse_s;
  const int g = blockIdx.x / H, h = blockIdx.x % H;
  const long long T = tile_start[n_groups];
  if (threadIdx.x < 32) {
    const long long first = tile_start[g], last = tile_start[g + 1] - 1;
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
}  // namespace

cudaError_t pkv_attn_tc_init(int) {
  cudaError_t e = set_attrs<128>();
  if (e == cudaSuccess) e = set_attrs<256>();
  if (e == cudaSuccess) e = set_attrs<512>();
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

size_t pkv_attn_tc_ws_bytes(int num_sms, int H, int D, int n_groups, int max_entries) {
  const size_t rows = (size_t)tc_grid(num_sms, n_groups, max_entries) + n_groups;
  const size_t plan = (size_t)(n_groups + 1 + tc_grid(num_sms, n_groups, max_entries)) * 4;
  return 256 + (plan + 255) / 256 * 256 + rows * H * D * 4 + rows * H * 4 + 256;
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
  plan_kernel<<<1, 1024, 0, st>>>(a, tile_start, G);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (e0 && e1) cudaEventRecord(e0, st);
  switch (a.D) {
    case 128: attn_tc_kernel<128><<<G, NTHREADS, Cfg<128>::DYN, st>>>(a, tile_start, part_o, part_lse); break;
    case 256: attn_tc_kernel<256><<<G, NTHREADS, Cfg<256>::DYN, st>>>(a, tile_start, part_o, part_lse); break;
    case 512: attn_tc_kernel<512><<<G, NTHREADS, Cfg<512>::DYN, st>>>(a, tile_start, part_o, part_lse); break;
    default: return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
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
  merge_tc_kernel<<<a.n_groups * a.H, a.D / 4, 0, st>>>(tile_start, a.n_groups, G, a.H, a.D, part_o, part_lse,
                                                        out, out_lse, ep);
  *n_launches = 3;
  return cudaGetLastError();
}
