// Tensor-core index scoring for the sparse MQA logits ("Logits MQA creux",
// vLLM blog "Kernels"):  score_t = sum_h w_h * ReLU(q_h . k_t)  over the
// 128-channel NVFP4 index keys, for every position of every sequence.
//
// One persistent CTA per SM, 896 threads, warp-specialized:
//   * warp 0 streams the 64-token key pages into a 24-page shared-memory ring
//     (1-D bulk copies);
//   * warps 4-11 and 20-27: four groups of four (one warp per TMEM lane
//     quarter, thread = token) that take every fourth 128-token tile and
//     dequantize it to f16 into TMEM (exact: E2M1 x E4M3 has <= 6 significant
//     bits), 32 channels at a time;
//   * warp 1 issues S^T = K Q^T on tcgen05 (M = 128 tokens, N = 64 index heads,
//     K = 128; Q = the FP8 index queries, exact in f16, in shared memory), the
//     whole warp running the schedule and one elected lane issuing;
//   * warps 12-19: two groups of four that take alternate tiles, read S^T back,
//     apply ReLU, the head weights and the two tensor scales, and store one
//     FP32 score per token.
// TMEM holds 4 K tiles and 4 S^T tiles (512 columns).
#include "attn_tc.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace tcscore {

constexpr int TILE = 128;
constexpr int NH = 64;
constexpr int D = 128;
constexpr int NTHREADS = 896;                          // 28 warps
constexpr int W_PROD = 0, W_MMA = 1, W_DEQ = 4, W_EPI = 12, W_DEQ2 = 20;
constexpr int NKG = 4;                                 // key dequant groups: warps 4-7, 8-11, 20-23, 24-27
constexpr int NR = 24;                                 // key ring: page slots
constexpr int NS = 4;                                  // K / S^T tile slots in TMEM
// A ring slot's consecutive uses (pages k and k + NR: tiles NR / 2 apart) must fall to
// the same dequant group, so that a group never waits on a slot one phase too early.
static_assert((NR / 2) % NKG == 0, "ring depth in tiles must be a multiple of the dequant groups");
constexpr int PAGE_DATA = PKV_PAGE * D / 2;            // 4096
constexpr int PAGE_SCALE = PKV_PAGE * D / 16;          // 512
constexpr int PSLOT = PAGE_DATA + PAGE_SCALE;          // 4608
constexpr int Q_BYTES = NH * D * 2;                    // 16 KB
constexpr int OFF_Q = 0;
constexpr int OFF_R = OFF_Q + Q_BYTES;
constexpr int DYN = OFF_R + NR * PSLOT + 1024;
constexpr uint32_t COL_S = 0;                          // NS x 64 columns
constexpr uint32_t COL_K = 256;                        // NS x 64 columns

struct Shared {
  uint64_t r_full[NR], r_empty[NR];
  uint64_t kfull[NS], kempty[NS], s_full[NS], s_empty[NS], q_full, drain;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float w[NH];
};

struct Args {
  const uint8_t* q;          // FP8 [B][Hi][128]
  float tq;
  const float* w;            // [B][Hi]
  pkv_idx_cache ic;
  const int32_t* page_table;
  int max_pages;
  const int32_t* seq_len;
  int B, Hi, Lmax;
  float* scores;             // [B][Lmax]
  int* err;
};

__device__ __forceinline__ int seq_tokens(const Args& a, int b) {
  int L = a.seq_len[b];
  if (L > a.Lmax) { L = a.Lmax; report(a.err, PKV_DEVERR_BAD_PAGE); }
  return L < 0 ? 0 : L;
}

__device__ __forceinline__ long long cta_start(long long T, int G, int c) { return (T * c) / G; }

__device__ __forceinline__ int group_of(const int* ts, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)ts[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// tile_start[b] = sum over b' < b of ceil(L(b')/128); tile_start[B] = total;
// then tile_start[B + 1 + c] = the sequence where CTA c (of G) starts.
__global__ void __launch_bounds__(1024) plan_kernel(Args a, int* tile_start, int G) {
  pkv::dep_wait();
  pkv::dep_trigger();
  __shared__ int wsum[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.B; base += 1024) {
    const int g = base + threadIdx.x;
    const int n = g < a.B ? (seq_tokens(a, g) + TILE - 1) / TILE : 0;
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
    if (g < a.B) tile_start[g] = pre + incl - n;
    __syncthreads();
    if (threadIdx.x == 1023) carry = pre + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_start[a.B] = carry;
  __syncthreads();
  const long long T = carry;
  for (int c = threadIdx.x; c < G; c += 1024) tile_start[a.B + 1 + c] = group_of(tile_start, a.B, cta_start(T, G, c));
}

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

__device__ __forceinline__ void fail(Shared& sh, int* err) {
  sh.abort_flag = 1;
  report(err, PKV_DEVERR_TIMEOUT);
}

// FP8 index queries of sequence b -> f16, K-major 128-byte swizzle; weights -> sh.w
// (128 threads; all loads of a thread are issued before the conversions)
__device__ __noinline__ void load_q(const Args& a, int b, uint8_t* sQ, float* sw, int tid) {
  const uint8_t* qb = a.q + (size_t)b * a.Hi * D;
  const uint32_t sq = tc::smem_u32(sQ);
  constexpr int NV = NH * D / 8 / 128;                  // 8 vectors of 8 channels per thread
  uint2 in[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = tid + 128 * k, h = v / (D / 8), c8 = v % (D / 8);
    in[k] = h < a.Hi ? *reinterpret_cast<const uint2*>(qb + (size_t)h * D + 8 * c8) : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = tid + 128 * k, h = v / (D / 8), c8 = v % (D / 8);
    uint32_t o[4];
    tc::e4m3x4_to_f16x2x2(in[k].x, &o[0]);
    tc::e4m3x4_to_f16x2x2(in[k].y, &o[2]);
    const int atom = c8 >> 3, ch = c8 & 7;
    tc::sts128(sq + atom * (NH * 128) + h * 128 + 16 * (ch ^ (h & 7)), make_uint4(o[0], o[1], o[2], o[3]));
  }
  if (tid < NH) sw[tid] = tid < a.Hi ? a.w[(size_t)b * a.Hi + tid] : 0.f;
  tc::fence_proxy_async_smem();
}

__global__ void __launch_bounds__(NTHREADS, 1) score_tc_kernel(Args a, const int* __restrict__ tile_start) {
  extern __shared__ uint8_t dyn_raw[];
  uint8_t* dyn = (uint8_t*)(((uintptr_t)dyn_raw + 1023) & ~(uintptr_t)1023);
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  if (tid == 0) {
    for (int i = 0; i < NR; ++i) {
      tc::mbar_init(&sh.r_full[i], 1);
      tc::mbar_init(&sh.r_empty[i], 4);
    }
    for (int i = 0; i < NS; ++i) {
      tc::mbar_init(&sh.kfull[i], 4);
      tc::mbar_init(&sh.kempty[i], 1);
      tc::mbar_init(&sh.s_full[i], 1);
      tc::mbar_init(&sh.s_empty[i], 4);
    }
    tc::mbar_init(&sh.q_full, 4);
    tc::mbar_init(&sh.drain, 1);
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
  // the set-up above may overlap the end of the plan kernel
  pkv::dep_wait();
  pkv::dep_trigger();
  const long long T = tile_start[a.B];
  const long long x0 = cta_start(T, G, cta), x1 = cta_start(T, G, cta + 1);
  const int g0 = tile_start[a.B + 1 + cta];
  volatile int* abort_p = &sh.abort_flag;
  uint8_t* sQ = dyn + OFF_Q;
  uint8_t* ring = dyn + OFF_R;

  if (x0 < x1) {
    if (warp == W_PROD) {
      // ======================================================== producer
      // The whole warp walks the pages; each lane reads one page-table entry and
      // issues that page's copies, so copies of consecutive pages go out in parallel.
      int pi = 0;
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int L = seq_tokens(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        // pages [2*j0, pend) of sequence g
        const int pend = min(2 * j1, (L + PKV_PAGE - 1) / PKV_PAGE);
        // up to 16 pages at a time, one lane each (16 <= NR: distinct ring slots)
        for (int pb = 2 * j0; pb < pend && ok; pb += 16) {
          const int cnt = min(16, pend - pb);
          bool lok = true;
          if (lane < cnt) {
            int p = a.page_table[(size_t)g * a.max_pages + pb + lane];
            if (p < 0 || p >= a.ic.num_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); p = 0; }
            const int k = pi + lane, slot = k % NR, use = k / NR;
            if (!tc::mbar_wait(&sh.r_empty[slot], (use & 1) ^ 1, abort_p)) {
              fail(sh, a.err);
              lok = false;
            } else {
              tc::mbar_arrive_expect_tx(&sh.r_full[slot], PSLOT);
              uint8_t* dst = ring + slot * PSLOT;
              tc::bulk_g2s(dst, a.ic.data + (size_t)p * PAGE_DATA, PAGE_DATA, &sh.r_full[slot]);
              tc::bulk_g2s(dst + PAGE_DATA, a.ic.scale + (size_t)p * PAGE_SCALE, PAGE_SCALE, &sh.r_full[slot]);
            }
          }
          ok = __all_sync(0xffffffffu, lok);
          pi += cnt;
        }
        x = tile_start[g] + j1;
        ++g;
      }
      if (lane == 0)
        for (int k = (pi > NR ? pi - NR : 0); k < pi; ++k)
          if (!tc::mbar_drain(&sh.r_full[k % NR], (k / NR) & 1)) report(a.err, PKV_DEVERR_TIMEOUT);
    } else if (warp == W_MMA) {
      // ======================================================== MMA issuer (whole warp, one elected lane issues)
      const uint32_t idq = tc::idesc_f16(128, NH, false, false);
      const uint64_t dq0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);
      int s = 0, item = 0;
      uint32_t ph = 0;
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        if (j1 > j0) {
          ok = tc::mbar_wait(&sh.q_full, item & 1, abort_p);
          ++item;
        }
        for (int j = j0; j < j1 && ok; ++j) {
          ok = tc::mbar_wait(&sh.kfull[s], ph, abort_p) && tc::mbar_wait(&sh.s_empty[s], ph ^ 1, abort_p);
          tc::compiler_fence();
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t dS = tbase + COL_S + 64 * s, aK = tbase + COL_K + 64 * s;
          if (tc::elect_one()) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_ts(dS, aK + 8 * k, dq0 + (uint64_t)((k >> 2) * (NH * 128 / 16) + (k & 3) * 2), idq, k != 0);
            tc::mma_commit(&sh.kempty[s]);
            tc::mma_commit(&sh.s_full[s]);
          }
          __syncwarp();
          if (++s == NS) { s = 0; ph ^= 1; }
        }
        x = tile_start[g] + j1;
        ++g;
      }
      if (!ok && lane == 0) fail(sh, a.err);
      if (tc::elect_one()) tc::mma_commit(&sh.drain);
      __syncwarp();
      if (!tc::mbar_drain(&sh.drain, 0) && lane == 0) report(a.err, PKV_DEVERR_TIMEOUT);
    } else if ((warp >= W_DEQ && warp < W_EPI) || warp >= W_DEQ2) {
      // ======================================================== key dequantizer (thread = token)
      // group kg takes the tiles n = kg, kg + NKG, ... of this CTA (n counted from x0)
      const int t = 32 * (warp & 3) + lane;
      const int kg = warp >= W_DEQ2 ? 2 + ((warp - W_DEQ2) >> 2) : (warp - W_DEQ) >> 2;
      const uint32_t lb = lane_base(warp);
      const uint32_t ring_s = tc::smem_u32(ring);
      int pc0 = 0, n0 = 0;      // ring pages and tiles of the CTA before this row's first tile in range
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int L = seq_tokens(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        // this group's tiles of the row (tile n = n0 + j - j0 with n % NKG == kg);
        // every tile but a sequence's last has two pages
        for (int j = j0 + (kg + NKG - n0 % NKG) % NKG; j < j1 && ok; j += NKG) {
          const int n = n0 + (j - j0), pc = pc0 + 2 * (j - j0);
          const int npg = (TILE * j + PKV_PAGE < L) ? 2 : 1;
          const int s = n % NS;
          const uint32_t ph = (n / NS) & 1;
          bool w_ok = tc::mbar_wait(&sh.kempty[s], ph ^ 1, abort_p);
          for (int q = 0; q < npg; ++q)
            w_ok = w_ok && tc::mbar_wait(&sh.r_full[(pc + q) % NR], ((pc + q) / NR) & 1, abort_p);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
          const bool valid = TILE * j + t < L;
          const uint32_t page = ring_s + ((pc + (t >> 6)) % NR) * PSLOT;
          const int slot = t & 63;
          const uint32_t row = page + slot * (D / 2);
          uint32_t sc[2] = {0u, 0u};
          if (valid) {
            const uint4 sv = tc::lds128(page + PAGE_DATA + (slot & ~1) * 8);   // 8 scale bytes of this token
            sc[0] = (slot & 1) ? sv.z : sv.x;
            sc[1] = (slot & 1) ? sv.w : sv.y;
          }
#pragma unroll
          for (int qt = 0; qt < 4; ++qt) {             // channels 32*qt .. 32*qt+31
            uint32_t r[16];
            if (valid) {
              const uint4 v = tc::lds128(row + 16 * (qt ^ (slot & 3)));
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
              uint32_t s4[2];
              tc::e4m3x4_to_f16x2x2(sc[qt >> 1], s4);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t e[4];
                tc::e2m1x8_to_f16x2x4(w[q], e);
                const int qq = 4 * (qt & 1) + q;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  r[4 * q + i] = (qq & 2) ? tc::hmul2_hi(e[i], s4[qq >> 2]) : tc::hmul2_lo(e[i], s4[qq >> 2]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) r[i] = 0u;
            }
            tc::tmem_st16(tbase + lb + COL_K + 64 * s + 16 * qt, r);
          }
          tc::tc_wait_st();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            tc::mbar_arrive(&sh.kfull[s]);
            for (int q = 0; q < npg; ++q) tc::mbar_arrive(&sh.r_empty[(pc + q) % NR]);
          }
        }
        n0 += j1 - j0;
        pc0 += 2 * (j1 - j0) - ((j1 == nt && j1 > j0 && TILE * (nt - 1) + PKV_PAGE >= L) ? 1 : 0);
        x = tile_start[g] + j1;
        ++g;
      }
    } else if (warp >= W_EPI && warp < W_DEQ2) {
      // ======================================================== epilogue (thread = token)
      // group eg takes the tiles n = eg, eg+2, ... of this CTA
      const int t = 32 * (warp & 3) + lane;
      const int eg = (warp - W_EPI) >> 2;
      const uint32_t lb = lane_base(warp);
      const float sc = a.tq * a.ic.ts;
      const uint32_t w_s = tc::smem_u32(sh.w);
      int n0 = 0;               // tiles of the CTA before this row's first tile in range
      bool ok = true;
      long long x = x0;
      int g = g0;
      while (x < x1 && ok) {
        const int L = seq_tokens(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        if (j1 > j0) {
          // every S^T of the previous sequence has been read (so its MMAs are done): new Q, w
          tc::named_bar(1, 256);
          if (eg == 0) {
            load_q(a, g, sQ, sh.w, t);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sh.q_full);
          }
          tc::named_bar(1, 256);                    // sh.w of this sequence visible to both groups
        }
        // this group's tiles of the row: tile n0 + j - j0 with n % 2 == eg
        for (int j = j0 + ((eg - n0) & 1); j < j1; j += 2) {
          const int n = n0 + (j - j0);
          const int s = n % NS;
          const uint32_t ph = (n / NS) & 1;
          const bool w_ok = tc::mbar_wait(&sh.s_full[s], ph, abort_p);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
          tc::tc_fence_after();
          float acc = 0.f;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {           // heads 32 hf .. 32 hf + 31
            uint32_t r[32];
            tc::tmem_ld32(tbase + lb + COL_S + 64 * s + 32 * hf, r);
            tc::tc_wait_ld();
            if (hf == 1) {
              tc::tc_fence_before();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.s_empty[s]);
            }
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const uint4 wv = tc::lds128(w_s + 16 * (8 * hf + i4));
              acc = fmaf(__uint_as_float(wv.x), fmaxf(__uint_as_float(r[4 * i4]), 0.f), acc);
              acc = fmaf(__uint_as_float(wv.y), fmaxf(__uint_as_float(r[4 * i4 + 1]), 0.f), acc);
              acc = fmaf(__uint_as_float(wv.z), fmaxf(__uint_as_float(r[4 * i4 + 2]), 0.f), acc);
              acc = fmaf(__uint_as_float(wv.w), fmaxf(__uint_as_float(r[4 * i4 + 3]), 0.f), acc);
            }
          }
          const int tok = TILE * j + t;
          if (tok < L) a.scores[(size_t)g * a.Lmax + tok] = acc * sc;
        }
        n0 += j1 - j0;
        x = tile_start[g] + j1;
        ++g;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == W_MMA) tc::tmem_dealloc(tbase, 512);
}

}  // namespace tcscore
}  // namespace pkv

size_t pkv_score_tc_ws_bytes(int B, int num_sms) { return ((size_t)(B + 1 + num_sms) * 4 + 255) / 256 * 256; }

cudaError_t pkv_score_tc_init() {
  return cudaFuncSetAttribute(pkv::tcscore::score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              pkv::tcscore::DYN);
}

// scores[b][t] for t < seq_len[b]; ws holds the tile plan ([B+1] ints)
cudaError_t pkv_launch_score_tc(const uint8_t* q_idx, float tq, const float* w, const pkv_idx_cache& ic,
                                const int32_t* page_table, int max_pages, const int32_t* seq_len, int B, int Hi,
                                float* scores, int Lmax, void* ws, int num_sms, int* err, cudaStream_t st,
                                cudaEvent_t prof_start, cudaEvent_t prof_stop) {
  using namespace pkv::tcscore;
  Args a;
  a.q = q_idx; a.tq = tq; a.w = w; a.ic = ic; a.page_table = page_table; a.max_pages = max_pages;
  a.seq_len = seq_len; a.B = B; a.Hi = Hi; a.Lmax = Lmax; a.scores = scores; a.err = err;
  int* tile_start = (int*)ws;
  const long long tmax = (long long)B * ((Lmax + TILE - 1) / TILE);
  const int G = (int)(tmax < num_sms ? (tmax > 0 ? tmax : 1) : num_sms);
  cudaError_t e = pkv::launch_pdl(plan_kernel, 1, 1024, 0, st, a, tile_start, G);
  if (e != cudaSuccess) return e;
  if (prof_start && prof_stop) cudaEventRecord(prof_start, st);
  e = pkv::launch_pdl(score_tc_kernel, G, NTHREADS, DYN, st, a, (const int*)tile_start);
  if (prof_start && prof_stop) cudaEventRecord(prof_stop, st);
  return e;
}
