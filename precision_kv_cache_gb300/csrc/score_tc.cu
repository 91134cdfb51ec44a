// Tensor-core index scoring for the sparse MQA logits ("Logits MQA creux",
// vLLM blog "Kernels"):  score_t = sum_h w_h * ReLU(q_h . k_t)  over the
// 128-channel NVFP4 index keys, for every position of every sequence.
//
// One persistent CTA per SM, 384 threads, warp-specialized like the attention
// kernel: warp 0 streams the 64-token key pages into a shared-memory ring
// (bulk copies), warps 4-7 (thread = token) dequantize a 128-token tile to f16
// into TMEM (exact: E2M1 x E4M3), warp 1 issues S^T = K Q^T on tcgen05
// (M = 128 tokens, N = 64 index heads, K = 128; Q = the FP8 index queries,
// exact in f16, in shared memory), warps 8-11 read S^T back, apply ReLU, the
// head weights and the two tensor scales, and store one FP32 score per token.
#include "attn_tc.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace pkv {
namespace tcscore {

constexpr int TILE = 128;
constexpr int NH = 64;
constexpr int D = 128;
constexpr int NTHREADS = 384;
constexpr int NR = 6;                                  // key ring: page slots
constexpr int PAGE_DATA = PKV_PAGE * D / 2;            // 4096
constexpr int PAGE_SCALE = PKV_PAGE * D / 16;          // 512
constexpr int PSLOT = PAGE_DATA + PAGE_SCALE;          // 4608
constexpr int Q_BYTES = NH * D * 2;                    // 16 KB
constexpr int OFF_Q = 0;
constexpr int OFF_R = OFF_Q + Q_BYTES;
constexpr int DYN = OFF_R + NR * PSLOT + 1024;
constexpr uint32_t COL_S = 0;                          // 2 x 64 columns
constexpr uint32_t COL_K = 128;                        // 2 x 64 columns

struct Shared {
  uint64_t r_full[NR], r_empty[NR];
  uint64_t kfull[2], kempty[2], s_full[2], s_empty[2], q_full, drain;
  uint32_t tmem_base;
  int abort_flag;
  float w[NH];
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

__global__ void __launch_bounds__(1024) plan_kernel(Args a, int* tile_start) {
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

__device__ __forceinline__ uint32_t lane_base(int warp) { return (uint32_t)((warp & 3) * 32) << 16; }

__device__ __forceinline__ void fail(Shared& sh, int* err) {
  sh.abort_flag = 1;
  report(err, PKV_DEVERR_TIMEOUT);
}

// FP8 index queries of sequence b -> f16, K-major 128-byte swizzle; weights -> sh.w
__device__ __noinline__ void load_q(const Args& a, int b, uint8_t* sQ, float* sw, int tid) {
  const uint8_t* qb = a.q + (size_t)b * a.Hi * D;
  for (int v = tid; v < NH * D / 8; v += 128) {
    const int h = v / (D / 8), c8 = v % (D / 8);
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (h < a.Hi) {
      const uint2 in = *reinterpret_cast<const uint2*>(qb + (size_t)h * D + 8 * c8);
      o = make_uint4(tc::e4m3x2_to_f16x2(in.x & 0xFFFFu), tc::e4m3x2_to_f16x2(in.x >> 16),
                     tc::e4m3x2_to_f16x2(in.y & 0xFFFFu), tc::e4m3x2_to_f16x2(in.y >> 16));
    }
    const int atom = c8 >> 3, ch = c8 & 7;
    *reinterpret_cast<uint4*>(sQ + atom * (NH * 128) + h * 128 + 16 * (ch ^ (h & 7))) = o;
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
  const long long T = tile_start[a.B];
  const long long x0 = cta_start(T, G, cta), x1 = cta_start(T, G, cta + 1);
  if (tid == 0) {
    for (int i = 0; i < NR; ++i) {
      tc::mbar_init(&sh.r_full[i], 1);
      tc::mbar_init(&sh.r_empty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
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
  if (warp == 1) {
    tc::tmem_alloc(&sh.tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;
  volatile int* abort_p = &sh.abort_flag;
  uint8_t* sQ = dyn + OFF_Q;
  uint8_t* ring = dyn + OFF_R;

  if (x0 < x1) {
    if (warp == 0) {
      // ======================================================== producer
      if (lane == 0) {
        int pi = 0;
        bool ok = true;
        long long x = x0;
        int g = group_of(tile_start, a.B, x);
        while (x < x1 && ok) {
          const int L = seq_tokens(a, g);
          const int nt = tile_start[g + 1] - tile_start[g];
          const int j0 = (int)(x - tile_start[g]);
          const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
          for (int j = j0; j < j1 && ok; ++j) {
            const int npg = (TILE * j + PKV_PAGE < L) ? 2 : 1;
            for (int q = 0; q < npg; ++q) {
              int p = a.page_table[(size_t)g * a.max_pages + 2 * j + q];
              if (p < 0 || p >= a.ic.num_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); p = 0; }
              const int slot = pi % NR, use = pi / NR;
              if (!tc::mbar_wait(&sh.r_empty[slot], (use & 1) ^ 1, abort_p)) { fail(sh, a.err); ok = false; break; }
              tc::mbar_arrive_expect_tx(&sh.r_full[slot], PSLOT);
              uint8_t* dst = ring + slot * PSLOT;
              tc::bulk_g2s(dst, a.ic.data + (size_t)p * PAGE_DATA, PAGE_DATA, &sh.r_full[slot]);
              tc::bulk_g2s(dst + PAGE_DATA, a.ic.scale + (size_t)p * PAGE_SCALE, PAGE_SCALE, &sh.r_full[slot]);
              ++pi;
            }
          }
          x = tile_start[g] + j1;
          ++g;
        }
        for (int k = (pi > NR ? pi - NR : 0); k < pi; ++k)
          tc::mbar_wait(&sh.r_full[k % NR], (k / NR) & 1, abort_p, 1LL << 31);
      }
    } else if (warp == 1) {
      // ======================================================== MMA issuer
      if (lane == 0) {
        const uint32_t idq = tc::idesc_f16(128, NH, false, false);
        const uint32_t qaddr = tc::smem_u32(sQ);
        int n = 0, item = 0;
        bool ok = true;
        long long x = x0;
        int g = group_of(tile_start, a.B, x);
        while (x < x1 && ok) {
          const int nt = tile_start[g + 1] - tile_start[g];
          const int j0 = (int)(x - tile_start[g]);
          const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
          if (j1 > j0) {
            if (!tc::mbar_wait(&sh.q_full, item & 1, abort_p)) { fail(sh, a.err); ok = false; break; }
            ++item;
          }
          for (int j = j0; j < j1 && ok; ++j) {
            const int s = n & 1;
            if (!tc::mbar_wait(&sh.s_empty[s], ((n >> 1) & 1) ^ 1, abort_p) ||
                !tc::mbar_wait(&sh.kfull[s], (n >> 1) & 1, abort_p)) {
              fail(sh, a.err);
              ok = false;
              break;
            }
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t bd = tc::sdesc_sw128(qaddr + (k >> 2) * (NH * 128) + (k & 3) * 32, 16, 1024);
              tc::mma_ts(tbase + COL_S + 64 * s, tbase + COL_K + 64 * s + 8 * k, bd, idq, k != 0);
            }
            tc::mma_commit(&sh.kempty[s]);
            tc::mma_commit(&sh.s_full[s]);
            ++n;
          }
          x = tile_start[g] + j1;
          ++g;
        }
        tc::mma_commit(&sh.drain);
        tc::mbar_wait(&sh.drain, 0, abort_p, 1LL << 31);
      }
    } else if (warp >= 4 && warp < 8) {
      // ======================================================== key dequantizer (thread = token)
      const int t = tid - 128;
      const uint32_t lb = lane_base(warp);
      int pc = 0, n = 0;
      bool ok = true;
      long long x = x0;
      int g = group_of(tile_start, a.B, x);
      while (x < x1 && ok) {
        const int L = seq_tokens(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        for (int j = j0; j < j1 && ok; ++j) {
          const int npg = (TILE * j + PKV_PAGE < L) ? 2 : 1;
          const int s = n & 1;
          bool w_ok = tc::mbar_wait(&sh.kempty[s], ((n >> 1) & 1) ^ 1, abort_p);
          for (int q = 0; q < npg; ++q)
            w_ok = w_ok && tc::mbar_wait(&sh.r_full[(pc + q) % NR], ((pc + q) / NR) & 1, abort_p);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(sh, a.err); ok = false; break; }
          const bool valid = TILE * j + t < L;
          const uint8_t* page = ring + ((pc + (t >> 6)) % NR) * PSLOT;
          const int slot = t & 63;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {             // channels 64*hf .. 64*hf+63
            uint32_t r[32];
            if (valid) {
              const uint8_t* row = page + slot * (D / 2);
              const uint4 lo = *reinterpret_cast<const uint4*>(row + 16 * ((2 * hf) ^ (slot & 3)));
              const uint4 hi = *reinterpret_cast<const uint4*>(row + 16 * ((2 * hf + 1) ^ (slot & 3)));
              const uint32_t sc = *reinterpret_cast<const uint32_t*>(page + PAGE_DATA + slot * 8 + 4 * hf);
              const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
              for (int bk = 0; bk < 4; ++bk) {
                const uint32_t sb = (sc >> (8 * bk)) & 0xFFu;
                const uint32_t s2 = tc::e4m3x2_to_f16x2(sb | (sb << 8));
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  r[8 * bk + i] = tc::hmul2(tc::e2m1x2_to_f16x2((w[2 * bk + (i >> 2)] >> (8 * (i & 3))) & 0xFFu), s2);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = 0u;
            }
            tc::tmem_st32(tbase + lb + COL_K + 64 * s + 32 * hf, r);
          }
          tc::tc_wait_st();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            tc::mbar_arrive(&sh.kfull[s]);
            for (int q = 0; q < npg; ++q) tc::mbar_arrive(&sh.r_empty[(pc + q) % NR]);
          }
          pc += npg;
          ++n;
        }
        x = tile_start[g] + j1;
        ++g;
      }
    } else if (warp >= 8) {
      // ======================================================== epilogue (thread = token)
      const int t = tid - 256;
      const uint32_t lb = lane_base(warp);
      const float sc = a.tq * a.ic.ts;
      int n = 0;
      bool ok = true;
      long long x = x0;
      int g = group_of(tile_start, a.B, x);
      bool loaded = false;
      while (x < x1 && ok) {
        const int L = seq_tokens(a, g);
        const int nt = tile_start[g + 1] - tile_start[g];
        const int j0 = (int)(x - tile_start[g]);
        const int j1 = (int)min((long long)nt, x1 - tile_start[g]);
        if (j1 > j0) {
          if (!loaded) {
            load_q(a, g, sQ, sh.w, t);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sh.q_full);
          }
          loaded = false;
        }
        tc::named_bar(1, 128);                      // sh.w of this sequence visible to all 4 warps
        for (int j = j0; j < j1; ++j) {
          const int s = n & 1;
          const bool w_ok = tc::mbar_wait(&sh.s_full[s], (n >> 1) & 1, abort_p);
          if (tc::named_bar_or(2, 128, !w_ok)) { fail(sh, a.err); ok = false; break; }
          tc::tc_fence_after();
          float acc = 0.f;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t r[32];
            tc::tmem_ld32(tbase + lb + COL_S + 64 * s + 32 * hf, r);
            tc::tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc = fmaf(sh.w[32 * hf + i], fmaxf(__uint_as_float(r[i]), 0.f), acc);
          }
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&sh.s_empty[s]);
          ++n;
          // all S^T of this sequence read: the next sequence's queries may replace these
          if (j == j1 - 1) {
            // next sequence with tiles in this CTA's range (empty sequences have none)
            int gn = g + 1;
            while (gn < a.B && tile_start[gn + 1] == tile_start[gn]) ++gn;
            if (gn < a.B && tile_start[gn] < x1) {
              tc::named_bar(1, 128);                // every warp is done with sh.w
              load_q(a, gn, sQ, sh.w, t);
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sh.q_full);
              loaded = true;
            }
          }
          const int tok = TILE * j + t;
          if (tok < L) a.scores[(size_t)g * a.Lmax + tok] = acc * sc;
        }
        x = tile_start[g] + j1;
        ++g;
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tbase, 256);
}

}  // namespace tcscore
}  // namespace pkv

size_t pkv_score_tc_ws_bytes(int B) { return ((size_t)(B + 1) * 4 + 255) / 256 * 256; }

cudaError_t pkv_score_tc_init() {
  return cudaFuncSetAttribute(pkv::tcscore::score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              pkv::tcscore::DYN);
}

// scores[b][t] for t < seq_len[b]; ws holds the tile plan ([B+1] ints)
cudaError_t pkv_launch_score_tc(const uint8_t* q_idx, float tq, const float* w, const pkv_idx_cache& ic,
                                const int32_t* page_table, int max_pages, const int32_t* seq_len, int B, int Hi,
                                float* scores, int Lmax, void* ws, int num_sms, int* err, cudaStream_t st) {
  using namespace pkv::tcscore;
  Args a;
  a.q = q_idx; a.tq = tq; a.w = w; a.ic = ic; a.page_table = page_table; a.max_pages = max_pages;
  a.seq_len = seq_len; a.B = B; a.Hi = Hi; a.Lmax = Lmax; a.scores = scores; a.err = err;
  int* tile_start = (int*)ws;
  plan_kernel<<<1, 1024, 0, st>>>(a, tile_start);
  const long long tmax = (long long)B * ((Lmax + TILE - 1) / TILE);
  const int G = (int)(tmax < num_sms ? (tmax > 0 ? tmax : 1) : num_sms);
  score_tc_kernel<<<G, NTHREADS, DYN, st>>>(a, tile_start);
  return cudaGetLastError();
}
