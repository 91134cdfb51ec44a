// Exact top-k over per-sequence float32 scores (ties to the lower position,
// output ascending) by radix select on the order-preserving 32-bit key.
//
//   pass 1  histogram of key bits [31:20] (4096 bins)       -> boundary bin b1
//   pass 2  emit keys above b1; histogram bits [19:8] of b1  -> boundary bin b2
//   pass 3  emit keys above (b1,b2); collect keys in (b1,b2) as candidates
//   finish  sort candidates by (key desc, position asc), emit what is still needed
//           (if the candidate buffer overflowed: an ordered scan of the sequence)
//   extract "emit" sets the position's bit in a per-sequence bitmap; the k
//           positions are read out of it in ascending order (no sort), one
//           block per 1024-word chunk of the bitmap
#include "pkv_common.cuh"
#include "launch.h"

namespace pkv {

constexpr int TK_BINS = 4096;
constexpr int TK_ITEMS = 16;            // scores per thread per pass
constexpr int TK_THREADS = 256;

// state words per sequence
enum { ST_BIN1 = 0, ST_NEED1, ST_BIN2, ST_NEED2, ST_OUT, ST_NCAND, ST_OVF, ST_L, ST_WORDS = 8 };

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int seq_length(const int32_t* seq_len, int b, int Lmax) {
  int L = seq_len[b];
  return L < 0 ? 0 : (L > Lmax ? Lmax : L);
}

__global__ void __launch_bounds__(TK_THREADS) tk_pass1(const float* __restrict__ scores, int Lmax,
                                                       const int32_t* __restrict__ seq_len,
                                                       uint32_t* __restrict__ hist) {
  pkv::dep_wait();
  pkv::dep_trigger();
  __shared__ uint32_t h[TK_BINS];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < TK_BINS; i += TK_THREADS) h[i] = 0u;
  __syncthreads();
  const int L = seq_length(seq_len, b, Lmax);
  const int base = blockIdx.x * TK_THREADS * TK_ITEMS;
  const float* s = scores + (size_t)b * Lmax;
  float v[TK_ITEMS];                      // every load in flight before any use
#pragma unroll
  for (int i = 0; i < TK_ITEMS; ++i) {
    const int t = base + i * TK_THREADS + threadIdx.x;
    v[i] = t < L ? s[t] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < TK_ITEMS; ++i) {
    const int t = base + i * TK_THREADS + threadIdx.x;
    if (t < L) atomicAdd(&h[order_key(v[i]) >> 20], 1u);
  }
  __syncthreads();
  uint32_t* g = hist + (size_t)b * TK_BINS;
  for (int i = threadIdx.x; i < TK_BINS; i += TK_THREADS)
    if (h[i]) atomicAdd(&g[i], h[i]);
}

// One block of 1024 threads per sequence: find the bin where the count of keys
// at or above it first reaches `need` (scanning from the top bin down).
__global__ void __launch_bounds__(1024) tk_find(const uint32_t* __restrict__ hist, int* __restrict__ state,
                                                const int32_t* __restrict__ seq_len, int Lmax, int k, int level) {
  pkv::dep_wait();
  pkv::dep_trigger();
  __shared__ uint32_t warp_tot[32];
  const int b = blockIdx.x;
  int* st = state + b * ST_WORDS;
  int need;
  if (level == 1) {
    const int L = seq_length(seq_len, b, Lmax);
    if (threadIdx.x == 0) st[ST_L] = L;
    if (L <= k) {            // everything is selected
      if (threadIdx.x == 0) { st[ST_BIN1] = -1; st[ST_NEED1] = 0; st[ST_BIN2] = -1; st[ST_NEED2] = 0; }
      return;
    }
    need = k;
  } else {
    if (st[ST_BIN1] < 0) return;
    need = st[ST_NEED1];
  }
  const uint32_t* hb = hist + (size_t)b * TK_BINS;
  // thread i owns bins 4095-4i .. 4092-4i (top first)
  const int top = TK_BINS - 1 - 4 * threadIdx.x;
  uint32_t c[4], sum = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) { c[j] = hb[top - j]; sum += c[j]; }
  // exclusive prefix over threads (thread order = descending bins)
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  uint32_t wpre = 0u;
  for (int i = 0; i < wid; ++i) wpre += warp_tot[i];
  uint32_t above = wpre + incl - sum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (above < (uint32_t)need && above + c[j] >= (uint32_t)need) {
      if (level == 1) { st[ST_BIN1] = top - j; st[ST_NEED1] = need - (int)above; }
      else { st[ST_BIN2] = top - j; st[ST_NEED2] = need - (int)above; }
    }
    above += c[j];
  }
}

// selected position t: count it and set its bit in the sequence's bitmap
__device__ __forceinline__ void emit(uint32_t* bm_b, int* st, int t) {
  atomicAdd(&st[ST_OUT], 1);
  atomicOr(&bm_b[t >> 5], 1u << (t & 31));
}

__global__ void __launch_bounds__(TK_THREADS) tk_pass2(const float* __restrict__ scores, int Lmax,
                                                       int* __restrict__ state, uint32_t* __restrict__ hist2,
                                                       uint32_t* __restrict__ bm, int W) {
  pkv::dep_wait();
  pkv::dep_trigger();
  __shared__ uint32_t h[TK_BINS];
  const int b = blockIdx.y;
  int* st = state + b * ST_WORDS;
  const int L = st[ST_L];
  const int bin1 = st[ST_BIN1];
  for (int i = threadIdx.x; i < TK_BINS; i += TK_THREADS) h[i] = 0u;
  __syncthreads();
  const int base = blockIdx.x * TK_THREADS * TK_ITEMS;
  const float* s = scores + (size_t)b * Lmax;
  uint32_t* bmb = bm + (size_t)b * W;
  float v[TK_ITEMS];
#pragma unroll
  for (int i = 0; i < TK_ITEMS; ++i) {
    const int t = base + i * TK_THREADS + threadIdx.x;
    v[i] = t < L ? s[t] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < TK_ITEMS; ++i) {
    const int t = base + i * TK_THREADS + threadIdx.x;
    if (t < L) {
      const uint32_t key = order_key(v[i]);
      const int hi = (int)(key >> 20);
      if (hi > bin1) emit(bmb, st, t);
      else if (hi == bin1) atomicAdd(&h[(key >> 8) & 0xFFFu], 1u);
    }
  }
  __syncthreads();
  if (bin1 < 0) return;
  uint32_t* g = hist2 + (size_t)b * TK_BINS;
  for (int i = threadIdx.x; i < TK_BINS; i += TK_THREADS)
    if (h[i]) atomicAdd(&g[i], h[i]);
}

__global__ void __launch_bounds__(TK_THREADS) tk_pass3(const float* __restrict__ scores, int Lmax,
                                                       int* __restrict__ state, unsigned long long* __restrict__ cand,
                                                       int cap, uint32_t* __restrict__ bm, int W) {
  pkv::dep_wait();
  pkv::dep_trigger();
  const int b = blockIdx.y;
  int* st = state + b * ST_WORDS;
  const int bin1 = st[ST_BIN1];
  if (bin1 < 0) return;
  const int bin2 = st[ST_BIN2];
  const int L = st[ST_L];
  const int base = blockIdx.x * TK_THREADS * TK_ITEMS;
  const float* s = scores + (size_t)b * Lmax;
  uint32_t* bmb = bm + (size_t)b * W;
  unsigned long long* cb = cand + (size_t)b * cap;
  float v[TK_ITEMS];
#pragma unroll
  for (int i = 0; i < TK_ITEMS; ++i) {
    const int t = base + i * TK_THREADS + threadIdx.x;
    v[i] = t < L ? s[t] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < TK_ITEMS; ++i) {
    const int t = base + i * TK_THREADS + threadIdx.x;
    if (t < L) {
      const uint32_t key = order_key(v[i]);
      if ((int)(key >> 20) != bin1) continue;
      const int mid = (int)((key >> 8) & 0xFFFu);
      if (mid > bin2) emit(bmb, st, t);
      else if (mid == bin2) {
        const int c = atomicAdd(&st[ST_NCAND], 1);
        if (c < cap) cb[c] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)t);
        else st[ST_OVF] = 1;
      }
    }
  }
}

// bitonic sort of n (power of two) 64-bit values in shared memory, descending
__device__ void bitonic_desc(unsigned long long* v, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const unsigned long long a = v[lo], c = v[hi];
        if ((a < c) == desc) { v[lo] = c; v[hi] = a; }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(1024) tk_finish(const float* __restrict__ scores, int Lmax,
                                                  int* __restrict__ state,
                                                  const unsigned long long* __restrict__ cand, int cap,
                                                  uint32_t* __restrict__ bm, int W) {
  pkv::dep_wait();
  pkv::dep_trigger();
  extern __shared__ unsigned long long sv[];
  const int b = blockIdx.x;
  int* st = state + b * ST_WORDS;
  const int bin1 = st[ST_BIN1];
  if (bin1 < 0) return;
  const int need = st[ST_NEED2];
  uint32_t* bmb = bm + (size_t)b * W;
  if (!st[ST_OVF]) {
    const int n = min(st[ST_NCAND], cap);
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += blockDim.x) sv[i] = i < n ? cand[(size_t)b * cap + i] : 0ull;
    __syncthreads();
    bitonic_desc(sv, n2);
    for (int i = threadIdx.x; i < need; i += blockDim.x) {
      const int t = (int)(0xFFFFFFFFu - (uint32_t)(sv[i] & 0xFFFFFFFFull));
      atomicOr(&bmb[t >> 5], 1u << (t & 31));
    }
    return;
  }
  // Overflow: many scores share the boundary's top 24 bits.  Ordered scan of the
  // sequence: histogram of the low 8 bits among the prefix, then emit in
  // position order so equal keys go to the lower positions first.
  __shared__ uint32_t h[256];
  __shared__ int sel_bin, sel_need, taken;
  __shared__ uint32_t wcnt[32];
  const uint32_t prefix = ((uint32_t)bin1 << 12) | (uint32_t)st[ST_BIN2];
  const int L = st[ST_L];
  const float* s = scores + (size_t)b * Lmax;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
  __syncthreads();
  for (int t = threadIdx.x; t < L; t += blockDim.x) {
    const uint32_t key = order_key(s[t]);
    if ((key >> 8) == prefix) atomicAdd(&h[key & 0xFFu], 1u);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int above = 0;
    for (int i = 255; i >= 0; --i) {
      if (above + (int)h[i] >= need) { sel_bin = i; sel_need = need - above; break; }
      above += (int)h[i];
    }
    taken = 0;
  }
  __syncthreads();
  const uint32_t T = (prefix << 8) | (uint32_t)sel_bin;
  for (int t0 = 0; t0 < L; t0 += blockDim.x) {
    const int t = t0 + threadIdx.x;
    uint32_t key = 0u;
    bool above = false, tie = false;
    if (t < L) {
      key = order_key(s[t]);
      above = ((key >> 8) == prefix) && (key > T);
      tie = (key == T);
    }
    if (above) atomicOr(&bmb[t >> 5], 1u << (t & 31));
    // rank of this tie among the ties of this block, in position order
    const unsigned bal = __ballot_sync(0xffffffffu, tie);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) wcnt[wid] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int i = 0; i < wid; ++i) before += (int)wcnt[i];
    const int rank = taken + before + __popc(bal & ((1u << lane) - 1u));
    if (tie && rank < sel_need) atomicOr(&bmb[t >> 5], 1u << (t & 31));
    __syncthreads();
    if (threadIdx.x == 0) { int tot = 0; for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += (int)wcnt[i]; taken += tot; }
    __syncthreads();
  }
}

// The selected positions of sequence b, ascending, from its bitmap.  Grid
// (chunks of 1024 words, sequences), 1024 threads: block j first counts the bits
// of the words before its chunk (its output offset), then thread i takes word
// 1024 j + i, a block scan gives the thread's offset inside the chunk, and the
// set bits are written in order.  The last chunk's block pads the row with -1.
__global__ void __launch_bounds__(1024) tk_extract(const uint32_t* __restrict__ bm, int W, int32_t* __restrict__ out,
                                                   int k) {
  pkv::dep_wait();
  pkv::dep_trigger();
  __shared__ int wsum[32];
  __shared__ int base_s;
  const int b = blockIdx.y, j = blockIdx.x;
  const uint32_t* bmb = bm + (size_t)b * W;
  int32_t* ob = out + (size_t)b * k;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // bits before this chunk
  int before = 0;
  for (int w = threadIdx.x; w < 1024 * j; w += 1024) before += __popc(bmb[w]);
#pragma unroll
  for (int o = 16; o; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) wsum[wid] = before;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < 32; ++i) t += wsum[i];
    base_s = t;
  }
  __syncthreads();
  const int base = base_s;
  // this chunk: one word per thread, offsets by a block scan
  const int w = 1024 * j + threadIdx.x;
  uint32_t y = w < W ? bmb[w] : 0u;
  const int cnt = __popc(y);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  __syncthreads();                       // every thread has read base_s / the first wsum use is over
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  int pos = base + incl - cnt;
  for (int i = 0; i < wid; ++i) pos += wsum[i];
  while (y) {
    const int bit = __ffs(y) - 1;
    if (pos < k) ob[pos] = 32 * w + bit;
    ++pos;
    y &= y - 1;
  }
  if (j == (int)gridDim.x - 1) {
    int total = base;
    for (int i = 0; i < 32; ++i) total += wsum[i];
    for (int i = min(total, k) + threadIdx.x; i < k; i += 1024) ob[i] = -1;
  }
}

}  // namespace pkv

size_t pkv_topk_ws_bytes(int B, int k, int Lmax) {
  (void)k;
  const size_t W = ((size_t)Lmax + 31) / 32;
  return (size_t)B * (2 * pkv::TK_BINS * 4 + pkv::ST_WORDS * 4 + W * 4 + PKV_TOPK_CAND * 8) + 512;
}

cudaError_t pkv_launch_topk(const float* scores, int Lmax, const int32_t* seq_len, int B, int k,
                            int32_t* out, void* ws, cudaStream_t st) {
  using namespace pkv;
  uint8_t* p = (uint8_t*)ws;
  uint32_t* hist1 = (uint32_t*)p;  p += (size_t)B * TK_BINS * 4;
  uint32_t* hist2 = (uint32_t*)p;  p += (size_t)B * TK_BINS * 4;
  int* state = (int*)p;            p += (size_t)B * ST_WORDS * 4;
  const int W = (Lmax + 31) / 32;
  uint32_t* bm = (uint32_t*)p;     p += (size_t)B * W * 4;
  p = (uint8_t*)(((uintptr_t)p + 15) & ~(uintptr_t)15);
  unsigned long long* cand = (unsigned long long*)p;
  cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)B * (2 * TK_BINS + ST_WORDS + W) * 4, st);
  if (e != cudaSuccess) return e;
  const int chunks = (Lmax + TK_THREADS * TK_ITEMS - 1) / (TK_THREADS * TK_ITEMS);
  dim3 grid(chunks > 0 ? chunks : 1, B);
  tk_pass1<<<grid, TK_THREADS, 0, st>>>(scores, Lmax, seq_len, hist1);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_pdl(tk_find, B, 1024, 0, st, hist1, state, seq_len, Lmax, k, 1);
  if (e == cudaSuccess) e = launch_pdl(tk_pass2, grid, TK_THREADS, 0, st, scores, Lmax, state, hist2, bm, W);
  if (e == cudaSuccess) e = launch_pdl(tk_find, B, 1024, 0, st, hist2, state, seq_len, Lmax, k, 2);
  if (e == cudaSuccess)
    e = launch_pdl(tk_pass3, grid, TK_THREADS, 0, st, scores, Lmax, state, cand, (int)PKV_TOPK_CAND, bm, W);
  if (e == cudaSuccess)
    e = launch_pdl(tk_finish, B, 1024, (size_t)PKV_TOPK_CAND * 8, st, scores, Lmax, state, cand,
                   (int)PKV_TOPK_CAND, bm, W);
  if (e == cudaSuccess) e = launch_pdl(tk_extract, dim3((W + 1023) / 1024, B), 1024, 0, st, bm, W, out, k);
  return e;
}
