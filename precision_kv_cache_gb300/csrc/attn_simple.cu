// Portable split-K attention over (global NVFP4 segment + FP8 window segment)
// on CUDA cores, and the LSE merge of partial results.
//
// This is the general path behind pkv_decode_attn (dense and sparse) and
// pkv_replay_attn for every supported shape; the tensor-core kernel
// (attn_tc.cu) takes over the dense global segment where its shape rules hold.
// Work unit = (split s, group of 8 query heads, query row g): a warp owns one
// head, a lane owns d/32 channels; entries are streamed with an online softmax
// (max-shifted exponentials, FP32) and each unit writes a normalized partial
// (O, LSE) that merge_splits combines ("flash-decoding": split along the
// sequence, then an LSE merge).
#include "pkv_common.cuh"
#include "attn_args.cuh"
#include "launch.h"

namespace pkv {

template <int D>
struct Slice {
  static constexpr int CPL = D / 32;   // channels per lane
};

// dequantized K (or V) channels [c0, c0+CPL) of token t of a page, without the tensor scale
template <int D>
__device__ __forceinline__ void load_k_slice(const uint8_t* __restrict__ pd, const uint8_t* __restrict__ psc,
                                             int t, int lane, float* kv) {
  constexpr int CPL = Slice<D>::CPL;
  const int c0 = lane * CPL;
  const float s = e4m3_value(psc[KLayout<D>::scale(t, c0 / 16)]);
  uint32_t w[2] = {0u, 0u};
  const uint8_t* p = pd + KLayout<D>::data(t, c0 / 2);
  if (CPL == 16) { const uint2 u = *reinterpret_cast<const uint2*>(p); w[0] = u.x; w[1] = u.y; }
  else if (CPL == 8) { w[0] = *reinterpret_cast<const uint32_t*>(p); }
  else { w[0] = *reinterpret_cast<const uint16_t*>(p); }
#pragma unroll
  for (int i = 0; i < CPL; ++i) kv[i] = e2m1_value((w[i >> 3] >> (4 * (i & 7))) & 0xFu) * s;
}

template <int D>
__device__ __forceinline__ void load_v_slice(const uint8_t* __restrict__ pd, const uint8_t* __restrict__ psc,
                                             int t, int lane, float* kv) {
  constexpr int CPL = Slice<D>::CPL;
  const int c0 = lane * CPL;
  const float s = e4m3_value(psc[VLayout<D>::scale(t, c0 / 16)]);
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(pd) + VLayout<D>::word(t, c0);
  const int sh = 4 * (t & 7);
#pragma unroll
  for (int q = 0; q < CPL / 4; ++q) {
    const uint4 u = *reinterpret_cast<const uint4*>(wp + 4 * q);
    kv[4 * q + 0] = e2m1_value((u.x >> sh) & 0xFu) * s;
    kv[4 * q + 1] = e2m1_value((u.y >> sh) & 0xFu) * s;
    kv[4 * q + 2] = e2m1_value((u.z >> sh) & 0xFu) * s;
    kv[4 * q + 3] = e2m1_value((u.w >> sh) & 0xFu) * s;
  }
}

template <int D>
__device__ __forceinline__ void load_fp8_slice(const uint8_t* __restrict__ row, int lane, float* kv) {
  constexpr int CPL = Slice<D>::CPL;
  const uint8_t* p = row + lane * CPL;
  uint32_t w[4];
  if (CPL == 16) { const uint4 u = *reinterpret_cast<const uint4*>(p); w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w; }
  else if (CPL == 8) { const uint2 u = *reinterpret_cast<const uint2*>(p); w[0] = u.x; w[1] = u.y; }
  else { w[0] = *reinterpret_cast<const uint32_t*>(p); }
#pragma unroll
  for (int i = 0; i < CPL; ++i) kv[i] = e4m3_value((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
}

template <int D>
__global__ void __launch_bounds__(256) attn_simple_kernel(AttnArgs a) {
  constexpr int CPL = Slice<D>::CPL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x, g = blockIdx.z;
  const int h = blockIdx.y * 8 + warp;
  if (h >= a.H) return;
  int b, n_glob, n_win;
  const uint8_t *wk, *wv;
  unit_extent(a, g, &b, &n_glob, &n_win, &wk, &wv);
  const int total = n_glob + n_win;
  const int e0 = s * a.chunk;
  const int e1 = min(total, e0 + a.chunk);

  const uint16_t* qp = a.q + ((size_t)g * a.H + h) * D + lane * CPL;
  float q[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) q[i] = bf16_bits_to_f32(qp[i]);

  const size_t pdb = (size_t)PKV_PAGE * D / 2, psb = (size_t)PKV_PAGE * D / 16;
  float m = -INFINITY, l = 0.f, o[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) o[i] = 0.f;

  for (int e = e0; e < e1; ++e) {
    float kv[CPL], vv[CPL];
    float zs, vs;
    if (e < n_glob) {
      const int t = a.sel ? a.sel[(size_t)b * a.k + e] : e;
      if (t < 0) continue;
      const int j = t >> 6;
      if (j >= a.max_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); continue; }
      const int pg = a.page_table[(size_t)b * a.max_pages + j];
      if (pg < 0 || pg >= a.cache.num_pages) { report(a.err, PKV_DEVERR_BAD_PAGE); continue; }
      const int slot = t & 63;
      load_k_slice<D>(a.cache.k_data + pg * pdb, a.cache.k_scale + pg * psb, slot, lane, kv);
      load_v_slice<D>(a.cache.v_data + pg * pdb, a.cache.v_scale + pg * psb, slot, lane, vv);
      zs = a.scale * a.cache.ts_k;
      vs = a.cache.ts_v;
    } else {
      const int w = e - n_glob;
      load_fp8_slice<D>(wk + (size_t)w * D, lane, kv);
      load_fp8_slice<D>(wv + (size_t)w * D, lane, vv);
      zs = a.scale * a.tw_k;
      vs = a.tw_v;
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) dot = fmaf(q[i], kv[i], dot);
#pragma unroll
    for (int off = 16; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float z = dot * zs;
    const float mn = fmaxf(m, z);
    const float corr = expf(m - mn);     // m = -inf on the first entry -> 0
    const float p = expf(z - mn);
    l = l * corr + p;
    const float pv = p * vs;
#pragma unroll
    for (int i = 0; i < CPL; ++i) o[i] = fmaf(pv, vv[i], o[i] * corr);
    m = mn;
  }
  const size_t row = ((size_t)g * a.n_split + s) * a.H + h;
  float* op = a.part_o + row * D + lane * CPL;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) op[i] = o[i] * inv;
  if (lane == 0) a.part_lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

// Combine n_split partials per (query row, head): lse = ln sum_s e^lse_s,
// O = sum_s e^(lse_s - lse) O_s.  One block per (g, h), threads over channels.
__global__ void merge_splits_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                    int n_split, int H, int D, float* __restrict__ out,
                                    float* __restrict__ out_lse) {
  const int gh = blockIdx.x;
  const int g = gh / H, h = gh % H;
  float m = -INFINITY;
  for (int s = 0; s < n_split; ++s) m = fmaxf(m, part_lse[((size_t)g * n_split + s) * H + h]);
  float sum = 0.f;
  if (m != -INFINITY)
    for (int s = 0; s < n_split; ++s) sum += expf(part_lse[((size_t)g * n_split + s) * H + h] - m);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < n_split; ++s) {
        const size_t row = ((size_t)g * n_split + s) * H + h;
        const float ls = part_lse[row];
        if (ls != -INFINITY) acc += expf(ls - m) * part_o[row * D + c];
      }
      acc /= sum;
    }
    out[(size_t)gh * D + c] = acc;
  }
  if (threadIdx.x == 0 && out_lse) out_lse[gh] = (m != -INFINITY) ? m + logf(sum) : -INFINITY;
}

__global__ void merge2_kernel(const float* o_a, const float* lse_a, const float* o_b,
                              const float* lse_b, float* o, float* lse, int rows, int dv) {
  const int r = blockIdx.x;
  if (r >= rows) return;
  const float la = lse_a[r], lb = lse_b[r];
  const float m = fmaxf(la, lb);
  const bool empty = (m == -INFINITY);
  const float wa = empty ? 0.f : expf(la - m), wb = empty ? 0.f : expf(lb - m);
  const float sum = wa + wb;
  for (int c = threadIdx.x; c < dv; c += blockDim.x) {
    const size_t i = (size_t)r * dv + c;
    o[i] = empty ? 0.f : (wa * o_a[i] + wb * o_b[i]) / sum;
  }
  __syncthreads();   // every thread has read lse_a/lse_b before they may be overwritten (aliasing)
  if (threadIdx.x == 0) lse[r] = empty ? -INFINITY : m + logf(sum);
}

}  // namespace pkv

cudaError_t pkv_launch_attn_simple(int d, const pkv::AttnArgs& a, cudaStream_t st) {
  dim3 grid(a.n_split, (a.H + 7) / 8, a.n_groups);
  switch (d) {
    case 128: pkv::attn_simple_kernel<128><<<grid, 256, 0, st>>>(a); break;
    case 256: pkv::attn_simple_kernel<256><<<grid, 256, 0, st>>>(a); break;
    case 512: pkv::attn_simple_kernel<512><<<grid, 256, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t pkv_launch_merge_splits(const float* part_o, const float* part_lse, int n_split, int rows_g,
                                    int H, int D, float* out, float* out_lse, cudaStream_t st) {
  pkv::merge_splits_kernel<<<rows_g * H, 128, 0, st>>>(part_o, part_lse, n_split, H, D, out, out_lse);
  return cudaGetLastError();
}

cudaError_t pkv_launch_merge2(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                              float* o, float* lse, int rows, int dv, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  pkv::merge2_kernel<<<rows, 128, 0, st>>>(o_a, lse_a, o_b, lse_b, o, lse, rows, dv);
  return cudaGetLastError();
}
