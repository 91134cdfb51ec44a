// NVFP4 quantize + append into the paged cache, and FP8 (E4M3) encode.
//
// The cache format is the one of "MegaAttention avec KV compressé NVFP4" (vLLM
// blog, "Kernels"): FP4 values with block scales.  Here: E2M1 codes, one E4M3
// scale per 16 consecutive channels of a token, one FP32 tensor scale.  The
// rounding contract (include/pkv.h) is followed step by step in float32 with
// correctly rounded multiply and divide, so the bytes are reproducible
// bit for bit.
#include "pkv_common.cuh"
#include "launch.h"

namespace pkv {

// One warp per (entry, tensor): lane handles 16-channel blocks lane, lane+32, ...
// LAYOUT: 0 = K cache (KLayout), 1 = V cache (VLayout), 2 = index keys (IdxLayout).
template <int D, int LAYOUT>
__device__ __forceinline__ void quantize_store_token(const float* __restrict__ x, float ts,
                                                     uint8_t* __restrict__ data,
                                                     uint8_t* __restrict__ scale, int t, int lane) {
  const float t6 = __fmul_rn(6.f, ts);
  for (int j = lane; j < D / 16; j += 32) {
    float v[16];
    const float4* x4 = reinterpret_cast<const float4*>(x + 16 * j);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 a = __ldg(x4 + q);
      v[4 * q + 0] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
    const uint32_t S = e4m3_code_pos(__fdiv_rn(amax, t6));
    uint32_t code[16];
    if (S == 0u) {
#pragma unroll
      for (int e = 0; e < 16; ++e) code[e] = 0u;
    } else {
      const float den = __fmul_rn(e4m3_value(S), ts);
#pragma unroll
      for (int e = 0; e < 16; ++e) code[e] = e2m1_code(__fdiv_rn(v[e], den));
    }
    if (LAYOUT != 1) {
      uint32_t lo = 0u, hi = 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        lo |= (code[2 * q] | (code[2 * q + 1] << 4)) << (8 * q);
        hi |= (code[8 + 2 * q] | (code[8 + 2 * q + 1] << 4)) << (8 * q);
      }
      const int off = LAYOUT == 2 ? IdxLayout::data(t, 8 * j) : KLayout<D>::data(t, 8 * j);
      *reinterpret_cast<uint2*>(data + off) = make_uint2(lo, hi);
      scale[KLayout<D>::scale(t, j)] = (uint8_t)S;
    } else {
      uint32_t* w = reinterpret_cast<uint32_t*>(data);
      const int sh = 4 * (t & 7);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        uint32_t* word = w + VLayout<D>::word(t, 16 * j + e);
        // other nibbles of the word belong to other tokens: update ours only
        atomicAnd(word, ~(0xFu << sh));
        atomicOr(word, code[e] << sh);
      }
      scale[VLayout<D>::scale(t, j)] = (uint8_t)S;
    }
  }
}

__device__ __forceinline__ bool locate(const int32_t* __restrict__ seq_idx,
                                       const int32_t* __restrict__ pos, int i,
                                       const int32_t* __restrict__ page_table, int max_pages,
                                       int num_pages, int* err, int* page, int* slot) {
  const int b = seq_idx[i], p = pos[i];
  if (b < 0 || p < 0 || p >= max_pages * PKV_PAGE) { report(err, PKV_DEVERR_BAD_PAGE); return false; }
  const int pg = page_table[(size_t)b * max_pages + p / PKV_PAGE];
  if (pg < 0 || pg >= num_pages) { report(err, PKV_DEVERR_BAD_PAGE); return false; }
  *page = pg;
  *slot = p % PKV_PAGE;
  return true;
}

template <int D>
__global__ void __launch_bounds__(256) append_kv_kernel(
    const float* __restrict__ k_new, const float* __restrict__ v_new,
    const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ pos, int n,
    pkv_kv_cache cache, const int32_t* __restrict__ page_table, int max_pages, int* err) {
  pkv::dep_wait();
  pkv::dep_trigger();
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int i = warp >> 1;
  if (i >= n) return;
  int page, slot;
  if (!locate(seq_idx, pos, i, page_table, max_pages, cache.num_pages, err, &page, &slot)) return;
  const size_t pd = (size_t)page * (PKV_PAGE * D / 2), ps = (size_t)page * (PKV_PAGE * D / 16);
  if ((warp & 1) == 0)
    quantize_store_token<D, 0>(k_new + (size_t)i * D, cache.ts_k, cache.k_data + pd,
                                   cache.k_scale + ps, slot, lane);
  else
    quantize_store_token<D, 1>(v_new + (size_t)i * D, cache.ts_v, cache.v_data + pd,
                                  cache.v_scale + ps, slot, lane);
}

__global__ void __launch_bounds__(256) append_index_kernel(
    const float* __restrict__ x, const int32_t* __restrict__ seq_idx,
    const int32_t* __restrict__ pos, int n, pkv_idx_cache ic,
    const int32_t* __restrict__ page_table, int max_pages, int* err) {
  pkv::dep_wait();
  pkv::dep_trigger();
  constexpr int D = 128;
  const int i = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  int page, slot;
  if (!locate(seq_idx, pos, i, page_table, max_pages, ic.num_pages, err, &page, &slot)) return;
  quantize_store_token<D, 2>(x + (size_t)i * D, ic.ts, ic.data + (size_t)page * (PKV_PAGE * D / 2),
                                 ic.scale + (size_t)page * (PKV_PAGE * D / 16), slot, lane);
}

__global__ void __launch_bounds__(256) quantize_fp8_kernel(const float* __restrict__ x, size_t n,
                                                           float tw, uint8_t* __restrict__ out) {
  pkv::dep_wait();
  pkv::dep_trigger();
  size_t i = (size_t)(blockIdx.x * blockDim.x + threadIdx.x) * 4;
  const size_t stride = (size_t)gridDim.x * blockDim.x * 4;
  for (; i < n; i += stride) {
    if (i + 4 <= n) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(x + i));
      const uint32_t c = e4m3_code(__fdiv_rn(a.x, tw)) | (e4m3_code(__fdiv_rn(a.y, tw)) << 8) |
                         (e4m3_code(__fdiv_rn(a.z, tw)) << 16) | (e4m3_code(__fdiv_rn(a.w, tw)) << 24);
      *reinterpret_cast<uint32_t*>(out + i) = c;
    } else {
      for (size_t e = i; e < n; ++e) out[e] = (uint8_t)e4m3_code(__fdiv_rn(x[e], tw));
    }
  }
}

}  // namespace pkv

// ---------------------------------------------------------------- launchers
cudaError_t pkv_launch_append_kv(int d, const float* k_new, const float* v_new, const int32_t* seq_idx,
                                 const int32_t* pos, int n, const pkv_kv_cache& cache,
                                 const int32_t* page_table, int max_pages, int* err, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long warps = 2LL * n;
  const int blocks = (int)((warps * 32 + 255) / 256);
  switch (d) {
    case 128: return pkv::launch_pdl(pkv::append_kv_kernel<128>, blocks, 256, 0, st, k_new, v_new, seq_idx, pos, n, cache, page_table, max_pages, err);
    case 256: return pkv::launch_pdl(pkv::append_kv_kernel<256>, blocks, 256, 0, st, k_new, v_new, seq_idx, pos, n, cache, page_table, max_pages, err);
    case 512: return pkv::launch_pdl(pkv::append_kv_kernel<512>, blocks, 256, 0, st, k_new, v_new, seq_idx, pos, n, cache, page_table, max_pages, err);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t pkv_launch_append_index(const float* x, const int32_t* seq_idx, const int32_t* pos, int n,
                                    const pkv_idx_cache& ic, const int32_t* page_table, int max_pages,
                                    int* err, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int blocks = (int)(((long long)n * 32 + 255) / 256);
  return pkv::launch_pdl(pkv::append_index_kernel, blocks, 256, 0, st, x, seq_idx, pos, n, ic, page_table, max_pages, err);
}

cudaError_t pkv_launch_quantize_fp8(const float* x, size_t n, float tw, uint8_t* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  size_t threads = (n + 3) / 4;
  int blocks = (int)((threads + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  return pkv::launch_pdl(pkv::quantize_fp8_kernel, blocks, 256, 0, st, x, n, tw, out);
}
