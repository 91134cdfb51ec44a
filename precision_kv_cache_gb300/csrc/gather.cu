// Sparse decode support: gather the selected positions of each sequence into a
// compact paged cache (same byte layouts), so the tensor-core attention kernel
// can run over them as a dense segment.
//
// "Logits MQA creux" (vLLM blog, "Kernels"): decode attention reads only the
// top-k positions the indexer selected.  Positions sel[b][0..k) are ascending
// and -1 padded; compact sequence b holds them, in order, in pages
// b*npb .. b*npb+npb-1 (npb = ceil(k/64)), and seq_len'[b] = number of valid
// positions.
#include "pkv_common.cuh"
#include "launch.h"

namespace pkv {

// one block (256 threads) per (compact page, octet of 8 tokens)
template <int D>
__global__ void __launch_bounds__(256) gather_kernel(pkv_kv_cache src, const int32_t* __restrict__ page_table,
                                                     int max_pages, const int32_t* __restrict__ sel, int k,
                                                     int npb, pkv_kv_cache dst, int32_t* __restrict__ dst_len,
                                                     int* err) {
  pkv::dep_wait();
  pkv::dep_trigger();
  constexpr int PD = PKV_PAGE * D / 2, PS = PKV_PAGE * D / 16;
  __shared__ int spage[8], sslot[8];
  const int page = blockIdx.x >> 3, o = blockIdx.x & 7;
  const int b = page / npb, jp = page % npb;
  const int tid = threadIdx.x;
  if (tid < 8) {
    const int i = jp * PKV_PAGE + 8 * o + tid;
    int pg = -1, sl = 0;
    if (i < k) {
      const int t = sel[(size_t)b * k + i];
      if (t >= 0) {
        const int j = t >> 6;
        if (j < max_pages) {
          const int p = page_table[(size_t)b * max_pages + j];
          if (p >= 0 && p < src.num_pages) { pg = p; sl = t & 63; }
          else report(err, PKV_DEVERR_BAD_PAGE);
        } else {
          report(err, PKV_DEVERR_BAD_PAGE);
        }
      }
    }
    spage[tid] = pg;
    sslot[tid] = sl;
  }
  // number of valid positions of sequence b (the list is ascending, -1 padded)
  if (jp == 0 && o == 0 && tid == 32) {
    int lo = 0, hi = k;                       // first index holding -1
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sel[(size_t)b * k + mid] >= 0) lo = mid + 1; else hi = mid;
    }
    dst_len[b] = lo;
  }
  __syncthreads();
  const size_t op = (size_t)page;
  // ---- K codes of the 8 tokens: 16-byte chunks, re-swizzled for the destination slot
  constexpr int NCH = D / 32;
  for (int w = tid; w < 8 * NCH; w += 256) {
    const int i = w / NCH, c = w % NCH, s = 8 * o + i;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (spage[i] >= 0) {
      const int ss = sslot[i];
      v = *reinterpret_cast<const uint4*>(src.k_data + (size_t)spage[i] * PD + KLayout<D>::chunk(ss, c));
    }
    *reinterpret_cast<uint4*>(dst.k_data + op * PD + KLayout<D>::chunk(s, c)) = v;
  }
  // ---- K scales: 8-byte words ([d/128][64][8])
  for (int w = tid; w < 8 * (D / 128); w += 256) {
    const int i = w % 8, gq = w / 8, s = 8 * o + i;
    uint2 v = make_uint2(0u, 0u);
    if (spage[i] >= 0)
      v = *reinterpret_cast<const uint2*>(src.k_scale + (size_t)spage[i] * PS + ((size_t)gq * PKV_PAGE + sslot[i]) * 8);
    *reinterpret_cast<uint2*>(dst.k_scale + op * PS + ((size_t)gq * PKV_PAGE + s) * 8) = v;
  }
  // ---- V codes: word (o, c) collects nibble i of its 8 tokens (coalesced over c)
  for (int c = tid; c < D; c += 256) {
    uint32_t word = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (spage[i] >= 0) {
        const int ss = sslot[i];
        const uint32_t sw = __ldg(reinterpret_cast<const uint32_t*>(src.v_data + (size_t)spage[i] * PD) + VLayout<D>::word(ss, c));
        word |= ((sw >> (4 * (ss & 7))) & 0xFu) << (4 * i);
      }
    }
    reinterpret_cast<uint32_t*>(dst.v_data + op * PD)[VLayout<D>::word(8 * o, c)] = word;
  }
  // ---- V scales: byte (block j, token s)
  for (int w = tid; w < 8 * (D / 16); w += 256) {
    const int j = w / 8, i = w % 8, s = 8 * o + i;
    uint8_t v = 0;
    if (spage[i] >= 0) v = src.v_scale[(size_t)spage[i] * PS + j * PKV_PAGE + sslot[i]];
    dst.v_scale[op * PS + j * PKV_PAGE + s] = v;
  }
}

__global__ void identity_table_kernel(int32_t* pt, int B, int npb) {
  pkv::dep_wait();
  pkv::dep_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B * npb) pt[i] = i;
}

}  // namespace pkv

size_t pkv_gather_ws_bytes(int d, int B, int k) {
  const size_t npb = (size_t)(k + PKV_PAGE - 1) / PKV_PAGE;
  const size_t pages = (size_t)B * npb;
  const size_t pool = pages * (2 * (size_t)PKV_PAGE * d / 2 + 2 * (size_t)PKV_PAGE * d / 16);
  return pool + pages * 4 + (size_t)B * 4 + 4 * 256;
}

// Carves the compact cache, page table and lengths out of ws; returns them.
cudaError_t pkv_launch_gather(int d, const pkv_kv_cache& src, const int32_t* page_table, int max_pages,
                              const int32_t* sel, int B, int k, void* ws, pkv_kv_cache* dst, int32_t** dst_pt,
                              int32_t** dst_len, int* npb_out, int* err, cudaStream_t st) {
  const int npb = (k + PKV_PAGE - 1) / PKV_PAGE;
  const size_t pages = (size_t)B * npb;
  const size_t PD = (size_t)PKV_PAGE * d / 2, PS = (size_t)PKV_PAGE * d / 16;
  uint8_t* p = (uint8_t*)ws;
  auto take = [&](size_t n) { uint8_t* r = p; p += (n + 255) / 256 * 256; return r; };
  dst->k_data = take(pages * PD);
  dst->k_scale = take(pages * PS);
  dst->v_data = take(pages * PD);
  dst->v_scale = take(pages * PS);
  dst->num_pages = (int)pages;
  dst->ts_k = src.ts_k;
  dst->ts_v = src.ts_v;
  *dst_pt = (int32_t*)take(pages * 4);
  *dst_len = (int32_t*)take((size_t)B * 4);
  *npb_out = npb;
  cudaError_t e = pkv::launch_pdl(pkv::identity_table_kernel, (int)((pages + 255) / 256), 256, 0, st, *dst_pt, B, npb);
  if (e != cudaSuccess) return e;
  const int grid = (int)pages * 8;
  switch (d) {
    case 128: return pkv::launch_pdl(pkv::gather_kernel<128>, grid, 256, 0, st, src, page_table, max_pages, sel, k, npb, *dst, *dst_len, err);
    case 256: return pkv::launch_pdl(pkv::gather_kernel<256>, grid, 256, 0, st, src, page_table, max_pages, sel, k, npb, *dst, *dst_len, err);
    case 512: return pkv::launch_pdl(pkv::gather_kernel<512>, grid, 256, 0, st, src, page_table, max_pages, sel, k, npb, *dst, *dst_len, err);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------- candidate index keys
// Candidate-list scoring ("Logits MQA creux": score a fixed candidate set per
// sequence): the index keys of the candidates cand[b][0..n) are gathered, in
// order, into compact pages b*npb .. b*npb+npb-1 (npb = ceil(n/64)) of an index
// pool with the same byte layout (128-channel K-layout: 64 code bytes per token,
// 16-byte pieces swizzled by slot mod 4; scales [1][64][8]).  cnt[b] = number
// of valid candidates (the list is ascending and -1 padded at the end).
namespace pkv {

__global__ void __launch_bounds__(256) gather_index_kernel(pkv_idx_cache src, const int32_t* __restrict__ page_table,
                                                           int max_pages, const int32_t* __restrict__ cand, int n,
                                                           int npb, pkv_idx_cache dst, int32_t* __restrict__ cnt,
                                                           int* err) {
  pkv::dep_wait();
  pkv::dep_trigger();
  constexpr int PD = PKV_PAGE * 64, PS = PKV_PAGE * 8;    // 128-channel index keys
  __shared__ int spage[64], sslot[64];
  const int page = blockIdx.x, b = page / npb, jp = page % npb;
  const int tid = threadIdx.x;
  if (tid < 64) {
    const int i = jp * PKV_PAGE + tid;
    int pg = -1, sl = 0;
    if (i < n) {
      const int t = cand[(size_t)b * n + i];
      if (t >= 0) {
        const int j = t >> 6;
        const int p = j < max_pages ? page_table[(size_t)b * max_pages + j] : -1;
        if (p >= 0 && p < src.num_pages) { pg = p; sl = t & 63; }
        else report(err, PKV_DEVERR_BAD_PAGE);
      }
    }
    spage[tid] = pg;
    sslot[tid] = sl;
  }
  if (jp == 0 && tid == 64) {
    int lo = 0, hi = n;                       // first index holding -1
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (cand[(size_t)b * n + mid] >= 0) lo = mid + 1; else hi = mid;
    }
    cnt[b] = lo;
  }
  __syncthreads();
  // codes: thread = (token s, 16-byte piece c)
  {
    const int s = tid >> 2, c = tid & 3;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (spage[s] >= 0) {
      const int ss = sslot[s];
      v = *reinterpret_cast<const uint4*>(src.data + (size_t)spage[s] * PD + ss * 64 + 16 * (c ^ (ss & 3)));
    }
    *reinterpret_cast<uint4*>(dst.data + (size_t)page * PD + s * 64 + 16 * (c ^ (s & 3))) = v;
  }
  // scales: one 8-byte word per token
  if (tid < 64) {
    uint2 v = make_uint2(0u, 0u);
    if (spage[tid] >= 0) v = *reinterpret_cast<const uint2*>(src.scale + (size_t)spage[tid] * PS + sslot[tid] * 8);
    *reinterpret_cast<uint2*>(dst.scale + (size_t)page * PS + tid * 8) = v;
  }
}

// out[b][i] (a candidate index, or -1) -> the candidate's position
__global__ void map_cand_kernel(int32_t* __restrict__ out, const int32_t* __restrict__ cand, int B, int n, int k) {
  pkv::dep_wait();
  pkv::dep_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * k) return;
  const int b = i / k, c = out[i];
  out[i] = c >= 0 ? cand[(size_t)b * n + c] : -1;
}

}  // namespace pkv

size_t pkv_gather_index_ws_bytes(int B, int n) {
  const size_t npb = (size_t)(n + PKV_PAGE - 1) / PKV_PAGE;
  const size_t pages = (size_t)B * npb;
  return pages * (PKV_PAGE * 64 + PKV_PAGE * 8) + pages * 4 + (size_t)B * 4 + 4 * 256;
}

cudaError_t pkv_launch_gather_index(const pkv_idx_cache& src, const int32_t* page_table, int max_pages,
                                    const int32_t* cand, int B, int n, void* ws, pkv_idx_cache* dst,
                                    int32_t** dst_pt, int32_t** dst_cnt, int* npb_out, int* err, cudaStream_t st) {
  const int npb = (n + PKV_PAGE - 1) / PKV_PAGE;
  const size_t pages = (size_t)B * npb;
  uint8_t* p = (uint8_t*)ws;
  auto take = [&](size_t bytes) { uint8_t* r = p; p += (bytes + 255) / 256 * 256; return r; };
  dst->data = take(pages * PKV_PAGE * 64);
  dst->scale = take(pages * PKV_PAGE * 8);
  dst->num_pages = (int)pages;
  dst->ts = src.ts;
  *dst_pt = (int32_t*)take(pages * 4);
  *dst_cnt = (int32_t*)take((size_t)B * 4);
  *npb_out = npb;
  const cudaError_t e = pkv::launch_pdl(pkv::identity_table_kernel, (int)((pages + 255) / 256), 256, 0, st, *dst_pt, B, npb);
  if (e != cudaSuccess) return e;
  return pkv::launch_pdl(pkv::gather_index_kernel, (int)pages, 256, 0, st, src, page_table, max_pages, cand, n, npb,
                         *dst, *dst_cnt, err);
}

cudaError_t pkv_launch_map_cand(int32_t* out, const int32_t* cand, int B, int n, int k, cudaStream_t st) {
  const int tot = B * k;
  return pkv::launch_pdl(pkv::map_cand_kernel, (tot + 255) / 256, 256, 0, st, out, cand, B, n, k);
}
