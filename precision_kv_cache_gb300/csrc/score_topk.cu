// Sparse MQA logits (index scoring) and exact top-k selection.
//
// "Logits MQA creux" (vLLM blog, "Kernels"): the late indexer layers pick their
// top-k positions from a score per position; the score is
//   score_t = sum_h w_h * ReLU(q_h . k_t)
// with FP8 index queries q_h, NVFP4 index keys k_t and per-head weights w_h.
// Top-k: the k highest scores, ties to the lower position, output ascending.
//
// Selection is an exact radix select on the order-preserving 32-bit image of
// the float scores: a 12-bit histogram pass, a second 12-bit pass restricted to
// the boundary bin, then the few elements that share the boundary's top 24
// bits are sorted by (key desc, position asc) in one block.  Scores live in a
// scratch buffer that stays in L2 between passes.
#include "pkv_common.cuh"
#include "launch.h"

namespace pkv {

// ---------------------------------------------------------------- scoring (CUDA cores)
__global__ void __launch_bounds__(128) score_simple_kernel(
    const uint8_t* __restrict__ q_idx, float tq, const float* __restrict__ w, pkv_idx_cache ic,
    const int32_t* __restrict__ page_table, int max_pages, const int32_t* __restrict__ seq_len,
    int Hi, float* __restrict__ scores, int Lmax, int* err) {
  constexpr int D = 128;
  __shared__ float qs[64][D + 1];
  __shared__ float wsh[64];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < Hi * D; i += blockDim.x)
    qs[i / D][i % D] = e4m3_value(q_idx[(size_t)b * Hi * D + i]);
  for (int i = threadIdx.x; i < Hi; i += blockDim.x) wsh[i] = w[(size_t)b * Hi + i];
  __syncthreads();
  int L = seq_len[b];
  if (L > Lmax) { L = Lmax; if (threadIdx.x == 0 && blockIdx.x == 0) report(err, PKV_DEVERR_BAD_PAGE); }
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= L) return;
  const int pg = page_table[(size_t)b * max_pages + (t >> 6)];
  if (pg < 0 || pg >= ic.num_pages) { report(err, PKV_DEVERR_BAD_PAGE); scores[(size_t)b * Lmax + t] = 0.f; return; }
  const int slot = t & 63;
  const uint8_t* pd = ic.data + (size_t)pg * (PKV_PAGE * D / 2);
  const uint8_t* ps = ic.scale + (size_t)pg * (PKV_PAGE * D / 16);
  float k[D];
#pragma unroll
  for (int c = 0; c < 4; ++c) {   // four 16-byte chunks = 32 channels each
    const uint4 u = *reinterpret_cast<const uint4*>(pd + KLayout<D>::data(slot, 16 * c));
    const float s0 = e4m3_value(ps[KLayout<D>::scale(slot, 2 * c)]);
    const float s1 = e4m3_value(ps[KLayout<D>::scale(slot, 2 * c + 1)]);
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 32; ++i)
      k[32 * c + i] = e2m1_value((wv[i >> 3] >> (4 * (i & 7))) & 0xFu) * (i < 16 ? s0 : s1);
  }
  float acc = 0.f;
  for (int h = 0; h < Hi; ++h) {
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < D; ++i) dot = fmaf(qs[h][i], k[i], dot);
    acc = fmaf(wsh[h], fmaxf(dot, 0.f), acc);
  }
  scores[(size_t)b * Lmax + t] = acc * (tq * ic.ts);
}

}  // namespace pkv

cudaError_t pkv_launch_score_simple(const uint8_t* q_idx, float tq, const float* w, const pkv_idx_cache& ic,
                                    const int32_t* page_table, int max_pages, const int32_t* seq_len, int B,
                                    int Hi, float* scores, int Lmax, int* err, cudaStream_t st) {
  dim3 grid((Lmax + 127) / 128, B);
  pkv::score_simple_kernel<<<grid, 128, 0, st>>>(q_idx, tq, w, ic, page_table, max_pages, seq_len, Hi,
                                                  scores, Lmax, err);
  return cudaGetLastError();
}
