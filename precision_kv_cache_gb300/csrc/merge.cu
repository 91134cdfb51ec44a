// LSE merge of two partial results over disjoint entry sets (pkv_merge): the
// combine step of flash-decoding, lse = ln(e^lse_a + e^lse_b),
// o = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b; a part with lse = -inf has
// weight 0, and two empty parts give o = 0, lse = -inf.
#include "pkv_common.cuh"
#include "launch.h"

namespace pkv {

// one block of 128 threads per row; o / lse may alias the a inputs
__global__ void merge2_kernel(const float* o_a, const float* lse_a, const float* o_b,
                              const float* lse_b, float* o, float* lse, int rows, int dv) {
  pkv::dep_wait();
  pkv::dep_trigger();
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

cudaError_t pkv_launch_merge2(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                              float* o, float* lse, int rows, int dv, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return pkv::launch_pdl(pkv::merge2_kernel, rows, 128, 0, st, o_a, lse_a, o_b, lse_b, o, lse, rows, dv);
}
