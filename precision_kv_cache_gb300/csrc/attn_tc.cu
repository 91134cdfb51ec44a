// Tensor-core attention: not enabled yet; every call takes the CUDA-core path.
#include "attn_tc.h"

cudaError_t pkv_attn_tc_init(int) { return cudaSuccess; }
bool pkv_attn_tc_supported(const pkv::AttnArgs&, int) { return false; }
size_t pkv_attn_tc_ws_bytes(int, int, int, int, int) { return 0; }
cudaError_t pkv_launch_attn_tc(pkv::AttnArgs&, int, int, float*, float*, void*, cudaStream_t, cudaEvent_t,
                               cudaEvent_t, int*) {
  return cudaErrorNotSupported;
}
