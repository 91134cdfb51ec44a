// Tensor-core (tcgen05 / TMEM) attention over the paged NVFP4 global segment.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "attn_args.cuh"

cudaError_t pkv_attn_tc_init(int device);
bool pkv_attn_tc_supported(const pkv::AttnArgs& a, int d);
size_t pkv_attn_tc_ws_bytes(int num_sms, int H, int D, int n_groups, int max_entries);
// prof_start/prof_stop (may be null): events recorded around the main kernel;
// *n_launches: kernels launched.
cudaError_t pkv_launch_attn_tc(pkv::AttnArgs& a, int num_sms, int max_entries, float* out, float* out_lse,
                               void* ws, cudaStream_t st, cudaEvent_t prof_start, cudaEvent_t prof_stop,
                               int* n_launches);
