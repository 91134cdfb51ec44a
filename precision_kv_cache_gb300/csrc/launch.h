// Host-side launchers of the library's kernels (internal; the public ABI is include/pkv.h).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pkv.h"

#define PKV_TOPK_CAND 4096
#define PKV_TOPK_MAX_K 4096
#define PKV_TOPK_LAUNCHES 8   // memset + 7 kernels of the radix select

namespace pkv { struct AttnArgs; }

cudaError_t pkv_launch_append_kv(int d, const float* k_new, const float* v_new, const int32_t* seq_idx,
                                 const int32_t* pos, int n, const pkv_kv_cache& cache,
                                 const int32_t* page_table, int max_pages, int* err, cudaStream_t st);
cudaError_t pkv_launch_append_index(const float* x, const int32_t* seq_idx, const int32_t* pos, int n,
                                    const pkv_idx_cache& ic, const int32_t* page_table, int max_pages,
                                    int* err, cudaStream_t st);
cudaError_t pkv_launch_quantize_fp8(const float* x, size_t n, float tw, uint8_t* out, cudaStream_t st);
cudaError_t pkv_launch_merge2(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                              float* o, float* lse, int rows, int dv, cudaStream_t st);
size_t pkv_topk_ws_bytes(int B, int k, int Lmax);
cudaError_t pkv_launch_topk(const float* scores, int Lmax, const int32_t* seq_len, int B, int k,
                            int32_t* out, void* ws, cudaStream_t st);

// device a context was created on
int pkv_internal_ctx_device(const pkv_ctx* c);

size_t pkv_gather_ws_bytes(int d, int B, int k);
cudaError_t pkv_launch_gather(int d, const pkv_kv_cache& src, const int32_t* page_table, int max_pages,
                              const int32_t* sel, int B, int k, void* ws, pkv_kv_cache* dst, int32_t** dst_pt,
                              int32_t** dst_len, int* npb_out, int* err, cudaStream_t st);

size_t pkv_gather_index_ws_bytes(int B, int n);
cudaError_t pkv_launch_gather_index(const pkv_idx_cache& src, const int32_t* page_table, int max_pages,
                                    const int32_t* cand, int B, int n, void* ws, pkv_idx_cache* dst,
                                    int32_t** dst_pt, int32_t** dst_cnt, int* npb_out, int* err, cudaStream_t st);
cudaError_t pkv_launch_map_cand(int32_t* out, const int32_t* cand, int B, int n, int k, cudaStream_t st);

size_t pkv_score_tc_ws_bytes(int B, int num_sms);
cudaError_t pkv_score_tc_init();
// prof_start/prof_stop (may be null): events recorded around the scoring kernel
cudaError_t pkv_launch_score_tc(const uint8_t* q_idx, float tq, const float* w, const pkv_idx_cache& ic,
                                const int32_t* page_table, int max_pages, const int32_t* seq_len, int B, int Hi,
                                float* scores, int Lmax, void* ws, int num_sms, int* err, cudaStream_t st,
                                cudaEvent_t prof_start = nullptr, cudaEvent_t prof_stop = nullptr);
