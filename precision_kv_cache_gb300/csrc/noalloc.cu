// Decode attention for callers that cannot allocate device memory.
//
// pkv_decode_attn needs scratch for the split-K partial results and takes it
// from the caller (ws, ws_bytes).  Some callers cannot produce that buffer:
// code that runs while another thread captures a CUDA graph in global capture
// mode (cudaMalloc is prohibited there), plugins living inside a host
// framework that owns every byte of device memory, and latency-critical loops
// that cannot pay the device-wide synchronization of cudaMalloc/cudaFree.
// pkv_decode_attn_noalloc serves them from a fixed scratch array that is part
// of the library image itself.
//
// The array is a file-scope __device__ object of PKV_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  Host
// code must not use the symbol itself as a device address; the device address
// is looked up once per device with cudaGetSymbolAddress (on the first call
// made on that device, which should therefore come before any stream capture).
// All calls share the array: two calls whose kernels overlap on the GPU (other
// streams, other host threads) race on it.  Each call rewrites every scratch
// word it later reads, so nothing has to be cleared between calls.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkv.h"
#include "launch.h"

#define PKV_NOALLOC_MAX_DEVICES 64

static __device__ __align__(256) unsigned char pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_mu;
void* g_addr[PKV_NOALLOC_MAX_DEVICES] = {};

// device address of the scratch array on `device` (set up once per device)
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= PKV_NOALLOC_MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[device]) {
    int prev = -1;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, pkv_noalloc_scratch);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess) return e;
    g_addr[device] = p;
  }
  *out = g_addr[device];
  return cudaSuccess;
}
}  // namespace

extern "C" pkv_status pkv_decode_attn_noalloc(pkv_ctx* ctx, const void* q_bf16,
                                              const pkv_kv_cache* cache, const int32_t* page_table,
                                              int max_pages, const int32_t* seq_len, int B,
                                              const int32_t* sel_idx, int k, const pkv_window* win,
                                              float softmax_scale, float* out, float* out_lse,
                                              void* stream) {
  if (!ctx || B <= 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
  // the same length limit as pkv_decode_attn, checked before the length is formed in int
  if ((long long)max_pages * 64 > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
  const size_t need = sel_idx ? pkv_workspace_bytes(ctx, PKV_OP_DECODE_SPARSE, B, k)
                              : pkv_workspace_bytes(ctx, PKV_OP_DECODE, B, max_pages * 64);
  if (need == 0) return PKV_ERR_INVALID_ARG;
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(pkv_internal_ctx_device(ctx), &ws) != cudaSuccess) return PKV_ERR_CUDA;
  return pkv_decode_attn(ctx, q_bf16, cache, page_table, max_pages, seq_len, B, sel_idx, k, win,
                         softmax_scale, out, out_lse, ws, (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
