// C ABI of the library (declared in include/pkv.h): argument validation,
// scratch carving and kernel selection.  Every compute step runs in the
// kernels of this directory; nothing here touches tensor data on the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <new>

#include "pkv_common.cuh"
#include "attn_args.cuh"
#include "attn_tc.h"
#include "launch.h"

struct pkv_ctx {
  pkv_config cfg;
  int device;
  int num_sms;
  int* d_err;
  cudaEvent_t prof_start = nullptr;   // one-shot events around the next attention or scoring kernel
  cudaEvent_t prof_stop = nullptr;
  long long launches = 0;
  int last_path = 0;                  // 2 = tensor-core attention ran (0 = no attention call yet)
  long long wait_limit = 1LL << 31;   // cycles a device-side bounded wait may take
  int hook_skip_copy = -1;            // testing aid: K-tile copy left out by the attention kernel
};

namespace {

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool valid_d(int d) { return d == 128 || d == 256 || d == 512; }

bool valid_cache(const pkv_ctx* c, const pkv_kv_cache* kc) {
  if (!kc || !kc->k_data || !kc->k_scale || !kc->v_data || !kc->v_scale) return false;
  if (!aligned16(kc->k_data) || !aligned16(kc->k_scale) || !aligned16(kc->v_data) || !aligned16(kc->v_scale))
    return false;
  if (kc->num_pages <= 0) return false;
  if (!(kc->ts_k > 0.f) || !(kc->ts_v > 0.f) || !(kc->ts_k < INFINITY) || !(kc->ts_v < INFINITY)) return false;
  (void)c;
  return true;
}

bool valid_window(const pkv_window* w) {
  if (!w || !w->k || !w->v || !aligned16(w->k) || !aligned16(w->v)) return false;
  return (w->tw_k > 0.f && w->tw_k < INFINITY && w->tw_v > 0.f && w->tw_v < INFINITY);
}

size_t attn_ws_bytes(const pkv_ctx* c, int n_groups, int max_entries) {
  return pkv_attn_tc_ws_bytes(c->num_sms, c->cfg.n_heads, c->cfg.d, n_groups, max_entries);
}

}  // namespace

int pkv_internal_ctx_device(const pkv_ctx* c) { return c ? c->device : -1; }

extern "C" {

const char* pkv_status_str(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_BAD_PAGE: return "page id out of range or sequence longer than its page table";
    case PKV_ERR_TIMEOUT: return "bounded wait timed out on the device";
    case PKV_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

pkv_status pkv_init(const pkv_config* cfg, int device, pkv_ctx** out) {
  if (!cfg || !out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!valid_d(cfg->d) || cfg->n_heads < 1 || cfg->n_heads > 64 || cfg->page_size != PKV_PAGE ||
      cfg->window != PKV_WINDOW || cfg->d_index != 128 || cfg->n_index_heads < 1 || cfg->n_index_heads > 64)
    return PKV_ERR_UNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return PKV_ERR_CUDA;
  DeviceGuard g(device);
  pkv_ctx* c = new (std::nothrow) pkv_ctx;
  if (!c) return PKV_ERR_CUDA;
  c->cfg = *cfg;
  c->device = device;
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete c;
    return PKV_ERR_CUDA;
  }
  if (cudaMalloc(&c->d_err, sizeof(int)) != cudaSuccess) { delete c; return PKV_ERR_CUDA; }
  if (cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess) { cudaFree(c->d_err); delete c; return PKV_ERR_CUDA; }
  if (pkv_attn_tc_init(device) != cudaSuccess || pkv_score_tc_init() != cudaSuccess) {
    cudaFree(c->d_err);
    delete c;
    return PKV_ERR_CUDA;
  }
  *out = c;
  return PKV_OK;
}

void pkv_destroy(pkv_ctx* c) {
  if (!c) return;
  DeviceGuard g(c->device);
  cudaFree(c->d_err);
  delete c;
}

size_t pkv_workspace_bytes(const pkv_ctx* c, int op, int batch, int max_len) {
  if (!c || batch <= 0 || max_len < 0) return 0;
  switch (op) {
    case PKV_OP_DECODE: return attn_ws_bytes(c, batch, max_len + PKV_WINDOW);
    case PKV_OP_REPLAY: return attn_ws_bytes(c, batch * PKV_WINDOW, max_len + PKV_WINDOW);
    case PKV_OP_DECODE_SPARSE: {
      const int kp = (max_len + PKV_PAGE - 1) / PKV_PAGE * PKV_PAGE;
      return pkv_gather_ws_bytes(c->cfg.d, batch, max_len) + 256 + attn_ws_bytes(c, batch, kp + PKV_WINDOW);
    }
    case PKV_OP_SCORE_CAND:
      return pkv_gather_index_ws_bytes(batch, max_len) + 256 + (size_t)batch * (size_t)max_len * 4 + 256 +
             pkv_score_tc_ws_bytes(batch, c->num_sms) + pkv_topk_ws_bytes(batch, PKV_TOPK_MAX_K, max_len) + 256;
    case PKV_OP_SCORE_TOPK:
      return (size_t)batch * (size_t)max_len * 4 + 256 + pkv_score_tc_ws_bytes(batch, c->num_sms) +
             pkv_topk_ws_bytes(batch, PKV_TOPK_MAX_K, max_len) + 256;
  }
  return 0;
}

pkv_status pkv_append_kv(pkv_ctx* c, const float* k_new, const float* v_new, const int32_t* seq_idx,
                         const int32_t* pos, int n, const pkv_kv_cache* cache, const int32_t* page_table,
                         int max_pages, void* stream) {
  if (!c || n < 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!k_new || !v_new || !seq_idx || !pos || !page_table || !aligned16(k_new) || !aligned16(v_new))
    return PKV_ERR_INVALID_ARG;
  if (!valid_cache(c, cache)) return PKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  c->launches += 1;
  return cuda_status(pkv_launch_append_kv(c->cfg.d, k_new, v_new, seq_idx, pos, n, *cache, page_table,
                                          max_pages, c->d_err, (cudaStream_t)stream));
}

pkv_status pkv_append_index(pkv_ctx* c, const float* x, const int32_t* seq_idx, const int32_t* pos, int n,
                            const pkv_idx_cache* ic, const int32_t* page_table, int max_pages, void* stream) {
  if (!c || n < 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!x || !seq_idx || !pos || !page_table || !ic || !ic->data || !ic->scale || !aligned16(x) ||
      !aligned16(ic->data) || !aligned16(ic->scale) || ic->num_pages <= 0 || !(ic->ts > 0.f) || !(ic->ts < INFINITY))
    return PKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  c->launches += 1;
  return cuda_status(pkv_launch_append_index(x, seq_idx, pos, n, *ic, page_table, max_pages, c->d_err,
                                             (cudaStream_t)stream));
}

pkv_status pkv_quantize_fp8(const float* x, size_t n, float tw, uint8_t* out, void* stream) {
  if (n == 0) return PKV_OK;
  if (!x || !out || !aligned16(x) || ((uintptr_t)out & 3u) || !(tw > 0.f) || !(tw < INFINITY))
    return PKV_ERR_INVALID_ARG;
  return cuda_status(pkv_launch_quantize_fp8(x, n, tw, out, (cudaStream_t)stream));
}

pkv_status pkv_score_topk(pkv_ctx* c, const uint8_t* q_idx, float tq, const float* w, const pkv_idx_cache* ic,
                          const int32_t* page_table, int max_pages, const int32_t* seq_len, int B, int k,
                          int32_t* out_idx, float* out_score, void* ws, size_t ws_bytes, void* stream) {
  if (!c || B <= 0 || max_pages <= 0 || k < 1 || k > PKV_TOPK_MAX_K) return PKV_ERR_INVALID_ARG;
  if (!q_idx || !w || !ic || !ic->data || !ic->scale || !page_table || !seq_len || !out_idx)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(ic->data) || !aligned16(ic->scale) || ic->num_pages <= 0 || !(ic->ts > 0.f) ||
      !(tq > 0.f) || !(tq < INFINITY) || !(ic->ts < INFINITY))
    return PKV_ERR_INVALID_ARG;
  if ((long long)max_pages * PKV_PAGE > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
  const int Lmax = max_pages * PKV_PAGE;
  const size_t need = pkv_workspace_bytes(c, PKV_OP_SCORE_TOPK, B, Lmax);
  if (!ws || ws_bytes < need || !aligned16(ws)) return PKV_ERR_WORKSPACE;
  DeviceGuard g(c->device);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* p = (uint8_t*)ws;
  float* scores = out_score;
  if (!scores) scores = (float*)p;
  p += (size_t)B * Lmax * 4;
  p = (uint8_t*)(((uintptr_t)p + 255) & ~(uintptr_t)255);
  void* plan = p;
  p += pkv_score_tc_ws_bytes(B, c->num_sms);
  c->launches += 2 + PKV_TOPK_LAUNCHES;
  cudaEvent_t e0 = c->prof_start, e1 = c->prof_stop;
  c->prof_start = c->prof_stop = nullptr;
  cudaError_t e = pkv_launch_score_tc(q_idx, tq, w, *ic, page_table, max_pages, seq_len, B, c->cfg.n_index_heads,
                                      scores, Lmax, plan, c->num_sms, c->d_err, st, e0, e1);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return cuda_status(pkv_launch_topk(scores, Lmax, seq_len, B, k, out_idx, p, st));
}

pkv_status pkv_score_topk_cand(pkv_ctx* c, const uint8_t* q_idx, float tq, const float* w, const pkv_idx_cache* ic,
                               const int32_t* page_table, int max_pages, const int32_t* cand, int n_cand, int B,
                               int k, int32_t* out_idx, float* out_score, void* ws, size_t ws_bytes, void* stream) {
  if (!c || B <= 0 || max_pages <= 0 || k < 1 || k > PKV_TOPK_MAX_K || n_cand < 1 || n_cand > (1 << 30))
    return PKV_ERR_INVALID_ARG;
  if (!q_idx || !w || !ic || !ic->data || !ic->scale || !page_table || !cand || !out_idx) return PKV_ERR_INVALID_ARG;
  if (!aligned16(ic->data) || !aligned16(ic->scale) || ic->num_pages <= 0 || !(ic->ts > 0.f) ||
      !(tq > 0.f) || !(tq < INFINITY) || !(ic->ts < INFINITY))
    return PKV_ERR_INVALID_ARG;
  if ((long long)max_pages * PKV_PAGE > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
  const size_t need = pkv_workspace_bytes(c, PKV_OP_SCORE_CAND, B, n_cand);
  if (!ws || ws_bytes < need || !aligned16(ws)) return PKV_ERR_WORKSPACE;
  DeviceGuard g(c->device);
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* p = (uint8_t*)ws;
  // candidate keys gathered into compact pages, one compact sequence per row
  pkv_idx_cache cc;
  int32_t *cpt = nullptr, *cnt = nullptr;
  int npb = 0;
  cudaError_t e = pkv_launch_gather_index(*ic, page_table, max_pages, cand, B, n_cand, p, &cc, &cpt, &cnt, &npb,
                                          c->d_err, st);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  p += pkv_gather_index_ws_bytes(B, n_cand);
  p = (uint8_t*)(((uintptr_t)p + 255) & ~(uintptr_t)255);
  float* scores = out_score;
  if (!scores) scores = (float*)p;
  p += (size_t)B * n_cand * 4;
  p = (uint8_t*)(((uintptr_t)p + 255) & ~(uintptr_t)255);
  void* plan = p;
  p += pkv_score_tc_ws_bytes(B, c->num_sms);
  c->launches += 2 + 2 + PKV_TOPK_LAUNCHES + 1;
  cudaEvent_t e0 = c->prof_start, e1 = c->prof_stop;
  c->prof_start = c->prof_stop = nullptr;
  e = pkv_launch_score_tc(q_idx, tq, w, cc, cpt, npb, cnt, B, c->cfg.n_index_heads, scores, n_cand, plan,
                          c->num_sms, c->d_err, st, e0, e1);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  // top-k over candidate indices (ascending candidates: lower index = lower position), then to positions
  e = pkv_launch_topk(scores, n_cand, cnt, B, k, out_idx, p, st);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return cuda_status(pkv_launch_map_cand(out_idx, cand, B, n_cand, k, st));
}

static pkv_status run_attention(pkv_ctx* c, pkv::AttnArgs& a, int max_entries, float* out, float* out_lse,
                                void* ws, size_t ws_bytes, cudaStream_t st) {
  // one kernel family: shapes outside it are refused, never sent elsewhere
  if (!pkv_attn_tc_supported(a, c->cfg.d)) return PKV_ERR_UNSUPPORTED;
  const size_t need = attn_ws_bytes(c, a.n_groups, max_entries);
  if (!ws || ws_bytes < need || !aligned16(ws)) return PKV_ERR_WORKSPACE;
  a.wait_limit = c->wait_limit;
  a.hook_skip_copy = c->hook_skip_copy;
  cudaEvent_t e0 = c->prof_start, e1 = c->prof_stop;
  c->prof_start = c->prof_stop = nullptr;
  int nl = 0;
  cudaError_t e = pkv_launch_attn_tc(a, c->num_sms, max_entries, out, out_lse, ws, st, e0, e1, &nl);
  c->launches += nl;
  c->last_path = 2;
  return cuda_status(e);
}

pkv_status pkv_decode_attn(pkv_ctx* c, const void* q, const pkv_kv_cache* cache, const int32_t* page_table,
                           int max_pages, const int32_t* seq_len, int B, const int32_t* sel_idx, int k,
                           const pkv_window* win, float softmax_scale, float* out, float* out_lse, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!c || B <= 0 || max_pages <= 0 || !q || !page_table || !seq_len || !out || !aligned16(q) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  if (!valid_cache(c, cache) || !valid_window(win)) return PKV_ERR_INVALID_ARG;
  if (sel_idx && (k < 1 || k > PKV_TOPK_MAX_K)) return PKV_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
    return PKV_ERR_INVALID_ARG;
  if ((long long)max_pages * PKV_PAGE > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
  DeviceGuard g(c->device);
  pkv::AttnArgs a{};
  a.q = (const uint16_t*)q;
  a.cache = *cache;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.lens = seq_len;
  a.sel = sel_idx;
  a.k = sel_idx ? k : 0;
  a.wk = win->k;
  a.wv = win->v;
  a.tw_k = win->tw_k;
  a.tw_v = win->tw_v;
  a.win_len = win->win_len;
  a.scale = softmax_scale;
  a.H = c->cfg.n_heads;
  a.D = c->cfg.d;
  a.n_groups = B;
  a.replay = 0;
  a.err = c->d_err;
  {
    pkv::AttnArgs chk = a;
    chk.sel = nullptr;
    if (!pkv_attn_tc_supported(chk, c->cfg.d)) return PKV_ERR_UNSUPPORTED;
  }
  if (sel_idx) {
    // the selected tokens are gathered into compact pages, then attended as a dense segment
    const size_t need = pkv_workspace_bytes(c, PKV_OP_DECODE_SPARSE, B, k);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PKV_ERR_WORKSPACE;
    pkv::AttnArgs ad = a;
    ad.sel = nullptr;
    ad.k = 0;
    const size_t gbytes = (pkv_gather_ws_bytes(c->cfg.d, B, k) + 255) / 256 * 256;
    pkv_kv_cache compact{};
    int32_t *cpt = nullptr, *clen = nullptr;
    int npb = 0;
    c->launches += 2;
    cudaError_t e = pkv_launch_gather(c->cfg.d, *cache, page_table, max_pages, sel_idx, B, k, ws, &compact, &cpt,
                                      &clen, &npb, c->d_err, (cudaStream_t)stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    ad.cache = compact;
    ad.page_table = cpt;
    ad.max_pages = npb;
    ad.lens = clen;
    return run_attention(c, ad, npb * PKV_PAGE + PKV_WINDOW, out, out_lse, (uint8_t*)ws + gbytes, ws_bytes - gbytes,
                         (cudaStream_t)stream);
  }
  const int max_entries = max_pages * PKV_PAGE + PKV_WINDOW;
  return run_attention(c, a, max_entries, out, out_lse, ws, ws_bytes, (cudaStream_t)stream);
}

pkv_status pkv_decode_attn_fused(pkv_ctx* c, const void* q, const pkv_kv_cache* cache, const int32_t* page_table,
                                 int max_pages, const int32_t* seq_len, int B, const int32_t* sel_idx, int k,
                                 const pkv_window* win, float softmax_scale, const pkv_rope_fp8* fz,
                                 uint8_t* out_fp8, float* out, float* out_lse, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (!c || B <= 0 || max_pages <= 0 || !q || !page_table || !seq_len || !fz || !out_fp8 || !aligned16(q) ||
      !aligned16(out_fp8) || (out && !aligned16(out)))
    return PKV_ERR_INVALID_ARG;
  if (!fz->pos || !fz->cos_sin || !aligned16(fz->cos_sin) || fz->max_pos < 1 || fz->rope_dim < 8 ||
      fz->rope_dim > c->cfg.d || fz->rope_dim % 8 != 0 || !(fz->out_scale > 0.f) || !(fz->out_scale < INFINITY))
    return PKV_ERR_INVALID_ARG;
  if ((long long)fz->max_pos * fz->rope_dim > (1LL << 40)) return PKV_ERR_INVALID_ARG;
  if (!valid_cache(c, cache) || !valid_window(win)) return PKV_ERR_INVALID_ARG;
  if (sel_idx && (k < 1 || k > PKV_TOPK_MAX_K)) return PKV_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
    return PKV_ERR_INVALID_ARG;
  if ((long long)max_pages * PKV_PAGE > (1LL << 30)) return PKV_ERR_UNSUPPORTED;
  pkv::AttnArgs a{};
  a.q = (const uint16_t*)q;
  a.cache = *cache;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.lens = seq_len;
  a.wk = win->k;
  a.wv = win->v;
  a.tw_k = win->tw_k;
  a.tw_v = win->tw_v;
  a.win_len = win->win_len;
  a.scale = softmax_scale;
  a.H = c->cfg.n_heads;
  a.D = c->cfg.d;
  a.n_groups = B;
  a.replay = 0;
  a.err = c->d_err;
  a.rope_pos = fz->pos;
  a.cos_sin = fz->cos_sin;
  a.max_pos = fz->max_pos;
  a.rope_dim = fz->rope_dim;
  a.out_scale = fz->out_scale;
  a.out_fp8 = out_fp8;
  // the fusion lives in the tensor-core kernel's Q load and merge epilogue
  if (!pkv_attn_tc_supported(a, c->cfg.d)) return PKV_ERR_UNSUPPORTED;
  DeviceGuard g(c->device);
  if (sel_idx) {
    const size_t need = pkv_workspace_bytes(c, PKV_OP_DECODE_SPARSE, B, k);
    if (!ws || ws_bytes < need || !aligned16(ws)) return PKV_ERR_WORKSPACE;
    const size_t gbytes = (pkv_gather_ws_bytes(c->cfg.d, B, k) + 255) / 256 * 256;
    pkv_kv_cache compact{};
    int32_t *cpt = nullptr, *clen = nullptr;
    int npb = 0;
    c->launches += 2;
    cudaError_t e = pkv_launch_gather(c->cfg.d, *cache, page_table, max_pages, sel_idx, B, k, ws, &compact, &cpt,
                                      &clen, &npb, c->d_err, (cudaStream_t)stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    a.cache = compact;
    a.page_table = cpt;
    a.max_pages = npb;
    a.lens = clen;
    return run_attention(c, a, npb * PKV_PAGE + PKV_WINDOW, out, out_lse, (uint8_t*)ws + gbytes, ws_bytes - gbytes,
                         (cudaStream_t)stream);
  }
  return run_attention(c, a, max_pages * PKV_PAGE + PKV_WINDOW, out, out_lse, ws, ws_bytes, (cudaStream_t)stream);
}

pkv_status pkv_replay_attn(pkv_ctx* c, const void* q, const pkv_kv_cache* cache, const int32_t* page_table,
                           int max_pages, const int32_t* prefix_len, int B, const pkv_window* cw,
                           float softmax_scale, float* out, float* out_lse, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!c || B <= 0 || max_pages <= 0 || !q || !page_table || !prefix_len || !out || !aligned16(q) ||
      !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  if (!valid_cache(c, cache) || !valid_window(cw)) return PKV_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
    return PKV_ERR_INVALID_ARG;
  if ((long long)max_pages * PKV_PAGE > (1LL << 30) || (long long)B * PKV_WINDOW > (1LL << 24))
    return PKV_ERR_UNSUPPORTED;
  DeviceGuard g(c->device);
  pkv::AttnArgs a{};
  a.q = (const uint16_t*)q;
  a.cache = *cache;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.lens = prefix_len;
  a.sel = nullptr;
  a.k = 0;
  a.wk = cw->k;
  a.wv = cw->v;
  a.tw_k = cw->tw_k;
  a.tw_v = cw->tw_v;
  a.win_len = nullptr;
  a.scale = softmax_scale;
  a.H = c->cfg.n_heads;
  a.D = c->cfg.d;
  a.n_groups = B * PKV_WINDOW;
  a.replay = 1;
  a.err = c->d_err;
  const int max_entries = max_pages * PKV_PAGE + PKV_WINDOW;
  return run_attention(c, a, max_entries, out, out_lse, ws, ws_bytes, (cudaStream_t)stream);
}

pkv_status pkv_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b, float* o,
                     float* lse, int rows, int dv, void* stream) {
  if (rows < 0 || dv <= 0) return PKV_ERR_INVALID_ARG;
  if (rows == 0) return PKV_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse) return PKV_ERR_INVALID_ARG;
  return cuda_status(pkv_launch_merge2(o_a, lse_a, o_b, lse_b, o, lse, rows, dv, (cudaStream_t)stream));
}

pkv_status pkv_get_error(pkv_ctx* c, void* stream) {
  if (!c) return PKV_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, c->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
  if (h & PKV_DEVERR_TIMEOUT) return PKV_ERR_TIMEOUT;
  if (h & PKV_DEVERR_BAD_PAGE) return PKV_ERR_BAD_PAGE;
  return PKV_OK;
}

pkv_status pkv_set_test_hooks(pkv_ctx* c, long long wait_limit_cycles, int skip_copy) {
  if (!c || wait_limit_cycles < 1000 || skip_copy < -1) return PKV_ERR_INVALID_ARG;
  c->wait_limit = wait_limit_cycles;
  c->hook_skip_copy = skip_copy;
  return PKV_OK;
}

pkv_status pkv_set_profile_events(pkv_ctx* c, void* start, void* stop) {
  if (!c) return PKV_ERR_INVALID_ARG;
  c->prof_start = (cudaEvent_t)start;
  c->prof_stop = (cudaEvent_t)stop;
  return PKV_OK;
}

long long pkv_launch_count(const pkv_ctx* c) { return c ? c->launches : 0; }

int pkv_attn_path(const pkv_ctx* c) { return c ? c->last_path : 0; }

}  // extern "C"
