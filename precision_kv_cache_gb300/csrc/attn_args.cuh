// Arguments of one attention launch over (global NVFP4 segment, FP8 window
// segment) for a set of query rows.
#pragma once
#include "pkv_common.cuh"

namespace pkv {

struct AttnArgs {
  const uint16_t* q;          // bf16 bits [n_groups][H][D]
  const uint8_t* qs;          // the query rows split into tensor-core terms (workspace, set by the launcher)
  pkv_kv_cache cache;
  const int32_t* page_table;  // [B][max_pages]
  int max_pages;
  const int32_t* lens;        // decode: seq_len[B]; replay: prefix_len[B]
  const int32_t* sel;         // decode sparse: [B][k] ascending, -1 padded; else NULL
  int k;
  const uint8_t* wk;          // FP8 window K [B][128][D]
  const uint8_t* wv;
  float tw_k, tw_v;
  const int32_t* win_len;     // decode: [B] or NULL (= 128); unused in replay
  float scale;                // softmax scale
  int H;
  int D;
  int n_groups;               // query rows: B (decode) or B*128 (replay)
  int replay;
  int* err;
  long long wait_limit;       // cycles a bounded wait may take before the kernel gives up
  int hook_skip_copy;         // testing aid: the K-tile copy with this index (CTA 0) is never issued; -1 = none
  // fused decode: query rotation before QK, inverse
  // rotation of O and its FP8 encoding in the merge; rope_dim 0 = none
  const int32_t* rope_pos;    // [n_groups] row of cos_sin of each query row
  const float* cos_sin;       // [max_pos][rope_dim]: cosines, then sines
  int max_pos, rope_dim;
  float out_scale;
  uint8_t* out_fp8;           // [n_groups][H][D] or NULL
};

// Which sequence a query row belongs to and how many global / window entries it sees.
//   decode:  b = g; global = seq_len[b] (or k selected positions); window = win_len[b]
//   replay:  b = g/128, r = g%128; global = [0, H_b - 128); window = entries [0, r]
__device__ __forceinline__ void unit_extent(const AttnArgs& a, int g, int* b, int* n_glob, int* n_win,
                                            const uint8_t** wk, const uint8_t** wv) {
  int bb, ng, nw;
  if (a.replay) {
    bb = g >> 7;
    const int r = g & 127;
    ng = a.lens[bb] - PKV_WINDOW;
    nw = r + 1;
  } else {
    bb = g;
    ng = a.sel ? a.k : a.lens[bb];
    nw = a.win_len ? a.win_len[bb] : PKV_WINDOW;
  }
  if (ng < 0) { ng = 0; report(a.err, PKV_DEVERR_BAD_PAGE); }
  if (!a.sel && ng > a.max_pages * PKV_PAGE) { ng = a.max_pages * PKV_PAGE; report(a.err, PKV_DEVERR_BAD_PAGE); }
  nw = nw < 0 ? 0 : (nw > PKV_WINDOW ? PKV_WINDOW : nw);
  *b = bb;
  *n_glob = ng;
  *n_win = nw;
  *wk = a.wk + (size_t)bb * PKV_WINDOW * a.D;
  *wv = a.wv + (size_t)bb * PKV_WINDOW * a.D;
}

}  // namespace pkv
