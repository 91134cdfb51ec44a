/*
 * pkv.h - C ABI of the GB300 (sm_103a) decode-attention library for a paged
 * NVFP4 global KV cache plus an FP8 sliding window.
 *
 * What the calls compute (sources: the vLLM blog "DeepSeek-V4.1-Flash sur
 * vLLM : 5x de débit agentique dès le jour 0" - sections "SWA bounded replay",
 * "Côté encodeur : reconstruire la fenêtre lors d'un hit de cache", "Kernels"
 * paragraphs "Logits MQA creux" and "MegaAttention avec KV compressé NVFP4",
 * "Performances agentiques"; and the cocoloop summary, section "Les
 * particularités du modèle lui-même"):
 *   - the global KV is compressed, shared by every query head (MQA over one
 *     latent) and stored in FP4 (NVFP4 here: E2M1 values, one E4M3 scale per
 *     16 consecutive channels of a token, one FP32 scale per tensor), in
 *     64-token pages reached through a page table;
 *   - a sliding window of the last 128 positions is kept uncompressed in FP8
 *     (E4M3, one FP32 scale per tensor);
 *   - decode attention = softmax over the global tokens plus the window entries;
 *   - sparse MQA logits: an index score per position picks the top-k positions
 *     that decode attention then reads;
 *   - bounded replay: after a prefix hit of length H the 128 tokens [H-128, H)
 *     are re-run with the window clipped at s = H-128.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned, on the device the context was created on.  Nothing is freed or
 *     retained by the library after a call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream; host-side validation happens
 *     before any launch and returns PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED
 *     without launching anything.  The library's kernels are launched with
 *     programmatic dependent launch: one may start while the kernel before it
 *     on the stream is finishing, but waits for it to complete before touching
 *     global memory, so stream order holds as for plain launches (a call sees
 *     what earlier work on the stream wrote; later work sees its results).
 *   - Faults found on the device (a page id outside [0, num_pages), a sequence
 *     longer than its page table) never trap: the kernel skips the access,
 *     records a code in the context's device error word and finishes.
 *     pkv_get_error() synchronizes the stream and returns/clears it.
 *   - A context is not thread-safe; use one per host thread / stream.
 *   - Nothing here allocates device memory per call: scratch comes from the
 *     caller through (ws, ws_bytes); pkv_workspace_bytes() gives the size.
 *
 * Cache byte layout (one 64-token page; d = head dim: 128, 256 or 512):
 *   K-layout (K): a token's d/2 code bytes in column blocks of R = min(128, d/2)
 *     bytes, stored [d/(2R)][64 tokens][R] (the K-major operand layout, with
 *     the 128- or 64-byte swizzle, of a block-scaled FP4 tensor-core
 *     contraction: pages are read as stored).  Channel pair (2j, 2j+1) of
 *     token t, q = j/16, w = t%8 (R = 128) or (t/2)%4 (R = 64), is at byte
 *     (q/(R/16))*64*R + t*R + 16*((q%(R/16)) ^ w) + j%16, channel 2j in the
 *     low nibble;
 *     scale [d/128][64][8]: block j of token t at ((j/8)*64 + t)*8 + j%8.
 *   Index-key layout (index keys, d_index = 128): data [64][64]: channel pair j
 *     of token t at t*64 + 16*((j/16) ^ (t & 3)) + j%16; scales as K.
 *   V-layout (V):
 *     data  [d/128][8][128][4]: channel c of token t is nibble t%8 of the
 *           little-endian 32-bit word ((c/128)*8 + t/8)*128 + c%128 (each
 *           128-channel block of a page is one contiguous 4 KB run);
 *     scale [d/16][64]: block j of token t at j*64 + t.
 *   Window: FP8 codes [B][128][d], row-major.  Queries: bf16 [.][H][d].
 *   Outputs: O float32 [.][H][d], LSE float32 [.][H] (natural log; -inf and
 *   O = 0 for an empty entry set).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, k > limit ... */
  PKV_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement */
  PKV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  PKV_ERR_BAD_PAGE = 4,      /* device: page id out of range / length beyond page table */
  PKV_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up */
  PKV_ERR_WORKSPACE = 6      /* ws_bytes smaller than pkv_workspace_bytes() */
} pkv_status;

typedef struct pkv_ctx pkv_ctx;

/* Shapes fixed for the life of a context. */
typedef struct {
  int d;              /* head dim of K, V and Q (d_qk = d_v): 128, 256 or 512 */
  int n_heads;        /* query heads sharing the KV: 1..64 */
  int page_size;      /* tokens per page: must be 64 */
  int window;         /* sliding-window entries: must be 128 */
  int d_index;        /* index-key width: must be 128 */
  int n_index_heads;  /* index heads: 1..64 */
} pkv_config;

/* One paged NVFP4 K/V cache (pools indexed by physical page id). */
typedef struct {
  uint8_t* k_data;    /* [num_pages][64*d/2]  K-layout */
  uint8_t* k_scale;   /* [num_pages][64*d/16] K-layout */
  uint8_t* v_data;    /* [num_pages][64*d/2]  V-layout */
  uint8_t* v_scale;   /* [num_pages][64*d/16] V-layout */
  int num_pages;
  float ts_k;         /* FP32 tensor scales, > 0, fixed when the cache is created */
  float ts_v;
} pkv_kv_cache;

/* Paged NVFP4 index keys (d_index channels, index-key layout). */
typedef struct {
  uint8_t* data;      /* [num_pages][64*d_index/2] */
  uint8_t* scale;     /* [num_pages][64*d_index/16] */
  int num_pages;
  float ts;
} pkv_idx_cache;

/* FP8 (E4M3) window K/V. */
typedef struct {
  const uint8_t* k;   /* [B][128][d] */
  const uint8_t* v;   /* [B][128][d] */
  float tw_k;         /* FP32 tensor scales, > 0 */
  float tw_v;
  const int32_t* win_len;  /* device [B]: valid entries 0..128 (decode only; NULL = 128) */
} pkv_window;

/* Operations for pkv_workspace_bytes. */
enum { PKV_OP_DECODE = 1, PKV_OP_SCORE_TOPK = 2, PKV_OP_REPLAY = 3, PKV_OP_DECODE_SPARSE = 4, PKV_OP_SCORE_CAND = 5 };

/* Create a context on CUDA device `device` (made current for the call).
 * Allocates the context's 4-byte device error word.  Returns
 * PKV_ERR_UNSUPPORTED for shapes outside the config rules above. */
pkv_status pkv_init(const pkv_config* cfg, int device, pkv_ctx** out);
void pkv_destroy(pkv_ctx* ctx);

/* Bytes of scratch (the `ws` argument) an op needs for `batch` sequences.
 * max_len: PKV_OP_DECODE - max_pages*64 of the page table;
 * PKV_OP_REPLAY - max_pages*64 (batch = sequences, 128 queries each);
 * PKV_OP_SCORE_TOPK - max_pages*64 (the score buffer and radix-select state);
 * PKV_OP_SCORE_CAND - n_cand, the candidates per sequence;
 * PKV_OP_DECODE_SPARSE - k, the number of selected positions per sequence
 * (decode over sel_idx: the selected tokens are first gathered into compact
 * pages inside the workspace). */
size_t pkv_workspace_bytes(const pkv_ctx* ctx, int op, int batch, int max_len);

/* NVFP4 quantize + append ("MegaAttention avec KV compressé NVFP4": the cache
 * format; the write side of it).  Token i (K row k_new[i], V row v_new[i],
 * float32 [n][d]) is written at position pos[i] of sequence seq_idx[i]: page
 * page_table[seq_idx[i]*max_pages + pos[i]/64], slot pos[i]%64.  Per block of
 * 16 channels: amax, s = fp32(amax / fp32(6*ts)), scale byte = E4M3(s) (nearest,
 * ties to even, saturating), codes = E2M1(fp32(x / fp32(E4M3[S]*ts))) (nearest,
 * ties to even, |v| >= 6 -> 6, sign kept; all 0 when S = 0).  Entries are
 * independent; two entries with the same (sequence, position) race. */
pkv_status pkv_append_kv(pkv_ctx* ctx, const float* k_new, const float* v_new,
                         const int32_t* seq_idx, const int32_t* pos, int n,
                         const pkv_kv_cache* cache, const int32_t* page_table,
                         int max_pages, void* stream);

/* Same quantize + append for index keys (float32 [n][d_index], index-key layout). */
pkv_status pkv_append_index(pkv_ctx* ctx, const float* k_idx_new, const int32_t* seq_idx,
                            const int32_t* pos, int n, const pkv_idx_cache* icache,
                            const int32_t* page_table, int max_pages, void* stream);

/* FP8 (E4M3) encode with a tensor scale: out[i] = E4M3(fp32(x[i] / tw)),
 * nearest, ties to even, saturating at 448, sign kept.  Used to write the
 * sliding window ("uncompressed FP8") and the FP8 index queries. */
pkv_status pkv_quantize_fp8(const float* x, size_t n, float tw, uint8_t* out, void* stream);

/* Sparse MQA logits + top-k ("Logits MQA creux"): for each sequence b and
 * position t < seq_len[b],
 *   score_t = sum_h w[b][h] * ReLU(tq * ts * (q_idx[b][h] . k_t))
 * with q_idx FP8 [B][n_index_heads][d_index] (scale tq), w float32
 * [B][n_index_heads], keys from `icache` through page_table.  Writes the k
 * positions of highest score (ties: lower position first) to out_idx
 * int32 [B][k] in ascending order, -1 padded when seq_len[b] < k, and the
 * scores to out_score float32 [B][max_pages*64] when not NULL.  1 <= k <= 4096. */
pkv_status pkv_score_topk(pkv_ctx* ctx, const uint8_t* q_idx, float tq, const float* w,
                          const pkv_idx_cache* icache, const int32_t* page_table,
                          int max_pages, const int32_t* seq_len, int B, int k,
                          int32_t* out_idx, float* out_score, void* ws, size_t ws_bytes,
                          void* stream);

/* The same scoring and top-k restricted to a candidate list per sequence (the
 * fixed candidate set of "Logits MQA creux", vLLM blog "Kernels"): only the
 * positions cand[b][0..n_cand) are scored.  cand int32 [B][n_cand], each row
 * strictly ascending and -1 padded at the end; every listed position must have
 * its page in page_table (else the error word is set and the position scores
 * as a zero key).  Writes the k highest-scoring candidates' positions to
 * out_idx int32 [B][k] in ascending order (ties: lower position first), -1
 * padded when a row has fewer than k candidates, and the candidates' scores to
 * out_score float32 [B][n_cand] (entry i = candidate i; unspecified after the
 * last valid one) when not NULL.  1 <= k <= 4096, 1 <= n_cand <= 2^30.
 * Workspace: pkv_workspace_bytes(ctx, PKV_OP_SCORE_CAND, B, n_cand). */
pkv_status pkv_score_topk_cand(pkv_ctx* ctx, const uint8_t* q_idx, float tq, const float* w,
                               const pkv_idx_cache* icache, const int32_t* page_table, int max_pages,
                               const int32_t* cand, int n_cand, int B, int k, int32_t* out_idx,
                               float* out_score, void* ws, size_t ws_bytes, void* stream);

/* Decode attention (flash-decoding split along the sequence + LSE merge).
 * For sequence b, query head h (q bf16 [B][n_heads][d]):
 *   entries = global tokens [0, seq_len[b]) (or, if sel_idx != NULL, the
 *             positions sel_idx[b][0..k), -1 entries skipped) followed by the
 *             window entries [0, win_len[b]);
 *   z = softmax_scale * q.k_hat, O = softmax(z) . v_hat, LSE = ln sum exp z,
 *   k_hat/v_hat the exact dequantized values.  Writes out float32 [B][H][d]
 *   and out_lse float32 [B][H] (may be NULL).
 * The contraction with the NVFP4 keys runs on block-scaled FP4 tensor cores:
 * q enters it as five FP4 terms per head, sigma_h * sum_{t<5} c_t 8^-t with c_t
 * E2M1 codes and sigma_h = max_i |q_h,i| / 4 (error at most sigma_h * 8^-4 / 2
 * per channel); the contraction with the FP8 window keys takes q as two E4M3
 * terms scaled by a power of two per head (exact for a bf16 q).  Each query
 * row is split into its terms once per call, into the workspace.
 * PKV_ERR_UNSUPPORTED when win->tw_v / cache->ts_v lies outside [2^-7, 2^7]
 * (the window's V scale is folded into the f16 softmax weights). */
pkv_status pkv_decode_attn(pkv_ctx* ctx, const void* q_bf16, const pkv_kv_cache* cache,
                           const int32_t* page_table, int max_pages, const int32_t* seq_len,
                           int B, const int32_t* sel_idx, int k, const pkv_window* win,
                           float softmax_scale, float* out, float* out_lse, void* ws,
                           size_t ws_bytes, void* stream);

/* Rotary and FP8-output parameters of the fused decode below. */
typedef struct {
  const int32_t* pos;     /* device [B]: position of each sequence's query token (a row of cos_sin) */
  const float* cos_sin;   /* device [max_pos][rope_dim], 16-byte aligned: per position the cosines of
                             the rope_dim/2 pair angles, then their sines (a serving engine's rotary cache) */
  int max_pos;            /* rows of cos_sin, >= 1 */
  int rope_dim;           /* rotated channels, the last rope_dim of d: a multiple of 8 in [8, d] */
  float out_scale;        /* FP8 output scale: finite, > 0 */
} pkv_rope_fp8;

/* Fused decode ("MegaAttention avec KV compressé NVFP4", vLLM blog "Kernels":
 * query RoPE, attention, inverse RoPE on the output and FP8 conversion in one
 * pass, writing the buffer the output projection reads).  With c_i, s_i the
 * entries i and rope_dim/2 + i of row pos[b] of cos_sin, and pair i the
 * channels (d - rope_dim + 2i, d - rope_dim + 2i + 1) of a head:
 *   q' = q with each pair (x0, x1) -> (x0 c_i - x1 s_i, x0 s_i + x1 c_i);
 *   (O, LSE) = pkv_decode_attn of q' (same entries, sel_idx, window, scale);
 *   O' = O with each pair (y0, y1) -> (y0 c_i + y1 s_i, -y0 s_i + y1 c_i);
 *   out_fp8 uint8 [B][H][d] = E4M3(fp32(O' / out_scale)) (nearest, ties to
 *   even, saturating at 448, sign kept);
 *   out float32 [B][H][d] = O' and out_lse float32 [B][H] when not NULL.
 * Channels outside the rotated part pass through.  q' is a bf16 tensor like
 * q: each rotated value is computed in FP32 (every product, the difference and
 * the sum rounded separately, no fused multiply-add) and rounded to bf16
 * (nearest, ties to even); q' then enters the contractions as the terms of
 * pkv_decode_attn (five FP4 terms; two E4M3 terms for the window, exact).  A position
 * outside [0, max_pos) sets the error
 * word (PKV_ERR_BAD_PAGE: an index out of range) and that row is not rotated.
 * Workspace as pkv_decode_attn.  PKV_ERR_UNSUPPORTED unless the tensor-core
 * kernel takes the shape (n_heads <= 64; tw_v / ts_v within [2^-7, 2^7]). */
pkv_status pkv_decode_attn_fused(pkv_ctx* ctx, const void* q_bf16, const pkv_kv_cache* cache,
                                 const int32_t* page_table, int max_pages, const int32_t* seq_len,
                                 int B, const int32_t* sel_idx, int k, const pkv_window* win,
                                 float softmax_scale, const pkv_rope_fp8* fz, uint8_t* out_fp8,
                                 float* out, float* out_lse, void* ws, size_t ws_bytes, void* stream);

/* Bounded replay ("SWA bounded replay", "Côté encodeur"): for sequence b with
 * prefix length H_b = prefix_len[b] >= 128 and s_b = H_b - 128, query r
 * (q bf16 [B][128][n_heads][d], position s_b + r) attends the global tokens
 * [0, s_b) and the chunk-window entries [0, r] (chunk_win->k/v [B][128][d]:
 * FP8 K/V of positions s_b..H_b-1; win_len ignored).
 * Writes out float32 [B][128][H][d], out_lse float32 [B][128][H] (may be NULL).
 * Query terms and PKV_ERR_UNSUPPORTED as pkv_decode_attn. */
pkv_status pkv_replay_attn(pkv_ctx* ctx, const void* q_bf16, const pkv_kv_cache* cache,
                           const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                           int B, const pkv_window* chunk_win, float softmax_scale,
                           float* out, float* out_lse, void* ws, size_t ws_bytes, void* stream);

/* LSE merge of two partial results over disjoint entry sets (the combine step
 * of flash-decoding; decode merges its global and window segments this way):
 *   lse = ln(e^lse_a + e^lse_b), o = e^(lse_a-lse) o_a + e^(lse_b-lse) o_b,
 * rows x dv float32; a part with lse = -inf has weight 0.  o/lse may alias a. */
pkv_status pkv_merge(const float* o_a, const float* lse_a, const float* o_b,
                     const float* lse_b, float* o, float* lse, int rows, int dv,
                     void* stream);

/* Synchronize `stream`, return and clear the context's device error word
 * (PKV_OK, PKV_ERR_BAD_PAGE or PKV_ERR_TIMEOUT), or PKV_ERR_CUDA. */
pkv_status pkv_get_error(pkv_ctx* ctx, void* stream);

const char* pkv_status_str(pkv_status s);

/* Decode attention without caller-provided scratch (no counterpart in the
 * pages: an interface for callers that cannot allocate device memory, e.g.
 * code running while a CUDA graph is being captured in global mode, where
 * cudaMalloc is prohibited; plugins inside a framework that owns the device
 * memory pool; loops that cannot afford cudaMalloc's implicit synchronization).
 * Same arguments and results as pkv_decode_attn minus (ws, ws_bytes): the
 * split-K scratch is a fixed array of PKV_NOALLOC_SCRATCH_BYTES inside the
 * library image, which every GPU that loads the library holds until exit.
 * Returns PKV_ERR_WORKSPACE when pkv_workspace_bytes(ctx, PKV_OP_DECODE, B,
 * max_len) exceeds that size.  Allocates nothing.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress), so make it
 * before any stream capture.  All calls share the array: calls whose kernels
 * overlap on the GPU race; each call rewrites all scratch it reads. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
pkv_status pkv_decode_attn_noalloc(pkv_ctx* ctx, const void* q_bf16, const pkv_kv_cache* cache,
                                   const int32_t* page_table, int max_pages, const int32_t* seq_len,
                                   int B, const int32_t* sel_idx, int k, const pkv_window* win,
                                   float softmax_scale, float* out, float* out_lse, void* stream);

/* Measurement aids (no counterpart in the pages; used by the benchmark).
 * pkv_set_profile_events: when both are non-NULL cudaEvent_t handles, the next
 * attention call (decode or replay) or scoring call (pkv_score_topk,
 * pkv_score_topk_cand) records `start` on its stream right before its main
 * kernel (attention, or index scoring) and `stop` right after it, then forgets
 * them.
 * pkv_launch_count: number of kernels this context has launched so far.
 * pkv_attn_path: 2 once an attention call has launched the tensor-core
 * (tcgen05) kernels on this context, 0 before (there is no other path). */
pkv_status pkv_set_profile_events(pkv_ctx* ctx, void* start, void* stop);
long long pkv_launch_count(const pkv_ctx* ctx);
int pkv_attn_path(const pkv_ctx* ctx);

/* Testing aid for the failure path (no counterpart in the pages).  Every wait
 * of the attention kernel on another of its roles (a copy landing, an MMA
 * completing, a buffer freed) gives up after wait_limit_cycles SM cycles
 * (default 2^31, about a second): the kernel then records PKV_ERR_TIMEOUT in
 * the error word, stops its roles, waits (bounded the same way) for the copies
 * and MMAs it has in flight, frees its tensor memory and returns.  skip_copy
 * >= 0 makes CTA 0 of the next attention calls leave out its K-tile copy
 * number skip_copy (counted from 0 in the CTA's issue order), so that the wait
 * for it runs out; -1 restores normal operation.  PKV_ERR_INVALID_ARG for a
 * limit below 1000 cycles or skip_copy < -1. */
pkv_status pkv_set_test_hooks(pkv_ctx* ctx, long long wait_limit_cycles, int skip_copy);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
