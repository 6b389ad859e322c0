/*
 * dllm_kv.h -- C ABI of one cached denoising step of a masked diffusion LM
 * on a single GB300 (sm_103a).
 *
 * One denoising step runs, in this order, on one CUDA stream:
 *   kv_refresh   gather the rows of the refresh set, RMSNorm, QKV projection,
 *                RoPE, scatter into the versioned per-layer cache (version = t);
 *   block_attn   the active block's queries attend bidirectionally over the
 *                whole cached sequence (or over the sink + rolling window);
 *   attn_out     residual stream h = x + O . W_o^T;
 *   lmhead_conf  per active row: argmax, top-1 probability and entropy of
 *                softmax(RMSNorm(h) . W_lm^T) with the mask id excluded;
 *                logits never reach memory;
 *   stab_update  Stable-Window-Decoding history push, stability test,
 *                commit, dilation by R, version expiry, and compaction of the
 *                refresh set of the next step.
 *
 * Sources (page title and section):
 *   "LaCache: Exact Caching and Precision-Adaptive Inference for Diffusion
 *     Large Language Models", Problem statement, Methodology 1 (LSM) and 3
 *     (Inference workflow): token-level operators (embedding, normalisation,
 *     QKV projection, RoPE) of unchanged tokens are reused; a block's first
 *     step runs a full forward.
 *   "Stable Window Decoding" page (wmrh.cn/news/51151), 3.1-3.3 and 4.2:
 *     stability over the last K steps with mean top-1 probability > tau,
 *     unstable positions dilated by R.
 *   "Diffusion latent cache with time anchors" page (mhpq.cn/news/1098081),
 *     2.3 and 3.1: every cache entry carries its write step; an entry with
 *     t - version > 2 is rejected.
 *   "Attention Sinks and Where to Cache Them" explainer (wmrh.cn/news/159578),
 *     2.3 and 3.1-3.3: S sink entries plus a rolling window of W entries, a
 *     cache of constant size S + W, positions that never roll.
 *   "I/O-aware KV cache and self-verifying parallel decoding"
 *     (bjdmk.com.cn/news/5926815), 3.1: per-position entropy.
 *
 * Conventions
 *   Pointers named *_dev or documented as device pointers are CUDA device
 *   pointers; every call is asynchronous on `stream` (a cudaStream_t, NULL =
 *   legacy default stream) and never synchronises, except dllm_cache_check
 *   and dllm_state_copy.  The caller owns every input, output and weight;
 *   the library owns only what dllm_cache_init allocates.
 *   Row layout: a dense cache row is r = b * L + pos; every row is d =
 *   n_heads * head_dim contiguous elements, heads contiguous inside a row.
 *   bf16 data is passed as 16-bit patterns (uint16), fp32 as float.
 *   Errors: an invalid argument returns a status != DLLM_OK, launches nothing
 *   and sets a message readable with dllm_last_error().  Problems found on
 *   the device (row or token out of range, a wait that timed out) set bits in
 *   the handle's device error word and skip the item; dllm_cache_check reads
 *   and clears that word.  No kernel traps.
 *   Handles are not thread-safe: one host thread per handle at a time.
 */
#ifndef DLLM_KV_H
#define DLLM_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DLLM_OK = 0,
  DLLM_EINVAL = 1,       /* bad argument: nothing launched */
  DLLM_ENOMEM = 2,       /* device allocation failed in dllm_cache_init */
  DLLM_ECUDA = 3,        /* a CUDA runtime call failed */
  DLLM_EDEVICE = 4,      /* the device error word was set (dllm_cache_check) */
  DLLM_EUNSUPPORTED = 5  /* shape outside what the kernels implement */
} dllm_status;

typedef enum { DLLM_F32 = 0, DLLM_BF16 = 1 } dllm_dtype;

/* device error word bits */
#define DLLM_ERR_ROW      0x1u   /* row index outside [0, rows) */
#define DLLM_ERR_TOKEN    0x2u   /* token id outside [0, vocab) */
#define DLLM_ERR_TIMEOUT  0x4u   /* a bounded wait on a barrier gave up */
#define DLLM_ERR_POS      0x8u   /* position outside the RoPE table */
#define DLLM_ERR_GUARD    0x10u  /* dllm_cache_check found a guard after one of the
                                    handle's buffers overwritten: some kernel
                                    wrote past the end of a buffer */

typedef struct {
  int n_layers;      /* layers with a cache (1 for a single attention layer) */
  int batch;         /* B sequences (1 in streaming mode) */
  int seq_len;       /* L positions of every sequence (dense mode) */
  int n_heads;       /* H */
  int head_dim;      /* dh; bf16 needs 64 or 128, fp32 needs 32, 64 or 128 */
  int dtype;         /* dllm_dtype of weights, caches and activations */
  int sink;          /* S sink entries; > 0 selects streaming mode */
  int window;        /* W rolling entries (streaming mode) */
  int expiry;        /* reject t - version > expiry; < 0 = no expiry */
  float rope_theta;  /* RoPE base, 10000 */
  float rms_eps;     /* RMSNorm epsilon, 1e-6 */
  int swd_K;         /* steps a top-1 token must persist (<= 8) */
  float swd_tau;     /* mean top-1 probability threshold (strict >) */
  int swd_R;         /* dilation radius of unstable positions */
  int block_len;     /* active block length (<= 64); streaming mode ignores it */
  int mask_id;       /* id of the mask token */
  int active_queries;/* 1 (multi-layer denoiser): every active-block row
                        passes through the layers as a query; the row list
                        stab_update writes is the refresh set plus the active
                        block, and kv_refresh rewrites K/V, version and
                        token-at-write only for refresh-set rows */
  int vocab;         /* V: token ids are checked against it; sizes the
                        LM-head workspace */
  int max_pos;       /* RoPE positions (streaming: stream length); 0 = L */
  int ffn;           /* FFN width F of the multi-layer denoiser (0 = none);
                        sizes the FFN workspace */
  int swd_R_min;     /* < 0: the dilation radius is swd_R at every step;
                        else it grows with the block-local step s:
                        R(s) = swd_R_min + floor((swd_R - swd_R_min + 1) s
                        / steps_per_block) ("Stable Window Decoding" 4.4) */
  int steps_per_block; /* Tb, the steps of a block (for the radius schedule) */
  int full_every;    /* > 0: the refresh set of block-local steps s with
                        s % full_every == 0 is every row ("I/O-aware KV cache
                        and self-verifying parallel decoding" 5.1) */
  int gate;          /* refresh criterion of the active block: 0 = the
                        unstable rows dilated by R ("Stable Window Decoding"
                        3.2); 1 = the unstable rows whose cache confidence
                        conf_alpha (1 - H / ln(vocab - 1)) + conf_beta
                        exp(-conf_lambda (t + 1 - version)) is below
                        conf_theta ("I/O-aware KV cache and self-verifying
                        parallel decoding" 3.1); fp32, in that order */
  float conf_alpha, conf_beta, conf_lambda, conf_theta;
  int early_exit;    /* 1: a sequence whose active rows are all stable after
                        a step (not its block's last) ends its block: the
                        block's later steps refresh none of its rows and skip
                        its attention, and when every sequence has ended,
                        W_o and the LM head too ("Stable Window Decoding" 3.2,
                        4.2: "compute all or end"); its argmax, top-1
                        probability and entropy are then unspecified */
  int facache;       /* 1: block_attn keeps the online-softmax state of the
                        key tiles outside the block's window and reuses it
                        while the block and its query tokens are unchanged
                        ("LaCache", Methodology 1, FACache); dense bf16
                        single-layer caches only */
} dllm_cache_cfg;

/* Opaque handle: per-layer Q/K/V cache, versions, the token each row was
   computed from, SWD history and stable flags, RoPE table, device error word
   and the scratch buffers of the kernels. */
typedef struct dllm_cache dllm_cache;

/* Allocate and zero a cache for `cfg` on the current device.  Validates the
   shape (EINVAL / EUNSUPPORTED), allocates with cudaMalloc (ENOMEM).
   *out receives the handle; free it with dllm_cache_free. */
dllm_status dllm_cache_init(const dllm_cache_cfg* cfg, void* stream, dllm_cache** out);

/* Free every buffer of the handle (synchronises the device first). */
dllm_status dllm_cache_free(dllm_cache* c);

/* Reset for a new generation: versions to "never written", token-at-write
   to -1, stable flags and SWD history to zero, error word to zero. */
dllm_status dllm_cache_reset(dllm_cache* c, void* stream);

/* Synchronise `stream`, read and clear the device error word into *err_word
   (may be NULL).  Returns DLLM_EDEVICE if any bit was set. */
dllm_status dllm_cache_check(dllm_cache* c, void* stream, uint32_t* err_word);

/* Message of the last failing call on this host thread ("" if none). */
const char* dllm_last_error(void);

/* Fields for dllm_state_copy (deterministic replay of a step in tests). */
typedef enum {
  /* Q, K, V of `layer`, in the cache's tiled layout: for each sequence b
     (1 in streaming mode) and head h, Lp rows (L, or S + W, rounded up to
     64) in tiles of 64; a tile holds head_dim * elem / 128 sub-tiles of 64
     rows x 128 bytes, and the 16-byte chunk c of row r of a sub-tile sits at
     chunk c ^ (r % 8).  Row pos of (b, h) is in tile (b * H + h) * Lp/64 +
     pos / 64.  Streaming mode indexes rows by ring slot. */
  DLLM_FIELD_Q = 0, DLLM_FIELD_K = 1, DLLM_FIELD_V = 2,
  DLLM_FIELD_VERSION = 3,   /* int32 [n_layers][B*L] */
  DLLM_FIELD_TOK_W = 4,     /* int32 [B*L]: token each row was computed from */
  DLLM_FIELD_STABLE = 5,    /* uint8 [B*L] */
  DLLM_FIELD_HIST_TOK = 6,  /* int32 [B][block_len][swd_K] ring of top-1 ids */
  DLLM_FIELD_HIST_P = 7,    /* float [B][block_len][swd_K] ring of top-1 probs */
  DLLM_FIELD_HIST_N = 8,    /* int32 [B][block_len] records pushed this block */
  DLLM_FIELD_FA_REBUILT = 9, /* int32 [1]: (sequence, head) attention states
                               rebuilt since the last reset (facache) */
  DLLM_FIELD_SEQ_DONE = 10, /* uint8 [B]: sequences whose block has ended
                               (early_exit) */
  /* int32 [4096][B][4], dense caches: for global step t (the t passed to
     stab_update, t < 4096) and sequence b, the counts stab_update found:
     rows of the next refresh set, stable rows of the active block, rows
     refreshed because their version expired, rows committed at this step
     (stable now, or forced at the block's last step) - the stability curve
     of [SWD] 4.4.  Zero for steps not run since the last reset. */
  DLLM_FIELD_STEP_STATS = 11
} dllm_field;

/* Blocking copy of one state field between the handle and HOST memory
   `host` (to_device = 1: host -> handle).  `bytes` must equal the field's
   size; *bytes_out (may be NULL) receives it. */
dllm_status dllm_state_copy(dllm_cache* c, int field, int layer, void* host, size_t bytes,
                            int to_device, size_t* bytes_out);

/* --- the step --------------------------------------------------------- */

/* Full refresh set of a block's first step ("LaCache", Inference workflow):
   every row b * L + pos of every sequence, ascending.
   rows_dev: int32 [B*L] device; n_rows_dev: int32 [1] device. */
dllm_status refresh_all(dllm_cache* c, int q_start, int32_t* rows_dev, int32_t* n_rows_dev,
                        void* stream);

/* Rows rows_dev[0 .. *n_rows_dev) (device count, never read by the host)
   are recomputed for layer `layer` ("LaCache", LSM: RoPECache holds the
   normalised hidden state after QKV projection and RoPE):
     x_i = x_dev[i] if x_dev != NULL (compact [n][d] layer input, i.e. the
           hidden state of row rows_dev[i]), else embed_dev[tok_dev[row]];
     [q k v] = RMSNorm(x_i) . W_qkv^T, W_qkv [3d][d] row-major;
     q, k rotated by RoPE at the row's position; stored into the layer's
     Q/K/V cache row; version[layer][row] = t; for layer 0 the token is
     recorded as the row's token-at-write.
   Dense mode: row = b * L + pos.  Streaming mode: row = stream index n,
   tok_dev is the stream, the entry goes to ring slot n (n < S) or
   S + (n - S) mod W, and RoPE uses position n.
   rows_dev == NULL means every dense row 0 .. B*L-1 (n_rows_dev ignored).
   At most B*L rows (dense) or S + W rows (streaming) per call; a larger
   device count sets DLLM_ERR_ROW and only the first rows are refreshed.
   A caller-given x_dev must hold that many rows (only the first *n_rows
   are used).  Out-of-range rows / tokens set the error word and are
   skipped. */
dllm_status kv_refresh(dllm_cache* c, int layer, const void* x_dev, const int32_t* tok_dev,
                       const void* embed_dev, const void* w_qkv_dev, const int32_t* rows_dev,
                       const int32_t* n_rows_dev, int t, void* stream);

/* Streaming pre-projection ("Attention Sinks and Where to Cache Them" 3.3:
   a token's entry depends only on its token and its absolute position, so
   the layer's Q/K/V of every stream token can be projected at once):
   stream tokens 0 .. n-1 (tok_dev[i], position i) -> embedding, RMSNorm,
   [q k v] = x W_qkv^T, RoPE at position i, stored row-major into
   staged_dev [n][3 * d] (q | k | v, heads contiguous) in the cache dtype,
   caller-owned.  Streaming caches only; n <= max_pos.  Asynchronous. */
dllm_status kv_project(dllm_cache* c, int layer, const int32_t* tok_dev, const void* embed_dev,
                       const void* w_qkv_dev, int n, void* staged_dev, void* stream);

/* Stream tokens n0 .. n0 + count - 1 join the sink + rolling cache: their
   staged rows (row n of staged_dev, as kv_project writes them) are copied
   into ring slot n (n < S) or S + (n - S) mod W of `layer`, in order.  A
   call takes at most W tokens (a later token may reuse an earlier one's
   slot).  Asynchronous on `stream`. */
dllm_status ring_append(dllm_cache* c, int layer, const void* staged_dev, int n0, int count, void* stream);

/* Bidirectional attention of cached queries over the cached sequence
   ("LaCache", Problem statement: a block's tokens are updated together over
   the full context; no causal mask):
   dense: queries are positions [q_start, q_start + q_len) of every sequence,
     keys/values all L positions; out_dev [B][q_len][d].
   streaming: the query is stream token n = q_start (q_len = 1), keys/values
     the min(n + 1, S + W) entries the ring holds; out_dev [1][d].
   Split-KV with an online-softmax merge; scratch owned by the handle.
   With cfg.facache (layer 0): the key tiles that [q_start - swd_R,
   q_start + q_len + swd_R) touches form the window; the online-softmax state
   (m, l, O~) of each (sequence, head, query) over all other tiles is kept
   with the block start, q_len and the queries' token-at-write, and while
   they are unchanged only the window's tiles are read and merged with it;
   otherwise every tile is read and the state rebuilt.  The result equals the
   plain attention up to fp32 rounding order. */
dllm_status block_attn(dllm_cache* c, int layer, int q_start, int q_len, void* out_dev,
                       void* stream);

/* Same attention for an explicit query row list (the multi-layer denoiser's
   rows that pass through every layer, [LaCache] "Inference workflow"; the
   queries are the refreshed rows, so the Q cache holds them):
   q_rows_dev[0 .. *n_q_dev) flat rows b * L + pos in ascending order (as
   stab_update and refresh_all write them), device int32; each query attends
   over all L positions of its own sequence in layer `layer`.
   out_dev [n][d] bf16, row i = query q_rows_dev[i], caller-owned.
   bf16 caches and batch <= 256 only (EUNSUPPORTED otherwise); rows outside
   [0, B*L) are skipped.  Asynchronous on `stream`. */
dllm_status block_attn_rows(dllm_cache* c, int layer, const int32_t* q_rows_dev,
                            const int32_t* n_q_dev, void* out_dev, void* stream);

/* The active block's rows out of a compact row-list buffer (no counterpart
   on the pages; plumbing of the multi-layer step): dst_dev[b * q_len + j] =
   src_dev[i] for the i with rows_dev[i] == b * L + q_start + j, for
   b < batch, j < q_len.  src_dev [*n_rows_dev][d] and dst_dev [B*q_len][d]
   in the cache dtype, caller-owned, 16-byte aligned; rows_dev sorted
   ascending.  A row missing from the list sets DLLM_ERR_ROW and its output
   row is zero.  Asynchronous on `stream`. */
dllm_status active_rows(dllm_cache* c, const void* src_dev, const int32_t* rows_dev,
                        const int32_t* n_rows_dev, int q_start, int q_len, void* dst_dev,
                        void* stream);

/* Residual stream after attention: h_dev[i] = x_i + o_dev[i] . W_o^T for
   i < M (M = B * q_len rows, row i = sequence i / q_len, position
   q_start + i % q_len), W_o [d][d] row-major.  x_i = x_res_dev[i] if given,
   else embed_dev[tok_dev[b * L + q_start + i % q_len]].
   m_dev (device int32, may be NULL) overrides M with a device count (at most
   B*L; o_dev, x_res_dev and h_dev then hold B*L rows).  With m_dev and no
   x_res_dev, x_i is row i of the layer-0 input the last kv_refresh gathered
   (the embeddings of its row list, compact). */
dllm_status attn_out(dllm_cache* c, const void* o_dev, const void* w_o_dev, const void* x_res_dev,
                     const int32_t* tok_dev, const void* embed_dev, int q_start, int q_len,
                     const int32_t* m_dev, void* h_dev, void* stream);

/* FFN of the multi-layer denoiser: out_dev[i] = h_i + W2 . GELU(W1 .
   RMSNorm(h_i)), W1 [F][d], W2 [d][F], exact (erf) GELU, the GELU output
   stored in the cache dtype.  M rows, or *m_dev if m_dev != NULL. */
dllm_status ffn_gelu(dllm_cache* c, const void* h_dev, const void* w1_dev, const void* w2_dev,
                     int F, int M, const int32_t* m_dev, void* out_dev, void* stream);

/* Fused LM head + confidence for M rows of h_dev [M][d]:
     logits = RMSNorm(h_i) . W_lm^T (W_lm [V][d]), logit[mask_id] excluded;
     argmax_dev[i] = first index of the largest logit,
     p_top1_dev[i] = its softmax probability,
     entropy_dev[i] = -sum p ln p.
   ("Stable Window Decoding" 3.1; "I/O-aware KV cache ..." 3.1.)
   Per vocab tile the epilogue reduces (max, argmax, sum e^(l-max),
   sum e^(l-max)(l-max)) from the accumulator; a merge kernel combines the
   tiles.  Logits are never written.  M <= B * block_len. */
dllm_status lmhead_conf(dllm_cache* c, const void* h_dev, const void* w_lm_dev, int M, int V,
                        int d, int mask_id, int32_t* argmax_dev, float* p_top1_dev,
                        float* entropy_dev, void* stream);

/* SWD update of the active block [q_start, q_start + block_len) of every
   sequence, then the refresh set of step t + 1 ("Stable Window Decoding"
   3.1-3.3, 4.2; "Diffusion latent cache with time anchors" 2.3):
     every active position not yet stable pushes (argmax, p_top1) into its
     ring of the last K; it becomes stable when K records exist, all K ids are
     equal and their mean (fp32, oldest to newest, / K) > tau; a position that
     becomes stable commits tok = argmax; stable positions are skipped.
     last_step != 0: every still-unstable active position commits its argmax,
     the history is cleared, and the next refresh set is the full set of the
     next block (as refresh_all(q_start + block_len)).
     Otherwise, with s = step_in_block (the block-local index of the step
     just run): if cfg.full_every > 0 and (s + 1) % full_every == 0 every
     row; else rows = dilate_R(unstable active) U {tok != token-at-write}
       U {(t + 1) - version > expiry}, R = the radius of step s + 1 (see
       cfg.swd_R_min), ascending b * L + pos; with
     active_queries the list also holds every active row (the refresh set
     itself stays in the handle and gates kv_refresh's K/V writes).
   With cfg.gate = 1 the dilated window is replaced by the unstable rows
   whose cache confidence is below conf_theta (entropy_dev then required).
   argmax_dev / p_top1_dev / entropy_dev: [B * block_len] device; tok_dev
   [B][L] device, updated in place; rows_dev [B * L], n_rows_dev [1] device
   outputs. */
dllm_status stab_update(dllm_cache* c, const int32_t* argmax_dev, const float* p_top1_dev,
                        const float* entropy_dev, int32_t* tok_dev, int q_start, int t, int step_in_block,
                        int last_step, int32_t* rows_dev, int32_t* n_rows_dev, void* stream);

/* --- without device allocation ---------------------------------------- */

/* lmhead_conf for callers that cannot call cudaMalloc: the same computation
   and kernels, no handle, and no allocation by the library.  (This entry
   point has no counterpart in the pages; it serves hosts such as a serving
   engine whose memory planner owns every device byte, code that must not hit
   cudaMalloc's implicit device synchronisation, or a caller that has no
   dllm_cache handle.)  The caller passes inputs and outputs as for
   lmhead_conf, plus the storage dtype and the RMSNorm epsilon.
   Scratch lives in one static device array of 4 MiB + 1.25 KiB that every GPU
   which loads the library keeps until the process exits; it bounds a call to
   M <= 256 rows and V <= 131072 (larger sizes return DLLM_EINVAL); d must
   be a multiple of 64.  There is no handle to hold a device error word: if a
   bounded wait inside the kernels gives up, the affected rows come back with
   argmax -1 and NaN top-1 probability and entropy.  The first
   call on a device resolves the array's address on that device (the device
   must be current); make that first call before any stream capture.  Every
   call shares the array and leaves its contents behind: calls whose kernels
   overlap on the GPU (different streams, or several host threads) race.
   The call allocates nothing: no cudaMalloc, cudaFree, or allocating library
   routine. */
dllm_status lmhead_conf_noalloc(const void* h_dev, const void* w_lm_dev, int M, int V, int d, int dtype,
                                int mask_id, float rms_eps, int32_t* argmax_dev, float* p_top1_dev,
                                float* entropy_dev, void* stream);

/* --- diagnostics ------------------------------------------------------ */

/* Exercise the bounded wait that every kernel's barrier waits use (no
   counterpart on the pages; it tests the failure path without faulting the
   GPU): one CTA waits on a shared-memory barrier that nothing arrives on,
   gives up after limit_ns nanoseconds (1e3 .. 2e9; the kernels' own limit is
   2 s), sets DLLM_ERR_TIMEOUT in the handle's error word and raises the
   CTA's abort flag, through which its other waiting warps leave; every
   thread then returns normally and the context stays usable.  Asynchronous
   on `stream`; read the result with dllm_cache_check. */
dllm_status dllm_wait_selftest(dllm_cache* c, uint64_t limit_ns, void* stream);

/* --- measurement ------------------------------------------------------ */

/* Kernels that dllm_profile_events can bracket. */
typedef enum {
  DLLM_PROF_QKV_GEMM = 1,   /* projection GEMM of kv_refresh */
  DLLM_PROF_ATTN = 2,       /* attention kernel of block_attn */
  DLLM_PROF_LM_GEMM = 3,    /* fused LM-head GEMM of lmhead_conf */
  DLLM_PROF_OUT_GEMM = 4,   /* output-projection GEMM of attn_out */
  DLLM_PROF_FFN = 5         /* row norm and both GEMMs of ffn_gelu */
} dllm_prof_kernel;

/* Record the CUDA events ev_begin / ev_end (cudaEvent_t, created by the
   caller with timing enabled) on the call's stream immediately before and
   after the next launches of `kernel`, until changed; NULL events clear the
   hook.  Under stream capture the records become graph nodes, so a captured
   generation can time one kernel per step. */
dllm_status dllm_profile_events(dllm_cache* c, int kernel, void* ev_begin, void* ev_end);

#ifdef __cplusplus
}
#endif

#endif /* DLLM_KV_H */
