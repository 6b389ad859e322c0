// Host-side internals shared by the translation units of libdllmkv.
#pragma once
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "dllm_kv.h"
#include "kv_layout.h"

struct dllm_cache {
  dllm_cache_cfg cfg;
  int device = 0;
  int num_sms = 0;
  int d = 0;            // n_heads * head_dim
  int rows = 0;         // cache rows per layer: B*L (dense) or S+W (streaming)
  int seq_rows = 0;     // B*L for bookkeeping arrays (dense), S+W streaming
  int max_pos = 0;      // RoPE table rows
  int Lw = 0;           // 32-position words per sequence
  size_t elem = 2;      // bytes per element of the cache dtype
  dllm::KvLayout kv{};  // tiled layout of every layer's Q/K/V cache
  size_t kv_layer_bytes = 0;
  // state
  void* q = nullptr;    // [n_layers] x tiled layout (kv), B (or 1) sequences
  void* k = nullptr;
  void* v = nullptr;
  int* version = nullptr;   // [n_layers][seq_rows]
  int* tok_w = nullptr;     // [seq_rows]
  uint8_t* stable = nullptr;
  int* hist_tok = nullptr;  // [B][blk][K]
  float* hist_p = nullptr;
  int* hist_n = nullptr;    // [B][blk]
  uint32_t* words = nullptr;// [B][Lw] refresh flags
  float2* rope = nullptr;   // [head_dim/2] RoPE frequencies as (hi, lo) float pairs
  unsigned* err = nullptr;  // device error word
  unsigned* ticket = nullptr; // arrival counter of the SWD kernel's blocks
  // scratch
  void* X = nullptr;        // gathered layer inputs [seq_rows][d]
  float* rs = nullptr;      // RMS scales [seq_rows]
  void* lm_part = nullptr;  // [B*blk][ceil(V/128)] LMPart
  float* lm_rs = nullptr;   // [B*blk]
  int lm_rows_cap = 0, lm_tiles_cap = 0;
  void* ffn_buf = nullptr;  // [seq_rows][ffn]
  int ffn_cap = 0;
  // kept online-softmax state of the unchanged key tiles (cfg.facache)
  float* fa_state = nullptr;  // [B][H][64][head_dim + 4]: O~, m (log2 domain), l
  int* fa_key = nullptr;      // [B][H][66]: block start, block length, token-at-write of the queries
  int* fa_rebuilt = nullptr;  // (sequence, head) states rebuilt since the last reset
  // early block exit: sequences whose block has ended, and the row count of
  // W_o and the LM head (B * block_len, or 0 once every sequence has ended)
  uint8_t* seq_done = nullptr;  // [B]
  int* m_live = nullptr;        // [1]
  // per-step stability counters of the dense step (the stability curve):
  // [kStatsSteps][B][4] = (refresh rows, stable rows, expired rows,
  // committed rows) of sequence b at global step t
  int* stats = nullptr;
  // guard bytes after every buffer above (a fixed pattern that
  // dllm_cache_check verifies): the device addresses, and a device copy of
  // the list
  std::vector<void*> guards;
  void** guard_dev = nullptr;
  // measurement hook: events bracketing a kernel (index = dllm_prof_kernel)
  cudaEvent_t prof_begin[8] = {};
  cudaEvent_t prof_end[8] = {};
};

namespace dllm {

constexpr int kStatsSteps = 4096;   // global steps the stability counters record

void set_error(const std::string& msg);

// Record the measurement hook's events around one launch.  Under stream
// capture a plain event record only orders streams; the external flag makes
// it an event-record node that the graph timestamps on every replay.
inline void record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}
struct ProfScope {
  cudaEvent_t end;
  cudaStream_t st;
  ProfScope(dllm_cache* c, int k, cudaStream_t s) : end(c->prof_end[k]), st(s) {
    if (c->prof_begin[k]) record_event(c->prof_begin[k], st);
  }
  ~ProfScope() {
    if (end) record_event(end, st);
  }
};

// Early block exit: the ended-sequence flags, or null when it is off.
inline const uint8_t* done_flags(const dllm_cache* c) { return c->cfg.early_exit ? c->seq_done : nullptr; }

// Refresh-set flag words that gate K/V writes: with active queries the row
// list of a step also holds query-only rows (dense mode only).
inline const uint32_t* kv_gate(const dllm_cache* c) {
  return (c->cfg.sink == 0 && c->cfg.active_queries) ? c->words : nullptr;
}

// tensor maps (driver entry point resolved once)
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer, bool bf16);

// gemm_launch.cu -----------------------------------------------------------
// bf16 or fp32 D = A . B^T with the named epilogue.  M: host rows, or the
// device count M_dev (then M_cap bounds the grid and A's row extent).
// stage (streaming pre-projection): rows row0 .. row0 + M_cap - 1 go to the
// row-major staging buffer instead of the cache
cudaError_t gemm_qkv(dllm_cache* c, int layer, const void* A, int M_cap, const int* M_dev, const int* rows,
                     const void* w_qkv, cudaStream_t st, void* stage = nullptr, int row0 = 0);
cudaError_t gemm_resid(dllm_cache* c, const void* A, const void* W, int M, int M_cap, const int* M_dev, int N,
                       int K, const void* xres, const int* tok, const void* embed, int q_start, int q_len,
                       void* out, cudaStream_t st);
cudaError_t gemm_gelu(dllm_cache* c, const void* A, const void* W, int M, int M_cap, const int* M_dev, int N,
                      int K, const float* rs, void* out, cudaStream_t st);
// M_dev (may be null): 0 skips every row, else M rows
cudaError_t gemm_lm(dllm_cache* c, const void* A, const void* W, int M, const int* M_dev, int V, int d,
                    const float* rs, int mask_id, void* part, int n_tiles, cudaStream_t st);
int lm_tile_cols(const dllm_cache* c, int M, int V);
// partial statistics per row of the LM head for M rows and V columns
int lm_slots(const dllm_cache* c, int M, int V);

// attn.cu ------------------------------------------------------------------
// Queries: positions [q_pos0, q_pos0 + q_len) (ring slot in streaming mode)
// of each of n_seq sequences; keys/values: positions [0, kv_len).  out:
// [n_seq][q_len][d] in the cache dtype.
// Launch `kernel` with programmatic stream serialisation (it may start while
// its predecessor on `st` finishes; it calls pdl_wait() before touching
// anything earlier work writes) and, if cluster > 0, clusters of that size
// along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  int n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 0) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Queries = the sorted row list rows[0, *n_rows) (bf16 caches, batch <= 256).
cudaError_t attn_rows_dense(dllm_cache* c, int layer, const int* rows, const int* n_rows, void* out,
                            cudaStream_t st);
cudaError_t launch_active_rows(dllm_cache* c, const void* src, const int* rows, const int* n_rows, int q_start,
                               int q_len, void* dst, cudaStream_t st);
// (the active rows of an ended sequence are skipped without an error)
cudaError_t attn_dense(dllm_cache* c, int layer, int q_pos0, int q_len, int kv_len, int n_seq, void* out,
                       cudaStream_t st);
// Layer-0 attention of the active block with the kept state of the
// unchanged key tiles (bf16, q_len <= 64).
cudaError_t attn_facache(dllm_cache* c, int q_pos0, int q_len, void* out, cudaStream_t st);

// misc.cu ------------------------------------------------------------------
cudaError_t launch_gather(dllm_cache* c, int layer, const int* rows, const int* n_rows, int n_host,
                          const void* x, const int* tok, const void* embed, int t, cudaStream_t st, int row0 = 0);
// Copy stream tokens n0 .. n0 + count - 1 from a row-major staging buffer
// [n][3d] into their ring slots of `layer`.
cudaError_t launch_ring_append(dllm_cache* c, int layer, const void* staged, int n0, int count, cudaStream_t st);
cudaError_t launch_rownorm(dllm_cache* c, const void* h, int M, const int* M_dev, int d, float* rs,
                           cudaStream_t st);
// fail_word: see lm_merge_kernel (null: always merge)
cudaError_t launch_lm_merge(const void* part, int M, const int* M_dev, int n_tiles, int* argmax, float* p1,
                            float* ent, const unsigned* fail_word, cudaStream_t st);
// R: dilation radius of the next step's refresh set; full: the next step
// refreshes every row (the schedules of stab_update)
// ent: the active rows' entropies with the confidence criterion, else null
cudaError_t launch_stab(dllm_cache* c, const int* argmax, const float* p1, const float* ent, int* tok, int q_start,
                        int t, int last, int R, int full, int* rows, int* n_rows, cudaStream_t st);
cudaError_t launch_refresh_all(dllm_cache* c, int q_start, int* rows, int* n_rows, cudaStream_t st);
cudaError_t launch_reset(dllm_cache* c, cudaStream_t st);
cudaError_t launch_wait_selftest(dllm_cache* c, uint64_t limit_ns, cudaStream_t st);

}  // namespace dllm
