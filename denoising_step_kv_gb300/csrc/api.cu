// C ABI of the cached denoising step: argument validation, buffers of the
// handle, the RoPE table, tensor-map encoding, and the entry points.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace dllm {

thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

namespace {

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

dllm_status fail(dllm_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

dllm_status cuda_fail(cudaError_t e, const char* where) {
  return fail(DLLM_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

#define DLLM_CHECK_HANDLE(c)                                     \
  do {                                                           \
    if (!(c)) return fail(DLLM_EINVAL, "null dllm_cache handle"); \
  } while (0)

// An NVTX range around each entry point of the step (host-side: it spans the
// call that enqueues the work; a profiler attached to the process shows the
// step's structure, and without one the calls cost a check of a pointer).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

#define DLLM_LAUNCH(expr, where)                 \
  do {                                           \
    cudaError_t e_ = (expr);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void free_all(dllm_cache* c) {
  void* bufs[] = {c->q, c->k, c->v, c->version, c->tok_w, c->stable, c->hist_tok, c->hist_p, c->hist_n, c->words,
                  c->rope, c->err, c->ticket, c->X, c->rs, c->lm_part, c->lm_rs, c->ffn_buf,
                  c->fa_state, c->fa_key, c->fa_rebuilt, c->seq_done, c->m_live, c->stats, c->guard_dev};
  for (void* b : bufs)
    if (b) cudaFree(b);
}

constexpr unsigned kGuardBytes = 256;     // after every buffer of the handle
constexpr unsigned kGuardByte = 0xA5;

template <typename T>
bool dalloc(dllm_cache* c, T** p, size_t bytes) {
  bytes = (std::max<size_t>(bytes, 16) + 255) / 256 * 256;
  if (cudaMalloc(reinterpret_cast<void**>(p), bytes + kGuardBytes) != cudaSuccess) return false;
  void* g = reinterpret_cast<uint8_t*>(*p) + bytes;
  c->guards.push_back(g);
  return cudaMemset(g, kGuardByte, kGuardBytes) == cudaSuccess;
}

// One CTA per guard: every word must still hold the pattern.
__global__ void guard_kernel(void* const* guards, unsigned* err) {
  const uint32_t* g = static_cast<const uint32_t*>(guards[blockIdx.x]);
  const uint32_t want = 0x01010101u * kGuardByte;
  if (threadIdx.x < kGuardBytes / 4 && g[threadIdx.x] != want) atomicOr(err, DLLM_ERR_GUARD);
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer, bool bf16) {
  EncodeFn fn = encode_fn();
  if (!fn || !aligned16(base) || row_bytes % 16 != 0 || outer == 0 || inner == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, static_cast<cuuint32_t>(std::min<uint64_t>(box_outer, 256))};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dllm

using namespace dllm;

extern "C" {

const char* dllm_last_error(void) { return g_last_error.c_str(); }

dllm_status dllm_cache_init(const dllm_cache_cfg* cfg, void* stream, dllm_cache** out) {
  if (!cfg || !out) return fail(DLLM_EINVAL, "dllm_cache_init: null cfg or out");
  *out = nullptr;
  const dllm_cache_cfg g = *cfg;
  const bool streaming = g.sink > 0;
  if (g.n_layers < 1 || g.batch < 1 || g.n_heads < 1 || g.head_dim < 1 || g.vocab < 1)
    return fail(DLLM_EINVAL, "dllm_cache_init: n_layers, batch, n_heads, head_dim and vocab must be >= 1");
  if (g.dtype != DLLM_F32 && g.dtype != DLLM_BF16) return fail(DLLM_EINVAL, "dllm_cache_init: bad dtype");
  if (streaming) {
    if (g.window < 1 || g.batch != 1 || g.max_pos < 1)
      return fail(DLLM_EINVAL, "dllm_cache_init: streaming needs window >= 1, batch 1 and max_pos >= 1");
  } else {
    if (g.seq_len < 1 || g.block_len < 1 || g.block_len > 64 || g.block_len > g.seq_len)
      return fail(DLLM_EINVAL, "dllm_cache_init: need 1 <= block_len <= min(64, seq_len)");
    if (g.swd_K < 1 || g.swd_K > 8 || g.swd_R < 0)
      return fail(DLLM_EINVAL, "dllm_cache_init: need 1 <= swd_K <= 8 and swd_R >= 0");
    if (g.gate != 0 && g.gate != 1) return fail(DLLM_EINVAL, "dllm_cache_init: gate must be 0 or 1");
    if (g.swd_R_min > g.swd_R || g.full_every < 0 || (g.swd_R_min >= 0 && g.steps_per_block < 1))
      return fail(DLLM_EINVAL, "dllm_cache_init: need swd_R_min <= swd_R, full_every >= 0 and, with a radius "
                               "schedule, steps_per_block >= 1");
    if (static_cast<long long>(g.batch) * g.seq_len > (1LL << 26))
      return fail(DLLM_EUNSUPPORTED, "dllm_cache_init: batch * seq_len above 2^26");
  }
  const int d = g.n_heads * g.head_dim;
  if (g.dtype == DLLM_BF16) {
    if ((g.head_dim != 64 && g.head_dim != 128) || d % 128 != 0)
      return fail(DLLM_EUNSUPPORTED, "dllm_cache_init: bf16 needs head_dim 64 or 128 and d % 128 == 0");
    if (g.ffn % 128 != 0) return fail(DLLM_EUNSUPPORTED, "dllm_cache_init: bf16 needs ffn % 128 == 0");
  } else {
    const bool ok = (d % 128 == 0 && (g.head_dim == 32 || g.head_dim == 64 || g.head_dim == 128)) ||
                    (d % 64 == 0 && (g.head_dim == 32 || g.head_dim == 64));
    if (!ok) return fail(DLLM_EUNSUPPORTED, "dllm_cache_init: fp32 needs head_dim 32/64 (d % 64 == 0) or 128");
    if (g.ffn % 32 != 0) return fail(DLLM_EUNSUPPORTED, "dllm_cache_init: fp32 needs ffn % 32 == 0");
  }
  if (!(g.rope_theta > 0.f) || !(g.rms_eps >= 0.f)) return fail(DLLM_EINVAL, "dllm_cache_init: bad theta/eps");
  if (g.facache && (streaming || g.dtype != DLLM_BF16 || g.n_layers != 1))
    return fail(DLLM_EUNSUPPORTED, "dllm_cache_init: facache needs a dense bf16 single-layer cache");

  dllm_cache* c = new dllm_cache();
  c->cfg = g;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return fail(DLLM_ECUDA, "dllm_cache_init: no CUDA device");
  }
  c->d = d;
  c->elem = g.dtype == DLLM_BF16 ? 2 : 4;
  c->rows = streaming ? g.sink + g.window : g.batch * g.seq_len;
  c->seq_rows = c->rows;
  c->max_pos = g.max_pos > 0 ? g.max_pos : g.seq_len;
  if (!streaming && c->max_pos < g.seq_len) c->max_pos = g.seq_len;
  c->Lw = streaming ? 1 : cdiv(g.seq_len, 32);
  const size_t nl = g.n_layers, sr = c->seq_rows;
  c->kv.H = g.n_heads;
  c->kv.Lp = cdiv(streaming ? g.sink + g.window : g.seq_len, 64) * 64;
  c->kv.row_bytes = static_cast<int>(g.head_dim * c->elem);
  c->kv_layer_bytes = c->kv.layer_bytes(streaming ? 1 : g.batch);
  const int blk = streaming ? 1 : g.block_len;
  const int K = streaming ? 1 : g.swd_K;
  c->lm_rows_cap = g.batch * blk;
  c->lm_tiles_cap = cdiv(g.vocab, 128);
  c->ffn_cap = g.ffn;
  bool ok = dalloc(c, &c->q, nl * c->kv_layer_bytes) && dalloc(c, &c->k, nl * c->kv_layer_bytes) &&
            dalloc(c, &c->v, nl * c->kv_layer_bytes) && dalloc(c, &c->version, nl * sr * sizeof(int)) &&
            dalloc(c, &c->tok_w, sr * sizeof(int)) && dalloc(c, &c->stable, sr) &&
            dalloc(c, &c->hist_tok, static_cast<size_t>(g.batch) * blk * K * sizeof(int)) &&
            dalloc(c, &c->hist_p, static_cast<size_t>(g.batch) * blk * K * sizeof(float)) &&
            dalloc(c, &c->hist_n, static_cast<size_t>(g.batch) * blk * sizeof(int)) &&
            dalloc(c, &c->words, static_cast<size_t>(g.batch) * c->Lw * sizeof(uint32_t)) &&
            dalloc(c, &c->rope, static_cast<size_t>(g.head_dim / 2) * sizeof(float2)) &&
            dalloc(c, &c->err, sizeof(unsigned)) && dalloc(c, &c->ticket, sizeof(unsigned)) && dalloc(c, &c->X, sr * d * c->elem) && dalloc(c, &c->rs, sr * sizeof(float)) &&
            dalloc(c, &c->lm_part, static_cast<size_t>(c->lm_rows_cap) * c->lm_tiles_cap * 16) &&
            dalloc(c, &c->lm_rs, static_cast<size_t>(c->lm_rows_cap) * sizeof(float)) &&
            dalloc(c, &c->ffn_buf, sr * static_cast<size_t>(g.ffn) * c->elem);
  if (ok && !streaming)
    ok = dalloc(c, &c->seq_done, static_cast<size_t>(g.batch)) && dalloc(c, &c->m_live, sizeof(int)) &&
         dalloc(c, &c->stats, static_cast<size_t>(kStatsSteps) * g.batch * 4 * sizeof(int));
  if (ok && g.facache) {
    const size_t bh = static_cast<size_t>(g.batch) * g.n_heads;
    ok = dalloc(c, &c->fa_state, bh * 64 * (g.head_dim + 4) * sizeof(float)) &&
         dalloc(c, &c->fa_key, bh * 66 * sizeof(int)) && dalloc(c, &c->fa_rebuilt, sizeof(int));
  }
  if (ok) {
    ok = cudaMalloc(reinterpret_cast<void**>(&c->guard_dev), c->guards.size() * sizeof(void*)) == cudaSuccess &&
         cudaMemcpy(c->guard_dev, c->guards.data(), c->guards.size() * sizeof(void*), cudaMemcpyHostToDevice) ==
             cudaSuccess;
  }
  if (!ok) {
    free_all(c);
    delete c;
    cudaGetLastError();
    return fail(DLLM_ENOMEM, "dllm_cache_init: cudaMalloc failed");
  }
  // RoPE frequencies theta^(-2i/dh), computed in double on the host and kept
  // as a float pair (hi, lo) so that kernels form pos * f to ~1e-10 relative
  {
    const int half = g.head_dim / 2;
    std::vector<float2> tab(half);
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow(static_cast<double>(g.rope_theta), -2.0 * i / g.head_dim);
      const float hi = static_cast<float>(inv);
      tab[i] = make_float2(hi, static_cast<float>(inv - static_cast<double>(hi)));
    }
    if (cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
      free_all(c);
      delete c;
      return fail(DLLM_ECUDA, "dllm_cache_init: RoPE frequency upload failed");
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t hist = static_cast<size_t>(g.batch) * blk * K;
  if (cudaMemsetAsync(c->q, 0, nl * c->kv_layer_bytes, st) != cudaSuccess ||
      cudaMemsetAsync(c->k, 0, nl * c->kv_layer_bytes, st) != cudaSuccess ||
      cudaMemsetAsync(c->v, 0, nl * c->kv_layer_bytes, st) != cudaSuccess ||
      cudaMemsetAsync(c->ticket, 0, sizeof(unsigned), st) != cudaSuccess ||
      cudaMemsetAsync(c->hist_tok, 0, hist * sizeof(int), st) != cudaSuccess ||
      cudaMemsetAsync(c->hist_p, 0, hist * sizeof(float), st) != cudaSuccess || launch_reset(c, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    free_all(c);
    delete c;
    return fail(DLLM_ECUDA, "dllm_cache_init: reset failed");
  }
  *out = c;
  return DLLM_OK;
}

dllm_status dllm_cache_free(dllm_cache* c) {
  DLLM_CHECK_HANDLE(c);
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
  return DLLM_OK;
}

dllm_status dllm_cache_reset(dllm_cache* c, void* stream) {
  DLLM_CHECK_HANDLE(c);
  DLLM_LAUNCH(launch_reset(c, static_cast<cudaStream_t>(stream)), "dllm_cache_reset");
  return DLLM_OK;
}

dllm_status dllm_cache_check(dllm_cache* c, void* stream, uint32_t* err_word) {
  DLLM_CHECK_HANDLE(c);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!c->guards.empty()) {
    guard_kernel<<<static_cast<unsigned>(c->guards.size()), kGuardBytes / 4, 0, st>>>(c->guard_dev, c->err);
    DLLM_LAUNCH(cudaGetLastError(), "dllm_cache_check: guards");
  }
  DLLM_LAUNCH(cudaStreamSynchronize(st), "dllm_cache_check: synchronize");
  unsigned w = 0;
  DLLM_LAUNCH(cudaMemcpy(&w, c->err, sizeof(w), cudaMemcpyDeviceToHost), "dllm_cache_check: read");
  DLLM_LAUNCH(cudaMemset(c->err, 0, sizeof(unsigned)), "dllm_cache_check: clear");
  if (err_word) *err_word = w;
  if (w) {
    std::string m = "device error word 0x";
    char buf[16];
    snprintf(buf, sizeof(buf), "%x", w);
    m += buf;
    if (w & DLLM_ERR_ROW) m += " (row out of range)";
    if (w & DLLM_ERR_TOKEN) m += " (token out of range)";
    if (w & DLLM_ERR_TIMEOUT) m += " (barrier wait timed out)";
    if (w & DLLM_ERR_POS) m += " (position outside the RoPE table)";
    if (w & DLLM_ERR_GUARD) m += " (a write past the end of a buffer of the handle)";
    return fail(DLLM_EDEVICE, m);
  }
  return DLLM_OK;
}

dllm_status dllm_state_copy(dllm_cache* c, int field, int layer, void* host, size_t bytes, int to_device,
                            size_t* bytes_out) {
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  void* ptr = nullptr;
  size_t size = 0;
  const size_t blk = g.sink > 0 ? 1 : g.block_len, K = g.sink > 0 ? 1 : g.swd_K;
  if (field < 0) return fail(DLLM_EINVAL, "dllm_state_copy: unknown field");
  if (field <= DLLM_FIELD_V) {
    if (layer < 0 || layer >= g.n_layers) return fail(DLLM_EINVAL, "dllm_state_copy: bad layer");
    size = c->kv_layer_bytes;
    void* base = field == DLLM_FIELD_Q ? c->q : field == DLLM_FIELD_K ? c->k : c->v;
    ptr = static_cast<char*>(base) + static_cast<size_t>(layer) * size;
  } else if (field == DLLM_FIELD_VERSION) {
    ptr = c->version;
    size = static_cast<size_t>(g.n_layers) * c->seq_rows * sizeof(int);
  } else if (field == DLLM_FIELD_TOK_W) {
    ptr = c->tok_w;
    size = static_cast<size_t>(c->seq_rows) * sizeof(int);
  } else if (field == DLLM_FIELD_STABLE) {
    ptr = c->stable;
    size = c->seq_rows;
  } else if (field == DLLM_FIELD_HIST_TOK) {
    ptr = c->hist_tok;
    size = g.batch * blk * K * sizeof(int);
  } else if (field == DLLM_FIELD_HIST_P) {
    ptr = c->hist_p;
    size = g.batch * blk * K * sizeof(float);
  } else if (field == DLLM_FIELD_HIST_N) {
    ptr = c->hist_n;
    size = g.batch * blk * sizeof(int);
  } else if (field == DLLM_FIELD_SEQ_DONE) {
    if (!c->seq_done) return fail(DLLM_EINVAL, "dllm_state_copy: streaming caches have no block state");
    ptr = c->seq_done;
    size = g.batch;
  } else if (field == DLLM_FIELD_STEP_STATS) {
    if (!c->stats) return fail(DLLM_EINVAL, "dllm_state_copy: streaming caches have no block state");
    ptr = c->stats;
    size = static_cast<size_t>(kStatsSteps) * g.batch * 4 * sizeof(int);
  } else if (field == DLLM_FIELD_FA_REBUILT) {
    if (!c->fa_rebuilt) return fail(DLLM_EINVAL, "dllm_state_copy: the cache keeps no attention state");
    ptr = c->fa_rebuilt;
    size = sizeof(int);
  } else {
    return fail(DLLM_EINVAL, "dllm_state_copy: unknown field");
  }
  if (bytes_out) *bytes_out = size;
  if (!host) return DLLM_OK;
  if (bytes != size) return fail(DLLM_EINVAL, "dllm_state_copy: byte count does not match the field");
  DLLM_LAUNCH(cudaDeviceSynchronize(), "dllm_state_copy: synchronize");
  DLLM_LAUNCH(cudaMemcpy(to_device ? ptr : host, to_device ? host : ptr, size,
                         to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost),
              "dllm_state_copy");
  return DLLM_OK;
}

dllm_status refresh_all(dllm_cache* c, int q_start, int32_t* rows_dev, int32_t* n_rows_dev, void* stream) {
  const NvtxRange nvtx("refresh_all");
  DLLM_CHECK_HANDLE(c);
  if (c->cfg.sink > 0) return fail(DLLM_EINVAL, "refresh_all: dense mode only");
  if (!rows_dev || !n_rows_dev) return fail(DLLM_EINVAL, "refresh_all: null rows or count");
  DLLM_LAUNCH(launch_refresh_all(c, q_start, rows_dev, n_rows_dev, static_cast<cudaStream_t>(stream)),
              "refresh_all");
  return DLLM_OK;
}

dllm_status kv_refresh(dllm_cache* c, int layer, const void* x_dev, const int32_t* tok_dev, const void* embed_dev,
                       const void* w_qkv_dev, const int32_t* rows_dev, const int32_t* n_rows_dev, int t,
                       void* stream) {
  const NvtxRange nvtx("kv_refresh");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  const bool streaming = g.sink > 0;
  if (layer < 0 || layer >= g.n_layers) return fail(DLLM_EINVAL, "kv_refresh: layer out of range");
  if (!w_qkv_dev) return fail(DLLM_EINVAL, "kv_refresh: null w_qkv");
  if (!x_dev && (!tok_dev || !embed_dev)) return fail(DLLM_EINVAL, "kv_refresh: need x, or tok and embed");
  if (!rows_dev != !n_rows_dev) return fail(DLLM_EINVAL, "kv_refresh: rows and n_rows go together");
  if (streaming && !rows_dev) return fail(DLLM_EINVAL, "kv_refresh: streaming mode needs a row list");
  if (!aligned16(w_qkv_dev) || (x_dev && !aligned16(x_dev)) || (embed_dev && !aligned16(embed_dev)))
    return fail(DLLM_EINVAL, "kv_refresh: pointers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int n_host = rows_dev ? 0 : c->seq_rows;
  DLLM_LAUNCH(launch_gather(c, layer, rows_dev, n_rows_dev, n_host, x_dev, tok_dev, embed_dev, t, st),
              "kv_refresh: gather");
  const void* A = x_dev ? x_dev : c->X;
  {
    ProfScope prof(c, DLLM_PROF_QKV_GEMM, st);
    DLLM_LAUNCH(gemm_qkv(c, layer, A, c->seq_rows, rows_dev ? n_rows_dev : nullptr, rows_dev, w_qkv_dev, st),
                "kv_refresh: projection");
  }
  return DLLM_OK;
}

dllm_status kv_project(dllm_cache* c, int layer, const int32_t* tok_dev, const void* embed_dev, const void* w_qkv_dev,
                       int n, void* staged_dev, void* stream) {
  const NvtxRange nvtx("kv_project");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (g.sink <= 0) return fail(DLLM_EINVAL, "kv_project: streaming caches only");
  if (layer < 0 || layer >= g.n_layers) return fail(DLLM_EINVAL, "kv_project: layer out of range");
  if (!tok_dev || !embed_dev || !w_qkv_dev || !staged_dev) return fail(DLLM_EINVAL, "kv_project: null pointer");
  if (n < 0 || n > c->max_pos) return fail(DLLM_EINVAL, "kv_project: n outside [0, max_pos]");
  if (!aligned16(w_qkv_dev) || !aligned16(embed_dev) || !aligned16(staged_dev))
    return fail(DLLM_EINVAL, "kv_project: pointers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // chunks of the compact buffer's rows: gather (embedding, RMS scale), then
  // the projection with the staging epilogue
  for (int r0 = 0; r0 < n; r0 += c->seq_rows) {
    const int cn = std::min(c->seq_rows, n - r0);
    DLLM_LAUNCH(launch_gather(c, layer, nullptr, nullptr, cn, nullptr, tok_dev, embed_dev, 0, st, r0),
                "kv_project: gather");
    ProfScope prof(c, DLLM_PROF_QKV_GEMM, st);
    DLLM_LAUNCH(gemm_qkv(c, layer, c->X, cn, nullptr, nullptr, w_qkv_dev, st, staged_dev, r0), "kv_project: projection");
  }
  return DLLM_OK;
}

dllm_status ring_append(dllm_cache* c, int layer, const void* staged_dev, int n0, int count, void* stream) {
  const NvtxRange nvtx("ring_append");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (g.sink <= 0) return fail(DLLM_EINVAL, "ring_append: streaming caches only");
  if (layer < 0 || layer >= g.n_layers) return fail(DLLM_EINVAL, "ring_append: layer out of range");
  if (!staged_dev || !aligned16(staged_dev)) return fail(DLLM_EINVAL, "ring_append: staged must be 16-byte aligned");
  if (count < 0 || n0 < 0 || n0 + count > c->max_pos) return fail(DLLM_EINVAL, "ring_append: tokens outside [0, max_pos)");
  if (count > g.window) return fail(DLLM_EINVAL, "ring_append: more tokens than the rolling window in one call");
  DLLM_LAUNCH(launch_ring_append(c, layer, staged_dev, n0, count, static_cast<cudaStream_t>(stream)), "ring_append");
  return DLLM_OK;
}

dllm_status block_attn(dllm_cache* c, int layer, int q_start, int q_len, void* out_dev, void* stream) {
  const NvtxRange nvtx("block_attn");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (layer < 0 || layer >= g.n_layers) return fail(DLLM_EINVAL, "block_attn: layer out of range");
  if (!out_dev) return fail(DLLM_EINVAL, "block_attn: null out");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (g.sink > 0) {
    if (q_len != 1 || q_start < 0 || q_start >= c->max_pos)
      return fail(DLLM_EINVAL, "block_attn: streaming takes one query 0 <= n < max_pos");
    const int slot = q_start < g.sink ? q_start : g.sink + (q_start - g.sink) % g.window;
    const int kv_len = std::min(q_start + 1, g.sink + g.window);
    ProfScope prof(c, DLLM_PROF_ATTN, st);
    DLLM_LAUNCH(attn_dense(c, layer, slot, 1, kv_len, 1, out_dev, st), "block_attn");
    return DLLM_OK;
  }
  if (q_start < 0 || q_len < 1 || q_start + q_len > g.seq_len)
    return fail(DLLM_EINVAL, "block_attn: query range outside the sequence");
  if (g.dtype == DLLM_BF16 && q_len > 64) return fail(DLLM_EUNSUPPORTED, "block_attn: q_len > 64");
  ProfScope prof(c, DLLM_PROF_ATTN, st);
  if (g.facache && layer == 0) {
    DLLM_LAUNCH(attn_facache(c, q_start, q_len, out_dev, st), "block_attn");
    return DLLM_OK;
  }
  DLLM_LAUNCH(attn_dense(c, layer, q_start, q_len, g.seq_len, g.batch, out_dev, st), "block_attn");
  return DLLM_OK;
}

dllm_status block_attn_rows(dllm_cache* c, int layer, const int32_t* q_rows_dev, const int32_t* n_q_dev,
                            void* out_dev, void* stream) {
  const NvtxRange nvtx("block_attn_rows");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (layer < 0 || layer >= g.n_layers) return fail(DLLM_EINVAL, "block_attn_rows: layer out of range");
  if (!q_rows_dev || !n_q_dev || !out_dev) return fail(DLLM_EINVAL, "block_attn_rows: null pointer");
  if (g.sink > 0) return fail(DLLM_EINVAL, "block_attn_rows: dense cache only");
  if (g.dtype != DLLM_BF16) return fail(DLLM_EUNSUPPORTED, "block_attn_rows: bf16 caches only");
  if (g.batch > 256) return fail(DLLM_EUNSUPPORTED, "block_attn_rows: batch above 256");
  if (!aligned16(out_dev)) return fail(DLLM_EINVAL, "block_attn_rows: out must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope prof(c, DLLM_PROF_ATTN, st);
  DLLM_LAUNCH(attn_rows_dense(c, layer, q_rows_dev, n_q_dev, out_dev, st), "block_attn_rows");
  return DLLM_OK;
}

dllm_status active_rows(dllm_cache* c, const void* src_dev, const int32_t* rows_dev, const int32_t* n_rows_dev,
                        int q_start, int q_len, void* dst_dev, void* stream) {
  const NvtxRange nvtx("active_rows");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (!src_dev || !rows_dev || !n_rows_dev || !dst_dev) return fail(DLLM_EINVAL, "active_rows: null pointer");
  if (g.sink > 0) return fail(DLLM_EINVAL, "active_rows: dense cache only");
  if (q_start < 0 || q_len < 1 || q_start + q_len > g.seq_len)
    return fail(DLLM_EINVAL, "active_rows: query range outside the sequence");
  if (!aligned16(src_dev) || !aligned16(dst_dev)) return fail(DLLM_EINVAL, "active_rows: pointers not 16-byte aligned");
  DLLM_LAUNCH(launch_active_rows(c, src_dev, rows_dev, n_rows_dev, q_start, q_len, dst_dev,
                                 static_cast<cudaStream_t>(stream)),
              "active_rows");
  return DLLM_OK;
}

dllm_status attn_out(dllm_cache* c, const void* o_dev, const void* w_o_dev, const void* x_res_dev,
                     const int32_t* tok_dev, const void* embed_dev, int q_start, int q_len, const int32_t* m_dev,
                     void* h_dev, void* stream) {
  const NvtxRange nvtx("attn_out");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (!o_dev || !w_o_dev || !h_dev) return fail(DLLM_EINVAL, "attn_out: null o, w_o or h");
  // with a device row count and no x_res, the residual rows are the compact
  // layer-0 input the last kv_refresh gathered (embeddings of its rows)
  const bool from_gather = !x_res_dev && m_dev;
  if (from_gather) x_res_dev = c->X;
  if (!x_res_dev && (!tok_dev || !embed_dev)) return fail(DLLM_EINVAL, "attn_out: need x_res, or tok and embed");
  if (!x_res_dev && (q_len < 1 || q_start < 0 || q_start + q_len > g.seq_len))
    return fail(DLLM_EINVAL, "attn_out: query range outside the sequence");
  if (!aligned16(o_dev) || !aligned16(w_o_dev) || !aligned16(h_dev))
    return fail(DLLM_EINVAL, "attn_out: pointers must be 16-byte aligned");
  const int M = g.batch * std::max(q_len, 1);
  ProfScope prof(c, DLLM_PROF_OUT_GEMM, static_cast<cudaStream_t>(stream));
  if (!m_dev && g.early_exit && g.sink == 0 && q_len == g.block_len) {
    // the active block's rows: none once every sequence has ended its block
    DLLM_LAUNCH(gemm_resid(c, o_dev, w_o_dev, M, M, c->m_live, c->d, c->d, x_res_dev, tok_dev, embed_dev, q_start,
                           q_len, h_dev, static_cast<cudaStream_t>(stream)),
                "attn_out");
    return DLLM_OK;
  }
  DLLM_LAUNCH(gemm_resid(c, o_dev, w_o_dev, M, c->seq_rows, m_dev, c->d, c->d, x_res_dev, tok_dev, embed_dev,
                         q_start, std::max(q_len, 1), h_dev, static_cast<cudaStream_t>(stream)),
              "attn_out");
  return DLLM_OK;
}

dllm_status ffn_gelu(dllm_cache* c, const void* h_dev, const void* w1_dev, const void* w2_dev, int F, int M,
                     const int32_t* m_dev, void* out_dev, void* stream) {
  const NvtxRange nvtx("ffn_gelu");
  DLLM_CHECK_HANDLE(c);
  if (!h_dev || !w1_dev || !w2_dev || !out_dev) return fail(DLLM_EINVAL, "ffn_gelu: null pointer");
  if (F != c->ffn_cap || F <= 0) return fail(DLLM_EINVAL, "ffn_gelu: F must equal the cache's ffn");
  if (!m_dev && (M < 0 || M > c->seq_rows)) return fail(DLLM_EINVAL, "ffn_gelu: M outside [0, B*L]");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int cap = m_dev ? c->seq_rows : M;
  ProfScope prof(c, DLLM_PROF_FFN, st);
  DLLM_LAUNCH(launch_rownorm(c, h_dev, cap, m_dev, c->d, c->rs, st), "ffn_gelu: norm");
  DLLM_LAUNCH(gemm_gelu(c, h_dev, w1_dev, M, c->seq_rows, m_dev, F, c->d, c->rs, c->ffn_buf, st), "ffn_gelu: W1");
  DLLM_LAUNCH(gemm_resid(c, c->ffn_buf, w2_dev, M, c->seq_rows, m_dev, c->d, F, h_dev, nullptr, nullptr, 0, 1,
                         out_dev, st),
              "ffn_gelu: W2");
  return DLLM_OK;
}

dllm_status lmhead_conf(dllm_cache* c, const void* h_dev, const void* w_lm_dev, int M, int V, int d, int mask_id,
                        int32_t* argmax_dev, float* p_top1_dev, float* entropy_dev, void* stream) {
  const NvtxRange nvtx("lmhead_conf");
  DLLM_CHECK_HANDLE(c);
  if (!h_dev || !w_lm_dev || !argmax_dev || !p_top1_dev || !entropy_dev)
    return fail(DLLM_EINVAL, "lmhead_conf: null pointer");
  if (M < 0 || M > c->lm_rows_cap) return fail(DLLM_EINVAL, "lmhead_conf: M outside [0, batch * block_len]");
  if (V < 2 || V > c->cfg.vocab) return fail(DLLM_EINVAL, "lmhead_conf: V outside [2, vocab]");
  if (d != c->d) return fail(DLLM_EINVAL, "lmhead_conf: d must equal n_heads * head_dim");
  if (mask_id >= V) return fail(DLLM_EINVAL, "lmhead_conf: mask_id >= V");
  if (!aligned16(h_dev) || !aligned16(w_lm_dev)) return fail(DLLM_EINVAL, "lmhead_conf: pointers not 16-byte aligned");
  if (M == 0) return DLLM_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int n_tiles = lm_slots(c, M, V);
  // with early exit, a device count: 0 once every sequence has ended its block
  const int* M_dev = (c->cfg.early_exit && c->m_live && M == c->lm_rows_cap) ? c->m_live : nullptr;
  DLLM_LAUNCH(launch_rownorm(c, h_dev, M, M_dev, d, c->lm_rs, st), "lmhead_conf: norm");
  {
    ProfScope prof(c, DLLM_PROF_LM_GEMM, st);
    DLLM_LAUNCH(gemm_lm(c, h_dev, w_lm_dev, M, M_dev, V, d, c->lm_rs, mask_id, c->lm_part, n_tiles, st),
                "lmhead_conf: gemm");
  }
  DLLM_LAUNCH(launch_lm_merge(c->lm_part, M, M_dev, n_tiles, argmax_dev, p_top1_dev, entropy_dev, nullptr, st),
              "lmhead_conf: merge");
  return DLLM_OK;
}

dllm_status stab_update(dllm_cache* c, const int32_t* argmax_dev, const float* p_top1_dev, const float* entropy_dev,
                        int32_t* tok_dev, int q_start, int t, int step_in_block, int last_step, int32_t* rows_dev,
                        int32_t* n_rows_dev, void* stream) {
  const NvtxRange nvtx("stab_update");
  DLLM_CHECK_HANDLE(c);
  const dllm_cache_cfg& g = c->cfg;
  if (g.sink > 0) return fail(DLLM_EINVAL, "stab_update: dense mode only");
  if (!argmax_dev || !p_top1_dev || !tok_dev || !rows_dev || !n_rows_dev)
    return fail(DLLM_EINVAL, "stab_update: null pointer");
  if (q_start < 0 || q_start + g.block_len > g.seq_len)
    return fail(DLLM_EINVAL, "stab_update: active block outside the sequence");
  if (step_in_block < 0) return fail(DLLM_EINVAL, "stab_update: step_in_block < 0");
  if (g.gate == 1 && !entropy_dev) return fail(DLLM_EINVAL, "stab_update: the confidence criterion needs entropy");
  // the schedules of the next step's refresh set
  const int s1 = step_in_block + 1;
  int R_next = g.swd_R;
  if (g.swd_R_min >= 0 && g.steps_per_block > 0)
    R_next = std::min(g.swd_R, g.swd_R_min + ((g.swd_R - g.swd_R_min + 1) * s1) / g.steps_per_block);
  const int full_next = (g.full_every > 0 && s1 % g.full_every == 0) ? 1 : 0;
  DLLM_LAUNCH(launch_stab(c, argmax_dev, p_top1_dev, g.gate == 1 ? entropy_dev : nullptr, tok_dev, q_start, t,
                          last_step ? 1 : 0, g.gate == 1 ? 0 : R_next, full_next, rows_dev, n_rows_dev,
                          static_cast<cudaStream_t>(stream)),
              "stab_update");
  return DLLM_OK;
}

dllm_status dllm_wait_selftest(dllm_cache* c, uint64_t limit_ns, void* stream) {
  DLLM_CHECK_HANDLE(c);
  if (limit_ns < 1000 || limit_ns > 2000000000ull)
    return fail(DLLM_EINVAL, "dllm_wait_selftest: limit_ns outside [1e3, 2e9]");
  DLLM_LAUNCH(launch_wait_selftest(c, limit_ns, static_cast<cudaStream_t>(stream)), "dllm_wait_selftest");
  return DLLM_OK;
}

dllm_status dllm_profile_events(dllm_cache* c, int kernel, void* ev_begin, void* ev_end) {
  DLLM_CHECK_HANDLE(c);
  if (kernel < DLLM_PROF_QKV_GEMM || kernel > DLLM_PROF_FFN)
    return fail(DLLM_EINVAL, "dllm_profile_events: unknown kernel");
  if (!ev_begin != !ev_end) return fail(DLLM_EINVAL, "dllm_profile_events: give both events or neither");
  c->prof_begin[kernel] = static_cast<cudaEvent_t>(ev_begin);
  c->prof_end[kernel] = static_cast<cudaEvent_t>(ev_end);
  return DLLM_OK;
}

}  // extern "C"
