// Instantiations and launchers of the projection GEMMs.
#include <algorithm>

#include "epilogue.cuh"
#include "gemm.cuh"
#include "internal.h"

namespace dllm {
namespace {


template <class Epi, int STAGES>
cudaError_t launch_persistent(dllm_cache* c, const CUtensorMap& ta, const CUtensorMap& tb, int a_rows, int M_host,
                              const int* M_dev, int M_min, int N, int K, const Epi& epi, cudaStream_t st) {
  constexpr size_t smem = tc::smem_bytes<STAGES>();
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, tc::gemm_tc_kernel<Epi, STAGES>, smem);
    if (e != cudaSuccess) return e;
  }
  const int m_rows = M_dev ? a_rows : M_host;
  const int tiles = cdiv(m_rows, tc::BM) * cdiv(N, tc::BN);
  const int per_sm = STAGES <= 3 ? 2 : 1;
  const int grid = std::max(1, std::min(tiles, per_sm * c->num_sms));
  return launch_ex(tc::gemm_tc_kernel<Epi, STAGES>, dim3(grid), dim3(tc::THREADS), smem, st, 0, ta, tb, M_host, M_dev,
                   a_rows, M_min, N, K, epi, c->err);
}

template <class Epi, int STAGES>
cudaError_t launch_pair(dllm_cache* c, const CUtensorMap& ta, const CUtensorMap& tb, int a_rows, int M_host,
                        const int* M_dev, int M_min, int N, int K, const Epi& epi, cudaStream_t st) {
  constexpr size_t smem = tc::pair_smem_bytes<STAGES>();
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, tc::gemm_pair_kernel<Epi, STAGES>, smem);
    if (e != cudaSuccess) return e;
  }
  const int m_rows = M_dev ? a_rows : M_host;
  const int pairs = cdiv(cdiv(m_rows, tc::BM), 2) * cdiv(N, tc::PBN);
  const int clusters = std::max(1, std::min(pairs, c->num_sms / 2));
  return launch_ex(tc::gemm_pair_kernel<Epi, STAGES>, dim3(2 * clusters), dim3(tc::THREADS), smem, st, 2, ta, tb,
                   M_host, M_dev, a_rows, M_min, N, K, epi, c->err);
}

template <class Epi, int STAGES, int CS, int SBN>
cudaError_t launch_sharea(dllm_cache* c, const void* A, int M, const int* M_dev, const void* B, int N, int K,
                          const Epi& epi, cudaStream_t st) {
  constexpr size_t smem = tc::sharea_smem_bytes<STAGES, SBN>();
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, tc::gemm_sharea_kernel<Epi, STAGES, CS, SBN>, smem);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, A, K, M, static_cast<uint64_t>(K) * 2, tc::BK, tc::BM / CS, true) ||
      !make_tmap_2d(&tb, B, K, N, static_cast<uint64_t>(K) * 2, tc::BK, SBN, true))
    return cudaErrorInvalidValue;
  const int tiles = cdiv(M, tc::BM) * cdiv(cdiv(N, SBN), CS);
  const int per_sm = 2 * tc::sharea_smem_bytes<STAGES, SBN>() <= 227 * 1024 ? 2 : 1;
  const int clusters = std::max(1, std::min(tiles, per_sm * c->num_sms / CS));
  return launch_ex(tc::gemm_sharea_kernel<Epi, STAGES, CS, SBN>, dim3(CS * clusters), dim3(tc::THREADS), smem, st, CS, ta,
                   tb, M, M_dev, N, K, epi, c->err);
}

template <class Epi, int S>
cudaError_t launch_skinny(dllm_cache* c, const void* A, int a_rows, int M_host, const int* M_dev, const void* W,
                          int N, int K, const Epi& epi, cudaStream_t st) {
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, tc::gemm_skinny_kernel<Epi, S>, tc::SKN_SMEM);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tw, tx;
  if (!make_tmap_2d(&tw, W, K, N, static_cast<uint64_t>(K) * 2, tc::BK, 128, true) ||
      !make_tmap_2d(&tx, A, K, a_rows, static_cast<uint64_t>(K) * 2, tc::BK, tc::SKN_XBOX, true))
    return cudaErrorInvalidValue;
  return launch_ex(tc::gemm_skinny_kernel<Epi, S>, dim3(cdiv(N, 128) * S), dim3(tc::THREADS), tc::SKN_SMEM, st, S, tw,
                   tx, M_host, M_dev, a_rows, N, K, epi, c->err);
}

// Clusters of the weight-streaming kernel (split s) that fit on the GPU at
// once: clusters must sit inside one GPC, so this can be below num_sms / s.
template <class Epi, int S>
int skinny_resident(dllm_cache* c) {
  static std::atomic<int> known[64];     // per device: clusters + 1, 0 = not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64) {
    const int k = known[dev].load(std::memory_order_acquire);
    if (k > 0) return k - 1;
  }
  if (set_smem(tc::gemm_skinny_kernel<Epi, S>, tc::SKN_SMEM) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S * c->num_sms);
  cfg.blockDim = dim3(tc::THREADS);
  cfg.dynamicSmemBytes = tc::SKN_SMEM;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = S;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int k = 0;
  if (cudaOccupancyMaxActiveClusters(&k, tc::gemm_skinny_kernel<Epi, S>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    k = 0;
  }
  if (dev < 64) known[dev].store(k + 1, std::memory_order_release);
  return k;
}

// Split of K for the weight-streaming kernel: the largest, up to 4, whose
// clusters (one per 128 output columns) are all resident at once, 0 if none
// is.  Past 4 the exchange of the partials costs more than the extra CTAs
// gain (W_o at 128 rows, d = 2048, L2 flushed: 19.1 us with 6 ranks, 17.0
// with 4 or 3).
template <class Epi>
int skinny_split(dllm_cache* c, int N) {
  const int nN = cdiv(N, 128);
  if (nN <= skinny_resident<Epi, 4>(c)) return 4;
  if (nN <= skinny_resident<Epi, 3>(c)) return 3;
  if (nN <= skinny_resident<Epi, 2>(c)) return 2;
  if (nN <= skinny_resident<Epi, 1>(c)) return 1;
  return 0;
}

template <class Epi>
cudaError_t run_skinny(dllm_cache* c, int split, const void* A, int a_rows, int M_host, const int* M_dev,
                       const void* W, int N, int K, const Epi& epi, cudaStream_t st) {
  switch (split) {
    case 4: return launch_skinny<Epi, 4>(c, A, a_rows, M_host, M_dev, W, N, K, epi, st);
    case 3: return launch_skinny<Epi, 3>(c, A, a_rows, M_host, M_dev, W, N, K, epi, st);
    case 2: return launch_skinny<Epi, 2>(c, A, a_rows, M_host, M_dev, W, N, K, epi, st);
    default: return launch_skinny<Epi, 1>(c, A, a_rows, M_host, M_dev, W, N, K, epi, st);
  }
}

// bf16 D = A . B^T with epilogue `epi`.  M is M_host, or the device count
// M_dev (at most a_rows).  Up to 256 rows with a split of K, 512 without, the
// weights are streamed once by the swapped-operand kernel (when their
// 128-column tiles fit on the SMs).  More rows are tensor-bound: the
// multicast pair kernel (256-wide
// tiles; `wide_ok` says the epilogue accepts them), else the persistent
// kernel.  With a device count both sizes are launched; each skips the
// other's range.
template <class Epi>
cudaError_t run_tc(dllm_cache* c, const void* A, int a_rows, int M_host, const int* M_dev, const void* B, int N,
                   int K, const Epi& epi, cudaStream_t st, bool wide_ok = true) {
  if (!M_dev && M_host <= 0) return cudaSuccess;
  const int split = skinny_split<Epi>(c, N);
  const int m_rows = M_dev ? a_rows : M_host;     // most rows this call can see
  cudaError_t e = cudaSuccess;
  const int skn_rows = split > 0 ? tc::skn_max_rows(split) : 0;
  if (split > 0 && (M_dev || M_host <= skn_rows)) {
    e = run_skinny(c, split, A, a_rows, M_host, M_dev, B, N, K, epi, st);
    if (e != cudaSuccess || m_rows <= skn_rows) return e;
  }
  const int M_min = skn_rows + 1;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, A, K, a_rows, static_cast<uint64_t>(K) * 2, tc::BK, tc::BM, true) ||
      !make_tmap_2d(&tb, B, K, N, static_cast<uint64_t>(K) * 2, tc::BK, tc::BN, true))
    return cudaErrorInvalidValue;
  if (m_rows <= 256) return launch_persistent<Epi, 3>(c, ta, tb, a_rows, M_host, M_dev, M_min, N, K, epi, st);
  if (wide_ok && N % tc::PBN == 0)
    return launch_pair<Epi, 4>(c, ta, tb, a_rows, M_host, M_dev, M_min, N, K, epi, st);
  return launch_persistent<Epi, 4>(c, ta, tb, a_rows, M_host, M_dev, M_min, N, K, epi, st);
}

template <int NCH, class Epi>
cudaError_t run_simt(const void* A, int m_cap, int M_host, const int* M_dev, const void* B, int N, int K,
                     const Epi& epi, cudaStream_t st) {
  const int m_rows = M_dev ? m_cap : M_host;
  if (m_rows <= 0) return cudaSuccess;
  dim3 grid(cdiv(m_rows, 128), cdiv(N, 32 * NCH));
  simt::gemm_simt_kernel<float, NCH, Epi><<<grid, 128, 0, st>>>(
      static_cast<const float*>(A), static_cast<const float*>(B), M_host, M_dev, m_cap, N, K, epi);
  return cudaGetLastError();
}

template <typename T, int DH>
EpiQKV<T, DH> make_qkv(dllm_cache* c, int layer, const int* rows) {
  EpiQKV<T, DH> e;
  const size_t off = static_cast<size_t>(layer) * c->kv_layer_bytes;
  e.rows = rows;
  e.rs = c->rs;
  e.q = static_cast<uint8_t*>(c->q) + off;
  e.k = static_cast<uint8_t*>(c->k) + off;
  e.v = static_cast<uint8_t*>(c->v) + off;
  e.kv = c->kv;
  e.rope = c->rope;
  e.L = c->cfg.seq_len;
  e.d = c->d;
  e.rows_cap = c->rows;
  e.streaming = c->cfg.sink > 0;
  e.S = c->cfg.sink;
  e.W = c->cfg.window;
  e.max_pos = c->max_pos;
  e.gate = kv_gate(c);
  e.Lw = c->Lw;
  e.stage = nullptr;
  e.row0 = 0;
  return e;
}

template <int DH>
cudaError_t qkv_dh(dllm_cache* c, int layer, const void* A, int M_cap, const int* M_dev, const int* rows,
                   const void* w, void* stage, int row0, cudaStream_t st) {
  const int d = c->d, N = 3 * d;
  const int M_host = M_dev ? 0 : M_cap;
  if (c->cfg.dtype == DLLM_BF16) {
    if constexpr (DH >= 64) {  // bf16 caches have head_dim 64 or 128
      auto e = make_qkv<bf16, DH>(c, layer, rows);
      e.stage = static_cast<bf16*>(stage);
      e.row0 = row0;
      return run_tc(c, A, M_cap, M_host, M_dev, w, N, d, e, st,
                    d % tc::PBN == 0);   // a 256-wide tile stays inside q, k or v
    }
    return cudaErrorInvalidValue;
  }
  auto e = make_qkv<float, DH>(c, layer, rows);
  e.stage = static_cast<float*>(stage);
  e.row0 = row0;
  if (d % 128 == 0) return run_simt<4>(A, M_cap, M_host, M_dev, w, N, d, e, st);
  if constexpr (DH <= 64) return run_simt<2>(A, M_cap, M_host, M_dev, w, N, d, e, st);
  return cudaErrorInvalidValue;
}

}  // namespace

// Vocab columns per partial of the LM head: 256 on the pair kernel (M > 128)
// and on the shared-A kernel (M <= 128, at least 8 such tiles), else 128.
int lm_tile_cols(const dllm_cache* c, int M, int V) {
  if (c->cfg.dtype != DLLM_BF16) return tc::BN;
  return M > tc::BM || (M > 0 && cdiv(V, tc::PBN) >= 8) ? tc::PBN : tc::BN;
}

int lm_slots(const dllm_cache* c, int M, int V) { return cdiv(V, lm_tile_cols(c, M, V)); }

cudaError_t gemm_qkv(dllm_cache* c, int layer, const void* A, int M_cap, const int* M_dev, const int* rows,
                     const void* w_qkv, cudaStream_t st, void* stage, int row0) {
  switch (c->cfg.head_dim) {
    case 32: return qkv_dh<32>(c, layer, A, M_cap, M_dev, rows, w_qkv, stage, row0, st);
    case 64: return qkv_dh<64>(c, layer, A, M_cap, M_dev, rows, w_qkv, stage, row0, st);
    case 128: return qkv_dh<128>(c, layer, A, M_cap, M_dev, rows, w_qkv, stage, row0, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_resid(dllm_cache* c, const void* A, const void* W, int M, int M_cap, const int* M_dev, int N,
                       int K, const void* xres, const int* tok, const void* embed, int q_start, int q_len,
                       void* out, cudaStream_t st) {
  if (c->cfg.dtype == DLLM_BF16) {
    EpiResid<bf16> e{static_cast<const bf16*>(xres), static_cast<const bf16*>(embed), tok, q_start, q_len,
                        c->cfg.seq_len, c->cfg.vocab, static_cast<bf16*>(out), c->err};
    return run_tc(c, A, M_dev ? M_cap : M, M, M_dev, W, N, K, e, st);
  }
  if (N % 128 == 0) {
    EpiResid<float> e{static_cast<const float*>(xres), static_cast<const float*>(embed), tok, q_start, q_len,
                         c->cfg.seq_len, c->cfg.vocab, static_cast<float*>(out), c->err};
    return run_simt<4>(A, M_cap, M, M_dev, W, N, K, e, st);
  }
  EpiResid<float> e{static_cast<const float*>(xres), static_cast<const float*>(embed), tok, q_start, q_len,
                       c->cfg.seq_len, c->cfg.vocab, static_cast<float*>(out), c->err};
  return run_simt<1>(A, M_cap, M, M_dev, W, N, K, e, st);
}

cudaError_t gemm_gelu(dllm_cache* c, const void* A, const void* W, int M, int M_cap, const int* M_dev, int N,
                      int K, const float* rs, void* out, cudaStream_t st) {
  if (c->cfg.dtype == DLLM_BF16) {
    EpiGelu<bf16> e{rs, static_cast<bf16*>(out)};
    return run_tc(c, A, M_dev ? M_cap : M, M, M_dev, W, N, K, e, st);
  }
  EpiGelu<float> e{rs, static_cast<float*>(out)};
  return run_simt<1>(A, M_cap, M, M_dev, W, N, K, e, st);
}

cudaError_t gemm_lm(dllm_cache* c, const void* A, const void* W, int M, const int* M_dev, int V, int d,
                    const float* rs, int mask_id, void* part, int n_tiles, cudaStream_t st) {
  EpiLM e{rs, mask_id, static_cast<LMPart*>(part), n_tiles};
  if (c->cfg.dtype == DLLM_BF16) {
    if (M > tc::BM) {   // pairs of row tiles share each 256-column weight tile
      CUtensorMap ta, tb;
      if (!make_tmap_2d(&ta, A, d, M, static_cast<uint64_t>(d) * 2, tc::BK, tc::BM, true) ||
          !make_tmap_2d(&tb, W, d, V, static_cast<uint64_t>(d) * 2, tc::BK, tc::BN, true))
        return cudaErrorInvalidValue;
      return launch_pair<EpiLM, 4>(c, ta, tb, M, M_dev ? 0 : M, M_dev, 0, V, d, e, st);
    }
    // one row tile, many vocab tiles: clusters of 4 share the rows' tile,
    // one 128 x 256 tile per CTA and SM
    if (M > 0 && cdiv(V, tc::PBN) >= 8) return launch_sharea<EpiLM, 4, 4, tc::PBN>(c, A, M, M_dev, W, V, d, e, st);
    return run_tc(c, A, M, M_dev ? 0 : M, M_dev, W, V, d, e, st);
  }
  return run_simt<4>(A, M, M_dev ? 0 : M, M_dev, W, V, d, e, st);
}

}  // namespace dllm
