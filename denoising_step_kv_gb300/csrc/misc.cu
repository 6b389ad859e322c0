// Row gather + RMS scale, LM-head tile merge, the Stable-Window-Decoding
// update with refresh-set construction, and state reset.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int NEVER = -(1 << 30);   // version of a never-written entry

template <typename T> struct Vec;
template <> struct Vec<bf16> { static constexpr int N = 8; };
template <> struct Vec<float> { static constexpr int N = 4; };

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// One warp per refreshed row: validate the row and its token, copy the layer
// input into the compact buffer X (layer-0 embedding rows; a caller-given
// input is used in place), compute the RMSNorm scale, and stamp the row's
// version and token-at-write.
//
// gate (may be null): refresh-set flag words [B][Lw]; a listed row whose flag
// is clear only queries, so its version and token-at-write stay as they are.
template <typename T>
__global__ void __launch_bounds__(256) gather_kernel(const int* __restrict__ rows, const int* __restrict__ n_rows,
                                                     int n_host, const T* __restrict__ x, const int* __restrict__ tok,
                                                     const T* __restrict__ embed, T* __restrict__ X,
                                                     float* __restrict__ rs, int* __restrict__ tok_w,
                                                     int* __restrict__ version, int t, int d, int rows_cap,
                                                     int max_pos, int streaming, int vocab, float eps, int x_cap,
                                                     const uint32_t* __restrict__ gate, int L, int Lw, int row0,
                                                     unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  pdl_launch();
  pdl_wait();
  int n = n_rows ? *n_rows : n_host;
  if (n > x_cap) {          // more rows than the compact buffers hold
    if (i == 0 && lane == 0) set_err(err, DLLM_ERR_ROW);
    n = x_cap;
  }
  if (i >= n) return;
  const int row = rows ? rows[i] : row0 + i;
  const bool row_ok = streaming ? (row >= 0 && row < max_pos) : (row >= 0 && row < rows_cap);
  if (!row_ok) {
    if (lane == 0) {
      set_err(err, DLLM_ERR_ROW);
      rs[i] = -1.f;
    }
    return;
  }
  const T* src;
  int token = -1;
  if (x) {
    src = x + static_cast<size_t>(i) * d;
  } else {
    token = tok[row];
    if (token < 0 || token >= vocab) {
      if (lane == 0) {
        set_err(err, DLLM_ERR_TOKEN);
        rs[i] = -1.f;
      }
      return;
    }
    src = embed + static_cast<size_t>(token) * d;
  }
  constexpr int VN = Vec<T>::N, U = 8;     // U vectors per lane in flight
  float ss = 0.f;
  for (int c0 = lane * VN; c0 < d; c0 += 32 * VN * U) {
    float v[U][VN];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + u * 32 * VN < d) load_row(src + c0 + u * 32 * VN, v[u], VN);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c0 + u * 32 * VN >= d) break;
#pragma unroll
      for (int j = 0; j < VN; ++j) ss = fmaf(v[u][j], v[u][j], ss);
      if (!x) store_row(X + static_cast<size_t>(i) * d + c0 + u * 32 * VN, v[u], VN);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) {
    rs[i] = rsqrtf(ss / static_cast<float>(d) + eps);
    if (!streaming) {
      const int b = row / L, pos = row - b * L;
      const bool writes = !gate || ((gate[b * Lw + (pos >> 5)] >> (pos & 31)) & 1u);
      if (version && writes) version[row] = t;
      if (tok_w && token >= 0 && writes) tok_w[row] = token;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) rownorm_kernel(const T* __restrict__ h, int M_host, const int* M_dev, int d,
                                                      float eps, float* __restrict__ rs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  pdl_launch();
  pdl_wait();
  const int M = M_dev ? *M_dev : M_host;
  if (i >= M) return;
  constexpr int VN = Vec<T>::N, U = 8;
  const T* row = h + static_cast<size_t>(i) * d;
  float ss = 0.f;
  for (int c0 = lane * VN; c0 < d; c0 += 32 * VN * U) {
    float v[U][VN];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + u * 32 * VN < d) load_row(row + c0 + u * 32 * VN, v[u], VN);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c0 + u * 32 * VN >= d) break;
#pragma unroll
      for (int j = 0; j < VN; ++j) ss = fmaf(v[u][j], v[u][j], ss);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) rs[i] = rsqrtf(ss / static_cast<float>(d) + eps);
}

// One 128-thread CTA per row: every thread merges its tiles in increasing
// vocab order, then a tree merge across threads (ties: lower index wins).
// fail_word (may be null): an error word of this call alone; when any bit is
// set (a wait of the GEMM gave up, so some partials were never written) the
// row gets argmax -1 and NaN probability and entropy instead.
constexpr int MERGE_THREADS = 128;
__global__ void __launch_bounds__(MERGE_THREADS) lm_merge_kernel(const LMPart* __restrict__ part, int M,
                                                                 const int* __restrict__ M_dev, int n_tiles,
                                                                 int* __restrict__ argmax, float* __restrict__ p1,
                                                                 float* __restrict__ ent,
                                                                 const unsigned* __restrict__ fail_word) {
  __shared__ float s_m[MERGE_THREADS / 32], s_s[MERGE_THREADS / 32], s_a[MERGE_THREADS / 32];
  __shared__ int s_i[MERGE_THREADS / 32];
  const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch();
  pdl_wait();
  if (i >= M || (M_dev && i >= *M_dev)) return;
  if (fail_word && *fail_word != 0u) {
    if (tid == 0) {
      argmax[i] = -1;
      p1[i] = __int_as_float(0x7fc00000);
      ent[i] = __int_as_float(0x7fc00000);
    }
    return;
  }
  float m = -INFINITY, s = 0.f, a = 0.f;
  int idx = 0x7fffffff;
  for (int tt = tid; tt < n_tiles; tt += MERGE_THREADS) {
    const LMPart p = part[static_cast<size_t>(i) * n_tiles + tt];
    lm_merge(m, s, a, idx, p.m, p.s, p.a, p.idx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float a2 = __shfl_xor_sync(0xffffffffu, a, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    lm_merge(m, s, a, idx, m2, s2, a2, i2);
  }
  if (lane == 0) {
    s_m[warp] = m; s_s[warp] = s; s_a[warp] = a; s_i[warp] = idx;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < MERGE_THREADS / 32; ++w) lm_merge(m, s, a, idx, s_m[w], s_s[w], s_a[w], s_i[w]);
    argmax[i] = idx;
    p1[i] = 1.f / s;
    ent[i] = logf(s) - a / s;
  }
}

__device__ void compact_words(const uint32_t* __restrict__ words, int nw, int L, int Lw, int q0, int nac,
                              const uint8_t* __restrict__ seq_done, int* __restrict__ rows,
                              int* __restrict__ n_rows);

// Stable-Window-Decoding update of the active block of sequence blockIdx.x,
// then one flag bit per position for the next step's refresh set.  With
// `stats`, the sequence's counters of step t (refresh rows, stable rows,
// expired rows, committed rows) go to stats[t][b][0..3].
//
// ent (may be null): the confidence criterion - an unstable active row joins
// the next refresh set when alpha (1 - ent / H_max) + beta exp(-lambda age)
// < theta (R is then 0); else every unstable active row is dilated by R.
struct ConfGate {
  float alpha, beta, lambda, theta, h_max;
};
__global__ void __launch_bounds__(1024, 1) swd_kernel(
    const int* __restrict__ argmax, const float* __restrict__ p1, const float* __restrict__ ent, ConfGate cg,
    int* __restrict__ tok,
    uint8_t* __restrict__ stable, int* __restrict__ hist_tok, float* __restrict__ hist_p, int* __restrict__ hist_n,
    const int* __restrict__ tok_w, const int* __restrict__ version, uint32_t* __restrict__ words, int L, int Lw,
    int seq_rows, int n_layers, int blk, int K, float tau, int R, int q0, int t, int last, int full, int expiry,
    int active_queries, uint8_t* __restrict__ seq_done, int* __restrict__ m_live, unsigned* __restrict__ ticket,
    int* __restrict__ rows, int* __restrict__ n_rows, int* __restrict__ stats) {
  __shared__ uint8_t s_unst[64];
  __shared__ uint8_t s_open[64];     // unstable after this update
  __shared__ int s_last;
  const int b = blockIdx.x;
  pdl_launch();
  pdl_wait();
  const int nac = min(blk, L - q0);
  int committed = 0, now_stable = 0;    // this row's counters
  if (threadIdx.x < nac) {
    const int j = threadIdx.x;
    const int r = b * L + q0 + j;
    const int h = b * blk + j;
    // every load of this row's state at once: its ring of K <= 8 records
    // stays in registers, so nothing written here is read back
    constexpr int KMAX = 8;
    bool st = stable[r] != 0;
    const bool st0 = st;
    const int a = argmax[h];
    const float pa = p1[h];
    int n = hist_n[h];
    int ht[KMAX];
    float hp[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (k < K) {
        ht[k] = hist_tok[h * K + k];
        hp[k] = hist_p[h * K + k];
      }
    if (!st) {
      const int slot_new = n % K;
      hist_tok[h * K + slot_new] = a;
      hist_p[h * K + slot_new] = pa;
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k == slot_new) {
          ht[k] = a;
          hp[k] = pa;
        }
      ++n;
      hist_n[h] = n;
      if (n >= K) {
        bool same = true;
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k)      // oldest -> newest: slot (n - K + k) % K
          if (k < K) {
            const int slot = (n - K + k) % K;
            int tk = 0;
            float pk = 0.f;
#pragma unroll
            for (int u = 0; u < KMAX; ++u)
              if (u == slot) {
                tk = ht[u];
                pk = hp[u];
              }
            same = same && tk == a;
            s = s + pk;
          }
        const float mean = s / static_cast<float>(K);
        if (same && mean > tau) {
          st = true;
          stable[r] = 1;
          tok[r] = a;
        }
      }
    }
    if (last) {
      if (!st) tok[r] = a;
      hist_n[h] = 0;
    }
    committed = (st && !st0) || (last && !st) ? 1 : 0;
    now_stable = st ? 1 : 0;
    s_open[j] = st ? 0 : 1;
    bool flag = !st;
    if (ent && flag) {   // cache confidence at step t + 1 of this row's layer-0 entry
      const float age = static_cast<float>(t + 1 - version[r]);
      const float conf = cg.alpha * (1.f - ent[h] / cg.h_max) + cg.beta * expf(-(cg.lambda * age));
      flag = conf < cg.theta;
    }
    s_unst[j] = flag ? 1 : 0;
  }
  // early exit: every active row stable after a step that is not the
  // block's last ends this sequence's block (no refresh from now on)
  const int n_open = __syncthreads_count(threadIdx.x < nac && s_open[threadIdx.x]);
  const int n_committed = __syncthreads_count(committed);
  const int n_stable = __syncthreads_count(now_stable);
  const bool ended = seq_done && !last && n_open == 0;
  int n_flag = 0, n_expired = 0;
  for (int base = 0; base < L; base += blockDim.x) {
    const int p = base + threadIdx.x;
    bool f = false, expired = false;
    if (p < L) {
      const int r = b * L + p;
      if (ended) {
        f = false;
      } else if (last || full) {
        f = true;
      } else {
        // independent loads (no short-circuit between them): any layer's
        // version expired <=> the oldest one did
        const int tk = tok[r], tw = tok_w[r];
        int vmin = 0x7fffffff;
        if (expiry >= 0)
          for (int l = 0; l < n_layers; ++l) vmin = min(vmin, version[l * seq_rows + r]);
        const int lo = max(p - R, q0), hi = min(p + R, q0 + nac - 1);
        for (int u = lo; u <= hi; ++u) f |= s_unst[u - q0] != 0;
        f |= tk != tw;
        expired = expiry >= 0 && (t + 1) - vmin > expiry;
        f |= expired;
      }
    }
    n_flag += __syncthreads_count(f);
    n_expired += __syncthreads_count(expired);
    const uint32_t word = __ballot_sync(0xffffffffu, f);
    const int w = (base + (threadIdx.x & ~31)) >> 5;
    if ((threadIdx.x & 31) == 0 && w < Lw) words[b * Lw + w] = word;
  }
  if (seq_done && threadIdx.x == 0) seq_done[b] = ended ? 1 : 0;
  if (stats && threadIdx.x == 0 && t >= 0 && t < kStatsSteps) {
    int* o = stats + (static_cast<size_t>(t) * gridDim.x + b) * 4;
    o[0] = n_flag;
    o[1] = n_stable;
    o[2] = n_expired;
    o[3] = n_committed;
  }
  // the last sequence block to finish compacts every sequence's flags
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the row list: the refresh set, plus the active rows of the running
  // sequences when they all query
  compact_words(words, gridDim.x * Lw, L, Lw, q0, active_queries && !last && !full ? nac : 0, seq_done, rows,
                n_rows);
  if (seq_done) {   // W_o and the LM head run while any sequence's block runs
    int open = 0;
    for (int i = threadIdx.x; i < gridDim.x; i += blockDim.x) open |= seq_done[i] == 0;
    open = __syncthreads_or(open);
    if (threadIdx.x == 0) *m_live = open ? gridDim.x * blk : 0;
  }
  if (threadIdx.x == 0) *ticket = 0u;
}

// Bits [lo, hi) of a 32-bit word (clipped to [0, 32)).
__device__ __forceinline__ uint32_t range_bits(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 32);
  if (hi <= lo) return 0u;
  const uint32_t up = hi == 32 ? 0xffffffffu : ((1u << hi) - 1u);
  return up & ~((1u << lo) - 1u);
}

// Compact the flag words, OR the positions [q0, q0 + nac) of every sequence,
// into ascending row ids b * L + pos (block-wide exclusive scan of the
// per-word popcounts, one word per thread per pass).  Run by one whole block
// of blockDim.x (a multiple of 32, <= 1024) threads.
__device__ void compact_words(const uint32_t* __restrict__ words, int nw, int L, int Lw, int q0, int nac,
                              const uint8_t* __restrict__ seq_done, int* __restrict__ rows,
                              int* __restrict__ n_rows) {
  __shared__ int s_warp[32];
  __shared__ int s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (int base = 0; base < nw; base += blockDim.x) {
    const int w = base + tid;
    uint32_t word = 0u;
    if (w < nw) {
      const bool run = !seq_done || !seq_done[w / Lw];      // an ended sequence adds no active rows
      word = words[w] | (run ? range_bits(q0 - (w % Lw) * 32, q0 + nac - (w % Lw) * 32) : 0u);
    }
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int x = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      s_warp[lane] = x;   // inclusive prefix of warp totals
    }
    __syncthreads();
    int off = s_base + incl - cnt + (warp > 0 ? s_warp[warp - 1] : 0);
    if (w < nw) {
      const int rb = (w / Lw) * L + (w % Lw) * 32;
      while (word) {
        const int bit = __ffs(word) - 1;
        word &= word - 1u;
        rows[off++] = rb + bit;
      }
    }
    __syncthreads();
    if (tid == 0) s_base += s_warp[nwarps - 1];
    __syncthreads();
  }
  if (tid == 0) *n_rows = s_base;
}

// Every refresh row 0 .. n-1 (the block-start full refresh), every refresh
// flag set.
__global__ void __launch_bounds__(256) all_rows_kernel(int* __restrict__ rows, int* __restrict__ n_rows, int n,
                                                       uint32_t* __restrict__ words, int nw) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) rows[i] = i;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nw; i += gridDim.x * blockDim.x) words[i] = 0xffffffffu;
  if (blockIdx.x == 0 && threadIdx.x == 0) *n_rows = n;
}

__global__ void reset_kernel(int* version, int n_version, int* tok_w, uint8_t* stable, int n_rows, int* hist_n,
                             int n_hist, int* m_live, unsigned* err) {
  const int i0 = blockIdx.x * blockDim.x + threadIdx.x, step = gridDim.x * blockDim.x;
  for (int i = i0; i < n_version; i += step) version[i] = NEVER;
  for (int i = i0; i < n_rows; i += step) {
    tok_w[i] = -1;
    stable[i] = 0;
  }
  for (int i = i0; i < n_hist; i += step) hist_n[i] = 0;
  if (i0 == 0) {
    *err = 0u;
    if (m_live) *m_live = n_hist;     // every active row of every sequence
  }
}

// Active-block rows out of a compact row-list buffer: dst[b * q_len + j] =
// src[i] for the i with rows[i] == b * L + q_start + j (binary search of the
// sorted list; one warp per output row).  A row missing from the list sets
// DLLM_ERR_ROW and its output row is zero-filled.
__global__ void __launch_bounds__(256) active_rows_kernel(const uint4* __restrict__ src, const int* __restrict__ rows,
                                                          const int* __restrict__ n_rows, int cap, int L,
                                                          int q_start, int q_len, int n_out, int row_vec,
                                                          const uint8_t* __restrict__ seq_done,
                                                          uint4* __restrict__ dst, unsigned* err) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  pdl_launch();
  pdl_wait();
  if (w >= n_out) return;
  const int b = w / q_len, j = w - b * q_len;
  if (seq_done && seq_done[b]) return;       // an ended sequence's rows are not in the list
  const int key = b * L + q_start + j;
  const int n = min(*n_rows, cap);
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (rows[mid] < key) lo = mid + 1; else hi = mid;
  }
  const bool found = lo < n && rows[lo] == key;
  if (!found && lane == 0) set_err(err, DLLM_ERR_ROW);
  const uint4* s = src + static_cast<size_t>(found ? lo : 0) * row_vec;
  uint4* o = dst + static_cast<size_t>(w) * row_vec;
  for (int c = lane; c < row_vec; c += 32) o[c] = found ? s[c] : make_uint4(0u, 0u, 0u, 0u);
}

// The bounded wait on a barrier that nothing arrives on: thread 0 gives up
// after limit_ns, sets DLLM_ERR_TIMEOUT and raises the CTA's abort flag; lane
// 0 of every other warp waits on a second such barrier (limit 4 x limit_ns)
// and leaves through that flag.  Every thread then returns normally.
__global__ void __launch_bounds__(128) wait_selftest_kernel(uint64_t limit_ns, unsigned* err) {
  __shared__ uint64_t bar_a, bar_b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar_a, 1);
    mbar_init(&bar_b, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_for(&bar_a, 0, &abort_flag, err, limit_ns);
  else if ((threadIdx.x & 31) == 0)
    mbar_wait_for(&bar_b, 0, &abort_flag, nullptr, 4 * limit_ns);
  __syncthreads();
}

// One warp per (token, part q/k/v, head): the head's dh values of the
// token's staging row (row-major [n][3d], RoPE applied) into the ring slot of
// the layer's tiled cache, 16 bytes per lane.
__global__ void __launch_bounds__(256) ring_append_kernel(const uint8_t* __restrict__ staged, uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ k, uint8_t* __restrict__ v,
                                                          KvLayout kv, int n0, int count, int H, int row_bytes,
                                                          int S, int W, int max_pos, unsigned* err) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  pdl_launch();
  pdl_wait();
  if (w >= count * 3 * H) return;
  const int i = w / (3 * H), part = (w / H) % 3, h = w % H;
  const int n = n0 + i;
  if (n < 0 || n >= max_pos) {
    if (lane == 0 && part == 0 && h == 0) set_err(err, DLLM_ERR_ROW);
    return;
  }
  const int slot = ring_slot(n, S, W);
  const uint8_t* src = staged + (static_cast<size_t>(n) * 3 * H + part * H + h) * row_bytes;
  uint8_t* base = part == 0 ? q : part == 1 ? k : v;
  for (int c = lane; c < row_bytes / 16; c += 32)
    *reinterpret_cast<uint4*>(base + kv.chunk_off(0, h, slot, c)) = *reinterpret_cast<const uint4*>(src + c * 16);
}

}  // namespace

cudaError_t launch_ring_append(dllm_cache* c, int layer, const void* staged, int n0, int count, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  const size_t off = static_cast<size_t>(layer) * c->kv_layer_bytes;
  const int H = c->cfg.n_heads, warps = count * 3 * H;
  return launch_ex(ring_append_kernel, dim3(cdiv(warps * 32, 256)), dim3(256), 0, st, 0,
                   static_cast<const uint8_t*>(staged), static_cast<uint8_t*>(c->q) + off,
                   static_cast<uint8_t*>(c->k) + off, static_cast<uint8_t*>(c->v) + off, c->kv, n0, count, H,
                   c->kv.row_bytes, c->cfg.sink, c->cfg.window, c->max_pos, c->err);
}

cudaError_t launch_wait_selftest(dllm_cache* c, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 128, 0, st>>>(limit_ns, c->err);
  return cudaGetLastError();
}

cudaError_t launch_active_rows(dllm_cache* c, const void* src, const int* rows, const int* n_rows, int q_start,
                               int q_len, void* dst, cudaStream_t st) {
  const int n_out = c->cfg.batch * q_len;
  if (n_out <= 0) return cudaSuccess;
  const int row_vec = c->d * c->elem / 16;
  return launch_ex(active_rows_kernel, dim3(cdiv(n_out * 32, 256)), dim3(256), 0, st, 0,
                   static_cast<const uint4*>(src), rows, n_rows, c->seq_rows, c->cfg.seq_len, q_start, q_len, n_out,
                   row_vec, done_flags(c), static_cast<uint4*>(dst), c->err);
}

cudaError_t launch_gather(dllm_cache* c, int layer, const int* rows, const int* n_rows, int n_host, const void* x,
                          const int* tok, const void* embed, int t, cudaStream_t st, int row0) {
  const bool dense = c->cfg.sink == 0;
  const int cap = rows ? c->seq_rows : n_host;    // rows of the compact buffers
  if (cap <= 0) return cudaSuccess;
  int* version = dense ? c->version + static_cast<size_t>(layer) * c->seq_rows : nullptr;
  int* tok_w = (dense && layer == 0 && !x) ? c->tok_w : nullptr;
  const dim3 grid(cdiv(cap, 8));
  const int* nr = rows ? n_rows : nullptr;
  const int streaming = dense ? 0 : 1;
  const uint32_t* gate = kv_gate(c);
  const int L = dense ? c->cfg.seq_len : 1;
  if (c->cfg.dtype == DLLM_BF16)
    return launch_ex(gather_kernel<bf16>, grid, dim3(256), 0, st, 0, rows, nr, n_host, static_cast<const bf16*>(x), tok,
                     static_cast<const bf16*>(embed), static_cast<bf16*>(c->X), c->rs, tok_w, version, t, c->d,
                     c->rows, c->max_pos, streaming, c->cfg.vocab, c->cfg.rms_eps, c->seq_rows, gate, L, c->Lw, row0,
                     c->err);
  return launch_ex(gather_kernel<float>, grid, dim3(256), 0, st, 0, rows, nr, n_host, static_cast<const float*>(x), tok,
                   static_cast<const float*>(embed), static_cast<float*>(c->X), c->rs, tok_w, version, t, c->d,
                   c->rows, c->max_pos, streaming, c->cfg.vocab, c->cfg.rms_eps, c->seq_rows, gate, L, c->Lw, row0,
                   c->err);
}

cudaError_t launch_rownorm(dllm_cache* c, const void* h, int M, const int* M_dev, int d, float* rs,
                           cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (c->cfg.dtype == DLLM_BF16)
    return launch_ex(rownorm_kernel<bf16>, dim3(cdiv(M, 8)), dim3(256), 0, st, 0, static_cast<const bf16*>(h), M, M_dev,
                     d, c->cfg.rms_eps, rs);
  return launch_ex(rownorm_kernel<float>, dim3(cdiv(M, 8)), dim3(256), 0, st, 0, static_cast<const float*>(h), M,
                   M_dev, d, c->cfg.rms_eps, rs);
}

cudaError_t launch_lm_merge(const void* part, int M, const int* M_dev, int n_tiles, int* argmax, float* p1,
                            float* ent, const unsigned* fail_word, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  return launch_ex(lm_merge_kernel, dim3(M), dim3(MERGE_THREADS), 0, st, 0, static_cast<const LMPart*>(part), M,
                   M_dev, n_tiles, argmax, p1, ent, fail_word);
}

cudaError_t launch_stab(dllm_cache* c, const int* argmax, const float* p1, const float* ent, int* tok, int q_start,
                        int t, int last, int R, int full, int* rows, int* n_rows, cudaStream_t st) {
  const dllm_cache_cfg& g = c->cfg;
  const ConfGate cg{g.conf_alpha, g.conf_beta, g.conf_lambda, g.conf_theta,
                    static_cast<float>(std::log(static_cast<double>(g.vocab - 1)))};
  uint8_t* done = g.early_exit ? c->seq_done : nullptr;
  return launch_ex(swd_kernel, dim3(g.batch), dim3(1024), 0, st, 0, argmax, p1, ent, cg, tok, c->stable, c->hist_tok, c->hist_p,
                   c->hist_n, c->tok_w, c->version, c->words, g.seq_len, c->Lw, c->seq_rows, g.n_layers, g.block_len,
                   g.swd_K, g.swd_tau, R, q_start, t, last, full, g.expiry, g.active_queries, done, c->m_live,
                   c->ticket, rows, n_rows, c->stats);
}

cudaError_t launch_refresh_all(dllm_cache* c, int q_start, int* rows, int* n_rows, cudaStream_t st) {
  (void)q_start;
  const int n = c->seq_rows;
  all_rows_kernel<<<std::min(cdiv(n, 256), 256), 256, 0, st>>>(rows, n_rows, n, c->words, c->cfg.batch * c->Lw);
  return cudaGetLastError();
}

cudaError_t launch_reset(dllm_cache* c, cudaStream_t st) {
  const dllm_cache_cfg& g = c->cfg;
  if (c->seq_done) {   // no block has ended (W_o and the LM head count: reset_kernel)
    cudaError_t e = cudaMemsetAsync(c->seq_done, 0, static_cast<size_t>(g.batch), st);
    if (e != cudaSuccess) return e;
  }
  {  // until a refresh set is built, every row may write its K/V (the gate of active queries)
    cudaError_t e = cudaMemsetAsync(c->words, 0xff, static_cast<size_t>(g.batch) * c->Lw * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  if (c->fa_key) {   // no kept attention state is valid (block start -1 never matches)
    cudaError_t e = cudaMemsetAsync(c->fa_key, 0xff, static_cast<size_t>(g.batch) * g.n_heads * 66 * sizeof(int), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->fa_rebuilt, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  if (c->stats) {   // no step recorded yet
    cudaError_t e = cudaMemsetAsync(c->stats, 0, static_cast<size_t>(kStatsSteps) * g.batch * 4 * sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  const int nv = g.n_layers * c->seq_rows;
  const int nh = g.batch * (g.sink > 0 ? 1 : g.block_len);   // the history counters the handle holds
  reset_kernel<<<std::max(1, std::min(cdiv(std::max(nv, c->seq_rows), 256), 1024)), 256, 0, st>>>(
      c->version, nv, c->tok_w, c->stable, c->seq_rows, c->hist_n, nh, c->m_live, c->err);
  return cudaGetLastError();
}

}  // namespace dllm
