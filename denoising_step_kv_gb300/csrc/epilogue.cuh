// Epilogues of the projection GEMMs (see gemm.cuh for the interface).
#pragma once
#include "common.cuh"

namespace dllm {

// Streaming-mode ring slot of stream token n: sinks keep slots 0..S-1, later
// tokens cycle through the W rolling slots.
__host__ __device__ __forceinline__ int ring_slot(int n, int S, int W) {
  return n < S ? n : S + (n - S) % W;
}

// Store 32 consecutive values of head h, dims [e0, e0 + 32), of cache row
// (b, pos) into the tiled KV layout (see KvLayout), 16 bytes at a time.
template <typename T>
__device__ __forceinline__ void store_kv32(uint8_t* base, const KvLayout& kv, int b, int h, int pos, int e0,
                                           const float* v) {
  constexpr int PER = 16 / sizeof(T);          // values per 16-byte chunk
  const int c0 = e0 / PER;
#pragma unroll
  for (int q = 0; q < 32 / PER; ++q) store_row(reinterpret_cast<T*>(base + kv.chunk_off(b, h, pos, c0 + q)),
                                               v + q * PER, PER);
}

// QKV projection: accumulator row m (compact refresh index) times the row's
// RMSNorm scale, RoPE on the q and k parts (rotate-half pairs (i, i + DH/2)
// with a cos/sin table), stored into the layer's tiled Q/K/V cache.
template <typename T, int DH>
struct EpiQKV {
  const int* rows;      // compact index -> row id (nullptr: identity)
  const float* rs;      // per compact row: RMS scale (< 0: skip the row)
  uint8_t* q;
  uint8_t* k;
  uint8_t* v;           // layer base pointers (tiled layout)
  KvLayout kv;
  const float2* rope;   // [max_pos][DH/2] (cos, sin)
  int L, d, rows_cap, streaming, S, W, max_pos;

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    bool ok = m < M;
    int b = 0, slot = 0, pos = 0;
    float sc = 0.f;
    if (ok) {
      const int row = rows ? rows[m] : m;
      if (streaming) {
        ok = row >= 0 && row < max_pos;
        pos = row;
        slot = ok ? ring_slot(row, S, W) : 0;
      } else {
        ok = row >= 0 && row < rows_cap;
        b = ok ? row / L : 0;
        pos = ok ? row - b * L : 0;
        slot = pos;
      }
      sc = ok ? rs[m] : -1.f;
      ok = ok && sc > 0.f;
    }
    const int part = n0 / d, c0 = n0 - part * d;   // c0: first column inside q, k or v
    uint8_t* base = part == 0 ? q : part == 1 ? k : v;
    auto put = [&](int col, const float* vals) {    // col: column inside the part
      const int h = col / DH;
      store_kv32<T>(base, kv, b, h, slot, col - h * DH, vals);
    };
    float a[32], bb[32];
    if (part == 2) {
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        ld(c * 32, a);
        if (ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] *= sc;
          put(c0 + c * 32, a);
        }
      }
    } else if (DH >= 64) {
      constexpr int HALF_CH = DH / 64;        // 32-column chunks in half a head
      const int heads = nch * 32 / DH;        // heads in the tile
#pragma unroll 1
      for (int hd = 0; hd < heads; ++hd) {
#pragma unroll 1
        for (int hc = 0; hc < HALF_CH; ++hc) {
          const int c1 = hd * DH + hc * 32, c2 = c1 + DH / 2;
          ld(c1, a);
          ld(c2, bb);
          if (ok) {
            const float2* rp = rope + static_cast<size_t>(pos) * (DH / 2) + hc * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float2 cs = rp[j];
              const float x1 = a[j] * sc, x2 = bb[j] * sc;
              a[j] = x1 * cs.x - x2 * cs.y;
              bb[j] = x2 * cs.x + x1 * cs.y;
            }
            put(c0 + c1, a);
            put(c0 + c2, bb);
          }
        }
      }
    } else {   // DH == 32: both halves of a head sit in one 32-column chunk
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        ld(c * 32, a);
        if (ok) {
          const float2* rp = rope + static_cast<size_t>(pos) * 16;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 cs = rp[j];
            const float x1 = a[j] * sc, x2 = a[j + 16] * sc;
            a[j] = x1 * cs.x - x2 * cs.y;
            a[j + 16] = x2 * cs.x + x1 * cs.y;
          }
          put(c0 + c * 32, a);
        }
      }
    }
  }
};

// out[m] = resid_m + acc[m]: resid_m = xres[m], or the embedding of the
// token at position q_start + m % q_len of sequence m / q_len.
template <typename T>
struct EpiResid {
  const T* xres;
  const T* embed;
  const int* tok;
  int q_start, q_len, L, vocab;
  T* out;
  unsigned* err;

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    bool ok = m < M;
    const T* rrow = nullptr;
    if (ok) {
      if (xres) {
        rrow = xres + static_cast<size_t>(m) * N;
      } else {
        const int b = m / q_len, j = m - b * q_len;
        const int t = tok[static_cast<size_t>(b) * L + q_start + j];
        if (t < 0 || t >= vocab) {
          if (n0 == 0) set_err(err, DLLM_ERR_TOKEN);
          ok = false;
        } else {
          rrow = embed + static_cast<size_t>(t) * N;
        }
      }
    }
    float a[32], r[32];
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      ld(c * 32, a);
      const int n = n0 + c * 32;
      if (ok && n < N) {
        load_row(rrow + n, r, 32);
#pragma unroll
        for (int j = 0; j < 32; ++j) a[j] += r[j];
        store_row(out + static_cast<size_t>(m) * N + n, a, 32);
      }
    }
  }
};

// out[m] = GELU(rs[m] * acc[m]) with the exact (erf) GELU.
template <typename T>
struct EpiGelu {
  const float* rs;
  T* out;

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    const bool ok = m < M;
    const float sc = ok ? rs[m] : 0.f;
    float a[32];
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      ld(c * 32, a);
      const int n = n0 + c * 32;
      if (ok && n < N) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = a[j] * sc;
          a[j] = 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
        }
        store_row(out + static_cast<size_t>(m) * N + n, a, 32);
      }
    }
  }
};

// Softmax statistics of one vocab tile of one row: max logit, its first
// index, S = sum e^(l - max), A = sum e^(l - max) (l - max).
struct LMPart {
  float m, s, a;
  int idx;
};

__device__ __forceinline__ void lm_merge(float& m, float& s, float& a, int& idx, float m2, float s2, float a2,
                                         int idx2) {
  // (m, s, a) rebased to a common maximum; ties keep the lower index
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2; s = s2; a = a2; idx = idx2;
    return;
  }
  const float mx = fmaxf(m, m2);
  const float e1 = __expf(m - mx), e2 = __expf(m2 - mx);
  const float s_new = s * e1 + s2 * e2;
  const float a_new = e1 * (a + (m - mx) * s) + e2 * (a2 + (m2 - mx) * s2);
  if (m2 > m || (m2 == m && idx2 < idx)) idx = idx2;
  m = mx; s = s_new; a = a_new;
}

struct EpiLM {
  const float* rs;   // RMSNorm scale of each row of h
  int mask_id;
  LMPart* part;      // [M][n_tiles]
  int n_tiles;

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    const bool ok = m < M;
    const float sc = ok ? rs[m] : 0.f;
    float mx = -INFINITY, S = 0.f, A = 0.f;
    int idx = -1;
    float v[32];
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      ld(c * 32, v);
      const int nb = n0 + c * 32;
      float cm = -INFINITY;
      int ci = -1;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = nb + j;
        const bool valid = n < N && n != mask_id;
        v[j] = valid ? v[j] * sc : -INFINITY;
        if (v[j] > cm) {
          cm = v[j];
          ci = n;
        }
      }
      if (cm == -INFINITY) continue;
      float cs = 0.f, ca = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float z = v[j] - cm;        // -inf for excluded columns
        const float e = __expf(z);        // 0 for excluded columns
        cs += e;
        ca += (e > 0.f) ? e * z : 0.f;
      }
      lm_merge(mx, S, A, idx, cm, cs, ca, ci);
    }
    if (ok) part[static_cast<size_t>(m) * n_tiles + n0 / (32 * nch)] = LMPart{mx, S, A, idx};
  }
};

}  // namespace dllm
