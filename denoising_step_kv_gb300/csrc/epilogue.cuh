// Epilogues of the projection GEMMs (see gemm.cuh for the interface).
#pragma once
#include "common.cuh"

namespace dllm {

// Streaming-mode ring slot of stream token n: sinks keep slots 0..S-1, later
// tokens cycle through the W rolling slots.
__host__ __device__ __forceinline__ int ring_slot(int n, int S, int W) {
  return n < S ? n : S + (n - S) % W;
}

// (cos, sin) of the angle pos * f for a frequency f = f.x + f.y held as a
// float pair.  The fp32 product a = pos * f.x is reduced by k * 2 pi (k the
// nearest integer to a / 2 pi) with two fused multiply-adds against 2 pi as
// a float pair (Cody and Waite's additive reduction), the product's rounding
// error and pos * f.y are added to the reduced angle, and the hardware sine
// and cosine evaluate it on [-pi, pi].  Absolute error ~1e-6 for |pos * f|
// up to 2^17.
__device__ __forceinline__ float2 rope_cs(int pos, float2 f) {
  constexpr float kTwoPiHi = 6.2831854820251465f, kTwoPiLo = -1.7484555314695172e-07f;
  constexpr float kInvTwoPi = 0.15915493667125702f;
  const float p = static_cast<float>(pos);
  const float a = p * f.x;
  const float da = fmaf(p, f.x, -a) + p * f.y;
  const float k = rintf(a * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a);
  r = fmaf(-k, kTwoPiLo, r) + da;
  float s, c;
  __sincosf(r, &s, &c);
  return make_float2(c, s);
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
// rotated by pos * theta^(-2i/DH)), stored into the layer's tiled Q/K/V cache.
//
// run_part(m, n0, p, ...) does piece p of the 128-column tile at n0 (PARTS
// independent pieces, used to spread a tile's epilogue over more threads):
// q/k: DH 128 - the rotate-half chunk pair (32p, 32p + 64); DH 64 - head p;
// v: chunks 2p and 2p + 1.
template <typename T, int DH>
struct EpiQKV {
  static constexpr int PARTS = 2;
  const int* rows;      // compact index -> row id (nullptr: identity)
  const float* rs;      // per compact row: RMS scale (< 0: skip the row)
  uint8_t* q;
  uint8_t* k;
  uint8_t* v;           // layer base pointers (tiled layout)
  KvLayout kv;
  const float2* rope;   // [DH/2] frequencies theta^(-2i/DH) as (hi, lo)
  const uint32_t* gate; // refresh-set flag words [B][Lw] (null: every row writes K/V)
  int L, d, rows_cap, streaming, S, W, max_pos, Lw;
  // staging instead of the cache (streaming pre-projection): row m is stream
  // token row0 + m (without a row list) and its q | k | v go to
  // stage[(row0 + m) * 3d ...] row-major, RoPE applied
  T* stage;
  int row0;

  // does row (b, pos) rewrite its K and V (a query-only row stores Q alone)
  __device__ __forceinline__ bool writes_kv(int b, int pos) const {
    return !gate || ((gate[b * Lw + (pos >> 5)] >> (pos & 31)) & 1u);
  }

  // where row m goes; false: store nothing
  __device__ __forceinline__ bool locate(int m, int M, int& b, int& slot, int& pos, float& sc) const {
    b = 0; slot = 0; pos = 0; sc = 0.f;
    if (m >= M) return false;
    const int row = rows ? rows[m] : row0 + m;
    bool ok;
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
    return ok && sc > 0.f;
  }

  // before the epilogue: the row's scale, its row id, its refresh-flag word
  // and the RoPE table into L1 (the epilogue's loads then hit)
  __device__ __forceinline__ void prefetch(int m, int n0, int M, int) const {
    if (m >= M) return;
    prefetch_l1(rs + m, 4);
    if ((m & 31) == 0) prefetch_l1(rope, DH / 2 * static_cast<int>(sizeof(float2)));
    if (!gate || streaming || n0 < d) return;
    const int row = rows ? rows[m] : row0 + m;
    if (row >= 0 && row < rows_cap) {
      const int b = row / L, pos = row - b * L;
      prefetch_l1(gate + b * Lw + (pos >> 5), 4);
    }
  }

  template <class LD>
  __device__ __forceinline__ void run_part(int m, int n0, int p, int M, int N, const LD& ld) const {
    int b, slot, pos;
    float sc;
    const bool ok_row = locate(m, M, b, slot, pos, sc);
    const int part = n0 / d, c0 = n0 - part * d;   // c0: first column inside q, k or v
    uint8_t* base = part == 0 ? q : part == 1 ? k : v;
    const bool ok = ok_row && (part == 0 || writes_kv(b, pos));
    auto put = [&](int col, const float* vals) {    // col: column inside the part
      if (stage) {
        store_row(stage + static_cast<size_t>(pos) * 3 * d + part * d + col, vals, 32);
        return;
      }
      const int h = col / DH;
      store_kv32<T>(base, kv, b, h, slot, col - h * DH, vals);
    };
    float a[32], bb[32];
    if (part == 2) {
      ld(64 * p, a);
      ld(64 * p + 32, bb);
      if (ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          a[j] *= sc;
          bb[j] *= sc;
        }
        put(c0 + 64 * p, a);
        put(c0 + 64 * p + 32, bb);
      }
      return;
    }
    static_assert(DH == 64 || DH == 128, "128-column pieces hold whole rotate-half pairs");
    const int c1 = DH == 128 ? 32 * p : 64 * p, c2 = c1 + DH / 2, hc = DH == 128 ? p : 0;
    ld(c1, a);
    ld(c2, bb);
    if (ok) {
      const float2* fr = rope + hc * 32;   // the same addresses in every lane
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 cs = rope_cs(pos, fr[j]);
        const float x1 = a[j] * sc, x2 = bb[j] * sc;
        a[j] = x1 * cs.x - x2 * cs.y;
        bb[j] = x2 * cs.x + x1 * cs.y;
      }
      put(c0 + c1, a);
      put(c0 + c2, bb);
    }
  }

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    if constexpr (DH >= 64) {
#pragma unroll 1
      for (int t = 0; t < nch / 4; ++t) {
        auto sub = [&](int col, float (&vals)[32]) { ld(t * 128 + col, vals); };
#pragma unroll 1
        for (int p = 0; p < PARTS; ++p) run_part(m, n0 + t * 128, p, M, N, sub);
      }
    } else {   // DH == 32: both halves of a head sit in one 32-column chunk
      int b, slot, pos;
      float sc;
      const bool ok_row = locate(m, M, b, slot, pos, sc);
      const int part = n0 / d, c0 = n0 - part * d;
      const bool ok = ok_row && (part == 0 || writes_kv(b, pos));
      uint8_t* base = part == 0 ? q : part == 1 ? k : v;
      float a[32];
#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        ld(c * 32, a);
        if (!ok) continue;
        if (part != 2) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 cs = rope_cs(pos, rope[j]);
            const float x1 = a[j] * sc, x2 = a[j + 16] * sc;
            a[j] = x1 * cs.x - x2 * cs.y;
            a[j + 16] = x2 * cs.x + x1 * cs.y;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) a[j] *= sc;
        }
        const int col = c0 + c * 32, h = col / DH;
        if (stage)
          store_row(stage + static_cast<size_t>(pos) * 3 * d + part * d + col, a, 32);
        else
          store_kv32<T>(base, kv, b, h, slot, col - h * DH, a);
      }
    }
  }
};

// out[m] = resid_m + acc[m]: resid_m = xres[m], or the embedding of the
// token at position q_start + m % q_len of sequence m / q_len.
template <typename T>
struct EpiResid {
  static constexpr int PARTS = 4;   // 32-column chunks of a 128-column tile
  const T* xres;
  const T* embed;
  const int* tok;
  int q_start, q_len, L, vocab;
  T* out;
  unsigned* err;

  // residual row of output row m (nullptr: skip the row)
  __device__ __forceinline__ const T* resid_row(int m, int M, int N, bool report) const {
    if (m >= M) return nullptr;
    if (xres) return xres + static_cast<size_t>(m) * N;
    const int b = m / q_len, j = m - b * q_len;
    const int t = tok[static_cast<size_t>(b) * L + q_start + j];
    if (t < 0 || t >= vocab) {
      if (report) set_err(err, DLLM_ERR_TOKEN);
      return nullptr;
    }
    return embed + static_cast<size_t>(t) * N;
  }

  // before the epilogue (the weight-streaming kernel calls this while its
  // MMAs run): the residual row's slice of this tile into L1
  __device__ __forceinline__ void prefetch(int m, int n0, int M, int N) const {
    const T* rrow = resid_row(m, M, N, false);
    if (rrow) prefetch_l1(rrow + n0, 128 * static_cast<int>(sizeof(T)));
  }

  template <class LD>
  __device__ __forceinline__ void run_part(int m, int n0, int p, int M, int N, const LD& ld) const {
    const T* rrow = resid_row(m, M, N, n0 == 0 && p == 0);
    const int n = n0 + 32 * p;
    float a[32], r[32];
    const bool ok = rrow && n < N;
    if (ok) load_row(rrow + n, r, 32);
    ld(32 * p, a);
    if (ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] += r[j];
      store_row(out + static_cast<size_t>(m) * N + n, a, 32);
    }
  }

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    const T* rrow = resid_row(m, M, N, n0 == 0);
    float a[32], r[32];
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      ld(c * 32, a);
      const int n = n0 + c * 32;
      if (rrow && n < N) {
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
  static constexpr int PARTS = 4;
  const float* rs;
  T* out;

  __device__ __forceinline__ void prefetch(int m, int, int M, int) const {
    if (m < M) prefetch_l1(rs + m, 4);
  }

  template <class LD>
  __device__ __forceinline__ void run_part(int m, int n0, int p, int M, int N, const LD& ld) const {
    const bool ok = m < M;
    const float sc = ok ? rs[m] : 0.f;
    float a[32];
    ld(32 * p, a);
    const int n = n0 + 32 * p;
    if (ok && n < N) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float x = a[j] * sc;
        a[j] = 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
      }
      store_row(out + static_cast<size_t>(m) * N + n, a, 32);
    }
  }

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
  static constexpr int PARTS = 1;   // tile statistics need the whole tile
  const float* rs;   // RMSNorm scale of each row of h
  int mask_id;
  LMPart* part;      // [M][n_tiles]
  int n_tiles;

  template <class LD>
  __device__ __forceinline__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const {
    run_slot(m, n0, nch, n0 / (32 * nch), M, N, ld);
  }

  // statistics of columns [n0, n0 + 32 nch) of row m into partial `slot`
  template <class LD>
  __device__ __forceinline__ void run_slot(int m, int n0, int nch, int slot, int M, int N, const LD& ld) const {
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
    if (ok) part[static_cast<size_t>(m) * n_tiles + slot] = LMPart{mx, S, A, idx};
  }

  __device__ __forceinline__ void prefetch(int, int, int, int) const {}

  template <class LD>
  __device__ __forceinline__ void run_part(int m, int n0, int, int M, int N, const LD& ld) const {
    run(m, n0, 4, M, N, ld);
  }
};

}  // namespace dllm
