// Cached attention with reuse of the online-softmax statistics of the
// unchanged key tiles ("LaCache", Methodology 1, FACache).
//
// Within an SAR block the prompt, the committed positions and the masked
// suffix keep their token ids, so their cached K/V rows do not change; only
// the key tiles that overlap the block's window [q0 - R, q0 + blk + R) can
// (the block's tokens are committed there, and the rows around them are
// re-projected).  For the block's queries the softmax over all keys splits
// into a part over the unchanged tiles U and a part over the window tiles W:
//   O = (e^(m_U - M) O~_U + e^(m_W - M) O~_W) / (e^(m_U - M) l_U + e^(m_W - M) l_W),
//   M = max(m_U, m_W),
// with (m, l, O~) the running maximum, normaliser and unnormalised
// accumulator of an online softmax.  The state (m_U, l_U, O~_U) of every
// (sequence, head, query) is kept in global memory with the key it is valid
// for: the block start q0, the block length and the token-at-write of every
// active row (a query row's Q is a function of that token and its
// position).  A CTA owns one (head, sequence):
//   * key unchanged: it streams only the W tiles and merges with the kept
//     state (the page seeds the accumulators from the cache; merging at the
//     end is the same sum in another order);
//   * otherwise (a block's first step, or a committed token): it streams the
//     U tiles, then the W tiles, into two TMEM accumulators with two online
//     softmax states, stores (m_U, l_U, O~_U) and the new key, and merges.
// The per-tile pipeline is the one of attn_tc_kernel (ring of K+V slots
// filled by bulk copies, S = Q K^T and O += P V on tcgen05 issued by one
// thread in a fixed order, P as a bf16 (hi, lo) pair in TMEM, R replicas of
// the queries in the 128 MMA rows, lazy rescaling in the log2 domain).
#pragma once
#include "attn_tc.cuh"

namespace dllm {
namespace attn_fa {

using attn_tc::KT;
using attn_tc::LAZY;
using attn_tc::QROWS;
// Two ring slots (K and V of two tiles) keep the CTA under 100 KB of shared
// memory, so two CTAs share an SM: the window-only pass of every (sequence,
// head) fits one wave, and a rebuild streams two CTAs' tiles per SM.
constexpr int NSLOT = 2;

constexpr int MAXQ = 64;                  // queries per (sequence, head) the state holds
constexpr int KEY_INTS = 2 + MAXQ;        // q0, q_len, token-at-write of each query row

template <int DH, int R>
struct Shape {
  static constexpr int QP = QROWS / R;
  static constexpr int KG = KT / R;
  static constexpr int Q_BYTES = QROWS * DH * 2;
  static constexpr int KV_TILE = KT * DH * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * 2 * KV_TILE;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  // TMEM: S/P double buffer, O~ of the window, then O~ of the unchanged
  // tiles (allocated only when the state is rebuilt)
  static constexpr uint32_t S_COL = 0, OW_COL = 2 * KT, OU_COL = 2 * KT + DH;
  static constexpr uint32_t COLS_W = (OW_COL + DH <= 256) ? 256 : 512;
  static constexpr uint32_t COLS_UW = (OU_COL + DH <= 256) ? 256 : 512;
  static constexpr int PLD = DH + 4;      // padded fp32 row of a partial
  // epilogue, one class at a time over the drained Q and ring: partial rows,
  // (m, l) pairs, merge weights
  static_assert(QROWS * PLD * 4 + QROWS * 8 + QROWS * 8 * 4 <= OFF_BAR, "tail fits in Q and the ring");
};

// Stored state row of (sequence, head, query): O~[DH], m (log2 domain), l.
__host__ __device__ constexpr int state_ld(int dh) { return dh + 4; }

// Ql, Kl, Vl: the layer's tiled caches.  Queries: positions [q_pos0,
// q_pos0 + q_len) of sequence blockIdx.y, head blockIdx.x; keys [0, kv_len)
// as n_all 64-key tiles, of which [w_lo, w_hi) are the window.  tok_w: the
// cache's token-at-write [B * L].  state: [B][H][MAXQ][DH + 4] fp32; key:
// [B][H][KEY_INTS] int32.  out [B][q_len][ld] bf16.
template <int DH, int R>
__global__ void __launch_bounds__(192, 2)
    attn_fa_kernel(const uint8_t* __restrict__ Ql, const uint8_t* __restrict__ Kl, const uint8_t* __restrict__ Vl,
                   KvLayout kv, int ld, int q_pos0, int q_len, int kv_len, int w_lo, int w_hi, float scale_log2,
                   const int* __restrict__ tok_w, int L, float* __restrict__ state, int* __restrict__ key,
                   const uint8_t* __restrict__ seq_done, bf16* __restrict__ out, unsigned* err,
                   int* __restrict__ rebuilt) {
  using S = Shape<DH, R>;
  using attn_tc::Bars;
  constexpr int QP = S::QP, KG = S::KG;
  const int h = blockIdx.x, b = blockIdx.y, H = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(sm + S::OFF_BAR);
  volatile int* abort = &bars->abort;

  const int n_all = cdiv(kv_len, KT);
  const int n_win = w_hi - w_lo;

  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
    }
    mbar_init(&bars->q_ready, 4);
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // the window tiles are read in every case: warm L2 with the first two
  if (warp >= 2 && lane == 0) {
    const int j = (warp - 2) >> 1;
    if (j < n_win) attn_tc::bulk_prefetch_l2(((warp & 1) ? Vl : Kl) + kv.tile_off(b, h, (w_lo + j) * KT), S::KV_TILE);
  }
  pdl_launch();
  pdl_wait();     // the cache rows and tokens of this step are written
  if (seq_done && seq_done[b]) return;     // the sequence has ended its block (no TMEM held yet)

  // ---- is the kept state valid for this block and these query tokens?
  int* mykey = key + static_cast<size_t>(b * H + h) * KEY_INTS;
  int same = 1;
  if (tid == 0) same = mykey[0] == q_pos0 && mykey[1] == q_len;
  if (tid >= 64 && tid - 64 < q_len) same = mykey[2 + tid - 64] == tok_w[static_cast<size_t>(b) * L + q_pos0 + tid - 64];
  const bool valid = __syncthreads_and(same) != 0;
  const int n_u = valid ? 0 : n_all - n_win;       // unchanged tiles streamed this time
  const uint32_t tmem_cols = n_u > 0 ? S::COLS_UW : S::COLS_W;
  if (warp == 1) tmem_alloc(&bars->tmem, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const int n_tiles = n_u + n_win;
  // virtual tile j -> physical 64-key tile
  auto phys = [&](int j) { return j < n_u ? (j < w_lo ? j : j + n_win) : w_lo + (j - n_u); };

  float m_ref = -INFINITY, l_sum = 0.f;      // the running state of the current class
  float m_u = -INFINITY, l_u = 0.f;          // the finished state of the unchanged tiles

  if (warp == 0) {
    if (lane < 4) {
      const bool is_k = (lane & 1) == 0;
      const uint8_t* src = is_k ? Kl : Vl;
      uint8_t* ring = sm + S::OFF_RING + (is_k ? 0 : S::KV_TILE);
      uint64_t* fullb = is_k ? bars->k_full : bars->v_full;
      uint32_t issued = 0, par = 0;
      for (int j = lane >> 1; j < n_tiles; j += 2) {
        const int s = j % NSLOT;
        const uint32_t ph = (j / NSLOT) & 1u;
        if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort, err)) break;
        mbar_expect_tx(&fullb[s], S::KV_TILE);
        bulk_load(ring + s * 2 * S::KV_TILE, src + kv.tile_off(b, h, phys(j) * KT), S::KV_TILE, &fullb[s]);
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
      }
      if (*abort)
        for (int s = 0; s < NSLOT; ++s)
          if (issued & (1u << s)) mbar_wait(&fullb[s], (par >> s) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(QROWS, KT);
      const uint32_t id_pv = attn_tc::idesc_bf16_bmn(QROWS, DH);
      const uint32_t q_base = smem_u32(sm + S::OFF_Q);
      auto issue_s = [&](int j) {
        const int sb = j & 1;
        tc_fence_after();
        const uint32_t kb = smem_u32(sm + S::OFF_RING + (j % NSLOT) * 2 * S::KV_TILE);
#pragma unroll
        for (int kc = 0; kc < DH / 16; ++kc)
          tc_mma_bf16(tmem + S::S_COL + sb * KT, sdesc_sw128(q_base + (kc >> 2) * (QROWS * 128) + (kc & 3) * 32),
                      sdesc_sw128(kb + (kc >> 2) * (KT * 128) + (kc & 3) * 32), id_s, kc > 0 ? 1u : 0u);
        tc_commit(&bars->s_full[sb]);
      };
      // O~ of the tile's class += P_i,hi V_i + P_i,lo V_i
      auto issue_pv = [&](int i) {
        const int s = i % NSLOT;
        const bool win = i >= n_u;
        const uint32_t o_col = win ? S::OW_COL : S::OU_COL;
        const int first = win ? n_u : 0;
        tc_fence_after();
        const uint32_t vb = smem_u32(sm + S::OFF_RING + s * 2 * S::KV_TILE + S::KV_TILE);
#pragma unroll
        for (int part = 0; part < attn_tc::P_PARTS; ++part) {
          const uint32_t pt = tmem + S::S_COL + (i & 1) * KT + part * (KT / 2);
#pragma unroll
          for (int k = 0; k < KT / 16; ++k)
            attn_tc::tc_mma_bf16_ta(tmem + o_col, pt + k * 8, attn_tc::sdesc_sw128_mn(vb + k * 2048), id_pv,
                                    (i > first || part > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&bars->empty[s]);
      };
      bool ok = n_tiles == 0 || (mbar_wait(&bars->q_ready, 0, abort, err) &&
                                 mbar_wait(&bars->k_full[0], 0, abort, err));
      if (ok && n_tiles > 0) issue_s(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          if (!mbar_wait(&bars->k_full[(j + 1) % NSLOT], ((j + 1) / NSLOT) & 1u, abort, err)) break;
          issue_s(j + 1);
        }
        if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1u, abort, err)) break;
        issue_pv(j);
      }
      tc_commit(&bars->done);
      mbar_wait(&bars->done, 0, nullptr, err);
    }
  } else {
    {   // stage Q: row g * QP + r holds query r (zero past q_len)
      const int st = tid - 64;
      constexpr int NQ = QP * (DH / 8), PER = (NQ + 127) / 128;
      uint4 v[PER];
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int e = st + u * 128, r = e / (DH / 8), c = e % (DH / 8);
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (e < NQ && r < q_len) v[u] = *reinterpret_cast<const uint4*>(Ql + kv.chunk_off(b, h, q_pos0 + r, c));
      }
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int e = st + u * 128, r = e / (DH / 8), c = e % (DH / 8);
        if (e >= NQ) continue;
#pragma unroll
        for (int g2 = 0; g2 < R; ++g2)
          *reinterpret_cast<uint4*>(sm + S::OFF_Q + (c >> 3) * (QROWS * 128) + attn_tc::sw128_off(g2 * QP + r, c & 7)) =
              v[u];
      }
      attn_tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_ready);
    }
    const int wq = warp & 3;
    const int m = wq * 32 + lane, g = m / QP, r = m % QP;
    const bool valid_row = r < q_len;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      const bool win = j >= n_u;
      if (j == n_u && n_u > 0) {      // the unchanged tiles are done: a fresh state for the window
        m_u = m_ref;
        l_u = l_sum;
        m_ref = -INFINITY;
        l_sum = 0.f;
      }
      const int first = win ? n_u : 0;
      const uint32_t o_col = win ? S::OW_COL : S::OU_COL;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bars->s_full[sb], (j >> 1) & 1u, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      float sv[KG];
      {
        const uint32_t col = tmem + lane_off + S::S_COL + sb * KT;
        if constexpr (KG == 16) {
          attn_tc::tmem_ld16(col + g * 16, sv);
        } else if constexpr (KG == 32) {
          float t[32];
          tmem_ld32(col + g * 32, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[i] = t[i];
        } else {
          float t0[32], t1[32];
          tmem_ld32(col, t0);
          tmem_ld32(col + 32, t1);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            sv[i] = t0[i];
            sv[i + 32] = t1[i];
          }
        }
      }
      const int key0 = phys(j) * KT + g * KG;
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < KG; ++i) {
        sv[i] = (valid_row && key0 + i < kv_len) ? sv[i] * scale_log2 : -INFINITY;
        mt = fmaxf(mt, sv[i]);
      }
      float alpha = 1.f;
      bool moved = false;
      if (mt > m_ref + LAZY || (m_ref == -INFINITY && mt != -INFINITY)) {
        alpha = m_ref == -INFINITY ? 0.f : exp2f(m_ref - mt);
        m_ref = mt;
        moved = j > first && alpha != 1.f;
      }
      float ls = 0.f;
#pragma unroll
      for (int i = 0; i < KG; ++i) {
        sv[i] = m_ref == -INFINITY ? 0.f : ex2_fast(sv[i] - m_ref);
        ls += sv[i];
      }
      l_sum = l_sum * alpha + ls;
      if (__any_sync(0xffffffffu, moved)) {
        int ok2 = 1;
        if (lane == 0) ok2 = mbar_wait(&bars->empty[(j - 1) % NSLOT], ((j - 1) / NSLOT) & 1u, abort, err) ? 1 : 0;
        ok2 = __shfl_sync(0xffffffffu, ok2, 0);
        if (!ok2) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DH / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_off + o_col + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          attn_tc::tmem_st32(tmem + lane_off + o_col + c * 32, o);
        }
      }
      {
        uint32_t ph[KG / 2], pl[KG / 2];
#pragma unroll
        for (int i = 0; i < KG / 2; ++i) {
          const float a = sv[2 * i], bb = sv[2 * i + 1];
          const __nv_bfloat162 hb = __floats2bfloat162_rn(a, bb);
          const float2 hf = __bfloat1622float2(hb);
          ph[i] = valid_row ? *reinterpret_cast<const uint32_t*>(&hb) : 0u;
          pl[i] = valid_row ? attn_tc::pack2(a - hf.x, bb - hf.y) : 0u;
        }
        uint32_t hi[KT / 2], lo[KT / 2];
#pragma unroll
        for (int gg = 0; gg < R; ++gg)
#pragma unroll
          for (int i = 0; i < KG / 2; ++i) {
            hi[gg * (KG / 2) + i] = gg == g ? ph[i] : 0u;
            lo[gg * (KG / 2) + i] = gg == g ? pl[i] : 0u;
          }
        const uint32_t pt = tmem + lane_off + S::S_COL + sb * KT;
        attn_tc::tmem_st32u(pt, hi);
        if constexpr (attn_tc::P_PARTS == 2) attn_tc::tmem_st32u(pt + KT / 2, lo);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      tc_fence_before();
      __syncwarp();
      int okv = 1;
      if (lane == 0) {
        okv = mbar_wait(&bars->v_full[j % NSLOT], (j / NSLOT) & 1u, abort, err) ? 1 : 0;
        if (okv) mbar_arrive(&bars->p_full[sb]);
      }
      okv = __shfl_sync(0xffffffffu, okv, 0);
      if (!okv) break;
    }
  }

  // ---- the partials, one class at a time, over the drained Q and ring:
  //   po[m][PLD] fp32 O~ row of MMA row m = g * QP + r, pml[m] = (m, l);
  // the unchanged tiles' class (rebuilt) goes to the kept state in global
  // memory, then the window's class stays in po for the merge
  tc_fence_before();
  __syncthreads();
  float* po = reinterpret_cast<float*>(sm + S::OFF_Q);
  float* pml = po + QROWS * S::PLD;                        // [QROWS][2]
  float* wts = pml + QROWS * 2;                            // [QROWS][8]
  float* my_state = state + static_cast<size_t>(b * H + h) * MAXQ * state_ld(DH);
  int last_ok = 1;
  if (warp >= 2 && n_tiles > 0) {
    if (lane == 0)
      last_ok = mbar_wait(&bars->empty[(n_tiles - 1) % NSLOT], ((n_tiles - 1) / NSLOT) & 1u, abort, err) ? 1 : 0;
    last_ok = __shfl_sync(0xffffffffu, last_ok, 0);
    tc_fence_after();
  }
#pragma unroll 1
  for (int cls = 0; cls < 2; ++cls) {
    if (cls == 0 && valid) continue;                       // the kept state stays
    // a rebuild with no unchanged tile (every tile in the window) stores the
    // empty state: m = -inf, l = 0, O~ = 0 (no TMEM columns were allocated)
    const bool from_tmem = cls == 1 || n_u > 0;
    if (warp >= 2) {
      const int wq = warp & 3;
      const int m = wq * 32 + lane, r = m % QP;
      const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
      const uint32_t o_col = cls == 0 ? S::OU_COL : S::OW_COL;
#pragma unroll 1
      for (int c = 0; c < DH / 32; ++c) {
        float o[32];
        if (from_tmem) {
          tmem_ld32(tmem + lane_off + o_col + c * 32, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (r < q_len) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(po + m * S::PLD + c * 32 + i) =
                last_ok ? make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (r < q_len) {
        pml[m * 2] = cls == 0 ? (n_u > 0 ? m_u : -INFINITY) : (n_win > 0 ? m_ref : -INFINITY);
        pml[m * 2 + 1] = cls == 0 ? (n_u > 0 ? l_u : 0.f) : l_sum;
      }
    }
    __syncthreads();
    // replicas of a query: weight each by 2^(m_g - M), sum into replica 0's
    // row, which then holds M, sum w l, sum w O~
    if constexpr (R > 1) {
      for (int r = tid; r < q_len; r += 192) {
        float M = -INFINITY;
#pragma unroll
        for (int g = 0; g < R; ++g) M = fmaxf(M, pml[(g * QP + r) * 2]);
        float l = 0.f;
#pragma unroll
        for (int g = 0; g < R; ++g) {
          const float mg = pml[(g * QP + r) * 2];
          const float w = mg == -INFINITY ? 0.f : exp2f(mg - M);
          wts[r * 8 + g] = w;
          l += w * pml[(g * QP + r) * 2 + 1];
        }
        wts[r * 8 + 7] = M;
        wts[r * 8 + 6] = l;
      }
      __syncthreads();
      for (int e = tid; e < q_len * (DH / 4); e += 192) {
        const int r = e / (DH / 4), c = (e % (DH / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int g = 0; g < R; ++g) {
          const float w = wts[r * 8 + g];
          const float4 v = *reinterpret_cast<const float4*>(po + (g * QP + r) * S::PLD + c);
          acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
        }
        *reinterpret_cast<float4*>(po + r * S::PLD + c) = acc;
      }
      __syncthreads();
      for (int r = tid; r < q_len; r += 192) {
        pml[r * 2] = wts[r * 8 + 7];
        pml[r * 2 + 1] = wts[r * 8 + 6];
      }
      __syncthreads();
    }
    if (cls == 0) {   // store the rebuilt state of the unchanged tiles
      for (int e = tid; e < q_len * (DH / 4); e += 192) {
        const int r = e / (DH / 4), c = (e % (DH / 4)) * 4;
        *reinterpret_cast<float4*>(my_state + r * state_ld(DH) + c) =
            *reinterpret_cast<const float4*>(po + r * S::PLD + c);
      }
      for (int r = tid; r < q_len; r += 192) {
        my_state[r * state_ld(DH) + DH] = pml[r * 2];
        my_state[r * state_ld(DH) + DH + 1] = pml[r * 2 + 1];
      }
      __syncthreads();      // the state is written before the merge reads it back
    }
  }
  // O = (w_U O~_U + w_W O~_W) / (w_U l_U + w_W l_W), O~_U from the kept state
  for (int r = tid; r < q_len; r += 192) {
    const float mu = my_state[r * state_ld(DH) + DH], mw = pml[r * 2];
    const float M = fmaxf(mu, mw);
    const float wu = mu == -INFINITY ? 0.f : exp2f(mu - M);
    const float ww = mw == -INFINITY ? 0.f : exp2f(mw - M);
    const float inv = 1.f / (wu * my_state[r * state_ld(DH) + DH + 1] + ww * pml[r * 2 + 1]);
    wts[r * 8] = wu * inv;
    wts[r * 8 + 1] = ww * inv;
  }
  __syncthreads();
  for (int e = tid; e < q_len * (DH / 4); e += 192) {
    const int r = e / (DH / 4), c = (e % (DH / 4)) * 4;
    const float wu = wts[r * 8], ww = wts[r * 8 + 1];
    const float4 u = *reinterpret_cast<const float4*>(my_state + r * state_ld(DH) + c);
    const float4 v = *reinterpret_cast<const float4*>(po + r * S::PLD + c);
    bf16* op = out + static_cast<size_t>(b * q_len + r) * ld + h * DH + c;
    *reinterpret_cast<__nv_bfloat162*>(op) = __floats2bfloat162_rn(fmaf(wu, u.x, ww * v.x), fmaf(wu, u.y, ww * v.y));
    *reinterpret_cast<__nv_bfloat162*>(op + 2) = __floats2bfloat162_rn(fmaf(wu, u.z, ww * v.z), fmaf(wu, u.w, ww * v.w));
  }
  // the key the stored state is valid for (only this CTA reads or writes it)
  if (!valid && !*abort) {
    if (tid == 0) {
      mykey[0] = q_pos0;
      mykey[1] = q_len;
      if (rebuilt) atomicAdd(rebuilt, 1);
    }
    if (tid >= 64 && tid - 64 < q_len) mykey[2 + tid - 64] = tok_w[static_cast<size_t>(b) * L + q_pos0 + tid - 64];
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace attn_fa
}  // namespace dllm
