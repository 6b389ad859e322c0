// Cached attention for queries given as a sorted list of flat rows b * L + pos
// (every row that passes through the layer stack of a multi-layer step):
// each query attends over all L cached positions of its own sequence.
//
// Persistent kernel, as many CTAs per SM as fit (two at dh 64, where a CTA
// takes about 107 KB of shared memory and 256 TMEM columns; one at dh 128).
// A work item is (sequence b, query tile
// of up to 128 of its rows, head h); items are numbered in (b, tile) order,
// heads fastest, and CTA i takes items i, i + gridDim.x, ...  The per-sequence
// row ranges come from a binary search of the sorted list at kernel start.
// Within an item there is one query per MMA row (no replicas, no key
// splits).  Lanes 0-3 of warp 0 stream K and V tiles through separate rings
// (lanes 0/2 K, 1/3 V, even and odd tiles).  One thread of warp 1 issues
// S = Q K^T and O += P_hi V + P_lo V on tcgen05 as each one's inputs are
// ready, polling the barriers (P is kept in TMEM over S).  Warps 2-5 run the
// online softmax, one query of 64 keys per thread per tile, and after the
// last tile normalise O and store it.  The barrier phases run on a tile
// counter shared by all items of the CTA.  Unlike attn_tc_kernel, whose
// issuing thread limits it, this kernel is bound by its softmax: a fixed
// issue order with one K+V ring and P in TMEM buffers of its own measured
// slower here (all 16 x 2048 rows of a 64-dim layer: 1202-1274 against
// 1109 us).
#pragma once
#include "attn_tc.cuh"

namespace dllm {
namespace attn_rows {

using attn_tc::KT;
using attn_tc::LAZY;
constexpr int KS = 5, VS = 6, QROWS = 128, MAX_SEQ = 256;

template <int DH>
struct Shape {
  static constexpr int Q_BYTES = QROWS * DH * 2;
  static constexpr int KV_TILE = KT * DH * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + KS * KV_TILE;
  static constexpr int OFF_SEQ = OFF_V + VS * KV_TILE;  // [MAX_SEQ + 1] first item, [MAX_SEQ + 1] first row
  static constexpr int OFF_BAR = OFF_SEQ + (2 * MAX_SEQ + 2) * 4;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr uint32_t TMEM_COLS = 256;           // S / P: 2 x 64 columns, O: DH columns
  static constexpr uint32_t S_COL = 0, O_COL = 128;
};

struct Bars {
  uint64_t k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t q_ready, done;
  uint32_t tmem;
  int abort;
};

// rows [0, n) sorted ascending; out [n][ld] bf16 (ld = H * DH).
template <int DH>
__global__ void __launch_bounds__(192, 1)
    attn_rows_kernel(const uint8_t* __restrict__ Ql, const uint8_t* __restrict__ Kl,
                     const uint8_t* __restrict__ Vl, KvLayout kv, int L, int n_seq, int n_heads,
                     const int* __restrict__ rows, const int* __restrict__ n_rows, int rows_cap, float scale_log2,
                     bf16* __restrict__ out, unsigned* err) {
  using S = Shape<DH>;
  using attn_tc::sw128_off;
  using attn_tc::pack2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(sm + S::OFF_BAR);
  int* first_item = reinterpret_cast<int*>(sm + S::OFF_SEQ);   // [n_seq + 1], in (b, tile) units
  int* row_start = first_item + MAX_SEQ + 1;                     // [n_seq + 1]
  volatile int* abort = &bars->abort;
  pdl_launch();
  pdl_wait();
  const int n = min(*n_rows, rows_cap);
  const int n_tiles = cdiv(L, KT);

  if (tid == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->q_ready, 4);
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  // per-sequence row ranges: rows of sequence b are [start_b, start_{b+1})
  for (int b = tid; b <= n_seq; b += 192) {
    int lo = 0, hi = n;   // first index with rows[i] >= b * L
    const long long key = static_cast<long long>(b) * L;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (rows[mid] < key) lo = mid + 1; else hi = mid;
    }
    row_start[b] = lo;    // rows past the last sequence (out of range) are left out
    first_item[b] = lo;   // overwritten below with tile prefix sums
  }
  if (warp == 1) tmem_alloc(&bars->tmem, S::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {   // row starts -> prefix sums of query tiles per sequence
    int acc = 0;
    for (int b = 0; b < n_seq; ++b) {
      const int cnt = row_start[b + 1] - row_start[b];
      first_item[b] = acc;
      acc += cdiv(cnt, QROWS);
    }
    first_item[n_seq] = acc;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const int n_items = first_item[n_seq] * n_heads;
  // item -> (b, query tile, head)
  auto decode = [&](int item, int& b, int& qt, int& h) {
    h = item % n_heads;
    const int bt = item / n_heads;
    int lo = 0, hi = n_seq - 1;   // last b with first_item[b] <= bt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (first_item[mid] <= bt) lo = mid; else hi = mid - 1;
    }
    b = lo;
    qt = bt - first_item[b];
  };

  if (warp == 0) {
    // lanes 0/2 stream K, lanes 1/3 V (even and odd tiles of the CTA's
    // running tile count J: two issuers per ring)
    if (lane < 4) {
      const bool is_k = (lane & 1) == 0;
      const int sub = lane >> 1;
      const uint8_t* src = is_k ? Kl : Vl;
      const int slots = is_k ? KS : VS;
      uint64_t* fullb = is_k ? bars->k_full : bars->v_full;
      uint64_t* emptyb = is_k ? bars->k_empty : bars->v_empty;
      uint8_t* ring = sm + (is_k ? S::OFF_K : S::OFF_V);
      uint32_t issued = 0, par = 0;
      int J = 0;   // tile counter over all items of this CTA
      for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
        int b, qt, h;
        decode(item, b, qt, h);
        for (int j = 0; j < n_tiles; ++j, ++J) {
          if ((J & 1) != sub) continue;
          const int s = J % slots;
          const uint32_t ph = (J / slots) & 1u;
          if (!mbar_wait(&emptyb[s], ph ^ 1u, abort, err)) break;
          mbar_expect_tx(&fullb[s], S::KV_TILE);
          bulk_load(ring + s * S::KV_TILE, src + kv.tile_off(b, h, j * KT), S::KV_TILE, &fullb[s]);
          issued |= 1u << s;
          par = (par & ~(1u << s)) | (ph << s);
        }
      }
      if (*abort)
        for (int s = 0; s < slots; ++s)
          if (issued & (1u << s)) mbar_wait(&fullb[s], (par >> s) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(QROWS, KT);
      const uint32_t id_pv = attn_tc::idesc_bf16_bmn(QROWS, DH);
      const uint32_t q_base = smem_u32(sm + S::OFF_Q);
      // the CTA's tiles J = 0, 1, ... run through its items in order; every
      // item has n_tiles tiles, so tile J belongs to item J / n_tiles
      const int my_items = blockIdx.x < n_items ? (n_items - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
      const int total = my_items * n_tiles;
      auto issue_s = [&](int J) {
        const int ks = J % KS, sb = J & 1;
        tc_fence_after();
        const uint32_t kb = smem_u32(sm + S::OFF_K + ks * S::KV_TILE);
#pragma unroll
        for (int kc = 0; kc < DH / 16; ++kc)
          tc_mma_bf16(tmem + S::S_COL + sb * KT, sdesc_sw128(q_base + (kc >> 2) * (QROWS * 128) + (kc & 3) * 32),
                      sdesc_sw128(kb + (kc >> 2) * (KT * 128) + (kc & 3) * 32), id_s, kc > 0 ? 1u : 0u);
        tc_commit(&bars->s_full[sb]);
        tc_commit(&bars->k_empty[ks]);
      };
      // O += P_J V_J with P from TMEM, N = DH in one MMA per 16 keys; the
      // first tile of an item overwrites O
      auto issue_pv = [&](int J) {
        const int pb = J & 1, vs = J % VS;
        const bool first = J % n_tiles == 0;
        tc_fence_after();
        const uint32_t vb = smem_u32(sm + S::OFF_V + vs * S::KV_TILE);
#pragma unroll
        for (int part = 0; part < attn_tc::P_PARTS; ++part) {
          const uint32_t pt = tmem + S::S_COL + pb * KT + part * (KT / 2);
#pragma unroll
          for (int k = 0; k < KT / 16; ++k)
            attn_tc::tc_mma_bf16_ta(tmem + S::O_COL, pt + k * 8, attn_tc::sdesc_sw128_mn(vb + k * 2048), id_pv,
                                    (!first || part > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&bars->pv_done[pb]);
        tc_commit(&bars->v_empty[vs]);
      };
      int js = 0, jp = 0;
      uint32_t idle = 0;
      uint64_t t_idle = 0;
      while (jp < total) {
        bool did = false;
        // S_js: its K tile, the item's Q (first tile), and P_{js-2} V_{js-2}
        // issued (S_js overwrites P_{js-2}; the MMAs run in order)
        if (js < total && js <= jp + 1 && mbar_test(&bars->k_full[js % KS], (js / KS) & 1u) &&
            (js % n_tiles != 0 || mbar_test(&bars->q_ready, static_cast<uint32_t>(js / n_tiles) & 1u))) {
          issue_s(js++);
          did = true;
        }
        if (jp < js && mbar_test(&bars->p_full[jp & 1], (jp >> 1) & 1u) &&
            mbar_test(&bars->v_full[jp % VS], (jp / VS) & 1u)) {
          issue_pv(jp++);
          did = true;
        }
        if (did) {
          idle = 0;
          continue;
        }
        if (idle++ == 0) {
          t_idle = globaltimer_ns();
        } else if ((idle & 63) == 0) {
          if (*abort) break;
          if (globaltimer_ns() - t_idle > kWaitLimitNs) {
            set_err(err, DLLM_ERR_TIMEOUT);
            *abort = 1;
            break;
          }
        }
      }
      tc_commit(&bars->done);
      mbar_wait(&bars->done, 0, nullptr, err);
    }
  } else {
    const int wq = warp & 3, m = wq * 32 + lane;   // this thread's query row (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int st = tid - 64;                        // 128 staging threads
    int J = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      int b, qt, h;
      decode(item, b, qt, h);
      const int r0 = row_start[b] + qt * QROWS;
      const int r_end = row_start[b + 1];
      const int nq = min(QROWS, r_end - r0);
      // ---- stage Q of rows r0 .. r0 + nq (zero past nq); the previous item's
      // S MMAs are done (its last P V has completed before we got here)
      {   // all loads in flight before the stores
        constexpr int PER = QROWS * (DH / 8) / 128;
        uint4 v[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int e = st + u * 128, q = e / (DH / 8), c = e % (DH / 8);
          v[u] = make_uint4(0u, 0u, 0u, 0u);
          if (q < nq) v[u] = *reinterpret_cast<const uint4*>(Ql + kv.chunk_off(b, h, rows[r0 + q] - b * L, c));
        }
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const int e = st + u * 128, q = e / (DH / 8), c = e % (DH / 8);
          *reinterpret_cast<uint4*>(sm + S::OFF_Q + (c >> 3) * (QROWS * 128) + sw128_off(q, c & 7)) = v[u];
        }
      }
      attn_tc::fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_ready);

      const bool valid = m < nq;
      float m_ref = -INFINITY, l_sum = 0.f;
      for (int j = 0; j < n_tiles; ++j, ++J) {
        const int sb = J & 1;
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&bars->s_full[sb], (J >> 1) & 1u, abort, err) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        float sv[KT];
        {
          float t0[32], t1[32];
          const uint32_t col = tmem + lane_off + S::S_COL + sb * KT;
          tmem_ld32(col, t0);
          tmem_ld32(col + 32, t1);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            sv[i] = t0[i];
            sv[i + 32] = t1[i];
          }
        }
        const int key0 = j * KT;
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < KT; ++i) {
          sv[i] = (valid && key0 + i < L) ? sv[i] * scale_log2 : -INFINITY;
          mt = fmaxf(mt, sv[i]);
        }
        float alpha = 1.f;
        bool moved = false;
        if (mt > m_ref + LAZY || (m_ref == -INFINITY && mt != -INFINITY)) {
          alpha = m_ref == -INFINITY ? 0.f : exp2f(m_ref - mt);
          m_ref = mt;
          moved = j > 0 && alpha != 1.f;
        }
        float ls = 0.f;
#pragma unroll
        for (int i = 0; i < KT; ++i) {
          sv[i] = m_ref == -INFINITY ? 0.f : ex2_fast(sv[i] - m_ref);
          ls += sv[i];
        }
        l_sum = l_sum * alpha + ls;
        if (__any_sync(0xffffffffu, moved)) {   // rescale O after the previous P V
          int ok2 = 1;
          if (lane == 0) ok2 = mbar_wait(&bars->pv_done[(J - 1) & 1], ((J - 1) >> 1) & 1u, abort, err) ? 1 : 0;
          ok2 = __shfl_sync(0xffffffffu, ok2, 0);
          if (!ok2) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DH / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_off + S::O_COL + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            attn_tc::tmem_st32(tmem + lane_off + S::O_COL + c * 32, o);
          }
        }
        // P_J over S_J in TMEM as hi + lo bf16 pairs (zeros past the tile's rows)
        {
          uint32_t hi[KT / 2], lo[KT / 2];
#pragma unroll
          for (int i = 0; i < KT / 2; ++i) {
            const float a = sv[2 * i], bb = sv[2 * i + 1];
            const __nv_bfloat162 hb = __floats2bfloat162_rn(a, bb);
            const float2 hf = __bfloat1622float2(hb);
            hi[i] = valid ? *reinterpret_cast<const uint32_t*>(&hb) : 0u;
            lo[i] = valid ? pack2(a - hf.x, bb - hf.y) : 0u;
          }
          const uint32_t pt = tmem + lane_off + S::S_COL + sb * KT;
          attn_tc::tmem_st32u(pt, hi);
          if constexpr (attn_tc::P_PARTS == 2) attn_tc::tmem_st32u(pt + KT / 2, lo);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[sb]);
      }
      if (!ok) break;
      // ---- the item's last P V done: O / l for this thread's query
      {
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&bars->pv_done[(J - 1) & 1], ((J - 1) >> 1) & 1u, abort, err) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        bf16* orow = out + static_cast<size_t>(r0 + m) * (n_heads * DH) + h * DH;
#pragma unroll 1
        for (int c = 0; c < DH / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_off + S::O_COL + c * 32, o);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= inv;
            store_row(orow + c * 32, o, 32);
          }
        }
        tc_fence_before();   // O reads ordered before the next item's first P V
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

}  // namespace attn_rows
}  // namespace dllm
