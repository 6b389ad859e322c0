// Cached attention on the 5th-generation tensor cores (bf16).
//
// One CTA = (key split, head, sequence); clusters of n_split CTAs along the
// key splits.  Four lanes of warp 0 stream 64-key tiles into a ring of
// NSLOT slots, each holding tile j's K and V (one bulk copy each: the cache
// stores every tile as the 128-byte-swizzled image the tensor cores read;
// lanes 0/1 take the K/V of even tiles, lanes 2/3 of odd ones, as one
// thread's bulk copies are served one after another).  One thread of warp 1
// issues, in a fixed order (S_{j+1} before P_j V_j),
//   S_j = Q K_j^T    M = 128 query rows, N = 64 keys, into one of two TMEM
//                    buffers (64 columns each),
//   O  += P_j,hi V_j + P_j,lo V_j   M = 128, N = DH, K = 16,
// with P read from TMEM as a bf16 pair (hi + lo, so that O keeps fp32-level
// accuracy; P_j overwrites S_j in place, and the fixed order puts S_{j+2}
// behind P_j V_j) and V as an MN-major operand straight from its tile.  At these sizes the issuing thread spends 50-65 clocks per
// MMA and about as much per commit or barrier test, so a tile costs it 16
// MMAs, 2 commits (S_j done; P_j V_j done, which frees the slot) and 2
// blocking waits (K_j landed; P_j written, which the softmax signals only
// once V_j has landed too).  The 128 MMA rows hold R replicas
// of the block's queries, row g * QP + r for replica g of query r; replica
// g's softmax thread (thread = row = TMEM lane, warps 2-5) takes only the
// tile's key columns [g 64/R, (g + 1) 64/R) and keeps its own running
// maximum, so a replica row is an independent partial softmax over its key
// group.  The online softmax runs in the log2 domain with a lazy reference
// (moved only when the max grows by more than 2^8, and then O is rescaled in
// TMEM).  A thread writes its whole P row: its segment, zeros elsewhere.  The partials (m, l, O) of every
// replica and every split are merged across the cluster through distributed
// shared memory.
#pragma once
#include "common.cuh"

namespace dllm {
namespace attn_tc {

constexpr int KT = 64;                  // keys per tile
constexpr int NSLOT = 6;                // ring slots (K and V of one tile each)
constexpr int QROWS = 128;              // MMA M (query rows, padded)
constexpr float LAZY = 8.f;             // log2 headroom before the reference moves
// P in TMEM for the P V products: 2 = a (hi, lo) bf16 pair whose sum
// carries P to about 16 bits (two MMAs per 16 keys); 1 = bf16 P alone, about
// 14% faster, but its 8-bit rounding of P moves O by up to 1.6e-2 when few
// keys carry the weight (a sink ring's first tokens)
constexpr int P_PARTS = 2;

template <int DH, int R>
struct Shape {
  static constexpr int QP = QROWS / R;                // queries per replica
  static constexpr int KG = KT / R;                   // keys per softmax thread
  static constexpr int SUB = DH / 64;                 // 64-dim sub-tiles
  static constexpr int Q_BYTES = QROWS * DH * 2;
  static constexpr int KV_TILE = KT * DH * 2;         // one K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;    // slot s: K at s * 2 KV_TILE, V after it
  static constexpr int OFF_BAR = OFF_RING + NSLOT * 2 * KV_TILE;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  // S_j: 64 fp32 columns of buffer j & 1, overwritten in place by P_j as
  // bf16 pairs (hi: columns 0-31, lo: 32-63); O: DH columns
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t S_COL = 0, O_COL = 2 * KT;
  static_assert(O_COL + DH <= TMEM_COLS, "TMEM budget");
  // tail: partials reuse the drained ring
  static constexpr int PLD = DH + 4;                  // padded fp32 row
  static_assert(QROWS * PLD * 4 + QROWS * 8 + QROWS * 8 * 4 <= NSLOT * 2 * KV_TILE, "tail fits in the ring");
};

struct Bars {
  uint64_t k_full[NSLOT], v_full[NSLOT], empty[NSLOT];
  uint64_t s_full[2], p_full[2];
  uint64_t q_ready, done;
  uint32_t tmem;
  int abort;
};

// K-major smem descriptor with the 128-byte swizzle is sdesc_sw128 (common).
// MN-major, 128-byte swizzle, one 64-element MN atom per MMA: K rows 128 B
// apart, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(8192 >> 4) << 16;                 // next 64-wide MN atom (N = 128)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16_bmn(int M, int N) {   // B MN-major
  return idesc_bf16(M, N) | (1u << 16);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// D += A B with A (M x 16 bf16, packed in pairs along TMEM columns, one row
// per lane) read from TMEM and B from shared memory.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 consecutive fp32 columns from TMEM (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}


__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float ld_peer_f(const float* p, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

template <int PER>
__device__ __forceinline__ void ld_peer_v(const float* p, int rank, float (&v)[PER]) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  if constexpr (PER == 4) {
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(ra)
                 : "memory");
  } else {
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v[0]), "=f"(v[1]) : "r"(ra) : "memory");
  }
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Bring `bytes` (a multiple of 16) at a 16-byte aligned address into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// Ql, Kl, Vl: the layer's tiled Q/K/V caches (KvLayout kv).  Queries are
// positions [q_pos0, q_pos0 + q_len) of sequence blockIdx.z, keys/values its
// positions [0, kv_len); out [n_seq][q_len][ld] bf16.
template <int DH, int R>
__global__ void __launch_bounds__(192, 1)
    attn_tc_kernel(const uint8_t* __restrict__ Ql, const uint8_t* __restrict__ Kl, const uint8_t* __restrict__ Vl,
                   KvLayout kv, int ld, int q_pos0, int q_len, int kv_len, int keys_per_split, float scale_log2,
                   const uint8_t* __restrict__ seq_done, bf16* __restrict__ out, unsigned* err) {
  using S = Shape<DH, R>;
  constexpr int QP = S::QP, KG = S::KG;
  static_assert(sizeof(Bars) <= 256, "barrier block");
  const int split = blockIdx.x, n_split = gridDim.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(sm + S::OFF_BAR);
  volatile int* abort = &bars->abort;

  const int k_begin = split * keys_per_split;
  const int k_end = min(kv_len, k_begin + keys_per_split);
  const int n_tiles = k_end > k_begin ? cdiv(k_end - k_begin, KT) : 0;

  // ---- barriers and TMEM first, so that the K/V streams start at once
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
  if (warp == 1) tmem_alloc(&bars->tmem, S::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  // K and V of the first two tiles into L2 while the projection may still
  // run (it writes only the refreshed rows, and L2 is where they meet): one
  // bulk prefetch per warp, as one warp's bulk operations issue one by one
  if (warp >= 2 && lane == 0) {
    const int j = (warp - 2) >> 1;
    if (j < n_tiles) bulk_prefetch_l2(((warp & 1) ? Vl : Kl) + kv.tile_off(b, h, k_begin + j * KT), S::KV_TILE);
  }
  pdl_launch();
  pdl_wait();     // the cache rows of this step are written by the projection
  // a sequence that has ended its block (every CTA of the cluster shares b):
  // no attention, leave before any cluster barrier
  if (seq_done && seq_done[b]) {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, S::TMEM_COLS);
    }
    return;
  }

  // per-row results of the softmax warps (kept for the merge)
  float m_ref = -INFINITY, l_sum = 0.f;

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
        bulk_load(ring + s * 2 * S::KV_TILE, src + kv.tile_off(b, h, k_begin + j * KT), S::KV_TILE, &fullb[s]);
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
      }
      if (*abort)   // drain this lane's copies in flight
        for (int s = 0; s < NSLOT; ++s)
          if (issued & (1u << s)) mbar_wait(&fullb[s], (par >> s) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(QROWS, KT);
      const uint32_t id_pv = idesc_bf16_bmn(QROWS, DH);
      const uint32_t q_base = smem_u32(sm + S::OFF_Q);
      // S_j = Q K_j^T into TMEM S buffer j & 1, where P_{j-2} was: P_{j-2}
      // V_{j-2} is issued before it, and the MMAs run in order
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
      // O += P_i,hi V_i + P_i,lo V_i
      auto issue_pv = [&](int i) {
        const int s = i % NSLOT;
        tc_fence_after();
        const uint32_t vb = smem_u32(sm + S::OFF_RING + s * 2 * S::KV_TILE + S::KV_TILE);
        // N = DH in one MMA: the V tile's 64-dim halves are MN atoms 8 KB apart
#pragma unroll
        for (int part = 0; part < P_PARTS; ++part) {
          const uint32_t pt = tmem + S::S_COL + (i & 1) * KT + part * (KT / 2);   // P_i hi / lo in TMEM
#pragma unroll
          for (int k = 0; k < KT / 16; ++k)
            tc_mma_bf16_ta(tmem + S::O_COL, pt + k * 8, sdesc_sw128_mn(vb + k * 2048), id_pv,
                           (i > 0 || part > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&bars->empty[s]);   // P_i V_i done: slot s free
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
    // ---- stage Q: row g * QP + r holds query r (zero past q_len); every
    // (query, chunk) is loaded once, all loads in flight before the stores
    {
      const int st = tid - 64;   // 128 staging threads
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
          *reinterpret_cast<uint4*>(sm + S::OFF_Q + (c >> 3) * (QROWS * 128) + sw128_off(g2 * QP + r, c & 7)) = v[u];
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_ready);
    }
    // softmax warps: thread = MMA row m = TMEM lane = replica g of query r,
    // owning the tile's key columns [g * KG, g * KG + KG)
    const int wq = warp & 3;
    const int m = wq * 32 + lane, g = m / QP, r = m % QP;
    const bool valid = r < q_len;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bars->s_full[sb], (j >> 1) & 1u, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      float sv[KG];
      {
        const uint32_t col = tmem + lane_off + S::S_COL + sb * KT;
        // g is the same for every lane of a warp (QP is a multiple of 32)
        if constexpr (KG == 16) {
          tmem_ld16(col + g * 16, sv);
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
      // this segment's maximum against the row's reference
      const int key0 = k_begin + j * KT + g * KG;
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < KG; ++i) {
        sv[i] = (valid && key0 + i < k_end) ? sv[i] * scale_log2 : -INFINITY;
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
      for (int i = 0; i < KG; ++i) {
        sv[i] = m_ref == -INFINITY ? 0.f : ex2_fast(sv[i] - m_ref);
        ls += sv[i];
      }
      l_sum = l_sum * alpha + ls;
      // rescale this warp's rows of O once the previous P V has landed (the
      // commit of P_i V_i completes phase i / NSLOT of slot i % NSLOT)
      if (__any_sync(0xffffffffu, moved)) {
        int ok2 = 1;
        if (lane == 0) ok2 = mbar_wait(&bars->empty[(j - 1) % NSLOT], ((j - 1) / NSLOT) & 1u, abort, err) ? 1 : 0;
        ok2 = __shfl_sync(0xffffffffu, ok2, 0);
        if (!ok2) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DH / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_off + S::O_COL + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + lane_off + S::O_COL + c * 32, o);
        }
      }
      // P_j over S_j in TMEM: this row's segment as hi + lo bf16 pairs, the
      // other replicas' keys (and rows past q_len) zero
      {
        uint32_t ph[KG / 2], pl[KG / 2];
#pragma unroll
        for (int i = 0; i < KG / 2; ++i) {
          const float a = sv[2 * i], bb = sv[2 * i + 1];
          const __nv_bfloat162 hb = __floats2bfloat162_rn(a, bb);
          const float2 hf = __bfloat1622float2(hb);
          ph[i] = valid ? *reinterpret_cast<const uint32_t*>(&hb) : 0u;
          pl[i] = valid ? pack2(a - hf.x, bb - hf.y) : 0u;
        }
        // segment g of the row (g is the same in every lane of the warp);
        // constant indices keep the row in registers
        uint32_t hi[KT / 2], lo[KT / 2];
#pragma unroll
        for (int gg = 0; gg < R; ++gg)
#pragma unroll
          for (int i = 0; i < KG / 2; ++i) {
            hi[gg * (KG / 2) + i] = gg == g ? ph[i] : 0u;
            lo[gg * (KG / 2) + i] = gg == g ? pl[i] : 0u;
          }
        const uint32_t pt = tmem + lane_off + S::S_COL + sb * KT;
        tmem_st32u(pt, hi);
        if constexpr (P_PARTS == 2) tmem_st32u(pt + KT / 2, lo);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      tc_fence_before();
      __syncwarp();
      int okv = 1;
      if (lane == 0) {   // P_j written and V_j landed: P_j V_j may go
        okv = mbar_wait(&bars->v_full[j % NSLOT], (j / NSLOT) & 1u, abort, err) ? 1 : 0;
        if (okv) mbar_arrive(&bars->p_full[sb]);
      }
      okv = __shfl_sync(0xffffffffu, okv, 0);
      if (!okv) break;
    }
  }

  // ---- partials of this CTA into the drained ring:
  //   po[m][PLD] fp32 O row of MMA row m = g * QP + r, pml[m] = (m_ref, l)
  tc_fence_before();
  __syncthreads();
  float* po = reinterpret_cast<float*>(sm + S::OFF_RING);
  float* pml = po + QROWS * S::PLD;
  float* wts = pml + QROWS * 2;                           // [QROWS][8] merge weights
  if (warp >= 2) {
    const int wq = warp & 3;
    const int m = wq * 32 + lane, r = m % QP;
    if (n_tiles > 0) {
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait(&bars->empty[(n_tiles - 1) % NSLOT], ((n_tiles - 1) / NSLOT) & 1u, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      tc_fence_after();
      const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
#pragma unroll 1
      for (int c = 0; c < DH / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_off + S::O_COL + c * 32, o);
        if (r < q_len) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(po + m * S::PLD + c * 32 + i) =
                ok ? make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    if (r < q_len) {
      pml[m * 2] = n_tiles > 0 ? m_ref : -INFINITY;
      pml[m * 2 + 1] = l_sum;
    }
  }
  __syncthreads();
  // a query's replicas: weight each by 2^(m_g - M) and sum O and l into
  // replica 0's row, whose reference becomes M
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
      pml[r * 2] = M;
      pml[r * 2 + 1] = l;
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
  }
  tc_fence_before();
  cluster_barrier();
  // CTA `split` finishes queries [split * qpc, split * qpc + qpc):
  //   1. one thread per query reads every split's (m, l) and keeps the weights
  //   2. every thread gathers float4 column groups of O from all splits
  const int qpc = cdiv(q_len, n_split);
  const int q0 = split * qpc, nq = max(0, min(qpc, q_len - q0));
  for (int t = tid; t < nq; t += 192) {
    const int q = q0 + t;
    float mr[8], lr[8];
    float M = -INFINITY;
    for (int p = 0; p < n_split; ++p) {
      mr[p] = ld_peer_f(pml + q * 2, p);
      lr[p] = ld_peer_f(pml + q * 2 + 1, p);
      M = fmaxf(M, mr[p]);
    }
    float den = 0.f;
    for (int p = 0; p < n_split; ++p) {
      mr[p] = mr[p] == -INFINITY ? 0.f : exp2f(mr[p] - M);
      den += mr[p] * lr[p];
    }
    const float inv = 1.f / den;
    for (int p = 0; p < n_split; ++p) wts[t * 8 + p] = mr[p] * inv;
  }
  __syncthreads();
  for (int e = tid; e < nq * (DH / 4); e += 192) {
    const int t = e / (DH / 4), c = (e % (DH / 4)) * 4, q = q0 + t;
    float4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p)
      if (p < n_split) {
        float x[4];
        ld_peer_v<4>(po + q * S::PLD + c, p, x);
        v[p] = make_float4(x[0], x[1], x[2], x[3]);
      }
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p)
      if (p < n_split) {
        const float w = wts[t * 8 + p];
        a0 = fmaf(w, v[p].x, a0); a1 = fmaf(w, v[p].y, a1); a2 = fmaf(w, v[p].z, a2); a3 = fmaf(w, v[p].w, a3);
      }
    bf16* op = out + static_cast<size_t>(b * q_len + q) * ld + h * DH + c;
    *reinterpret_cast<__nv_bfloat162*>(op) = __floats2bfloat162_rn(a0, a1);
    *reinterpret_cast<__nv_bfloat162*>(op + 2) = __floats2bfloat162_rn(a2, a3);
  }
  cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

}  // namespace attn_tc
}  // namespace dllm
