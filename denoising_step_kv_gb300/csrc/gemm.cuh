// D = A . B^T for K-major A [M][K] (rows) and B [N][K] (weights), finished
// by an epilogue functor that receives one output row of a tile at a time.
//
// bf16, four tcgen05 kernels (TMA loads with 128-byte swizzle into an
// mbarrier ring, one thread issuing the MMAs, fp32 accumulators in TMEM):
//   gemm_tc_kernel      persistent, 128 x 128 tiles, two TMEM accumulators so
//                       the epilogue of one tile overlaps the next tile's MMAs;
//   gemm_pair_kernel    the same with clusters of two CTAs on 128 x 256 tiles
//                       that share (multicast) the weight tile - large M;
//                       both persistent kernels run their tiles in column
//                       bands so that the tiles in flight share L2;
//   gemm_sharea_kernel  clusters of CTAs on adjacent weight tiles of the same
//                       128 rows, which they share (multicast) - the LM head;
//   gemm_skinny_kernel  weights as the MMA's A operand, the few rows as its B
//                       operand, K split over a cluster - weight streaming for
//                       M <= 256 with a split, M <= 512 without.
// fp32: a SIMT kernel whose "loader" computes 32 dot products on demand, used
// only by the fp32 workload (tensor cores have no fp32 path within 1e-5).
#pragma once
#include "common.cuh"

namespace dllm {

// Epilogue interface:
//   template <class LD> __device__ void run(int m, int n0, int nch, int M, int N, const LD& ld) const;
// m: output row (may be >= M: then store nothing), n0: first column of the
// tile, nch: the tile's width in 32-column chunks; ld(col, v) fills v[0..31]
// with accumulator columns n0+col .. n0+col+31.
// On the tensor-core path ld is warp-collective: every lane calls it the same
// number of times whatever its row.

namespace tc {
constexpr int BM = 128, BN = 128, BK = 64, MAX_STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;

struct Bars {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem;
  int abort;
};
// Persistent kernel: 4 stages (one CTA per SM) for compute-bound shapes, 3
// stages (two CTAs per SM, twice the weight bytes in flight) for streaming.
template <int STAGES>
constexpr size_t smem_bytes() { return 1024 + STAGES * STAGE_BYTES + sizeof(Bars); }

// Column-banded tile order of the persistent kernels: bands of gw column
// tiles (about 32 MB of weights), the column tile fastest inside a band, so
// that the tiles in flight at once share a few row tiles and one band of
// weights in L2 (rows fastest would stream every row tile from HBM once per
// column tile when the rows do not fit in L2).
__host__ __device__ __forceinline__ int band_width(int tile_cols, int K) {
  const long long w = (32ll << 20) / (static_cast<long long>(tile_cols) * K * 2);
  return static_cast<int>(w < 1 ? 1 : w);
}
__device__ __forceinline__ void band_tile(int tile, int nM, int nN, int gw, int& m, int& n) {
  const int per = nM * gw;                      // tiles of a full band
  const int band = tile / per;
  const int bw = min(gw, nN - band * gw);       // this band's width
  const int rem = tile - band * per;
  m = rem / bw;
  n = band * gw + rem % bw;
}

struct TmemLoader {
  uint32_t taddr;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const { tmem_ld32(taddr + col, v); }
};

template <class Epi, int STAGES>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   int M_host, const int* __restrict__ M_dev, int M_cap, int M_min, int N, int K, Epi epi,
                   unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 4);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem, TMEM_COLS);
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  pdl_launch();
  pdl_wait();
  const int M = M_dev ? min(*M_dev, M_cap) : M_host;   // never past A's rows
  const int nM = (M + BM - 1) / BM, nN = (N + BN - 1) / BN, nK = (K + BK - 1) / BK;
  // M below M_min belongs to the kernel launched beside this one
  const int tiles = (M > 0 && M >= M_min) ? nM * nN : 0;
  const int gw = band_width(BN, K);

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, par = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort; tile += gridDim.x) {
        int mb, nb;
        band_tile(tile, nM, nN, gw, mb, nb);
        for (int kb = 0; kb < nK; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, err)) break;
          mbar_expect_tx(&bars->full[stage], STAGE_BYTES);
          tma_load_2d(sa + stage * A_BYTES, &tmA, kb * BK, mb * BM, &bars->full[stage]);
          tma_load_2d(sb + stage * B_BYTES, &tmB, kb * BK, nb * BN, &bars->full[stage]);
          issued |= 1u << stage;
          par = (par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort) {   // let every copy already issued land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&bars->full[s], (par >> s) & 1u, nullptr, err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort; tile += gridDim.x) {
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nK; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sa + stage * A_BYTES), b0 = smem_u32(sb + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_bf16(d_tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          tc_commit(&bars->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bars->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      tc_commit(&bars->done);
      mbar_wait(&bars->done, 0, nullptr, err);
    }
  } else {
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bars->tfull[acc], acc_phase, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int mb, nb;
      band_tile(tile, nM, nN, gw, mb, nb);
      const int m = mb * BM + q * 32 + lane;
      TmemLoader ld{tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN)};
      epi.run(m, nb * BN, BN / 32, M, N, ld);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Pair kernel for large M: persistent clusters of two CTAs; cluster tile p
// covers rows [256 mp, 256 mp + 256) x columns [256 nb, 256 nb + 256), CTA
// rank r the 128-row half 2 mp + r.  Each CTA loads its own 128 x 64 A tile
// and one 128-row half of the 256 x 64 B tile, multicast into both CTAs, so a
// CTA fetches 32 KB per k-block for 512 tensor cycles (M=128, N=256, K=64)
// instead of 32 KB per 256 cycles with 128 x 128 tiles.  A stage is reloaded
// only once both CTAs' MMAs have read it: every MMA commit arrives on the
// empty barrier of both CTAs (count 2).  Accumulators: 2 x 256 TMEM columns.
constexpr int PBN = 256;
constexpr int PB_BYTES = PBN * BK * 2;             // two 16 KB halves
constexpr int PSTAGE_BYTES = A_BYTES + PB_BYTES;   // 48 KB
constexpr uint32_t PTMEM_COLS = 2 * PBN;
template <int STAGES>
constexpr size_t pair_smem_bytes() { return 1024 + STAGES * PSTAGE_BYTES + sizeof(Bars); }

template <class Epi, int STAGES>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     int M_host, const int* __restrict__ M_dev, int M_cap, int M_min, int N, int K, Epi epi,
                     unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * PSTAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cl = blockIdx.x >> 1, n_cl = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 2);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 4);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem, PTMEM_COLS);
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();       // the peer's barriers exist before any multicast lands
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  pdl_launch();
  pdl_wait();
  const int M = M_dev ? min(*M_dev, M_cap) : M_host;
  const int nM = (M + BM - 1) / BM, nMP = (nM + 1) / 2, nN = (N + PBN - 1) / PBN, nK = (K + BK - 1) / BK;
  // the same in both CTAs of a cluster: both run the same tiles and k-blocks
  const int tiles = (M > 0 && M >= M_min) ? nMP * nN : 0;
  const int gw = band_width(PBN, K);

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, par = 0;
      for (int tile = cl; tile < tiles && !*abort; tile += n_cl) {
        int mp, nb;
        band_tile(tile, nMP, nN, gw, mp, nb);
        // a half past the last row tile loads the last valid one again (its
        // rows are >= M, the epilogue stores nothing for them)
        const int mb_ld = min(2 * mp + rank, nM - 1);
        for (int kb = 0; kb < nK; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, err)) break;
          mbar_expect_tx(&bars->full[stage], PSTAGE_BYTES);
          tma_load_2d(sa + stage * A_BYTES, &tmA, kb * BK, mb_ld * BM, &bars->full[stage]);
          tma_load_2d_mc(sb + stage * PB_BYTES + rank * B_BYTES, &tmB, kb * BK, nb * PBN + rank * BN,
                         &bars->full[stage], 0x3);
          issued |= 1u << stage;
          par = (par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort) {
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&bars->full[s], (par >> s) & 1u, nullptr, err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, PBN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = cl; tile < tiles && !*abort; tile += n_cl) {
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * PBN);
        bool ok = true;
        for (int kb = 0; kb < nK; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sa + stage * A_BYTES), b0 = smem_u32(sb + stage * PB_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_bf16(d_tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          tc_commit_mc(&bars->empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bars->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs (and the empty-barrier arrivals they owe the peer) complete
      // before the cluster barrier below
      tc_commit(&bars->done);
      mbar_wait(&bars->done, 0, nullptr, err);
    }
  } else {
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cl; tile < tiles; tile += n_cl) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bars->tfull[acc], acc_phase, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int mp, nb;
      band_tile(tile, nMP, nN, gw, mp, nb);
      const int m = (2 * mp + rank) * BM + q * 32 + lane;
      TmemLoader ld{tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * PBN)};
      epi.run(m, nb * PBN, PBN / 32, M, N, ld);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();       // no multicast copy or commit still targets this CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, PTMEM_COLS);
  }
}

// Shared-A kernel for few rows and many output columns (the LM head):
// persistent clusters of CS CTAs on CS adjacent 128 x SBN tiles of the same
// 128 rows.  Each CTA loads its own weight tile and a 128/CS-row piece of the
// rows' tile, multicast into every CTA of the cluster, so the rows are read
// once per cluster instead of once per CTA.  A stage is reloaded once all CS
// CTAs' MMAs have read it (every commit arrives on all CS empty barriers).
// The row count is a host value: before the grid dependency each CTA warms
// L2 with the first PREF k-blocks of its first weight tile, which no earlier
// kernel writes.  With SBN = 256, one CTA per SM keeps four stages of 32 KB
// of weights in flight.
template <int STAGES, int SBN>
constexpr size_t sharea_smem_bytes() { return 1024 + STAGES * (A_BYTES + SBN * BK * 2) + sizeof(Bars); }

template <class Epi, int STAGES, int CS, int SBN>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_sharea_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M,
                       const int* __restrict__ M_dev, int N, int K, Epi epi, unsigned* err) {
  static_assert(CS == 2 || CS == 4, "the rows' tile splits into CS whole 8-row swizzle groups");
  static_assert(SBN == 128 || SBN == 256, "one MMA per 16-deep slice (N <= 256)");
  constexpr int SB_BYTES = SBN * BK * 2, S_BYTES = A_BYTES + SB_BYTES, PREF = 8;
  constexpr uint32_t S_TMEM = 2 * SBN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * S_BYTES);
  constexpr uint16_t ALL = (1u << CS) - 1;
  constexpr int PIECE = BM / CS;                  // rows of the shared tile each CTA loads

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const int cl = blockIdx.x / CS, n_cl = gridDim.x / CS;
  const int nM = (M + BM - 1) / BM, nN = (N + SBN - 1) / SBN, nK = (K + BK - 1) / BK;
  const int nG = (nN + CS - 1) / CS;
  int tiles = M > 0 ? nM * nG : 0;                // cluster tiles (row tile, group of CS column tiles)

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], CS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 4);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem, S_TMEM);
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (cl < tiles) {
      const int nb = (cl / nM) * CS + rank;
      if (nb < nN)
        for (int kb = 0; kb < min(nK, PREF); ++kb) tma_prefetch_l2_2d(&tmB, kb * BK, nb * SBN);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();       // every CTA's barriers exist before any multicast lands
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  pdl_launch();
  pdl_wait();
  if (M_dev && *M_dev <= 0) tiles = 0;            // a device count of 0 (the same in every CTA): no work

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, par = 0;
      for (int tile = cl; tile < tiles && !*abort; tile += n_cl) {
        const int mb = tile % nM, nb = (tile / nM) * CS + rank;
        for (int kb = 0; kb < nK; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, err)) break;
          mbar_expect_tx(&bars->full[stage], S_BYTES);
          tma_load_2d_mc(sa + stage * A_BYTES + rank * (PIECE * 128), &tmA, kb * BK, mb * BM + rank * PIECE,
                         &bars->full[stage], ALL);
          tma_load_2d(sb + stage * SB_BYTES, &tmB, kb * BK, nb * SBN, &bars->full[stage]);
          issued |= 1u << stage;
          par = (par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort) {
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&bars->full[s], (par >> s) & 1u, nullptr, err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, SBN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = cl; tile < tiles && !*abort; tile += n_cl) {
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort, err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * SBN);
        bool ok = true;
        for (int kb = 0; kb < nK; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sa + stage * A_BYTES), b0 = smem_u32(sb + stage * SB_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_bf16(d_tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          tc_commit_mc(&bars->empty[stage], ALL);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bars->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA and the empty-barrier arrivals it owes the peers complete
      // before the cluster barrier below
      tc_commit(&bars->done);
      mbar_wait(&bars->done, 0, nullptr, err);
    }
  } else {
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cl; tile < tiles; tile += n_cl) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bars->tfull[acc], acc_phase, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int mb = tile % nM, nb = (tile / nM) * CS + rank;
      if (nb < nN) {   // the last group may run past the columns
        const int m = mb * BM + q * 32 + lane;
        TmemLoader ld{tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * SBN)};
        epi.run(m, nb * SBN, SBN / 32, M, N, ld);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();       // no multicast copy or commit still targets this CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S_TMEM);
  }
}

// Weight-streaming GEMM for few rows: D^T = B . A^T.  The weights B [N][K]
// are the MMA's A operand (128 output columns per CTA, on the TMEM lanes) and
// the rows A [M][K] its B operand (on the TMEM columns: one MMA of N = M
// rounded up to 16, or two past 256 rows), so every weight byte is read from
// HBM once and no MMA work goes to padding rows.
//
// Before the grid dependency (the weights are no earlier kernel's output)
// each CTA loads its first SKN_EARLY weight k-blocks into the stage ring and
// asks L2 for the next ones; the rows and the device row count wait for the
// dependency.  A stage holds a weight tile at a fixed offset and the rows'
// tile (32-row boxes, only as many as M needs) after all weight tiles.
//
// A cluster of SPLITK CTAs splits K.  Rank r owns rows [r * tpr, (r + 1) *
// tpr) (tpr a multiple of 32).  Once every rank's MMAs are done (cluster
// barrier) each rank writes its fp32 partial of every other owner's rows
// from TMEM into a local send block and hands the block to the owner with
// one bulk shared::cluster copy that completes on the owner's receive
// barrier; the owner adds the partials in rank order (its own from TMEM)
// into its first receive block and runs the epilogue over (row, piece)
// items.  Without a split the accumulator is staged through shared memory
// in one pass (up to 384 rows, else two).  Blocks are [128 columns][tpr rows] fp32 with each
// column's 16-byte chunks rotated by the column index, so that a warp's
// column-wise writes and its row-wise reads both spread over all banks.
constexpr int SKN_MAX_ROWS = 512;                // without a split of K
constexpr int SKN_SPLIT_ROWS = 256;              // with one
constexpr int SKN_W_BYTES = 128 * BK * 2;        // 16 KB of weights per k-block
constexpr int SKN_XBOX = 32;                     // rows per load of A
constexpr int SKN_RING = 192 * 1024;
constexpr int SKN_MAX_ST = 8;
constexpr int SKN_EARLY = 2;                     // weight k-blocks loaded before the grid dependency
constexpr int SKN_PF = 16;                       // weight k-blocks warmed in L2 before it
constexpr int SKN_CHUNK = 384;                   // most rows staged in one pass without a split
constexpr uint32_t SKN_TMEM_COLS = 512;
struct SknBars {
  uint64_t full[SKN_MAX_ST];
  uint64_t empty[SKN_MAX_ST];
  uint64_t tfull;
  uint64_t recv;
  uint32_t tmem;
  int abort;
};
constexpr size_t SKN_SMEM = 1024 + SKN_RING + sizeof(SknBars);

__host__ __device__ constexpr int skn_max_rows(int S) { return S == 1 ? SKN_MAX_ROWS : SKN_SPLIT_ROWS; }
__host__ __device__ constexpr int skn_tpr(int M, int S) { return ((M + S - 1) / S + 31) & ~31; }
// send and receive blocks of every other rank
static_assert(2 * 3 * 128 * skn_tpr(SKN_SPLIT_ROWS, 4) * 4 <= SKN_RING, "exchange blocks fit in the ring");
static_assert(2 * 2 * 128 * skn_tpr(SKN_SPLIT_ROWS, 3) * 4 <= SKN_RING, "exchange blocks fit in the ring");
static_assert(2 * 1 * 128 * skn_tpr(SKN_SPLIT_ROWS, 2) * 4 <= SKN_RING, "exchange blocks fit in the ring");
static_assert(128 * SKN_CHUNK * 4 <= SKN_RING && 128 * 256 * 4 <= SKN_RING, "a staged pass fits in the ring");
static_assert(SKN_RING / (SKN_W_BYTES + SKN_MAX_ROWS * 128) >= SKN_EARLY, "the early loads' stages exist for any M");

// Element (column f, row rr) of a [128][tpr] block: column f's 16-byte
// chunks rotated by f mod 8 (tpr / 4 is a multiple of 8).
__device__ __forceinline__ int skn_at(int f, int rr, int tpr) {
  int c = (rr >> 2) + (f & 7);
  if (c >= (tpr >> 2)) c -= tpr >> 2;
  return f * tpr + (c << 2) + (rr & 3);
}

// Columns [col, col + 32) of row rr of a staged block (col a multiple of 32).
struct SknLoader {
  const float* blk;
  int tpr, rr;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = blk[skn_at(col + j, rr, tpr)];
  }
};

// This thread's 32 accumulator values of column f (rows r0 .. r0 + 31, as
// read from its TMEM lane) into a staged block.
__device__ __forceinline__ void skn_put32(float* blk, int f, int r0, int tpr, const float (&v)[32]) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<float4*>(blk + skn_at(f, r0 + 4 * u, tpr)) =
        make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}

// Local shared memory -> a cluster peer's shared memory, completing on the
// peer's barrier (both addresses in the peer, mapped with mapa).
__device__ __forceinline__ void bulk_s2c(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                         uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ uint32_t mapa_u32(const void* p, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  return ra;
}

template <class Epi, int SPLITK>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       int M_host, const int* __restrict__ M_dev, int M_cap, int N, int K, Epi epi,
                       unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  SknBars* bars = reinterpret_cast<SknBars*>(smem + SKN_RING);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = SPLITK > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int nb = blockIdx.x / SPLITK;
  const int nK = (K + BK - 1) / BK, kpc = (nK + SPLITK - 1) / SPLITK;
  const int kb0 = rank * kpc, n_kb = max(0, min(nK, kb0 + kpc) - kb0);
  const int n_early = min(n_kb, SKN_EARLY);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SKN_MAX_ST; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->tfull, 1);
    mbar_init(&bars->recv, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&bars->tmem, SKN_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  // before the grid dependency: the weights only
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
    for (int i = 0; i < n_early; ++i) {
      mbar_expect_tx_only(&bars->full[i], SKN_W_BYTES);
      tma_load_2d(smem + i * SKN_W_BYTES, &tmW, (kb0 + i) * BK, nb * 128, &bars->full[i]);
    }
    for (int i = n_early; i < min(n_kb, SKN_PF); ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * BK, nb * 128);
  }
  pdl_launch();
  pdl_wait();
  const int M = M_dev ? min(*M_dev, M_cap) : M_host;
  // the same decision in every CTA of the cluster
  if (M <= 0 || M > skn_max_rows(SPLITK)) {
    if (threadIdx.x == 0)      // the early loads land before the CTA ends
      for (int i = 0; i < n_early; ++i) {
        mbar_arrive(&bars->full[i]);
        mbar_wait(&bars->full[i], 0, nullptr, err);
      }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, SKN_TMEM_COLS);
    }
    return;
  }
  const int xrows = (M + SKN_XBOX - 1) / SKN_XBOX * SKN_XBOX;   // rows loaded per k-block
  const int x_bytes = xrows * 128;
  const int n_st = min(SKN_MAX_ST, SKN_RING / (SKN_W_BYTES + x_bytes));
  uint8_t* xring = smem + n_st * SKN_W_BYTES;
  const int n1 = (min(M, 256) + 15) / 16 * 16;                   // the MMAs' N
  const int n2 = M > 256 ? (M - 256 + 15) / 16 * 16 : 0;
  // rows per owner with a split; without one, rows staged per pass (all of
  // them up to SKN_CHUNK, else halves of at most 256)
  const int tpr = SPLITK > 1 ? skn_tpr(M, SPLITK) : (xrows <= SKN_CHUNK ? xrows : 256);
  const int r0 = rank * tpr, r1 = SPLITK > 1 ? min(M, r0 + tpr) : M;   // rows this CTA finishes

  int ok = 1;
  if (warp == 0) {
    if (lane == 0) {
      uint32_t issued = 0, par = 0;
      for (int i = 0; i < n_kb; ++i) {
        const int kb = kb0 + i, stage = i % n_st;
        const uint32_t phase = (i / n_st) & 1u;
        if (i >= n_early) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, err)) break;
          mbar_expect_tx(&bars->full[stage], SKN_W_BYTES + x_bytes);
          tma_load_2d(smem + stage * SKN_W_BYTES, &tmW, kb * BK, nb * 128, &bars->full[stage]);
        } else {
          mbar_expect_tx(&bars->full[stage], x_bytes);   // its weight bytes are already expected
        }
        for (int j = 0; j < xrows / SKN_XBOX; ++j)
          tma_load_2d(xring + stage * x_bytes + j * (SKN_XBOX * 128), &tmX, kb * BK, j * SKN_XBOX,
                      &bars->full[stage]);
        issued |= 1u << stage;
        par = (par & ~(1u << stage)) | (phase << stage);
      }
      if (*abort) {
        for (int s = 0; s < n_st; ++s)
          if (issued & (1u << s)) mbar_wait(&bars->full[s], (par >> s) & 1u, nullptr, err);
        // early loads the loop never reached
        for (int i = 0; i < n_early; ++i)
          if (!(issued & (1u << i))) {
            mbar_arrive(&bars->full[i]);
            mbar_wait(&bars->full[i], 0, nullptr, err);
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16(128, n1), id2 = idesc_bf16(128, n2 > 0 ? n2 : 16);
      for (int i = 0; i < n_kb; ++i) {
        const int stage = i % n_st;
        const uint32_t phase = (i / n_st) & 1u;
        if (!mbar_wait(&bars->full[stage], phase, abort, err)) break;
        tc_fence_after();
        const uint32_t w0 = smem_u32(smem + stage * SKN_W_BYTES), x0 = smem_u32(xring + stage * x_bytes);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          tc_mma_bf16(tmem, sdesc_sw128(w0 + k * 32), sdesc_sw128(x0 + k * 32), id1, (i | k) != 0 ? 1u : 0u);
          if (n2 > 0)
            tc_mma_bf16(tmem + 256, sdesc_sw128(w0 + k * 32), sdesc_sw128(x0 + 256 * 128 + k * 32), id2,
                        (i | k) != 0 ? 1u : 0u);
        }
        tc_commit(&bars->empty[stage]);
      }
      tc_commit(&bars->tfull);   // completes once every MMA above is done
    }
  } else {
    // while the MMAs run: warm L2 with the epilogue's side data of our rows
    for (int r = r0 + static_cast<int>(threadIdx.x) - 64; r < r1; r += THREADS - 64) epi.prefetch(r, nb * 128, M, N);
    if (lane == 0) ok = mbar_wait(&bars->tfull, 0, abort, err) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
  }
  const int q = warp & 3, f = q * 32 + lane;                 // epilogue warps: this thread's output column
  const uint32_t lane_tm = tmem + (static_cast<uint32_t>(q * 32) << 16);
  const bool live = ok && n_kb > 0 && !*abort;               // a rank with no k-blocks adds zeros
  float* blk0 = reinterpret_cast<float*>(smem);
  tc_fence_before();
  if constexpr (SPLITK > 1) {
    const int bsz = 128 * tpr;                               // floats per block
    float* send = blk0;                                      // [SPLITK - 1][128][tpr]
    float* recv = blk0 + (SPLITK - 1) * bsz;                 // [SPLITK - 1][128][tpr], by sender
    cluster_barrier();   // every rank's MMAs are done: the rings are free for the exchange
    if (warp >= 2) {
      tc_fence_after();
#pragma unroll 1
      for (int o = 0, oi = 0; o < SPLITK; ++o) {
        if (o == rank) continue;
        float* dst = send + (oi++) * bsz;
#pragma unroll 1
        for (int c = 0; c < tpr / 32; ++c) {
          float v[32];
          tmem_ld32(lane_tm + o * tpr + c * 32, v);
          if (!live)
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          skn_put32(dst, f, c * 32, tpr, v);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // writes visible to the bulk copies
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (threadIdx.x == 64) {
        mbar_expect_tx(&bars->recv, static_cast<uint32_t>((SPLITK - 1) * bsz * 4));
#pragma unroll 1
        for (int o = 0, oi = 0; o < SPLITK; ++o) {
          if (o == rank) continue;
          const int slot = rank < o ? rank : rank - 1;        // senders skip the owner
          bulk_s2c(mapa_u32(recv + slot * bsz, o), send + (oi++) * bsz, static_cast<uint32_t>(bsz * 4),
                   mapa_u32(&bars->recv, o));
        }
      }
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&bars->recv, 0, abort, err) ? 1 : 0;
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      // the rank-order sum of this CTA's rows into the first receive block
#pragma unroll 1
      for (int c = 0; c < (r1 - r0 + 31) / 32 && w_ok; ++c) {
        float acc[32], v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
#pragma unroll 1
        for (int s = 0; s < SPLITK; ++s) {
          if (s == rank) {
            tmem_ld32(lane_tm + r0 + c * 32, v);
            if (!live)
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
          } else {
            const float* src = recv + (s < rank ? s : s - 1) * bsz;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 x = *reinterpret_cast<const float4*>(src + skn_at(f, c * 32 + 4 * u, tpr));
              v[4 * u] = x.x;
              v[4 * u + 1] = x.y;
              v[4 * u + 2] = x.z;
              v[4 * u + 3] = x.w;
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] += v[j];
        }
        skn_put32(recv, f, c * 32, tpr, acc);
      }
    }
    __syncthreads();
    const int nrows = r1 - r0;
    if (!*abort)
      for (int it = threadIdx.x; it < nrows * Epi::PARTS; it += THREADS) {
        const int rr = it % nrows, piece = it / nrows;
        epi.run_part(r0 + rr, nb * 128, piece, M, N, SknLoader{recv, tpr, rr});
      }
    tc_fence_before();
    cluster_barrier();   // every copy into this CTA has landed and every copy out of it was read
  } else {
    __syncthreads();     // the MMAs are done: the ring is free for staging
#pragma unroll 1
    for (int c0 = 0; c0 < M; c0 += tpr) {
      const int nrows = min(tpr, M - c0);
      if (warp >= 2) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < (nrows + 31) / 32; ++c) {
          float v[32];
          tmem_ld32(lane_tm + c0 + c * 32, v);
          skn_put32(blk0, f, c * 32, tpr, v);
        }
      }
      __syncthreads();
      if (live)
        for (int it = threadIdx.x; it < nrows * Epi::PARTS; it += THREADS) {
          const int rr = it % nrows, piece = it / nrows;
          epi.run_part(c0 + rr, nb * 128, piece, M, N, SknLoader{blk0, tpr, rr});
        }
      __syncthreads();
    }
    tc_fence_before();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SKN_TMEM_COLS);
  }
}

}  // namespace tc

namespace simt {
template <typename T>
struct DotLoader {
  const T* A;
  const T* B;
  int m, n0, M, N, K;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const {
#pragma unroll 1
    for (int j = 0; j < 32; ++j) {
      const int n = n0 + col + j;
      float s = 0.f;
      if (m < M && n < N) {
        const T* a = A + static_cast<size_t>(m) * K;
        const T* b = B + static_cast<size_t>(n) * K;
        for (int k = 0; k < K; ++k) s = fmaf(to_f(a[k]), to_f(b[k]), s);
      }
      v[j] = s;
    }
  }
};

// One thread per output row, blockIdx.y selects a tile of 32*NCH columns.
template <typename T, int NCH, class Epi>
__global__ void __launch_bounds__(128) gemm_simt_kernel(const T* __restrict__ A, const T* __restrict__ B,
                                                        int M_host, const int* __restrict__ M_dev, int M_cap,
                                                        int N, int K, Epi epi) {
  const int M = M_dev ? min(*M_dev, M_cap) : M_host;
  if (static_cast<int>(blockIdx.x * blockDim.x) >= M) return;
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  const int n0 = blockIdx.y * 32 * NCH;
  DotLoader<T> ld{A, B, m, n0, M, N, K};
  epi.run(m, n0, NCH, M, N, ld);
}
}  // namespace simt

}  // namespace dllm
