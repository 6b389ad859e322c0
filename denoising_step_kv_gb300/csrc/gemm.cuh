// D = A . B^T for K-major A [M][K] (rows) and B [N][K] (weights), finished
// by an epilogue functor that receives one output row of a tile at a time.
//
// bf16, four tcgen05 kernels (TMA loads with 128-byte swizzle into an
// mbarrier ring, one thread issuing the MMAs, fp32 accumulators in TMEM):
//   gemm_tc_kernel      persistent, 128 x 128 tiles, two TMEM accumulators so
//                       the epilogue of one tile overlaps the next tile's MMAs;
//   gemm_pair_kernel    the same with clusters of two CTAs on 128 x 256 tiles
//                       that share (multicast) the weight tile - large M;
//   gemm_sharea_kernel  clusters of CTAs on adjacent weight tiles of the same
//                       128 rows, which they share (multicast) - the LM head;
//   gemm_skinny_kernel  weights as the MMA's A operand, the few rows as its B
//                       operand, K split over a cluster - M <= 256, weight
//                       streaming.
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

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, par = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort; tile += gridDim.x) {
        const int mb = tile % nM, nb = tile / nM;
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
      const int mb = tile % nM, nb = tile / nM;
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

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, par = 0;
      for (int tile = cl; tile < tiles && !*abort; tile += n_cl) {
        const int mp = tile % nMP, nb = tile / nMP;
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
      const int mp = tile % nMP, nb = tile / nMP;
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

// Weight-streaming GEMM for small M (at most 256 rows): D^T = B . A^T.  The
// weights B [N][K] are the MMA's A operand (128 output columns per CTA, on
// the TMEM lanes) and the rows A [M][K] its B operand (M rounded up to 16, on
// the TMEM columns), so every weight byte is read from HBM once and no MMA
// work goes to padding rows.  A cluster of SPLITK CTAs splits K.  Rank r owns
// rows [r * tpr, (r + 1) * tpr) of the tile: after every rank's MMAs are done
// (cluster barrier), each rank pushes its fp32 partial of those rows into the
// owner's shared memory (16-byte remote stores, no round trips), and after
// a second barrier the owner sums the SPLITK partials (rank order) while
// running the epilogue, spread over (row, piece) items.  The epilogue warps
// warm L2 with the epilogue's side data while the MMAs run.  The stage ring holds as many
// stages as fit for this M (rows are loaded in 64-row boxes, only as needed).
constexpr int SKN_MAX_ROWS = 256;
constexpr int SKN_W_BYTES = 128 * BK * 2;        // 16 KB of weights per k-block
constexpr int SKN_XBOX = 64;                     // rows per load of A
constexpr int SKN_RING = 192 * 1024;
constexpr int SKN_MAX_ST = 8;
struct SknBars {
  uint64_t full[SKN_MAX_ST];
  uint64_t empty[SKN_MAX_ST];
  uint64_t tfull;
  uint32_t tmem;
  int abort;
};
constexpr size_t SKN_SMEM = 1024 + SKN_RING + sizeof(SknBars);

// Rows per rank (a multiple of 4) and the row stride of the receive buffer
// recv[rank][column][ldr], padded so that ldr / 4 is odd: a warp's 16-byte
// pushes (a lane per column, four rows each) spread over all banks.
__host__ __device__ constexpr int skn_tpr(int M, int S) { return ((M + S - 1) / S + 3) & ~3; }
__host__ __device__ constexpr int skn_ldr(int tpr) { return (tpr / 4) % 2 ? tpr : tpr + 4; }
static_assert(4 * 128 * skn_ldr(skn_tpr(SKN_MAX_ROWS, 4)) * 4 <= SKN_RING, "receive buffer fits in the ring");
static_assert(3 * 128 * skn_ldr(skn_tpr(SKN_MAX_ROWS, 3)) * 4 <= SKN_RING, "receive buffer fits in the ring");
static_assert(2 * 128 * skn_ldr(skn_tpr(SKN_MAX_ROWS, 2)) * 4 <= SKN_RING, "receive buffer fits in the ring");

// Columns [col, col + 32) of local row rr of the owner's tile: the sum, in
// rank order, of the SPLITK partials pushed into recv.
template <int SPLITK>
struct RecvSumLoader {
  const float* recv;
  int ldr, rr;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = recv[(col + j) * ldr + rr];
#pragma unroll
    for (int p = 1; p < SPLITK; ++p)
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += recv[((p * 128) + col + j) * ldr + rr];
  }
};

template <class Epi, int SPLITK>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       int M_host, const int* __restrict__ M_dev, int M_cap, int N, int K, Epi epi,
                       unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  SknBars* bars = reinterpret_cast<SknBars*>(smem + SKN_RING);
  float* recv = reinterpret_cast<float*>(smem);    // [SPLITK][128][ldr], after the mainloop

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch();
  pdl_wait();
  const int M = M_dev ? min(*M_dev, M_cap) : M_host;
  // the same decision in every CTA of the cluster
  if (M <= 0 || M > SKN_MAX_ROWS) return;
  const int rank = static_cast<int>(cluster_rank());
  const int nb = blockIdx.x / SPLITK;
  const int nK = (K + BK - 1) / BK, kpc = (nK + SPLITK - 1) / SPLITK;
  const int kb0 = rank * kpc, kb1 = min(nK, kb0 + kpc);
  const bool has_k = kb1 > kb0;
  const int xrows = (M + SKN_XBOX - 1) / SKN_XBOX * SKN_XBOX;   // rows loaded per k-block
  const int nx = xrows / SKN_XBOX;
  const int n_mma = (M + 15) / 16 * 16;
  const int stage_bytes = SKN_W_BYTES + xrows * 128;
  const int n_st = min(SKN_MAX_ST, SKN_RING / stage_bytes);
  const int tpr = skn_tpr(M, SPLITK), ldr = skn_ldr(tpr);
  const int r0 = rank * tpr, r1 = min(M, r0 + tpr);

  if (threadIdx.x == 0) {
    for (int s = 0; s < n_st; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->tfull, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &bars->abort;
  // the producer starts at once; warps 1-5 meet after the TMEM allocation
  uint32_t tmem = 0;
  if (warp >= 1) {
    if (warp == 1) tmem_alloc(&bars->tmem, 256);
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS - 32) : "memory");
    tc_fence_after();
    tmem = bars->tmem;
  }

  int ok = 1;
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmX);
      uint32_t issued = 0, par = 0;
      for (int kb = kb0, i = 0; kb < kb1; ++kb, ++i) {
        const int stage = i % n_st;
        const uint32_t phase = (i / n_st) & 1u;
        if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort, err)) break;
        uint8_t* st = smem + stage * stage_bytes;
        mbar_expect_tx(&bars->full[stage], stage_bytes);
        tma_load_2d(st, &tmW, kb * BK, nb * 128, &bars->full[stage]);
        for (int j = 0; j < nx; ++j)
          tma_load_2d(st + SKN_W_BYTES + j * SKN_XBOX * 128, &tmX, kb * BK, j * SKN_XBOX, &bars->full[stage]);
        issued |= 1u << stage;
        par = (par & ~(1u << stage)) | (phase << stage);
      }
      if (*abort)
        for (int s = 0; s < n_st; ++s)
          if (issued & (1u << s)) mbar_wait(&bars->full[s], (par >> s) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, n_mma);
      for (int kb = kb0, i = 0; kb < kb1; ++kb, ++i) {
        const int stage = i % n_st;
        const uint32_t phase = (i / n_st) & 1u;
        if (!mbar_wait(&bars->full[stage], phase, abort, err)) break;
        tc_fence_after();
        const uint32_t w0 = smem_u32(smem + stage * stage_bytes), x0 = w0 + SKN_W_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc_mma_bf16(tmem, sdesc_sw128(w0 + k * 32), sdesc_sw128(x0 + k * 32), idesc, (i | k) != 0 ? 1u : 0u);
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
  // every rank's MMAs are done: the stage rings are free to receive partials
  tc_fence_before();
  cluster_barrier();
  if (warp >= 2) {
    tc_fence_after();
    const int q = warp & 3, f = q * 32 + lane;   // this thread's output column
    const bool live = ok && has_k;
    float v[32];
#pragma unroll 1
    for (int c = 0; c < xrows / 32; ++c) {
      tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 32, v);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const int r = c * 32 + j;   // four rows, never split between owners
        if (r >= M) break;
        const int owner = r / tpr, rr = r - owner * tpr;
        const uint32_t la = smem_u32(recv + (rank * 128 + f) * ldr + rr);
        uint32_t ra;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(owner));
        const float4 x = live ? make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(x.x), "f"(x.y),
                     "f"(x.z), "f"(x.w)
                     : "memory");
      }
    }
  }
  tc_fence_before();
  cluster_barrier();       // every partial has landed; no remote access follows
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
  // (row, piece) items, rows fastest so a warp reads consecutive rows
  const int nrows = r1 - r0;
  for (int it = threadIdx.x; it < nrows * Epi::PARTS; it += THREADS) {
    const int rr = it % nrows, piece = it / nrows;
    RecvSumLoader<SPLITK> ldr_{recv, ldr, rr};
    epi.run_part(r0 + rr, nb * 128, piece, M, N, ldr_);
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
