// D = A . B^T for K-major A [M][K] and B [N][K], finished by an epilogue
// functor that receives one accumulator row at a time.
//
// bf16: persistent tcgen05 kernel.  Warp 0 issues TMA loads of 128x64 A and B
// tiles (128-byte swizzle) into a STAGES-deep ring; one thread of warp 1
// issues tcgen05.mma (M=128, N=128, K=16) into one of two TMEM accumulators
// (2 x 128 columns) and commits to mbarriers; warps 2-5 read the finished
// accumulator with tcgen05.ld (warp w owns TMEM lanes 32*(w%4) ...) and run
// the epilogue while the next tile accumulates into the other buffer.
// fp32: a SIMT kernel whose "loader" computes 32 dot products on demand, used
// only by the fp32 workload (tensor cores have no fp32 path within 1e-5).
#pragma once
#include "common.cuh"

namespace dllm {

// Epilogue interface:
//   template <class LD> __device__ void run(int m, int n0, int M, int N, const LD& ld) const;
// m: output row (may be >= M: then store nothing), n0: first column of the
// tile; ld(col, v) fills v[0..31] with accumulator columns n0+col .. n0+col+31.
// On the tensor-core path ld is warp-collective: every lane calls it the same
// number of times whatever its row.

namespace tc {
constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;

struct Bars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem;
  int abort;
};
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + sizeof(Bars);

struct TmemLoader {
  uint32_t taddr;
  __device__ __forceinline__ void operator()(int col, float (&v)[32]) const { tmem_ld32(taddr + col, v); }
};

template <class Epi>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   int M_host, const int* __restrict__ M_dev, int M_cap, int N, int K, Epi epi, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = M_dev ? min(*M_dev, M_cap) : M_host;   // never past A's rows
  const int nM = (M + BM - 1) / BM, nN = (N + BN - 1) / BN, nK = (K + BK - 1) / BK;
  const int tiles = M > 0 ? nM * nN : 0;

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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
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
      epi.run(m, nb * BN, M, N, ld);
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
  epi.run(m, n0, M, N, ld);
}
}  // namespace simt

}  // namespace dllm
