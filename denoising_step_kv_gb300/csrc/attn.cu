// Cached bidirectional attention of a few queries per (sequence, head) over
// the whole cached sequence: HBM-bound streaming of K/V.
//
// bf16: grid (n_split, H, B) launched as clusters of n_split CTAs.  In each
// CTA a producer warp streams 64-key K and V tiles of its key range with TMA
// (128-byte swizzle) into a 3-stage mbarrier ring; two groups of NQW consumer
// warps (16 queries per warp) each take one 32-key half of every tile and
// compute S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in, fp32
// accumulate) from ldmatrix fragments, keeping an online softmax in the log2
// domain.  The partials (m, l, O) of both groups of every CTA are merged
// across the cluster through distributed shared memory, so no partial ever
// reaches HBM.
// fp32: one warp per (query, head, sequence), online softmax in fp32.
#include <algorithm>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace dllm {
namespace {


constexpr int KT = 64;        // keys per tile
constexpr int ASTAGES = 3;    // ring depth

template <int DH>
struct AttnShape {
  static constexpr int TILE = KT * DH * 2;   // bytes of one K (or V) tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int RING = ASTAGES * STAGE;
};

constexpr int QLD_PAD = 8;   // bf16 padding of a staged Q row (ldmatrix without bank conflicts)

template <int DH, int NQW>
constexpr size_t attn_smem_bytes() {
  return 1024 + AttnShape<DH>::RING + 2 * ASTAGES * sizeof(uint64_t) + 16 +
         static_cast<size_t>(NQW) * 16 * (DH + QLD_PAD) * 2;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// (a, b) -> bf16 pairs hi = rn(a, b) and lo = rn(a - hi_a, b - hi_b)
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}
// Byte offset of (key, dim) in a tile stored as DH/64 sub-tiles of 64 keys x
// 128 bytes with the 128-byte swizzle (16-byte chunk index ^= key % 8).
__device__ __forceinline__ uint32_t swz(int key, int dim) {
  return static_cast<uint32_t>((dim >> 6) * (KT * 128) + key * 128 + ((((dim & 63) >> 3) ^ (key & 7)) << 4) +
                               ((dim & 7) << 1));
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer(const float* p, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}
// PER consecutive floats (16- or 8-byte aligned) from the same offset in the
// shared memory of cluster CTA `rank`.
template <int PER>
__device__ __forceinline__ void ld_peer_vec(const float* p, int rank, float (&v)[PER]) {
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

constexpr int GROUPS = 2;    // consumer warp groups, one per 32-key half of a tile

template <int DH, int NQW>
__global__ void __launch_bounds__((GROUPS * NQW + 1) * 32, NQW <= 2 ? 2 : 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const bf16* __restrict__ Q, int ld, int q_row0, int q_seq_stride, int q_len, int kv_row0,
                     int kv_seq_stride, int kv_len, int keys_per_split, float scale_log2, bf16* __restrict__ out,
                     int out_seq_stride, unsigned* err) {
  using S = AttnShape<DH>;
  constexpr int CW = GROUPS * NQW;   // consumer warps; warp CW is the producer
  const int split = blockIdx.x, n_split = gridDim.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + S::RING);
  uint64_t* empty = full + ASTAGES;
  int* abort_flag = reinterpret_cast<int*>(empty + ASTAGES);
  volatile int* abort = abort_flag;
  constexpr int QLD = DH + QLD_PAD;
  bf16* qs = reinterpret_cast<bf16*>(reinterpret_cast<uint8_t*>(full) + 2 * ASTAGES * sizeof(uint64_t) + 16);

  // stage the queries (16 rows per query warp, zero rows past q_len)
  for (int e = tid; e < NQW * 16 * (DH / 8); e += (GROUPS * NQW + 1) * 32) {
    const int r = e / (DH / 8), c = (e % (DH / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < q_len)
      v = *reinterpret_cast<const uint4*>(Q + static_cast<size_t>(q_row0 + b * q_seq_stride + r) * ld + h * DH + c);
    *reinterpret_cast<uint4*>(qs + r * QLD + c) = v;
  }
  if (tid == 0) {
    for (int s = 0; s < ASTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CW);    // every consumer warp releases every stage
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int k_begin = split * keys_per_split;
  const int k_end = min(kv_len, k_begin + keys_per_split);
  const int n_tiles = k_end > k_begin ? cdiv(k_end - k_begin, KT) : 0;
  const int kv_base = kv_row0 + b * kv_seq_stride + k_begin;

  float o[DH / 8][4];
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int g = lane >> 2, t4 = lane & 3;
  const int grp = warp / NQW, qw = warp % NQW;
  const int qi0 = qw * 16 + g, qi1 = qi0 + 8;

  if (warp == CW) {
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      uint32_t issued = 0, par = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % ASTAGES;
        const uint32_t ph = (it / ASTAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort, err)) break;
        mbar_expect_tx(&full[s], S::STAGE);
        uint8_t* kd = ring + s * S::STAGE;
#pragma unroll
        for (int sub = 0; sub < DH / 64; ++sub) {
          tma_load_2d(kd + sub * KT * 128, &tmK, h * DH + sub * 64, kv_base + it * KT, &full[s]);
          tma_load_2d(kd + S::TILE + sub * KT * 128, &tmV, h * DH + sub * 64, kv_base + it * KT, &full[s]);
        }
        issued |= 1u << s;
        par = (par & ~(1u << s)) | (ph << s);
      }
      if (*abort)
        for (int s = 0; s < ASTAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (par >> s) & 1u, nullptr, err);
    }
  } else {
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // ldmatrix row address of this lane in the warp's staged Q tile
    const uint32_t qrow = smem_u32(qs + (qw * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * QLD + (lane >> 4) * 8);
    // every consumer warp takes every tile, in order (so each wait targets the
    // stage's next phase); group grp covers keys [grp * HK, grp * HK + HK)
    constexpr int HK = KT / GROUPS, NT = HK / 8;
    for (int it = 0; it < n_tiles; ++it) {
      const int s = it % ASTAGES;
      const uint32_t ph = (it / ASTAGES) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&full[s], ph, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t kb = smem_u32(ring + s * S::STAGE), vb = kb + S::TILE;
      float sc[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < DH / 16; ++kc) {
        uint32_t qa[4];
        ldsm_x4(qrow + kc * 32, qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int key = grp * HK + np * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int dim = kc * 16 + (((lane >> 3) & 1) << 3);
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kb + swz(key, dim), r0, r1, r2, r3);
          mma16816(sc[2 * np], qa, r0, r1);
          mma16816(sc[2 * np + 1], qa, r2, r3);
        }
      }
      const int key0 = k_begin + it * KT + grp * HK;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int kidx = key0 + nt * 8 + 2 * t4 + (c & 1);
          sc[nt][c] = kidx < k_end ? sc[nt][c] * scale_log2 : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
      }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(mrow[0], mx0), mn1 = fmaxf(mrow[1], mx1);
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(mrow[0] - ref0), al1 = exp2f(mrow[1] - ref1);
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - ref0);
        sc[nt][1] = exp2f(sc[nt][1] - ref0);
        sc[nt][2] = exp2f(sc[nt][2] - ref1);
        sc[nt][3] = exp2f(sc[nt][3] - ref1);
        ls0 += sc[nt][0] + sc[nt][1];
        ls1 += sc[nt][2] + sc[nt][3];
      }
      lrow[0] = lrow[0] * al0 + ls0;
      lrow[1] = lrow[1] * al1 + ls1;
      mrow[0] = mn0;
      mrow[1] = mn1;
#pragma unroll
      for (int i = 0; i < DH / 8; ++i) {
        o[i][0] *= al0; o[i][1] *= al0;
        o[i][2] *= al1; o[i][3] *= al1;
      }
      // P = P_hi + P_lo, both bf16: the PV product keeps ~16 significant
      // bits of every softmax weight instead of bf16's 8 (hi pass, then lo
      // pass, so no accumulator is hit twice back to back)
#pragma unroll
      for (int kc2 = 0; kc2 < NT / 2; ++kc2) {
        uint32_t pp[2][4];
        split_bf16(sc[2 * kc2][0], sc[2 * kc2][1], pp[0][0], pp[1][0]);
        split_bf16(sc[2 * kc2][2], sc[2 * kc2][3], pp[0][1], pp[1][1]);
        split_bf16(sc[2 * kc2 + 1][0], sc[2 * kc2 + 1][1], pp[0][2], pp[1][2]);
        split_bf16(sc[2 * kc2 + 1][2], sc[2 * kc2 + 1][3], pp[0][3], pp[1][3]);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int dp = 0; dp < DH / 16; ++dp) {
            const int key = grp * HK + kc2 * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
            const int dim = dp * 16 + ((lane >> 4) << 3);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(vb + swz(key, dim), r0, r1, r2, r3);
            mma16816(o[2 * dp], pp[part], r0, r1);
            mma16816(o[2 * dp + 1], pp[part], r2, r3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      lrow[0] += __shfl_xor_sync(0xffffffffu, lrow[0], off);
      lrow[1] += __shfl_xor_sync(0xffffffffu, lrow[1], off);
    }
  }

  // ---- split merge across the cluster (distributed shared memory)
  __syncthreads();
  constexpr int QP = NQW * 16;                     // padded queries per CTA
  float* po = reinterpret_cast<float*>(ring);      // [GROUPS][QP][DH] unnormalised O
  float* pml = po + GROUPS * QP * DH;              // [GROUPS][QP][2] (m, l), log2 domain
  if (warp < CW) {
    float* pg = po + grp * QP * DH;
    float* mg = pml + grp * QP * 2;
#pragma unroll
    for (int dt = 0; dt < DH / 8; ++dt) {
      const int col = dt * 8 + 2 * t4;
      pg[qi0 * DH + col] = o[dt][0];
      pg[qi0 * DH + col + 1] = o[dt][1];
      pg[qi1 * DH + col] = o[dt][2];
      pg[qi1 * DH + col + 1] = o[dt][3];
    }
    if (t4 == 0) {
      mg[qi0 * 2] = mrow[0];
      mg[qi0 * 2 + 1] = lrow[0];
      mg[qi1 * 2] = mrow[1];
      mg[qi1 * 2 + 1] = lrow[1];
    }
  }
  cluster_sync_all();
  // CTA `split` finishes queries [split * qpc, split * qpc + qpc): one warp per
  // query; lane p < 2 n_split fetches partial p = (CTA p / 2, group p % 2)'s
  // (m, l), then every lane gathers its DH/32 output columns from all
  // partials with vector loads.
  constexpr int NW = CW + 1, PER = DH / 32;
  const int qpc = cdiv(q_len, n_split);
  const int n_part = GROUPS * n_split;
  for (int wq = warp; wq < qpc; wq += NW) {
    const int q = split * qpc + wq;
    if (q >= q_len) break;
    float m_r = -INFINITY, l_r = 0.f;
    if (lane < n_part) {
      const float* mg = pml + (lane % GROUPS) * QP * 2 + q * 2;
      m_r = ld_peer(mg, lane / GROUPS);
      l_r = ld_peer(mg + 1, lane / GROUPS);
    }
    float M = m_r;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float wr = (m_r == -INFINITY) ? 0.f : exp2f(m_r - M);
    float den = wr * l_r;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int p = 0; p < n_part; ++p) {
      const float wgt = __shfl_sync(0xffffffffu, wr, p);
      if (wgt == 0.f) continue;
      float v[PER];
      ld_peer_vec<PER>(po + (p % GROUPS) * QP * DH + q * DH + lane * PER, p / GROUPS, v);
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(wgt, v[i], acc[i]);
    }
    const float inv = 1.f / den;
    bf16* op = out + static_cast<size_t>(b * out_seq_stride + q) * ld + h * DH + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; i += 2)
      *reinterpret_cast<__nv_bfloat162*>(op + i) = __floats2bfloat162_rn(acc[i] * inv, acc[i + 1] * inv);
  }
  cluster_sync_all();
}

template <int DH>
__global__ void __launch_bounds__(32)
    attn_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V, int ld,
                    int q_row0, int q_seq_stride, int kv_row0, int kv_seq_stride, int kv_len, float scale,
                    float* __restrict__ out, int out_seq_stride) {
  constexpr int PER = DH / 32;
  const int qi = blockIdx.x, h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x;
  const float* qp = Q + static_cast<size_t>(q_row0 + b * q_seq_stride + qi) * ld + h * DH;
  float q[PER], acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    q[i] = qp[lane + 32 * i];
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < kv_len; ++j) {
    const size_t row = static_cast<size_t>(kv_row0 + b * kv_seq_stride + j) * ld + h * DH;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) s = fmaf(q[i], K[row + lane + 32 * i], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    s *= scale;
    const float mn = fmaxf(m, s);
    const float a = expf(m - mn), p = expf(s - mn);
    l = l * a + p;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = acc[i] * a + p * V[row + lane + 32 * i];
    m = mn;
  }
  float* op = out + static_cast<size_t>(b * out_seq_stride + qi) * ld + h * DH;
#pragma unroll
  for (int i = 0; i < PER; ++i) op[lane + 32 * i] = acc[i] / l;
}

template <int DH, int NQW>
cudaError_t launch_bf16(dllm_cache* c, const CUtensorMap& tk, const CUtensorMap& tv, const bf16* Q, int q_row0,
                        int q_seq_stride, int q_len, int kv_row0, int kv_seq_stride, int kv_len, int n_seq,
                        bf16* out, int out_seq_stride, cudaStream_t st) {
  const int H = c->cfg.n_heads;
  const int tiles = cdiv(kv_len, KT);
  // one wave at two CTAs per SM, every CTA with >= 2 tiles
  int n_split = std::min(8, std::max(1, (2 * c->num_sms) / (n_seq * H)));
  n_split = std::max(1, std::min(n_split, tiles / 2));
  const int per = cdiv(tiles, n_split);
  n_split = cdiv(tiles, per);
  const int keys_per_split = per * KT;
  constexpr size_t smem = attn_smem_bytes<DH, NQW>();
  static bool attr = false;
  if (!attr) {
    cudaError_t e = set_smem(attn_bf16_kernel<DH, NQW>, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_split, H, n_seq);
  cfg.blockDim = dim3((GROUPS * NQW + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = n_split;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  return cudaLaunchKernelEx(&cfg, attn_bf16_kernel<DH, NQW>, tk, tv, Q, c->d, q_row0, q_seq_stride, q_len, kv_row0,
                            kv_seq_stride, kv_len, keys_per_split, scale_log2, out, out_seq_stride, c->err);
}

template <int DH>
cudaError_t dispatch_nqw(dllm_cache* c, const CUtensorMap& tk, const CUtensorMap& tv, const bf16* Q, int q_row0,
                         int q_seq_stride, int q_len, int kv_row0, int kv_seq_stride, int kv_len, int n_seq,
                         bf16* out, int out_seq_stride, cudaStream_t st) {
  const int nqw = cdiv(q_len, 16);
  switch (nqw) {
    case 1: return launch_bf16<DH, 1>(c, tk, tv, Q, q_row0, q_seq_stride, q_len, kv_row0, kv_seq_stride, kv_len, n_seq, out, out_seq_stride, st);
    case 2: return launch_bf16<DH, 2>(c, tk, tv, Q, q_row0, q_seq_stride, q_len, kv_row0, kv_seq_stride, kv_len, n_seq, out, out_seq_stride, st);
    case 3: return launch_bf16<DH, 3>(c, tk, tv, Q, q_row0, q_seq_stride, q_len, kv_row0, kv_seq_stride, kv_len, n_seq, out, out_seq_stride, st);
    case 4: return launch_bf16<DH, 4>(c, tk, tv, Q, q_row0, q_seq_stride, q_len, kv_row0, kv_seq_stride, kv_len, n_seq, out, out_seq_stride, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t attn_dense(dllm_cache* c, int layer, int q_row0, int q_seq_stride, int q_len, int kv_row0,
                       int kv_seq_stride, int kv_len, int n_seq, void* out, int out_seq_stride, cudaStream_t st) {
  if (q_len <= 0 || kv_len <= 0 || n_seq <= 0) return cudaSuccess;
  const int d = c->d, dh = c->cfg.head_dim;
  const size_t layer_off = static_cast<size_t>(layer) * c->rows * d;
  if (c->cfg.dtype == DLLM_F32) {
    const float* Q = static_cast<const float*>(c->q) + layer_off;
    const float* K = static_cast<const float*>(c->k) + layer_off;
    const float* V = static_cast<const float*>(c->v) + layer_off;
    const dim3 grid(q_len, c->cfg.n_heads, n_seq);
    const float scale = 1.f / sqrtf(static_cast<float>(dh));
    switch (dh) {
      case 32: attn_f32_kernel<32><<<grid, 32, 0, st>>>(Q, K, V, d, q_row0, q_seq_stride, kv_row0, kv_seq_stride, kv_len, scale, static_cast<float*>(out), out_seq_stride); break;
      case 64: attn_f32_kernel<64><<<grid, 32, 0, st>>>(Q, K, V, d, q_row0, q_seq_stride, kv_row0, kv_seq_stride, kv_len, scale, static_cast<float*>(out), out_seq_stride); break;
      case 128: attn_f32_kernel<128><<<grid, 32, 0, st>>>(Q, K, V, d, q_row0, q_seq_stride, kv_row0, kv_seq_stride, kv_len, scale, static_cast<float*>(out), out_seq_stride); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  const uint64_t total_rows = static_cast<uint64_t>(c->cfg.n_layers) * c->rows;
  CUtensorMap tk, tv;
  if (!make_tmap_2d(&tk, c->k, d, total_rows, static_cast<uint64_t>(d) * 2, 64, KT, true) ||
      !make_tmap_2d(&tv, c->v, d, total_rows, static_cast<uint64_t>(d) * 2, 64, KT, true))
    return cudaErrorInvalidValue;
  const bf16* Q = static_cast<const bf16*>(c->q) + layer_off;
  const int kv0 = layer * c->rows + kv_row0;
  bf16* o = static_cast<bf16*>(out);
  if (dh == 128)
    return dispatch_nqw<128>(c, tk, tv, Q, q_row0, q_seq_stride, q_len, kv0, kv_seq_stride, kv_len, n_seq, o, out_seq_stride, st);
  if (dh == 64)
    return dispatch_nqw<64>(c, tk, tv, Q, q_row0, q_seq_stride, q_len, kv0, kv_seq_stride, kv_len, n_seq, o, out_seq_stride, st);
  return cudaErrorInvalidValue;
}

}  // namespace dllm
