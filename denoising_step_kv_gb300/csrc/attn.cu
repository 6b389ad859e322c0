// Cached bidirectional attention of a few queries per (sequence, head) over
// the whole cached sequence: HBM-bound streaming of K/V.
//
// bf16: grid (n_split, H, B) launched as clusters of n_split CTAs.  In each
// CTA a producer warp streams 64-key K and V tiles of its key range with TMA
// (128-byte swizzle) into a 3-stage mbarrier ring; NQW consumer warps (16
// queries each) compute S = Q K^T and O += P V with mma.sync m16n8k16 (bf16
// in, fp32 accumulate) from ldmatrix fragments and keep an online softmax in
// the log2 domain.  The split partials (m, l, O) are merged across the cluster
// through distributed shared memory, so no partial ever reaches HBM.
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

template <int DH, int NQW>
constexpr size_t attn_smem_bytes() {
  return 1024 + AttnShape<DH>::RING + 2 * ASTAGES * sizeof(uint64_t) + 16;
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
__device__ __forceinline__ uint32_t ld_u32(const bf16* p) { return *reinterpret_cast<const uint32_t*>(p); }

template <int DH, int NQW>
__global__ void __launch_bounds__((NQW + 1) * 32)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const bf16* __restrict__ Q, int ld, int q_row0, int q_seq_stride, int q_len, int kv_row0,
                     int kv_seq_stride, int kv_len, int keys_per_split, float scale_log2, bf16* __restrict__ out,
                     int out_seq_stride, unsigned* err) {
  using S = AttnShape<DH>;
  constexpr int NT = (NQW + 1) * 32;
  const int split = blockIdx.x, n_split = gridDim.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + S::RING);
  uint64_t* empty = full + ASTAGES;
  int* abort_flag = reinterpret_cast<int*>(empty + ASTAGES);
  volatile int* abort = abort_flag;

  if (tid == 0) {
    for (int s = 0; s < ASTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NQW);
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
  const int qi0 = warp * 16 + g, qi1 = qi0 + 8;

  if (warp == NQW) {
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
    // Q fragments (A operand, rows qi0 / qi1) straight from the cache
    uint32_t qa[DH / 16][4];
    const bool v0 = qi0 < q_len, v1 = qi1 < q_len;
    const bf16* q0p = Q + static_cast<size_t>(q_row0 + b * q_seq_stride + (v0 ? qi0 : 0)) * ld + h * DH;
    const bf16* q1p = Q + static_cast<size_t>(q_row0 + b * q_seq_stride + (v1 ? qi1 : 0)) * ld + h * DH;
#pragma unroll
    for (int kc = 0; kc < DH / 16; ++kc) {
      qa[kc][0] = v0 ? ld_u32(q0p + kc * 16 + 2 * t4) : 0u;
      qa[kc][1] = v1 ? ld_u32(q1p + kc * 16 + 2 * t4) : 0u;
      qa[kc][2] = v0 ? ld_u32(q0p + kc * 16 + 8 + 2 * t4) : 0u;
      qa[kc][3] = v1 ? ld_u32(q1p + kc * 16 + 8 + 2 * t4) : 0u;
    }
    for (int it = 0; it < n_tiles; ++it) {
      const int s = it % ASTAGES;
      const uint32_t ph = (it / ASTAGES) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&full[s], ph, abort, err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t kb = smem_u32(ring + s * S::STAGE), vb = kb + S::TILE;
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < DH / 16; ++kc) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int key = np * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int dim = kc * 16 + (((lane >> 3) & 1) << 3);
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kb + swz(key, dim), r0, r1, r2, r3);
          mma16816(sc[2 * np], qa[kc], r0, r1);
          mma16816(sc[2 * np + 1], qa[kc], r2, r3);
        }
      }
      const int key0 = k_begin + it * KT;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
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
      for (int nt = 0; nt < 8; ++nt) {
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
      // bits of every softmax weight instead of bf16's 8
#pragma unroll
      for (int kc2 = 0; kc2 < 4; ++kc2) {
        uint32_t ph[4], pl[4];
        split_bf16(sc[2 * kc2][0], sc[2 * kc2][1], ph[0], pl[0]);
        split_bf16(sc[2 * kc2][2], sc[2 * kc2][3], ph[1], pl[1]);
        split_bf16(sc[2 * kc2 + 1][0], sc[2 * kc2 + 1][1], ph[2], pl[2]);
        split_bf16(sc[2 * kc2 + 1][2], sc[2 * kc2 + 1][3], ph[3], pl[3]);
#pragma unroll
        for (int dp = 0; dp < DH / 16; ++dp) {
          const int key = kc2 * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int dim = dp * 16 + ((lane >> 4) << 3);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vb + swz(key, dim), r0, r1, r2, r3);
          mma16816(o[2 * dp], ph, r0, r1);
          mma16816(o[2 * dp + 1], ph, r2, r3);
          mma16816(o[2 * dp], pl, r0, r1);
          mma16816(o[2 * dp + 1], pl, r2, r3);
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
  float* po = reinterpret_cast<float*>(ring);      // [NQW*16][DH] unnormalised O
  float* pml = po + NQW * 16 * DH;                 // [NQW*16][2] (m, l), log2 domain
  if (warp < NQW) {
#pragma unroll
    for (int dt = 0; dt < DH / 8; ++dt) {
      const int col = dt * 8 + 2 * t4;
      po[qi0 * DH + col] = o[dt][0];
      po[qi0 * DH + col + 1] = o[dt][1];
      po[qi1 * DH + col] = o[dt][2];
      po[qi1 * DH + col + 1] = o[dt][3];
    }
    if (t4 == 0) {
      pml[qi0 * 2] = mrow[0];
      pml[qi0 * 2 + 1] = lrow[0];
      pml[qi1 * 2] = mrow[1];
      pml[qi1 * 2 + 1] = lrow[1];
    }
  }
  cluster_sync_all();
  const int qpc = cdiv(q_len, n_split);
  for (int idx = tid; idx < qpc * DH; idx += NT) {
    const int q = split * qpc + idx / DH, e = idx % DH;
    if (q >= q_len) continue;
    float M = -INFINITY;
    for (int r = 0; r < n_split; ++r) M = fmaxf(M, ld_peer(pml + q * 2, r));
    float num = 0.f, den = 0.f;
    for (int r = 0; r < n_split; ++r) {
      const float m = ld_peer(pml + q * 2, r);
      if (m == -INFINITY) continue;
      const float w = exp2f(m - M);
      den += w * ld_peer(pml + q * 2 + 1, r);
      num += w * ld_peer(po + q * DH + e, r);
    }
    out[static_cast<size_t>(b * out_seq_stride + q) * ld + h * DH + e] = __float2bfloat16_rn(num / den);
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
  int n_split = std::min(8, std::max(1, cdiv(3 * c->num_sms, n_seq * H)));
  n_split = std::min(n_split, tiles);
  const int per = cdiv(tiles, n_split);
  n_split = cdiv(tiles, per);
  const int keys_per_split = per * KT;
  constexpr size_t smem = attn_smem_bytes<DH, NQW>();
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel<DH, NQW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_split, H, n_seq);
  cfg.blockDim = dim3((NQW + 1) * 32);
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
