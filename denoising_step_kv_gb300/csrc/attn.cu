// Cached bidirectional attention of a few queries per (sequence, head) over
// the whole cached sequence: HBM-bound streaming of K/V from the tiled cache.
// bf16: the tensor-core kernel of attn_tc.cuh.  fp32: one warp per (query,
// head, sequence) with an online softmax in fp32.
#include <algorithm>
#include <atomic>

#include "attn_tc.cuh"
#include "attn_fa.cuh"
#include "attn_rows.cuh"
#include "common.cuh"
#include "internal.h"

namespace dllm {
namespace {

// element e of head h, row pos of sequence b in a tiled fp32 cache
__device__ __forceinline__ float kv_at(const uint8_t* base, const KvLayout& kv, int b, int h, int pos, int e) {
  return *reinterpret_cast<const float*>(base + kv.chunk_off(b, h, pos, e >> 2) + (e & 3) * 4);
}

template <int DH>
__global__ void __launch_bounds__(32)
    attn_f32_kernel(const uint8_t* __restrict__ Ql, const uint8_t* __restrict__ Kl, const uint8_t* __restrict__ Vl,
                    KvLayout kv, int ld, int q_pos0, int q_len, int kv_len, float scale,
                    const uint8_t* __restrict__ seq_done, float* __restrict__ out) {
  constexpr int PER = DH / 32;
  const int qi = blockIdx.x, h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x;
  if (seq_done && seq_done[b]) return;       // the sequence has ended its block
  float q[PER], acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    q[i] = kv_at(Ql, kv, b, h, q_pos0 + qi, lane + 32 * i);
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < kv_len; ++j) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) s = fmaf(q[i], kv_at(Kl, kv, b, h, j, lane + 32 * i), s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    s *= scale;
    const float mn = fmaxf(m, s);
    const float a = expf(m - mn), p = expf(s - mn);
    l = l * a + p;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = acc[i] * a + p * kv_at(Vl, kv, b, h, j, lane + 32 * i);
    m = mn;
  }
  float* op = out + static_cast<size_t>(b * q_len + qi) * ld + h * DH;
#pragma unroll
  for (int i = 0; i < PER; ++i) op[lane + 32 * i] = acc[i] / l;
}

template <int DH, int R>
cudaError_t launch_tc_r(dllm_cache* c, const uint8_t* Ql, const uint8_t* Kl, const uint8_t* Vl, int q_pos0, int q_len,
                        int kv_len, int n_seq, bf16* out, cudaStream_t st) {
  using S = attn_tc::Shape<DH, R>;
  const int H = c->cfg.n_heads;
  const int tiles = cdiv(kv_len, attn_tc::KT);
  // one CTA per SM (about 210 KB of shared memory), one wave
  int n_split = std::min(8, std::max(1, c->num_sms / (n_seq * H)));
  n_split = std::max(1, std::min(n_split, tiles));
  const int per = cdiv(tiles, n_split);
  n_split = cdiv(tiles, per);
  const int keys_per_split = per * attn_tc::KT;
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, attn_tc::attn_tc_kernel<DH, R>, S::SMEM);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  const uint8_t* done = c->cfg.sink == 0 ? done_flags(c) : nullptr;
  return launch_ex(attn_tc::attn_tc_kernel<DH, R>, dim3(n_split, H, n_seq), dim3(192), S::SMEM, st, n_split, Ql, Kl,
                   Vl, c->kv, c->d, q_pos0, q_len, kv_len, keys_per_split, scale_log2, done, out, c->err);
}

// Replicas R of the queries in the 128 MMA rows: as many as fit.
template <int DH>
cudaError_t launch_tc(dllm_cache* c, const uint8_t* Ql, const uint8_t* Kl, const uint8_t* Vl, int q_pos0, int q_len,
                      int kv_len, int n_seq, bf16* out, cudaStream_t st) {
  if (q_len <= 32) return launch_tc_r<DH, 4>(c, Ql, Kl, Vl, q_pos0, q_len, kv_len, n_seq, out, st);
  if (q_len <= 64) return launch_tc_r<DH, 2>(c, Ql, Kl, Vl, q_pos0, q_len, kv_len, n_seq, out, st);
  return launch_tc_r<DH, 1>(c, Ql, Kl, Vl, q_pos0, q_len, kv_len, n_seq, out, st);
}

}  // namespace

template <int DH>
cudaError_t launch_rows(dllm_cache* c, const uint8_t* Ql, const uint8_t* Kl, const uint8_t* Vl, const int* rows,
                        const int* n_rows, bf16* out, cudaStream_t st) {
  using S = attn_rows::Shape<DH>;
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, attn_rows::attn_rows_kernel<DH>, S::SMEM);
    if (e != cudaSuccess) return e;
  }
  // CTAs resident per SM (two at dh 64: twice the softmax warps to hide
  // each one's TMEM and barrier latency), asked once per device
  static std::atomic<int> resident[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  int per_sm = dev < 64 ? resident[dev].load(std::memory_order_acquire) : 0;
  if (per_sm == 0) {
    // from the SM's shared memory and registers (the largest carveout is
    // requested, so that two CTAs' worth of shared memory is there)
    cudaFuncSetAttribute(attn_rows::attn_rows_kernel<DH>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    cudaFuncAttributes fa;
    int smem_sm = 0, resv = 0, regs_sm = 0;
    per_sm = 1;
    if (cudaFuncGetAttributes(&fa, attn_rows::attn_rows_kernel<DH>) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) == cudaSuccess) {
      const size_t per_cta = S::SMEM + fa.sharedSizeBytes + resv;
      const int regs_cta = ((fa.numRegs + 7) / 8 * 8) * 192;
      per_sm = static_cast<int>(std::min<size_t>(smem_sm / per_cta, regs_sm / std::max(1, regs_cta)));
    }
    cudaGetLastError();
    per_sm = std::max(1, std::min(per_sm, 2));
    if (dev < 64) resident[dev].store(per_sm, std::memory_order_release);
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  return launch_ex(attn_rows::attn_rows_kernel<DH>, dim3(per_sm * c->num_sms), dim3(192), S::SMEM, st, 0, Ql, Kl, Vl,
                   c->kv, c->cfg.seq_len, c->cfg.batch, c->cfg.n_heads, rows, n_rows, c->seq_rows, scale_log2, out,
                   c->err);
}

cudaError_t attn_rows_dense(dllm_cache* c, int layer, const int* rows, const int* n_rows, void* out,
                            cudaStream_t st) {
  const size_t off = static_cast<size_t>(layer) * c->kv_layer_bytes;
  const uint8_t* Ql = static_cast<const uint8_t*>(c->q) + off;
  const uint8_t* Kl = static_cast<const uint8_t*>(c->k) + off;
  const uint8_t* Vl = static_cast<const uint8_t*>(c->v) + off;
  bf16* o = static_cast<bf16*>(out);
  if (c->cfg.head_dim == 128) return launch_rows<128>(c, Ql, Kl, Vl, rows, n_rows, o, st);
  if (c->cfg.head_dim == 64) return launch_rows<64>(c, Ql, Kl, Vl, rows, n_rows, o, st);
  return cudaErrorInvalidValue;
}

template <int DH, int R>
cudaError_t launch_fa_r(dllm_cache* c, int q_pos0, int q_len, bf16* out, cudaStream_t st) {
  using S = attn_fa::Shape<DH, R>;
  static PerDeviceOnce attr;
  {
    const cudaError_t e = set_smem_once(attr, attn_fa::attn_fa_kernel<DH, R>, S::SMEM);
    if (e != cudaSuccess) return e;
  }
  const int L = c->cfg.seq_len, Rd = c->cfg.swd_R;
  // the window: every 64-key tile that [q0 - R, q0 + q_len + R) touches
  const int w_lo = std::max(0, q_pos0 - Rd) / attn_tc::KT;
  const int w_hi = (std::min(L, q_pos0 + q_len + Rd) - 1) / attn_tc::KT + 1;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  const uint8_t* Ql = static_cast<const uint8_t*>(c->q);     // layer 0
  const uint8_t* Kl = static_cast<const uint8_t*>(c->k);
  const uint8_t* Vl = static_cast<const uint8_t*>(c->v);
  return launch_ex(attn_fa::attn_fa_kernel<DH, R>, dim3(c->cfg.n_heads, c->cfg.batch), dim3(192), S::SMEM, st, 0, Ql,
                   Kl, Vl, c->kv, c->d, q_pos0, q_len, L, w_lo, w_hi, scale_log2, c->tok_w, L, c->fa_state,
                   c->fa_key, done_flags(c), out, c->err, c->fa_rebuilt);
}

cudaError_t attn_facache(dllm_cache* c, int q_pos0, int q_len, void* out, cudaStream_t st) {
  bf16* o = static_cast<bf16*>(out);
  const int dh = c->cfg.head_dim;
  if (dh == 128) {
    if (q_len <= 32) return launch_fa_r<128, 4>(c, q_pos0, q_len, o, st);
    return launch_fa_r<128, 2>(c, q_pos0, q_len, o, st);
  }
  if (dh == 64) {
    if (q_len <= 32) return launch_fa_r<64, 4>(c, q_pos0, q_len, o, st);
    return launch_fa_r<64, 2>(c, q_pos0, q_len, o, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t attn_dense(dllm_cache* c, int layer, int q_pos0, int q_len, int kv_len, int n_seq, void* out,
                       cudaStream_t st) {
  if (q_len <= 0 || kv_len <= 0 || n_seq <= 0) return cudaSuccess;
  const int dh = c->cfg.head_dim;
  const size_t off = static_cast<size_t>(layer) * c->kv_layer_bytes;
  const uint8_t* Ql = static_cast<const uint8_t*>(c->q) + off;
  const uint8_t* Kl = static_cast<const uint8_t*>(c->k) + off;
  const uint8_t* Vl = static_cast<const uint8_t*>(c->v) + off;
  // early exit applies to the active block of a dense cache, not to a stream
  const uint8_t* done = c->cfg.sink == 0 ? done_flags(c) : nullptr;
  if (c->cfg.dtype == DLLM_F32) {
    const dim3 grid(q_len, c->cfg.n_heads, n_seq);
    const float scale = 1.f / sqrtf(static_cast<float>(dh));
    float* o = static_cast<float*>(out);
    switch (dh) {
      case 32: attn_f32_kernel<32><<<grid, 32, 0, st>>>(Ql, Kl, Vl, c->kv, c->d, q_pos0, q_len, kv_len, scale, done, o); break;
      case 64: attn_f32_kernel<64><<<grid, 32, 0, st>>>(Ql, Kl, Vl, c->kv, c->d, q_pos0, q_len, kv_len, scale, done, o); break;
      case 128: attn_f32_kernel<128><<<grid, 32, 0, st>>>(Ql, Kl, Vl, c->kv, c->d, q_pos0, q_len, kv_len, scale, done, o); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  bf16* o = static_cast<bf16*>(out);
  if (dh == 128) return launch_tc<128>(c, Ql, Kl, Vl, q_pos0, q_len, kv_len, n_seq, o, st);
  if (dh == 64) return launch_tc<64>(c, Ql, Kl, Vl, q_pos0, q_len, kv_len, n_seq, o, st);
  return cudaErrorInvalidValue;
}

}  // namespace dllm
