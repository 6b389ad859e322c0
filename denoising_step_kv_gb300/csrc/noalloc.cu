// lmhead_conf for callers that cannot allocate device memory: the same
// kernels as lmhead_conf, with their scratch (per-tile softmax statistics,
// row scales and an error word) in one file-scope static device array.
#include <mutex>
#include <string>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace dllm {
namespace {

constexpr int NA_MAX_ROWS = 256;             // rows of h per call
constexpr int NA_MAX_VOCAB = 131072;         // vocabulary size per call
constexpr int NA_MAX_TILES = NA_MAX_VOCAB / 128;
constexpr size_t NA_PART_BYTES = static_cast<size_t>(NA_MAX_ROWS) * NA_MAX_TILES * sizeof(LMPart);
constexpr size_t NA_RS_OFF = NA_PART_BYTES;
constexpr size_t NA_ERR_OFF = NA_RS_OFF + NA_MAX_ROWS * sizeof(float);
constexpr size_t NA_BYTES = NA_ERR_OFF + 256;   // 4 MiB + 1.25 KiB

// Held by every GPU that loads the library, until the process exits.  Host
// code must not use this name as a pointer: it resolves the device address
// with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_lmhead_scratch[NA_BYTES];

std::mutex g_scratch_mu;
constexpr int MAX_DEVICES = 64;
void* g_scratch_addr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device, resolved once
// per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

dllm_status na_fail(dllm_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" dllm_status lmhead_conf_noalloc(const void* h_dev, const void* w_lm_dev, int M, int V, int d, int dtype,
                                           int mask_id, float rms_eps, int32_t* argmax_dev, float* p_top1_dev,
                                           float* entropy_dev, void* stream) {
  if (!h_dev || !w_lm_dev || !argmax_dev || !p_top1_dev || !entropy_dev)
    return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: null pointer");
  if (dtype != DLLM_F32 && dtype != DLLM_BF16) return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: bad dtype");
  if (M < 0 || M > NA_MAX_ROWS)
    return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: M outside [0, 256] (the static scratch's row limit)");
  if (V < 2 || V > NA_MAX_VOCAB)
    return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: V outside [2, 131072] (the static scratch's vocab limit)");
  if (d < 64 || d % 64 != 0) return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: d must be a positive multiple of 64");
  if (mask_id >= V) return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: mask_id >= V");
  if (!(rms_eps >= 0.f)) return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: rms_eps < 0");
  if ((reinterpret_cast<uintptr_t>(h_dev) | reinterpret_cast<uintptr_t>(w_lm_dev)) & 15u)
    return na_fail(DLLM_EINVAL, "lmhead_conf_noalloc: h and w_lm must be 16-byte aligned");
  if (M == 0) return DLLM_OK;

  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess)
    return na_fail(DLLM_ECUDA, std::string("lmhead_conf_noalloc: scratch address: ") + cudaGetErrorString(e));
  uint8_t* scratch = static_cast<uint8_t*>(base);

  // launch context on the host stack (no device memory is allocated)
  dllm_cache ctx;
  ctx.cfg = dllm_cache_cfg{};
  ctx.cfg.dtype = dtype;
  ctx.cfg.rms_eps = rms_eps;
  ctx.err = reinterpret_cast<unsigned*>(scratch + NA_ERR_OFF);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return na_fail(DLLM_ECUDA, "lmhead_conf_noalloc: no CUDA device");
  ctx.d = d;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* rs = reinterpret_cast<float*>(scratch + NA_RS_OFF);
  const int n_tiles = lm_slots(&ctx, M, V);
  // the error word is the only scratch that must start at zero; the
  // statistics and row scales are fully rewritten by every call.  A wait
  // that gives up leaves some statistics unwritten and sets the word, and
  // the merge then writes argmax -1 and NaN instead of stale results.
  if ((e = cudaMemsetAsync(ctx.err, 0, sizeof(unsigned), st)) != cudaSuccess ||
      (e = launch_rownorm(&ctx, h_dev, M, nullptr, d, rs, st)) != cudaSuccess ||
      (e = gemm_lm(&ctx, h_dev, w_lm_dev, M, nullptr, V, d, rs, mask_id, scratch, n_tiles, st)) != cudaSuccess ||
      (e = launch_lm_merge(scratch, M, nullptr, n_tiles, argmax_dev, p_top1_dev, entropy_dev, ctx.err, st)) !=
          cudaSuccess)
    return na_fail(DLLM_ECUDA, std::string("lmhead_conf_noalloc: ") + cudaGetErrorString(e));
  return DLLM_OK;
}
