// Tiled layout of the Q/K/V cache (shared by host and device code).
#pragma once
#include <stddef.h>

#include <cuda_runtime.h>

namespace dllm {

// A layer's Q, K and V caches hold, for every (sequence, head), Lp rows (the
// sequence length or ring size rounded up to 64) as tiles of 64 rows.  A tile
// is the exact shared-memory image the tensor cores read: row_bytes / 128
// sub-tiles of 64 rows x 128 bytes, and inside a sub-tile the 16-byte chunk c
// of row r sits at chunk position c ^ (r % 8) (the 128-byte swizzle).  One
// tile is therefore one contiguous bulk copy.
struct KvLayout {
  int H;          // heads
  int Lp;         // rows per (sequence, head) block, multiple of 64
  int row_bytes;  // head_dim * element size, multiple of 128
  // byte offset of the 16-byte chunk `chunk` (of row_bytes / 16) of row `pos`
  // of head h of sequence b
  __host__ __device__ __forceinline__ size_t chunk_off(int b, int h, int pos, int chunk) const {
    const size_t block = static_cast<size_t>(b * H + h) * Lp;
    const int sub = chunk >> 3, cc = chunk & 7, r = pos & 63;
    return (block + (pos & ~63)) * row_bytes + static_cast<size_t>(sub) * 8192 + r * 128 +
           (static_cast<size_t>(cc ^ (r & 7)) << 4);
  }
  // byte offset of the first row of the 64-row tile holding row `pos`
  __host__ __device__ __forceinline__ size_t tile_off(int b, int h, int pos) const {
    return (static_cast<size_t>(b * H + h) * Lp + (pos & ~63)) * row_bytes;
  }
  __host__ __device__ __forceinline__ size_t layer_bytes(int B) const {
    return static_cast<size_t>(B) * H * Lp * row_bytes;
  }
};

}  // namespace dllm
