// prune.cu — the two memory-bound kernels of the path.
//
//   prune24_kernel            2:4 magnitude prune-and-compress of W (A1).
//   double_prune24_kernel     transpose of the pruned W, pruned 2:4 again
//                             along the old out dimension (A2).
//
// Source: "SLoPe: Double-Pruned Sparse Plus Lazy Low-Rank Adapter Pretraining
// of LLMs", §1 and §2.1 (N:M pruning of the weight, then of its transpose)
// and §2.3 / App. K (compressed formats for both).  Ranking uses the exact
// magnitude key (bits & 0x7FFF) with ties to the lower index; the
// compressed format is the one slope.h documents.
#include <cuda_runtime.h>

#include <cstdint>

#include "slope_internal.h"

namespace slope {
namespace {

// Packs a 16-bit bf16 pattern and its in-group index into one integer whose
// order is the ranking: larger magnitude first, then lower index.  The sign
// sits below the index so the pattern can be rebuilt from the winner.
__device__ __forceinline__ uint32_t rank_key(uint32_t bits16, uint32_t j) {
  return ((bits16 & 0x7FFFu) << 3) | ((3u - j) << 1) | (bits16 >> 15);
}

__device__ __forceinline__ uint32_t pattern_of(uint32_t key) {
  return (key >> 3) | ((key & 1u) << 15);
}

// Top two of a group of four bf16 patterns.  Returns the kept pair packed
// (lower column in the low half) and writes the nibble i0 | i1 << 2.
__device__ __forceinline__ uint32_t top2of4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3,
                                            uint32_t& nibble) {
  const uint32_t k0 = rank_key(b0, 0), k1 = rank_key(b1, 1);
  const uint32_t k2 = rank_key(b2, 2), k3 = rank_key(b3, 3);
  const uint32_t a = max(k0, k1), b = min(k0, k1);
  const uint32_t c = max(k2, k3), d = min(k2, k3);
  const uint32_t first = max(a, c);
  const uint32_t second = max(min(a, c), max(b, d));
  const uint32_t j1 = 3u - ((first >> 1) & 3u);
  const uint32_t j2 = 3u - ((second >> 1) & 3u);
  const bool ordered = j1 < j2;
  const uint32_t lo = ordered ? j1 : j2, hi = ordered ? j2 : j1;
  const uint32_t vlo = pattern_of(ordered ? first : second);
  const uint32_t vhi = pattern_of(ordered ? second : first);
  nibble = lo | (hi << 2);
  return vlo | (vhi << 16);
}

// ---------------------------------------------------------------- A1 ------
// One 16-byte chunk = 8 consecutive weights of a row = 2 groups -> 8 bytes of
// kept values and one metadata byte.  Row-major contiguity makes chunk c of
// the flattened matrix map to vals[c] (uint2) and meta[c]; every warp access
// is fully coalesced.

constexpr int kPruneThreads = 256;
constexpr int kPruneUnroll = 4;

__global__ void __launch_bounds__(kPruneThreads) prune24_kernel(const uint4* __restrict__ W,
                                                                uint2* __restrict__ vals,
                                                                uint8_t* __restrict__ meta,
                                                                int64_t nchunks) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       base < nchunks; base += stride * kPruneUnroll) {
    uint4 w[kPruneUnroll];
#pragma unroll
    for (int u = 0; u < kPruneUnroll; ++u) {
      const int64_t c = base + u * stride;
      if (c < nchunks) w[u] = __ldcs(W + c);
    }
#pragma unroll
    for (int u = 0; u < kPruneUnroll; ++u) {
      const int64_t c = base + u * stride;
      if (c < nchunks) {
        uint32_t n0, n1;
        const uint32_t p0 = top2of4(w[u].x & 0xFFFFu, w[u].x >> 16, w[u].y & 0xFFFFu,
                                    w[u].y >> 16, n0);
        const uint32_t p1 = top2of4(w[u].z & 0xFFFFu, w[u].z >> 16, w[u].w & 0xFFFFu,
                                    w[u].w >> 16, n1);
        __stcs(vals + c, make_uint2(p0, p1));
        meta[c] = static_cast<uint8_t>(n0 | (n1 << 4));
      }
    }
  }
}

// ---------------------------------------------------------------- A2 ------
// Work item: 8 consecutive rows (one "octet" h8) x 16 consecutive columns
// (chunk c16) of the rows x cols pruned weight.  It reads 8 x 16 B of kept
// values and 8 x 2 B of metadata, rebuilds the 8 x 16 block (pruned = +0),
// and for each of the 16 columns i prunes the two row-quadruples along the
// old row dimension: 4 kept values (8 B) and one metadata byte for row i of
// the transposed output, at column octet h8.  Lanes of a warp take
// consecutive octets of the same chunk, so each output row segment a warp
// writes is 256 B (values) / 32 B (metadata) contiguous.

constexpr int kDpThreads = 256;  // 8 warps = 8 column chunks per tile

__device__ __forceinline__ uint32_t expanded(uint32_t pair, uint32_t nib, uint32_t j) {
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  return (j == i0) ? (pair & 0xFFFFu) : ((j == i1) ? (pair >> 16) : 0u);
}

__global__ void __launch_bounds__(kDpThreads) double_prune24_kernel(
    const uint4* __restrict__ vals, const uint16_t* __restrict__ meta, uint2* __restrict__ t_vals,
    uint8_t* __restrict__ t_meta, int64_t rows, int64_t cols) {
  const int64_t n_h8 = rows / 8, n_c16 = cols / 16;
  const int64_t tiles_h = (n_h8 + 31) / 32, tiles_c = (n_c16 + 7) / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t tile = blockIdx.x; tile < tiles_h * tiles_c; tile += gridDim.x) {
    const int64_t h8 = (tile % tiles_h) * 32 + lane;
    const int64_t c16 = (tile / tiles_h) * 8 + warp;
    if (h8 >= n_h8 || c16 >= n_c16) continue;
    uint4 v[8];
    uint32_t m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t row = 8 * h8 + k;
      v[k] = __ldcs(vals + row * n_c16 + c16);
      m[k] = __ldcs(meta + row * n_c16 + c16);
    }
    const int64_t out_stride = rows / 8;  // uint2 / bytes per output row
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // group of 4 columns within the chunk
      uint32_t pair[8], nib[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        pair[k] = (q == 0) ? v[k].x : (q == 1) ? v[k].y : (q == 2) ? v[k].z : v[k].w;
        nib[k] = (m[k] >> (4 * q)) & 0xFu;
      }
#pragma unroll
      for (uint32_t j = 0; j < 4; ++j) {
        uint32_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = expanded(pair[k], nib[k], j);
        uint32_t na, nb;
        const uint32_t pa = top2of4(e[0], e[1], e[2], e[3], na);
        const uint32_t pb = top2of4(e[4], e[5], e[6], e[7], nb);
        const int64_t i = 16 * c16 + 4 * q + j;
        __stcs(t_vals + i * out_stride + h8, make_uint2(pa, pb));
        t_meta[i * out_stride + h8] = static_cast<uint8_t>(na | (nb << 4));
      }
    }
  }
}

}  // namespace

cudaError_t launch_prune24(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream) {
  const int64_t nchunks = rows * cols / 8;
  if (nchunks == 0) return cudaSuccess;
  const int64_t per_block = static_cast<int64_t>(kPruneThreads) * kPruneUnroll;
  int64_t blocks = (nchunks + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  prune24_kernel<<<static_cast<unsigned>(blocks), kPruneThreads, 0, stream>>>(
      static_cast<const uint4*>(W), static_cast<uint2*>(vals), meta, nchunks);
  return cudaGetLastError();
}

cudaError_t launch_double_prune24(const void* vals, const uint8_t* meta, int64_t rows,
                                  int64_t cols, void* t_vals, uint8_t* t_meta,
                                  cudaStream_t stream) {
  const int64_t tiles = ((rows / 8 + 31) / 32) * ((cols / 16 + 7) / 8);
  if (tiles == 0) return cudaSuccess;
  int64_t blocks = tiles;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  double_prune24_kernel<<<static_cast<unsigned>(blocks), kDpThreads, 0, stream>>>(
      static_cast<const uint4*>(vals), reinterpret_cast<const uint16_t*>(meta),
      static_cast<uint2*>(t_vals), t_meta, rows, cols);
  return cudaGetLastError();
}

}  // namespace slope
