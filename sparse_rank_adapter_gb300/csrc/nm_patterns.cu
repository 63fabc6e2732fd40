// nm_patterns.cu — the 1:2 and 2:8 patterns of the method's N:M family.
//
// Source: "SLoPe: Double-Pruned Sparse Plus Lazy Low-Rank Adapter Pretraining
// of LLMs", §2.1 "Double-pruned backward pass" (the weight is pruned N:M,
// its transpose N:M again; 1:2, 2:4 and 2:8 are the patterns it counts the
// added zeros of, derived in §T.1 "Lemma 2.1").
//
// 1:2 keeps the entry of larger magnitude of every aligned pair.  Two pairs
// make a quadruple with exactly two kept entries, one per half, so a 1:2
// matrix is a 2:4 matrix and is written in the 2:4 format (slope.h): the
// 2:4 sparse tensor-core GEMMs take it as it is.
//
// 2:8 keeps the two entries of largest magnitude of every aligned group of
// eight, in its own format: vals rows x cols/4 (the two kept values of a
// group, ascending), meta rows x cols/8 bytes (i0 | i1 << 3, i0 < i1).  It
// is also a 2:4 matrix; expand28_kernel writes that 2:4 form for the GEMMs
// (each quadruple's kept entries padded to two with its lowest free
// positions, +0 there), and the weight gradient masks with the 2:8 bytes.
//
// Ranking: the key bf16 bits & 0x7FFF (exact magnitude), the lower index on
// ties; pruned-away positions of a double pruning's input count as +0.
// Every kernel here is memory-bound: one pass over its input, coalesced row
// segments, no shared state between threads.
#include <cuda_runtime.h>

#include <cstdint>

#include "slope_internal.h"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t key15(uint32_t bf16) { return bf16 & 0x7FFFu; }

// ------------------------------------------------------------------ 1:2 ---

// One aligned pair (a word: lower column in the low half): 1 if the upper
// entry's magnitude is strictly larger (ties keep the lower column).
__device__ __forceinline__ uint32_t pick_upper(uint32_t w) {
  return key15(w >> 16) > key15(w & 0xFFFFu) ? 1u : 0u;
}

// The kept entries of two pairs (x: columns 0-1, y: columns 2-3 of a
// quadruple) packed as one word, and the quadruple's nibble.
__device__ __forceinline__ uint32_t keep12(uint32_t x, uint32_t y, uint32_t& nib) {
  const uint32_t px = pick_upper(x), py = pick_upper(y);
  nib = px | ((2u + py) << 2);
  const uint32_t sel = (px ? 0x32u : 0x10u) | ((py ? 0x76u : 0x54u) << 8);
  return __byte_perm(x, y, sel);
}

// A1 for 1:2: one 16-byte chunk (8 weights = 2 quadruples) per item.
__global__ void __launch_bounds__(kThreads) prune12_kernel(const uint4* __restrict__ W,
                                                           uint2* __restrict__ vals,
                                                           uint8_t* __restrict__ meta,
                                                           int64_t nchunks) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks; c += stride) {
    const uint4 w = __ldcs(W + c);
    uint32_t n0, n1;
    const uint32_t a = keep12(w.x, w.y, n0);
    const uint32_t b = keep12(w.z, w.w, n1);
    __stcs(vals + c, make_uint2(a, b));
    meta[c] = static_cast<uint8_t>(n0 | (n1 << 4));
  }
}

// Column j (0-3) of a quadruple stored as a kept pair `word` with nibble
// `nib`: the kept value at its position, +0 elsewhere.
__device__ __forceinline__ uint32_t quad_col(uint32_t word, uint32_t nib, uint32_t j) {
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  return j == i0 ? (word & 0xFFFFu) : (j == i1 ? (word >> 16) : 0u);
}

// A2 for 1:2: the transpose of a rows x cols 2:4-format matrix, pruned 1:2
// along the old rows.  Work item: 8 consecutive rows (octet h8) x one
// 16-column chunk c16 (16 B of values and 2 B of metadata per row).  Lanes
// take consecutive octets, the block's 8 warps adjacent chunks (their loads
// of a row share 128 B in L1); the 16 output rows a thread writes get 8 B
// of values (4 pairs of old rows) and one metadata byte at column octet h8,
// 256 B / 32 B contiguous per warp.
__global__ void __launch_bounds__(kThreads) double_prune12_kernel(const uint4* __restrict__ vals,
                                                                  const uint16_t* __restrict__ meta,
                                                                  uint2* __restrict__ t_vals,
                                                                  uint8_t* __restrict__ t_meta,
                                                                  int64_t rows, int64_t cols) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t n_h8 = rows / 8, n_c16 = cols / 16;
  const int64_t tiles_h = (n_h8 + 31) / 32, tiles_c = (n_c16 + 7) / 8;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  for (int64_t tile = blockIdx.x; tile < tiles_h * tiles_c; tile += gridDim.x) {
    const int64_t h8 = (tile % tiles_h) * 32 + lane;
    const int64_t c16 = (tile / tiles_h) * 8 + warp;
    if (h8 >= n_h8 || c16 >= n_c16) continue;
    uint4 pw[8];
    uint32_t m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t at = (8 * h8 + k) * n_c16 + c16;
      pw[k] = __ldg(vals + at);
      m[k] = __ldg(meta + at);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // quadruple q of the chunk: columns 4q .. 4q + 3
#pragma unroll
      for (uint32_t j = 0; j < 4; ++j) {
        uint32_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t word = q == 0 ? pw[k].x : q == 1 ? pw[k].y : q == 2 ? pw[k].z : pw[k].w;
          e[k] = quad_col(word, (m[k] >> (4 * q)) & 15u, j);
        }
        // old rows (2p, 2p + 1) form pair p; pairs 0-1 and 2-3 form the two
        // output quadruples of this octet
        uint32_t n0, n1;
        const uint32_t a = keep12(e[0] | (e[1] << 16), e[2] | (e[3] << 16), n0);
        const uint32_t b = keep12(e[4] | (e[5] << 16), e[6] | (e[7] << 16), n1);
        const int64_t i = 16 * c16 + 4 * q + j;  // output row = old column
        __stcs(t_vals + i * n_h8 + h8, make_uint2(a, b));
        t_meta[i * n_h8 + h8] = static_cast<uint8_t>(n0 | (n1 << 4));
      }
    }
  }
}

// ------------------------------------------------------------------ 2:8 ---

// The two largest of eight candidates e[0..7] (bf16 patterns) by magnitude,
// the lower index first on ties: keys (magnitude << 3) | (7 - index) are
// distinct, so a running top two decides.  Returns the packed values (lower
// index in the low half) and the byte i0 | i1 << 3.
__device__ __forceinline__ uint32_t top2_of_8(const uint32_t (&e)[8], uint32_t& byte) {
  uint32_t t1 = (key15(e[0]) << 3) | 7u, t2 = 0;
#pragma unroll
  for (uint32_t j = 1; j < 8; ++j) {
    const uint32_t k = (key15(e[j]) << 3) | (7u - j);
    const uint32_t nt2 = max(t2, min(t1, k));
    t1 = max(t1, k);
    t2 = nt2;
  }
  const uint32_t ia = 7u - (t1 & 7u), ib = 7u - (t2 & 7u);
  const uint32_t i0 = min(ia, ib), i1 = max(ia, ib);
  uint32_t v0 = 0, v1 = 0;
#pragma unroll
  for (uint32_t j = 0; j < 8; ++j) {
    v0 = j == i0 ? e[j] : v0;
    v1 = j == i1 ? e[j] : v1;
  }
  byte = i0 | (i1 << 3);
  return v0 | (v1 << 16);
}

// A1 for 2:8: one group of eight (16 B) per item -> 4 B of values, 1 byte.
__global__ void __launch_bounds__(kThreads) prune28_kernel(const uint4* __restrict__ W,
                                                           uint32_t* __restrict__ vals,
                                                           uint8_t* __restrict__ meta,
                                                           int64_t ngroups) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < ngroups; g += stride) {
    const uint4 w = __ldcs(W + g);
    const uint32_t e[8] = {w.x & 0xFFFFu, w.x >> 16, w.y & 0xFFFFu, w.y >> 16,
                           w.z & 0xFFFFu, w.z >> 16, w.w & 0xFFFFu, w.w >> 16};
    uint32_t byte;
    __stcs(vals + g, top2_of_8(e, byte));
    meta[g] = static_cast<uint8_t>(byte);
  }
}

// A2 for 2:8: the transpose of a rows x cols 2:8-format matrix, pruned 2:8
// along the old rows.  Work item: 8 consecutive rows (octet h8) x one group
// of 8 columns g (4 B of values and 1 byte per row).  Lanes take consecutive
// octets, the block's 8 warps adjacent groups (a row's loads share one
// 32 B sector); each of the 8 output rows (old columns 8g .. 8g + 7) gets
// 4 B of values and one byte at column octet h8, 128 B / 32 B contiguous
// per warp.
__global__ void __launch_bounds__(kThreads) double_prune28_kernel(const uint32_t* __restrict__ vals,
                                                                  const uint8_t* __restrict__ meta,
                                                                  uint32_t* __restrict__ t_vals,
                                                                  uint8_t* __restrict__ t_meta,
                                                                  int64_t rows, int64_t cols) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t n_h8 = rows / 8, n_g = cols / 8;
  const int64_t tiles_h = (n_h8 + 31) / 32, tiles_g = (n_g + 7) / 8;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  for (int64_t tile = blockIdx.x; tile < tiles_h * tiles_g; tile += gridDim.x) {
    const int64_t h8 = (tile % tiles_h) * 32 + lane;
    const int64_t g = (tile / tiles_h) * 8 + warp;
    if (h8 >= n_h8 || g >= n_g) continue;
    uint32_t w[8], a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t at = (8 * h8 + k) * n_g + g;
      w[k] = __ldg(vals + at);
      const uint32_t byte = __ldg(meta + at);
      a[k] = byte & 7u;
      b[k] = (byte >> 3) & 7u;
    }
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
      uint32_t e[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) e[k] = a[k] == c ? (w[k] & 0xFFFFu) : (b[k] == c ? (w[k] >> 16) : 0u);
      uint32_t byte;
      const uint32_t v = top2_of_8(e, byte);
      const int64_t i = 8 * g + c;  // output row = old column
      __stcs(t_vals + i * n_h8 + h8, v);
      t_meta[i * n_h8 + h8] = static_cast<uint8_t>(byte);
    }
  }
}

// One quadruple of the 2:4 form: kept positions (p < q) and their values
// packed as a word (p's in the low half), with the nibble p | q << 2.
__device__ __forceinline__ uint32_t quad24(uint32_t p, uint32_t vp, uint32_t q, uint32_t vq, uint32_t& nib) {
  nib = p | (q << 2);
  return vp | (vq << 16);
}

// The 2:4 form of a 2:8-format matrix: one group of eight per item -> two
// quadruples (8 B of values, one metadata byte).  A quadruple with both of
// the group's entries keeps them; with one, it adds its lowest other
// position (+0); with none, it keeps positions 0 and 1 (+0, +0).
__global__ void __launch_bounds__(kThreads) expand28_kernel(const uint32_t* __restrict__ vals,
                                                            const uint8_t* __restrict__ meta,
                                                            uint2* __restrict__ vals24,
                                                            uint8_t* __restrict__ meta24,
                                                            int64_t ngroups) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < ngroups; g += stride) {
    const uint32_t w = __ldcs(vals + g), byte = meta[g];
    const uint32_t i0 = byte & 7u, i1 = (byte >> 3) & 7u;
    const uint32_t va = w & 0xFFFFu, vb = w >> 16;
    uint32_t lo, hi, n0, n1;
    if (i1 < 4) {  // both in quadruple 0
      lo = quad24(i0, va, i1, vb, n0);
      hi = quad24(0, 0, 1, 0, n1);
    } else if (i0 >= 4) {  // both in quadruple 1
      lo = quad24(0, 0, 1, 0, n0);
      hi = quad24(i0 - 4, va, i1 - 4, vb, n1);
    } else {  // one in each: pad with the lowest other position
      const uint32_t p0 = i0 == 0 ? 1u : 0u, j1 = i1 - 4, p1 = j1 == 0 ? 1u : 0u;
      lo = p0 < i0 ? quad24(p0, 0, i0, va, n0) : quad24(i0, va, p0, 0, n0);
      hi = p1 < j1 ? quad24(p1, 0, j1, vb, n1) : quad24(j1, vb, p1, 0, n1);
    }
    __stcs(vals24 + g, make_uint2(lo, hi));
    meta24[g] = static_cast<uint8_t>(n0 | (n1 << 4));
  }
}

int64_t grid_for(int64_t items) {
  int64_t blocks = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return blocks < 1 ? 1 : (blocks > cap ? cap : blocks);
}

template <typename Kernel, typename... Args>
cudaError_t launch(Kernel kernel, int64_t blocks, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_prune12(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream) {
  const int64_t n = rows * cols / 8;
  if (n == 0) return cudaSuccess;
  return launch(prune12_kernel, grid_for(n), stream, static_cast<const uint4*>(W), static_cast<uint2*>(vals),
                meta, n);
}

cudaError_t launch_double_prune12(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* t_vals, uint8_t* t_meta, cudaStream_t stream) {
  const int64_t tiles = ((rows / 8 + 31) / 32) * ((cols / 16 + 7) / 8);
  if (tiles == 0) return cudaSuccess;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return launch(double_prune12_kernel, tiles < cap ? tiles : cap, stream, static_cast<const uint4*>(vals),
                reinterpret_cast<const uint16_t*>(meta), static_cast<uint2*>(t_vals), t_meta, rows, cols);
}

cudaError_t launch_prune28(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream) {
  const int64_t n = rows * cols / 8;
  if (n == 0) return cudaSuccess;
  return launch(prune28_kernel, grid_for(n), stream, static_cast<const uint4*>(W),
                static_cast<uint32_t*>(vals), meta, n);
}

cudaError_t launch_double_prune28(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* t_vals, uint8_t* t_meta, cudaStream_t stream) {
  const int64_t tiles = ((rows / 8 + 31) / 32) * ((cols / 8 + 7) / 8);
  if (tiles == 0) return cudaSuccess;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return launch(double_prune28_kernel, tiles < cap ? tiles : cap, stream, static_cast<const uint32_t*>(vals),
                meta, static_cast<uint32_t*>(t_vals), t_meta, rows, cols);
}

cudaError_t launch_expand28(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols, void* vals24,
                            uint8_t* meta24, cudaStream_t stream) {
  const int64_t n = rows * cols / 8;
  if (n == 0) return cudaSuccess;
  return launch(expand28_kernel, grid_for(n), stream, static_cast<const uint32_t*>(vals), meta,
                static_cast<uint2*>(vals24), meta24, n);
}

}  // namespace slope
