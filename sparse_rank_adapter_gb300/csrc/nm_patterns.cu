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
// 2:4 sparse tensor-core GEMMs take it as it is, and its double pruning is
// the 2:4 A2 kernels' data movement with a per-pair selection (prune.cu).
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

// ------------------------------------------------------------------ 2:8 ---

// Rank key of a candidate bf16 value v at index j of its group of eight:
// (|v| << 4) | ((7 - j) << 1) | sign.  Keys of one group are distinct and
// order by magnitude, then the lower index; the value is recovered from
// its key (value_of_key), so a running top two yields the kept values too.
__device__ __forceinline__ uint32_t key28(uint32_t v, uint32_t j) {
  return ((v & 0x7FFFu) << 4) | ((7u - j) << 1) | (v >> 15);
}
__device__ __forceinline__ uint32_t value_of_key(uint32_t k) { return ((k & 1u) << 15) | (k >> 4); }
__device__ __forceinline__ uint32_t index_of_key(uint32_t k) { return 7u - ((k >> 1) & 7u); }

// Running top two of keys (t1 > t2): insert k.
__device__ __forceinline__ void top2_insert(uint32_t& t1, uint32_t& t2, uint32_t k) {
  t2 = max(t2, min(t1, k));
  t1 = max(t1, k);
}

// The group's output from its top two keys: the two values in ascending
// index order (lower index in the low half) and the byte i0 | i1 << 3.
__device__ __forceinline__ uint32_t pack28(uint32_t t1, uint32_t t2, uint32_t& byte) {
  const uint32_t ia = index_of_key(t1), ib = index_of_key(t2);
  const bool a_first = ia < ib;
  const uint32_t lo = a_first ? t1 : t2, hi = a_first ? t2 : t1;
  byte = index_of_key(lo) | (index_of_key(hi) << 3);
  return value_of_key(lo) | (value_of_key(hi) << 16);
}

constexpr int kUnroll = 4;  // groups in flight per thread in the elementwise kernels

// A1 for 2:8: one group of eight (16 B) per item -> 4 B of values, 1 byte.
__global__ void __launch_bounds__(kThreads) prune28_kernel(const uint4* __restrict__ W,
                                                           uint32_t* __restrict__ vals,
                                                           uint8_t* __restrict__ meta,
                                                           int64_t ngroups) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < ngroups;
       base += stride * kUnroll) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (base + u * stride < ngroups) w[u] = __ldcs(W + base + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t g = base + u * stride;
      if (g >= ngroups) break;
      const uint32_t words[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
      uint32_t t1 = key28(words[0] & 0xFFFFu, 0), t2 = 0;
#pragma unroll
      for (uint32_t j = 1; j < 8; ++j) top2_insert(t1, t2, key28((words[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, j));
      uint32_t byte;
      __stcs(vals + g, pack28(t1, t2, byte));
      meta[g] = static_cast<uint8_t>(byte);
    }
  }
}

// A2 for 2:8 at any width (rows % 8 == 0, cols % 8 == 0): work item = 8
// consecutive rows (octet h8) x one group of 8 columns g (4 B of values and
// one byte per row), read straight from global memory.  Lanes take
// consecutive octets, the block's 8 warps adjacent groups (a row's loads
// share one 32 B sector); each of the 8 output rows (old columns 8g ..
// 8g + 7) gets 4 B of values and one byte at column octet h8.
__device__ __forceinline__ void transpose_prune28_group(const uint32_t (&w)[8], const uint32_t (&mb)[8],
                                                        int shift, int64_t g, int64_t h8, int64_t n_h8,
                                                        uint32_t* __restrict__ t_vals,
                                                        uint8_t* __restrict__ t_meta) {
  uint32_t klo[8], khi[8], a[8], b[8];
#pragma unroll
  for (uint32_t k = 0; k < 8; ++k) {
    const uint32_t byte = (mb[k] >> shift) & 0xFFu;
    a[k] = byte & 7u;
    b[k] = (byte >> 3) & 7u;
    klo[k] = key28(w[k] & 0xFFFFu, k);
    khi[k] = key28(w[k] >> 16, k);
  }
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c) {
    // candidate of old row k at column c: its kept value there, or +0
    uint32_t t1 = a[0] == c ? klo[0] : (b[0] == c ? khi[0] : key28(0, 0)), t2 = 0;
#pragma unroll
    for (uint32_t k = 1; k < 8; ++k) top2_insert(t1, t2, a[k] == c ? klo[k] : (b[k] == c ? khi[k] : key28(0, k)));
    uint32_t byte;
    const uint32_t v = pack28(t1, t2, byte);
    const int64_t i = 8 * g + c;  // output row = old column
    __stcs(t_vals + i * n_h8 + h8, v);
    t_meta[i * n_h8 + h8] = static_cast<uint8_t>(byte);
  }
}

__global__ void __launch_bounds__(kThreads) double_prune28_direct_kernel(const uint32_t* __restrict__ vals,
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
    uint32_t w[8], mb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t at = (8 * h8 + k) * n_g + g;
      w[k] = __ldg(vals + at);
      mb[k] = __ldg(meta + at);
    }
    transpose_prune28_group(w, mb, 0, g, h8, n_h8, t_vals, t_meta);
  }
}

// A2 for 2:8, cols % 256 == 0 (every row's segment of a tile is whole
// 16-byte pieces): tiles of 256 rows x 256 columns (32
// groups): the tile's rows (128 B of values, 32 B of metadata each) are
// copied into shared memory with whole-row, coalesced loads; then thread
// (lane o, warp G) takes row octet o and the four groups 4G .. 4G + 3, and
// writes, for each of their 32 columns (output rows), 4 B of values and one
// byte at column octet o, so a warp's stores to an output row are 128 B /
// 32 B contiguous.  Shared layout: value word (row, group g) at
// row·32 + (g ^ (row / 8 % 32)) and metadata word (row, G) at
// row·8 + (G ^ (row / 8 % 8)), which spreads the lanes of a read over the
// banks.
constexpr int kDp8Rows = 256, kDp8Groups = 32;
constexpr int kDp8Pieces = kDp8Rows * 10 / kThreads;  // 16 B pieces per thread and tile (8 of values, 2 of metadata per row)

__global__ void __launch_bounds__(kThreads, 2) double_prune28_kernel(const uint32_t* __restrict__ vals,
                                                                     const uint8_t* __restrict__ meta,
                                                                     uint32_t* __restrict__ t_vals,
                                                                     uint8_t* __restrict__ t_meta,
                                                                     int64_t rows, int64_t cols) {
  __shared__ uint32_t sv[kDp8Rows * kDp8Groups];      // 32 KB
  __shared__ uint32_t sm[kDp8Rows * kDp8Groups / 4];  // 8 KB
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t n_g = cols / 8, n_h8 = rows / 8;
  const int64_t tiles_h = (rows + kDp8Rows - 1) / kDp8Rows, tiles = tiles_h * (n_g / kDp8Groups);
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  // piece u = threadIdx.x + kThreads·i of a tile: row u / 10, piece u % 10
  // (0-7: four value words each, 8-9: sixteen metadata bytes each)
  auto fetch = [&](int64_t tile, uint4 (&x)[kDp8Pieces]) {
    const int64_t row0 = (tile % tiles_h) * kDp8Rows, g0 = (tile / tiles_h) * kDp8Groups;
#pragma unroll
    for (int i = 0; i < kDp8Pieces; ++i) {
      const int u = static_cast<int>(threadIdx.x) + kThreads * i, piece = u % 10;
      const int64_t row = row0 + u / 10;
      x[i] = make_uint4(0, 0, 0, 0);
      if (row < rows)
        x[i] = piece < 8 ? __ldcs(reinterpret_cast<const uint4*>(vals + row * n_g + g0 + 4 * piece))
                         : __ldcs(reinterpret_cast<const uint4*>(meta + row * n_g + g0 + 16 * (piece - 8)));
    }
  };
  uint4 x[kDp8Pieces];
  int64_t tile = blockIdx.x;
  if (tile < tiles) fetch(tile, x);
  for (; tile < tiles; tile += gridDim.x) {
    const int64_t row0 = (tile % tiles_h) * kDp8Rows, g0 = (tile / tiles_h) * kDp8Groups;
    __syncthreads();  // the previous tile's reads of shared memory are done
#pragma unroll
    for (int i = 0; i < kDp8Pieces; ++i) {
      const int u = static_cast<int>(threadIdx.x) + kThreads * i, r = u / 10, piece = u % 10;
      if (piece < 8) {
        const uint32_t sw = static_cast<uint32_t>(r >> 3) & 31u;
        uint32_t* d = sv + r * kDp8Groups;
        d[(4 * piece + 0) ^ sw] = x[i].x;
        d[(4 * piece + 1) ^ sw] = x[i].y;
        d[(4 * piece + 2) ^ sw] = x[i].z;
        d[(4 * piece + 3) ^ sw] = x[i].w;
      } else {
        const uint32_t sw = static_cast<uint32_t>(r >> 3) & 7u, w0 = 4 * (piece - 8);
        uint32_t* d = sm + r * (kDp8Groups / 4);
        d[(w0 + 0) ^ sw] = x[i].x;
        d[(w0 + 1) ^ sw] = x[i].y;
        d[(w0 + 2) ^ sw] = x[i].z;
        d[(w0 + 3) ^ sw] = x[i].w;
      }
    }
    __syncthreads();
    // the next tile's pieces are in flight while this one is pruned
    if (tile + gridDim.x < tiles) fetch(tile + gridDim.x, x);
    const int64_t h8 = row0 / 8 + lane;
    if (h8 >= n_h8) continue;
    uint32_t w[8][4], mb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = 8 * static_cast<int>(lane) + k;
#pragma unroll
      for (int j = 0; j < 4; ++j) w[k][j] = sv[r * kDp8Groups + ((4 * warp + j) ^ lane)];
      mb[k] = sm[r * (kDp8Groups / 4) + (warp ^ (lane & 7u))];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // group 4·warp + j of the tile
      uint32_t wj[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) wj[k] = w[k][j];
      transpose_prune28_group(wj, mb, 8 * j, g0 + 4 * warp + j, h8, n_h8, t_vals, t_meta);
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
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < ngroups;
       base += stride * kUnroll) {
    uint32_t wv[kUnroll], mv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (base + u * stride < ngroups) {
        wv[u] = __ldcs(vals + base + u * stride);
        mv[u] = meta[base + u * stride];
      }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t g = base + u * stride;
      if (g >= ngroups) break;
      const uint32_t w = wv[u], byte = mv[u];
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

cudaError_t launch_prune28(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream) {
  const int64_t n = rows * cols / 8;
  if (n == 0) return cudaSuccess;
  return launch(prune28_kernel, grid_for(n), stream, static_cast<const uint4*>(W),
                static_cast<uint32_t*>(vals), meta, n);
}

cudaError_t launch_double_prune28(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* t_vals, uint8_t* t_meta, cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 256 == 0) {  // whole 16-byte row pieces: the staged kernel
    const int64_t tiles = ((rows + kDp8Rows - 1) / kDp8Rows) * (cols / 8 / kDp8Groups);
    const int64_t cap = static_cast<int64_t>(sm_count()) * 2;
    return launch(double_prune28_kernel, tiles < cap ? tiles : cap, stream, static_cast<const uint32_t*>(vals),
                  meta, static_cast<uint32_t*>(t_vals), t_meta, rows, cols);
  }
  const int64_t tiles = ((rows / 8 + 31) / 32) * ((cols / 8 + 7) / 8);
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return launch(double_prune28_direct_kernel, tiles < cap ? tiles : cap, stream,
                static_cast<const uint32_t*>(vals), meta, static_cast<uint32_t*>(t_vals), t_meta, rows, cols);
}

cudaError_t launch_expand28(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols, void* vals24,
                            uint8_t* meta24, cudaStream_t stream) {
  const int64_t n = rows * cols / 8;
  if (n == 0) return cudaSuccess;
  return launch(expand28_kernel, grid_for(n), stream, static_cast<const uint32_t*>(vals), meta,
                static_cast<uint2*>(vals24), meta24, n);
}

}  // namespace slope
