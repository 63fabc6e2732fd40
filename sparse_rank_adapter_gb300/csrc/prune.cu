// prune.cu — the two memory-bound kernels of the path.
//
//   prune24_kernel            2:4 magnitude prune-and-compress of W (A1).
//   double_prune24_staged_kernel / double_prune24_kernel
//                             transpose of the pruned W, pruned 2:4 again
//                             along the old out dimension (A2); the staged
//                             kernel (cols % 128 == 0) moves its tiles
//                             through shared memory, the other reads global
//                             memory directly and takes any legal shape.
//   prune_double24_kernel     A1 and A2 from one read of W (cols % 128 == 0).
//   The two A2 kernels also prune the transpose 1:2 (one entry per row pair)
//   for the 1:2 pattern, whose matrices are written in the 2:4 format.
//
// Source: "SLoPe: Double-Pruned Sparse Plus Lazy Low-Rank Adapter Pretraining
// of LLMs", §1 and §2.1 (N:M pruning of the weight, then of its transpose)
// and §2.3 / App. K (compressed formats for both).  Ranking uses the exact
// magnitude key (bits & 0x7FFF) with ties to the lower index; the
// compressed format is the one slope.h documents.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "slope_internal.h"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

// ---------------------------------------------------------------- A2 ------

constexpr int kDpThreads = 256;  // direct kernel: 8 warps = 8 column chunks per tile

// Byte-permute selectors that expand a compressed group (kept pair: lower
// column in bytes 0-1, upper in 2-3 of one word; the permute's second word
// is zero) into its four columns, two per output word: .x builds columns
// 0-1, .y columns 2-3.  Indexed by the metadata nibble.
__device__ __forceinline__ uint2 expand_selectors(uint32_t nib) {
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  uint32_t sel = 0;
#pragma unroll
  for (uint32_t pos = 0; pos < 4; ++pos) {
    const uint32_t src = pos == i0 ? 0u : (pos == i1 ? 2u : 4u);  // 4: a zero byte
    sel |= (src | ((src + 1) << 4)) << (8 * pos);
  }
  return make_uint2(sel & 0xFFFFu, sel >> 16);
}

// Output of a transposed group from the in-quadruple codes (3 - row) of its
// two winners, first and second by rank: the low 16 bits are the permute
// selector that packs the kept pair in ascending row order (candidate k
// sits in bytes 2k, 2k+1 of the two candidate words); bits 16 + nib_shift
// and up hold the metadata nibble i0 | i1 << 2.
__device__ __forceinline__ uint32_t output_entry(uint32_t code_first, uint32_t code_second,
                                                 uint32_t nib_shift) {
  const uint32_t j1 = 3u - code_first, j2 = 3u - code_second;
  const uint32_t lo = j1 < j2 ? j1 : j2, hi = j1 < j2 ? j2 : j1;
  const uint32_t sel = (2 * lo) | ((2 * lo + 1) << 4) | ((2 * hi) << 8) | ((2 * hi + 1) << 12);
  return sel | ((lo | (hi << 2)) << (16 + nib_shift));
}

// Byte-permute selector that picks a group's two entries at the positions a
// metadata nibble names (i0 | i1 << 2) out of its four (two words, two
// entries each), in the order of the nibble's fields.
__device__ __forceinline__ uint32_t gather_selector(uint32_t nib) {
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  return (2 * i0) | ((2 * i0 + 1) << 4) | ((2 * i1) << 8) | ((2 * i1 + 1) << 12);
}

struct DpTables {
  uint2 expand[16];     // by metadata nibble
  uint32_t out[2][16];  // [upper / lower quadruple of the octet][code_first * 4 + code_second]
  uint32_t gather[16];  // by metadata nibble
};

__device__ __forceinline__ void fill_tables(DpTables& t) {
  if (threadIdx.x < 16) t.expand[threadIdx.x] = expand_selectors(threadIdx.x);
  if (threadIdx.x < 32) {
    const uint32_t g = threadIdx.x >> 4, idx = threadIdx.x & 15;
    t.out[g][idx] = output_entry(idx >> 2, idx & 3, 4 * g);
  }
  if (threadIdx.x >= 32 && threadIdx.x < 48) t.gather[threadIdx.x - 32] = gather_selector(threadIdx.x - 32);
}

// Top two of the four candidates of a transposed group, packed as two rows
// per word (w01: rows 0 and 1, w23: rows 2 and 3, lower row in the low
// half).  Rank key of row k: magnitude in bits 17-31, 3 - k in bits 15-16,
// zeros below: larger magnitude first, then the lower row.  Multiplying a
// word by 2^17 moves its low half's magnitude to the top and drops the sign
// and the high half; the high half is shifted by one and masked.  Returns
// the table entry of the two winners.  `k17` = 2^17 and `k1` = 2 come in at
// run time: as unknown factors they stay integer multiply-adds, on a pipe
// this kernel otherwise leaves idle, instead of becoming shifts on the logic
// pipe, which is its bottleneck.
__device__ __forceinline__ uint32_t top2_entry(uint32_t w01, uint32_t w23, const uint32_t* out,
                                               uint32_t k17, uint32_t k1) {
  const uint32_t c0 = w01 * k17 + 0x18000u;
  const uint32_t c1 = ((w01 * k1) & 0xFFFE0000u) | 0x10000u;
  const uint32_t c2 = w23 * k17 + 0x08000u;
  const uint32_t c3 = (w23 * k1) & 0xFFFE0000u;
  const uint32_t a = max(c0, c1), b = min(c0, c1);
  const uint32_t c = max(c2, c3), d = min(c2, c3);
  const uint32_t first = max(a, c);
  const uint32_t second = max(min(a, c), max(b, d));
  // byte offset 16·code_first + 4·code_second; bits 0-14 of the keys are
  // zero, so the +1 in each multiplier never reaches the bits kept
  const uint32_t off = (__umulhi(first, 0x200001u) & 0x30u) | (__umulhi(second, 0x80001u) & 0x0Cu);
  return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(out) + off);
}

// The 1:2 counterpart of top2_entry: each of the transposed group's two
// row pairs (w01: rows 0 and 1, w23: rows 2 and 3, lower row in the low
// half) keeps its entry of larger magnitude, the lower row on ties.  Same
// encoding: the permute selector that packs the two kept entries in the low
// 16 bits (below 0x8000), the nibble i0 | i1 << 2 (i0 in {0, 1}, i1 in
// {2, 3}) at bit 16 + nib_shift.
__device__ __forceinline__ uint32_t pair12_entry(uint32_t w01, uint32_t w23, uint32_t nib_shift) {
  const uint32_t p0 = ((w01 >> 16) & 0x7FFFu) > (w01 & 0x7FFFu) ? 1u : 0u;
  const uint32_t p1 = ((w23 >> 16) & 0x7FFFu) > (w23 & 0x7FFFu) ? 1u : 0u;
  const uint32_t sel = (p0 ? 0x32u : 0x10u) | ((p1 ? 0x76u : 0x54u) << 8);
  return sel | ((p0 | ((2u + p1) << 2)) << (16 + nib_shift));
}

// ---------------------------------------------------------------- A1 ------
// One 16-byte chunk = 8 consecutive weights of a row = 2 groups -> 8 bytes of
// kept values and one metadata byte.  Row-major contiguity makes chunk c of
// the flattened matrix map to vals[c] (uint2) and meta[c]; every warp access
// is fully coalesced.  A row group of four bf16 is two words with two
// entries each, the layout top2_entry takes (it was written for a group of
// the transpose, four rows packed two per word), so A1 ranks with the same
// multiply-add keys and table: magnitude first, the lower column on ties.

constexpr int kPruneThreads = 256;
constexpr int kPruneUnroll = 4;

__global__ void __launch_bounds__(kPruneThreads) prune24_kernel(const uint4* __restrict__ W,
                                                                uint2* __restrict__ vals,
                                                                uint8_t* __restrict__ meta,
                                                                int64_t nchunks, uint32_t k17) {
  __shared__ DpTables tab;
  fill_tables(tab);
  __syncthreads();
  grid_dependency_wait();
  allow_dependents_launch();
  const uint32_t k1 = k17 >> 16;
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
        const uint32_t ea = top2_entry(w[u].x, w[u].y, tab.out[0], k17, k1);
        const uint32_t eb = top2_entry(w[u].z, w[u].w, tab.out[1], k17, k1);
        __stcs(vals + c, make_uint2(__byte_perm(w[u].x, w[u].y, ea), __byte_perm(w[u].z, w[u].w, eb)));
        // the selectors stay below 0x8000: the sum carries nothing into the nibbles
        meta[c] = static_cast<uint8_t>((ea + eb) >> 16);
      }
    }
  }
}

// Work item: 8 consecutive rows (one "octet" h8) x 4·Q consecutive columns
// (groups q0 .. q0 + Q - 1 of chunk c16) of the rows x cols pruned weight,
// given as each row's kept-pair words pw[k][q] of those groups and its
// metadata m[k] shifted so that group q0 is the low nibble.  It expands each
// row's groups with byte permutes (pruned positions become +0) and, for each
// column, prunes the two row-quadruples along the old row dimension: 4 kept
// values (8 B) and one metadata byte for row i of the transposed output, at
// column octet h8.  Lanes of a warp take consecutive octets of the same
// chunk, so each output row segment a warp writes is 256 B (values) / 32 B
// (metadata) contiguous.
// FROZEN: the transposed metadata is an input (the column-wise mask is
// kept): each transposed group takes the two positions its byte of
// `t_meta_in` names, through the byte-permute selector of the nibble, and
// no metadata is written.
// P12: the transposed groups are pruned 1:2 (one entry per row pair)
// instead of 2:4; the input format, the output format and the data
// movement are the same.
template <int Q, bool FROZEN = false, bool P12 = false>
__device__ __forceinline__ void transpose_prune_octet(const uint32_t (&pw)[8][Q], const uint32_t (&m)[8],
                                                      const DpTables& tab,
                                                      uint2* __restrict__ t_vals,
                                                      uint8_t* __restrict__ t_meta,
                                                      int64_t out_stride, uint32_t h8,
                                                      uint32_t c16, uint32_t k17, int q0,
                                                      const uint8_t* __restrict__ t_meta_in = nullptr) {
  const uint32_t k1 = k17 >> 16, k8 = k17 >> 14;
  const int64_t first = (16 * static_cast<int64_t>(c16) + 4 * q0) * out_stride + h8;
  uint2* tv = t_vals + first;
  uint8_t* tm = FROZEN ? nullptr : t_meta + first;
  // FROZEN: the given bytes of all this thread's output rows, loaded up
  // front so that their latency overlaps the expansion below
  uint32_t dmv[Q][4];
  if constexpr (FROZEN) {
    const uint8_t* tmi = t_meta_in + first;
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) dmv[q][j] = tmi[(4 * q + j) * out_stride];
  }
#pragma unroll
  for (int q = 0; q < Q; ++q) {  // group of 4 columns
    uint32_t e0[8], e1[8];        // row k, columns 0-1 / 2-3 of the group
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      // byte offset 8·nibble: the shift comes from a multiply-high, whose
      // +1 term only adds below bit 3
      const uint32_t m8 = (q == 0) ? m[k] * k8 : __umulhi(m[k], (1u << (35 - 4 * q)) + 1u);
      const uint2 sel = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(tab.expand) + (m8 & 0x78u));
      e0[k] = __byte_perm(pw[k][q], 0u, sel.x);
      e1[k] = __byte_perm(pw[k][q], 0u, sel.y);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t* e = (j < 2) ? e0 : e1;
      const uint32_t pick = (j & 1) ? 0x7632u : 0x5410u;  // high or low halves of two words
      const uint32_t a01 = __byte_perm(e[0], e[1], pick), a23 = __byte_perm(e[2], e[3], pick);
      const uint32_t b01 = __byte_perm(e[4], e[5], pick), b23 = __byte_perm(e[6], e[7], pick);
      const int64_t i = 4 * q + j;
      uint32_t ea, eb;
      if constexpr (FROZEN) {
        const uint32_t dm = dmv[q][j];  // low nibble: rows 0-3 of the octet
        ea = tab.gather[dm & 15u];
        eb = tab.gather[dm >> 4];
      } else if constexpr (P12) {
        ea = pair12_entry(a01, a23, 0);
        eb = pair12_entry(b01, b23, 4);
      } else {
        ea = top2_entry(a01, a23, tab.out[0], k17, k1);
        eb = top2_entry(b01, b23, tab.out[1], k17, k1);
      }
      __stcs(tv + i * out_stride, make_uint2(__byte_perm(a01, a23, ea), __byte_perm(b01, b23, eb)));
      // the selectors stay below 0x8000, so the sum carries nothing into the nibbles
      if constexpr (!FROZEN) tm[i * out_stride] = static_cast<uint8_t>((ea + eb) >> 16);
    }
  }
}

// Any shape (rows % 8 == 0, cols % 16 == 0): each thread loads its octet's
// rows straight from global memory; the eight warps of a block take
// adjacent chunks, whose loads share sectors in L1.
template <bool FROZEN, bool P12 = false>
__global__ void __launch_bounds__(kDpThreads) double_prune24_kernel(
    const uint4* __restrict__ vals, const uint16_t* __restrict__ meta, uint2* __restrict__ t_vals,
    uint8_t* __restrict__ t_meta, int64_t rows, int64_t cols, uint32_t k17,
    const uint8_t* __restrict__ t_meta_in) {
  __shared__ DpTables tab;
  fill_tables(tab);
  __syncthreads();
  grid_dependency_wait();
  allow_dependents_launch();
  const uint32_t n_h8 = static_cast<uint32_t>(rows / 8), n_c16 = static_cast<uint32_t>(cols / 16);
  const uint32_t tiles_h = (n_h8 + 31) / 32, tiles_c = (n_c16 + 7) / 8;
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (uint32_t tile = blockIdx.x; tile < tiles_h * tiles_c; tile += gridDim.x) {
    const uint32_t h8 = (tile % tiles_h) * 32 + lane;
    const uint32_t c16 = (tile / tiles_h) * 8 + warp;
    if (h8 >= n_h8 || c16 >= n_c16) continue;
    uint32_t pw[8][4];
    uint32_t m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t at = (static_cast<int64_t>(8) * h8 + k) * n_c16 + c16;
      const uint4 v = __ldg(vals + at);
      pw[k][0] = v.x; pw[k][1] = v.y; pw[k][2] = v.z; pw[k][3] = v.w;
      m[k] = __ldg(meta + at);
    }
    transpose_prune_octet<4, FROZEN, P12>(pw, m, tab, t_vals, t_meta, rows / 8, h8, c16, k17, 0, t_meta_in);
  }
}

// cols % 128 == 0: tiles of 256 rows x 16·CH columns staged through shared
// memory.  Global reads are whole row segments (16·CH bytes of values,
// 2·CH bytes of metadata per row) copied with cp.async into a layout where
// the per-thread reads of the compute phase are free of bank conflicts:
// values of row 8·o + k, chunk c at k·plane + o·16·CH + 16·(c ^ f(o)) with
// f(o) = (o / (8 / CH)) % CH, so any 8 consecutive lanes (octets o) reading
// chunk c hit 8 different 16 B bank groups; metadata of that row at
// k·(32·16) + o·16 + 2·c.  Two stages: the copies of the next tile are in
// flight while the current one is pruned.
template <int CH>
__device__ __forceinline__ uint32_t swz(uint32_t o) { return (o / (8 / CH)) % CH; }

// QS threads share an octet and chunk, each taking 4 / QS groups of 4
// columns: for small weights (narrow tiles), shorter per-thread work.
template <int CH, int QS = 1>
struct DpStaged {
  static constexpr int kThreads = 32 * CH * QS;
  static constexpr int kValPitch = 16 * CH;
  static constexpr int kValPlane = 32 * kValPitch;
  static constexpr int kValBytes = 8 * kValPlane;
  static constexpr int kMetaBytes = 256 * 16;
  static constexpr int kStage = kValBytes + kMetaBytes;
  static constexpr int kSmem = 2 * kStage;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

template <int CH, int QS, bool FROZEN, bool P12 = false>
__global__ void __launch_bounds__(32 * CH * QS) double_prune24_staged_kernel(
    const uint8_t* __restrict__ vals, const uint8_t* __restrict__ meta, uint2* __restrict__ t_vals,
    uint8_t* __restrict__ t_meta, int64_t rows, int64_t cols, uint32_t k17,
    const uint8_t* __restrict__ t_meta_in) {
  using C = DpStaged<CH, QS>;
  constexpr int kQ = 4 / QS;  // groups of 4 columns per thread
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ DpTables tab;
  fill_tables(tab);
  const uint32_t n_h8 = static_cast<uint32_t>(rows / 8);
  const uint32_t tiles_h = (static_cast<uint32_t>(rows) + 255) / 256;
  const uint32_t tiles_c = static_cast<uint32_t>(cols / (16 * CH));
  const uint32_t lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) % CH;  // warp: the chunk
  const int q0 = static_cast<int>(threadIdx.x >> 5) / CH * kQ;               // first column group
  const int64_t val_pitch = cols, meta_pitch = cols / 8;  // bytes per input row
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));

  auto issue = [&](uint32_t th, uint32_t tc, int stage) {
    const uint32_t row0 = th * 256, ch0 = tc * CH;
    const uint32_t st = sbase + stage * C::kStage;
#pragma unroll
    for (int i = 0; i < 8 / QS; ++i) {  // 256 rows x CH chunks of 16 B values
      const uint32_t u = threadIdx.x + i * C::kThreads;
      const uint32_t r = u / CH, c = u % CH;
      if (row0 + r < rows)
        cp_async16(st + (r & 7) * C::kValPlane + (r >> 3) * C::kValPitch + 16 * (c ^ swz<CH>(r >> 3)),
                   vals + (row0 + r) * val_pitch + 16 * (ch0 + c));
    }
    // One 16 B piece of metadata per row, holding the tile's 2·CH bytes
    // (and, for CH < 8, neighbouring bytes that are never read).
    for (uint32_t r = threadIdx.x; r < 256; r += C::kThreads)
      if (row0 + r < rows) {
        const int64_t off = (row0 + r) * meta_pitch + 2 * ch0;
        cp_async16(st + C::kValBytes + (r & 7) * 512 + (r >> 3) * 16, meta + (off & ~int64_t(15)));
      }
  };

  // tile t covers row tile t % tiles_h and chunk tile t / tiles_h; the
  // (row, chunk) pair of the next tile is stepped without dividing
  const uint32_t step_c = gridDim.x / tiles_h, step_h = gridDim.x % tiles_h;
  auto advance = [&](uint32_t& th, uint32_t& tc) {
    th += step_h;
    tc += step_c;
    if (th >= tiles_h) { th -= tiles_h; ++tc; }
  };
  uint32_t th = blockIdx.x % tiles_h, tc = blockIdx.x / tiles_h;
  grid_dependency_wait();
  allow_dependents_launch();
  if (tc < tiles_c) issue(th, tc, 0);
  cp_async_commit();
  int stage = 0;
  for (; tc < tiles_c; stage ^= 1) {
    uint32_t nh = th, nc = tc;
    advance(nh, nc);
    if (nc < tiles_c) issue(nh, nc, stage ^ 1);
    cp_async_commit();
    cp_async_wait_1();
    __syncthreads();
    const uint32_t h8 = th * 32 + lane;
    const uint32_t ch0 = tc * CH;
    if (h8 < n_h8) {
      const uint8_t* st = smem + stage * C::kStage;
      // offset of this tile's metadata inside the 16 B piece that was copied
      const uint32_t moff = static_cast<uint32_t>((2 * ch0) & 15);
      uint32_t pw[8][kQ];
      uint32_t m[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint8_t* row = st + k * C::kValPlane + lane * C::kValPitch + 16 * (warp ^ swz<CH>(lane));
        if constexpr (kQ == 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(row);
          pw[k][0] = v.x; pw[k][1] = v.y; pw[k][2] = v.z; pw[k][3] = v.w;
        } else {
#pragma unroll
          for (int q = 0; q < kQ; ++q) pw[k][q] = *reinterpret_cast<const uint32_t*>(row + 4 * (q0 + q));
        }
        m[k] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(st + C::kValBytes + k * 512 +
                                                                          lane * 16 + moff + 2 * warp)) >> (4 * q0);
      }
      transpose_prune_octet<kQ, FROZEN, P12>(pw, m, tab, t_vals, t_meta, rows / 8, h8, ch0 + warp, k17, q0,
                                             t_meta_in);
    }
    __syncthreads();
    th = nh;
    tc = nc;
  }
}

// ------------------------------------------------------------ A1 + A2 ------
// Both compressed formats from one read of W.  Tiles and the compressed
// shared-memory layout are the staged A2 kernel's (256 rows x 16·CH
// columns).  The tile's rows of W are copied into shared memory with
// cp.async (row-major, 32·CH bytes a row); the copy of the next tile runs
// while the current one is double-pruned.  Phase 1: lanes take consecutive
// 16 B chunks (8 weights = 2 groups) of a row.  A row group of four bf16 is
// two words with two entries each, the same layout as a transposed group,
// so top2_entry ranks it too (magnitude key, lower column on ties).  The
// kept pairs and nibbles go to global memory (A1's output, coalesced) and
// into the compressed layout in shared memory.  Phase 2 is the staged A2
// kernel's compute step on that tile.
// GIVEN: the row mask is an input (the weight is re-compressed at the
// positions its metadata names instead of selecting them): the tile's
// metadata bytes are staged beside W, phase 1 gathers with the byte-permute
// selector of each nibble and writes no metadata.
template <int CH, int QS, bool GIVEN = false>
struct FusedCfg {
  using D = DpStaged<CH, QS>;
  static constexpr int kRawPitch = 32 * CH;          // bytes of one tile row of W
  static constexpr int kRawBytes = 256 * kRawPitch;
  static constexpr int kRawMeta = GIVEN ? 256 * 16 : 0;  // a 16 B piece of each row's metadata
  static constexpr int kSmem = kRawBytes + kRawMeta + D::kStage;
  static constexpr int kMinBlocks = CH == 8 ? 2 : 3;
};

template <int CH, int QS, bool GIVEN, bool FROZEN>
__global__ void __launch_bounds__(32 * CH * QS, (FusedCfg<CH, QS, GIVEN>::kMinBlocks)) prune_double24_kernel(
    const uint4* __restrict__ W, const uint8_t* __restrict__ meta_in, uint2* __restrict__ vals,
    uint8_t* __restrict__ meta, uint2* __restrict__ t_vals, uint8_t* __restrict__ t_meta, int64_t rows,
    int64_t cols, uint32_t k17, const uint8_t* __restrict__ t_meta_in) {
  using C = DpStaged<CH, QS>;
  using F = FusedCfg<CH, QS, GIVEN>;
  constexpr int kQ = 4 / QS;                     // groups of 4 columns per thread in phase 2
  constexpr int kRowChunks = 2 * CH;             // 8-column chunks per tile row
  constexpr int kItems = 256 * kRowChunks / C::kThreads;  // chunks per thread in phase 1
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ DpTables tab;
  uint8_t* raw = smem;                // the tile's rows of W
  uint8_t* rawm = smem + F::kRawBytes;  // GIVEN: their metadata, 16 B per row
  uint8_t* st = smem + F::kRawBytes + F::kRawMeta;  // the compressed tile, A2's staged layout
  fill_tables(tab);
  const uint32_t k1 = k17 >> 16;
  const uint32_t n_h8 = static_cast<uint32_t>(rows / 8);
  const uint32_t tiles_h = (static_cast<uint32_t>(rows) + 255) / 256;
  const uint32_t tiles_c = static_cast<uint32_t>(cols / (16 * CH));
  const uint32_t lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) % CH;
  const int q0 = static_cast<int>(threadIdx.x >> 5) / CH * kQ;
  const int64_t row_chunks = cols / 8;  // 8-column chunks per row of W
  const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(raw));
  const uint32_t rawm_s = static_cast<uint32_t>(__cvta_generic_to_shared(rawm));

  auto issue = [&](uint32_t th, uint32_t tc) {
    const uint32_t row0 = th * 256;
    const int64_t chunk0 = static_cast<int64_t>(tc) * kRowChunks;
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const uint32_t i = threadIdx.x + it * C::kThreads;
      const uint32_t r = i / kRowChunks, cc = i % kRowChunks;
      if (row0 + r < rows) cp_async16(raw_s + r * F::kRawPitch + 16 * cc, W + (row0 + r) * row_chunks + chunk0 + cc);
    }
    if constexpr (GIVEN) {
      for (uint32_t r = threadIdx.x; r < 256; r += C::kThreads)
        if (row0 + r < rows)
          cp_async16(rawm_s + r * 16, meta_in + (((row0 + r) * row_chunks + chunk0) & ~int64_t(15)));
    }
    cp_async_commit();
  };

  const uint32_t step_c = gridDim.x / tiles_h, step_h = gridDim.x % tiles_h;
  uint32_t th = blockIdx.x % tiles_h, tc = blockIdx.x / tiles_h;
  grid_dependency_wait();
  allow_dependents_launch();
  if (tc < tiles_c) issue(th, tc);
  while (tc < tiles_c) {
    cp_async_wait_all();
    __syncthreads();  // the tile's W is in; every thread is done with the last tile
    const uint32_t row0 = th * 256;
    const int64_t chunk0 = static_cast<int64_t>(tc) * kRowChunks;
#pragma unroll 4
    for (int it = 0; it < kItems; ++it) {
      const uint32_t i = threadIdx.x + it * C::kThreads;
      const uint32_t r = i / kRowChunks, cc = i % kRowChunks;
      if (row0 + r < rows) {
        const uint4 w = *reinterpret_cast<const uint4*>(raw + r * F::kRawPitch + 16 * cc);
        uint2 kept;
        uint8_t nib;
        if constexpr (GIVEN) {
          // the chunk's metadata byte: rows hold cols / 8 bytes, a multiple
          // of 16, so the tile's bytes sit at chunk0 % 16 in each row's piece
          nib = rawm[r * 16 + (static_cast<uint32_t>(chunk0) & 15u) + cc];
          kept = make_uint2(__byte_perm(w.x, w.y, tab.gather[nib & 15u]), __byte_perm(w.z, w.w, tab.gather[nib >> 4]));
        } else {
          const uint32_t ea = top2_entry(w.x, w.y, tab.out[0], k17, k1);
          const uint32_t eb = top2_entry(w.z, w.w, tab.out[1], k17, k1);
          kept = make_uint2(__byte_perm(w.x, w.y, ea), __byte_perm(w.z, w.w, eb));
          nib = static_cast<uint8_t>((ea + eb) >> 16);
        }
        const int64_t at = (row0 + r) * row_chunks + chunk0 + cc;
        __stcs(vals + at, kept);
        if constexpr (!GIVEN) meta[at] = nib;
        const uint32_t o = r >> 3, c = cc >> 1, h = cc & 1;
        *reinterpret_cast<uint2*>(st + (r & 7) * C::kValPlane + o * C::kValPitch +
                                  16 * (c ^ swz<CH>(o)) + 8 * h) = kept;
        st[C::kValBytes + (r & 7) * 512 + o * 16 + 2 * c + h] = nib;
      }
    }
    __syncthreads();  // compressed tile complete; W's buffer is free
    uint32_t nh = th + step_h, nc = tc + step_c;
    if (nh >= tiles_h) { nh -= tiles_h; ++nc; }
    if (nc < tiles_c) issue(nh, nc);
    const uint32_t h8 = th * 32 + lane;
    if (h8 < n_h8) {
      uint32_t pw[8][kQ];
      uint32_t m[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint8_t* row = st + k * C::kValPlane + lane * C::kValPitch + 16 * (warp ^ swz<CH>(lane));
        if constexpr (kQ == 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(row);
          pw[k][0] = v.x; pw[k][1] = v.y; pw[k][2] = v.z; pw[k][3] = v.w;
        } else {
#pragma unroll
          for (int q = 0; q < kQ; ++q) pw[k][q] = *reinterpret_cast<const uint32_t*>(row + 4 * (q0 + q));
        }
        m[k] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(st + C::kValBytes + k * 512 +
                                                                          lane * 16 + 2 * warp)) >> (4 * q0);
      }
      transpose_prune_octet<kQ, FROZEN>(pw, m, tab, t_vals, t_meta, rows / 8, h8, tc * CH + warp, k17, q0,
                                        t_meta_in);
    }
    th = nh;
    tc = nc;
  }
}

// ------------------------------------------------ optimizer side ---------
// Re-compression of an updated weight at a kept mask (any width with
// cols % 8 == 0): one 16-byte chunk = 8 weights = 2 groups and its metadata
// byte in, the two kept pairs out; coalesced like the prune kernel.
__global__ void __launch_bounds__(kPruneThreads) gather24_kernel(const uint4* __restrict__ W,
                                                                 const uint8_t* __restrict__ meta,
                                                                 uint2* __restrict__ vals,
                                                                 int64_t nchunks) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks; c += stride) {
    const uint4 w = __ldcs(W + c);
    const uint32_t nib = meta[c];
    __stcs(vals + c, make_uint2(__byte_perm(w.x, w.y, gather_selector(nib & 15u)),
                                __byte_perm(w.z, w.w, gather_selector(nib >> 4))));
  }
}

// beta·A + gamma·B on the compressed values of two matrices that share a 2:4
// pattern: the metadata is common, so the combination is element-wise on the
// value arrays.  fp32 arithmetic (one fused multiply-add on gamma·b), inputs
// and output each fp32 or bf16 (the output rounded to nearest even).  Eight
// values per thread and step.
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 y = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 x = __ldcs(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
}

template <typename TA, typename TB, typename TO>
__global__ void __launch_bounds__(256) axpby_kernel(float beta, const TA* a, float gamma, const TB* b,
                                                    TO* out, int64_t n8) {  // out may be a or b
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    float va[8], vb[8], vo[8];
    load8(a + 8 * i, va);
    load8(b + 8 * i, vb);
#pragma unroll
    for (int k = 0; k < 8; ++k) vo[k] = fmaf(beta, va[k], gamma * vb[k]);
    store8(out + 8 * i, vo);
  }
}

// Blocks per SM of a persistent kernel at its launch shape, cached per device.
template <typename Kernel>
static cudaError_t blocks_per_sm(Kernel kernel, int threads, int smem, std::atomic<int> (&cache)[64],
                                 int& out) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  out = cache[dev].load();
  if (out) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&out, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (out < 1) out = 1;
  cache[dev].store(out);
  return cudaSuccess;
}

}  // namespace

constexpr uint32_t kKeyShift = 1u << 17;  // the k17 argument of the prune kernels

cudaError_t launch_prune24(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream) {
  const int64_t nchunks = rows * cols / 8;
  if (nchunks == 0) return cudaSuccess;
  // one chunk per thread while the grid stays under 8 blocks per SM (short
  // latency for small weights); beyond that, up to kPruneUnroll per thread
  int64_t blocks = (nchunks + kPruneThreads - 1) / kPruneThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kPruneThreads);
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, prune24_kernel, static_cast<const uint4*>(W),
                                     static_cast<uint2*>(vals), meta, nchunks, kKeyShift);
  return e != cudaSuccess ? e : cudaGetLastError();
}


template <int CH, int QS, bool FROZEN = false, bool P12 = false>
static cudaError_t run_staged(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                              void* t_vals, uint8_t* t_meta, const uint8_t* t_meta_in,
                              cudaStream_t stream) {
  using C = DpStaged<CH, QS>;
  auto kernel = double_prune24_staged_kernel<CH, QS, FROZEN, P12>;
  static std::atomic<int> per_sm[64];
  int per = 0;
  if (cudaError_t e = blocks_per_sm(kernel, C::kThreads, C::kSmem, per_sm, per)) return e;
  const int64_t tiles = ((rows + 255) / 256) * (cols / (16 * CH));
  const int64_t cap = static_cast<int64_t>(sm_count()) * per;
  const int64_t blocks = tiles < cap ? tiles : cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<const uint8_t*>(vals), meta,
                                     static_cast<uint2*>(t_vals), t_meta, rows, cols, kKeyShift, t_meta_in);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int CH, int QS, bool GIVEN = false, bool FROZEN = false>
static cudaError_t run_fused(const void* W, const uint8_t* meta_in, int64_t rows, int64_t cols,
                             void* vals, uint8_t* meta, void* t_vals, uint8_t* t_meta,
                             const uint8_t* t_meta_in, cudaStream_t stream) {
  using C = DpStaged<CH, QS>;
  using F = FusedCfg<CH, QS, GIVEN>;
  auto kernel = prune_double24_kernel<CH, QS, GIVEN, FROZEN>;
  static std::atomic<int> per_sm[64];
  int per = 0;
  if (cudaError_t e = blocks_per_sm(kernel, C::kThreads, F::kSmem, per_sm, per)) return e;
  const int64_t tiles = ((rows + 255) / 256) * (cols / (16 * CH));
  const int64_t cap = static_cast<int64_t>(sm_count()) * per;
  const int64_t blocks = tiles < cap ? tiles : cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = F::kSmem;
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<const uint4*>(W), meta_in,
                                     static_cast<uint2*>(vals), meta, static_cast<uint2*>(t_vals), t_meta,
                                     rows, cols, kKeyShift, t_meta_in);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_prune_double24(const void* W, int64_t rows, int64_t cols, void* vals,
                                  uint8_t* meta, void* t_vals, uint8_t* t_meta,
                                  cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 128 == 0) {  // tile widths as A2's staged kernel
    const int64_t tiles_h = (rows + 255) / 256;
    if (tiles_h * (cols / 128) >= sm_count())
      return run_fused<8, 1>(W, nullptr, rows, cols, vals, meta, t_vals, t_meta, nullptr, stream);
    if (tiles_h * (cols / 64) >= sm_count())
      return run_fused<4, 2>(W, nullptr, rows, cols, vals, meta, t_vals, t_meta, nullptr, stream);
    return run_fused<2, 4>(W, nullptr, rows, cols, vals, meta, t_vals, t_meta, nullptr, stream);
  }
  // other widths: the two kernels one after the other
  if (cudaError_t e = launch_prune24(W, rows, cols, vals, meta, stream)) return e;
  return launch_double_prune24(vals, meta, rows, cols, t_vals, t_meta, stream);
}

cudaError_t launch_gather24(const void* W, const uint8_t* meta, int64_t rows, int64_t cols, void* vals,
                            cudaStream_t stream) {
  const int64_t nchunks = rows * cols / 8;
  if (nchunks == 0) return cudaSuccess;
  int64_t blocks = (nchunks + kPruneThreads - 1) / kPruneThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kPruneThreads);
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, gather24_kernel, static_cast<const uint4*>(W), meta,
                                     static_cast<uint2*>(vals), nchunks);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_recompress_double24(const void* W, const uint8_t* meta, int64_t rows, int64_t cols,
                                       void* vals, void* t_vals, uint8_t* t_meta, cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 128 == 0) {
    const int64_t tiles_h = (rows + 255) / 256;
    if (tiles_h * (cols / 128) >= sm_count())
      return run_fused<8, 1, true>(W, meta, rows, cols, vals, nullptr, t_vals, t_meta, nullptr, stream);
    if (tiles_h * (cols / 64) >= sm_count())
      return run_fused<4, 2, true>(W, meta, rows, cols, vals, nullptr, t_vals, t_meta, nullptr, stream);
    return run_fused<2, 4, true>(W, meta, rows, cols, vals, nullptr, t_vals, t_meta, nullptr, stream);
  }
  // other widths: the gather, then the second pruning of its output
  if (cudaError_t e = launch_gather24(W, meta, rows, cols, vals, stream)) return e;
  return launch_double_prune24(vals, meta, rows, cols, t_vals, t_meta, stream);
}

template <typename TA, typename TB, typename TO>
static cudaError_t run_axpby(float beta, const void* a, float gamma, const void* b, void* out, int64_t n,
                             cudaStream_t stream) {
  const int64_t n8 = n / 8;
  int64_t blocks = (n8 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, axpby_kernel<TA, TB, TO>, beta, static_cast<const TA*>(a), gamma,
                                     static_cast<const TB*>(b), static_cast<TO*>(out), n8);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_axpby(float beta, const void* a, int a_dt, float gamma, const void* b, int b_dt,
                         void* out, int out_dt, int64_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  using F = float;
  using H = __nv_bfloat16;
  const int key = a_dt * 4 + b_dt * 2 + out_dt;  // 0 = f32, 1 = bf16 each
  switch (key) {
    case 0: return run_axpby<F, F, F>(beta, a, gamma, b, out, n, stream);
    case 1: return run_axpby<F, F, H>(beta, a, gamma, b, out, n, stream);
    case 2: return run_axpby<F, H, F>(beta, a, gamma, b, out, n, stream);
    case 3: return run_axpby<F, H, H>(beta, a, gamma, b, out, n, stream);
    case 4: return run_axpby<H, F, F>(beta, a, gamma, b, out, n, stream);
    case 5: return run_axpby<H, F, H>(beta, a, gamma, b, out, n, stream);
    case 6: return run_axpby<H, H, F>(beta, a, gamma, b, out, n, stream);
    default: return run_axpby<H, H, H>(beta, a, gamma, b, out, n, stream);
  }
}

template <bool FROZEN, bool P12 = false>
static cudaError_t double_prune24_any(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                      void* t_vals, uint8_t* t_meta, const uint8_t* t_meta_in,
                                      cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 128 == 0) {
    // the widest tile that still gives every SM a tile
    const int64_t tiles_h = (rows + 255) / 256;
    // (narrower tiles split each octet's columns over more threads)
    if (tiles_h * (cols / 128) >= sm_count())
      return run_staged<8, 1, FROZEN, P12>(vals, meta, rows, cols, t_vals, t_meta, t_meta_in, stream);
    if (tiles_h * (cols / 64) >= sm_count())
      return run_staged<4, 2, FROZEN, P12>(vals, meta, rows, cols, t_vals, t_meta, t_meta_in, stream);
    return run_staged<2, 4, FROZEN, P12>(vals, meta, rows, cols, t_vals, t_meta, t_meta_in, stream);
  }
  const int64_t tiles = ((rows / 8 + 31) / 32) * ((cols / 16 + 7) / 8);
  int64_t blocks = tiles;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kDpThreads);
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, double_prune24_kernel<FROZEN, P12>, static_cast<const uint4*>(vals),
                                     reinterpret_cast<const uint16_t*>(meta),
                                     static_cast<uint2*>(t_vals), t_meta, rows, cols, kKeyShift, t_meta_in);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_double_prune24(const void* vals, const uint8_t* meta, int64_t rows,
                                  int64_t cols, void* t_vals, uint8_t* t_meta,
                                  cudaStream_t stream) {
  return double_prune24_any<false>(vals, meta, rows, cols, t_vals, t_meta, nullptr, stream);
}

cudaError_t launch_double_prune12(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* t_vals, uint8_t* t_meta, cudaStream_t stream) {
  return double_prune24_any<false, true>(vals, meta, rows, cols, t_vals, t_meta, nullptr, stream);
}

cudaError_t launch_double_prune24_frozen(const void* vals, const uint8_t* meta, int64_t rows,
                                         int64_t cols, const uint8_t* t_meta, void* t_vals,
                                         cudaStream_t stream) {
  return double_prune24_any<true>(vals, meta, rows, cols, t_vals, nullptr, t_meta, stream);
}

cudaError_t launch_recompress_frozen24(const void* W, const uint8_t* meta, const uint8_t* t_meta,
                                       int64_t rows, int64_t cols, void* vals, void* t_vals,
                                       cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 128 == 0) {
    const int64_t tiles_h = (rows + 255) / 256;
    if (tiles_h * (cols / 128) >= sm_count())
      return run_fused<8, 1, true, true>(W, meta, rows, cols, vals, nullptr, t_vals, nullptr, t_meta, stream);
    if (tiles_h * (cols / 64) >= sm_count())
      return run_fused<4, 2, true, true>(W, meta, rows, cols, vals, nullptr, t_vals, nullptr, t_meta, stream);
    return run_fused<2, 4, true, true>(W, meta, rows, cols, vals, nullptr, t_vals, nullptr, t_meta, stream);
  }
  if (cudaError_t e = launch_gather24(W, meta, rows, cols, vals, stream)) return e;
  return launch_double_prune24_frozen(vals, meta, rows, cols, t_meta, t_vals, stream);
}

}  // namespace slope
