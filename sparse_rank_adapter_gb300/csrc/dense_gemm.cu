// dense_gemm.cu — dense tcgen05 GEMMs of the path.
//
//   A5  dW  = M ⊙ (dYᵀ·X)   masked weight gradient; the epilogue applies the
//       weight's own 2:4 mask and writes only the kept entries (or a dense
//       masked matrix).  Source: "SLoPe: Double-Pruned Sparse Plus Lazy
//       Low-Rank Adapter Pretraining of LLMs", §2.3 and App. K (gradients of
//       pruned weights are masked and stored without their zeros).
//   A6  the adapter products of §2.2: XL = X·L and G = dY·Rᵀ, written as
//       hi/lo bf16 pairs (hi = bf16(v), lo = bf16(v - hi): about 16
//       significant bits, so the tensor cores can take them at nearly fp32
//       accuracy), then dL = Xᵀ·G and dR = XLᵀ·dY over both parts, folded
//       back onto r columns in the epilogue.
//
//   D[m][n] = Σ_k A[m][k]·B[n][k]; A and B are bf16, stored either K-major
//   (row = m or n) or MN-major (row = k), as the row-major tensors of the
//   layer happen to be.  Tile 128 x BN x 64, TMA-fed smem ring, fp32 TMEM
//   accumulator, optional split-K with atomic fp32 accumulation.
//
// Persistent kernel, one CTA per SM, tiles (m, n, split) taken round-robin.
// Roles (192 threads): warp 0 TMA, warp 1 TMEM owner + MMA issuer, warps
// 2..5 epilogue.  The accumulator is double-buffered in TMEM so a tile's
// epilogue overlaps the next tile's K-loop.  Every mbarrier wait is bounded.
//
// dw_pair_kernel (below) runs dW on CTA pairs (pair-wide MMA, 256 x 256
// tiles) and, when asked, dL and dR as extra tiles of the same launch:
// dRᵀ = dYᵀ·XL shares dW's A operand and dLᵀ = Gᵀ·X its B operand.  The
// outputs a split launch adds into are zeroed first by zero3_kernel, a
// programmatic dependent like the GEMMs (a memset node would break the
// chain of early launches).
//
// The hi/lo store needs the whole sum before it rounds, so its split-K goes
// through a thread-block cluster instead of atomics: the cluster's CTAs take
// K ranges of the one tile the cluster owns; each writes its fp32 partial
// into its own stage ring (drained: its last MMA has completed) and arrives
// (release, cluster scope) on every other CTA's barrier; then each adds one
// slice of the tile's rows over all the partials (distributed shared
// memory), stores it, and arrives on every other CTA's second barrier; a
// cluster barrier at the end keeps each CTA until the others have read its
// partial.  This is what
// gives a handful of token tiles (small T) more than one SM each, at every
// tile width.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "slope_internal.h"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kA_BYTES = kBM * kBK * 2;  // 16 KB
constexpr int kThreads = 192;

template <int BN>
struct DnCfg {
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE = kA_BYTES + B_BYTES;
  // fp32 partial tile that each CTA of a cluster leaves for the others when
  // a tile's K is split over the cluster (column-major: [BN][128]).  A
  // split cluster owns one tile, so by then every stage fill has been
  // consumed: the partial lives in the stage ring.
  static constexpr int RED_BYTES = kBM * BN * 4;
  static constexpr int STAGES_FIT = 192 * 1024 / STAGE;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC_COLS = BN < 32 ? 32 : BN;  // one accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS;       // double-buffered
  // stages | barriers (1 KB) | alignment slack
  static constexpr int SMEM = STAGES * STAGE + 1024 + 1024;
  // MN-major B: swizzle atom width in elements (64 for SW128) and its code.
  static constexpr int B_ATOM = BN >= 64 ? 64 : BN;
  static constexpr uint32_t B_SWZ = BN >= 64 ? kSwizzle128 : BN == 32 ? kSwizzle64 : kSwizzle32;
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(RED_BYTES <= STAGES * STAGE, "the split partial fits in the stage ring");
};

struct DnParams {
  int M, N, K;
  int kb_per_split, num_kb;
  int tiles_m, tiles_n, num_tiles;  // tiles = tiles_m x tiles_n x splits
  int group_m;                      // pair kernel: M pairs per raster band
  int64_t ldo;
  void* out;
  const uint8_t* meta;  // masked dW: metadata, N/8 bytes per row
  int dense_dw, accumulate, atomic_out;
  int nm28;  // masked dW: `meta` holds 2:8 bytes (i0 | i1 << 3 per 8 columns); compressed dW has N/4 per row
  unsigned int* wave_ctr;  // pair dW: producers' arrival counter (zeroed before the launch), or NULL
  int lo_off, fold;
  int csplit;  // CTAs of a cluster that split one tile's K (hi/lo store only); 1 = none
  int fuse_r;  // pair dW kernel: r of the adapter gradients computed alongside; 0 = none
  float* dl;   // in x r fp32 (added into)
  float* dr;   // r x out fp32 (added into)
  unsigned int* status;
};

__device__ __forceinline__ float pick3(uint32_t i, float a, float b, float c) {
  return i == 0 ? a : (i == 1 ? b : c);
}

// One 32-column (or BN-column, when narrower) chunk of a tile row, already in
// registers: row m of the tile, columns n0 + c0 .. n0 + c0 + CH - 1.
template <int BN, int CH, DenseEpi EPI>
__device__ __forceinline__ void epilogue_chunk(const DnParams& p, const uint32_t (&v)[32], int m,
                                               int n0, int c0, const uint4 (&mrow)[2]) {
  if constexpr (EPI == DenseEpi::StoreBf16HiLo) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(m) * p.ldo;
#pragma unroll
    for (int j = 0; j < CH; j += 8) {
      const int n = n0 + c0 + j;
      if (n < p.N) {  // N % 8 == 0
        uint4 hi, lo;
        uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
        uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = __uint_as_float(v[j + 2 * u]), b = __uint_as_float(v[j + 2 * u + 1]);
          const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
          const __nv_bfloat162 l =
              __floats2bfloat162_rn(a - __bfloat162float(h.x), b - __bfloat162float(h.y));
          ph[u] = *reinterpret_cast<const uint32_t*>(&h);
          pl[u] = *reinterpret_cast<const uint32_t*>(&l);
        }
        *reinterpret_cast<uint4*>(o + n) = hi;
        *reinterpret_cast<uint4*>(o + p.lo_off + n) = lo;
      }
    }
  } else if constexpr (EPI == DenseEpi::AddF32) {
    float* o = static_cast<float*>(p.out) + static_cast<size_t>(m) * p.ldo;
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int n = n0 + c0 + j;
      if (n < p.N) red_add_f32(o + (p.fold && n >= p.fold ? n - p.fold : n), __uint_as_float(v[j]));
    }
  } else if constexpr (EPI == DenseEpi::AddF32Transposed) {
    float* o = static_cast<float*>(p.out);
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int n = n0 + c0 + j;
      const int nf = p.fold && n >= p.fold ? n - p.fold : n;
      if (n < p.N) red_add_f32(o + static_cast<size_t>(nf) * p.ldo + m, __uint_as_float(v[j]));
    }
  } else {  // MaskedWeightGrad: 32 columns = 8 groups = one metadata word
    const int nb = n0 + c0;
    if (nb >= p.N) return;
    const uint32_t word = reinterpret_cast<const uint32_t*>(mrow)[c0 / 32];
    float* orow = static_cast<float*>(p.out) + static_cast<size_t>(m) * p.ldo;
    if (p.nm28) {
      // 2:8 mask: the word's four bytes are the 32 columns' four groups of
      // eight; group b keeps columns 8b + i0 and 8b + i1
      float d[32];
      float kept[8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (word >> (8 * b)) & 0xFFu;
        const uint32_t i0 = byte & 7u, i1 = (byte >> 3) & 7u;
        float k0 = 0.0f, k1 = 0.0f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float x = __uint_as_float(v[8 * b + jj]);
          const bool on0 = jj == static_cast<int>(i0), on1 = jj == static_cast<int>(i1);
          k0 = on0 ? x : k0;
          k1 = on1 ? x : k1;
          d[8 * b + jj] = (on0 || on1) ? x : 0.0f;
        }
        kept[2 * b] = k0;
        kept[2 * b + 1] = k1;
      }
      const int nvec = p.dense_dw ? 8 : 2;
      float4* dst = reinterpret_cast<float4*>(orow + (p.dense_dw ? nb : nb / 4));
      const float* src = p.dense_dw ? d : kept;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u >= nvec) break;
        float4 x = make_float4(src[4 * u], src[4 * u + 1], src[4 * u + 2], src[4 * u + 3]);
        if (p.atomic_out) {
          red_add_f32x4(reinterpret_cast<float*>(&dst[u]), x);
        } else {
          if (p.accumulate) {
            const float4 y = dst[u];
            x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
          }
          dst[u] = x;
        }
      }
    } else if (p.dense_dw) {
      float d[32];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint32_t nib = (word >> (4 * g)) & 0xFu;
        const uint32_t i0 = nib & 3u, i1 = nib >> 2;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          d[4 * g + jj] = (jj == static_cast<int>(i0) || jj == static_cast<int>(i1))
                              ? __uint_as_float(v[4 * g + jj]) : 0.0f;
      }
      float4* dst = reinterpret_cast<float4*>(orow + nb);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float4 x = make_float4(d[4 * u], d[4 * u + 1], d[4 * u + 2], d[4 * u + 3]);
        if (p.atomic_out) {
          red_add_f32x4(reinterpret_cast<float*>(&dst[u]), x);
        } else {
          if (p.accumulate) {
            const float4 y = dst[u];
            x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
          }
          dst[u] = x;
        }
      }
    } else {
      float kept[16];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint32_t nib = (word >> (4 * g)) & 0xFu;
        const uint32_t i0 = nib & 3u, i1 = nib >> 2;
        const float a = __uint_as_float(v[4 * g]), b = __uint_as_float(v[4 * g + 1]);
        const float c = __uint_as_float(v[4 * g + 2]), d = __uint_as_float(v[4 * g + 3]);
        kept[2 * g] = pick3(i0, a, b, c);
        kept[2 * g + 1] = i1 == 3 ? d : (i1 == 2 ? c : b);
      }
      float4* dst = reinterpret_cast<float4*>(orow + nb / 2);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float4 x = make_float4(kept[4 * u], kept[4 * u + 1], kept[4 * u + 2], kept[4 * u + 3]);
        if (p.atomic_out) {
          red_add_f32x4(reinterpret_cast<float*>(&dst[u]), x);
        } else {
          if (p.accumulate) {
            const float4 y = dst[u];
            x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
          }
          dst[u] = x;
        }
      }
    }
  }
}

template <bool A_MN, bool B_MN, int BN, DenseEpi EPI>
__global__ void __launch_bounds__(kThreads, 1)
    dense_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const DnParams p) {
  using C = DnCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* red_full = mma_done + 1;   // cluster split: every CTA's partial is in place
  uint64_t* red_empty = red_full + 1;  // cluster split: every CTA has read this CTA's partial
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(red_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* red = reinterpret_cast<float*>(smem);  // split partial, over the drained stage ring

  const int warp = warp_id(), lane = lane_id();
  const int cs = p.csplit;
  const uint32_t crank = cs > 1 ? cluster_ctarank() : 0u;
  const int tiles_mn = p.tiles_m * p.tiles_n;
  const int units = p.num_tiles;
  const int unit0 = static_cast<int>(cs > 1 ? blockIdx.x / cs : blockIdx.x);
  const int ustep = static_cast<int>(cs > 1 ? gridDim.x / cs : gridDim.x);
  // unit -> (tile m0, n0, split z); in a cluster the split is the CTA's rank
  auto decode = [&](int u, int& m0, int& n0, int& z) {
    const int mn = u % tiles_mn;
    z = cs > 1 ? static_cast<int>(crank) : u / tiles_mn;
    m0 = (mn % p.tiles_m) * kBM;
    n0 = (mn / p.tiles_m) * BN;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    mbar_init(red_full, 4 * (cs > 1 ? cs - 1 : 1));   // every other CTA's epilogue warps
    mbar_init(red_empty, 4 * (cs > 1 ? cs - 1 : 1));
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  if (cs > 1)
    cluster_sync();  // the peers' barriers exist before anyone arrives on them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dependency_wait();  // the previous kernel's outputs are visible from here
  allow_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer -------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int it = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep) {
        int m0, n0, z;
        decode(u, m0, n0, z);
        const int kb0 = z * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { stop = true; break; }
          uint8_t* sA = smem + s * C::STAGE;
          uint8_t* sB = sA + kA_BYTES;
          const int k0 = kb * kBK;
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          if (A_MN) {
            tma_load_2d(sA, &tmA, &full[s], m0, k0);
            tma_load_2d(sA + 8192, &tmA, &full[s], m0 + 64, k0);
          } else {
            tma_load_2d(sA, &tmA, &full[s], k0, m0);
          }
          if (B_MN) {
#pragma unroll
            for (int a = 0; a < BN / C::B_ATOM; ++a)
              tma_load_2d(sB + a * (C::B_ATOM * kBK * 2), &tmB, &full[s], n0 + a * C::B_ATOM, k0);
          } else {
            tma_load_2d(sB, &tmB, &full[s], k0, n0);
          }
        }
      }
      for (int i = it - 1; i >= 0 && i >= it - C::STAGES; --i) {
        volatile int no_abort = 0;
        mbar_wait(&full[i % C::STAGES], (i / C::STAGES) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------- MMA issuer ---------
      const uint32_t idesc = idesc_bf16(kBM, BN, A_MN, B_MN, false);
      constexpr uint32_t b_swz_bytes = C::B_ATOM * 2;  // MN-major B swizzle span
      int it = 0, local = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep, ++local) {
        int m0, n0, z;
        decode(u, m0, n0, z);
        const int kb0 = z * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * C::ACC_COLS;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&full[s], ph, abort_flag, p.status)) { stop = true; break; }
          tc_fence_after();
          const uint32_t aA = smem_u32(smem + s * C::STAGE);
          const uint32_t aB = aA + kA_BYTES;
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j) {
            const uint64_t da = A_MN ? smem_desc(aA + j * 2048, 8192, 1024, kSwizzle128)
                                     : smem_desc(aA + j * 32, 0, 1024, kSwizzle128);
            const uint64_t db =
                B_MN ? smem_desc(aB + j * 16 * b_swz_bytes, C::B_ATOM * kBK * 2, 8 * b_swz_bytes,
                                 C::B_SWZ)
                     : smem_desc(aB + j * 32, 0, 1024, kSwizzle128);
            mma_bf16_ss(d, da, db, idesc, (kb > kb0 || j > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (!stop) mma_commit(&acc_full[buf]);
      }
      mma_commit(mma_done);
    }
  } else {
    // ------------------------------------------------ epilogue -----------
    const int q = warp & 3;
    int local = 0;
    for (int u = unit0; u < units; u += ustep, ++local) {
      int m0, n0, z;
      decode(u, m0, n0, z);
      const int m = m0 + 32 * q + lane;
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t trow = tmem + buf * C::ACC_COLS + (static_cast<uint32_t>(32 * q) << 16);
      constexpr int CH = BN < 32 ? BN : 32;
      if constexpr (EPI == DenseEpi::StoreBf16HiLo) {
        if (cs > 1) {
          // Cluster split of K, reduce-scatter: every CTA leaves its fp32
          // partial in its own shared memory ([column][row]); then each
          // adds one slice of the rows over all the CTAs' partials and
          // stores it.  The buffer is overwritten only after every CTA
          // has read the previous tile's.
          if (!mbar_wait_cluster(red_empty, (local & 1) ^ 1, abort_flag, p.status)) break;
          const int row = 32 * q + lane;
#pragma unroll
          for (int c0 = 0; c0 < BN; c0 += CH) {
            uint32_t v[32];
            if constexpr (CH == 32) {
              tmem_ld_32x32b_x32(trow + c0, v);
            } else {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < CH / 4; ++u) {
                tmem_ld_32x32b_x4(trow + c0 + 4 * u, w);
                v[4 * u] = w[0]; v[4 * u + 1] = w[1]; v[4 * u + 2] = w[2]; v[4 * u + 3] = w[3];
              }
            }
            tmem_ld_wait();
            if (c0 + CH >= BN) {  // last chunk read: hand the accumulator back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
#pragma unroll
            for (int j = 0; j < CH; ++j) red[(c0 + j) * kBM + row] = __uint_as_float(v[j]);
          }
          asm volatile("fence.acq_rel.cluster;" ::: "memory");
          __syncwarp();
          if (lane == 0)
            for (int pr = 0; pr < cs; ++pr)
              if (pr != static_cast<int>(crank))
                mbar_arrive_cluster(mapa_shared(smem_u32(red_full), static_cast<uint32_t>(pr)));
          if (!mbar_wait_cluster(red_full, local & 1, abort_flag, p.status)) break;
          // this CTA's slice: rows [r0, r0 + nrow), 8 columns per work item,
          // consecutive threads on consecutive rows (coalesced remote loads)
          const int rows = (kBM + cs - 1) / cs;
          const int r0 = static_cast<int>(crank) * rows;
          const int nrow = min(kBM, r0 + rows) - r0;
          const int items = nrow * (BN / 8);
          for (int w = static_cast<int>(threadIdx.x) - 64; w < items; w += 128) {
            const int rr = r0 + w % nrow, cg = w / nrow;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int pr = 0; pr < cs; ++pr) {
              const uint32_t base = mapa_shared(smem_u32(red), static_cast<uint32_t>(pr));
              float t[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) t[j] = ld_shared_cluster_f32(base + 4u * ((8 * cg + j) * kBM + rr));
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[j] += t[j];
            }
            const int mm = m0 + rr, n = n0 + 8 * cg;
            if (mm < p.M && n < p.N) {  // N % 8 == 0
              uint4 hi, lo;
              uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
              uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
                const __nv_bfloat162 l = __floats2bfloat162_rn(acc[2 * u] - __bfloat162float(h.x),
                                                               acc[2 * u + 1] - __bfloat162float(h.y));
                ph[u] = *reinterpret_cast<const uint32_t*>(&h);
                pl[u] = *reinterpret_cast<const uint32_t*>(&l);
              }
              __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(mm) * p.ldo;
              *reinterpret_cast<uint4*>(o + n) = hi;
              *reinterpret_cast<uint4*>(o + p.lo_off + n) = lo;
            }
          }
          asm volatile("fence.acq_rel.cluster;" ::: "memory");
          __syncwarp();
          if (lane == 0)
            for (int pr = 0; pr < cs; ++pr)
              if (pr != static_cast<int>(crank))
                mbar_arrive_cluster(mapa_shared(smem_u32(red_empty), static_cast<uint32_t>(pr)));
          continue;
        }
      }
      uint4 mrow[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if constexpr (EPI == DenseEpi::MaskedWeightGrad) {
        if (m < p.M) {
          const uint4* mp = reinterpret_cast<const uint4*>(p.meta + static_cast<size_t>(m) * (p.N / 8) + n0 / 8);
          mrow[0] = mp[0];
          if (n0 + 128 < p.N) mrow[1] = mp[1];
        }
      }
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += CH) {
        uint32_t v[32];
        if constexpr (CH == 32) {
          tmem_ld_32x32b_x32(trow + c0, v);
        } else {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < CH / 4; ++u) {
            tmem_ld_32x32b_x4(trow + c0 + 4 * u, w);
            v[4 * u] = w[0]; v[4 * u + 1] = w[1]; v[4 * u + 2] = w[2]; v[4 * u + 3] = w[3];
          }
        }
        tmem_ld_wait();
        if (c0 + CH >= BN) {  // last chunk read: hand the buffer back early
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (m >= p.M) continue;
        epilogue_chunk<BN, CH, EPI>(p, v, m, n0, c0, mrow);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.status);
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // No CTA leaves while the leader may still read its partial or arrive on
  // its barrier.
  if (cs > 1) cluster_sync();
}

// Zeroes up to four fp32 arrays (the outputs a launch adds into and its
// wave counter) in one launch.  Unlike memset nodes it is a programmatic
// dependent of the kernel before it (set-up overlaps that kernel's tail) and
// lets the next kernel launch early; it writes only after the previous
// kernel is done.
__global__ void __launch_bounds__(256) zero3_kernel(float4* a, int64_t na, float4* b, int64_t nb, float4* c,
                                                    int64_t nc, float4* d, int64_t nd) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb + nc + nd; i += stride) {
    if (i < na) a[i] = z;
    else if (i < na + nb) b[i - na] = z;
    else if (i < na + nb + nc) c[i - na - nb] = z;
    else d[i - na - nb - nc] = z;
  }
}

// ---------------------------------------------------------------------------
// dW on CTA pairs: the pair-wide MMA (M = 256 = two 128-row weight tiles, one
// per CTA, N = 256 input columns, half of them in each CTA's shared memory)
// halves the bytes each SM takes in per flop.  The even CTA issues the MMAs
// and owns the full barriers, which both CTAs' TMA loads signal; its MMA
// commits release the stages and the accumulators in both CTAs; both CTAs'
// epilogue warps hand accumulator buffers back to the even CTA.
// ---------------------------------------------------------------------------

constexpr int kPairBN = 256;          // N of the pair tile
constexpr int kPairHalfB = kPairBN / 2;  // B columns each CTA holds
constexpr int kPairStage = kA_BYTES + kPairHalfB * kBK * 2;  // 32 KB
constexpr int kPairStages = 6;
constexpr int kPairSmem = kPairStages * kPairStage + 1024 + 1024;
constexpr int kPairTmemCols = 2 * kPairBN;  // double-buffered 256-column accumulator
// 10 warps: TMA, MMA, and eight epilogue warps (two per TMEM lane quadrant,
// alternate 32-column chunks), so the last tile's epilogue, which nothing
// overlaps, is short
constexpr int kPairThreads = 320;

__global__ void __launch_bounds__(kPairThreads, 1)
    dw_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmXL,
                   const DnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStage);
  uint64_t* empty = full + kPairStages;
  uint64_t* acc_full = empty + kPairStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2], counted in the even CTA
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const int pairs_m = p.tiles_m / 2;
  const int w_tiles = pairs_m * p.tiles_n;  // dW tiles of one split
  // With the adapter gradients fused, each split also has pairs_m dRᵀ tiles
  // (dYᵀ·XL: the pair's weight rows against the 2r columns of XL) and
  // tiles_n dLᵀ tiles (Gᵀ·X: the 2r columns of G, as rows, against X).
  const int per_split = w_tiles + (p.fuse_r > 0 ? pairs_m + p.tiles_n : 0);
  const int units = per_split * p.num_tiles;  // num_tiles holds the split count here
  const int unit0 = static_cast<int>(blockIdx.x >> 1);
  const int ustep = static_cast<int>(gridDim.x >> 1);
  // unit -> (this CTA's rows m0, the pair's columns n0, split z, kind: 0 dW,
  // 1 dRᵀ, 2 dLᵀ).  dW tiles in raster order within a split: bands of
  // group_m M pairs; within a band the M pairs turn fastest, then the N
  // tiles.  The pairs in flight (consecutive units) then cover a block about
  // as tall as it is wide, which loads the fewest operand slabs (256 rows of
  // dY or 256 columns of X over the split's K range) per wave of tiles.
  auto decode = [&](int u, int& m0, int& n0, int& z, int& kind) {
    const int mn = u % per_split;
    z = u / per_split;
    if (mn < w_tiles) {
      kind = 0;
      const int per_band = p.group_m * p.tiles_n;
      const int b = mn / per_band, w = mn % per_band;
      const int first = b * p.group_m;
      const int gm = min(p.group_m, pairs_m - first);
      m0 = (2 * (first + w % gm) + static_cast<int>(rank)) * kBM;  // this CTA's 128 rows
      n0 = (w / gm) * kPairBN;                                       // the pair's 256 columns
    } else if (mn < w_tiles + pairs_m) {
      kind = 1;
      m0 = (2 * (mn - w_tiles) + static_cast<int>(rank)) * kBM;
      n0 = 0;
    } else {
      kind = 2;
      m0 = static_cast<int>(rank) * kBM;  // rows = columns of G (2r of them are real)
      n0 = (mn - w_tiles - pairs_m) * kPairBN;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 16);  // eight epilogue warps in each CTA
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kPairTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dependency_wait();  // the previous kernel's outputs are visible from here
  allow_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer -------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (p.fuse_r > 0) {
        tma_prefetch_desc(&tmG);
        tma_prefetch_desc(&tmXL);
      }
      int it = 0;
      bool stop = false;
      // Waves in step: before the loads of its unit of wave w (w >= 1), every
      // producer of the grid waits until all have issued wave w - 1's.  The
      // units in flight then stay one compact raster block, whose slabs of
      // dY and X the pairs share in L2.  Only waves in which every pair has
      // a unit take part.  The wait only saves DRAM traffic: it is bounded
      // at about 50 µs, after which this producer stops waiting for the
      // rest of the launch (e.g. when CTAs of the grid cannot be resident
      // together because other kernels hold SMs).
      const int full_waves = units / ustep;
      bool in_step = p.wave_ctr != nullptr;
      int wave = 0;
      for (int u = unit0; u < units && !stop; u += ustep, ++wave) {
        if (in_step && wave >= 1 && wave < full_waves) {
          atomicAdd(p.wave_ctr, 1u);
          in_step = counter_wait_geq(p.wave_ctr, static_cast<unsigned int>(wave) * gridDim.x, 100000);
        }
        int m0, n0, z, kind;
        decode(u, m0, n0, z, kind);
        const CUtensorMap* mA = kind == 2 ? &tmG : &tmA;   // rows: weight rows, or G's columns
        const CUtensorMap* mB = kind == 1 ? &tmXL : &tmB;  // columns: X's, or XL's
        const int nb = n0 + static_cast<int>(rank) * kPairHalfB;  // this CTA's half of B
        const int kb0 = z * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { stop = true; break; }
          uint8_t* sA = smem + s * kPairStage;
          uint8_t* sB = sA + kA_BYTES;
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);  // the even CTA's barrier
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kPairStage);
          const int k0 = kb * kBK;
          // (boxes past G's or XL's 2r columns are zero-filled and still
          // count their full bytes)
          tma_load_2d_pair(sA, mA, bar, m0, k0);
          tma_load_2d_pair(sA + 8192, mA, bar, m0 + 64, k0);
          tma_load_2d_pair(sB, mB, bar, nb, k0);
          tma_load_2d_pair(sB + 8192, mB, bar, nb + 64, k0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------- MMA issuer ---------
      const uint32_t idesc = idesc_bf16(2 * kBM, kPairBN, true, true, false);
      int it = 0, local = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep, ++local) {
        int m0, n0, z, kind;
        decode(u, m0, n0, z, kind);
        const int kb0 = z * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * kPairBN;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kPairStages;
          const uint32_t ph = (it / kPairStages) & 1;
          if (!mbar_wait(&full[s], ph, abort_flag, p.status)) { stop = true; break; }
          tc_fence_after();
          const uint32_t aA = smem_u32(smem + s * kPairStage);
          const uint32_t aB = aA + kA_BYTES;
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j) {
            const uint64_t da = smem_desc(aA + j * 2048, 8192, 1024, kSwizzle128);
            const uint64_t db = smem_desc(aB + j * 2048, 8192, 1024, kSwizzle128);
            mma_bf16_ss_pair(d, da, db, idesc, (kb > kb0 || j > 0) ? 1u : 0u);
          }
          mma_commit_pair_mc(&empty[s], 3);
        }
        if (!stop) mma_commit_pair_mc(&acc_full[buf], 3);
      }
      mma_commit_pair_mc(mma_done, 3);
    }
  } else {
    // ------------------------------------------------ epilogue -----------
    const int q = warp & 3;
    const int half = warp >= 6 ? 1 : 0;  // which alternate column chunks
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
    int local = 0;
    for (int u = unit0; u < units; u += ustep, ++local) {
      int m0, n0, z, kind;
      decode(u, m0, n0, z, kind);
      const int m = m0 + 32 * q + lane;
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t trow = tmem + buf * kPairBN + (static_cast<uint32_t>(32 * q) << 16);
      if (kind != 0) {
        // Adapter gradients.  Columns (dRᵀ) or rows (dLᵀ) j < 2r are real;
        // the lo half j >= r folds onto j - r.  fp32 adds into dR (r x out:
        // lanes = consecutive weight rows) or dL (in x r: lanes = consecutive
        // j of one input column).
        const int r = p.fuse_r;
        const int ncols = kind == 1 ? (2 * r + 31) / 32 * 32 : kPairBN;
        const int jrow = static_cast<int>(rank) * kBM + 32 * q + lane;  // dLᵀ: j of this lane
        const bool live = kind == 1 || static_cast<int>(rank) * kBM + 32 * q < 2 * r;
        bool handed = false;
        if (live) {
          for (int c0 = 32 * half; c0 < ncols; c0 += 64) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(trow + c0, v);
            tmem_ld_wait();
            if (c0 + 64 >= ncols) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8 * buf);
              handed = true;
            }
            if (kind == 1) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int c = c0 + jj;
                if (c < 2 * r) red_add_f32(p.dr + static_cast<size_t>(c < r ? c : c - r) * p.M + m,
                                           __uint_as_float(v[jj]));
              }
            } else if (jrow < 2 * r) {
              const int jf = jrow < r ? jrow : jrow - r;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int i = n0 + c0 + jj;
                if (i < p.N) red_add_f32(p.dl + static_cast<size_t>(i) * r + jf, __uint_as_float(v[jj]));
              }
            }
          }
        }
        if (!handed) {  // nothing of this tile for this warp: hand the buffer back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8 * buf);
        }
        continue;
      }
      uint4 mrow[2];
      {
        const uint4* mp = reinterpret_cast<const uint4*>(p.meta + static_cast<size_t>(m) * (p.N / 8) + n0 / 8);
        mrow[0] = mp[0];
        mrow[1] = (n0 + 128 < p.N) ? mp[1] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int c0 = 0; c0 < kPairBN; c0 += 32) {
        if (((c0 >> 5) & 1) != half) continue;  // the other warp of this quadrant's chunk
        uint32_t v[32];
        tmem_ld_32x32b_x32(trow + c0, v);
        tmem_ld_wait();
        if (c0 + 64 >= kPairBN) {  // this warp's last chunk read: hand the buffer back early
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8 * buf);
        }
        epilogue_chunk<kPairBN, 32, DenseEpi::MaskedWeightGrad>(p, v, m, n0, c0, mrow);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.status);
    tmem_dealloc_pair(tmem, kPairTmemCols);
  }
  cluster_sync();  // no CTA leaves while its peer may still signal it
}

cudaError_t run_dw_pair(const DenseGemmArgs& a, cudaStream_t stream) {
  static std::atomic<int> attr_set[64];
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = stream;
  if (!attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(dw_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    e = cudaOccupancyMaxActiveClusters(&n, dw_pair_kernel, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters[dev].store(n > 0 ? n : 1);
    attr_set[dev].store(1);
  }
  const uint64_t M = a.M, N = a.N, K = a.K;
  CUtensorMap tA, tB;  // dY (K x M) and X (K x N), both MN-major, 64 x 64 boxes
  bool ok = make_tmap_2d(&tA, a.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, 2 * a.lda, 64, kBK, Swz::B128) &&
            make_tmap_2d(&tB, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, 2 * a.ldb, 64, kBK, Swz::B128);
  const int fr = a.fuse_r;
  CUtensorMap tG, tXL;  // G and XL (K x 2r), MN-major, 64 x 64 boxes (past 2r: zeros)
  if (fr > 0) {
    ok = ok &&
         make_tmap_2d(&tG, a.g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2 * fr, K, 4 * fr, 64, kBK, Swz::B128) &&
         make_tmap_2d(&tXL, a.xl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2 * fr, K, 4 * fr, 64, kBK, Swz::B128);
  } else {
    tG = tA;  // unused
    tXL = tB;
  }
  if (!ok) return cudaErrorInvalidValue;
  const int num_kb = static_cast<int>((K + kBK - 1) / kBK);
  const int tiles_m = static_cast<int>(M / kBM);  // even
  const int tiles_n = static_cast<int>((N + kPairBN - 1) / kPairBN);
  const int clusters_max = max_clusters[dev].load();
  const int pair_tiles = (tiles_m / 2) * tiles_n + (fr > 0 ? tiles_m / 2 + tiles_n : 0);
  int splits = choose_splits(pair_tiles, clusters_max, num_kb);
  const int kbs = (num_kb + splits - 1) / splits;
  splits = (num_kb + kbs - 1) / kbs;

  DnParams p = {};
  p.csplit = 1;
  p.M = static_cast<int>(M); p.N = static_cast<int>(N); p.K = static_cast<int>(K);
  p.kb_per_split = kbs; p.num_kb = num_kb;
  p.tiles_m = tiles_m; p.tiles_n = tiles_n;
  p.num_tiles = splits;  // the kernel's units: (dW + adapter tiles of one split) x splits
  p.fuse_r = fr;
  p.dl = a.dl;
  p.dr = a.dr;
  {
    // The units in flight (about one per resident pair) should form a
    // block whose slabs of dY (M) and X (N), equal in bytes, are fewest:
    // about sqrt(pairs) M pairs tall.  Bands of as even a height as that
    // allows, so no thin band is left at the bottom.
    int want = static_cast<int>(std::lround(std::sqrt(static_cast<double>(clusters_max))));
    const int pairs_m = tiles_m / 2;
    want = want < 1 ? 1 : (want > pairs_m ? pairs_m : want);
    const int bands = (pairs_m + want - 1) / want;
    p.group_m = (pairs_m + bands - 1) / bands;
  }
  p.ldo = a.ldo; p.out = a.out; p.meta = a.meta;
  p.nm28 = a.nm28 ? 1 : 0;
  p.dense_dw = a.dense_dw ? 1 : 0;
  p.accumulate = a.accumulate ? 1 : 0;
  p.atomic_out = splits > 1 ? 1 : 0;
  p.wave_ctr = a.wave_ctr;
  {
    // dW when split K adds its parts; the adapter gradients are always
    // added; the wave counter starts at zero (4 floats: 16 bytes)
    const bool zero_out = !a.accumulate;
    const size_t ndw = zero_out && p.atomic_out ? static_cast<size_t>(M) * a.ldo : 0;
    const size_t nl = zero_out && fr > 0 ? static_cast<size_t>(N) * fr : 0;
    const size_t nr = zero_out && fr > 0 ? static_cast<size_t>(fr) * M : 0;
    const size_t nw = a.wave_ctr != nullptr ? 4 : 0;
    if (ndw + nl + nr + nw > 0)
      if (cudaError_t e = launch_zero3(static_cast<float*>(a.out), ndw, a.dl, nl, a.dr, nr, stream,
                                       reinterpret_cast<float*>(a.wave_ctr), nw))
        return e;
  }
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  const int units = pair_tiles * splits;
  const int clusters = units < clusters_max ? units : clusters_max;
  cfg.gridDim = dim3(2 * clusters);
  add_pdl_attr(cfg, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, dw_pair_kernel, tA, tB, tG, tXL, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool A_MN, bool B_MN, int BN, DenseEpi EPI>
cudaError_t run(const DenseGemmArgs& a, cudaStream_t stream) {
  using C = DnCfg<BN>;
  auto kernel = dense_gemm_kernel<A_MN, B_MN, BN, EPI>;
  static std::atomic<int> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1);
  }
  const uint64_t M = a.M, N = a.N, K = a.K;
  CUtensorMap tA, tB;
  bool ok;
  if (A_MN)  // stored K x M (row stride lda)
    ok = make_tmap_2d(&tA, a.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, 2 * a.lda, 64, kBK, Swz::B128);
  else       // stored M x K
    ok = make_tmap_2d(&tA, a.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M, 2 * a.lda, kBK, kBM, Swz::B128);
  if (B_MN) {
    const Swz sw = C::B_ATOM == 64 ? Swz::B128 : C::B_ATOM == 32 ? Swz::B64 : Swz::B32;
    ok = ok && make_tmap_2d(&tB, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, 2 * a.ldb, C::B_ATOM, kBK, sw);
  } else {
    ok = ok && make_tmap_2d(&tB, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, 2 * a.ldb, kBK, BN, Swz::B128);
  }
  if (!ok) return cudaErrorInvalidValue;

  const int num_kb = static_cast<int>((K + kBK - 1) / kBK);
  const int tiles_m = static_cast<int>((M + kBM - 1) / kBM);
  const int tiles_n = static_cast<int>((N + BN - 1) / BN);
  int splits = a.splits;
  if (splits <= 0) splits = choose_splits(tiles_m * tiles_n, sm_count(), num_kb);
  int csplit = 1;
  if (EPI == DenseEpi::StoreBf16HiLo) {
    // no atomic split for the rounding store; when the tiles leave SMs
    // idle, split K over a cluster of up to 8 CTAs.  The hand-over costs
    // about 2.5 us (cluster-scope fences and arrivals), so each CTA keeps
    // at least 16 K-blocks.
    splits = 1;
    const int tiles = tiles_m * tiles_n;
    int want = sm_count() / tiles;
    want = want < 8 ? want : 8;
    want = want < num_kb / 16 ? want : num_kb / 16;
    if (want >= 2) {
      const int kbs = (num_kb + want - 1) / want;
      csplit = (num_kb + kbs - 1) / kbs;  // every CTA of the cluster owns >= 1 K-block
    }
  }
  const int kbs = csplit > 1 ? (num_kb + csplit - 1) / csplit : (num_kb + splits - 1) / splits;
  splits = csplit > 1 ? 1 : (num_kb + kbs - 1) / kbs;  // every split owns >= 1 K-block

  DnParams p = {};
  p.M = static_cast<int>(M); p.N = static_cast<int>(N); p.K = static_cast<int>(K);
  p.kb_per_split = kbs; p.num_kb = num_kb;
  p.ldo = a.ldo; p.out = a.out; p.meta = a.meta;
  p.nm28 = a.nm28 ? 1 : 0;
  p.dense_dw = a.dense_dw ? 1 : 0;
  p.accumulate = a.accumulate ? 1 : 0;
  p.atomic_out = 0;
  p.lo_off = a.lo_off;
  p.fold = a.fold;
  p.csplit = csplit;
  if (EPI == DenseEpi::MaskedWeightGrad && splits > 1) {
    p.atomic_out = 1;
    if (!a.accumulate) {
      if (cudaError_t e = launch_zero3(static_cast<float*>(a.out), static_cast<size_t>(M) * a.ldo, nullptr, 0,
                                       nullptr, 0, stream))
        return e;
    }
  }
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  p.tiles_m = tiles_m; p.tiles_n = tiles_n;
  p.num_tiles = tiles_m * tiles_n * splits;
  // with a cluster split, one cluster per tile (tiles * csplit <= SMs)
  const int grid = csplit > 1 ? p.num_tiles * csplit
                              : (p.num_tiles < sm_count() ? p.num_tiles : sm_count());
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  if (csplit > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  add_pdl_attr(cfg, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tA, tB, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// N tile for the skinny (rank-wide) products.
template <bool A_MN, bool B_MN, DenseEpi EPI>
cudaError_t run_rank(const DenseGemmArgs& a, cudaStream_t stream) {
  if (a.N <= 16) return run<A_MN, B_MN, 16, EPI>(a, stream);
  if (a.N <= 32) return run<A_MN, B_MN, 32, EPI>(a, stream);
  if (a.N <= 64) return run<A_MN, B_MN, 64, EPI>(a, stream);
  if (a.N <= 128) return run<A_MN, B_MN, 128, EPI>(a, stream);
  return run<A_MN, B_MN, 256, EPI>(a, stream);
}

}  // namespace

cudaError_t launch_zero3(float* a, size_t na, float* b, size_t nb, float* c, size_t nc,
                         cudaStream_t stream, float* d, size_t nd) {
  // counts in floats, each a multiple of 4 (16-byte aligned arrays)
  const int64_t n4 = static_cast<int64_t>((na + nb + nc + nd) / 4);
  if (n4 == 0) return cudaSuccess;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 4;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[1];
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  add_pdl_attr(cfg, attrs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, zero3_kernel, reinterpret_cast<float4*>(a), static_cast<int64_t>(na / 4),
                                     reinterpret_cast<float4*>(b), static_cast<int64_t>(nb / 4),
                                     reinterpret_cast<float4*>(c), static_cast<int64_t>(nc / 4),
                                     reinterpret_cast<float4*>(d), static_cast<int64_t>(nd / 4));
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dense_gemm(const DenseGemmArgs& a, cudaStream_t stream) {
  switch (a.epi) {
    case DenseEpi::MaskedWeightGrad:  // dW: A = dY (T x out), B = X (T x in), both MN-major
      if (a.a_mn_major && a.b_mn_major) {
        if ((a.M / kBM) % 2 == 0) return run_dw_pair(a, stream);  // CTA pairs on M-adjacent tiles
        return run<true, true, 256, DenseEpi::MaskedWeightGrad>(a, stream);
      }
      break;
    case DenseEpi::StoreBf16HiLo:  // XL = X·L (B MN-major) or G = dY·Rᵀ (B K-major)
      if (!a.a_mn_major && a.b_mn_major) return run_rank<false, true, DenseEpi::StoreBf16HiLo>(a, stream);
      if (!a.a_mn_major && !a.b_mn_major) return run_rank<false, false, DenseEpi::StoreBf16HiLo>(a, stream);
      break;
    case DenseEpi::AddF32:  // dL = Xᵀ·G
      if (a.a_mn_major && a.b_mn_major) return run_rank<true, true, DenseEpi::AddF32>(a, stream);
      break;
    case DenseEpi::AddF32Transposed:  // dRᵀ = dYᵀ·XL
      if (a.a_mn_major && a.b_mn_major) return run_rank<true, true, DenseEpi::AddF32Transposed>(a, stream);
      break;
  }
  return cudaErrorNotSupported;
}

}  // namespace slope
