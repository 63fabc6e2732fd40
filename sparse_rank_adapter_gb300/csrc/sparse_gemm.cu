// sparse_gemm.cu — 2:4-sparse tcgen05 GEMM with the low-rank adapter fused
// into the same TMEM accumulator (A3 forward, A4 input gradient).
//
// Source: "SLoPe: Double-Pruned Sparse Plus Lazy Low-Rank Adapter Pretraining
// of LLMs", §2.1 (sparse forward and, with the double-pruned transpose,
// sparse backward) and §2.4 / App. D (the adapter concatenated with the
// sparse weight and fused with the result addition, so one accumulator takes
// both).  Here the adapter is an extra dense K-segment: after the sparse
// K-loop, dense MMAs add A2·B2ᵀ into the same TMEM tile, once for the hi and
// once for the lo bf16 part of the rank-r intermediate.
//
//   D[m][n] = Σ_k A[m][k]·B[n][k] + Σ_j A2[m][j]·B2[n][j],   out[n][m] = D[m][n]
//
// The sparse operand has to be the MMA's A, so the weight rows are M and the
// tokens are N; the result is the transpose of the row-major output, which
// the epilogue writes directly (lane = m, so a warp's stores of one column
// n are 128 contiguous bytes).
//
// Two kernels.  sparse_gemm_kernel: one CTA per tile, persistent, one CTA
// per SM, tiles taken round-robin; it serves up to 128 tokens and weights
// with an odd number of 128-row tiles.  sparse_pair_kernel (below): CTA
// pairs on the pair-wide MMA for the large batches, with one 128-row weight
// tile per CTA, or two (256 rows apart) for long K-loops, where a stage's
// bytes then serve eight MMAs instead of four.
//
// Roles (576 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues
// the MMAs (one thread), warps 2..5 and 14..17 drain the accumulator (two
// warps per TMEM lane quadrant, alternate 32-column chunks, so that the
// epilogue of a tile stays shorter than the K-loop of the next even for
// short K), and two groups of four warps (6..9 for the even stages of the
// ring, 10..13 for the odd ones) move each stage's 2:4 metadata from shared
// memory into TMEM, so the short stages of narrow tiles do not wait on it.
// The accumulator is double-buffered in TMEM, so the epilogue of one tile
// overlaps the K-loop of the next.  Every mbarrier wait is bounded.
//
// Metadata in TMEM: k-step j (32 logical columns = 8 groups = one 32-bit
// word per row) of stage s sits in its own column META_COL + 16 s + 4 j, so
// every sparse MMA reads a 4-column-aligned address with sparsity selector 0.
// Within each 16-row block the hardware pairs rows i and i + 8 (i < 8) by
// 16-bit halves: lane i holds [row i groups 0-3 | row i+8 groups 0-3] and
// lane i + 8 holds [row i groups 4-7 | row i+8 groups 4-7] (measured with
// identity inputs on sm_103a).  One shuffle per word turns the row-major
// metadata into that arrangement.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "slope_internal.h"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

constexpr int kBM = 128;               // weight rows per tile (MMA M)
constexpr int kBKc = 64;               // compressed A columns per stage (= 128 logical K)
constexpr int kA_BYTES = kBM * 128;    // 16 KB: 128 rows x 128 B (SW128)
constexpr int kMETA_BYTES = kBM * 16;  // 2 KB: 128 rows x 16 B (32 groups)
constexpr int kThreads = 576;
constexpr int kEpiWarps = 8;

template <int BN>
struct SpCfg {
  static constexpr int B_BYTES = BN * 256;  // two 64-column SW128 atoms of BN rows
  static constexpr int STAGE = kA_BYTES + B_BYTES + kMETA_BYTES;
  // fp32 partial tile a cluster peer hands to its leader when a tile's K is
  // split over a cluster (column-major: [BN][128]).  A split cluster owns
  // exactly one tile, so by the time the partial exists every stage fill has
  // been consumed: the partial lives in the stage ring.
  static constexpr int RED_BYTES = kBM * BN * 4;
  static constexpr int STAGES_FIT = 200 * 1024 / STAGE;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC_COLS = BN < 32 ? 32 : BN;  // one accumulator buffer
  static constexpr int META_COL = 2 * ACC_COLS;        // after the two buffers
  static constexpr int TMEM_NEED = META_COL + 16 * STAGES;
  static constexpr int TMEM_COLS =
      TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int SMEM = STAGES * STAGE + 1024 /*barriers*/ + 1024 /*align slack*/;
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert(STAGES * STAGE >= RED_BYTES, "the split partial fits in the stage ring");
};

// Row-major metadata word of this lane's row -> the word the sparse MMA
// expects in this lane (rows i and i+8 of a 16-row block exchange halves).
__device__ __forceinline__ uint32_t pair_rows(uint32_t w, int lane) {
  const uint32_t p = __shfl_xor_sync(0xFFFFFFFFu, w, 8);
  return (lane & 8) ? ((p >> 16) | (w & 0xFFFF0000u)) : ((w & 0xFFFFu) | (p << 16));
}

struct SpParams {
  int M, N, K, r;
  int tiles_m, num_tiles;
  int group_m;     // M tiles (or pairs) per raster group: a band of weight tiles kept in L2
  int num_kb;      // sparse K-blocks (K / 128)
  int num_ab;      // adapter blocks per part (ceil(r / 64)); parts: hi, lo
  int out_bf16;
  int csplit;        // CTAs of a cluster that split one tile's K (one-CTA kernel); 1 = none
  int kb_per_split;  // sparse K-blocks per CTA of such a cluster
  void* out;
  unsigned int* status;
};

template <int BN, bool A2_MN>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmMeta,
                       const __grid_constant__ CUtensorMap tmA2,
                       const __grid_constant__ CUtensorMap tmB2, const SpParams p) {
  using C = SpCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty = full + C::STAGES;
  uint64_t* meta_full = empty + C::STAGES;
  uint64_t* acc_full = meta_full + C::STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* red_full = mma_done + 1;   // split leader: every peer's partial is in place
  uint64_t* red_empty = red_full + 1;  // split peer: the leader has read this CTA's partial
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(red_empty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* red = reinterpret_cast<float*>(smem);  // split partial, over the drained stage ring

  const int warp = warp_id(), lane = lane_id();
  // Cluster split of K (narrow tiles): CTA `crank` of the
  // cluster takes sparse K-blocks [crank * kb_per_split, ...); the last one
  // also runs the adapter steps.  Its fp32 partial goes to the leader.
  const int cs = p.csplit;
  const uint32_t crank = cs > 1 ? cluster_ctarank() : 0u;
  const int kb0 = cs > 1 ? static_cast<int>(crank) * p.kb_per_split : 0;
  const int nsp = cs > 1 ? min(p.num_kb - kb0, p.kb_per_split) : p.num_kb;
  const int nad = (cs == 1 || static_cast<int>(crank) == cs - 1) ? 2 * p.num_ab : 0;
  const int per_tile = nsp + nad;
  // step kk of a tile -> K-block index: sparse blocks kb0.., then the adapter
  // blocks, numbered from num_kb as in the unsplit tile
  auto kblock = [&](int kk) { return kk < nsp ? kb0 + kk : p.num_kb + (kk - nsp); };
  // Work units: tiles (one per cluster when K is split).
  const int units = p.num_tiles;
  const int unit0 = static_cast<int>(cs > 1 ? blockIdx.x / cs : blockIdx.x);
  const int ustep = static_cast<int>(cs > 1 ? gridDim.x / cs : gridDim.x);
  // Raster order: bands of group_m M tiles; within a band the M tiles turn
  // fastest, then the N tiles, so the band's weight tiles stay in L2 while
  // every token tile passes over them once.
  const int rows_m = p.tiles_m;
  const int tiles_n = units / rows_m;
  auto band = [&](int u, int& mi, int& ni) {
    const int per_band = p.group_m * tiles_n;
    const int b = u / per_band, w = u % per_band;
    const int first = b * p.group_m;
    const int gm = min(p.group_m, rows_m - first);
    mi = first + w % gm;
    ni = w / gm;
  };
  auto tile_m0 = [&](int u) {
    int mi, ni;
    band(u, mi, ni);
    return mi * kBM;
  };
  auto tile_n0 = [&](int u) {
    int mi, ni;
    band(u, mi, ni);
    return ni * BN;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&meta_full[s], 4);  // one arrival per metadata warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    mbar_init(red_full, kEpiWarps * (cs > 1 ? cs - 1 : 1));  // every epilogue warp of each peer
    mbar_init(red_empty, kEpiWarps);                         // the leader's epilogue warps
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  if (cs > 1)
    cluster_sync();  // the peers' barriers exist before any arrival reaches them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // With the adapter (r > 0) the kernel before this one on the stream is
  // the call's own rank-r GEMM, which produces only the adapter's B operand
  // (XL or G); its CTAs could start only after everything before it had
  // completed.  So the weights and tokens may be read at once and only the
  // TMA producer waits, before its first adapter load: the rank-r GEMM runs
  // alongside the sparse K-loop.  Without the adapter the predecessor is
  // unknown, and every thread waits here.
  if (p.r == 0) grid_dependency_wait();
  allow_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer -------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmMeta);
      bool dep_done = p.r == 0;
      int it = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep) {
        const int m0 = tile_m0(u);
        const int n0 = tile_n0(u);
        for (int kk = 0; kk < per_tile; ++kk, ++it) {
          const int kb = kblock(kk);
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { stop = true; break; }
          uint8_t* sA = smem + s * C::STAGE;
          uint8_t* sB = sA + kA_BYTES;
          uint8_t* sMeta = sB + C::B_BYTES;
          if (kb < p.num_kb) {
            mbar_arrive_expect_tx(&full[s], kA_BYTES + C::B_BYTES + kMETA_BYTES);
            tma_load_2d(sA, &tmA, &full[s], kb * kBKc, m0);
            tma_load_2d(sB, &tmB, &full[s], kb * 128, n0);
            tma_load_2d(sB + BN * 128, &tmB, &full[s], kb * 128 + 64, n0);
            tma_load_2d(sMeta, &tmMeta, &full[s], kb * 16, m0);
          } else {
            // adapter block c of part `part` (0 = hi, 1 = lo): rank columns
            // 64c .. 64c+63 of A2, and the same columns of that part of B2.
            // A2 rows/columns past r are zero-filled, so whatever B2 holds
            // past the part's r columns adds nothing.
            if (!dep_done) {  // the rank-r GEMM's output is visible from here
              grid_dependency_wait();
              dep_done = true;
            }
            const int a = kb - p.num_kb;
            const int part = a / p.num_ab, c = a % p.num_ab;
            mbar_arrive_expect_tx(&full[s], kA_BYTES + BN * 128);
            if (A2_MN) {  // R: r x M, two 64-wide M atoms of 64 rank rows
              tma_load_2d(sA, &tmA2, &full[s], m0, c * 64);
              tma_load_2d(sA + 8192, &tmA2, &full[s], m0 + 64, c * 64);
            } else {      // L: M x r, 128 rows of 64 rank columns
              tma_load_2d(sA, &tmA2, &full[s], c * 64, m0);
            }
            tma_load_2d(sB, &tmB2, &full[s], part * p.r + c * 64, n0);
          }
        }
      }
      // Leave no copy in flight: wait (bounded) for the last fill of each stage.
      for (int i = it - 1; i >= 0 && i >= it - C::STAGES; --i) {
        volatile int no_abort = 0;
        mbar_wait(&full[i % C::STAGES], (i / C::STAGES) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------- MMA issuer ---------
      const uint32_t id_sp = idesc_bf16(kBM, BN, false, false, true);
      const uint32_t id_ad = idesc_bf16(kBM, BN, A2_MN, false, false);
      const int r16 = (p.r + 15) / 16;  // dense K=16 steps of the adapter
      int it = 0, local = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep, ++local) {
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * C::ACC_COLS;
        for (int kk = 0; kk < per_tile; ++kk, ++it) {
          const int kb = kblock(kk);
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          // meta_full[s] completes once per fill of stage s (metadata or not),
          // so its phase parity always matches full[s]'s.
          if (!mbar_wait(&full[s], ph, abort_flag, p.status)) { stop = true; break; }
          if (!mbar_wait(&meta_full[s], ph, abort_flag, p.status)) { stop = true; break; }
          tc_fence_after();
          const uint32_t aA = smem_u32(smem + s * C::STAGE);
          const uint32_t aB = aA + kA_BYTES;
          if (kb < p.num_kb) {
            const uint32_t tmeta = tmem + C::META_COL + 16 * s;
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // 4 x (K = 32 logical)
              const uint64_t da = smem_desc(aA + j * 32, 0, 1024, kSwizzle128);
              const uint64_t db = smem_desc(aB + (j >> 1) * (BN * 128) + (j & 1) * 64, 0, 1024,
                                            kSwizzle128);
              mma_sp_bf16_ss(d, da, db, tmeta + 4 * j, id_sp, (kk > 0 || j > 0) ? 1u : 0u);
            }
          } else {
            const int c = (kb - p.num_kb) % p.num_ab;
            const int steps = min(4, r16 - 4 * c);
            for (int j = 0; j < steps; ++j) {
              const uint64_t da = A2_MN ? smem_desc(aA + j * 2048, 8192, 1024, kSwizzle128)
                                        : smem_desc(aA + j * 32, 0, 1024, kSwizzle128);
              const uint64_t db = smem_desc(aB + j * 32, 0, 1024, kSwizzle128);
              mma_bf16_ss(d, da, db, id_ad, 1u);
            }
          }
          mma_commit(&empty[s]);
        }
        if (!stop) mma_commit(&acc_full[buf]);
      }
      mma_commit(mma_done);
    }
  } else if (warp < 6 || warp >= 14) {
    // ------------------------------------------------ epilogue -----------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int half = warp >= 14 ? 1 : 0;  // which alternate column chunks
    int local = 0;
    for (int u = unit0; u < units; u += ustep, ++local) {
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      const int m = tile_m0(u) + 32 * q + lane;
      const int n0 = tile_n0(u);
      if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, p.status)) break;
      tc_fence_after();
      // cluster split of K: a peer first waits until the leader has read its
      // previous partial; the leader waits until every peer's is in place
      const bool peer = cs > 1 && crank != 0, leader = cs > 1 && crank == 0;
      if (peer && !mbar_wait_cluster(red_empty, (local & 1) ^ 1, abort_flag, p.status)) break;
      if (leader && !mbar_wait_cluster(red_full, local & 1, abort_flag, p.status)) break;
      const uint32_t trow = tmem + buf * C::ACC_COLS + (static_cast<uint32_t>(32 * q) << 16);
      constexpr int CH = BN < 32 ? BN : 32;
      if (half * CH >= BN) {  // no chunk for this warp: release the buffer at once
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
#pragma unroll 1
      for (int c0 = half * CH; c0 < BN; c0 += 2 * CH) {
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
        if (c0 + 2 * CH >= BN) {  // this warp's last chunk read: hand the buffer back early
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (cs > 1) {
          const int row = 32 * q + lane;
          if (peer) {  // hand the partial over; the leader stores
#pragma unroll
            for (int j = 0; j < CH; ++j) red[(c0 + j) * kBM + row] = __uint_as_float(v[j]);
            continue;
          }
          if (leader) {
            for (int pr = 1; pr < cs; ++pr) {
              const uint32_t base = mapa_shared(smem_u32(red), static_cast<uint32_t>(pr));
              // eight coalesced remote loads in flight (one 128-byte column
              // segment per warp each), then their adds
#pragma unroll
              for (int g = 0; g < CH; g += 8) {
                float t[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  t[j] = ld_shared_cluster_f32(base + 4u * ((c0 + g + j) * kBM + row));
#pragma unroll
                for (int j = 0; j < 8; ++j) v[g + j] = __float_as_uint(__uint_as_float(v[g + j]) + t[j]);
              }
            }
          }
        }
        const int nlim = p.N - (n0 + c0);
        if (p.out_bf16) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(n0 + c0) * p.M + m;
#pragma unroll
          for (int j = 0; j < CH; ++j)
            if (j < nlim) o[static_cast<size_t>(j) * p.M] = __float2bfloat16_rn(__uint_as_float(v[j]));
        } else {
          float* o = static_cast<float*>(p.out) + static_cast<size_t>(n0 + c0) * p.M + m;
#pragma unroll
          for (int j = 0; j < CH; ++j)
            if (j < nlim) o[static_cast<size_t>(j) * p.M] = __uint_as_float(v[j]);
        }
      }
      if (cs > 1) {
        // peer: the partial is written; leader: the peers' partials are read
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (peer) {
            mbar_arrive_cluster(mapa_shared(smem_u32(red_full), 0u));
          } else {
            for (int pr = 1; pr < cs; ++pr)
              mbar_arrive_cluster(mapa_shared(smem_u32(red_empty), static_cast<uint32_t>(pr)));
          }
        }
      }
    }
  } else {
    // ------------------------------------------------ metadata -> TMEM ---
    // Row m's 16 metadata bytes of stage s (4 k-steps) go to the 4 aligned
    // columns of that stage.  The stage's previous metadata is no longer in
    // use once its TMA fill has landed again (the refill waited for the
    // MMAs of the previous use).  Every fill of a stage is acknowledged on
    // meta_full, adapter fills (no metadata) included, so both barriers of a
    // stage move through the same phases.
    const int q = warp & 3;
    // Group g owns the stages of parity g and takes every fill of them in
    // order, so it never waits on a barrier more than one phase ahead (a
    // parity wait cannot tell phase p from phase p + 2).
    const int group = (warp - 6) >> 2;
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::META_COL;
    int it = 0;
    bool stop = false;
    for (int u = unit0; u < units && !stop; u += ustep) {
      for (int kk = 0; kk < per_tile; ++kk, ++it) {
        const int kb = kblock(kk);
        const int s = it % C::STAGES;
        if ((s & 1) != group) continue;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&full[s], ph, abort_flag, p.status)) { stop = true; break; }
        if (kb < p.num_kb) {  // adapter stages carry no metadata
          const uint4 w = *reinterpret_cast<const uint4*>(smem + s * C::STAGE + kA_BYTES +
                                                          C::B_BYTES + 16 * (32 * q + lane));
          const uint32_t col = tq + 16 * s;
          tmem_st_32x32b_x1(col + 0, pair_rows(w.x, lane));
          tmem_st_32x32b_x1(col + 4, pair_rows(w.y, lane));
          tmem_st_32x32b_x1(col + 8, pair_rows(w.z, lane));
          tmem_st_32x32b_x1(col + 12, pair_rows(w.w, lane));
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_full[s]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    // every MMA this CTA issued must be complete before its columns are released
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.status);
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // No CTA leaves while a peer may still read its partial or arrive on its
  // barriers.
  if (cs > 1) cluster_sync();
}

// Tiles that leave SMs idle split K over a cluster of up to 8 CTAs; the
// partials meet in the leader's registers.  The hand-over costs about 2.5 us,
// so each CTA keeps at least 16 sparse K-blocks.  Returns the CTAs per tile
// (1 = no split) and the sparse K-blocks each takes.
int split_of(int num_tiles, int num_kb, int* kb_per_split) {
  *kb_per_split = num_kb;
  if (num_tiles <= 0) return 1;
  int want = sm_count() / num_tiles;
  want = want < 8 ? want : 8;
  want = want < num_kb / 16 ? want : num_kb / 16;
  if (want < 2) return 1;
  *kb_per_split = (num_kb + want - 1) / want;
  return (num_kb + *kb_per_split - 1) / *kb_per_split;  // each CTA >= 1 block
}

// CTAs the one-CTA kernel keeps busy with BN-token tiles.
int busy_ctas(int64_t M, int64_t N, int64_t K, int bn) {
  const int tiles = static_cast<int>((M / kBM) * ((N + bn - 1) / bn));
  int per = 0;
  const int cs = split_of(tiles, static_cast<int>(K / 128), &per);
  if (cs > 1) return tiles * cs;
  return tiles < sm_count() ? tiles : sm_count();
}

template <int BN, bool A2_MN>
cudaError_t run(const SparseGemmArgs& a, cudaStream_t stream) {
  using C = SpCfg<BN>;
  auto kernel = sparse_gemm_kernel<BN, A2_MN>;
  static std::atomic<int> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  if (!attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1);
  }
  CUtensorMap tA, tB, tMeta, tA2, tB2;
  const uint64_t M = a.M, N = a.N, K = a.K, r = a.r;
  const uint32_t b_rows = BN;  // rows of B one TMA box brings
  bool ok = make_tmap_2d(&tA, a.a_vals, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K / 2, M, K, 64, kBM,
                         Swz::B128) &&
            make_tmap_2d(&tB, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, 2 * K, 64, b_rows,
                         Swz::B128) &&
            make_tmap_2d(&tMeta, a.a_meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 8, M, K / 8, 16,
                         kBM, Swz::None);
  if (r > 0) {
    ok = ok && (A2_MN ? make_tmap_2d(&tA2, a.a2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, r, 2 * M,
                                     64, 64, Swz::B128)
                      : make_tmap_2d(&tA2, a.a2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, r, M, 2 * r,
                                     64, kBM, Swz::B128));
    ok = ok && make_tmap_2d(&tB2, a.b2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2 * r, N, 4 * r, 64,
                            b_rows, Swz::B128);
  } else {
    tA2 = tA;  // unused
    tB2 = tB;
  }
  if (!ok) return cudaErrorInvalidValue;
  SpParams p;
  p.M = static_cast<int>(M); p.N = static_cast<int>(N); p.K = static_cast<int>(K);
  p.r = static_cast<int>(r);
  p.tiles_m = static_cast<int>(M / kBM);
  p.num_tiles = p.tiles_m * static_cast<int>((N + BN - 1) / BN);
  p.num_kb = static_cast<int>(K / 128);
  p.num_ab = static_cast<int>((r + 63) / 64);
  {  // a band of weight tiles (values + metadata, all of K) of about 40 MB
    const double tile_bytes = static_cast<double>(kBM) * K * 1.125;
    int g = static_cast<int>(40.0e6 / tile_bytes);
    p.group_m = g < 1 ? 1 : (g > p.tiles_m ? p.tiles_m : g);
  }
  p.out_bf16 = a.out_bf16 ? 1 : 0;
  p.csplit = split_of(p.num_tiles, p.num_kb, &p.kb_per_split);
  p.out = a.out;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  const int grid = p.csplit > 1 ? p.num_tiles * p.csplit  // one cluster per tile
                                 : (p.num_tiles < sm_count() ? p.num_tiles : sm_count());
  if (p.csplit > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.csplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cfg.gridDim = dim3(grid);
  add_pdl_attr(cfg, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tA, tB, tMeta, tA2, tB2, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Sparse GEMM on CTA pairs: the pair-wide sparse MMA (M = 256 = two 128-row
// weight tiles, one per CTA; N = BN tokens, of which each CTA holds half)
// halves the token bytes each SM takes in per flop, which is what bounds the
// one-CTA kernel at large sizes.  The even CTA issues the MMAs and owns the
// full barriers that both CTAs' operand loads signal.  Each CTA loads its own
// rows' metadata on a barrier of its own; its metadata warps copy them into
// its own TMEM (the pair MMA reads each CTA's metadata at the same column)
// and then arrive on the even CTA's meta_full.  The even CTA's commits
// release stages and accumulators in both CTAs; both CTAs' epilogue warps
// hand accumulator buffers back to the even CTA.
// ---------------------------------------------------------------------------

// MT = 2: each CTA holds two 128-row weight tiles 256 rows apart, so the
// pair computes two pair-wide 256-row tiles against the same token tile and
// a stage brings 2 x 16 KB of weights, one half token tile and 2 x 2 KB of
// metadata for eight MMAs: 30 % fewer bytes per flop, the bound of the
// MT = 1 kernel.  The two accumulators then fill TMEM with the metadata of
// three stages, so they are single-buffered: the next tile waits for the
// epilogue to read both.
template <int BN, int MT = 1>
struct Sp2Cfg {
  static constexpr int HB = BN / 2;              // token rows each CTA holds
  static constexpr int B_BYTES = HB * 256;       // two 64-column SW128 atoms of HB rows
  static constexpr int A_ALL = MT * kA_BYTES;    // the stage's weight tiles
  static constexpr int STAGE = A_ALL + B_BYTES + MT * kMETA_BYTES;
  static constexpr int NBUF = MT == 1 ? 2 : 1;   // accumulator buffers
  static constexpr int ACC_COLS = BN;            // per weight tile
  static constexpr int META_COL = NBUF * MT * ACC_COLS;
  static constexpr int META_STAGE = 16 * MT;     // metadata columns per stage
  static constexpr int STAGES_SMEM = (212 * 1024) / STAGE;
  static constexpr int STAGES_TMEM = (512 - META_COL) / META_STAGE;
  static constexpr int STAGES_FIT = STAGES_SMEM < STAGES_TMEM ? STAGES_SMEM : STAGES_TMEM;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int TMEM_NEED = META_COL + META_STAGE * STAGES;
  static constexpr int TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
  // output staging for the TMA stores: two 1 KB buffers per epilogue warp,
  // so one store can read its buffer while the next is filled
  static constexpr int STG_BYTES = 2048;
  // Stage s goes to metadata group s % 4, so with three stages or fewer the
  // fourth group (warps 22..25) has no stage: it joins the epilogue as a
  // third set, which drains the accumulators in two thirds of the time.
  static constexpr int EPI_SETS = STAGES <= 3 ? 3 : 2;
  static constexpr int EPI_WARPS = 4 * EPI_SETS;
  static constexpr int SMEM = STAGES * STAGE + 1024 /*barriers*/ + EPI_WARPS * STG_BYTES +
                              1024 /*align slack*/;
  static_assert(STAGE % 1024 == 0 && (HB * 128) % 1024 == 0, "1024-byte aligned atoms");
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert(MT == 1 || MT == 2, "one or two weight tiles per CTA");
  static_assert(BN > 32 * (EPI_SETS - 1), "every epilogue warp has a chunk");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// 26 warps: the 18 roles of the one-CTA kernel plus two more groups of four
// metadata warps (warps 18..25), so that four stages' metadata move into
// TMEM at once (stage s goes to group s % 4).  With three stages or fewer,
// warps 22..25 are a third set of epilogue warps instead.
constexpr int kThreadsPair = 832;

template <int BN, bool A2_MN, int MT>
__global__ void __launch_bounds__(kThreadsPair, 1)
    sparse_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmMeta,
                       const __grid_constant__ CUtensorMap tmA2,
                       const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ CUtensorMap tmOut, const SpParams p) {
  using C = Sp2Cfg<BN, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);  // even CTA's
  uint64_t* empty = full + C::STAGES;
  uint64_t* meta_ready = empty + C::STAGES;     // this CTA's metadata tile landed
  uint64_t* meta_full = meta_ready + C::STAGES; // even CTA's: both CTAs' metadata in TMEM
  uint64_t* acc_full = meta_full + C::STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;           // [2], counted in the even CTA
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const int per_tile = p.num_kb + 2 * p.num_ab;
  // units: groups of 2·MT M-adjacent tiles x token tiles
  const int units = p.num_tiles / (2 * MT);
  const int unit0 = static_cast<int>(blockIdx.x >> 1);
  const int ustep = static_cast<int>(gridDim.x >> 1);
  // Raster order as in the one-CTA kernel: bands of group_m M groups, the M
  // groups turning fastest within a band.
  const int rows_m = p.tiles_m / (2 * MT);
  const int tiles_n = units / rows_m;
  auto decode = [&](int u, int& m0, int& n0) {
    const int per_band = p.group_m * tiles_n;
    const int b = u / per_band, w = u % per_band;
    const int first = b * p.group_m;
    const int gm = min(p.group_m, rows_m - first);
    // this CTA's first 128 weight rows; its tile t (MT = 2) is 256 rows on
    m0 = (2 * MT * (first + w % gm) + static_cast<int>(rank)) * kBM;
    n0 = (w / gm) * BN;  // the pair's token tile
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&meta_ready[s], 1);
      mbar_init(&meta_full[s], 8);  // four metadata warps in each CTA
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * C::EPI_WARPS);  // the epilogue warps of both CTAs
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if (warp >= 6 && warp < 10) {
    // Every metadata column starts with a legal pattern (each group keeps
    // positions 0 and 1), so no MMA can ever meet an unwritten one.
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + C::META_COL;
    const uint32_t legal[4] = {0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u};
    for (int c = 0; c < C::META_STAGE * C::STAGES; c += 4) tmem_st_32x32b_x4(tq + c, legal);
    tmem_st_wait();
  }
  tc_fence_before();
  cluster_sync();  // every barrier of both CTAs exists before anything reaches it
  tc_fence_after();
  // With the adapter (r > 0) the kernel before this one on the stream is
  // the call's own rank-r GEMM, which produces only the adapter's B operand
  // (XL or G); its CTAs could start only after everything before it had
  // completed.  So the weights and tokens may be read at once and only the
  // TMA producer waits, before its first adapter load: the rank-r GEMM runs
  // alongside the sparse K-loop.  Without the adapter the predecessor is
  // unknown, and every thread waits here.
  if (p.r == 0) grid_dependency_wait();
  allow_dependents_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer -------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmMeta);
      bool dep_done = p.r == 0;
      int it = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep) {
        int m0, n0;
        decode(u, m0, n0);
        const int nb = n0 + static_cast<int>(rank) * C::HB;  // this CTA's half of the tokens
        for (int kb = 0; kb < per_tile; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { stop = true; break; }
          uint8_t* sA = smem + s * C::STAGE;
          uint8_t* sB = sA + C::A_ALL;
          uint8_t* sMeta = sB + C::B_BYTES;
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);  // the even CTA's barrier
          if (kb < p.num_kb) {
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (C::A_ALL + C::B_BYTES));
#pragma unroll
            for (int t = 0; t < MT; ++t) tma_load_2d_pair(sA + t * kA_BYTES, &tmA, bar, kb * kBKc, m0 + 256 * t);
            tma_load_2d_pair(sB, &tmB, bar, kb * 128, nb);
            tma_load_2d_pair(sB + C::HB * 128, &tmB, bar, kb * 128 + 64, nb);
            mbar_arrive_expect_tx(&meta_ready[s], MT * kMETA_BYTES);
#pragma unroll
            for (int t = 0; t < MT; ++t)
              tma_load_2d(sMeta + t * kMETA_BYTES, &tmMeta, &meta_ready[s], kb * 16, m0 + 256 * t);
          } else {
            // adapter block c of part `part` (0 = hi, 1 = lo), as in the
            // one-CTA kernel; each CTA brings its rows of A2 and its half of B2
            if (!dep_done) {  // the rank-r GEMM's output is visible from here
              grid_dependency_wait();
              dep_done = true;
            }
            const int a = kb - p.num_kb;
            const int part = a / p.num_ab, c = a % p.num_ab;
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (C::A_ALL + C::HB * 128));
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              uint8_t* sAt = sA + t * kA_BYTES;
              if (A2_MN) {
                tma_load_2d_pair(sAt, &tmA2, bar, m0 + 256 * t, c * 64);
                tma_load_2d_pair(sAt + 8192, &tmA2, bar, m0 + 256 * t + 64, c * 64);
              } else {
                tma_load_2d_pair(sAt, &tmA2, bar, c * 64, m0 + 256 * t);
              }
            }
            tma_load_2d_pair(sB, &tmB2, bar, part * p.r + c * 64, nb);
            mbar_arrive(&meta_ready[s]);  // no metadata in this stage
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------- MMA issuer ---------
      const uint32_t id_sp = idesc_bf16(2 * kBM, BN, false, false, true);
      const uint32_t id_ad = idesc_bf16(2 * kBM, BN, A2_MN, false, false);
      const int r16 = (p.r + 15) / 16;
      int it = 0, local = 0;
      bool stop = false;
      for (int u = unit0; u < units && !stop; u += ustep, ++local) {
        const int buf = local % C::NBUF;
        const uint32_t use = static_cast<uint32_t>(local / C::NBUF);
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * MT * C::ACC_COLS;  // tile t at + t * ACC_COLS
        for (int kb = 0; kb < per_tile; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&full[s], ph, abort_flag, p.status)) { stop = true; break; }
          // both CTAs' metadata of this fill is in TMEM (the odd CTA's
          // warps arrive with release at cluster scope)
          if (!mbar_wait_cluster(&meta_full[s], ph, abort_flag, p.status)) { stop = true; break; }
          tc_fence_after();
          const uint32_t aA = smem_u32(smem + s * C::STAGE);
          const uint32_t aB = aA + C::A_ALL;
          if (kb < p.num_kb) {
            const uint32_t tmeta = tmem + C::META_COL + C::META_STAGE * s;
#pragma unroll
            for (int t = 0; t < MT; ++t)
#pragma unroll
              for (int j = 0; j < 4; ++j) {  // 4 x (K = 32 logical)
                const uint64_t da = smem_desc(aA + t * kA_BYTES + j * 32, 0, 1024, kSwizzle128);
                const uint64_t db = smem_desc(aB + (j >> 1) * (C::HB * 128) + (j & 1) * 64, 0, 1024,
                                              kSwizzle128);
                mma_sp_bf16_ss_pair(d + t * C::ACC_COLS, da, db, tmeta + 16 * t + 4 * j, id_sp,
                                    (kb > 0 || j > 0) ? 1u : 0u);
              }
          } else {
            const int c = (kb - p.num_kb) % p.num_ab;
            const int steps = min(4, r16 - 4 * c);
#pragma unroll
            for (int t = 0; t < MT; ++t)
              for (int j = 0; j < steps; ++j) {
                const uint32_t aAt = aA + t * kA_BYTES;
                const uint64_t da = A2_MN ? smem_desc(aAt + j * 2048, 8192, 1024, kSwizzle128)
                                          : smem_desc(aAt + j * 32, 0, 1024, kSwizzle128);
                const uint64_t db = smem_desc(aB + j * 32, 0, 1024, kSwizzle128);
                mma_bf16_ss_pair(d + t * C::ACC_COLS, da, db, id_ad, 1u);
              }
          }
          mma_commit_pair_mc(&empty[s], 3);  // release the stage in both CTAs
        }
        if (!stop) mma_commit_pair_mc(&acc_full[buf], 3);
      }
      mma_commit_pair_mc(mma_done, 3);
    }
  } else if (warp < 6 || (warp >= 14 && warp < 18) || (C::EPI_SETS == 3 && warp >= 22)) {
    // ------------------------------------------------ epilogue -----------
    const int q = warp & 3;
    const int half = warp < 6 ? 0 : warp < 18 ? 1 : 2;  // this warp's set: chunks half, half + EPI_SETS, ...
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&acc_empty[0]), 0);
    // this warp's two 1 KB staging buffers: [token][32 weight rows] of the
    // output, 16 tokens (bf16) or 8 (fp32) at a time, each written out by a
    // TMA store; they alternate, so a store overlaps the next buffer's fill
    uint8_t* stg0 = smem + C::STAGES * C::STAGE + 1024 + (q + 4 * half) * C::STG_BYTES;
    int nstore = 0;
    int local = 0;
    for (int u = unit0; u < units; u += ustep, ++local) {
      int m0, n0;
      decode(u, m0, n0);
      const int buf = local % C::NBUF;
      const uint32_t use = static_cast<uint32_t>(local / C::NBUF);
      if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, p.status)) break;
      tc_fence_after();
#pragma unroll 1
      for (int t = 0; t < MT; ++t) {
      const uint32_t trow = tmem + (buf * MT + t) * C::ACC_COLS + (static_cast<uint32_t>(32 * q) << 16);
      const int mt = m0 + 256 * t;  // this tile's rows in this CTA
#pragma unroll 1
      for (int c0 = 32 * half; c0 < BN; c0 += 32 * C::EPI_SETS) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(trow + c0, v);
        tmem_ld_wait();
        if (t == MT - 1 && c0 + 32 * C::EPI_SETS >= BN) {  // this warp's last chunk read: hand the buffer back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8 * buf);
        }
        // stage 16 tokens (bf16) or 8 (fp32) at a time and store them
        auto buffer = [&]() {  // the next buffer, once the store that last used it has read it
          if (lane == 0) bulk_wait_read_but_one();
          __syncwarp();
          return stg0 + (nstore & 1) * 1024;
        };
        auto flush = [&](uint8_t* stg, int t0) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmOut, stg, mt + 32 * q, n0 + c0 + t0);  // tokens past N are clipped
            bulk_commit();
          }
          ++nstore;
        };
        if (p.out_bf16) {
#pragma unroll
          for (int g = 0; g < 32; g += 16) {
            __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(buffer());
#pragma unroll
            for (int j = 0; j < 16; ++j) sb[j * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[g + j]));
            flush(reinterpret_cast<uint8_t*>(sb), g);
          }
        } else {
#pragma unroll
          for (int g = 0; g < 32; g += 8) {
            float* sf = reinterpret_cast<float*>(buffer());
#pragma unroll
            for (int j = 0; j < 8; ++j) sf[j * 32 + lane] = __uint_as_float(v[g + j]);
            flush(reinterpret_cast<uint8_t*>(sf), g);
          }
        }
      }
      }
    }
    if (lane == 0) bulk_wait_all();
  } else {
    // ------------------------------------------------ metadata -> TMEM ---
    // As in the one-CTA kernel, on this CTA's own metadata and TMEM, with
    // four groups taking the stages by s % 4 (each group takes every fill
    // of its stages in order); the arrival goes to the even CTA's meta_full.
    const int q = warp & 3;
    const int group = warp < 14 ? (warp - 6) >> 2 : 2 + ((warp - 18) >> 2);
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::META_COL;
    const uint32_t meta_full0 = mapa_shared(smem_u32(&meta_full[0]), 0);
    int it = 0;
    bool stop = false;
    for (int u = unit0; u < units && !stop; u += ustep) {
      for (int kb = 0; kb < per_tile; ++kb, ++it) {
        const int s = it % C::STAGES;
        if ((s & 3) != group) continue;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&meta_ready[s], ph, abort_flag, p.status)) { stop = true; break; }
        if (kb < p.num_kb) {
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            const uint4 w = *reinterpret_cast<const uint4*>(smem + s * C::STAGE + C::A_ALL + C::B_BYTES +
                                                            t * kMETA_BYTES + 16 * (32 * q + lane));
            const uint32_t col = tq + C::META_STAGE * s + 16 * t;
            tmem_st_32x32b_x1(col + 0, pair_rows(w.x, lane));
            tmem_st_32x32b_x1(col + 4, pair_rows(w.y, lane));
            tmem_st_32x32b_x1(col + 8, pair_rows(w.z, lane));
            tmem_st_32x32b_x1(col + 12, pair_rows(w.w, lane));
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // the stores are complete (tcgen05.wait::st); the signal orders no
          // generic-memory writes, so the odd CTA arrives without a release
          if (rank == 0)
            mbar_arrive(&meta_full[s]);
          else
            mbar_arrive_cluster_relaxed(meta_full0 + 8 * s);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    volatile int no_abort = 0;
    mbar_wait(mma_done, 0, &no_abort, p.status);
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
  cluster_sync();  // no CTA leaves while its peer may still signal it or read its TMEM
}

template <int BN, bool A2_MN, int MT = 1>
cudaError_t run_pair2(const SparseGemmArgs& a, cudaStream_t stream) {
  using C = Sp2Cfg<BN, MT>;
  auto kernel = sparse_pair_kernel<BN, A2_MN, MT>;
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
  cfg.blockDim = dim3(kThreadsPair);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  if (!attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(2 * (sm_count() / 2));
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters[dev].store(n > 0 ? n : 1);
    attr_set[dev].store(1);
  }
  CUtensorMap tA, tB, tMeta, tA2, tB2;
  const uint64_t M = a.M, N = a.N, K = a.K, r = a.r;
  const uint32_t b_rows = BN / 2;  // rows of B one CTA's TMA box brings
  bool ok = make_tmap_2d(&tA, a.a_vals, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K / 2, M, K, 64, kBM,
                         Swz::B128) &&
            make_tmap_2d(&tB, a.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, 2 * K, 64, b_rows,
                         Swz::B128) &&
            make_tmap_2d(&tMeta, a.a_meta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 8, M, K / 8, 16,
                         kBM, Swz::None);
  if (r > 0) {
    ok = ok && (A2_MN ? make_tmap_2d(&tA2, a.a2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, r, 2 * M,
                                     64, 64, Swz::B128)
                      : make_tmap_2d(&tA2, a.a2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, r, M, 2 * r,
                                     64, kBM, Swz::B128));
    ok = ok && make_tmap_2d(&tB2, a.b2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 2 * r, N, 4 * r, 64,
                            b_rows, Swz::B128);
  } else {
    tA2 = tA;  // unused
    tB2 = tB;
  }
  // output: N x M (tokens x weight rows), boxes of 32 rows x 16 (bf16) or
  // 8 (fp32) tokens
  CUtensorMap tOut;
  ok = ok && (a.out_bf16 ? make_tmap_2d(&tOut, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, N,
                                        2 * M, 32, 16, Swz::None)
                         : make_tmap_2d(&tOut, a.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, N,
                                        4 * M, 32, 8, Swz::None));
  if (!ok) return cudaErrorInvalidValue;
  SpParams p = {};
  p.M = static_cast<int>(M); p.N = static_cast<int>(N); p.K = static_cast<int>(K);
  p.r = static_cast<int>(r);
  p.tiles_m = static_cast<int>(M / kBM);  // a multiple of 2·MT
  p.num_tiles = p.tiles_m * static_cast<int>((N + BN - 1) / BN);
  p.num_kb = static_cast<int>(K / 128);
  p.num_ab = static_cast<int>((r + 63) / 64);
  {  // a band of weight-tile groups (values + metadata, all of K) of about 40 MB
    const double tile_bytes = 2.0 * MT * kBM * K * 1.125;
    int g = static_cast<int>(40.0e6 / tile_bytes);
    const int rows = p.tiles_m / (2 * MT);
    p.group_m = g < 1 ? 1 : (g > rows ? rows : g);
  }
  p.out_bf16 = a.out_bf16 ? 1 : 0;
  p.csplit = 1;
  p.kb_per_split = p.num_kb;
  p.out = a.out;
  p.status = device_status_ptr();
  if (!p.status) return cudaErrorInvalidDevicePointer;
  const int units = p.num_tiles / (2 * MT);
  const int clusters = units < max_clusters[dev].load() ? units : max_clusters[dev].load();
  cfg.gridDim = dim3(2 * clusters);
  add_pdl_attr(cfg, attr);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tA, tB, tMeta, tA2, tB2, tOut, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// N tile by token count: the smallest tile that covers small batches (up to
// 128 tokens; while the weight has fewer 128-row tiles than there are SMs,
// 128-token tiles with K split over a cluster, unless 64-token tiles keep
// more SMs busy); for large
// batches CTA pairs with 224- or 128-token tiles (an even number of weight
// tiles), else one CTA with 192 (the widest that still double-buffers in
// TMEM beside the metadata) unless 128 gives the grid noticeably more tiles.
template <bool A2_MN>
cudaError_t dispatch(const SparseGemmArgs& a, cudaStream_t stream) {
  if (a.N <= 16) return run<16, A2_MN>(a, stream);
  if (a.N <= 64) return run<64, A2_MN>(a, stream);
  const int64_t tiles_m = a.M / kBM;
  const bool pair = tiles_m % 2 == 0;  // clusters pair M-adjacent tiles
  if (a.N <= 128 && tiles_m < sm_count()) {
    // 128-token tiles read each weight row once; 64-token ones twice, but
    // they give twice the tiles when K is too short to split over a cluster
    const bool wide = busy_ctas(a.M, a.N, a.K, 128) >= busy_ctas(a.M, a.N, a.K, 64);
    return wide ? run<128, A2_MN>(a, stream) : run<64, A2_MN>(a, stream);
  }
  if (a.N <= 128)
    return pair ? run_pair2<128, A2_MN>(a, stream) : run<128, A2_MN>(a, stream);
  if (pair) {
    // CTA pairs: 224 or 128 tokens per tile, whichever needs fewer rounds of
    // the pairs the GPU holds, counting 32 columns' worth of fixed cost per
    // tile; or two weight tiles per CTA with 192 tokens (when the weight has
    // a multiple of four 128-row tiles), whose stages move 30 % fewer bytes
    // per flop, counted as 1.4 times the throughput per column.  Its
    // single-buffered accumulators expose one epilogue per tile, which only
    // a long K-loop (K >= 4096) amortises.
    const int64_t clusters = sm_count() / 2;
    auto cost = [&](int64_t bn, int64_t mt) {
      const int64_t units = (tiles_m / (2 * mt)) * ((a.N + bn - 1) / bn);
      const double c = static_cast<double>((units + clusters - 1) / clusters) * mt * (bn + 32);
      return mt == 2 ? c / 1.4 : c;
    };
    const double c224 = cost(224, 1), c128 = cost(128, 1);
    if (tiles_m % 4 == 0 && a.K >= 4096 && cost(192, 2) < (c224 < c128 ? c224 : c128))
      return run_pair2<192, A2_MN, 2>(a, stream);
    return c224 <= c128 ? run_pair2<224, A2_MN>(a, stream) : run_pair2<128, A2_MN>(a, stream);
  }
  const int64_t t192 = tiles_m * ((a.N + 191) / 192);
  if (t192 < 2 * sm_count()) return run<128, A2_MN>(a, stream);
  return run<192, A2_MN>(a, stream);
}

}  // namespace

cudaError_t launch_sparse_gemm(const SparseGemmArgs& a, cudaStream_t stream) {
  return a.a2_mn_major ? dispatch<true>(a, stream) : dispatch<false>(a, stream);
}

}  // namespace slope
