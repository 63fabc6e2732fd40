// mma_rate.cu — tensor-core rate self test.
//
// Measures the rate the GEMM kernels are judged against: every SM (or SM
// pair) issues rounds of four back-to-back tcgen05.mma instructions of
// kind::f16 (bf16 operands, fp32 accumulation, N = 256) on operands that
// stay in shared memory, so nothing but the tensor pipe limits it.  The
// variants are the ones the path's kernels use: dense (K = 16 per
// instruction) and 2:4 sparse (.sp, K = 32 dense-equivalent, metadata in
// TMEM: one fixed pattern, or random legal pairs as pruned weights have), on
// one SM (M = 128) or on an SM pair (cta_group::2, M = 256).  The
// operand layouts and descriptors are those of the path's kernels: 128-byte
// swizzled K-major atoms, the sparse B operand in two atoms of 64 K each.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "slope_internal.h"
#include "sm103_ptx.cuh"

namespace slope {
namespace {

constexpr int kRateThreads = 128;
constexpr int kRateN = 256;
// Shared memory asked for at launch: more than half an SM's, so one CTA
// (and its 512 TMEM columns) per SM.
constexpr int kRateSmem = 120 * 1024;
constexpr uint32_t kRateMetaCol = kRateN;  // sparse metadata columns, after the accumulator

template <bool SPARSE, bool PAIR>
struct RateCfg {
  static constexpr int A_BYTES = 128 * 128;              // 128 rows x one 128 B atom
  static constexpr int B_ROWS = PAIR ? kRateN / 2 : kRateN;  // this CTA's rows of B
  static constexpr int B_ATOMS = SPARSE ? 2 : 1;         // 64 K per atom
  static constexpr int B_BYTES = B_ATOMS * B_ROWS * 128;
  static constexpr int M = PAIR ? 256 : 128;
  static constexpr int K_STEP = SPARSE ? 32 : 16;        // dense-equivalent K per instruction
  static_assert(1024 + A_BYTES + B_BYTES + 1024 <= kRateSmem, "operands fit");
};

// A legal 2:4 metadata nibble (i0 | i1 << 2, i0 < i1) picked by x % 6.
__device__ __forceinline__ uint32_t legal_nibble(uint32_t x) {
  const uint32_t i = x % 6u;
  const uint32_t i0 = i < 3u ? 0u : (i < 5u ? 1u : 2u);
  const uint32_t i1 = i < 3u ? i + 1u : (i < 5u ? i - 1u : 3u);
  return i0 | (i1 << 2);
}

template <bool SPARSE, bool PAIR>
__global__ void __launch_bounds__(kRateThreads, 1) mma_rate_kernel(int64_t iters, int random_meta,
                                                                   unsigned int* status) {
  using C = RateCfg<SPARSE, PAIR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::A_BYTES;
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const int warp = warp_id(), lane = lane_id();
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;

  // operands: pseudo-random bf16 of magnitude in [2^-7, 2^-6), either sign
  // (a 32-bit LCG per word)
  for (int i = threadIdx.x; i < (C::A_BYTES + C::B_BYTES) / 4; i += kRateThreads) {
    uint32_t x = 1664525u * (static_cast<uint32_t>(i) + 977u * blockIdx.x) + 1013904223u;
    x ^= x >> 15;
    const uint32_t lo = 0x3C00u | (x & 0x807Fu), hi = 0x3C00u | ((x >> 16) & 0x807Fu);
    reinterpret_cast<uint32_t*>(smem)[i] = lo | (hi << 16);
  }
  fence_proxy_async_smem();  // the tensor core reads what the threads wrote
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&tmem_holder, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_holder, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  if constexpr (SPARSE) {
    // the 16 metadata columns of the four k-steps: every group keeps
    // positions 0 and 1, or (random_meta) each group one of the six legal
    // pairs at random, as pruned weights have
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * warp) << 16) + kRateMetaCol;
    for (int c = 0; c < 16; c += 4) {
      uint32_t words[4] = {0x44444444u, 0x44444444u, 0x44444444u, 0x44444444u};
      if (random_meta) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t x = 2654435761u * (threadIdx.x + 131u * (c + k) + 7919u * blockIdx.x) + 12345u;
          uint32_t w = 0;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            x = 1664525u * x + 1013904223u;
            w |= legal_nibble(x >> 8) << (4 * g);
          }
          words[k] = w;
        }
      }
      tmem_st_32x32b_x4(tq + c, words);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync(); else __syncthreads();
  tc_fence_after();

  if (warp == 1 && lane == 0 && rank == 0) {
    const uint32_t id = idesc_bf16(C::M, kRateN, false, false, SPARSE);
    const uint32_t aA = smem_u32(sA), aB = smem_u32(sB);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t acc = (it > 0 || j > 0) ? 1u : 0u;
        const uint64_t da = smem_desc(aA + j * 32, 0, 1024, kSwizzle128);
        if constexpr (SPARSE) {
          const uint64_t db = smem_desc(aB + (j >> 1) * (C::B_ROWS * 128) + (j & 1) * 64, 0, 1024,
                                        kSwizzle128);
          if constexpr (PAIR) mma_sp_bf16_ss_pair(tmem, da, db, tmem + kRateMetaCol + 4 * j, id, acc);
          else mma_sp_bf16_ss(tmem, da, db, tmem + kRateMetaCol + 4 * j, id, acc);
        } else {
          const uint64_t db = smem_desc(aB + j * 32, 0, 1024, kSwizzle128);
          if constexpr (PAIR) mma_bf16_ss_pair(tmem, da, db, id, acc);
          else mma_bf16_ss(tmem, da, db, id, acc);
        }
      }
    }
    if constexpr (PAIR) mma_commit_pair_mc(&done, 3);
    else mma_commit(&done);
  }
  __syncwarp();
  if (warp == 1) {
    // bounded: a wait that runs out records a timeout and returns
    mbar_wait(&done, 0, abort_flag, status);
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
  if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
}

template <bool SPARSE, bool PAIR>
cudaError_t run_rate(int64_t iters, int random_meta, double* flops, cudaStream_t stream) {
  using C = RateCfg<SPARSE, PAIR>;
  auto kernel = mma_rate_kernel<SPARSE, PAIR>;
  static std::atomic<int> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1);
  }
  unsigned int* status = device_status_ptr();
  if (!status) return cudaErrorUnknown;
  const int sms = sm_count();
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kRateThreads);
  cfg.dynamicSmemBytes = kRateSmem;
  cfg.stream = stream;
  int issuers = sms;
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    cfg.gridDim = dim3(2);
    cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) clusters = 1;
    if (clusters > sms / 2) clusters = sms / 2;
    issuers = clusters;
    cfg.gridDim = dim3(2 * clusters);
  } else {
    cfg.gridDim = dim3(sms);
  }
  *flops = static_cast<double>(issuers) * static_cast<double>(iters) * 4.0 * 2.0 * C::M * kRateN * C::K_STEP;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, iters, random_meta, status);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma_rate(int kind, bool pair, int64_t iters, double* flops,
                            cudaStream_t stream) {
  const int rnd = kind == 2 ? 1 : 0;
  if (kind > 0)
    return pair ? run_rate<true, true>(iters, rnd, flops, stream) : run_rate<true, false>(iters, rnd, flops, stream);
  return pair ? run_rate<false, true>(iters, 0, flops, stream) : run_rate<false, false>(iters, 0, flops, stream);
}

}  // namespace slope
