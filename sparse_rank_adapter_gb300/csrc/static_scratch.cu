// static_scratch.cu — the sparse forward for callers that cannot allocate
// device memory.
//
// slope_linear_fwd keeps the rank-r plane (X·L as hi/lo bf16, T x 2r) in a
// buffer the caller passes: XL, or the workspace when XL is NULL.  Some
// callers have neither to give.  A plugin running inside a host runtime
// that owns every device allocation gets only its inputs and outputs, and a
// serving loop that must never call cudaMalloc on its hot path (it can
// synchronise the device and stall other streams) has no workspace to hand
// over either.  For them this file keeps the plane in a fixed array of
// device memory that the library itself declares, so no call allocates.
//
// The array lives in every GPU's memory from the moment the library's
// module is loaded on that GPU until the process exits.  Its device address
// is taken once per device (the entry point's first call on that device),
// with that device current; in host code the array's name only stands for
// the symbol and is never passed to a kernel.  The entry point then runs
// the same calls as slope_linear_fwd with XL = NULL and the array as the
// workspace: the kernels, and so the results, are the same.
//
// No counterpart on the SLoPe pages: this is a deployment variant of the
// forward (A3), not a step of the method.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/slope.h"

namespace {

// The forward's rank-r plane: 4·T·r bytes.  Nothing in it needs to start at
// zero (the rank-r GEMM writes every byte the sparse GEMM reads), and every
// call overwrites it.
static __device__ __align__(256) uint8_t g_static_scratch[SLOPE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the array on the current device (resolved once per
// device, with that device current), or NULL on a CUDA error.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* q = nullptr;
  if (cudaGetSymbolAddress(&q, g_static_scratch) != cudaSuccess || q == nullptr) return nullptr;
  g_scratch_addr[dev].store(q, std::memory_order_release);
  return q;
}

}  // namespace

extern "C" int slope_linear_fwd_static_scratch(const void* X, int64_t T, int64_t in, int64_t out,
                                               const void* Wv, const uint8_t* Wm, const void* L,
                                               const void* R, int r, void* Y, int y_dtype,
                                               void* stream) {
  // No adapter (nothing to keep), no tokens (nothing to do), or sizes the
  // forward refuses: the plain forward, which needs no plane, does or
  // reports it.
  const size_t need = (r > 0 && T > 0) ? slope_workspace_size(T, in, out, r) : 0;
  if (need == 0)
    return slope_linear_fwd(X, T, in, out, Wv, Wm, L, R, r, Y, y_dtype, nullptr, nullptr, 0,
                            stream);
  // Sizes beyond the array are refused before anything touches the GPU.
  if (need > SLOPE_STATIC_SCRATCH_BYTES) return SLOPE_ERR_SHAPE;
  void* scratch = scratch_on_current_device();
  if (!scratch) return SLOPE_ERR_CUDA;
  return slope_linear_fwd(X, T, in, out, Wv, Wm, L, R, r, Y, y_dtype, nullptr, scratch,
                          SLOPE_STATIC_SCRATCH_BYTES, stream);
}
