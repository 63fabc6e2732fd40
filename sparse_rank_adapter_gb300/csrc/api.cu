// api.cu — the C ABI declared in include/slope.h: argument validation,
// device checks, tensor-map encoding and kernel launches.  Every step of
// the computation runs in this library's kernels; nothing here computes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/slope.h"
#include "slope_internal.h"
#include "sm103_ptx.cuh"

namespace slope {

// --------------------------------------------------------- device state ---

constexpr int kMaxDevices = 64;

namespace {
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_device_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
}  // namespace

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 148;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int choose_splits(int tiles, int slots, int num_kb) {
  if (tiles <= 0 || slots <= 0 || num_kb <= 0) return 1;
  const int max_split = num_kb / 4 > 0 ? num_kb / 4 : 1;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= max_split; ++s) {
    const long long waves = (static_cast<long long>(tiles) * s + slots - 1) / slots;
    const long long per_unit = (num_kb + s - 1) / s + (s > 1 ? 8 : 4);
    const long long cost = waves * per_unit + (s > 1 ? 8 : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// The kernels are built for sm_103a only; any other device is refused.
static int check_device() {
  const int dev = current_device();
  if (dev < 0) return SLOPE_ERR_CUDA;
  int ok = g_device_ok[dev].load(std::memory_order_relaxed);
  if (ok == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SLOPE_ERR_CUDA;
    ok = (major == 10 && minor == 3) ? 1 : -1;
    g_device_ok[dev].store(ok, std::memory_order_relaxed);
  }
  return ok == 1 ? SLOPE_OK : SLOPE_ERR_UNSUPPORTED;
}

// ------------------------------------------------------- tensor maps ------

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::atomic<EncodeTiledFn> g_encode{nullptr};

EncodeTiledFn encode_fn() {
  EncodeTiledFn f = g_encode.load(std::memory_order_acquire);
  if (f) return f;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr)
    return nullptr;
  f = reinterpret_cast<EncodeTiledFn>(p);
  g_encode.store(f, std::memory_order_release);
  return f;
}
}  // namespace

// Encoded tensor maps, cached by everything that goes into them (address,
// element type, extents, row stride, box, swizzle): a hit is exactly the map
// that encoding would produce, so a call on the same buffers skips the
// driver's encoder.  Direct-mapped, 256 entries, one lock.
namespace {
struct TmapKey {
  const void* base;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  int dtype, swz;
  bool operator==(const TmapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes &&
           box_inner == o.box_inner && box_outer == o.box_outer && dtype == o.dtype && swz == o.swz;
  }
};
struct TmapSlot {
  bool used = false;
  TmapKey key;
  CUtensorMap map;
};
constexpr int kTmapSlots = 256;
TmapSlot g_tmap_cache[kTmapSlots];
std::mutex g_tmap_mutex;

size_t tmap_hash(const TmapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
  for (uint64_t v : {k.inner, k.outer, k.row_bytes, uint64_t(k.box_inner) << 32 | k.box_outer,
                     uint64_t(k.dtype) << 8 | uint64_t(k.swz)})
    h = (h ^ v) * 0x100000001B3ull;
  return static_cast<size_t>(h >> 32) % kTmapSlots;
}
}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                  uint32_t box_outer, Swz swz) {
  (void)elem_bytes;
  const TmapKey key{base, inner, outer, row_bytes, box_inner, box_outer, static_cast<int>(dtype),
                    static_cast<int>(swz)};
  const size_t slot = tmap_hash(key);
  {
    std::lock_guard<std::mutex> lock(g_tmap_mutex);
    if (g_tmap_cache[slot].used && g_tmap_cache[slot].key == key) {
      *map = g_tmap_cache[slot].map;
      return true;
    }
  }
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle s = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swz == Swz::B32) s = CU_TENSOR_MAP_SWIZZLE_32B;
  if (swz == Swz::B64) s = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swz == Swz::B128) s = CU_TENSOR_MAP_SWIZZLE_128B;
  std::memset(map, 0, sizeof(*map));
  const CUresult r =
      f(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
        CU_TENSOR_MAP_INTERLEAVE_NONE, s, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(g_tmap_mutex);
  g_tmap_cache[slot].used = true;
  g_tmap_cache[slot].key = key;
  g_tmap_cache[slot].map = *map;
  return true;
}

// ----------------------------------------------------- status word --------

namespace {
__device__ unsigned int g_status_word;
std::atomic<unsigned int*> g_status_ptr[kMaxDevices];
}  // namespace

unsigned int* device_status_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  unsigned int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* q = nullptr;
  if (cudaGetSymbolAddress(&q, g_status_word) != cudaSuccess) return nullptr;
  p = static_cast<unsigned int*>(q);
  g_status_ptr[dev].store(p, std::memory_order_release);
  return p;
}

// A wait that nothing will end: one thread waits, with the given limit, on
// a fresh mbarrier no one arrives on, through the same bounded wait every
// pipeline kernel uses, which records the timeout in the status word.
__global__ void wait_timeout_probe_kernel(unsigned int* status, long long limit_cycles) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, limit_cycles);
}

}  // namespace slope

// ================================================================ C ABI ===

using namespace slope;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int from_cuda(cudaError_t e) { return e == cudaSuccess ? SLOPE_OK : SLOPE_ERR_CUDA; }

extern "C" const char* slope_status_string(int s) {
  switch (s) {
    case SLOPE_OK: return "ok";
    case SLOPE_ERR_INVALID_ARG: return "invalid argument";
    case SLOPE_ERR_SHAPE: return "unsupported shape";
    case SLOPE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SLOPE_ERR_UNSUPPORTED: return "unsupported device or n:m pattern";
    case SLOPE_ERR_CUDA: return "CUDA error";
    case SLOPE_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

extern "C" int slope_version(void) { return 10000; }

// Scratch of the two sparse-product calls: the T x 2r bf16 plane of the
// rank-r intermediate (XL or G, hi parts then lo parts) when the caller does
// not keep it, rounded up to 256 bytes.  The weight-gradient call uses the
// first kWaveSyncBytes of a workspace, when given, for the counter that
// keeps its waves of tiles in step.
constexpr size_t kWaveSyncBytes = 16;

static size_t plane_bytes(int64_t T, int r) {
  const size_t b = static_cast<size_t>(T) * static_cast<size_t>(2 * r) * 2;
  return (b + 255) & ~static_cast<size_t>(255);
}

extern "C" size_t slope_workspace_size(int64_t T, int64_t in, int64_t out, int r) {
  if (T < 0 || in <= 0 || out <= 0 || in % 128 != 0 || out % 128 != 0) return 0;
  if (r < 0 || r > 256 || r % 8 != 0 || T > (int64_t(1) << 31) - 1) return 0;
  const size_t plane = r > 0 ? plane_bytes(T, r) : 0;
  return plane > 256 ? plane : 256;
}

// The rank-r plane of a sparse-product call: the caller's output when given,
// else the front of the workspace, which must then hold plane_bytes(T, r).
static int rank_plane(void* given, void* workspace, size_t workspace_bytes, int64_t T, int r,
                      void** plane) {
  *plane = given;
  if (r == 0 || given) return SLOPE_OK;
  if (!workspace || workspace_bytes < plane_bytes(T, r)) return SLOPE_ERR_INVALID_ARG;
  *plane = workspace;
  return SLOPE_OK;
}

// The N:M patterns the library prunes: 2:4, 1:2 (written in the 2:4
// format) and 2:8 (its own format).
static bool known_pattern(int n, int m) {
  return (n == 2 && m == 4) || (n == 1 && m == 2) || (n == 2 && m == 8);
}

extern "C" int slope_prune_nm(const void* W, int64_t rows, int64_t cols, int n, int m, void* vals,
                              uint8_t* meta, void* stream) {
  if (!known_pattern(n, m)) return SLOPE_ERR_UNSUPPORTED;
  if (rows < 0 || cols <= 0 || cols % 8 != 0) return SLOPE_ERR_SHAPE;
  if (rows == 0) return SLOPE_OK;
  if (!W || !vals || !meta) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(vals) || !aligned16(meta)) return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (m == 8) return from_cuda(launch_prune28(W, rows, cols, vals, meta, st));
  if (m == 2) return from_cuda(launch_prune12(W, rows, cols, vals, meta, st));
  return from_cuda(launch_prune24(W, rows, cols, vals, meta, st));
}

extern "C" int slope_double_prune_nm(const void* vals, const uint8_t* meta, int64_t rows,
                                     int64_t cols, int n, int m, void* t_vals, uint8_t* t_meta,
                                     void* stream) {
  if (!known_pattern(n, m)) return SLOPE_ERR_UNSUPPORTED;
  if (m == 4) return slope_double_prune(vals, meta, rows, cols, t_vals, t_meta, stream);
  if (rows <= 0 || cols <= 0 || rows % 8 != 0 || cols % 16 != 0) return SLOPE_ERR_SHAPE;
  if (!vals || !meta || !t_vals || !t_meta) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(vals) || !aligned16(meta) || !aligned16(t_vals) || !aligned16(t_meta))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (m == 8) return from_cuda(launch_double_prune28(vals, meta, rows, cols, t_vals, t_meta, st));
  return from_cuda(launch_double_prune12(vals, meta, rows, cols, t_vals, t_meta, st));
}

extern "C" int slope_expand_nm_to_24(const void* vals, const uint8_t* meta, int64_t rows,
                                     int64_t cols, int n, int m, void* vals24, uint8_t* meta24,
                                     void* stream) {
  if (n != 2 || m != 8) return SLOPE_ERR_UNSUPPORTED;
  if (rows < 0 || cols <= 0 || cols % 8 != 0) return SLOPE_ERR_SHAPE;
  if (rows == 0) return SLOPE_OK;
  if (!vals || !meta || !vals24 || !meta24) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(vals) || !aligned16(meta) || !aligned16(vals24) || !aligned16(meta24))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_expand28(vals, meta, rows, cols, vals24, meta24,
                                   static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_double_prune(const void* vals, const uint8_t* meta, int64_t rows,
                                  int64_t cols, void* t_vals, uint8_t* t_meta, void* stream) {
  if (rows <= 0 || cols <= 0 || rows % 8 != 0 || cols % 16 != 0) return SLOPE_ERR_SHAPE;
  if (!vals || !meta || !t_vals || !t_meta) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(vals) || !aligned16(meta) || !aligned16(t_vals) || !aligned16(t_meta))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_double_prune24(vals, meta, rows, cols, t_vals, t_meta,
                                         static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_prune_and_double_prune(const void* W, int64_t rows, int64_t cols, int n,
                                            int m, void* vals, uint8_t* meta, void* t_vals,
                                            uint8_t* t_meta, void* stream) {
  if (n != 2 || m != 4) return SLOPE_ERR_UNSUPPORTED;
  if (rows <= 0 || cols <= 0 || rows % 8 != 0 || cols % 16 != 0) return SLOPE_ERR_SHAPE;
  if (!W || !vals || !meta || !t_vals || !t_meta) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(vals) || !aligned16(meta) || !aligned16(t_vals) ||
      !aligned16(t_meta))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_prune_double24(W, rows, cols, vals, meta, t_vals, t_meta,
                                         static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_recompress_double_prune(const void* W, const uint8_t* meta, int64_t rows,
                                             int64_t cols, void* vals, void* t_vals,
                                             uint8_t* t_meta, void* stream) {
  if (rows <= 0 || cols <= 0 || rows % 8 != 0 || cols % 16 != 0) return SLOPE_ERR_SHAPE;
  if (!W || !meta || !vals || !t_vals || !t_meta) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(meta) || !aligned16(vals) || !aligned16(t_vals) ||
      !aligned16(t_meta))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_recompress_double24(W, meta, rows, cols, vals, t_vals, t_meta,
                                              static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_double_prune_frozen(const void* vals, const uint8_t* meta, int64_t rows,
                                         int64_t cols, const uint8_t* t_meta, void* t_vals,
                                         void* stream) {
  if (rows <= 0 || cols <= 0 || rows % 8 != 0 || cols % 16 != 0) return SLOPE_ERR_SHAPE;
  if (!vals || !meta || !t_meta || !t_vals) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(vals) || !aligned16(meta) || !aligned16(t_meta) || !aligned16(t_vals))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_double_prune24_frozen(vals, meta, rows, cols, t_meta, t_vals,
                                                static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_recompress_frozen(const void* W, const uint8_t* meta, const uint8_t* t_meta,
                                       int64_t rows, int64_t cols, void* vals, void* t_vals,
                                       void* stream) {
  if (rows <= 0 || cols <= 0 || rows % 8 != 0 || cols % 16 != 0) return SLOPE_ERR_SHAPE;
  if (!W || !meta || !t_meta || !vals || !t_vals) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(meta) || !aligned16(t_meta) || !aligned16(vals) ||
      !aligned16(t_vals))
    return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_recompress_frozen24(W, meta, t_meta, rows, cols, vals, t_vals,
                                              static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_sparse_axpby(float beta, const void* A, int a_dtype, float gamma,
                                  const void* B, int b_dtype, void* out, int out_dtype, int64_t n,
                                  void* stream) {
  auto ok_dt = [](int d) { return d == SLOPE_F32 || d == SLOPE_BF16; };
  if (!ok_dt(a_dtype) || !ok_dt(b_dtype) || !ok_dt(out_dtype)) return SLOPE_ERR_INVALID_ARG;
  if (n < 0 || n % 8 != 0) return SLOPE_ERR_SHAPE;
  if (n == 0) return SLOPE_OK;
  if (!A || !B || !out) return SLOPE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  return from_cuda(launch_axpby(beta, A, a_dtype, gamma, B, b_dtype, out, out_dtype, n,
                                static_cast<cudaStream_t>(stream)));
}

// Shared size rules of the three GEMM calls.
static int check_linear(int64_t T, int64_t in, int64_t out, int r) {
  if (T < 0 || in <= 0 || out <= 0 || in % 128 != 0 || out % 128 != 0) return SLOPE_ERR_SHAPE;
  if (r < 0 || r > 256 || r % 8 != 0) return SLOPE_ERR_SHAPE;
  if (T > (int64_t(1) << 31) - 1 || in > (int64_t(1) << 31) - 1 || out > (int64_t(1) << 31) - 1)
    return SLOPE_ERR_SHAPE;
  return SLOPE_OK;
}

extern "C" int slope_linear_fwd(const void* X, int64_t T, int64_t in, int64_t out, const void* Wv,
                                const uint8_t* Wm, const void* L, const void* R, int r, void* Y,
                                int y_dtype, void* XL, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (int s = check_linear(T, in, out, r)) return s;
  if (y_dtype != SLOPE_F32 && y_dtype != SLOPE_BF16) return SLOPE_ERR_INVALID_ARG;
  if (T == 0) return SLOPE_OK;
  if (!X || !Wv || !Wm || !Y) return SLOPE_ERR_INVALID_ARG;
  if (r > 0 && (!L || !R)) return SLOPE_ERR_INVALID_ARG;
  if (int s = rank_plane(XL, workspace, workspace_bytes, T, r, &XL)) return s;
  if (!aligned16(X) || !aligned16(Wv) || !aligned16(Wm) || !aligned16(Y)) return SLOPE_ERR_ALIGNMENT;
  if (r > 0 && (!aligned16(L) || !aligned16(R) || !aligned16(XL))) return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (r > 0) {
    // XL = X·L as hi/lo bf16 (T x 2r): M = T, N = r, K = in; A = X K-major, B = L MN-major.
    DenseGemmArgs g{};
    g.a = X; g.b = L; g.a_mn_major = false; g.b_mn_major = true;
    g.M = T; g.N = r; g.K = in; g.lda = in; g.ldb = r;
    g.epi = DenseEpi::StoreBf16HiLo; g.out = XL; g.ldo = 2 * r; g.lo_off = r; g.splits = 1;
    if (cudaError_t e = launch_dense_gemm(g, st)) return SLOPE_ERR_CUDA;
  }
  SparseGemmArgs a{};
  a.a_vals = Wv; a.a_meta = Wm; a.b = X;
  a.a2 = r > 0 ? R : nullptr; a.b2 = r > 0 ? XL : nullptr; a.a2_mn_major = true;
  a.M = out; a.N = T; a.K = in; a.r = r; a.out = Y; a.out_bf16 = (y_dtype == SLOPE_BF16);
  return from_cuda(launch_sparse_gemm(a, st));
}

extern "C" int slope_linear_bwd_input(const void* dY, int64_t T, int64_t in, int64_t out,
                                      const void* Dv, const uint8_t* Dm, const void* L,
                                      const void* R, int r, void* dX, int dx_dtype, void* G,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (int s = check_linear(T, in, out, r)) return s;
  if (dx_dtype != SLOPE_F32 && dx_dtype != SLOPE_BF16) return SLOPE_ERR_INVALID_ARG;
  if (T == 0) return SLOPE_OK;
  if (!dY || !Dv || !Dm || !dX) return SLOPE_ERR_INVALID_ARG;
  if (r > 0 && (!L || !R)) return SLOPE_ERR_INVALID_ARG;
  if (int s = rank_plane(G, workspace, workspace_bytes, T, r, &G)) return s;
  if (!aligned16(dY) || !aligned16(Dv) || !aligned16(Dm) || !aligned16(dX))
    return SLOPE_ERR_ALIGNMENT;
  if (r > 0 && (!aligned16(L) || !aligned16(R) || !aligned16(G))) return SLOPE_ERR_ALIGNMENT;
  if (int s = check_device()) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (r > 0) {
    // G = dY·Rᵀ as hi/lo bf16 (T x 2r): M = T, N = r, K = out; A = dY K-major, B = R K-major.
    DenseGemmArgs g{};
    g.a = dY; g.b = R; g.a_mn_major = false; g.b_mn_major = false;
    g.M = T; g.N = r; g.K = out; g.lda = out; g.ldb = out;
    g.epi = DenseEpi::StoreBf16HiLo; g.out = G; g.ldo = 2 * r; g.lo_off = r; g.splits = 1;
    if (cudaError_t e = launch_dense_gemm(g, st)) return SLOPE_ERR_CUDA;
  }
  SparseGemmArgs a{};
  a.a_vals = Dv; a.a_meta = Dm; a.b = dY;
  a.a2 = r > 0 ? L : nullptr; a.b2 = r > 0 ? G : nullptr; a.a2_mn_major = false;
  a.M = in; a.N = T; a.K = out; a.r = r; a.out = dX; a.out_bf16 = (dx_dtype == SLOPE_BF16);
  return from_cuda(launch_sparse_gemm(a, st));
}

extern "C" int slope_linear_bwd_weight(const void* dY, const void* X, int64_t T, int64_t in,
                                       int64_t out, const uint8_t* Wm, const void* XL,
                                       const void* G, int r, float* dW, uint32_t flags, float* dL,
                                       float* dR, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (int s = check_linear(T, in, out, r)) return s;
  const uint32_t known =
      SLOPE_DW_DENSE | SLOPE_ACCUMULATE | SLOPE_SKIP_DW | SLOPE_SKIP_ADAPTER | SLOPE_DW_NM28;
  if (flags & ~known) return SLOPE_ERR_INVALID_ARG;
  if ((flags & SLOPE_SKIP_DW) && (flags & SLOPE_SKIP_ADAPTER)) return SLOPE_ERR_INVALID_ARG;
  const bool do_dw = !(flags & SLOPE_SKIP_DW);
  const bool do_ad = r > 0 && !(flags & SLOPE_SKIP_ADAPTER);
  if (do_dw && (!Wm || !dW)) return SLOPE_ERR_INVALID_ARG;
  if (T > 0 && (!dY || !X)) return SLOPE_ERR_INVALID_ARG;
  if (do_ad && (!dL || !dR || (T > 0 && (!XL || !G)))) return SLOPE_ERR_INVALID_ARG;
  if (do_dw && (!aligned16(Wm) || !aligned16(dW))) return SLOPE_ERR_ALIGNMENT;
  if (T > 0 && (!aligned16(dY) || !aligned16(X))) return SLOPE_ERR_ALIGNMENT;
  if (do_ad && (!aligned16(dL) || !aligned16(dR) || (T > 0 && (!aligned16(XL) || !aligned16(G)))))
    return SLOPE_ERR_ALIGNMENT;
  // an optional workspace keeps the dW launch's waves of tiles in step
  unsigned int* wave_ctr = nullptr;
  if (workspace != nullptr) {
    if (workspace_bytes < kWaveSyncBytes) return SLOPE_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return SLOPE_ERR_ALIGNMENT;
    wave_ctr = static_cast<unsigned int*>(workspace);
  }
  if (int s = check_device()) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool dense = flags & SLOPE_DW_DENSE, acc = flags & SLOPE_ACCUMULATE;
  const bool nm28 = flags & SLOPE_DW_NM28;
  const int64_t dw_cols = dense ? in : (nm28 ? in / 4 : in / 2);  // fp32 per row of dW
  const size_t dw_bytes = static_cast<size_t>(out) * dw_cols * sizeof(float);
  if (T == 0) {
    if (!acc && launch_zero3(do_dw ? dW : nullptr, do_dw ? dw_bytes / sizeof(float) : 0,
                             do_ad ? dL : nullptr, do_ad ? static_cast<size_t>(in) * r : 0,
                             do_ad ? dR : nullptr, do_ad ? static_cast<size_t>(out) * r : 0,
                             st) != cudaSuccess)
      return SLOPE_ERR_CUDA;
    return SLOPE_OK;
  }
  // dW and the adapter gradients in one launch when the dW GEMM runs on CTA
  // pairs (an even number of 128-row weight tiles) and 2r fits one tile:
  // dRᵀ = dYᵀ·XL shares dW's A operand and dLᵀ = Gᵀ·X its B operand.
  const bool fuse = do_dw && do_ad && r <= 128 && (out / 128) % 2 == 0;
  if (do_dw) {
    // dW = M ⊙ (dYᵀ·X): M = out, N = in, K = T; A = dY MN-major, B = X MN-major.
    DenseGemmArgs w{};
    w.a = dY; w.b = X; w.a_mn_major = true; w.b_mn_major = true;
    w.M = out; w.N = in; w.K = T; w.lda = out; w.ldb = in;
    w.epi = DenseEpi::MaskedWeightGrad; w.out = dW; w.ldo = dw_cols;
    w.meta = Wm; w.dense_dw = dense; w.accumulate = acc; w.splits = 0; w.nm28 = nm28;
    w.wave_ctr = wave_ctr;
    if (fuse) {
      w.fuse_r = r; w.xl = XL; w.g = G; w.dl = dL; w.dr = dR;
    }
    if (launch_dense_gemm(w, st) != cudaSuccess) return SLOPE_ERR_CUDA;
  }
  if (!do_ad || fuse) return SLOPE_OK;
  if (!acc && launch_zero3(dL, static_cast<size_t>(in) * r, dR, static_cast<size_t>(out) * r, nullptr, 0,
                           st) != cudaSuccess)
    return SLOPE_ERR_CUDA;
  // dL = Xᵀ·G (in x r): M = in, N = 2r (hi and lo parts of G), K = T;
  // A = X MN-major, B = G MN-major; column j + r folds onto column j.
  DenseGemmArgs l{};
  l.a = X; l.b = G; l.a_mn_major = true; l.b_mn_major = true;
  l.M = in; l.N = 2 * r; l.K = T; l.lda = in; l.ldb = 2 * r;
  l.epi = DenseEpi::AddF32; l.out = dL; l.ldo = r; l.fold = r; l.splits = 0;  // 0 = choose
  if (launch_dense_gemm(l, st) != cudaSuccess) return SLOPE_ERR_CUDA;
  // dR = XLᵀ·dY (r x out), computed as dRᵀ = dYᵀ·XL: M = out, N = 2r, K = T;
  // A = dY MN-major, B = XL MN-major, stored transposed and folded onto r rows.
  DenseGemmArgs q{};
  q.a = dY; q.b = XL; q.a_mn_major = true; q.b_mn_major = true;
  q.M = out; q.N = 2 * r; q.K = T; q.lda = out; q.ldb = 2 * r;
  q.epi = DenseEpi::AddF32Transposed; q.out = dR; q.ldo = out; q.fold = r; q.splits = 0;
  return from_cuda(launch_dense_gemm(q, st));
}

extern "C" int slope_selftest_mma_rate(int kind, int pair, int64_t iters, double* flops,
                                       void* stream) {
  if (kind < 0 || kind > 2 || (pair != 0 && pair != 1)) return SLOPE_ERR_INVALID_ARG;
  if (iters < 1 || iters > (int64_t(1) << 20) || !flops) return SLOPE_ERR_INVALID_ARG;
  if (int s = check_device()) return s;
  return from_cuda(launch_mma_rate(kind, pair != 0, iters, flops,
                                   static_cast<cudaStream_t>(stream)));
}

extern "C" int slope_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles <= 0 || limit_cycles > (int64_t(1) << 34)) return SLOPE_ERR_INVALID_ARG;
  if (int s = check_device()) return s;
  unsigned int* status = device_status_ptr();
  if (!status) return SLOPE_ERR_CUDA;
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_cycles);
  return from_cuda(cudaGetLastError());
}

extern "C" int slope_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SLOPE_ERR_CUDA;
  unsigned int* p = device_status_ptr();
  if (!p) return SLOPE_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SLOPE_ERR_CUDA;
  if (v == 0) return SLOPE_OK;
  const unsigned int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return SLOPE_ERR_CUDA;
  return SLOPE_ERR_TIMEOUT;
}
