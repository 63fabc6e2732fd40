// slope_internal.h — declarations shared by the library's translation units
// (kernel launchers, device queries).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace slope {

// Appends the programmatic stream-serialization attribute (the kernel may
// begin its set-up while the previous kernel on the stream finishes; every
// kernel of this library waits for that kernel before touching global
// memory) to a launch configuration whose attrs array has room for it.
inline void add_pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attrs) {
  attrs[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  ++cfg.numAttrs;
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Split-K factor for `tiles` output tiles of `num_kb` K-blocks each, run on
// `slots` concurrent CTAs (or CTA pairs): the s that minimises
//   ceil(tiles * s / slots) * (ceil(num_kb / s) + epilogue) (+ zero-fill),
// in K-block units, with a dearer epilogue once partial sums are added
// atomically.  At most max(num_kb / 4, 1).
int choose_splits(int tiles, int slots, int num_kb);

// Device address of the status word that bounded waits report into (per
// device, resolved once with the device current), or NULL on error.
unsigned int* device_status_ptr();

// ---- memory-bound kernels (prune.cu)
cudaError_t launch_prune24(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream);
cudaError_t launch_double_prune24(const void* vals, const uint8_t* meta, int64_t rows,
                                  int64_t cols, void* t_vals, uint8_t* t_meta,
                                  cudaStream_t stream);
cudaError_t launch_prune_double24(const void* W, int64_t rows, int64_t cols, void* vals,
                                  uint8_t* meta, void* t_vals, uint8_t* t_meta,
                                  cudaStream_t stream);
cudaError_t launch_gather24(const void* W, const uint8_t* meta, int64_t rows, int64_t cols, void* vals,
                            cudaStream_t stream);
cudaError_t launch_recompress_double24(const void* W, const uint8_t* meta, int64_t rows, int64_t cols,
                                       void* vals, void* t_vals, uint8_t* t_meta, cudaStream_t stream);
cudaError_t launch_double_prune24_frozen(const void* vals, const uint8_t* meta, int64_t rows,
                                         int64_t cols, const uint8_t* t_meta, void* t_vals,
                                         cudaStream_t stream);
cudaError_t launch_recompress_frozen24(const void* W, const uint8_t* meta, const uint8_t* t_meta,
                                       int64_t rows, int64_t cols, void* vals, void* t_vals,
                                       cudaStream_t stream);
// dtype codes: 0 f32, 1 bf16
cudaError_t launch_axpby(float beta, const void* a, int a_dt, float gamma, const void* b, int b_dt,
                         void* out, int out_dt, int64_t n, cudaStream_t stream);

// ---- the 1:2 and 2:8 patterns (nm_patterns.cu)
// 1:2 prune of W into the 2:4 format; its double pruning (2:4 format in and out).
cudaError_t launch_prune12(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream);
cudaError_t launch_double_prune12(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* t_vals, uint8_t* t_meta, cudaStream_t stream);
// 2:8 prune of W into the 2:8 format (vals rows x cols/4, meta rows x cols/8);
// its double pruning (2:8 format in and out); its 2:4 form.
cudaError_t launch_prune28(const void* W, int64_t rows, int64_t cols, void* vals, uint8_t* meta,
                           cudaStream_t stream);
cudaError_t launch_double_prune28(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* t_vals, uint8_t* t_meta, cudaStream_t stream);
cudaError_t launch_expand28(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols, void* vals24,
                            uint8_t* meta24, cudaStream_t stream);

// Zeroes up to three fp32 arrays, and a fourth small one (counts in floats,
// multiples of 4) in one programmatic-dependent launch (dense_gemm.cu).
cudaError_t launch_zero3(float* a, size_t na, float* b, size_t nb, float* c, size_t nc,
                         cudaStream_t stream, float* d = nullptr, size_t nd = 0);

// ---- tensor-core rate self test (mma_rate.cu): enqueues the launch and
// writes the dense-equivalent flops it executes to *flops.
// kind: 0 dense, 1 sparse with one fixed metadata pattern, 2 sparse with
// random legal metadata.
cudaError_t launch_mma_rate(int kind, bool pair, int64_t iters, double* flops,
                            cudaStream_t stream);

// ---- tensor-map encoding (api.cu): 2-D row-major tensor [outer][inner]
// with `row_bytes` between rows, box [box_outer][box_inner], given swizzle.
enum class Swz { None, B32, B64, B128 };
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                  uint32_t box_outer, Swz swz);

// ---- sparse GEMM with the fused adapter (sparse_gemm.cu)
//   D[m][n] = Σ_k A[m][k]·B[n][k] + Σ_j A2[m][j]·B2[n][j], stored transposed:
//   out[n][m].  A is 2:4 compressed (vals M x K/2, meta M x K/8), B is N x K.
//   fwd: M = out, N = T, K = in, A2 = R (MN-major), B2 = XL.
//   dX:  M = in,  N = T, K = out, A2 = L (K-major),  B2 = G.
//   B2 holds 2r columns: the hi and lo bf16 parts of the rank-r product;
//   the adapter segment runs once per part against the same A2.
struct SparseGemmArgs {
  const void* a_vals;
  const uint8_t* a_meta;
  const void* b;       // N x K bf16
  const void* a2;      // adapter operand of the m index (R or L), may be NULL
  const void* b2;      // adapter operand of the n index (XL or G), may be NULL
  bool a2_mn_major;    // true: a2 is r x M (R); false: a2 is M x r (L)
  int64_t M, N, K;
  int r;
  void* out;           // N x M, f32 or bf16
  bool out_bf16;
};
cudaError_t launch_sparse_gemm(const SparseGemmArgs& a, cudaStream_t stream);

// ---- dense GEMMs (dense_gemm.cu)
//   D[m][n] = Σ_k A[m][k]·B[n][k] with A, B bf16 in K-major (row = m/n) or
//   MN-major (row = k) storage.
enum class DenseEpi {
  StoreBf16HiLo,    // out[m][n] = bf16(v), out[m][lo_off + n] = bf16(v - bf16(v))
  AddF32,           // out[m][n'] f32 += v, n' = n folded by `fold` (atomic, split-K)
  AddF32Transposed, // out[n'][m] f32 += v, same folding
  MaskedWeightGrad  // dW: mask by meta, compressed or dense, f32
};
struct DenseGemmArgs {
  const void* a;
  const void* b;
  bool a_mn_major, b_mn_major;
  int64_t M, N, K;
  int64_t lda, ldb;  // elements between rows of the stored matrices
  DenseEpi epi;
  void* out;
  int64_t ldo;       // elements between rows of the output
  const uint8_t* meta;  // MaskedWeightGrad: out x in/8 metadata
  bool dense_dw, accumulate;
  bool nm28 = false;    // MaskedWeightGrad: meta is the 2:8 format (one byte per 8 columns)
  int splits;        // split-K factor; 0 chooses one from the grid size
  int lo_off;        // StoreBf16HiLo: column offset of the low parts (= r)
  int fold;          // AddF32*: columns n >= fold add into column n - fold (0: none)
  // MaskedWeightGrad on CTA pairs may also compute the adapter gradients in
  // the same launch (fuse_r > 0): dR += XLᵀ·dY and dL += Xᵀ·G, with XL and G
  // T x 2r bf16 (hi | lo), dL in x r and dR r x out fp32, added into.
  int fuse_r = 0;
  const void* xl = nullptr;
  const void* g = nullptr;
  float* dl = nullptr;
  float* dr = nullptr;
  // MaskedWeightGrad on CTA pairs: 16 bytes of the caller's workspace for the
  // counter that keeps the pairs' waves of tiles in step, or NULL
  unsigned int* wave_ctr = nullptr;
};
cudaError_t launch_dense_gemm(const DenseGemmArgs& a, cudaStream_t stream);

}  // namespace slope
