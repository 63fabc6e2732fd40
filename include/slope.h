/*
 * slope.h — C ABI of the 2:4-sparse plus low-rank adapter linear layer
 * (SLoPe) on one NVIDIA GB300 (sm_103a).
 *
 * The operation is defined on the page "SLoPe: Double-Pruned Sparse Plus Lazy
 * Low-Rank Adapter Pretraining of LLMs" (an AI summary of arXiv 2405.16325v3):
 *   §1 and §2.1 "Double-pruned backward pass" — N:M pruning of the weight and
 *      a second N:M pruning of its transpose for the input gradient;
 *   §2.2 "Lazy low-rank adapters" — the rank-r term (X·L)·R;
 *   §2.3 "Sparse kernels" and App. K "Implementation details" — compressed
 *      formats for the weight and its transpose, gradients masked with the
 *      weight's own mask and stored without their zeros;
 *   §2.4 / App. D — the adapter fused into the sparse product.
 *
 * Notation: T tokens, `in` input features, `out` output features, r adapter
 * rank.  W is out x in.  X is T x in, Y and dY are T x out, L is in x r,
 * R is r x out.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All matrices are dense, row-major and contiguous, in device memory.
 *    bf16 means IEEE bfloat16 bit patterns (uint16); f32 is IEEE binary32.
 *  - Every pointer must be 16-byte aligned (the tensor-memory-access unit's
 *    rule); otherwise SLOPE_ERR_ALIGNMENT.
 *  - The caller owns and allocates every buffer; the library allocates no
 *    device memory and keeps no handle.  Scratch, where a call needs it, is
 *    passed in (`workspace`, sized by slope_workspace_size()).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are returned synchronously, before any
 *    launch, and leave every buffer untouched.  Launch failures return
 *    SLOPE_ERR_CUDA.  Faults inside a kernel surface at the next
 *    synchronisation as a CUDA error; a device-side wait that gave up (a
 *    bounded wait ran out) is reported by slope_device_status().
 *  - Compressed 2:4 format ("vals, meta") of a rows x cols matrix that is 2:4
 *    along its rows: groups are the aligned column quadruples 4g..4g+3.
 *      vals: rows x cols/2 bf16, the two kept entries of each group in
 *            ascending column order;
 *      meta: rows x cols/8 bytes; group g of a row is the nibble
 *            (i0 | i1 << 2), i0 < i1 its kept positions; byte b holds group
 *            2b in its low nibble and group 2b+1 in its high nibble.
 *    The sparse GEMMs read this format as it is (no reordering pass).
 *  - Magnitude ranking uses the exact key (bf16 bits & 0x7FFF); ties go to
 *    the lower index.  No floating-point arithmetic decides a mask.
 *  - Thread safety: calls may be made from several host threads.  Shared
 *    state: a per-device capability cache, a device status word, and a
 *    process-wide cache of encoded TMA tensor maps (256 slots behind one
 *    lock) keyed by every field that goes into a map (address, element type,
 *    extents, row stride, box, swizzle).  A hit is bit for bit the map that
 *    encoding would produce, so a buffer freed and re-allocated at the same
 *    address is still described correctly; the cache holds no reference to
 *    device memory and nothing needs releasing.
 *  - Adapter rank: 0 <= r <= 256 with r % 8 == 0.  The rank-r operands are
 *    read by the tensor-memory-access unit, whose row strides must be
 *    multiples of 16 bytes: L (in x r bf16) has rows of 2r bytes, so r must
 *    be a multiple of 8.  A rank that is not can be zero-padded by the
 *    caller (zero columns of L and zero rows of R add nothing).
 */
#ifndef SLOPE_H_
#define SLOPE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SLOPE_OK = 0,
  SLOPE_ERR_INVALID_ARG = 1, /* NULL pointer, bad flag or dtype, short workspace */
  SLOPE_ERR_SHAPE = 2,       /* a size breaks the rules of the call */
  SLOPE_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
  SLOPE_ERR_UNSUPPORTED = 4, /* device is not sm_103, or an n:m the call does not take */
  SLOPE_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
  SLOPE_ERR_TIMEOUT = 6      /* a bounded device-side wait ran out */
} slope_status;

typedef enum { SLOPE_F32 = 0, SLOPE_BF16 = 1 } slope_dtype;

/* flags of slope_linear_bwd_weight */
#define SLOPE_DW_DENSE 1u     /* write dW dense (out x in, zeros where pruned) */
#define SLOPE_ACCUMULATE 2u   /* add into dW, dL, dR instead of overwriting */
#define SLOPE_SKIP_DW 4u      /* compute dL, dR only (dW is not touched) */
#define SLOPE_SKIP_ADAPTER 8u /* compute dW only (dL, dR are not touched) */
#define SLOPE_DW_NM28 16u     /* Wm is a 2:8 metadata; compressed dW is out x in/4 */

/* Human-readable name of a status code (static string, never NULL). */
const char* slope_status_string(int status);

/* ABI version (major * 10000 + minor * 100 + patch). */
int slope_version(void);

/*
 * Bytes of scratch memory that is always enough as the `workspace` of any of
 * the compute calls below for one linear of these sizes (T tokens, in, out,
 * rank r): the larger of the T x 2r bf16 plane of the rank-r intermediate
 * (4·T·r bytes, rounded up to 256), which slope_linear_fwd and
 * slope_linear_bwd_input use when the caller passes XL (or G) as NULL, and
 * 256 bytes (slope_linear_bwd_weight uses 16 of them, when given, to keep
 * its launch's tiles in step).  Returns 0 for invalid sizes (the call
 * itself then reports them).
 */
size_t slope_workspace_size(int64_t T, int64_t in, int64_t out, int r);

/*
 * A1 — N:M magnitude prune-and-compress (§1, §2.1, §2.3; App. K, where the
 * weight is pruned and packed for the sparse product).  For each row of W
 * (rows x cols bf16), keep the n entries of largest |w| (lower index on
 * ties) of every aligned group of m columns:
 *   2:4 — `vals` rows x cols/2 bf16, `meta` rows x cols/8, the 2:4 format;
 *   1:2 — one entry per aligned pair, written in the 2:4 format (each
 *         quadruple keeps one entry of each half: i0 in {0, 1}, i1 in
 *         {2, 3}), so the 2:4 sparse products take it as it is;
 *   2:8 — the 2:8 format: `vals` rows x cols/4 bf16 (a group's two kept
 *         entries, ascending), `meta` rows x cols/8 bytes, one per group of
 *         eight columns: i0 | i1 << 3 (i0 < i1).  slope_expand_nm_to_24
 *         gives the 2:4 form the sparse products read.
 * Other n:m return SLOPE_ERR_UNSUPPORTED.  Requires rows >= 0 and
 * cols % 8 == 0 (else SLOPE_ERR_SHAPE).  rows == 0 is a no-op.
 */
int slope_prune_nm(const void* W, int64_t rows, int64_t cols, int n, int m, void* vals,
                   uint8_t* meta, void* stream);

/*
 * A2 — double pruning (§1, §2.1; §2.3, which keeps compressed copies of both
 * the weight and its transpose).  Input: the compressed rows x cols (= out x in) weight from
 * slope_prune_nm.  Output: D = P(Wsᵀ), the cols x rows transpose of the
 * pruned weight pruned 2:4 again along its rows (the old out dimension, the
 * reduction dimension of the input gradient), as `t_vals` (cols x rows/2
 * bf16) and `t_meta` (cols x rows/8 bytes).  Positions removed by the first
 * pruning count as +0 (key 0), so a group with fewer than two non-zeros
 * keeps its lowest-index positions and stores +0 there.
 * Requires rows % 8 == 0 and cols % 16 == 0 (else SLOPE_ERR_SHAPE).
 */
int slope_double_prune(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                       void* t_vals, uint8_t* t_meta, void* stream);

/*
 * A2 for any of the library's patterns (§2.1: the transpose is pruned with
 * the same N:M pattern along the input gradient's reduction dimension).
 * n:m = 2:4 is slope_double_prune.  1:2: `vals`/`meta` are a rows x cols
 * matrix in the 2:4 format (e.g. slope_prune_nm's 1:2 output); `t_vals`
 * (cols x rows/2) and `t_meta` (cols x rows/8) receive its transpose pruned
 * 1:2 along the old rows, in the 2:4 format.  2:8: `vals` (rows x cols/4)
 * and `meta` (rows x cols/8) in the 2:8 format; `t_vals` (cols x rows/4)
 * and `t_meta` (cols x rows/8) receive the transpose pruned 2:8, in the 2:8
 * format.  Pruned-away positions count as +0 (key 0): a group with fewer
 * than n non-zeros keeps its lowest-index remaining positions, +0 there.
 * Requires rows % 8 == 0 and cols % 16 == 0 (else SLOPE_ERR_SHAPE); other
 * n:m return SLOPE_ERR_UNSUPPORTED.
 */
int slope_double_prune_nm(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                          int n, int m, void* t_vals, uint8_t* t_meta, void* stream);

/*
 * The 2:4 form of a 2:8-format rows x cols matrix (§2.1's 2:8 pattern run on
 * the 2:4 sparse tensor cores): `vals24` (rows x cols/2 bf16) and `meta24`
 * (rows x cols/8) in the 2:4 format.  Each quadruple keeps the group's
 * entries that fall in it, padded to two with its lowest-index other
 * positions, which hold +0; the dense matrix is unchanged.  Only n:m = 2:8
 * (else SLOPE_ERR_UNSUPPORTED).  Requires cols % 8 == 0 (else
 * SLOPE_ERR_SHAPE); rows == 0 is a no-op.
 */
int slope_expand_nm_to_24(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                          int n, int m, void* vals24, uint8_t* meta24, void* stream);

/*
 * A1 + A2 in one call (§2.3: both compressed copies are made from the same
 * weight; one read of W serves both).  Writes exactly what slope_prune_nm
 * followed by slope_double_prune on its output would write: (vals, meta) of
 * the pruned rows x cols weight and (t_vals, t_meta) of D = P(Wsᵀ), in the
 * layouts of those two calls.  The four outputs must not overlap W or each
 * other.  Requires n == 2 and m == 4 (else SLOPE_ERR_UNSUPPORTED),
 * rows % 8 == 0 and cols % 16 == 0 with both positive (else SLOPE_ERR_SHAPE).
 * Widths with cols % 128 == 0 run as one kernel; other widths run the two
 * kernels of the separate calls.
 */
int slope_prune_and_double_prune(const void* W, int64_t rows, int64_t cols, int n, int m,
                                 void* vals, uint8_t* meta, void* t_vals, uint8_t* t_meta,
                                 void* stream);

/*
 * Optimizer side, weight re-compression (App. K: the kernel that copies
 * optimizer-updated weights into the compressed format; §2.1: the training
 * policy keeps the initialised row mask while the transposed, column-wise
 * mask may change; §2.3: both sparse representations are updated during
 * optimisation).  W is the updated rows x cols bf16 weight and `meta` its
 * kept metadata (rows x cols/8, from slope_prune_nm at initialisation).
 * Writes `vals` (rows x cols/2 bf16): group g of a row takes W's columns
 * 4g + i0 and 4g + i1, (i0, i1) the fields of its nibble, in that order;
 * and (t_vals, t_meta), exactly what slope_double_prune(vals, meta, rows,
 * cols, ...) would write.  One pass over W for cols % 128 == 0, a gather
 * then the second pruning otherwise.  `meta` is read only; the outputs must
 * not overlap the inputs or each other.  Requires rows % 8 == 0 and
 * cols % 16 == 0, both positive (else SLOPE_ERR_SHAPE).
 */
int slope_recompress_double_prune(const void* W, const uint8_t* meta, int64_t rows, int64_t cols,
                                  void* vals, void* t_vals, uint8_t* t_meta, void* stream);

/*
 * A2 with its column-wise mask frozen (§2.1: the transposed mask may be
 * re-derived or kept; this is the kept form): `t_vals` (cols x rows/2 bf16)
 * receives the transpose of the single-pruned matrix (vals, meta) gathered
 * at the positions the given `t_meta` (cols x rows/8, e.g. an earlier
 * slope_double_prune output) names, with no new selection; a position the
 * first pruning removed gives +0.  `t_meta` is read only.  Size rules as
 * slope_double_prune.
 */
int slope_double_prune_frozen(const void* vals, const uint8_t* meta, int64_t rows, int64_t cols,
                              const uint8_t* t_meta, void* t_vals, void* stream);

/*
 * Optimizer side with both masks kept: the updated weight W gathered at the
 * row mask `meta` into `vals` (as slope_recompress_double_prune does), and
 * its transpose gathered at the column mask `t_meta` into `t_vals` (as
 * slope_double_prune_frozen does), in one pass over W for cols % 128 == 0.
 * `meta` and `t_meta` are read only.  Size rules as
 * slope_recompress_double_prune.
 */
int slope_recompress_frozen(const void* W, const uint8_t* meta, const uint8_t* t_meta, int64_t rows,
                            int64_t cols, void* vals, void* t_vals, void* stream);

/*
 * Optimizer side, sparse linear combination (App. K: beta·A + gamma·B for
 * matrices that share a sparsity pattern, for weight decay).  A, B and out
 * are the compressed value arrays (n values each, e.g. rows x cols/2) of
 * matrices with the same metadata, so the combination is element-wise:
 * out[i] = beta·A[i] + gamma·B[i], computed in fp32 as one fused
 * multiply-add on gamma·B[i], each array SLOPE_F32 or SLOPE_BF16 by its
 * dtype argument (a bf16 output is rounded to nearest even).  `out` may be
 * A or B (an in-place update) but must not partly overlap either.  Requires
 * n % 8 == 0 (else SLOPE_ERR_SHAPE; n == 0 is a no-op) and known dtypes
 * (else SLOPE_ERR_INVALID_ARG).
 */
int slope_sparse_axpby(float beta, const void* A, int a_dtype, float gamma, const void* B,
                       int b_dtype, void* out, int out_dtype, int64_t n, void* stream);

/*
 * A3 — sparse forward with the fused adapter (§2.1, §2.2, §2.4, App. D):
 *     Y  = X·Wsᵀ + (X·L)·R          (bf16 inputs, fp32 accumulation)
 *     XL = X·L                        (kept for the backward)
 * X: T x in bf16.  (Wv, Wm): the compressed out x in weight.  L: in x r
 * bf16, R: r x out bf16.  Y: T x out, `y_dtype` SLOPE_F32 or SLOPE_BF16.
 * XL: T x 2r bf16 output when r > 0: row t holds the r values of (X·L)[t]
 * as bf16 "hi" parts followed by their bf16 "lo" remainders (hi = bf16(v),
 * lo = bf16(v - hi)); hi + lo keeps about 16 significant bits, and the
 * adapter product uses both.  XL may be NULL when the caller does not keep
 * it (e.g. inference): the plane then lives in `workspace`, which must be
 * 16-byte aligned and hold slope_workspace_size(T, in, out, r) bytes
 * (else SLOPE_ERR_INVALID_ARG).  The workspace's contents on entry do not
 * matter, and it must not be reused by another call until this one's work
 * on `stream` is done.  With XL given, `workspace` is not used (NULL, 0).
 * Requires in % 128 == 0, out % 128 == 0, T >= 0 (T == 0 is a no-op),
 * 0 <= r <= 256 and r % 8 == 0; r == 0 disables the adapter (L, R, XL may
 * then be NULL).
 */
int slope_linear_fwd(const void* X, int64_t T, int64_t in, int64_t out, const void* Wv,
                     const uint8_t* Wm, const void* L, const void* R, int r, void* Y, int y_dtype,
                     void* XL, void* workspace, size_t workspace_bytes, void* stream);

/*
 * A4 — sparse input gradient with the fused adapter (§1, §2.1):
 *     dX = dY·Dᵀ + (dY·Rᵀ)·Lᵀ        G = dY·Rᵀ (kept for dL)
 * dY: T x out bf16.  (Dv, Dm): the compressed in x out double-pruned matrix
 * from slope_double_prune.  dX: T x in, `dx_dtype` SLOPE_F32 or SLOPE_BF16.
 * G: T x 2r bf16 output (hi parts, then lo parts, as XL) when r > 0; it
 * may be NULL, with the plane then in `workspace`, under the rules
 * slope_linear_fwd gives for XL.  Size rules as slope_linear_fwd.
 */
int slope_linear_bwd_input(const void* dY, int64_t T, int64_t in, int64_t out, const void* Dv,
                           const uint8_t* Dm, const void* L, const void* R, int r, void* dX,
                           int dx_dtype, void* G, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * A5 + A6 — masked weight gradient and adapter gradients (§2.3, gradients of
 * pruned weights are masked; App. K, the gradient stored without the mask's
 * zeros; §2.2 for the adapter):
 *     dW = M ⊙ (dYᵀ·X)     M = the weight's own mask (decoded from Wm)
 *     dL = Xᵀ·G            dR = XLᵀ·dY
 * dY: T x out bf16, X: T x in bf16, Wm: out x in/8 metadata of the weight.
 * dW (f32): compressed out x in/2 (the kept entries in Wv's order) by
 * default, dense out x in with zeros at pruned positions with SLOPE_DW_DENSE.
 * XL (T x 2r) and G (T x 2r) are the hi/lo outputs of the two calls above;
 * dL (in x r f32) and dR (r x out f32) are written when r > 0.
 * SLOPE_ACCUMULATE adds into dW, dL, dR (gradient accumulation) instead of
 * overwriting them.  SLOPE_DW_NM28: Wm is the 2:8 metadata of a 2:8 weight
 * (out x in/8 bytes, slope_prune_nm's 2:8 output) and M its 2:8 mask; the
 * compressed dW is then out x in/4 (the kept entries in the 2:8 `vals`
 * order).  SLOPE_SKIP_DW computes only dL and dR (dW and Wm may be
 * NULL); SLOPE_SKIP_ADAPTER computes only dW (XL, G, dL, dR may be NULL);
 * both together are SLOPE_ERR_INVALID_ARG.  T == 0 writes zeros (or leaves
 * them, when accumulating).  `workspace` is optional (NULL, 0 works): given
 * at least 16 bytes, 16-byte aligned (else SLOPE_ERR_INVALID_ARG or
 * SLOPE_ERR_ALIGNMENT), the call keeps a counter there that holds the dW
 * launch's waves of tiles in step, so the tiles in flight share their
 * slabs of dY and X in L2 and DRAM re-reads fall; its contents on entry do
 * not matter, and it must not be used by another call until this one's
 * work on `stream` is done.  The waiting is advisory: a wave that does not
 * come together within about 50 µs (e.g. when other kernels hold SMs so
 * that the launch's CTAs are not resident together) ends it for the rest of
 * the launch, without error and with the same results.  Size rules as
 * slope_linear_fwd.
 */
int slope_linear_bwd_weight(const void* dY, const void* X, int64_t T, int64_t in, int64_t out,
                            const uint8_t* Wm, const void* XL, const void* G, int r, float* dW,
                            uint32_t flags, float* dL, float* dR, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Size of the library's own scratch array used by
 * slope_linear_fwd_static_scratch: 8 MiB, room for the rank-r plane of
 * T·r <= 2,097,152 (for example T = 16384 tokens at rank 128).
 */
#define SLOPE_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * The forward A3 (as slope_linear_fwd) for callers that cannot allocate
 * device memory and so have no workspace to pass: a plugin inside a host
 * runtime that owns every allocation and hands it only inputs and outputs,
 * or a serving loop that must never call cudaMalloc on its hot path (an
 * allocation can synchronise the device and stall other streams).  This
 * call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine): the rank-r plane X·L that slope_linear_fwd would keep in XL or
 * in the workspace lives in a fixed SLOPE_STATIC_SCRATCH_BYTES array of
 * device memory that the library declares and every GPU that loads the
 * library holds until the process exits.  The caller still passes the
 * inputs and Y; the plane itself is not returned (use slope_linear_fwd with
 * XL when the backward needs it).  Arguments, layouts and results are those
 * of slope_linear_fwd with XL = NULL: the same kernels run.
 *  - Sizes whose plane (4·T·r bytes) exceeds SLOPE_STATIC_SCRATCH_BYTES
 *    return SLOPE_ERR_SHAPE before any work; other argument errors are
 *    slope_linear_fwd's.  r == 0 and T == 0 use no scratch.
 *  - The first call on a device looks up the array's device address on that
 *    device (with it current) and keeps it; make that first call before any
 *    stream capture.
 *  - All calls share the one array, which keeps the last call's plane.
 *    Calls whose work overlaps on the GPU (different streams with no
 *    ordering between them, or different host threads) race on it: order
 *    them on one stream, or with events.
 * The SLoPe pages have no counterpart: this is a deployment form of the
 * forward, not a step of the method.
 */
int slope_linear_fwd_static_scratch(const void* X, int64_t T, int64_t in, int64_t out,
                                    const void* Wv, const uint8_t* Wm, const void* L,
                                    const void* R, int r, void* Y, int y_dtype, void* stream);

/*
 * Synchronises `stream`, then reports and clears the device status word in
 * which kernels record a bounded wait that ran out (SLOPE_ERR_TIMEOUT), or
 * returns SLOPE_OK.  A CUDA error seen while synchronising returns
 * SLOPE_ERR_CUDA.
 */
int slope_device_status(void* stream);

/*
 * Failure-detection self test (no counterpart in the method: it exercises
 * the library's own bounded waits).  Launches one kernel whose single wait
 * can never be satisfied, bounded by `limit_cycles` SM clocks (1 .. 2^34;
 * about 2e6 is one millisecond).  The kernel then records a timeout in the
 * device status word and returns, leaving the context usable; a following
 * slope_device_status() returns SLOPE_ERR_TIMEOUT and clears the word.
 * Returns SLOPE_ERR_INVALID_ARG for a limit outside the range.
 */
int slope_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/*
 * Tensor-core rate self test (no counterpart in the method: it measures the
 * rate the GEMM calls above are judged against).  Every SM (pair = 0) or SM
 * pair (pair = 1, tcgen05 cta_group::2) issues `iters` rounds of four
 * back-to-back tcgen05.mma instructions of kind::f16 (bf16 operands, fp32
 * accumulation, N = 256; M = 128 per SM, 256 per pair) on operands that stay
 * in shared memory: dense (kind = 0, K = 16 per instruction) or 2:4 sparse
 * (the .sp form, K = 32 dense-equivalent, metadata in TMEM), with every
 * group keeping positions 0 and 1 (kind = 1) or each group a random one of
 * the six legal position pairs, as pruned weights have (kind = 2).
 * Writes the dense-equivalent flops the launch executes to *flops and
 * returns once it is enqueued on `stream`; time it with events there.
 * kind must be 0, 1 or 2, pair 0 or 1 and 1 <= iters <= 2^20, else
 * SLOPE_ERR_INVALID_ARG.  A bounded wait that ran out is reported by
 * slope_device_status().
 */
int slope_selftest_mma_rate(int kind, int pair, int64_t iters, double* flops, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SLOPE_H_ */
