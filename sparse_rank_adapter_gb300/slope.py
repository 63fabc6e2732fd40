"""ctypes binding of libslope.so, with the C ABI's names (include/slope.h).

Argument marshalling only: each function checks that the torch tensors it
is given are contiguous device tensors of the right dtype and shape, passes
their device pointers and the current (or given) CUDA stream to the
library, and raises ``SlopeError`` on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  A
missing or unloadable library is an error.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libslope.so")

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(7)
F32, BF16 = 0, 1
DW_DENSE, ACCUMULATE, SKIP_DW, SKIP_ADAPTER, DW_NM28 = 1, 2, 4, 8, 16

# (name, restype, argtypes) of every exported function, in header order.
_vp, _i64, _i, _u32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
SIGNATURES = (
    ("slope_status_string", ctypes.c_char_p, (_i,)),
    ("slope_version", _i, ()),
    ("slope_workspace_size", _sz, (_i64, _i64, _i64, _i)),
    ("slope_prune_nm", _i, (_vp, _i64, _i64, _i, _i, _vp, _vp, _vp)),
    ("slope_double_prune", _i, (_vp, _vp, _i64, _i64, _vp, _vp, _vp)),
    ("slope_double_prune_nm", _i, (_vp, _vp, _i64, _i64, _i, _i, _vp, _vp, _vp)),
    ("slope_expand_nm_to_24", _i, (_vp, _vp, _i64, _i64, _i, _i, _vp, _vp, _vp)),
    ("slope_prune_and_double_prune", _i, (_vp, _i64, _i64, _i, _i, _vp, _vp, _vp, _vp, _vp)),
    ("slope_recompress_double_prune", _i, (_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp)),
    ("slope_double_prune_frozen", _i, (_vp, _vp, _i64, _i64, _vp, _vp, _vp)),
    ("slope_recompress_frozen", _i, (_vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp)),
    ("slope_sparse_axpby", _i, (ctypes.c_float, _vp, _i, ctypes.c_float, _vp, _i, _vp, _i, _i64, _vp)),
    ("slope_linear_fwd", _i, (_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp)),
    ("slope_linear_bwd_input", _i, (_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp)),
    ("slope_linear_bwd_weight", _i, (_vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _i, _vp, _u32, _vp, _vp, _vp, _sz, _vp)),
    ("slope_linear_fwd_static_scratch", _i, (_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp)),
    ("slope_device_status", _i, (_vp,)),
    ("slope_selftest_wait_timeout", _i, (_i64, _vp)),
    ("slope_selftest_mma_rate", _i, (_i, _i, _i64, ctypes.POINTER(ctypes.c_double), _vp)),
)

_lib = None
_lock = threading.Lock()


class SlopeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """The loaded library (loaded once; raises if it is missing)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with sparse_rank_adapter_gb300.build.build()"
                    )
                handle = ctypes.CDLL(LIB_PATH)
                for name, res, args in SIGNATURES:
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = list(args)
                _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().slope_status_string(status).decode()


def _check(status: int, where: str):
    if status != OK:
        raise SlopeError(status, where)


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t, dtype=None, shape=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _dtype_code(t):
    import torch

    return BF16 if t.dtype == torch.bfloat16 else F32


def slope_workspace_size(T: int, inp: int, out: int, r: int) -> int:
    return lib().slope_workspace_size(T, inp, out, r)


def _vals_cols(cols: int, m: int) -> int:
    """Stored values per row: half the columns (2:4, and 1:2 in the 2:4
    format), a quarter for 2:8."""
    return cols // 4 if m == 8 else cols // 2


def slope_prune_nm(W, vals, meta, n: int = 2, m: int = 4, stream=None):
    """A1: n:m prune-and-compress of W (rows x cols bf16) into vals/meta:
    2:4 and 1:2 in the 2:4 format (vals cols/2), 2:8 in the 2:8 format
    (vals cols/4); meta is cols/8 bytes per row in every case."""
    import torch

    rows, cols = W.shape
    st = lib().slope_prune_nm(
        _ptr(W, torch.bfloat16, name="W"), rows, cols, n, m,
        _ptr(vals, torch.bfloat16, (rows, _vals_cols(cols, m)), "vals"),
        _ptr(meta, torch.uint8, (rows, cols // 8), "meta"), _stream(stream))
    _check(st, "slope_prune_nm")


def slope_double_prune_nm(vals, meta, rows: int, cols: int, t_vals, t_meta, n: int = 2, m: int = 4,
                          stream=None):
    """A2 for 2:4, 1:2 (2:4 format) or 2:8 (2:8 format): the transpose of the
    compressed rows x cols matrix pruned n:m again along the old rows."""
    import torch

    st = lib().slope_double_prune_nm(
        _ptr(vals, torch.bfloat16, (rows, _vals_cols(cols, m)), "vals"),
        _ptr(meta, torch.uint8, (rows, cols // 8), "meta"), rows, cols, n, m,
        _ptr(t_vals, torch.bfloat16, (cols, _vals_cols(rows, m)), "t_vals"),
        _ptr(t_meta, torch.uint8, (cols, rows // 8), "t_meta"), _stream(stream))
    _check(st, "slope_double_prune_nm")


def slope_expand_nm_to_24(vals, meta, rows: int, cols: int, vals24, meta24, n: int = 2, m: int = 8,
                          stream=None):
    """The 2:4 form (vals24 cols/2, meta24 cols/8) of a 2:8-format matrix."""
    import torch

    st = lib().slope_expand_nm_to_24(
        _ptr(vals, torch.bfloat16, (rows, _vals_cols(cols, m)), "vals"),
        _ptr(meta, torch.uint8, (rows, cols // 8), "meta"), rows, cols, n, m,
        _ptr(vals24, torch.bfloat16, (rows, cols // 2), "vals24"),
        _ptr(meta24, torch.uint8, (rows, cols // 8), "meta24"), _stream(stream))
    _check(st, "slope_expand_nm_to_24")


def slope_double_prune(vals, meta, rows: int, cols: int, t_vals, t_meta, stream=None):
    """A2: D = P(Wsᵀ) from the compressed rows x cols weight."""
    import torch

    st = lib().slope_double_prune(
        _ptr(vals, torch.bfloat16, (rows, cols // 2), "vals"),
        _ptr(meta, torch.uint8, (rows, cols // 8), "meta"), rows, cols,
        _ptr(t_vals, torch.bfloat16, (cols, rows // 2), "t_vals"),
        _ptr(t_meta, torch.uint8, (cols, rows // 8), "t_meta"), _stream(stream))
    _check(st, "slope_double_prune")


def slope_prune_and_double_prune(W, vals, meta, t_vals, t_meta, n: int = 2, m: int = 4, stream=None):
    """A1 and A2 in one call: (vals, meta) of the pruned W and (t_vals, t_meta)
    of D = P(Wsᵀ), exactly as the two separate calls write them."""
    import torch

    rows, cols = W.shape
    st = lib().slope_prune_and_double_prune(
        _ptr(W, torch.bfloat16, name="W"), rows, cols, n, m,
        _ptr(vals, torch.bfloat16, (rows, cols // 2), "vals"),
        _ptr(meta, torch.uint8, (rows, cols // 8), "meta"),
        _ptr(t_vals, torch.bfloat16, (cols, rows // 2), "t_vals"),
        _ptr(t_meta, torch.uint8, (cols, rows // 8), "t_meta"), _stream(stream))
    _check(st, "slope_prune_and_double_prune")


def slope_recompress_double_prune(W, meta, vals, t_vals, t_meta, stream=None):
    """Re-compress the updated weight W at its kept mask `meta` into `vals`,
    and write the second pruning of the result into (t_vals, t_meta)."""
    import torch

    rows, cols = W.shape
    st = lib().slope_recompress_double_prune(
        _ptr(W, torch.bfloat16, name="W"), _ptr(meta, torch.uint8, (rows, cols // 8), "meta"), rows, cols,
        _ptr(vals, torch.bfloat16, (rows, cols // 2), "vals"),
        _ptr(t_vals, torch.bfloat16, (cols, rows // 2), "t_vals"),
        _ptr(t_meta, torch.uint8, (cols, rows // 8), "t_meta"), _stream(stream))
    _check(st, "slope_recompress_double_prune")


def slope_double_prune_frozen(vals, meta, rows: int, cols: int, t_meta, t_vals, stream=None):
    """A2 with the column mask frozen: the transpose of (vals, meta) gathered
    at the given t_meta into t_vals."""
    import torch

    st = lib().slope_double_prune_frozen(
        _ptr(vals, torch.bfloat16, (rows, cols // 2), "vals"), _ptr(meta, torch.uint8, (rows, cols // 8), "meta"),
        rows, cols, _ptr(t_meta, torch.uint8, (cols, rows // 8), "t_meta"),
        _ptr(t_vals, torch.bfloat16, (cols, rows // 2), "t_vals"), _stream(stream))
    _check(st, "slope_double_prune_frozen")


def slope_recompress_frozen(W, meta, t_meta, vals, t_vals, stream=None):
    """Both masks kept: W gathered at meta into vals, its transpose at t_meta into t_vals."""
    import torch

    rows, cols = W.shape
    st = lib().slope_recompress_frozen(
        _ptr(W, torch.bfloat16, name="W"), _ptr(meta, torch.uint8, (rows, cols // 8), "meta"),
        _ptr(t_meta, torch.uint8, (cols, rows // 8), "t_meta"), rows, cols,
        _ptr(vals, torch.bfloat16, (rows, cols // 2), "vals"),
        _ptr(t_vals, torch.bfloat16, (cols, rows // 2), "t_vals"), _stream(stream))
    _check(st, "slope_recompress_frozen")


def slope_sparse_axpby(beta: float, A, gamma: float, B, out, stream=None):
    """out = beta·A + gamma·B on the compressed values of matrices sharing a
    2:4 pattern (fp32 or bf16 tensors of the same number of values)."""
    import torch

    n = out.numel()
    if A.numel() != n or B.numel() != n:
        raise ValueError("A, B and out must hold the same number of values")
    for t, name in ((A, "A"), (B, "B"), (out, "out")):
        if t.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError(f"{name} must be float32 or bfloat16, got {t.dtype}")
    st = lib().slope_sparse_axpby(
        float(beta), _ptr(A, None, name="A"), _dtype_code(A), float(gamma), _ptr(B, None, name="B"),
        _dtype_code(B), _ptr(out, None, name="out"), _dtype_code(out), n, _stream(stream))
    _check(st, "slope_sparse_axpby")


def slope_linear_fwd(X, Wv, Wm, L, R, Y, XL=None, workspace=None, stream=None):
    """A3: Y = X·Wsᵀ + (X·L)·R, XL = X·L as hi/lo bf16 (T x 2r).  Y is f32 or bf16."""
    import torch

    T, inp = X.shape
    out = Wv.shape[0]
    r = 0 if L is None else L.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().slope_linear_fwd(
        _ptr(X, torch.bfloat16, name="X"), T, inp, out,
        _ptr(Wv, torch.bfloat16, (out, inp // 2), "Wv"), _ptr(Wm, torch.uint8, (out, inp // 8), "Wm"),
        _ptr(L, torch.bfloat16, (inp, r), "L"), _ptr(R, torch.bfloat16, (r, out), "R"), r,
        _ptr(Y, None, (T, out), "Y"), _dtype_code(Y),
        _ptr(XL, torch.bfloat16, (T, 2 * r), "XL"), _ptr(workspace, name="workspace"), ws_bytes,
        _stream(stream))
    _check(st, "slope_linear_fwd")


def slope_linear_bwd_input(dY, Dv, Dm, L, R, dX, G=None, workspace=None, stream=None):
    """A4: dX = dY·Dᵀ + (dY·Rᵀ)·Lᵀ, G = dY·Rᵀ as hi/lo bf16 (T x 2r).  dX is f32 or bf16."""
    import torch

    T, out = dY.shape
    inp = Dv.shape[0]
    r = 0 if L is None else L.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().slope_linear_bwd_input(
        _ptr(dY, torch.bfloat16, name="dY"), T, inp, out,
        _ptr(Dv, torch.bfloat16, (inp, out // 2), "Dv"), _ptr(Dm, torch.uint8, (inp, out // 8), "Dm"),
        _ptr(L, torch.bfloat16, (inp, r), "L"), _ptr(R, torch.bfloat16, (r, out), "R"), r,
        _ptr(dX, None, (T, inp), "dX"), _dtype_code(dX),
        _ptr(G, torch.bfloat16, (T, 2 * r), "G"), _ptr(workspace, name="workspace"), ws_bytes,
        _stream(stream))
    _check(st, "slope_linear_bwd_input")


def slope_linear_bwd_weight(dY, X, Wm, XL, G, dW, dL=None, dR=None, flags: int = 0,
                            workspace=None, stream=None):
    """A5 + A6: dW = M ⊙ (dYᵀ·X) (compressed, or dense with DW_DENSE), dL, dR."""
    import torch

    T, out = dY.shape
    inp = X.shape[1]
    r = 0 if XL is None else XL.shape[1] // 2
    if r == 0 and dL is not None:
        r = dL.shape[1]
    dw_shape = (out, inp) if flags & DW_DENSE else (out, inp // 4 if flags & DW_NM28 else inp // 2)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().slope_linear_bwd_weight(
        _ptr(dY, torch.bfloat16, name="dY"), _ptr(X, torch.bfloat16, (T, inp), "X"), T, inp, out,
        _ptr(Wm, torch.uint8, (out, inp // 8), "Wm"),
        _ptr(XL, torch.bfloat16, (T, 2 * r), "XL"), _ptr(G, torch.bfloat16, (T, 2 * r), "G"), r,
        _ptr(dW, torch.float32, dw_shape, "dW"), flags,
        _ptr(dL, torch.float32, (inp, r), "dL"), _ptr(dR, torch.float32, (r, out), "dR"),
        _ptr(workspace, name="workspace"), ws_bytes, _stream(stream))
    _check(st, "slope_linear_bwd_weight")


STATIC_SCRATCH_BYTES = 8 << 20  # SLOPE_STATIC_SCRATCH_BYTES


def slope_linear_fwd_static_scratch(X, Wv, Wm, L, R, Y, stream=None):
    """A3 for callers that cannot allocate device memory: Y = X·Wsᵀ + (X·L)·R
    with the rank-r plane in the library's own fixed device array (4·T·r
    bytes at most STATIC_SCRATCH_BYTES).  Calls that overlap on the GPU race
    on that array; the first call on a device must come before any stream
    capture."""
    import torch

    T, inp = X.shape
    out = Wv.shape[0]
    r = 0 if L is None else L.shape[1]
    st = lib().slope_linear_fwd_static_scratch(
        _ptr(X, torch.bfloat16, name="X"), T, inp, out,
        _ptr(Wv, torch.bfloat16, (out, inp // 2), "Wv"), _ptr(Wm, torch.uint8, (out, inp // 8), "Wm"),
        _ptr(L, torch.bfloat16, (inp, r), "L"), _ptr(R, torch.bfloat16, (r, out), "R"), r,
        _ptr(Y, None, (T, out), "Y"), _dtype_code(Y), _stream(stream))
    _check(st, "slope_linear_fwd_static_scratch")


def slope_device_status(stream=None):
    _check(lib().slope_device_status(_stream(stream)), "slope_device_status")


MMA_DENSE, MMA_SPARSE_FIXED_META, MMA_SPARSE_RANDOM_META = 0, 1, 2


def slope_selftest_mma_rate(kind: int, pair: bool, iters: int, stream=None) -> float:
    """Enqueue the tensor-core rate self test (kind::f16 MMAs from resident
    shared-memory operands, on every SM or SM pair): dense, 2:4 sparse with
    one fixed metadata pattern, or 2:4 sparse with random legal metadata.
    Returns the dense-equivalent flops the launch executes; time it with
    events on `stream`."""
    flops = ctypes.c_double(0.0)
    _check(lib().slope_selftest_mma_rate(int(kind), int(bool(pair)), iters, ctypes.byref(flops),
                                         _stream(stream)), "slope_selftest_mma_rate")
    return flops.value


def slope_selftest_wait_timeout(limit_cycles: int, stream=None):
    """Launch the bounded-wait self test (a wait nothing ends, limited to
    `limit_cycles` SM clocks); slope_device_status() then reports the timeout."""
    _check(lib().slope_selftest_wait_timeout(limit_cycles, _stream(stream)), "slope_selftest_wait_timeout")
