"""The C-ABI library builds, loads, exports every function the header
declares, and rejects bad arguments with status codes before any launch.
Runs without a GPU (the argument checks return before touching CUDA)."""

import os
import re

import pytest

from tests.helpers import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def header_functions():
    src = open(os.path.join(ROOT, "include", "slope.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(slope_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_five_path_calls():
    names = header_functions()
    for n in ("slope_prune_nm", "slope_double_prune", "slope_linear_fwd",
              "slope_linear_bwd_input", "slope_linear_bwd_weight"):
        assert n in names


def test_every_declared_function_is_exported_and_bound(L):
    lib = L.lib()
    bound = {name for name, _, _ in L.SIGNATURES}
    for name in header_functions():
        assert hasattr(lib, name), name
        assert name in bound, name


def test_status_strings(L):
    assert L.status_string(0) == "ok"
    for s in range(1, 7):
        assert L.status_string(s) and L.status_string(s) != "unknown status"
    assert L.status_string(99) == "unknown status"
    assert L.lib().slope_version() >= 10000


def no_gpu():
    try:
        import torch

        return not torch.cuda.is_available()
    except Exception:
        return True


# Fake device addresses: every case below breaks exactly one rule that the
# library checks before any CUDA call, so nothing is dereferenced.  Skipped
# when a GPU is present, where a checking bug would launch on them.
A = 0x10000
MIS = 0x10008

cpu_only = pytest.mark.skipif(not no_gpu(), reason="fake pointers are only safe without a GPU")


@cpu_only
def test_prune_argument_checks(L):
    f = L.lib().slope_prune_nm
    assert f(A, 4, 16, 1, 4, A, A, None) == L.ERR_UNSUPPORTED  # 2:4, 1:2 and 2:8 only
    assert f(A, 4, 16, 4, 8, A, A, None) == L.ERR_UNSUPPORTED
    assert f(A, 4, 12, 1, 2, A, A, None) == L.ERR_SHAPE
    assert f(A, 4, 12, 2, 8, A, A, None) == L.ERR_SHAPE
    assert f(A, 4, 16, 2, 8, A, MIS, None) == L.ERR_ALIGNMENT
    assert f(A, 4, 12, 2, 4, A, A, None) == L.ERR_SHAPE
    assert f(A, -1, 16, 2, 4, A, A, None) == L.ERR_SHAPE
    assert f(None, 4, 16, 2, 4, A, A, None) == L.ERR_INVALID_ARG
    assert f(A, 4, 16, 2, 4, MIS, A, None) == L.ERR_ALIGNMENT
    assert f(A, 0, 16, 2, 4, A, A, None) == L.OK  # empty: nothing to do


@cpu_only
def test_double_prune_argument_checks(L):
    f = L.lib().slope_double_prune
    assert f(A, A, 12, 16, A, A, None) == L.ERR_SHAPE
    assert f(A, A, 16, 24, A, A, None) == L.ERR_SHAPE
    assert f(A, None, 16, 16, A, A, None) == L.ERR_INVALID_ARG
    assert f(A, A, 16, 16, A, MIS, None) == L.ERR_ALIGNMENT


@cpu_only
def test_pattern_argument_checks(L):
    d = L.lib().slope_double_prune_nm
    assert d(A, A, 16, 16, 3, 4, A, A, None) == L.ERR_UNSUPPORTED
    for n, m in ((1, 2), (2, 8), (2, 4)):
        assert d(A, A, 12, 16, n, m, A, A, None) == L.ERR_SHAPE  # rows % 8
        assert d(A, A, 16, 24, n, m, A, A, None) == L.ERR_SHAPE  # cols % 16
        assert d(A, None, 16, 16, n, m, A, A, None) == L.ERR_INVALID_ARG
        assert d(A, A, 16, 16, n, m, MIS, A, None) == L.ERR_ALIGNMENT
    e = L.lib().slope_expand_nm_to_24
    assert e(A, A, 16, 16, 2, 4, A, A, None) == L.ERR_UNSUPPORTED  # 2:8 only
    assert e(A, A, 16, 12, 2, 8, A, A, None) == L.ERR_SHAPE
    assert e(A, A, 16, 16, 2, 8, A, None, None) == L.ERR_INVALID_ARG
    assert e(A, A, 16, 16, 2, 8, A, MIS, None) == L.ERR_ALIGNMENT
    assert e(None, None, 0, 16, 2, 8, None, None, None) == L.OK  # no rows
    bw = L.lib().slope_linear_bwd_weight
    # the 2:8 flag is known: a bad dW alignment is what fails next
    assert bw(A, A, 64, 256, 256, A, A, A, 8, MIS, 16, A, A, None, 0, None) == L.ERR_ALIGNMENT
    assert bw(A, A, 64, 256, 256, A, A, A, 8, A, 32, A, A, None, 0, None) == L.ERR_INVALID_ARG


@cpu_only
def test_prune_and_double_prune_argument_checks(L):
    f = L.lib().slope_prune_and_double_prune
    assert f(A, 16, 16, 1, 2, A, A, A, A, None) == L.ERR_UNSUPPORTED
    assert f(A, 12, 16, 2, 4, A, A, A, A, None) == L.ERR_SHAPE  # rows % 8
    assert f(A, 16, 24, 2, 4, A, A, A, A, None) == L.ERR_SHAPE  # cols % 16
    assert f(A, 0, 16, 2, 4, A, A, A, A, None) == L.ERR_SHAPE
    assert f(A, 16, 16, 2, 4, A, A, None, A, None) == L.ERR_INVALID_ARG
    assert f(A, 16, 16, 2, 4, A, A, A, MIS, None) == L.ERR_ALIGNMENT


@cpu_only
def test_optimizer_side_argument_checks(L):
    f = L.lib().slope_recompress_double_prune
    assert f(A, A, 12, 16, A, A, A, None) == L.ERR_SHAPE
    assert f(A, A, 16, 24, A, A, A, None) == L.ERR_SHAPE
    assert f(A, None, 16, 16, A, A, A, None) == L.ERR_INVALID_ARG
    assert f(A, A, 16, 16, A, A, MIS, None) == L.ERR_ALIGNMENT
    h = L.lib().slope_double_prune_frozen
    assert h(A, A, 12, 16, A, A, None) == L.ERR_SHAPE
    assert h(A, A, 16, 16, None, A, None) == L.ERR_INVALID_ARG
    assert h(A, A, 16, 16, A, MIS, None) == L.ERR_ALIGNMENT
    k = L.lib().slope_recompress_frozen
    assert k(A, A, A, 16, 24, A, A, None) == L.ERR_SHAPE
    assert k(A, A, None, 16, 16, A, A, None) == L.ERR_INVALID_ARG
    assert k(A, A, A, 16, 16, MIS, A, None) == L.ERR_ALIGNMENT
    g = L.lib().slope_sparse_axpby
    assert g(1.0, A, 0, 1.0, A, 2, A, 0, 16, None) == L.ERR_INVALID_ARG  # unknown dtype
    assert g(1.0, A, 0, 1.0, A, 0, A, 0, 12, None) == L.ERR_SHAPE        # n % 8
    assert g(1.0, A, 0, 1.0, A, 0, A, 0, -8, None) == L.ERR_SHAPE
    assert g(1.0, A, 0, 1.0, None, 0, A, 0, 16, None) == L.ERR_INVALID_ARG
    assert g(1.0, A, 1, 1.0, A, 1, MIS, 1, 16, None) == L.ERR_ALIGNMENT
    assert g(1.0, None, 0, 1.0, None, 0, None, 0, 0, None) == L.OK      # n == 0


@cpu_only
def test_linear_argument_checks(L):
    fwd = L.lib().slope_linear_fwd
    bi = L.lib().slope_linear_bwd_input
    bw = L.lib().slope_linear_bwd_weight
    # in/out must be multiples of 128, r a multiple of 8 in [0, 256]
    assert fwd(A, 64, 200, 256, A, A, A, A, 8, A, 0, A, None, 0, None) == L.ERR_SHAPE
    assert fwd(A, 64, 256, 256, A, A, A, A, 12, A, 0, A, None, 0, None) == L.ERR_SHAPE
    assert fwd(A, 64, 256, 256, A, A, A, A, 264, A, 0, A, None, 0, None) == L.ERR_SHAPE
    assert fwd(A, -1, 256, 256, A, A, A, A, 8, A, 0, A, None, 0, None) == L.ERR_SHAPE
    assert fwd(A, 64, 256, 256, A, A, A, A, 8, A, 7, A, None, 0, None) == L.ERR_INVALID_ARG
    assert fwd(A, 64, 256, 256, A, A, None, A, 8, A, 0, A, None, 0, None) == L.ERR_INVALID_ARG
    assert fwd(A, 64, 256, 256, A, A, A, A, 8, A, 0, None, None, 0, None) == L.ERR_INVALID_ARG  # no XL, no workspace
    assert fwd(A, 64, 256, 256, A, A, A, A, 8, MIS, 0, A, None, 0, None) == L.ERR_ALIGNMENT
    assert fwd(A, 0, 256, 256, A, A, A, A, 8, A, 0, A, None, 0, None) == L.OK  # T == 0
    assert bi(A, 64, 256, 384, A, A, A, A, 16, A, 1, None, None, 0, None) == L.ERR_INVALID_ARG
    assert bi(A, 64, 256, 130, A, A, A, A, 16, A, 1, A, None, 0, None) == L.ERR_SHAPE
    assert bw(A, A, 64, 256, 256, A, A, A, 8, A, 32, A, A, None, 0, None) == L.ERR_INVALID_ARG  # unknown flag
    assert bw(A, A, 64, 256, 256, A, A, A, 8, A, 4 | 8, A, A, None, 0, None) == L.ERR_INVALID_ARG  # skip both
    assert bw(A, A, 64, 256, 256, A, A, A, 8, None, 4, None, A, None, 0, None) == L.ERR_INVALID_ARG  # no dL
    assert bw(A, A, 64, 256, 256, None, A, A, 8, A, 0, A, A, None, 0, None) == L.ERR_INVALID_ARG
    assert bw(A, A, 64, 256, 256, A, A, A, 8, A, 0, None, A, None, 0, None) == L.ERR_INVALID_ARG
    assert bw(A, A, 64, 256, 256, A, A, A, 8, MIS, 0, A, A, None, 0, None) == L.ERR_ALIGNMENT


@cpu_only
def test_mma_rate_argument_checks(L):
    import ctypes

    f = L.lib().slope_selftest_mma_rate
    out = ctypes.c_double(0.0)
    assert f(3, 0, 16, ctypes.byref(out), None) == L.ERR_INVALID_ARG
    assert f(-1, 0, 16, ctypes.byref(out), None) == L.ERR_INVALID_ARG
    assert f(1, -1, 16, ctypes.byref(out), None) == L.ERR_INVALID_ARG
    assert f(1, 1, 0, ctypes.byref(out), None) == L.ERR_INVALID_ARG
    assert f(0, 1, (1 << 20) + 1, ctypes.byref(out), None) == L.ERR_INVALID_ARG
    assert f(0, 0, 16, None, None) == L.ERR_INVALID_ARG


@cpu_only
def test_selftest_argument_checks(L):
    f = L.lib().slope_selftest_wait_timeout
    assert f(0, None) == L.ERR_INVALID_ARG
    assert f(-5, None) == L.ERR_INVALID_ARG
    assert f(1 << 40, None) == L.ERR_INVALID_ARG


def test_workspace_size_is_the_rank_plane(L):
    # the T x 2r bf16 plane of XL or G, rounded up to 256 bytes
    assert L.slope_workspace_size(4096, 1024, 1024, 16) == 4 * 4096 * 16
    assert L.slope_workspace_size(1, 256, 256, 8) == 256
    assert L.slope_workspace_size(16384, 7168, 28672, 64) == 4 * 16384 * 64
    assert L.slope_workspace_size(4096, 1024, 1024, 0) == 256  # the weight gradient's wave counter
    assert L.slope_workspace_size(4096, 1024, 1024, 12) == 0  # invalid rank
    assert L.slope_workspace_size(-1, 1024, 1024, 16) == 0
    assert L.slope_workspace_size(64, 200, 256, 8) == 0


@cpu_only
def test_workspace_argument_checks(L):
    fwd = L.lib().slope_linear_fwd
    bi = L.lib().slope_linear_bwd_input
    need = L.slope_workspace_size(64, 256, 256, 8)
    # XL (or G) NULL: the workspace must be there and large enough
    assert fwd(A, 64, 256, 256, A, A, A, A, 8, A, 0, None, None, need, None) == L.ERR_INVALID_ARG
    assert fwd(A, 64, 256, 256, A, A, A, A, 8, A, 0, None, A, need - 16, None) == L.ERR_INVALID_ARG
    assert fwd(A, 64, 256, 256, A, A, A, A, 8, A, 0, None, MIS, need, None) == L.ERR_ALIGNMENT
    assert bi(A, 64, 256, 256, A, A, A, A, 8, A, 0, None, A, 0, None) == L.ERR_INVALID_ARG
    assert bi(A, 64, 256, 256, A, A, A, A, 8, A, 0, None, MIS, need, None) == L.ERR_ALIGNMENT
    # no adapter: nothing is needed
    assert fwd(A, 64, 256, 256, A, A, None, None, 0, MIS, 0, None, None, 0, None) == L.ERR_ALIGNMENT
    # the weight gradient's optional workspace: at least 16 bytes, aligned
    bw = L.lib().slope_linear_bwd_weight
    assert bw(A, A, 64, 256, 256, A, A, A, 8, A, 0, A, A, A, 8, None) == L.ERR_INVALID_ARG
    assert bw(A, A, 64, 256, 256, A, A, A, 8, A, 0, A, A, MIS, 16, None) == L.ERR_ALIGNMENT


def test_binding_refuses_cpu_tensors(L):
    import torch

    W = torch.zeros(4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        L.slope_prune_nm(W, torch.zeros(4, 8, dtype=torch.bfloat16), torch.zeros(4, 2, dtype=torch.uint8), stream=0)


def test_product_code_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "sparse_rank_adapter_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("CPU oracle", ""), os.path.join(dirpath, f)
