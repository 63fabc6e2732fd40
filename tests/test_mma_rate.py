"""Tensor-core rate self test: every variant (dense, 2:4 sparse with fixed
and with random legal metadata; one SM and SM pair) runs, leaves the status word clear, and reports a rate between
a tenth of and a little above the nominal dense-equivalent peak of its kind
(a rate far above it would mean the launch skipped work)."""

import pytest

from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu

NOMINAL_DENSE_TFLOPS = 2250.0  # bf16 dense, GB300


@pytest.mark.parametrize("kind", [0, 1, 2])  # dense, sparse fixed metadata, sparse random metadata
@pytest.mark.parametrize("pair", [False, True])
def test_mma_rate_runs_and_is_plausible(kind, pair):
    import torch

    ensure_built()
    from sparse_rank_adapter_gb300 import slope as S

    stream = torch.cuda.current_stream()
    S.slope_selftest_mma_rate(kind, pair, 64)  # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    flops = S.slope_selftest_mma_rate(kind, pair, 1024)
    e1.record(stream)
    torch.cuda.synchronize()
    S.slope_device_status()
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    nominal = NOMINAL_DENSE_TFLOPS * (2 if kind else 1)
    assert 0.1 * nominal < tflops < 1.2 * nominal, tflops
