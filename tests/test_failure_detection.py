"""Failure detection without a GPU fault: a kernel wait that can never end
runs out its (short) limit, the kernel records a timeout in the device status
word and returns, the host reads SLOPE_ERR_TIMEOUT, and the context keeps
working afterwards."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import bits_of, ensure_built, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch

    ensure_built()
    from sparse_rank_adapter_gb300 import slope as S

    S.slope_device_status()  # start from a clear status word
    S.slope_selftest_wait_timeout(2_000_000)  # about a millisecond of SM clocks
    with pytest.raises(S.SlopeError) as e:
        S.slope_device_status()
    assert e.value.status == S.ERR_TIMEOUT
    S.slope_device_status()  # cleared by the read above
    # the context is intact: a real call still runs and is still exact
    W = synth.normal_bf16(0, 1, "W", (64, 128))
    vals = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(64, 16, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(to_dev(W), vals, meta)
    torch.cuda.synchronize()
    ov, om, _ = O.prune24(W)
    np.testing.assert_array_equal(bits_of(vals), ov)
    np.testing.assert_array_equal(meta.cpu().numpy(), om)


def test_selftest_rejects_bad_limits():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope as S

    assert S.lib().slope_selftest_wait_timeout(0, None) == S.ERR_INVALID_ARG
    assert S.lib().slope_selftest_wait_timeout(1 << 40, None) == S.ERR_INVALID_ARG
