"""Failure detection without a GPU fault: a kernel whose wait runs out (an
mbarrier that nothing arrives on, bounded by the global timer) records
HC_ERR_TIMEOUT; the host reads it through hc_sync_check, the status word is
cleared, and the context keeps computing correct results."""
import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available()
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def test_timeout_is_reported_and_context_survives(hc, orc):
    assert hc.hc_sync_check() == hc.HC_OK
    assert hc.hc_selftest_timeout(0) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_selftest_timeout(20000) == hc.HC_OK      # 20 ms wait that nothing ends
    assert hc.hc_sync_check() == hc.HC_ERR_TIMEOUT
    assert hc.hc_sync_check() == hc.HC_OK                  # read and cleared
    cfg = P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4)
    x, w, b, gy = P.rand_case(cfg, 3)
    y = R.fwd(cfg, x, w, b)
    assert R.normwise(y, orc.conv2d_fwd(cfg, x, w, b)) <= 1e-5


def test_timeout_on_a_side_stream(hc):
    s = torch.cuda.Stream()
    assert hc.hc_selftest_timeout(5000, s) == hc.HC_OK
    assert hc.hc_sync_check(s) == hc.HC_ERR_TIMEOUT
    assert hc.hc_sync_check(s) == hc.HC_OK
