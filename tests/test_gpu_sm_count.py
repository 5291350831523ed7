"""Determinism across SM counts.

The persistent kernels size their grids, work partitions and the tensor-core
weight-gradient split count from the SM count, so the fixed-order sums are
partitioned by it: results are bit-identical from call to call on one GPU model
and may round differently on another.  hc_set_sm_count imposes a smaller count
on this GPU: every kernel family is run at the device's count and at two
smaller ones; each result matches the oracle within the usual bars, repeats at
a fixed count are bit-identical, and the counts agree with each other within
those bars.
"""
import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P
from spatially_sharded_cnn_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    from spatially_sharded_cnn_gb300 import hc as mod
    yield mod
    mod.hc_set_sm_count(0)


def _cases():
    dw = P.cfg_of(2, 8, 70, 512, 8, 7, 1, 3, 8, 4)
    tc = P.cfg_of(1, 128, 6, 256, 128, 5, 1, 2, 1, 2)
    pw = P.cfg_of(2, 128, 4, 256, 256, 1, 1, 0, 1, 4)
    out = []
    for cfg, wstd in ((dw, 0.02), (tc, (2.0 / 3200) ** 0.5), (pw, (2.0 / 128) ** 0.5)):
        x = synth.normal((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), 1.0, 7, 1)
        w = synth.normal((cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"]), wstd, 7, 2)
        b = synth.normal((cfg["C_out"],), 0.05, 7, 3)
        gy = synth.normal((cfg["N"], cfg["C_out"], cfg["H"], cfg["W"]), 1.0, 7, 4)
        out.append((cfg, x, w, b, gy))
    return out


@pytest.mark.parametrize("idx", [0, 1, 2], ids=["depthwise7x7", "tc3xtf32_5x5", "bf16x6_1x1"])
def test_results_across_sm_counts(hc, orc, idx):
    cfg, x, w, b, gy = _cases()[idx]
    ref = {"y": orc.conv2d_fwd(cfg, x, w, b), "gx": orc.conv2d_bwd_input(cfg, w, gy),
           "gw": orc.conv2d_bwd_weight(cfg, x, gy), "gb": orc.conv2d_bwd_bias(cfg, gy)}
    tol = {"y": 1e-5, "gx": 1e-5, "gw": 1e-4, "gb": 1e-4}
    runs = {}
    try:
        for sms in (0, 57, 19):
            hc.check(hc.hc_set_sm_count(sms))
            got = []
            for _ in range(2):
                out = R.bwd(cfg, x, w, gy)
                out["y"] = R.fwd(cfg, x, w, b)
                got.append(out)
            for k in ("y", "gx", "gw", "gb", "gw_partials", "gb_partials"):
                assert np.array_equal(got[0][k], got[1][k]), (sms, k)  # bit-identical at a fixed count
            for k in ref:
                assert R.normwise(got[0][k], ref[k]) <= tol[k], (sms, k)
            runs[sms] = got[0]
    finally:
        hc.hc_set_sm_count(0)
    for sms in (57, 19):  # other partitions of the same fixed-order sums: equal within the bars
        for k in ref:
            assert R.normwise(runs[sms][k], runs[0][k]) <= tol[k], (sms, k)


def test_set_sm_count_rejects_negative(hc):
    assert hc.hc_set_sm_count(-1) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_set_sm_count(0) == hc.HC_OK
