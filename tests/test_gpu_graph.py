"""A fwd + bwd step captured as a CUDA graph replays to exactly the eager result.

The replay check is bitwise, as the LibreYOLO "Grafy CUDA" page requires of a
capturable family ("Obsługa inferencji"), and the graph is bound to buffer
addresses, not values ("Co jest przechwytywane"): rewriting the input in place
and replaying gives the eager result for the new input.
"""
import numpy as np
import pytest
import torch

from spatially_sharded_cnn_gb300 import synth
import hc_run as R
from test_gpu_conv import CASES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def _eager(hc, cfg, x, w, b, gy):
    y = R.fwd(cfg, x, w, b)
    out = R.bwd(cfg, x, w, gy, partials=False)
    return y, out["gx"], out["gw"], out["gb"]


@pytest.mark.parametrize("name", ["config1_dense5x5", "dw7_ragged_S4", "tc_5x5_S2", "tc_down2x2s2_S2", "stem4x4s4",
                                  "tc_1x1"])
def test_step_graph_bitwise(hc, orc, name):
    cfg, x, w, b, gy = CASES[name]()
    d = hc.desc(cfg)
    Ho, Wo = R.out_hw(cfg)
    wshape = (cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"])
    xd, wd, bd, gyd = R.dev(x), R.dev(w), R.dev(b), R.dev(gy)
    y = torch.full((cfg["N"], cfg["C_out"], Ho, Wo), float("nan"), device="cuda")
    gx = torch.full(x.shape, float("nan"), device="cuda")
    gw = torch.full(wshape, float("nan"), device="cuda")
    gb = torch.full((cfg["C_out"],), float("nan"), device="cuda")
    wsf, nbf = R.workspace(d, 0)
    wsb, nbb = R.workspace(d, 1)
    st, g = hc.hc_conv2d_step_graph_create(d, xd, wd, bd, y, gyd, gx, gw, gb, wsf, nbf, wsb, nbb)
    hc.check(st, "graph create")
    try:
        torch.cuda.synchronize()
        assert torch.isnan(y).all(), "capture must not run the step"
        for _ in range(2):  # replays are repeatable
            hc.check(hc.hc_step_graph_launch(g), "graph launch")
            hc.check(hc.hc_sync_check(), "graph sync")
            ref = _eager(hc, cfg, x, w, b, gy)
            for got, want in zip((y, gx, gw, gb), ref):
                assert np.array_equal(got.cpu().numpy(), want)
        # new input values in the same buffer: the replay computes the new step
        x2 = synth.normal(x.shape, 1.0, 99, 1)
        xd.copy_(torch.from_numpy(x2).cuda())
        hc.check(hc.hc_step_graph_launch(g), "graph launch")
        hc.check(hc.hc_sync_check(), "graph sync")
        ref = _eager(hc, cfg, x2, w, b, gy)
        for got, want in zip((y, gx, gw, gb), ref):
            assert np.array_equal(got.cpu().numpy(), want)
        assert R.normwise(y.cpu().numpy(), orc.conv2d_fwd(cfg, x2, w, b)) <= 1e-5
    finally:
        hc.check(hc.hc_step_graph_destroy(g), "graph destroy")


@pytest.mark.parametrize("name", ["tc_1x1", "tc_down2x2s2_S2"])
def test_step_graph_shared_workspace(hc, orc, name):
    """One buffer as both workspaces: the backward pass may not read x's operand
    copy from the forward workspace (it overwrites it), so the graph runs the
    plain backward pass -- same results."""
    cfg, x, w, b, gy = CASES[name]()
    d = hc.desc(cfg)
    Ho, Wo = R.out_hw(cfg)
    wshape = (cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"])
    xd, wd, bd, gyd = R.dev(x), R.dev(w), R.dev(b), R.dev(gy)
    y = torch.empty((cfg["N"], cfg["C_out"], Ho, Wo), device="cuda")
    gx = torch.empty(x.shape, device="cuda")
    gw = torch.empty(wshape, device="cuda")
    gb = torch.empty((cfg["C_out"],), device="cuda")
    nb = max(R.workspace(d, 0)[1], R.workspace(d, 1)[1])
    ws = torch.empty(nb // 4 + 64, device="cuda")
    st, g = hc.hc_conv2d_step_graph_create(d, xd, wd, bd, y, gyd, gx, gw, gb, ws, nb, ws, nb)
    hc.check(st, "graph create")
    try:
        hc.check(hc.hc_step_graph_launch(g), "graph launch")
        hc.check(hc.hc_sync_check(), "graph sync")
        for got, want in zip((y, gx, gw, gb), _eager(hc, cfg, x, w, b, gy)):
            assert np.array_equal(got.cpu().numpy(), want)
    finally:
        hc.check(hc.hc_step_graph_destroy(g), "graph destroy")


def test_step_graph_rejects_bad_args(hc):
    cfg = CASES["config1_dense5x5"]()[0]
    d = hc.desc(cfg)
    st, g = hc.hc_conv2d_step_graph_create(d, None, None, None, None, None, None, None, None, None, 0, None, 0)
    assert st == hc.HC_ERR_INVALID_ARG and not g.value
    assert hc.hc_step_graph_destroy(None) == 0
