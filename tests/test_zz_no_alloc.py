"""The depthwise backward entry point that allocates nothing.

Some callers may not allocate device memory when they call the backward pass
(their memory belongs to another framework's allocator, or they must not
allocate after start-up), so they cannot hand hc_conv2d_bwd a workspace.
hc_conv2d_bwd_depthwise_noalloc keeps that scratch in a library-owned static
device array instead.  This test checks, through the C ABI, that two calls in a
row give the same results as the workspace-taking entry point (within the
tolerances the other GPU tests use), and that sizes beyond the array are
refused.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P
from spatially_sharded_cnn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_GX = 1e-5
TOL_W = 1e-4


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def _case(N, C, H, W, S, seed):
    cfg = P.cfg_of(N, C, H, W, C, 7, 1, 3, C, S)
    x = synth.normal((N, C, H, W), 1.0, seed, 1)
    w = synth.trunc_normal((C, 1, 7, 7), 0.02, seed, 2)
    gy = synth.normal((N, C, H, W), 1.0, seed, 4)
    return cfg, x, w, gy


def _outputs(cfg, S):
    wshape = (cfg["C_out"], 1, 7, 7)
    return dict(gx=R.Guarded((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"])), gw=R.Guarded(wshape),
                gb=R.Guarded((cfg["C_out"],)), gwp=R.Guarded((S,) + wshape), gbp=R.Guarded((S, cfg["C_out"])))


@pytest.mark.parametrize("shape", [(2, 4, 70, 512, 4), (1, 8, 40, 512, 2)], ids=["ragged_S4", "two_tiles_S2"])
def test_noalloc_matches_workspace_entry_point(hc, shape):
    N, C, H, W, S = shape
    cfg, x, w, gy = _case(N, C, H, W, S, seed=11)
    d = hc.desc(cfg)
    xd, wd, gyd = R.dev(x), R.dev(w), R.dev(gy)
    ref = _outputs(cfg, S)
    ws, nb = R.workspace(d, 1, hc.HC_ALGO_DEPTHWISE)
    hc.check(hc.hc_conv2d_bwd(d, xd, wd, gyd, ref["gx"].view, ref["gw"].view, ref["gb"].view, ref["gwp"].view,
                              ref["gbp"].view, ws, nb, algo=hc.HC_ALGO_DEPTHWISE), "workspace bwd")
    hc.check(hc.hc_sync_check(), "workspace bwd sync")
    want = {k: v.numpy() for k, v in ref.items()}
    for call in range(2):  # the shared scratch keeps the previous call's contents
        got = _outputs(cfg, S)
        hc.check(hc.hc_conv2d_bwd_depthwise_noalloc(d, xd, wd, gyd, got["gx"].view, got["gw"].view, got["gb"].view,
                                                     got["gwp"].view, got["gbp"].view), f"noalloc call {call}")
        hc.check(hc.hc_sync_check(), f"noalloc sync {call}")
        g = {k: v.numpy() for k, v in got.items()}
        assert R.normwise(g["gx"], want["gx"]) <= TOL_GX
        for k in ("gw", "gb", "gwp", "gbp"):
            assert R.normwise(g[k], want[k]) <= TOL_W, (call, k)
    # weight gradients only (grad_input skipped, partials kept in the scratch)
    got = _outputs(cfg, S)
    hc.check(hc.hc_conv2d_bwd_depthwise_noalloc(d, xd, wd, gyd, None, got["gw"].view, got["gb"].view), "noalloc w")
    hc.check(hc.hc_sync_check(), "noalloc w sync")
    assert R.normwise(got["gw"].numpy(), want["gw"]) <= TOL_W
    assert R.normwise(got["gb"].numpy(), want["gb"]) <= TOL_W


def test_noalloc_refuses_oversized_and_unsupported(hc):
    # 64 images x 1024 channels x 16 column tiles of 7x7 partials: far beyond 16 MiB
    big = hc.desc(P.cfg_of(64, 1024, 8, 2048, 1024, 7, 1, 3, 1024, 1))
    assert hc.hc_conv2d_bwd_depthwise_noalloc(big, 256, 256, 256, 256, 256, 256) == hc.HC_ERR_WORKSPACE
    dense = hc.desc(P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4))
    assert hc.hc_conv2d_bwd_depthwise_noalloc(dense, 256, 256, 256, 256, 256, 256) == hc.HC_ERR_UNSUPPORTED
