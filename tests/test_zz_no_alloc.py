"""The depthwise backward entry point that allocates nothing.

Some callers may not allocate device memory when they call the backward pass
(their memory belongs to another framework's allocator, or they must not
allocate after start-up), so they cannot hand hc_conv2d_bwd a workspace.
hc_conv2d_bwd_depthwise_noalloc keeps that scratch in a library-owned static
device array instead.  This test checks, through the C ABI, that two calls in a
row give bit-for-bit the results of the workspace-taking entry point (same
kernels, same sums in the same order), that they match the oracle within the
tolerances the other GPU tests use -- including a case whose scratch reaches
past the middle of the 16 MiB array -- and that sizes beyond the array are
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


def _scratch_bytes(N, C, W, S):
    """The entry point's scratch for a depthwise 7x7 desc: shard partials of the
    weight and bias gradients, then per-(shard, channel, 128-column tile, image)
    partials of 49 + 1 floats, each region rounded up to 256 bytes."""
    r = lambda b: (b + 255) // 256 * 256
    return r(4 * S * C * 49) + r(4 * S * C) + r(4 * S * C * (W // S // 128) * N * 50)


# (N, C, H, W, S): a ragged row tile over 4 shards; two column tiles per shard; and
# 12 images x 256 channels x 8 tiles per shard x 2 shards, whose 9.9 MB of scratch
# runs past the first 8 MiB of the array
SHAPES = [(2, 4, 70, 512, 4), (1, 8, 40, 512, 2), (12, 256, 8, 2048, 2)]


@pytest.mark.parametrize("shape", SHAPES, ids=["ragged_S4", "two_tiles_S2", "scratch_past_8MiB"])
def test_noalloc_matches_workspace_entry_point_and_oracle(hc, orc, shape):
    N, C, H, W, S = shape
    cfg, x, w, gy = _case(N, C, H, W, S, seed=11)
    if shape == SHAPES[2]:
        assert _scratch_bytes(N, C, W, S) > (8 << 20)
    d = hc.desc(cfg)
    xd, wd, gyd = R.dev(x), R.dev(w), R.dev(gy)
    ref = _outputs(cfg, S)
    ws, nb = R.workspace(d, 1, hc.HC_ALGO_DEPTHWISE)
    hc.check(hc.hc_conv2d_bwd(d, xd, wd, gyd, ref["gx"].view, ref["gw"].view, ref["gb"].view, ref["gwp"].view,
                              ref["gbp"].view, ws, nb, algo=hc.HC_ALGO_DEPTHWISE), "workspace bwd")
    hc.check(hc.hc_sync_check(), "workspace bwd sync")
    want = {k: v.numpy() for k, v in ref.items()}
    # the oracle: unsharded gradients and the sharded method's per-shard partials
    o_gx = orc.conv2d_bwd_input(cfg, w, gy)
    o_gw = orc.conv2d_bwd_weight(cfg, x, gy)
    o_gb = orc.conv2d_bwd_bias(cfg, gy)
    _, o_gwp, o_gbp = orc.sharded_bwd(cfg, x, w, gy)
    oracle_ref = dict(gx=o_gx, gw=o_gw, gb=o_gb, gwp=o_gwp, gbp=o_gbp)
    for call in range(2):  # the shared scratch keeps the previous call's contents
        got = _outputs(cfg, S)
        hc.check(hc.hc_conv2d_bwd_depthwise_noalloc(d, xd, wd, gyd, got["gx"].view, got["gw"].view, got["gb"].view,
                                                     got["gwp"].view, got["gbp"].view), f"noalloc call {call}")
        hc.check(hc.hc_sync_check(), f"noalloc sync {call}")
        g = {k: v.numpy() for k, v in got.items()}
        for k in want:
            assert np.array_equal(g[k], want[k]), (call, k)  # same kernels and sums: bit-identical
        assert R.normwise(g["gx"], oracle_ref["gx"]) <= TOL_GX, call
        for k in ("gw", "gb", "gwp", "gbp"):
            assert R.normwise(g[k], oracle_ref[k]) <= TOL_W, (call, k)
    # weight gradients only (grad_input skipped, partials kept in the scratch)
    got = _outputs(cfg, S)
    hc.check(hc.hc_conv2d_bwd_depthwise_noalloc(d, xd, wd, gyd, None, got["gw"].view, got["gb"].view), "noalloc w")
    hc.check(hc.hc_sync_check(), "noalloc w sync")
    assert np.array_equal(got["gw"].numpy(), want["gw"])
    assert np.array_equal(got["gb"].numpy(), want["gb"])


def test_noalloc_refuses_oversized_and_unsupported(hc):
    # 64 images x 1024 channels x 16 column tiles of 7x7 partials: far beyond 16 MiB
    big = hc.desc(P.cfg_of(64, 1024, 8, 2048, 1024, 7, 1, 3, 1024, 1))
    assert hc.hc_conv2d_bwd_depthwise_noalloc(big, 256, 256, 256, 256, 256, 256) == hc.HC_ERR_WORKSPACE
    dense = hc.desc(P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4))
    assert hc.hc_conv2d_bwd_depthwise_noalloc(dense, 256, 256, 256, 256, 256, 256) == hc.HC_ERR_UNSUPPORTED
