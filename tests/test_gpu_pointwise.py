"""GPU parity of the ConvNeXt block's pointwise ops (LayerNorm over C, GELU,
layer scale + residual) against the fp64 oracle, through the C ABI.
Tolerances (normwise): outputs and input gradients 1e-5, parameter gradients 1e-4."""
import numpy as np
import pytest
import torch

import hc_run as R
from spatially_sharded_cnn_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available()
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def _ws(hc, N, C, HW):
    st, nb = hc.hc_pointwise_workspace_size(N, C, HW)
    hc.check(st)
    return torch.empty(nb // 4 + 64, device="cuda"), nb


# C = 256 runs the persistent register kernel: (2, 256, 128, 160) gives 1280
# 32-pixel groups, several per block; (1, 256, 97, 113) a ragged last group
@pytest.mark.parametrize("shape", [(2, 256, 37, 29), (1, 96, 8, 64), (3, 32, 1, 5), (2, 256, 128, 160),
                                   (1, 256, 97, 113)])
def test_layernorm(hc, orc, shape):
    N, C, H, W = shape
    HW = H * W
    x = synth.normal(shape, 2.0, 5, 1) + np.float32(0.3)
    gamma = (1.0 + synth.normal((C,), 0.1, 5, 2)).astype(np.float32)
    beta = synth.normal((C,), 0.1, 5, 3)
    gy = synth.normal(shape, 1.0, 5, 4)
    eps = 1e-6
    y, mean, rstd = R.Guarded(shape), R.Guarded((N, HW)), R.Guarded((N, HW))
    xd, gd, bd, gyd = R.dev(x), R.dev(gamma), R.dev(beta), R.dev(gy)
    hc.check(hc.hc_layernorm_c_fwd(N, C, HW, xd, gd, bd, eps, y.view, mean.view, rstd.view))
    hc.check(hc.hc_sync_check())
    yr, mr, rr = orc.layernorm_c_fwd(x, gamma, beta, eps)
    assert R.normwise(y.numpy(), yr) <= 1e-5
    assert R.normwise(mean.numpy(), mr) <= 1e-5
    assert R.normwise(rstd.numpy(), rr) <= 1e-5
    gx, gg, gb = R.Guarded(shape), R.Guarded((C,)), R.Guarded((C,))
    ws, nb = _ws(hc, N, C, HW)
    hc.check(hc.hc_layernorm_c_bwd(N, C, HW, xd, gd, mean.view, rstd.view, gyd, gx.view, gg.view, gb.view, ws, nb))
    hc.check(hc.hc_sync_check())
    gxr, ggr, gbr = orc.layernorm_c_bwd(x, gamma, gy, eps)
    assert R.normwise(gx.numpy(), gxr) <= 1e-5
    assert R.normwise(gg.numpy(), ggr) <= 1e-4
    assert R.normwise(gb.numpy(), gbr) <= 1e-4
    # a second call gives the same bits (fixed summation order)
    gx2, gg2, gb2 = R.Guarded(shape), R.Guarded((C,)), R.Guarded((C,))
    hc.check(hc.hc_layernorm_c_bwd(N, C, HW, xd, gd, mean.view, rstd.view, gyd, gx2.view, gg2.view, gb2.view, ws, nb))
    hc.check(hc.hc_sync_check())
    for a, b in ((gx, gx2), (gg, gg2), (gb, gb2)):
        assert np.array_equal(a.numpy(), b.numpy())


@pytest.mark.parametrize("n", [4096 * 3 + 3, 7, 1 << 20])
def test_gelu(hc, orc, n):
    x = synth.normal((n,), 2.5, 6, 1)
    gy = synth.normal((n,), 1.0, 6, 2)
    y, gx = R.Guarded((n,)), R.Guarded((n,))
    hc.check(hc.hc_gelu_fwd(n, R.dev(x), y.view))
    hc.check(hc.hc_gelu_bwd(n, R.dev(x), R.dev(gy), gx.view))
    hc.check(hc.hc_sync_check())
    assert R.normwise(y.numpy(), orc.gelu_fwd(x)) <= 1e-5
    assert R.normwise(gx.numpy(), orc.gelu_bwd(x, gy)) <= 1e-5


@pytest.mark.parametrize("shape", [(2, 64, 9, 33), (1, 256, 16, 128)])
def test_layerscale_residual(hc, orc, shape):
    N, C, H, W = shape
    HW = H * W
    res = synth.normal(shape, 1.0, 7, 1)
    br = synth.normal(shape, 1.0, 7, 2)
    gamma = synth.normal((C,), 1e-2, 7, 3)
    gy = synth.normal(shape, 1.0, 7, 4)
    out = R.Guarded(shape)
    hc.check(hc.hc_layerscale_residual_fwd(N, C, HW, R.dev(res), R.dev(br), R.dev(gamma), out.view))
    gbr, gg = R.Guarded(shape), R.Guarded((C,))
    ws, nb = _ws(hc, N, C, HW)
    hc.check(hc.hc_layerscale_residual_bwd(N, C, HW, R.dev(br), R.dev(gamma), R.dev(gy), gbr.view, gg.view, ws, nb))
    hc.check(hc.hc_sync_check())
    assert R.normwise(out.numpy(), orc.layerscale_residual_fwd(res, br, gamma)) <= 1e-5
    _, gbrr, ggr = orc.layerscale_residual_bwd(br, gamma, gy)
    assert R.normwise(gbr.numpy(), gbrr) <= 1e-5
    assert R.normwise(gg.numpy(), ggr) <= 1e-4


@pytest.mark.parametrize("n", [1 << 16, 4097])
def test_add_inplace(hc, n):
    a = synth.normal((n,), 1.0, 8, 1)
    b = synth.normal((n,), 1.0, 8, 2)
    y = R.Guarded((n,))
    y.view.copy_(torch.from_numpy(a))
    hc.check(hc.hc_add_inplace(n, y.view, R.dev(b)))
    hc.check(hc.hc_sync_check())
    assert np.array_equal(y.numpy(), (a + b).astype(np.float32))


@pytest.mark.parametrize("N,p,seed,offset", [(7, 0.1, 0, 0), (4096, 0.3, 12345, 0), (100_003, 0.5, 2 ** 63 + 5, 77),
                                             (33, 0.0, 9, 1), (1, 0.999, 3, 2 ** 40)])
def test_drop_path_mask_bitexact(hc, orc, N, p, seed, offset):
    """The device draw equals the oracle's SplitMix64 draw bit for bit."""
    m = R.Guarded((N,))
    hc.check(hc.hc_drop_path_mask(N, p, seed, offset, m.view))
    hc.check(hc.hc_sync_check())
    assert np.array_equal(m.numpy(), orc.drop_path_mask(N, p, seed, offset))


def test_drop_path_mask_shard_consistent(hc, orc):
    """A slice of the batch drawn with offset = its first sample (what a device or
    shard holding those samples would call) equals that slice of the full draw."""
    N, p, seed = 1000, 0.25, 31337
    full = R.Guarded((N,))
    hc.check(hc.hc_drop_path_mask(N, p, seed, 0, full.view))
    parts = []
    for a, b in ((0, 250), (250, 500), (500, 1000)):
        g = R.Guarded((b - a,))
        hc.check(hc.hc_drop_path_mask(b - a, p, seed, a, g.view))
        parts.append(g)
    hc.check(hc.hc_sync_check())
    assert np.array_equal(np.concatenate([g.numpy() for g in parts]), full.numpy())
    st = hc.hc_drop_path_mask(N, 1.0, seed, 0, full.view)
    assert st == hc.HC_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [(8, 64, 9, 17), (3, 256, 4, 128)])
def test_layerscale_droppath(hc, orc, shape):
    N, C, H, W = shape
    HW = H * W
    res = synth.normal(shape, 1.0, 9, 1)
    br = synth.normal(shape, 1.0, 9, 2)
    gamma = synth.normal((C,), 1e-1, 9, 3)
    gy = synth.normal(shape, 1.0, 9, 4)
    mask = R.dev(orc.drop_path_mask(N, 0.4, 2024, 0))
    hmask = mask.cpu().numpy()
    assert 0 < np.count_nonzero(hmask) < N   # both kept and dropped samples
    out = R.Guarded(shape)
    hc.check(hc.hc_layerscale_droppath_fwd(N, C, HW, R.dev(res), R.dev(br), R.dev(gamma), mask, out.view))
    gbr, gg = R.Guarded(shape), R.Guarded((C,))
    ws, nb = _ws(hc, N, C, HW)
    hc.check(hc.hc_layerscale_droppath_bwd(N, C, HW, R.dev(br), R.dev(gamma), mask, R.dev(gy), gbr.view, gg.view,
                                           ws, nb))
    hc.check(hc.hc_sync_check())
    o = out.numpy()
    assert R.normwise(o, orc.layerscale_droppath_fwd(res, br, gamma, hmask)) <= 1e-5
    for n in np.flatnonzero(hmask == 0):
        assert np.array_equal(o[n], res[n]) and np.all(gbr.numpy()[n] == 0)
    _, gbrr, ggr = orc.layerscale_droppath_bwd(br, gamma, hmask, gy)
    assert R.normwise(gbr.numpy(), gbrr) <= 1e-5
    assert R.normwise(gg.numpy(), ggr) <= 1e-4
    # no mask: bit-identical to the plain layer scale
    o1, o2 = R.Guarded(shape), R.Guarded(shape)
    hc.check(hc.hc_layerscale_droppath_fwd(N, C, HW, R.dev(res), R.dev(br), R.dev(gamma), None, o1.view))
    hc.check(hc.hc_layerscale_residual_fwd(N, C, HW, R.dev(res), R.dev(br), R.dev(gamma), o2.view))
    hc.check(hc.hc_sync_check())
    assert np.array_equal(o1.numpy(), o2.numpy())
