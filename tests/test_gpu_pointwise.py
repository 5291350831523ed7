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


@pytest.mark.parametrize("shape", [(2, 256, 37, 29), (1, 96, 8, 64), (3, 32, 1, 5)])
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
