"""One rank of the pages' multi-device layout, on one GPU.

Each rank of a W-sharded depthwise convolution keeps its column block in the
halo-padded layout and gets its halo columns from its neighbours (NVIDIA blog
"Perception model training for autonomous vehicles with tensor parallelism",
design section and Figure 1; kwkr.cn news/18980, 2.2), computing the tiles
away from the block edges while the halo is in flight (kwkr.cn 5.2).  Here the
ranks run one after another on one device and their exchange is a device copy
of the packed columns (hc_halo_pack on the sender, hc_halo_unpack on the
receiver), so no kernel waits on another.  Checked:

* the exchanged margins equal the oracle's halo columns bit for bit;
* forward and grad_input of every rank equal the single-device sharded call
  bit for bit, and the oracle within 1e-5;
* interior tiles then edge tiles give the same bits as all tiles at once;
* each rank's _Partial grad_weight / grad_bias equal the oracle's shard
  partials within 1e-4, and their rank-order sum (hc_sum_partials) the full
  gradients.
"""
import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P
from spatially_sharded_cnn_gb300 import synth

pytestmark = pytest.mark.gpu
H4 = 4  # HC_HALO_COLS


@pytest.fixture(scope="module")
def hc():
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def _case(N, C, H, W, K, S, seed=21):
    cfg = P.cfg_of(N, C, H, W, C, K, 1, (K - 1) // 2, C, S)
    x = synth.normal((N, C, H, W), 1.0, seed, 1)
    w = synth.trunc_normal((C, 1, K, K), 0.02, seed, 2)
    b = synth.normal((C,), 0.1, seed, 3)
    gy = synth.normal((N, C, H, W), 1.0, seed, 4)
    return cfg, x, w, b, gy


def _padded_blocks(hc, d, t, S, Wl):
    """Every rank's halo-padded block of device tensor t, margins exchanged."""
    N, C, H, _ = t.shape
    pads = []
    for r in range(S):
        loc = t[..., r * Wl:(r + 1) * Wl].contiguous()
        xp = torch.full((N, C, H, Wl + 2 * H4), float("nan"), device="cuda")
        hc.check(hc.hc_halo_pad(d, loc, xp), "pad")
        pads.append(xp)
    buf = torch.empty((N * C * H, H4), device="cuda")
    for r in range(S):  # the exchange: r's edge columns into its neighbours' margins
        for side, nb, nb_side in ((0, r - 1, 1), (1, r + 1, 0)):
            if 0 <= nb < S:
                hc.check(hc.hc_halo_pack(d, pads[r], side, buf), "pack")
                hc.check(hc.hc_halo_unpack(d, buf, nb_side, pads[nb]), "unpack")
    hc.check(hc.hc_halo_unpack(d, None, 0, pads[0]), "left image edge")
    hc.check(hc.hc_halo_unpack(d, None, 1, pads[S - 1]), "right image edge")
    return pads


# (N, C, H, W, K, S): 4 tiles per rank (interior tiles 1-2), 2 (edges only), 1; K = 3, 5, 7; ragged rows
CASES = [(2, 8, 70, 1024, 7, 2), (1, 4, 64, 1024, 7, 4), (2, 4, 40, 1024, 5, 8), (1, 4, 20, 768, 3, 2)]


@pytest.mark.parametrize("shape", CASES, ids=[f"K{c[4]}_S{c[5]}_T{c[3] // c[5] // 128}" for c in CASES])
def test_rank_path(hc, orc, shape):
    N, C, H, W, K, S = shape
    cfg, x, w, b, gy = _case(*shape)
    d = hc.desc(cfg)
    Wl, p = W // S, (K - 1) // 2
    xd, wd, bd, gyd = R.dev(x), R.dev(w), R.dev(b), R.dev(gy)
    xpads = _padded_blocks(hc, d, xd, S, Wl)
    gypads = _padded_blocks(hc, d, gyd, S, Wl)
    # the margins are the pages' halo columns (oracle: halo exchange + concat)
    for r in range(S):
        ext = orc.halo_extend(cfg, r, x)
        got = xpads[r][..., H4 - p:H4 + Wl + p].cpu().numpy()
        assert np.array_equal(got, ext[..., :Wl + 2 * p]), r
    # single-device sharded reference (the same kernels over the whole tensor)
    y_ref = R.fwd(cfg, x, w, b, algo=hc.HC_ALGO_DEPTHWISE)
    out_ref = R.bwd(cfg, x, w, gy, algo=hc.HC_ALGO_DEPTHWISE)
    o_y = orc.conv2d_fwd(cfg, x, w, b)
    o_gx = orc.conv2d_bwd_input(cfg, w, gy)
    o_gw, o_gb = orc.conv2d_bwd_weight(cfg, x, gy), orc.conv2d_bwd_bias(cfg, gy)
    _, o_gwp, o_gbp = orc.sharded_bwd(cfg, x, w, gy)
    st, nb = hc.hc_conv2d_workspace_size_rank(d)
    hc.check(st, "ws")
    ws = torch.empty(nb // 4 + 64, device="cuda")
    ys, gxs, gwps, gbps = [], [], [], []
    for r in range(S):
        y_all = torch.full((N, C, H, Wl), float("nan"), device="cuda")
        hc.check(hc.hc_conv2d_fwd_rank(d, xpads[r], wd, bd, y_all, hc.HC_TILES_ALL), "fwd all")
        y_split = torch.full_like(y_all, float("nan"))
        hc.check(hc.hc_conv2d_fwd_rank(d, xpads[r], wd, bd, y_split, hc.HC_TILES_INTERIOR), "fwd interior")
        hc.check(hc.hc_conv2d_fwd_rank(d, xpads[r], wd, bd, y_split, hc.HC_TILES_EDGE), "fwd edge")
        gx_all = torch.full_like(y_all, float("nan"))
        gwp = torch.empty_like(wd)
        gbp = torch.empty_like(bd)
        hc.check(hc.hc_conv2d_bwd_rank(d, xpads[r], wd, gypads[r], gx_all, gwp, gbp, ws, nb, hc.HC_TILES_ALL),
                 "bwd all")
        gx_split = torch.full_like(y_all, float("nan"))
        gwp2, gbp2 = torch.empty_like(wd), torch.empty_like(bd)
        hc.check(hc.hc_conv2d_bwd_rank(d, xpads[r], wd, gypads[r], gx_split, gwp2, gbp2, ws, nb,
                                       hc.HC_TILES_INTERIOR), "bwd interior")
        hc.check(hc.hc_conv2d_bwd_rank(d, xpads[r], wd, gypads[r], gx_split, gwp2, gbp2, ws, nb, hc.HC_TILES_EDGE),
                 "bwd edge")
        hc.check(hc.hc_sync_check(), "sync")
        assert torch.equal(y_all, y_split) and torch.equal(gx_all, gx_split), r
        assert R.normwise(gwp2.cpu().numpy(), gwp.cpu().numpy()) <= 1e-6
        ys.append(y_all.cpu().numpy())
        gxs.append(gx_all.cpu().numpy())
        gwps.append(gwp)
        gbps.append(gbp)
    y = np.concatenate(ys, axis=3)
    gx = np.concatenate(gxs, axis=3)
    assert np.array_equal(y, y_ref) and np.array_equal(gx, out_ref["gx"])
    assert R.normwise(y, o_y) <= 1e-5 and R.normwise(gx, o_gx) <= 1e-5
    for r in range(S):
        assert R.normwise(gwps[r].cpu().numpy(), o_gwp[r]) <= 1e-4, r
        assert R.normwise(gbps[r].cpu().numpy(), o_gbp[r]) <= 1e-4, r
    gw_sum, gb_sum = torch.empty_like(wd), torch.empty_like(bd)
    hc.check(hc.hc_sum_partials(torch.stack(gwps), S, wd.numel(), gw_sum), "sum gw")
    hc.check(hc.hc_sum_partials(torch.stack(gbps), S, bd.numel(), gb_sum), "sum gb")
    assert R.normwise(gw_sum.cpu().numpy(), o_gw) <= 1e-4 and R.normwise(gb_sum.cpu().numpy(), o_gb) <= 1e-4


def test_rank_path_rejects(hc):
    d = hc.desc(P.cfg_of(1, 4, 16, 256, 4, 5, 1, 2, 1, 2))  # dense: not the depthwise kernels
    assert hc.hc_conv2d_fwd_rank(d, 256, 256, None, 256) == hc.HC_ERR_UNSUPPORTED
    d = hc.desc(P.cfg_of(1, 4, 16, 384, 4, 7, 1, 3, 4, 2))  # 192-column blocks: not whole 128-column tiles
    assert hc.hc_conv2d_fwd_rank(d, 256, 256, None, 256) == hc.HC_ERR_UNSUPPORTED
    d = hc.desc(P.cfg_of(1, 4, 16, 512, 4, 7, 1, 3, 4, 2))
    assert hc.hc_conv2d_fwd_rank(d, 256, 256, None, 256, 3) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_halo_pack(d, 256, 2, 256) == hc.HC_ERR_INVALID_ARG
