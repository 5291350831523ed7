"""Full-size parity of the two multi-op workloads the bench times.

* The depthwise 7x7 + 2x2/s2 downsample on (7,256,128,2048), 8 shards.
* The ConvNeXt stage-1 block on the stem output of a (7,3,512,4096) image,
  8 shards.

Each runs one fwd+bwd step through bench.py's own workload classes: same
shapes, shard counts, algorithms, workspaces and call sequence.  The results
are checked against the oracle, computed from the workloads' original inputs.
Where an output depends on another op's output, the oracle computes that
intermediate itself, in full or on the slice a sample needs.  No value the
GPU computed is ever an oracle input.

Tolerances are the parity bar: normwise 1e-5 for outputs and input
gradients, 1e-4 for parameter gradients.  The block's parameter gradients
sum over all 917,504 pixels of a chain that LayerNorm couples across
channels.  Computing those sums needs the whole fp64 block, so they are
covered by the small-size family tests, not here.
"""
import os
import sys

import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_FWD = 1e-5
TOL_W = 1e-4


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def run_step(hc, wl):
    """One forward + backward step of a bench workload on cuda:0."""
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    runner = bench.Runner(hc, torch, torch.device("cuda", 0), stream)
    wl.setup(runner)
    wl.fwd()
    wl.bwd()
    hc.check(hc.hc_sync_check(stream), "workload step")


def host(t):
    return t.detach().cpu().numpy()


def at(t, pts):
    """Values of a device tensor at a list of index tuples (gathered on the device)."""
    idx = torch.as_tensor(np.array(pts, dtype=np.int64).T, device=t.device)
    return t[tuple(idx)].cpu().numpy()


def f32(a):
    return np.ascontiguousarray(a, np.float32)


# ---------------------------------------------------------------------------
# depthwise 7x7 + 2x2/s2 downsample, (7,256,128,2048), 8 shards of 256 columns

def down_grad_input(orc, w_dn, gz, n0, n1, c, r0, r1, c0, c1):
    """The downsample's grad_input for input channel c on images [n0, n1), rows
    [r0, r1) and columns [c0, c1) (even bounds): with kernel = stride = 2 every
    input position feeds one output, so it is the grad_input of that slice alone."""
    cfg = P.cfg_of(n1 - n0, 1, r1 - r0, c1 - c0, 512, 2, 2, 0, 1)
    return orc.conv2d_bwd_input(cfg, f32(w_dn[:, c:c + 1]), f32(gz[n0:n1, :, r0 // 2:r1 // 2, c0 // 2:c1 // 2]))


def test_dwdown_full_size(hc, orc):
    wl = bench.DwDownWorkload()
    run_step(hc, wl)
    N, C, H, W, S = 7, 256, 128, 2048, 8
    Wl = W // S
    x, gz = wl.h_x, wl.h_gz
    w_dw, w_dn = host(wl.w_dw), host(wl.w_dn)
    b_dw, b_dn = np.zeros(C, np.float32), np.zeros(512, np.float32)
    cd, cn = wl.dw, wl.down
    rng = np.random.default_rng(5)

    # depthwise forward, every output: the oracle's own depthwise output is the downsample's input
    dwo = orc.conv2d_fwd(cd, x, w_dw, b_dw).astype(np.float32)
    assert R.normwise(host(wl.dwo), dwo) <= TOL_FWD

    # downsample forward and grad_input on random points plus shard-edge columns
    zpts = [tuple(int(rng.integers(0, s)) for s in (N, 512, 64, 1024)) for _ in range(1500)]
    zpts += [(int(rng.integers(0, N)), int(rng.integers(0, 512)), i, j)
             for j in (0, 127, 128, 129, 511, 512, 895, 896, 1023) for i in (0, 31, 63)]
    zr = np.array([orc.fwd_at(cn, dwo, w_dn, b_dn, *p) for p in zpts])
    assert R.normwise(at(wl.z, zpts), zr) <= TOL_FWD
    gpts = [tuple(int(rng.integers(0, s)) for s in (N, C, H, W)) for _ in range(1500)]
    gpts += [(int(rng.integers(0, N)), int(rng.integers(0, C)), i, j)
             for j in (0, 1, 255, 256, 257, 1023, 1024, 2046, 2047) for i in (0, 1, 127)]
    gr = np.array([orc.gx_at(cn, w_dn, gz, *p) for p in gpts])
    assert R.normwise(at(wl.gd, gpts), gr) <= TOL_FWD

    # downsample grad_weight (sampled elements) and grad_bias (every channel)
    wpts = [tuple(int(rng.integers(0, s)) for s in (512, C, 2, 2)) for _ in range(12)] + [(0, 0, 0, 0), (511, 255, 1, 1)]
    gw_dn = host(wl.gw_dn)
    wr = np.array([orc.gw_at(cn, dwo, gz, *p, 0, 1024) for p in wpts])
    assert R.normwise(np.array([gw_dn[p] for p in wpts]), wr) <= TOL_W
    br = np.array([orc.gb_at(cn, gz, co, 0, 1024) for co in range(512)])
    assert R.normwise(host(wl.gb_dn), br) <= TOL_W

    # depthwise grad_input on sampled points: the oracle's downsample grad_input on
    # the even-aligned patch covering the point's 7x7 neighbourhood, then the
    # depthwise grad_input of that patch (zeros past the patch are past the image)
    xpts = [tuple(int(rng.integers(0, s)) for s in (N, C, H, W)) for _ in range(120)]
    xpts += [(int(rng.integers(0, N)), int(rng.integers(0, C)), i, j)
             for j in (0, 2, 254, 255, 256, 258, 1791, 1792, 2045, 2047) for i in (0, 2, 64, 125, 127)]
    ref = []
    for (n, c, h, w) in xpts:
        r0, r1 = max(0, (h - 3) & ~1), min(H, (h + 5) & ~1)
        c0, c1 = max(0, (w - 3) & ~1), min(W, (w + 5) & ~1)
        gd = f32(down_grad_input(orc, w_dn, gz, n, n + 1, c, r0, r1, c0, c1))
        cfg = P.cfg_of(1, 1, r1 - r0, c1 - c0, 1, 7, 1, 3, 1)
        ref.append(orc.gx_at(cfg, f32(w_dw[c:c + 1]), gd, 0, 0, h - r0, w - c0))
    assert R.normwise(at(wl.gx, xpts), np.array(ref)) <= TOL_FWD

    # depthwise grad_weight / grad_bias of two channels, as the sum of their
    # per-shard partials: each shard's grad_output slice from the oracle, and the
    # shard's input block with its 3-column halos (zeros past the image) and 3 zero rows
    gw_dw, gb_dw = host(wl.gw_dw), host(wl.gb_dw)
    chans, gw_all, gb_all = (0, 201), [], []
    for c in chans:
        gw_ref, gb_ref = np.zeros((7, 7)), 0.0
        for r in range(S):
            j0, j1 = r * Wl, (r + 1) * Wl
            gd = f32(down_grad_input(orc, w_dn, gz, 0, N, c, 0, H, j0, j1))
            xs = np.zeros((N, 1, H + 6, Wl + 6), np.float32)
            lo, hi = max(0, j0 - 3), min(W, j1 + 3)
            xs[:, 0, 3:3 + H, lo - (j0 - 3):hi - (j0 - 3)] = x[:, c, :, lo:hi]
            cfg = P.cfg_of(N, 1, H + 6, Wl + 6, 1, 7, 1, 0, 1)
            gw_ref += orc.conv2d_bwd_weight(cfg, xs, gd)[0, 0]
            gb_ref += orc.conv2d_bwd_bias(cfg, gd)[0]
        gw_all.append(gw_ref)
        gb_all.append(gb_ref)
    assert R.normwise(gw_dw[list(chans), 0], np.array(gw_all)) <= TOL_W
    assert R.normwise(gb_dw[list(chans)], np.array(gb_all)) <= TOL_W


# ---------------------------------------------------------------------------
# ConvNeXt stage-1 block on the stem output of a (7,3,512,4096) image, 8 shards

def stem_patch(orc, img, w_stem, n, i, j, r):
    """The stem output (256 channels) on rows i-r..i+r and columns j-r..j+r of
    the (128, 1024) output grid, zeros outside it (the depthwise conv's padding):
    the oracle's 4x4/s4 conv of the image rows and columns under those outputs."""
    Ho, Wo = 128, 1024
    ra, rb, ca, cb = max(0, i - r), min(Ho, i + r + 1), max(0, j - r), min(Wo, j + r + 1)
    cfg = P.cfg_of(1, 3, 4 * (rb - ra), 4 * (cb - ca), 256, 4, 4, 0, 1)
    sub = orc.conv2d_fwd(cfg, f32(img[n:n + 1, :, 4 * ra:4 * rb, 4 * ca:4 * cb]), w_stem, np.zeros(256, np.float32))
    out = np.zeros((1, 256, 2 * r + 1, 2 * r + 1), np.float32)
    out[:, :, ra - (i - r):rb - (i - r), ca - (j - r):cb - (j - r)] = sub
    return out


def test_block_full_size(hc, orc):
    wl = bench.BlockWorkload()
    run_step(hc, wl)
    img, gy = wl.h_img, wl.h_gy
    w_stem, w_dw, w1, w2 = (host(t) for t in (wl.w_stem, wl.w_dw, wl.w1, wl.w2))
    ls = host(wl.ls_g)
    ones, zeros = np.ones(256), np.zeros(256)
    z256, z1024 = np.zeros(256, np.float32), np.zeros(1024, np.float32)
    eps = 1e-6
    rng = np.random.default_rng(6)
    pix = [tuple(int(rng.integers(0, s)) for s in (7, 128, 1024)) for _ in range(24)]
    pix += [(int(rng.integers(0, 7)), i, j) for (i, j) in
            ((0, 0), (127, 1023), (64, 127), (64, 128), (3, 511), (124, 512), (1, 895), (126, 896))]

    got = {k: [] for k in ("s", "dwo", "ln", "mean", "rstd", "h", "b2", "out", "g_b2", "g_a", "g_l", "g_d")}
    ref = {k: [] for k in got}
    dw7 = P.cfg_of(1, 256, 13, 13, 256, 7, 1, 0, 256)       # valid 7x7 conv: 13x13 -> 7x7
    pw1 = P.cfg_of(1, 256, 7, 7, 1024, 1, 1, 0, 1)
    pw2 = P.cfg_of(1, 1024, 7, 7, 256, 1, 1, 0, 1)
    for (n, i, j) in pix:
        # forward on the 7x7 pixels around (i, j): every op after the depthwise conv is per pixel
        s13 = stem_patch(orc, img, w_stem, n, i, j, 6)
        dwo = f32(orc.conv2d_fwd(dw7, s13, w_dw, z256))                # (1,256,7,7)
        ln, mean, rstd = orc.layernorm_c_fwd(dwo, ones, zeros, eps)
        h = f32(orc.conv2d_fwd(pw1, f32(ln), w1, z1024))
        a = f32(orc.gelu_fwd(h))
        b2 = f32(orc.conv2d_fwd(pw2, a, w2, z256))
        s7 = s13[:, :, 3:10, 3:10]
        out = orc.layerscale_residual_fwd(s7, b2, ls)
        # backward on the same pixels from the original grad_output
        ra, ca = i - 3, j - 3
        g7 = np.zeros((1, 256, 7, 7), np.float32)
        rr = slice(max(0, ra), min(128, ra + 7))
        cc = slice(max(0, ca), min(1024, ca + 7))
        g7[:, :, rr.start - ra:rr.stop - ra, cc.start - ca:cc.stop - ca] = gy[n:n + 1, :, rr, cc]
        _, g_b2, _ = orc.layerscale_residual_bwd(b2, ls, g7)
        g_a = orc.conv2d_bwd_input(pw2, w2, f32(g_b2))
        g_h = orc.gelu_bwd(h, g_a)
        g_l = orc.conv2d_bwd_input(pw1, w1, f32(g_h))
        g_d, _, _ = orc.layernorm_c_bwd(dwo, ones, g_l, eps)
        c = (0, slice(None), 3, 3)
        for k, v in (("s", s7), ("dwo", dwo), ("ln", ln), ("h", h), ("b2", b2), ("out", out), ("g_b2", g_b2),
                     ("g_a", g_a), ("g_l", g_l), ("g_d", g_d)):
            ref[k].append(v[c])
        ref["mean"].append(mean[0, 24])
        ref["rstd"].append(rstd[0, 24])
        g = lambda t: t[n, :, i, j].cpu().numpy()
        for k, t in (("s", wl.s), ("dwo", wl.dwo), ("ln", wl.ln), ("h", wl.h), ("b2", wl.b2), ("out", wl.out),
                     ("g_b2", wl.g_b2), ("g_a", wl.g_a), ("g_l", wl.g_l), ("g_d", wl.g_d)):
            got[k].append(g(t))
        got["mean"].append(float(wl.mean[n, i * 1024 + j]))
        got["rstd"].append(float(wl.rstd[n, i * 1024 + j]))
    for k in got:
        err = R.normwise(np.array(got[k]), np.array(ref[k]))
        assert err <= TOL_FWD, (k, err)
