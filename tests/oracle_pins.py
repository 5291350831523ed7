"""Pins of the CPU oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch.  ``test_oracle.py`` runs them against the oracle, and
``test_oracle_mutants.py`` runs them against copies of the oracle with a
planted mistake, each of which must fail at least one pin.

What pins what:
  * forward conv        -- torch CPU conv2d in fp64 (a library routine),
                           scipy.signal.correlate2d, the 1x1 case as a numpy
                           matrix product, one-hot (delta) kernels as exact shifts;
  * grad_input / weight / bias -- torch autograd in fp64, the dense Jacobian
                           enumerated column by column, the adjoint identities;
  * shard plan, halo, crop -- the shapes printed on the pages (tests/golden),
                           numpy slicing of a zero-padded array, and the
                           invariant that the sharded result equals the unsharded
                           one for every shard count;
  * LayerNorm / GELU / layer scale -- torch fp64 functions and autograd, closed
                           forms (mean 0, variance 1, GELU(0) = 0, GELU'(0) = 1/2,
                           Phi(1)), central finite differences;
  * DropPath mask         -- the published first outputs of SplitMix64
                           (tests/golden/splitmix64.json), the keep decision on
                           those bits, p = 0, the Bernoulli rate within 5 sigma,
                           unbiased scaling, slices drawn with an offset;
  * layer scale + DropPath -- the unmasked op (all-ones mask), dropped samples,
                           torch autograd.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from spatially_sharded_cnn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_facts.json")


def cfg_of(N, Ci, H, W, Co, k, s, p, g, S=1):
    return dict(N=N, C_in=Ci, H=H, W=W, C_out=Co, kh=k, kw=k, stride=s, padding=p, groups=g, num_shards=S)


def rand_case(cfg, seed, bias=True):
    x = synth.uniform((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), -1, 1, seed, 1)
    w = synth.normal((cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"]), 0.3, seed, 2)
    b = synth.normal((cfg["C_out"],), 0.1, seed, 3) if bias else None
    Ho = (cfg["H"] + 2 * cfg["padding"] - cfg["kh"]) // cfg["stride"] + 1
    Wo = (cfg["W"] + 2 * cfg["padding"] - cfg["kw"]) // cfg["stride"] + 1
    gy = synth.normal((cfg["N"], cfg["C_out"], Ho, Wo), 1.0, seed, 4)
    return x, w, b, gy


def _t(a):
    return torch.from_numpy(np.asarray(a, np.float64))


SMALL_CASES = [
    cfg_of(2, 3, 9, 8, 4, 3, 1, 1, 1),
    cfg_of(1, 4, 7, 10, 4, 5, 1, 2, 1),
    cfg_of(2, 4, 6, 9, 4, 7, 1, 3, 4),   # depthwise
    cfg_of(1, 6, 8, 8, 4, 3, 2, 1, 2),   # grouped, strided
    cfg_of(1, 3, 8, 12, 5, 4, 4, 0, 1),  # stem-like 4x4 / s4
    cfg_of(2, 4, 6, 8, 6, 2, 2, 0, 1),   # downsample-like 2x2 / s2
    cfg_of(1, 2, 5, 5, 3, 1, 1, 0, 1),   # 1x1
    cfg_of(1, 2, 5, 7, 2, 3, 2, 0, 1),   # ragged stride
]


def pin_out_size(orc):
    for n, k, s, p in itertools.product(range(1, 12), range(1, 8), range(1, 4), range(0, 4)):
        if n + 2 * p < k:
            continue
        ref = F.conv2d(torch.zeros(1, 1, n, n, dtype=torch.float64), torch.zeros(1, 1, k, k, dtype=torch.float64),
                       stride=s, padding=p).shape[-1]
        assert orc.out_size(n, k, s, p) == ref == (n + 2 * p - k) // s + 1, (n, k, s, p)


def pin_fwd_vs_torch(orc):
    for i, cfg in enumerate(SMALL_CASES):
        x, w, b, _ = rand_case(cfg, 10 + i)
        y = orc.conv2d_fwd(cfg, x, w, b)
        ref = F.conv2d(_t(x), _t(w), _t(b), stride=cfg["stride"], padding=cfg["padding"], groups=cfg["groups"])
        assert y.shape == tuple(ref.shape), (cfg, y.shape, ref.shape)
        assert np.abs(y - ref.numpy()).max() <= 1e-12 * max(1.0, np.abs(y).max()), cfg


def pin_fwd_vs_scipy(orc):
    from scipy.signal import correlate2d
    cfg = cfg_of(1, 3, 9, 11, 2, 5, 1, 2, 1)
    x, w, b, _ = rand_case(cfg, 3)
    y = orc.conv2d_fwd(cfg, x, w, b)
    for co in range(cfg["C_out"]):
        ref = np.full((9, 11), float(b[co]))
        for ci in range(cfg["C_in"]):
            xp = np.pad(x[0, ci].astype(np.float64), 2)
            ref += correlate2d(xp, w[co, ci].astype(np.float64), mode="valid")
        assert np.abs(y[0, co] - ref).max() <= 1e-12


def pin_fwd_1x1_is_matmul(orc):
    cfg = cfg_of(2, 5, 4, 6, 3, 1, 1, 0, 1)
    x, w, b, _ = rand_case(cfg, 4)
    y = orc.conv2d_fwd(cfg, x, w, b)
    W2 = w[:, :, 0, 0].astype(np.float64)
    for n in range(2):
        X2 = x[n].reshape(5, -1).astype(np.float64)
        ref = (W2 @ X2 + b[:, None]).reshape(3, 4, 6)
        assert np.abs(y[n] - ref).max() <= 1e-12


def pin_fwd_delta_kernel(orc):
    # One-hot weight at tap (u, v): the output is the input shifted by (u - p, v - p),
    # with zeros where the tap falls in the padding -- exactly.
    for k, p in ((5, 2), (7, 3), (3, 0)):
        cfg = cfg_of(1, 2, 6, 9, 2, k, 1, p, 2)
        x, _, _, _ = rand_case(cfg, 5)
        for u, v in itertools.product(range(k), range(k)):
            w = np.zeros((2, 1, k, k), np.float32)
            w[:, 0, u, v] = 1.0
            y = orc.conv2d_fwd(cfg, x, w)
            xp = np.pad(x.astype(np.float64), ((0, 0), (0, 0), (p, p), (p, p)))
            Ho, Wo = y.shape[2:]
            ref = xp[:, :, u:u + Ho, v:v + Wo]
            assert np.array_equal(y, ref), (k, p, u, v)


def pin_bwd_vs_autograd(orc):
    for i, cfg in enumerate(SMALL_CASES):
        x, w, b, gy = rand_case(cfg, 20 + i)
        xt, wt, bt = (_t(a).requires_grad_() for a in (x, w, b))
        yt = F.conv2d(xt, wt, bt, stride=cfg["stride"], padding=cfg["padding"], groups=cfg["groups"])
        yt.backward(_t(gy))
        gx = orc.conv2d_bwd_input(cfg, w, gy)
        gw = orc.conv2d_bwd_weight(cfg, x, gy)
        gb = orc.conv2d_bwd_bias(cfg, gy)
        for got, ref in ((gx, xt.grad), (gw, wt.grad), (gb, bt.grad)):
            ref = ref.numpy()
            assert got.shape == ref.shape
            assert np.abs(got - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max()), cfg


def pin_bwd_jacobian(orc):
    # Dense Jacobian J[:, k] = conv(e_k) (bias 0) enumerated column by column:
    # gx must equal J^T gy; gw likewise from the weight Jacobian.
    for cfg in (cfg_of(1, 2, 4, 5, 2, 3, 2, 1, 1), cfg_of(1, 2, 5, 4, 2, 3, 1, 1, 2)):
        x, w, _, gy = rand_case(cfg, 7, bias=False)
        nx = x.size
        J = np.zeros((gy.size, nx))
        for kk in range(nx):
            e = np.zeros(nx, np.float32)
            e[kk] = 1.0
            J[:, kk] = orc.conv2d_fwd(cfg, e.reshape(x.shape), w).ravel()
        gx = orc.conv2d_bwd_input(cfg, w, gy)
        assert np.abs(gx.ravel() - J.T @ gy.ravel().astype(np.float64)).max() <= 1e-12
        nw = w.size
        Jw = np.zeros((gy.size, nw))
        for kk in range(nw):
            e = np.zeros(nw, np.float32)
            e[kk] = 1.0
            Jw[:, kk] = orc.conv2d_fwd(cfg, x, e.reshape(w.shape)).ravel()
        gw = orc.conv2d_bwd_weight(cfg, x, gy)
        assert np.abs(gw.ravel() - Jw.T @ gy.ravel().astype(np.float64)).max() <= 1e-12


def pin_adjoint(orc):
    for i, cfg in enumerate(SMALL_CASES):
        x, w, b, gy = rand_case(cfg, 30 + i)
        y0 = orc.conv2d_fwd(cfg, x, w)          # no bias: y is linear in x and in w
        gx = orc.conv2d_bwd_input(cfg, w, gy)
        gw = orc.conv2d_bwd_weight(cfg, x, gy)
        lhs = float(np.sum(y0 * gy))
        scale = float(np.sum(np.abs(y0 * gy))) + 1.0
        assert abs(lhs - float(np.sum(x * gx))) <= 1e-12 * scale, cfg
        assert abs(lhs - float(np.sum(w * gw))) <= 1e-12 * scale, cfg
        gb = orc.conv2d_bwd_bias(cfg, gy)
        assert np.abs(gb - gy.astype(np.float64).sum(axis=(0, 2, 3))).max() <= 1e-12


def pin_point_evaluators(orc):
    rng = np.random.default_rng(0)
    for i, cfg in enumerate(SMALL_CASES):
        x, w, b, gy = rand_case(cfg, 40 + i)
        y = orc.conv2d_fwd(cfg, x, w, b)
        gx = orc.conv2d_bwd_input(cfg, w, gy)
        gw = orc.conv2d_bwd_weight(cfg, x, gy)
        gb = orc.conv2d_bwd_bias(cfg, gy)
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in y.shape)
            assert abs(orc.fwd_at(cfg, x, w, b, *idx) - y[idx]) <= 1e-12
            idx = tuple(int(rng.integers(0, s)) for s in gx.shape)
            assert abs(orc.gx_at(cfg, w, gy, *idx) - gx[idx]) <= 1e-12
            idx = tuple(int(rng.integers(0, s)) for s in gw.shape)
            assert abs(orc.gw_at(cfg, x, gy, *idx, 0, y.shape[3]) - gw[idx]) <= 1e-12
            co = int(rng.integers(0, cfg["C_out"]))
            assert abs(orc.gb_at(cfg, gy, co, 0, y.shape[3]) - gb[co]) <= 1e-12


def pin_shard_plan_pages(orc):
    facts = json.load(open(GOLDEN))
    f = facts["shard3_split"]
    N, Cc, H, W = f["global_shape"]
    cfg = cfg_of(N, Cc, H, W, Cc, 1, 1, 0, 1, f["num_shards"])
    rc, plan, Ho, Wo = orc.shard_plan(cfg)
    assert rc == 0
    for r, e in enumerate(plan):
        assert [N, Cc, H, e[1] - e[0]] == f["local_shape"]
        assert e[0] == r * f["local_shape"][3]
    h = facts["halo_5x5"]
    cfg = cfg_of(1, 1, 16, 32, 1, h["kernel"], h["stride"], h["padding"], 1, 4)
    rc, plan, Ho, Wo = orc.shard_plan(cfg)
    assert rc == 0 and (Ho, Wo) == (16, 32)
    for e in plan:
        assert e[2] == e[3] == h["halo_columns_each_side"]
        assert e[5] - e[4] == 8                      # each shard keeps its own 8 output columns
    # Crop of [KW] 3.2: the local conv (padding p on the (Wl + 2p)-wide tile) has
    # Wl + 2p output columns; the crop removes p on each side.
    c = facts["crop"]
    Wl = 8
    local_out = (Wl + 2 * c["padding"] + 2 * c["padding"] - 5) // 1 + 1
    assert local_out - Wl == 2 * c["local_output_columns_dropped_each_side"]


def pin_shard_plan_cover(orc):
    # Owned output columns partition [0, Wout); halos are exactly the columns read
    # outside the shard; unsupported layouts are refused.
    for W, S, k, s, p in itertools.product((8, 12, 16, 24), (1, 2, 4), (1, 2, 3, 4, 5, 7), (1, 2, 4), (0, 1, 2, 3)):
        cfg = cfg_of(1, 1, 8, W, 1, k, s, p, 1, S)
        rc, plan, Ho, Wo = orc.shard_plan(cfg)
        Wl = W // S
        if W % S or Wl % s or p % s:
            assert rc != 0, (W, S, k, s, p)
            continue
        if rc:
            # refused only because some halo would be wider than a neighbouring shard
            Wout = (W + 2 * p - k) // s + 1
            widest = 0
            for r in range(S):
                o0, o1 = r * Wl // s, (Wout if r == S - 1 else min((r + 1) * Wl // s, Wout))
                if o1 > o0:
                    widest = max(widest, r * Wl - (o0 * s - p), (o1 - 1) * s - p + k - (r + 1) * Wl)
            assert widest > Wl, (W, S, k, s, p)
            continue
        owned = [j for e in plan for j in range(e[4], e[5])]
        assert owned == list(range(Wo)), (W, S, k, s, p)
        for e in plan:
            if e[5] == e[4]:
                continue
            cols = [j * s - p + v for j in range(e[4], e[5]) for v in range(k)]
            assert e[0] - e[2] == min(min(cols), e[0])
            assert e[1] + e[3] == max(max(cols) + 1, e[1])


def pin_halo_extend(orc):
    for cfg in (cfg_of(2, 3, 4, 16, 3, 5, 1, 2, 1, 4), cfg_of(1, 2, 3, 24, 2, 7, 1, 3, 2, 4),
                cfg_of(1, 2, 3, 16, 2, 2, 2, 0, 1, 2), dict(cfg_of(1, 2, 8, 16, 2, 3, 1, 1, 1, 2), num_shards_h=2),
                dict(cfg_of(2, 1, 12, 8, 1, 5, 1, 2, 1, 1), num_shards_h=3)):
        x, _, _, _ = rand_case(cfg, 8)
        rc, plan, _, _ = orc.shard_plan(cfg)
        rc2, plan_h = orc.shard_plan_h(cfg)
        assert rc == 0 and rc2 == 0
        P = 8
        xp = np.pad(x, ((0, 0), (0, 0), (P, P), (P, P)))   # zeros past every image edge
        for q in range(len(plan_h) * len(plan)):
            e, f = plan[q % len(plan)], plan_h[q // len(plan)]
            xe = orc.halo_extend(cfg, q, x)
            ref = xp[:, :, P + f[0] - f[2]: P + f[1] + f[3], P + e[0] - e[2]: P + e[1] + e[3]]
            assert np.array_equal(xe, ref), (cfg, q)


def pin_shard_plan_rows(orc):
    # The row plan follows the column rule on H: owned output rows partition
    # [0, Hout); halos are exactly the rows read outside the shard.
    for H, Sh, k, s, p in itertools.product((8, 12, 16), (1, 2, 4), (1, 2, 3, 5), (1, 2), (0, 1, 2)):
        cfg = dict(cfg_of(1, 1, H, 8, 1, k, s, p, 1, 1), num_shards_h=Sh)
        rc, plan = orc.shard_plan_h(cfg)
        Hl = H // Sh
        Ho = (H + 2 * p - k) // s + 1
        if Sh == 1:   # no row neighbours: every row, no halo rows (padding supplies the edges)
            assert rc == 0 and plan == [(0, H, 0, 0, 0, Ho)], (H, k, s, p)
            continue
        if H % Sh or Hl % s or p % s:
            assert rc != 0, (H, Sh, k, s, p)
            continue
        if rc:
            continue    # a halo wider than a neighbouring shard
        assert [i for f in plan for i in range(f[4], f[5])] == list(range(Ho)), (H, Sh, k, s, p)
        for f in plan:
            if f[5] > f[4]:
                rows = [i * s - p + u for i in range(f[4], f[5]) for u in range(k)]
                assert f[0] - f[2] == min(min(rows), f[0]) and f[1] + f[3] == max(max(rows) + 1, f[1])


SHARD_CASES = [
    cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1),      # the small dense case, any S
    cfg_of(2, 3, 6, 24, 3, 7, 1, 3, 3),       # depthwise 7x7
    cfg_of(1, 2, 6, 16, 4, 2, 2, 0, 1),       # 2x2 / s2 downsample
    cfg_of(1, 3, 8, 32, 4, 4, 4, 0, 1),       # 4x4 / s4 stem
    cfg_of(1, 2, 5, 12, 3, 1, 1, 0, 1),       # 1x1
    cfg_of(1, 2, 6, 16, 2, 3, 2, 2, 1),       # 3x3 / s2 / p2 (stride divides padding)
]


def pin_sharded_equals_unsharded(orc):
    for i, base in enumerate(SHARD_CASES):
        x, w, b, gy = rand_case(base, 50 + i)
        y = orc.conv2d_fwd(base, x, w, b)
        gx = orc.conv2d_bwd_input(base, w, gy)
        gw = orc.conv2d_bwd_weight(base, x, gy)
        gb = orc.conv2d_bwd_bias(base, gy)
        tried = tried_h = 0
        for S, Sh in itertools.product(range(1, base["W"] + 1), (1, 2, 3)):
            cfg = dict(base, num_shards=S, num_shards_h=Sh)
            rc, plan, _, _ = orc.shard_plan(cfg)
            rc2, plan_h = orc.shard_plan_h(cfg)
            if rc or rc2:
                continue
            tried += 1
            tried_h += Sh > 1
            ys = orc.sharded_fwd(cfg, x, w, b)
            assert np.abs(ys - y).max() <= 1e-12, (base, S, Sh)
            gxs, gwp, gbp = orc.sharded_bwd(cfg, x, w, gy)
            assert np.abs(gxs - gx).max() <= 1e-12, (base, S, Sh)
            assert np.abs(gwp.sum(0) - gw).max() <= 1e-12 * max(1, np.abs(gw).max()), (base, S, Sh)
            assert np.abs(gbp.sum(0) - gb).max() <= 1e-12 * max(1, np.abs(gb).max()), (base, S, Sh)
            # each partial is the gradient restricted to the shard's own output rows and columns
            for q in range(len(plan_h) * len(plan)):
                e, f = plan[q % len(plan)], plan_h[q // len(plan)]
                co, cl, u, v = 0, 0, base["kh"] - 1, 0
                ref = orc.gw_at(base, x, gy, co, cl, u, v, e[4], e[5], f[4], f[5])
                assert abs(gwp[q, co, cl, u, v] - ref) <= 1e-12, (base, S, Sh, q)
                if Sh == 1:  # the bias evaluator restricts columns only: each column shard's own partial
                    for co in range(base["C_out"]):
                        assert abs(gbp[q, co] - orc.gb_at(base, gy, co, e[4], e[5])) <= 1e-12, (base, S, q, co)
        assert tried >= 2 and (tried_h >= 1 or (base["H"] % 2 and base["H"] % 3)), base


def pin_layernorm(orc):
    x = synth.normal((2, 16, 3, 5), 2.0, 1, 1).astype(np.float64) + 0.5
    gamma = 1.0 + synth.normal((16,), 0.2, 1, 2).astype(np.float64)
    beta = synth.normal((16,), 0.2, 1, 3).astype(np.float64)
    gy = synth.normal(x.shape, 1.0, 1, 4).astype(np.float64)
    eps = 1e-6
    y, mean, rstd = orc.layernorm_c_fwd(x, gamma, beta, eps)
    # closed form with gamma = 1, beta = 0: mean 0, variance var/(var+eps) per position
    y1, _, _ = orc.layernorm_c_fwd(x, np.ones(16), np.zeros(16), eps)
    var = x.var(axis=1)
    assert np.abs(y1.mean(axis=1)).max() <= 1e-12
    assert np.abs(y1.var(axis=1) - var / (var + eps)).max() <= 1e-12
    xt = _t(x).requires_grad_()
    gt, bt = _t(gamma).requires_grad_(), _t(beta).requires_grad_()
    yt = F.layer_norm(xt.permute(0, 2, 3, 1), (16,), gt, bt, eps).permute(0, 3, 1, 2)
    assert np.abs(y - yt.detach().numpy()).max() <= 1e-12
    yt.backward(_t(gy))
    gx, gg, gb = orc.layernorm_c_bwd(x, gamma, gy, eps)
    assert np.abs(gx - xt.grad.numpy()).max() <= 1e-11
    assert np.abs(gg - gt.grad.numpy()).max() <= 1e-11
    assert np.abs(gb - bt.grad.numpy()).max() <= 1e-11
    assert np.abs(gx.sum(axis=1)).max() <= 1e-11   # LN grad_input sums to 0 over C when beta-shift invariant
    # central differences on a few entries
    h = 1e-5
    for idx in ((0, 0, 0, 0), (1, 7, 2, 4), (0, 15, 1, 3)):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = (np.sum(orc.layernorm_c_fwd(xp, gamma, beta, eps)[0] * gy) -
              np.sum(orc.layernorm_c_fwd(xm, gamma, beta, eps)[0] * gy)) / (2 * h)
        assert abs(fd - gx[idx]) <= 1e-6 * max(1, abs(gx[idx]))


def pin_gelu(orc):
    x = np.concatenate([np.linspace(-6, 6, 241), synth.normal((500,), 2.0, 2, 1).astype(np.float64)])
    y = orc.gelu_fwd(x)
    ref = np.array([v * 0.5 * (1 + math.erf(v / math.sqrt(2))) for v in x])
    assert np.abs(y - ref).max() <= 1e-15 * 8
    assert np.abs(y - F.gelu(_t(x)).numpy()).max() <= 1e-14
    assert orc.gelu_fwd(np.array([0.0]))[0] == 0.0
    assert abs(orc.gelu_fwd(np.array([1.0]))[0] - 0.8413447460685429) <= 1e-15   # Phi(1)
    assert abs(orc.gelu_bwd(np.array([0.0]), np.array([1.0]))[0] - 0.5) <= 1e-15
    gy = synth.normal(x.shape, 1.0, 2, 2).astype(np.float64)
    xt = _t(x).requires_grad_()
    F.gelu(xt).backward(_t(gy))
    assert np.abs(orc.gelu_bwd(x, gy) - xt.grad.numpy()).max() <= 1e-13
    h = 1e-6
    fd = (orc.gelu_fwd(x + h) - orc.gelu_fwd(x - h)) / (2 * h)
    assert np.abs(orc.gelu_bwd(x, np.ones_like(x)) - fd).max() <= 1e-7


def pin_layerscale(orc):
    res = synth.normal((2, 6, 3, 4), 1.0, 3, 1).astype(np.float64)
    br = synth.normal(res.shape, 1.0, 3, 2).astype(np.float64)
    gamma = synth.normal((6,), 1e-2, 3, 3).astype(np.float64)
    gy = synth.normal(res.shape, 1.0, 3, 4).astype(np.float64)
    out = orc.layerscale_residual_fwd(res, br, gamma)
    assert np.abs(out - (res + gamma[None, :, None, None] * br)).max() <= 1e-15
    rt, bt, gt = (_t(a).requires_grad_() for a in (res, br, gamma))
    (rt + gt[None, :, None, None] * bt).backward(_t(gy))
    gres, gbr, gg = orc.layerscale_residual_bwd(br, gamma, gy)
    assert np.array_equal(gres, gy)
    assert np.abs(gbr - bt.grad.numpy()).max() <= 1e-15
    assert np.abs(gg - gt.grad.numpy()).max() <= 1e-13


def pin_splitmix64_published(orc):
    g = json.load(open(os.path.join(os.path.dirname(GOLDEN), "splitmix64.json")))
    for i, hx in enumerate(g["outputs_hex"]):
        assert orc.splitmix64(g["seed"], i) == int(hx, 16), (i, hex(orc.splitmix64(g["seed"], i)))


def pin_drop_path_mask(orc):
    # the keep decision on the published first output of seed 0: top 24 bits 0xe220a8
    u0 = int(json.load(open(os.path.join(os.path.dirname(GOLDEN), "splitmix64.json")))["outputs_hex"][0], 16) >> 40
    p_keep = math.floor(u0 / 2 ** 24 * 100) / 100          # largest p (2 decimals) that still keeps sample 0
    assert orc.drop_path_mask(1, p_keep, 0, 0)[0] == np.float32(1.0) / (np.float32(1.0) - np.float32(p_keep))
    assert orc.drop_path_mask(1, p_keep + 0.01, 0, 0)[0] == 0.0
    assert np.all(orc.drop_path_mask(1000, 0.0, 7, 3) == 1.0)          # p = 0 keeps every sample, scale 1
    p = 0.3
    m = orc.drop_path_mask(400_000, p, 12345, 0)
    scale = np.float32(1.0) / (np.float32(1.0) - np.float32(p))
    assert set(np.unique(m).tolist()) <= {0.0, float(scale)}
    kept = float(np.mean(m > 0))
    sd = math.sqrt(p * (1 - p) / m.size)
    assert abs(kept - (1 - p)) <= 5 * sd, kept                        # Bernoulli(1 - p) within 5 sigma
    assert abs(float(np.mean(m, dtype=np.float64)) - 1.0) <= 5 * sd / (1 - p) + 1e-6   # unbiased scaling
    # shard consistency: a slice of the batch drawn with offset = its first sample matches
    for k, n in ((0, 10), (17, 100), (399_000, 1000)):
        assert np.array_equal(orc.drop_path_mask(n, p, 12345, k), m[k:k + n]), k
    assert not np.array_equal(orc.drop_path_mask(1000, p, 12346, 0), m[:1000])


def pin_layerscale_droppath(orc):
    res = synth.normal((4, 6, 3, 4), 1.0, 5, 1).astype(np.float64)
    br = synth.normal(res.shape, 1.0, 5, 2).astype(np.float64)
    gamma = synth.normal((6,), 1e-2, 5, 3).astype(np.float64)
    gy = synth.normal(res.shape, 1.0, 5, 4).astype(np.float64)
    ones = np.ones(4)
    assert np.array_equal(orc.layerscale_droppath_fwd(res, br, gamma, ones), orc.layerscale_residual_fwd(res, br, gamma))
    for a, b in zip(orc.layerscale_droppath_bwd(br, gamma, ones, gy), orc.layerscale_residual_bwd(br, gamma, gy)):
        assert np.array_equal(a, b)
    mask = np.array([0.0, 1.25, 0.0, 1.25])
    out = orc.layerscale_droppath_fwd(res, br, gamma, mask)
    assert np.array_equal(out[0], res[0]) and np.array_equal(out[2], res[2])   # a dropped sample passes res through
    rt, bt, gt = (_t(a).requires_grad_() for a in (res, br, gamma))
    (rt + _t(mask)[:, None, None, None] * gt[None, :, None, None] * bt).backward(_t(gy))
    gres, gbr, gg = orc.layerscale_droppath_bwd(br, gamma, mask, gy)
    assert np.array_equal(gres, gy)
    assert np.abs(gbr - bt.grad.numpy()).max() <= 1e-15
    assert np.all(gbr[0] == 0) and np.all(gbr[2] == 0)
    assert np.abs(gg - gt.grad.numpy()).max() <= 1e-13


ALL_PINS = [
    pin_out_size, pin_fwd_vs_torch, pin_fwd_vs_scipy, pin_fwd_1x1_is_matmul, pin_fwd_delta_kernel,
    pin_bwd_vs_autograd, pin_bwd_jacobian, pin_adjoint, pin_point_evaluators, pin_shard_plan_pages,
    pin_shard_plan_cover, pin_shard_plan_rows, pin_halo_extend, pin_sharded_equals_unsharded, pin_layernorm, pin_gelu, pin_layerscale,
    pin_splitmix64_published, pin_drop_path_mask, pin_layerscale_droppath,
]
