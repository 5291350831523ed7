"""The patchify stem's weight / bias gradient (4x4 kernel, stride 4, 3 input
channels) on the direct FP32 reduction, against the oracle.

The library takes that kernel when hc_conv2d_bwd is asked for weight and bias
gradients only (no grad_input: the image needs none) with the algorithm left
to it; grad_output is then read once instead of split into bf16 pieces.
Checked: the gradients and their per-shard partials within the weight
tolerance on column, row x column and two-channel-block grids, including CTAs
that get no job; bit-exact on dyadic inputs (every product and sum exact in
fp32); bit-identical repeats; the full image width of the ConvNeXt stem (two
images) on sampled channels; and that the trace names the kernel.
"""
import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P
from spatially_sharded_cnn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_W = 1e-4


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def stem_cfg(N, H, W, Co, S, Sh=1):
    cfg = P.cfg_of(N, 3, H, W, Co, 4, 4, 0, 1, S)
    if Sh > 1:
        cfg["num_shards_h"] = Sh
    return cfg


def stem_inputs(cfg, seed):
    x = synth.uniform((cfg["N"], 3, cfg["H"], cfg["W"]), 0.0, 1.0, seed, 1)
    gy = synth.normal((cfg["N"], cfg["C_out"], cfg["H"] // 4, cfg["W"] // 4), 1.0, seed, 4)
    w = synth.trunc_normal((cfg["C_out"], 3, 4, 4), 0.02, seed, 2)
    return x, w, gy


def traced_names(hc, fn):
    hc.hc_trace_collect()
    hc.hc_trace_enable(True)
    try:
        fn()
    finally:
        hc.hc_trace_enable(False)
    st, tab = hc.hc_trace_collect()
    hc.check(st, "trace collect")
    return set(tab)


CASES = {
    # 4 column shards of 128 output columns; 2 images
    "S4": stem_cfg(2, 16, 2048, 256, 4),
    # a 2 x 2 grid: row shards of 2 output rows
    "grid_2x2": stem_cfg(1, 16, 1024, 256, 2, 2),
    # two 256-channel blocks
    "Co512_S2": stem_cfg(1, 8, 512, 512, 2),
    # 2 jobs per group and far more CTAs: most slots are zero
    "few_jobs": stem_cfg(1, 8, 256, 256, 2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_patchify_wgrad_matches_oracle(hc, orc, name):
    cfg = CASES[name]
    x, w, gy = stem_inputs(cfg, 11)
    names = traced_names(hc, lambda: R.bwd_subset(cfg, x, w, gy, ("gw", "gb", "gw_partials", "gb_partials")))
    assert "patchify_wgrad_kernel" in names and "dw_shard_partials_kernel" in names, names
    assert not any(n.startswith("tc_conv_kernel") or n.startswith("bias_rows") for n in names), names
    out = R.bwd_subset(cfg, x, w, gy, ("gw", "gb", "gw_partials", "gb_partials"))
    _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, x, w, gy)
    assert R.normwise(out["gw"], orc.conv2d_bwd_weight(cfg, x, gy)) <= TOL_W
    assert R.normwise(out["gb"], orc.conv2d_bwd_bias(cfg, gy)) <= TOL_W
    for q in range(gwp_ref.shape[0]):
        assert R.normwise(out["gw_partials"][q], gwp_ref[q]) <= TOL_W, q
        assert R.normwise(out["gb_partials"][q], gbp_ref[q]) <= TOL_W, q
    # the shard partials add up to the full gradients in shard order
    acc_w = out["gw_partials"][0].copy()
    acc_b = out["gb_partials"][0].copy()
    for q in range(1, gwp_ref.shape[0]):
        acc_w = (acc_w + out["gw_partials"][q]).astype(np.float32)
        acc_b = (acc_b + out["gb_partials"][q]).astype(np.float32)
    assert np.array_equal(acc_w, out["gw"]) and np.array_equal(acc_b, out["gb"])


@pytest.mark.parametrize("name", ["S4", "grid_2x2"])
def test_patchify_wgrad_dyadic_exact(hc, orc, name):
    """Multiples of 1/4 in [-4, 4]: every product and partial sum is exact in fp32,
    so gradients and partials equal the oracle bit for bit, whatever the order."""
    cfg = CASES[name]
    x = synth.dyadic((cfg["N"], 3, cfg["H"], cfg["W"]), 2, 4, 5, 1)
    gy = synth.dyadic((cfg["N"], cfg["C_out"], cfg["H"] // 4, cfg["W"] // 4), 2, 4, 5, 4)
    w = synth.dyadic((cfg["C_out"], 3, 4, 4), 2, 4, 5, 2)
    out = R.bwd_subset(cfg, x, w, gy, ("gw", "gb", "gw_partials", "gb_partials"))
    _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, x, w, gy)
    assert np.array_equal(out["gw"], orc.conv2d_bwd_weight(cfg, x, gy).astype(np.float32))
    assert np.array_equal(out["gb"], orc.conv2d_bwd_bias(cfg, gy).astype(np.float32))
    assert np.array_equal(out["gw_partials"], gwp_ref.astype(np.float32))
    assert np.array_equal(out["gb_partials"], gbp_ref.astype(np.float32))


def test_patchify_wgrad_repeat_bit_identical(hc):
    cfg = CASES["S4"]
    x, w, gy = stem_inputs(cfg, 12)
    a = R.bwd_subset(cfg, x, w, gy, ("gw", "gb", "gw_partials"))
    b = R.bwd_subset(cfg, x, w, gy, ("gw", "gb", "gw_partials"))
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_patchify_wgrad_bias_only_and_weights_only(hc, orc):
    cfg = CASES["S4"]
    x, w, gy = stem_inputs(cfg, 13)
    ob = R.bwd_subset(cfg, x, w, gy, ("gb",))
    assert R.normwise(ob["gb"], orc.conv2d_bwd_bias(cfg, gy)) <= TOL_W
    ow = R.bwd_subset(cfg, x, w, gy, ("gw",))
    assert R.normwise(ow["gw"], orc.conv2d_bwd_weight(cfg, x, gy)) <= TOL_W


def test_patchify_wgrad_stem_width_sampled(hc, orc):
    """The ConvNeXt stem's full image (512 x 4096, 8 shards) for two images:
    every shard's partial of sampled output channels against the oracle's
    per-element sums over that shard's own output columns."""
    cfg = stem_cfg(2, 512, 4096, 256, 8)
    x, w, gy = stem_inputs(cfg, 14)
    out = R.bwd_subset(cfg, x, w, gy, ("gw", "gb", "gw_partials", "gb_partials"))
    Wlo = cfg["W"] // 4 // cfg["num_shards"]
    rng = np.random.default_rng(3)
    for co in rng.choice(256, 3, replace=False).tolist():
        for q in (0, 3, 7):
            j0, j1 = q * Wlo, (q + 1) * Wlo
            ref = np.array([[[orc.gw_at(cfg, x, gy, co, ci, u, v, j0, j1) for v in range(4)] for u in range(4)]
                            for ci in range(3)])
            assert R.normwise(out["gw_partials"][q][co], ref) <= TOL_W, (co, q)
            gb = orc.gb_at(cfg, gy, co, j0, j1)
            assert abs(out["gb_partials"][q][co] - gb) <= TOL_W * max(abs(gb), 1.0), (co, q)
