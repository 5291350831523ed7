"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances (normwise max relative error, max|gpu - oracle| / max|oracle| per
output tensor): forward and grad_input 1e-5, grad_weight / grad_bias and their
per-shard partials 1e-4.  Halo gathers and one-hot (delta) kernels on dyadic
inputs must match bit for bit; two runs of the same call must be identical.
"""
import numpy as np
import pytest
import torch

import hc_run as R
import oracle_pins as P
from spatially_sharded_cnn_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-5
TOL_W = 1e-4


@pytest.fixture(scope="module")
def hc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def config1():
    """Dense 5x5 / s1 / p2, (1,4,16,32), 4 shards of width 8; seed 0."""
    cfg = P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4)
    x = synth.uniform((1, 4, 16, 32), -1, 1, 0, 1)
    w = synth.normal((4, 4, 5, 5), 0.1, 0, 2)
    b = synth.normal((4,), 0.1, 0, 3)
    gy = synth.normal((1, 4, 16, 32), 1.0, 0, 4)
    return cfg, x, w, b, gy


def dw_case(N, C, H, W, K, S, seed=1):
    cfg = P.cfg_of(N, C, H, W, C, K, 1, (K - 1) // 2, C, S)
    x = synth.normal((N, C, H, W), 1.0, seed, 1)
    w = synth.trunc_normal((C, 1, K, K), 0.02, seed, 2)
    b = synth.normal((C,), 0.1, seed, 3)
    gy = synth.normal((N, C, H, W), 1.0, seed, 4)
    return cfg, x, w, b, gy


def tc_case(N, Ci, H, W, Co, K, S, seed=3):
    cfg = P.cfg_of(N, Ci, H, W, Co, K, 1, (K - 1) // 2, 1, S)
    x = synth.normal((N, Ci, H, W), 1.0, seed, 1)
    w = synth.normal((Co, Ci, K, K), (2.0 / (Ci * K * K)) ** 0.5, seed, 2)
    b = synth.normal((Co,), 0.01, seed, 3)
    gy = synth.normal((N, Co, H, W), 1.0, seed, 4)
    return cfg, x, w, b, gy


def tc_strided_case(N, Ci, H, W, Co, s, S, seed=4):
    cfg = P.cfg_of(N, Ci, H, W, Co, s, s, 0, 1, S)
    x = synth.uniform((N, Ci, H, W), 0.0, 1.0, seed, 1)
    w = synth.trunc_normal((Co, Ci, s, s), 0.02, seed, 2)
    b = synth.normal((Co,), 0.01, seed, 3)
    gy = synth.normal((N, Co, H // s, W // s), 1.0, seed, 4)
    return cfg, x, w, b, gy


def generic_case(cfg, seed=2):
    x, w, b, gy = P.rand_case(cfg, seed)
    return cfg, x, w, b, gy


CASES = {
    "config1_dense5x5": config1,
    "dw7_ragged_S4": lambda: dw_case(2, 3, 70, 512, 7, 4),
    "dw7_S2_two_tiles_per_shard": lambda: dw_case(1, 2, 40, 512, 7, 2),
    "dw7_S1": lambda: dw_case(1, 2, 33, 256, 7, 1),
    "dw5_S2": lambda: dw_case(2, 2, 45, 256, 5, 2),
    "dw3_S4": lambda: dw_case(1, 3, 31, 512, 3, 4),
    "dw7_H1": lambda: dw_case(1, 2, 1, 256, 7, 2),
    "dw7_narrow_shards_direct": lambda: dw_case(1, 4, 20, 64, 7, 4),
    "grouped_strided": lambda: generic_case(P.cfg_of(2, 6, 12, 16, 4, 3, 2, 2, 2, 2)),
    "stem4x4s4": lambda: generic_case(P.cfg_of(1, 3, 16, 64, 8, 4, 4, 0, 1, 4)),
    "down2x2s2_S8": lambda: generic_case(P.cfg_of(1, 4, 8, 32, 6, 2, 2, 0, 1, 8)),
    "pointwise1x1": lambda: generic_case(P.cfg_of(2, 5, 6, 16, 7, 1, 1, 0, 1, 2)),
    # tensor-core (3xTF32) path: C_in, C_out multiples of 128
    "tc_5x5_S2": lambda: tc_case(1, 128, 6, 256, 128, 5, 2),
    "tc_3x3_two_mblocks": lambda: tc_case(1, 128, 5, 256, 256, 3, 1),
    "tc_1x1": lambda: tc_case(2, 256, 4, 128, 128, 1, 1),
    # 1x1 convs on three bf16 pieces: half slot pair (C_in 128), 128-pixel tiles
    # (H*W = 384) with a half pair (C_in 384), the block's 256->1024 and 1024->256
    # shapes at 8 shards, a 2 x 4 grid
    "pw_128to256_S4_half_pair": lambda: tc_case(2, 128, 4, 256, 256, 1, 4),
    "pw_384to128_tiles128": lambda: tc_case(1, 384, 3, 128, 128, 1, 2),
    "pw_256to1024_S8": lambda: tc_case(1, 256, 2, 1024, 1024, 1, 8),
    "pw_1024to256_S8": lambda: tc_case(1, 1024, 2, 1024, 256, 1, 8),
    "tc_5x5_ragged_two_tiles": lambda: tc_case(1, 128, 7, 512, 128, 5, 1),
    # weight-gradient slot pairs: 7 kernel rows (a single in every column), and
    # C_in = 256 (channel-block pairs of one tap)
    "tc_7x7_S2": lambda: tc_case(1, 128, 9, 256, 128, 7, 2),
    "tc_3x3_Cin256_S2": lambda: tc_case(1, 256, 6, 256, 128, 3, 2),
    "tc_1x1_Cin384_S2": lambda: tc_case(1, 384, 3, 256, 128, 1, 2),  # 3 channel blocks: a pair and a single
    # strided k = stride convs through space-to-depth (stem- and downsample-like)
    "tc_stem4x4s4": lambda: tc_strided_case(2, 3, 12, 512, 128, 4, 1),
    "tc_down2x2s2_S2": lambda: tc_strided_case(1, 128, 6, 512, 256, 2, 2),
    # s = 3 with a zero channel tail (Kp 640 > 576) and the scalar depth-to-space store
    "tc_down3x3s3_C64_S2": lambda: tc_strided_case(1, 64, 6, 768, 128, 3, 2),
    # C % 64 != 0: the generic space-to-depth prep; 256-wide tiles over 128-wide shards
    "tc_down2x2s2_C96_S4": lambda: tc_strided_case(1, 96, 4, 1024, 128, 2, 4),
    # 256-wide conv tiles across 128-wide shards, the halo read inside a tile
    "tc_5x5_S4_tiles_cross_shards": lambda: tc_case(1, 128, 5, 512, 128, 5, 4),
    # 2048 columns: the bias partials walk two 1024-column groups, 8 shards
    "tc_3x3_wide_S8": lambda: tc_case(1, 128, 2, 2048, 128, 3, 8),
    # row x column shard grids (Shard(2) and Shard(3) together)
    "tc_5x5_grid_2x2": lambda: _rows(tc_case(1, 128, 8, 256, 128, 5, 2), 2),
    "tc_down2x2s2_grid_2x2": lambda: _rows(tc_strided_case(1, 128, 8, 512, 256, 2, 2), 2),
    "pw_grid_2x4": lambda: _rows(tc_case(1, 256, 8, 256, 128, 1, 4), 2),
    "dw7_grid_2x2": lambda: _rows(dw_case(1, 2, 128, 256, 7, 2), 2),          # 64-row shards: depthwise
    "dw7_grid_4x2": lambda: _rows(dw_case(1, 2, 128, 256, 7, 2), 4),          # 32-row shards: depthwise
    "dw7_grid_8x2_direct": lambda: _rows(dw_case(1, 2, 128, 256, 7, 2), 8),   # 16-row shards: direct
    "grouped_strided_grid_3x2": lambda: _rows(generic_case(P.cfg_of(2, 6, 12, 16, 4, 3, 2, 2, 2, 2)), 3),
}


def _rows(case, Sh):
    cfg, *rest = case
    return (dict(cfg, num_shards_h=Sh), *rest)


def check_case(hc, orc, cfg, x, w, b, gy, algo=None):
    y = R.fwd(cfg, x, w, b, algo)
    ref = orc.conv2d_fwd(cfg, x, w, b)
    assert R.normwise(y, ref) <= TOL_FWD, R.normwise(y, ref)
    out = R.bwd(cfg, x, w, gy, algo)
    gx_ref = orc.conv2d_bwd_input(cfg, w, gy)
    gw_ref = orc.conv2d_bwd_weight(cfg, x, gy)
    gb_ref = orc.conv2d_bwd_bias(cfg, gy)
    assert R.normwise(out["gx"], gx_ref) <= TOL_FWD, R.normwise(out["gx"], gx_ref)
    assert R.normwise(out["gw"], gw_ref) <= TOL_W, R.normwise(out["gw"], gw_ref)
    assert R.normwise(out["gb"], gb_ref) <= TOL_W, R.normwise(out["gb"], gb_ref)
    # per-shard _Partial values against the oracle's sharded backward
    _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, x, w, gy)
    assert R.normwise(out["gw_partials"], gwp_ref) <= TOL_W
    assert R.normwise(out["gb_partials"], gbp_ref) <= TOL_W
    return y, out


@pytest.mark.parametrize("name", list(CASES))
def test_parity_auto(hc, orc, name):
    check_case(hc, orc, *CASES[name]())


@pytest.mark.parametrize("name", ["config1_dense5x5", "dw7_ragged_S4", "stem4x4s4"])
def test_parity_direct(hc, orc, name):
    check_case(hc, orc, *CASES[name](), algo=hc.HC_ALGO_DIRECT)


def test_grid_family_choice(hc):
    """Row shards keep the depthwise kernels when each row shard is whole 32-row
    tiles of the backward, and fall back to the direct kernels otherwise."""
    sel = lambda n: hc.hc_conv2d_select(hc.desc(CASES[n]()[0]), 1)
    assert sel("dw7_grid_2x2") == (0, hc.HC_ALGO_DEPTHWISE)
    assert sel("dw7_grid_4x2") == (0, hc.HC_ALGO_DEPTHWISE)
    assert sel("dw7_grid_8x2_direct") == (0, hc.HC_ALGO_DIRECT)
    assert sel("tc_5x5_grid_2x2") == (0, hc.HC_ALGO_TC_3XTF32)
    assert sel("tc_down2x2s2_grid_2x2") == (0, hc.HC_ALGO_TC_BF16X6)
    assert sel("pw_grid_2x4") == (0, hc.HC_ALGO_TC_BF16X6)


@pytest.mark.parametrize("name", ["dw7_ragged_S4", "dw5_S2", "dw3_S4"])
def test_parity_depthwise_explicit(hc, orc, name):
    cfg = CASES[name]()[0]
    st, algo = hc.hc_conv2d_select(hc.desc(cfg), 1)
    assert st == 0 and algo == hc.HC_ALGO_DEPTHWISE
    check_case(hc, orc, *CASES[name](), algo=hc.HC_ALGO_DEPTHWISE)


@pytest.mark.parametrize("name", ["tc_5x5_S2", "tc_3x3_two_mblocks", "tc_1x1", "tc_5x5_ragged_two_tiles",
                                  "tc_stem4x4s4", "tc_down2x2s2_S2", "tc_down3x3s3_C64_S2", "tc_down2x2s2_C96_S4",
                                  "tc_5x5_S4_tiles_cross_shards", "tc_3x3_wide_S8", "tc_7x7_S2", "tc_3x3_Cin256_S2",
                                  "tc_1x1_Cin384_S2"])
def test_parity_tensor_cores_explicit(hc, orc, name):
    cfg = CASES[name]()[0]
    auto = hc.HC_ALGO_TC_BF16X6 if name in BF16_CASES else hc.HC_ALGO_TC_3XTF32
    assert hc.hc_conv2d_select(hc.desc(cfg), 0) == (0, auto)
    check_case(hc, orc, *CASES[name](), algo=hc.HC_ALGO_TC_3XTF32)


# 1x1 convs and k = stride convs (space-to-depth) with 128-multiple output
# channels take the bf16-piece GEMM
BF16_CASES = ["tc_1x1", "pw_128to256_S4_half_pair", "pw_384to128_tiles128", "pw_256to1024_S8", "pw_1024to256_S8",
              "pw_grid_2x4", "tc_stem4x4s4", "tc_down2x2s2_S2", "tc_down3x3s3_C64_S2", "tc_down2x2s2_C96_S4",
              "tc_down2x2s2_grid_2x2", "tc_1x1_Cin384_S2"]


@pytest.mark.parametrize("name", BF16_CASES)
def test_parity_bf16x6_explicit(hc, orc, name):
    cfg = CASES[name]()[0]
    assert hc.hc_conv2d_select(hc.desc(cfg), 0) == (0, hc.HC_ALGO_TC_BF16X6)
    assert hc.hc_conv2d_select(hc.desc(cfg), 1) == (0, hc.HC_ALGO_TC_BF16X6)
    check_case(hc, orc, *CASES[name](), algo=hc.HC_ALGO_TC_BF16X6)


def test_bf16x6_space_to_depth_moves_bit_exact(hc):
    """A 2x2/s2 conv whose weights pick one input tap per output channel:
    y[co] = x[c][2ho + u][2wo + v] exactly, and grad_input puts each grad_output
    value back at that tap (zeros elsewhere), for 20-bit significands."""
    N, C, H, W, Co, s = 1, 64, 8, 512, 128, 2
    cfg = P.cfg_of(N, C, H, W, Co, s, s, 0, 1, 2)
    pick = [(co % C, co // C, 1 - co // C) for co in range(Co)]  # (c, u, v)
    w = np.zeros((Co, C, s, s), np.float32)
    for co, (c, u, v) in enumerate(pick):
        w[co, c, u, v] = 1.0
    x = synth.dyadic((N, C, H, W), 20, 1, 9, 1)
    gy = synth.dyadic((N, Co, H // s, W // s), 20, 1, 9, 2)
    algo = hc.HC_ALGO_TC_BF16X6
    y = R.fwd(cfg, x, w, None, algo)
    want = np.stack([x[:, c, u::s, v::s] for c, u, v in pick], axis=1)
    assert np.array_equal(y, want)
    gx = R.bwd_subset(cfg, x, w, gy, ("gx",), algo)["gx"]
    want = np.zeros_like(x)
    for co, (c, u, v) in enumerate(pick):
        want[:, c, u::s, v::s] = gy[:, co]
    assert np.array_equal(gx, want)


@pytest.mark.parametrize("S", [1, 4])
def test_bf16x6_permutation_bit_exact(hc, S):
    """A 1x1 conv whose weight is a permutation matrix moves values: y = x[perm]
    and grad_input = grad_output[perm^-1], exactly, for values with 20-bit
    significands -- so all three bf16 pieces reach the output, every channel and
    pixel lands where the tile layouts say, and nothing else is added."""
    N, C, H, W = 2, 256, 2, 256
    cfg = P.cfg_of(N, C, H, W, C, 1, 1, 0, 1, S)
    rng = np.random.default_rng(5)
    perm = rng.permutation(C)
    w = np.zeros((C, C, 1, 1), np.float32)
    w[np.arange(C), perm, 0, 0] = 1.0
    x = synth.dyadic((N, C, H, W), 20, 1, 6, 1)
    gy = synth.dyadic((N, C, H, W), 20, 1, 6, 2)
    algo = hc.HC_ALGO_TC_BF16X6
    y = R.fwd(cfg, x, w, None, algo)
    assert np.array_equal(y, x[:, perm])
    out = R.bwd_subset(cfg, x, w, gy, ("gx",), algo)
    inv = np.argsort(perm)
    assert np.array_equal(out["gx"], gy[:, inv])


@pytest.mark.parametrize("cfg", [P.cfg_of(2, 256, 4, 256, 256, 1, 1, 0, 1, 4),
                                 P.cfg_of(2, 128, 8, 512, 128, 2, 2, 0, 1, 2),
                                 P.cfg_of(1, 3, 16, 512, 128, 4, 4, 0, 1, 1)])
def test_bf16x6_dyadic_exact(hc, orc, cfg):
    """Multiples of 1/4 in [-4, 4]: every piece split and every fp32 sum of the
    GEMMs is exact, so forward, grad_input, grad_weight and their per-shard
    partials equal the oracle bit for bit (1x1, 2x2/s2, and a 4x4/s4 stem whose
    48-deep K ends inside a 32-chunk)."""
    Ho, Wo = R.out_hw(cfg)
    x = synth.dyadic((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), 2, 4, 8, 1)
    w = synth.dyadic((cfg["C_out"], cfg["C_in"], cfg["kh"], cfg["kw"]), 2, 4, 8, 2)
    b = synth.dyadic((cfg["C_out"],), 2, 4, 8, 3)
    gy = synth.dyadic((cfg["N"], cfg["C_out"], Ho, Wo), 2, 4, 8, 4)
    algo = hc.HC_ALGO_TC_BF16X6
    assert hc.hc_conv2d_select(hc.desc(cfg), 1) == (0, algo)
    assert np.array_equal(R.fwd(cfg, x, w, b, algo), orc.conv2d_fwd(cfg, x, w, b))
    out = R.bwd(cfg, x, w, gy, algo)
    assert np.array_equal(out["gx"], orc.conv2d_bwd_input(cfg, w, gy))
    assert np.array_equal(out["gw"], orc.conv2d_bwd_weight(cfg, x, gy))
    _, gwp_ref, _ = orc.sharded_bwd(cfg, x, w, gy)
    assert np.array_equal(out["gw_partials"], gwp_ref.astype(np.float32))


@pytest.mark.parametrize("cfg", [P.cfg_of(1, 128, 6, 256, 128, 5, 1, 2, 1, 2),
                                 P.cfg_of(1, 256, 5, 256, 128, 3, 1, 1, 1, 2),
                                 P.cfg_of(1, 128, 4, 512, 128, 7, 1, 3, 1, 4),
                                 dict(P.cfg_of(1, 128, 8, 256, 128, 5, 1, 2, 1, 2), num_shards_h=2)])
def test_tc_kxk_dyadic_exact(hc, orc, cfg):
    """K x K convs on the tensor-core path (3xTF32 conv passes, the weight gradient
    on bf16 pieces with every tap's shift a box coordinate), on multiples of 1/4 in
    [-4, 4]: every split and every fp32 sum is exact, so forward, grad_input,
    grad_weight and the per-shard partials equal the oracle bit for bit -- a tap
    read from a wrong row or column, or a slot written to the wrong tap or channel
    block, would show (5x5 over 2 shards, 3x3 with two 128-channel blocks, 7x7 over
    4 shards, a 2 x 2 grid)."""
    Ho, Wo = R.out_hw(cfg)
    x = synth.dyadic((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), 2, 4, 9, 1)
    w = synth.dyadic((cfg["C_out"], cfg["C_in"], cfg["kh"], cfg["kw"]), 2, 4, 9, 2)
    b = synth.dyadic((cfg["C_out"],), 2, 4, 9, 3)
    gy = synth.dyadic((cfg["N"], cfg["C_out"], Ho, Wo), 2, 4, 9, 4)
    algo = hc.HC_ALGO_TC_3XTF32
    assert hc.hc_conv2d_select(hc.desc(cfg), 1) == (0, algo)
    assert np.array_equal(R.fwd(cfg, x, w, b, algo), orc.conv2d_fwd(cfg, x, w, b))
    out = R.bwd(cfg, x, w, gy, algo)
    assert np.array_equal(out["gx"], orc.conv2d_bwd_input(cfg, w, gy))
    assert np.array_equal(out["gw"], orc.conv2d_bwd_weight(cfg, x, gy))
    assert np.array_equal(out["gb"], orc.conv2d_bwd_bias(cfg, gy))
    _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, x, w, gy)
    assert np.array_equal(out["gw_partials"], gwp_ref.astype(np.float32))
    assert np.array_equal(out["gb_partials"], gbp_ref.astype(np.float32))


@pytest.mark.parametrize("want", [("gx",), ("gw",), ("gb",), ("gw", "gb"), ("gw_partials", "gb_partials"),
                                  ("gx", "gb_partials")])
@pytest.mark.parametrize("name", ["config1_dense5x5", "dw7_ragged_S4", "tc_5x5_S2", "tc_down2x2s2_S2"])
def test_backward_output_subsets(hc, orc, name, want):
    """Outputs passed as NULL are skipped; the requested ones still match the oracle."""
    cfg, x, w, b, gy = CASES[name]()
    out = R.bwd_subset(cfg, x, w, gy, want)
    refs = dict(gx=lambda: orc.conv2d_bwd_input(cfg, w, gy), gw=lambda: orc.conv2d_bwd_weight(cfg, x, gy),
                gb=lambda: orc.conv2d_bwd_bias(cfg, gy))
    if "gw_partials" in want or "gb_partials" in want:
        _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, x, w, gy)
        refs["gw_partials"] = lambda: gwp_ref
        refs["gb_partials"] = lambda: gbp_ref
    for k in want:
        tol = TOL_FWD if k == "gx" else TOL_W
        assert R.normwise(out[k], refs[k]()) <= tol, (k, R.normwise(out[k], refs[k]()))


@pytest.mark.parametrize("name", ["tc_1x1", "pw_128to256_S4_half_pair", "pw_grid_2x4", "tc_down2x2s2_S2",
                                  "tc_stem4x4s4", "tc_5x5_S2", "dw7_ragged_S4"])
def test_bwd_reuse_bit_identical(hc, name):
    """hc_conv2d_bwd_reuse, reading x's operand copy from the forward workspace
    (bf16 pieces; other families keep nothing), gives hc_conv2d_bwd's results
    bit for bit, including the per-shard partials."""
    cfg, x, w, b, gy = CASES[name]()
    ref = R.bwd(cfg, x, w, gy)
    d = hc.desc(cfg)
    Ho, Wo = R.out_hw(cfg)
    xd, wd, bd, gyd = R.dev(x), R.dev(w), R.dev(b), R.dev(gy)
    y = torch.empty((cfg["N"], cfg["C_out"], Ho, Wo), device="cuda")
    wsf, nbf = R.workspace(d, 0)
    wsb, nbb = R.workspace(d, 2)
    Q = R.num_partials(cfg)
    gx = R.Guarded(x.shape)
    gw = R.Guarded(w.shape)
    gb = R.Guarded((cfg["C_out"],))
    gwp = R.Guarded((Q,) + w.shape)
    gbp = R.Guarded((Q, cfg["C_out"]))
    hc.check(hc.hc_conv2d_fwd(d, xd, wd, bd, y, wsf, nbf), "fwd")
    hc.check(hc.hc_conv2d_bwd_reuse(d, xd, wd, gyd, gx.view, gw.view, gb.view, gwp.view, gbp.view, wsb, nbb, wsf, nbf),
             "bwd reuse")
    hc.check(hc.hc_sync_check(), "sync")
    for k, g in (("gx", gx), ("gw", gw), ("gb", gb), ("gw_partials", gwp), ("gb_partials", gbp)):
        assert np.array_equal(g.numpy(), ref[k]), k


def _bwd_act(hc, cfg, xd, wd, gyd, act, y_pre=None, fwd_ws=None, want=("gx", "gw", "gb", "gw_partials",
                                                                          "gb_partials")):
    d = hc.desc(cfg)
    Q = R.num_partials(cfg)
    wshape = (cfg["C_out"], cfg["C_in"], 1, 1)
    shapes = dict(gx=tuple(xd.shape), gw=wshape, gb=(cfg["C_out"],), gw_partials=(Q,) + wshape,
                  gb_partials=(Q, cfg["C_out"]))
    o = {k: R.Guarded(shapes[k]) for k in want}
    ws, nb = R.workspace(d, 2 if fwd_ws else 1)
    fws, fnb = fwd_ws if fwd_ws else (None, 0)
    v = lambda k: o[k].view if k in o else None
    hc.check(hc.hc_conv2d_bwd_act(d, xd, wd, gyd, v("gx"), v("gw"), v("gb"), v("gw_partials"), v("gb_partials"), ws,
                                  nb, fws, fnb, algo=hc.HC_ALGO_TC_BF16X6, act=act, y_pre=y_pre), "bwd act")
    hc.check(hc.hc_sync_check(), "sync")
    return {k: g.numpy() for k, g in o.items()}


@pytest.mark.parametrize("name", ["pw_128to256_S4_half_pair", "pw_1024to256_S8", "pw_grid_2x4"])
def test_gelu_input_fusion(hc, orc, name):
    """HC_ACT_GELU_INPUT: the conv of GELU(x) against the oracle's GELU followed by
    its convolution; grad_input is the gradient with respect to GELU(x); the
    backward pass taking GELU(x)'s pieces from the forward workspace equals the
    one that splits them itself, bit for bit."""
    cfg, x, w, b, gy = CASES[name]()
    x = (2.0 * x).astype(np.float32)  # spread the pre-activations over GELU's curved part
    d = hc.desc(cfg)
    act = hc.HC_ACT_GELU_INPUT
    xd, wd, bd, gyd = R.dev(x), R.dev(w), R.dev(b), R.dev(gy)
    y = R.Guarded(gy.shape)
    wsf, nbf = R.workspace(d, 0)
    hc.check(hc.hc_conv2d_fwd_act(d, xd, wd, bd, y.view, wsf, nbf, algo=hc.HC_ALGO_TC_BF16X6, act=act), "fwd act")
    a = orc.gelu_fwd(x).astype(np.float32)
    assert R.normwise(y.numpy(), orc.conv2d_fwd(cfg, a, w, b)) <= TOL_FWD
    out = _bwd_act(hc, cfg, xd, wd, gyd, act, fwd_ws=(wsf, nbf))
    own = _bwd_act(hc, cfg, xd, wd, gyd, act)
    for k in out:
        assert np.array_equal(out[k], own[k]), k
    assert R.normwise(out["gx"], orc.conv2d_bwd_input(cfg, w, gy)) <= TOL_FWD
    assert R.normwise(out["gw"], orc.conv2d_bwd_weight(cfg, a, gy)) <= TOL_W
    assert R.normwise(out["gb"], orc.conv2d_bwd_bias(cfg, gy)) <= TOL_W
    _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, a, w, gy)
    assert R.normwise(out["gw_partials"], gwp_ref) <= TOL_W
    assert R.normwise(out["gb_partials"], gbp_ref) <= TOL_W


@pytest.mark.parametrize("name", ["pw_128to256_S4_half_pair", "pw_256to1024_S8", "pw_grid_2x4"])
def test_gelu_output_fusion(hc, orc, name):
    """HC_ACT_GELU_OUTPUT: gy is the gradient of GELU(y_pre); every gradient is the
    conv's for gy * GELU'(y_pre) (oracle: its GELU backward, then its conv
    backward), with and without the forward workspace, and with gb alone."""
    cfg, x, w, b, gy = CASES[name]()
    y_pre = synth.normal(gy.shape, 2.0, 11, 1)
    xd, wd, gyd, yd = R.dev(x), R.dev(w), R.dev(gy), R.dev(y_pre)
    d = hc.desc(cfg)
    act = hc.HC_ACT_GELU_OUTPUT
    y = torch.empty(gy.shape, device="cuda")
    wsf, nbf = R.workspace(d, 0)
    hc.check(hc.hc_conv2d_fwd_act(d, xd, wd, None, y, wsf, nbf, algo=hc.HC_ALGO_TC_BF16X6, act=act), "fwd")
    out = _bwd_act(hc, cfg, xd, wd, gyd, act, y_pre=yd, fwd_ws=(wsf, nbf))
    own = _bwd_act(hc, cfg, xd, wd, gyd, act, y_pre=yd)
    for k in out:
        assert np.array_equal(out[k], own[k]), k
    g = orc.gelu_bwd(y_pre, gy).astype(np.float32)
    assert R.normwise(out["gx"], orc.conv2d_bwd_input(cfg, w, g)) <= TOL_FWD
    assert R.normwise(out["gw"], orc.conv2d_bwd_weight(cfg, x, g)) <= TOL_W
    assert R.normwise(out["gb"], orc.conv2d_bwd_bias(cfg, g)) <= TOL_W
    _, gwp_ref, gbp_ref = orc.sharded_bwd(cfg, x, w, g)
    assert R.normwise(out["gw_partials"], gwp_ref) <= TOL_W
    assert R.normwise(out["gb_partials"], gbp_ref) <= TOL_W
    only_b = _bwd_act(hc, cfg, xd, wd, gyd, act, y_pre=yd, want=("gb",))
    assert np.array_equal(only_b["gb"], out["gb"])


def test_gelu_mlp_chain(hc, orc):
    """1x1 -> GELU -> 1x1 with the GELU folded into both convs (h = conv1(x),
    out = conv2(GELU(h)); backward: conv2 with HC_ACT_GELU_INPUT, conv1 with
    HC_ACT_GELU_OUTPUT on h) against the oracle's unfused chain."""
    c1 = P.cfg_of(1, 128, 2, 256, 256, 1, 1, 0, 1, 2)
    c2 = P.cfg_of(1, 256, 2, 256, 128, 1, 1, 0, 1, 2)
    x = synth.normal((1, 128, 2, 256), 1.0, 12, 1)
    w1 = synth.normal((256, 128, 1, 1), 0.15, 12, 2)
    w2 = synth.normal((128, 256, 1, 1), 0.1, 12, 3)
    b1, b2 = synth.normal((256,), 0.1, 12, 4), synth.normal((128,), 0.1, 12, 5)
    gout = synth.normal((1, 128, 2, 256), 1.0, 12, 6)
    d1, d2 = hc.desc(c1), hc.desc(c2)
    bf, gi, go = hc.HC_ALGO_TC_BF16X6, hc.HC_ACT_GELU_INPUT, hc.HC_ACT_GELU_OUTPUT
    xd, w1d, w2d, b1d, b2d, god = (R.dev(a) for a in (x, w1, w2, b1, b2, gout))
    h = torch.empty((1, 256, 2, 256), device="cuda")
    out = torch.empty((1, 128, 2, 256), device="cuda")
    ws1, n1 = R.workspace(d1, 0)
    ws2, n2 = R.workspace(d2, 0)
    hc.check(hc.hc_conv2d_fwd_act(d1, xd, w1d, b1d, h, ws1, n1, algo=bf, act=go), "fwd 1")
    hc.check(hc.hc_conv2d_fwd_act(d2, h, w2d, b2d, out, ws2, n2, algo=bf, act=gi), "fwd 2")
    g2 = _bwd_act(hc, c2, h, w2d, god, gi, fwd_ws=(ws2, n2))
    g1 = _bwd_act(hc, c1, xd, w1d, R.dev(g2["gx"]), go, y_pre=h, fwd_ws=(ws1, n1))
    h_ref = orc.conv2d_fwd(c1, x, w1, b1)
    a_ref = orc.gelu_fwd(h_ref).astype(np.float32)
    assert R.normwise(out.cpu().numpy(), orc.conv2d_fwd(c2, a_ref, w2, b2)) <= TOL_FWD
    ga_ref = orc.conv2d_bwd_input(c2, w2, gout)
    gh_ref = orc.gelu_bwd(h_ref, ga_ref).astype(np.float32)
    assert R.normwise(g1["gx"], orc.conv2d_bwd_input(c1, w1, gh_ref)) <= TOL_FWD
    assert R.normwise(g1["gw"], orc.conv2d_bwd_weight(c1, x, gh_ref)) <= TOL_W
    assert R.normwise(g1["gb"], orc.conv2d_bwd_bias(c1, gh_ref)) <= TOL_W
    assert R.normwise(g2["gw"], orc.conv2d_bwd_weight(c2, a_ref, gout)) <= TOL_W


@pytest.mark.parametrize("name", ["config1_dense5x5", "dw7_ragged_S4", "grouped_strided", "tc_5x5_S2",
                                  "pw_128to256_S4_half_pair"])
def test_deterministic(hc, name):
    cfg, x, w, b, gy = CASES[name]()
    y1, y2 = R.fwd(cfg, x, w, b), R.fwd(cfg, x, w, b)
    o1, o2 = R.bwd(cfg, x, w, gy), R.bwd(cfg, x, w, gy)
    assert np.array_equal(y1, y2)
    for k in o1:
        assert np.array_equal(o1[k], o2[k]), k


@pytest.mark.parametrize("cfg", [P.cfg_of(2, 3, 5, 32, 3, 5, 1, 2, 1, 4), P.cfg_of(1, 2, 4, 48, 2, 7, 1, 3, 2, 4),
                                 P.cfg_of(1, 2, 3, 16, 2, 3, 2, 2, 1, 2), P.cfg_of(1, 2, 3, 16, 2, 2, 2, 0, 1, 8),
                                 dict(P.cfg_of(2, 3, 12, 32, 3, 5, 1, 2, 1, 4), num_shards_h=3),
                                 dict(P.cfg_of(1, 2, 16, 16, 2, 3, 2, 2, 1, 2), num_shards_h=2)])
def test_halo_gather_bit_exact(hc, orc, cfg):
    x = synth.normal((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), 1.0, 3, 1)
    d = hc.desc(cfg)
    st, plan, _, _ = hc.hc_shard_plan(d)
    st2, plan_h = hc.hc_shard_plan_rows(d)
    assert st == 0 and st2 == 0
    We = max(e[2] + (e[1] - e[0]) + e[3] for e in plan)
    He = max(f[2] + (f[1] - f[0]) + f[3] for f in plan_h)
    Q = len(plan) * len(plan_h)
    xe = R.Guarded((Q, cfg["N"], cfg["C_in"], He, We))
    hc.check(hc.hc_halo_gather(d, R.dev(x), xe.view), "halo")
    hc.check(hc.hc_sync_check(), "halo sync")
    got = xe.numpy()
    for q in range(Q):
        ref = orc.halo_extend(cfg, q, x)
        hr, wr = ref.shape[-2:]
        assert np.array_equal(got[q, :, :, :hr, :wr], ref), q
        assert np.all(got[q, :, :, hr:, :] == 0) and np.all(got[q, :, :, :, wr:] == 0)


@pytest.mark.parametrize("K,S,groups", [(7, 4, "dw"), (5, 4, "dw"), (3, 2, "dw"), (5, 4, "dense"), (3, 2, "dense")])
def test_delta_kernels_bit_exact(hc, K, S, groups):
    """One-hot kernels on dyadic inputs: every output is one input value (or a
    zero of the padding), so the result must be the shifted input exactly, at
    every tap and across every shard edge."""
    p = (K - 1) // 2
    C = 2
    W = 128 * S if groups == "dw" else 8 * S
    cfg = P.cfg_of(1, C, 11, W, C, K, 1, p, C if groups == "dw" else 1, S)
    x = synth.dyadic((1, C, 11, W), 6, 4, 5, 1)
    xp = np.pad(x, ((0, 0), (0, 0), (p, p), (p, p)))
    for u in range(K):
        for v in range(K):
            w = np.zeros((C, 1 if groups == "dw" else C, K, K), np.float32)
            for c in range(C):
                w[c, 0 if groups == "dw" else c, u, v] = 1.0
            y = R.fwd(cfg, x, w, None)
            assert np.array_equal(y, xp[:, :, u:u + 11, v:v + W]), (u, v)


@pytest.mark.slow
def test_config2_full_size_sampled(hc, orc):
    """Depthwise 7x7, (7,256,128,512), 4 shards -- the size and launch the bench
    times -- checked on sampled outputs that the oracle computes one by one:
    random positions plus every shard-edge column of some rows."""
    N, C, H, W, K, S = 7, 256, 128, 512, 7, 4
    cfg = P.cfg_of(N, C, H, W, C, K, 1, 3, C, S)
    x = synth.normal((N, C, H, W), 1.0, 0, 1)
    w = synth.trunc_normal((C, 1, K, K), 0.02, 0, 2)
    b = np.zeros((C,), np.float32)
    gy = synth.normal((N, C, H, W), 1.0, 0, 4)
    y = R.fwd(cfg, x, w, b)
    out = R.bwd(cfg, x, w, gy)
    rng = np.random.default_rng(0)
    pts = [tuple(int(rng.integers(0, s)) for s in (N, C, H, W)) for _ in range(3000)]
    for col in (0, 1, 2, 3, 125, 126, 127, 128, 129, 130, 255, 256, 257, 383, 384, 385, 509, 510, 511):
        for hrow in (0, 1, 2, 64, 125, 126, 127):
            pts.append((int(rng.integers(0, N)), int(rng.integers(0, C)), hrow, col))
    yg = np.array([y[p] for p in pts])
    yr = np.array([orc.fwd_at(cfg, x, w, b, *p) for p in pts])
    assert R.normwise(yg, yr) <= TOL_FWD
    gg = np.array([out["gx"][p] for p in pts])
    gr = np.array([orc.gx_at(cfg, w, gy, *p) for p in pts])
    assert R.normwise(gg, gr) <= TOL_FWD
    chans = [0, 1, 100, 255]
    gwp_ref = np.array([[[orc.gw_at(cfg, x, gy, c, 0, u, v, r * 128, (r + 1) * 128) for u in range(K) for v in range(K)]
                         for c in chans] for r in range(S)])
    gwp = out["gw_partials"][:, chans, 0].reshape(S, len(chans), K * K)
    assert R.normwise(gwp, gwp_ref) <= TOL_W
    assert R.normwise(out["gw"][chans, 0].reshape(len(chans), K * K), gwp_ref.sum(0)) <= TOL_W
    gbp_ref = np.array([[orc.gb_at(cfg, gy, c, r * 128, (r + 1) * 128) for c in chans] for r in range(S)])
    assert R.normwise(out["gb_partials"][:, chans], gbp_ref) <= TOL_W
    assert R.normwise(out["gb"][chans], gbp_ref.sum(0)) <= TOL_W
    # properties that hold at any size: sum over shards of the partials is the full gradient
    assert np.abs(out["gw_partials"].astype(np.float64).sum(0) - out["gw"]).max() <= 1e-5 * np.abs(out["gw"]).max()


@pytest.mark.slow
def test_config3_full_size_sampled(hc, orc):
    """Dense 5x5 128->128, (7,128,128,1024), 4 shards on the tensor-core path,
    checked on sampled outputs the oracle computes one by one (random positions
    plus shard-edge columns) and on sampled per-shard weight-gradient partials."""
    N, C, H, W, K, S = 7, 128, 128, 1024, 5, 4
    cfg = P.cfg_of(N, C, H, W, C, K, 1, 2, 1, S)
    assert hc.hc_conv2d_select(hc.desc(cfg), 1) == (0, hc.HC_ALGO_TC_3XTF32)
    x = synth.normal((N, C, H, W), 1.0, 0, 1)
    w = synth.kaiming_normal((C, C, K, K), C * K * K, 0, 2)
    b = synth.normal((C,), 0.01, 0, 3)
    gy = synth.normal((N, C, H, W), 1.0, 0, 4)
    y = R.fwd(cfg, x, w, b)
    out = R.bwd(cfg, x, w, gy)
    rng = np.random.default_rng(1)
    pts = [tuple(int(rng.integers(0, s)) for s in (N, C, H, W)) for _ in range(1500)]
    for col in (0, 1, 254, 255, 256, 257, 511, 512, 767, 768, 1022, 1023):
        for hrow in (0, 1, 64, 126, 127):
            pts.append((int(rng.integers(0, N)), int(rng.integers(0, C)), hrow, col))
    yr = np.array([orc.fwd_at(cfg, x, w, b, *p) for p in pts])
    assert R.normwise(np.array([y[p] for p in pts]), yr) <= TOL_FWD
    gr = np.array([orc.gx_at(cfg, w, gy, *p) for p in pts])
    assert R.normwise(np.array([out["gx"][p] for p in pts]), gr) <= TOL_FWD
    wpts = [tuple(int(rng.integers(0, s)) for s in (C, C, K, K)) for _ in range(6)] + [(0, 0, 0, 0), (127, 127, 4, 4)]
    got, ref = [], []
    for r in range(S):
        for (co, ci, u, v) in wpts:
            got.append(out["gw_partials"][r, co, ci, u, v])
            ref.append(orc.gw_at(cfg, x, gy, co, ci, u, v, r * 256, (r + 1) * 256))
    assert R.normwise(np.array(got), np.array(ref)) <= TOL_W
    assert np.abs(out["gw_partials"].astype(np.float64).sum(0) - out["gw"]).max() <= 1e-5 * np.abs(out["gw"]).max()


@pytest.mark.parametrize("name,family", [("dw7_ragged_S4", "DEPTHWISE"), ("dw5_S2", "DEPTHWISE"),
                                         ("dw3_S4", "DEPTHWISE"), ("dw7_grid_2x2", "DEPTHWISE"),
                                         ("dw7_grid_4x2", "DEPTHWISE"), ("tc_5x5_S2", "TC_3XTF32"),
                                         ("tc_down2x2s2_S2", "TC_BF16X6"), ("config1_dense5x5", "DIRECT")])
def test_bwd_residual(hc, orc, name, family):
    """hc_conv2d_bwd_residual: grad_input plus the gradient reaching x along a
    skip connection, against the oracle's grad_input plus that gradient; the
    parameter gradients equal hc_conv2d_bwd's bit for bit.  Aliasing the
    residual with gx, or passing no gx, is refused."""
    cfg, x, w, b, gy = CASES[name]()
    algo = getattr(hc, "HC_ALGO_" + family)
    d = hc.desc(cfg)
    res = synth.normal(x.shape, 1.0, 17, 1)
    wshape = (cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"])
    gx, gw, gb = R.Guarded(x.shape), R.Guarded(wshape), R.Guarded((cfg["C_out"],))
    ws, nb = R.workspace(d, 1, algo)
    xd, wd, gyd, rd = R.dev(x), R.dev(w), R.dev(gy), R.dev(res)
    hc.check(hc.hc_conv2d_bwd_residual(d, xd, wd, gyd, rd, gx.view, gw.view, gb.view, ws=ws, ws_bytes=nb, algo=algo),
             "bwd residual")
    hc.check(hc.hc_sync_check(), "bwd residual sync")
    ref = orc.conv2d_bwd_input(cfg, w, gy) + res.astype(np.float64)
    assert R.normwise(gx.numpy(), ref) <= TOL_FWD
    plain = R.bwd(cfg, x, w, gy, algo, partials=False)
    assert np.array_equal(gw.numpy(), plain["gw"]) and np.array_equal(gb.numpy(), plain["gb"])
    assert np.array_equal(rd.cpu().numpy(), res)  # the residual is only read
    # grad_input alone (no parameter gradients): the same values
    gx_only = R.Guarded(x.shape)
    hc.check(hc.hc_conv2d_bwd_residual(d, xd, wd, gyd, rd, gx_only.view, None, None, ws=ws, ws_bytes=nb, algo=algo),
             "bwd residual gx only")
    hc.check(hc.hc_sync_check(), "bwd residual gx only sync")
    assert np.array_equal(gx_only.numpy(), gx.numpy())
    assert hc.hc_conv2d_bwd_residual(d, xd, wd, gyd, gx.view, gx.view, gw.view, gb.view, ws=ws, ws_bytes=nb,
                                     algo=algo) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_conv2d_bwd_residual(d, xd, wd, gyd, rd, None, gw.view, gb.view, ws=ws, ws_bytes=nb,
                                     algo=algo) == hc.HC_ERR_INVALID_ARG
