"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every function include/hc.h declares; the shard plan and the argument
checks behave as documented."""
import itertools
import os
import re
import subprocess

import pytest

import oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hc():
    from spatially_sharded_cnn_gb300 import build
    build.build()
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def declared_functions():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(hc_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(hc):
    names = declared_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", hc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (hc_\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(hc._lib, n)
    assert set(hc.EXPORTS) <= set(names)


def test_trace_without_launches(hc):
    """The per-kernel trace API on the host: enabling, collecting with nothing
    recorded, and argument errors."""
    assert hc.hc_trace_enable(True) == hc.HC_OK
    assert hc.hc_trace_enable(False) == hc.HC_OK
    st, table = hc.hc_trace_collect()
    assert table == {}
    import ctypes as C
    n = C.c_int(7)
    assert hc._lib.hc_trace_collect(None, 4, C.byref(n)) == hc.HC_ERR_INVALID_ARG
    assert hc._lib.hc_trace_collect(None, 0, None) == hc.HC_ERR_INVALID_ARG


def test_status_strings(hc):
    for s in range(6):
        assert hc.hc_status_string(s) and hc.hc_status_string(s) != "unknown status"
    assert hc.hc_status_string(99) == "unknown status"


def test_plan_matches_oracle(hc, orc):
    for W, S, k, s, p in itertools.product((8, 12, 16, 32, 48), (1, 2, 3, 4, 8), (1, 2, 3, 4, 5, 7),
                                            (1, 2, 4), (0, 1, 2, 3)):
        cfg = P.cfg_of(2, 3, 9, W, 3, k, s, p, 1, S)
        if W + 2 * p < k:
            continue
        st, ext, Ho, Wo = hc.hc_shard_plan(hc.desc(cfg))
        rc, plan, oHo, oWo = orc.shard_plan(cfg)
        if rc:
            assert st == hc.HC_ERR_UNSUPPORTED, (cfg, st, rc)
            continue
        assert st == hc.HC_OK, cfg
        assert ext == plan and (Ho, Wo) == (oHo, oWo), cfg


def test_row_plan_matches_oracle(hc, orc):
    for H, Sh, k, s, p in itertools.product((8, 12, 16, 24), (0, 1, 2, 3, 4), (1, 2, 3, 5), (1, 2), (0, 1, 2)):
        cfg = dict(P.cfg_of(1, 2, H, 16, 2, k, s, p, 1, 2), num_shards_h=Sh)
        if H + 2 * p < k:
            continue
        st, ext = hc.hc_shard_plan_rows(hc.desc(cfg))
        rc, plan = orc.shard_plan_h(cfg)
        rcw = orc.shard_plan(cfg)[0]
        if rc or rcw:
            assert st == hc.HC_ERR_UNSUPPORTED, (cfg, st, rc, rcw)
            continue
        assert st == hc.HC_OK and ext == plan, (cfg, ext, plan)


def test_plan_pages_example(hc):
    # (7,3,512,2048) over 4 shards -> 4 blocks of 512 columns; 5x5/p2/s1 -> 2-column halos
    st, ext, Ho, Wo = hc.hc_shard_plan(hc.desc(P.cfg_of(7, 3, 512, 2048, 3, 5, 1, 2, 1, 4)))
    assert st == 0 and (Ho, Wo) == (512, 2048)
    assert [e[1] - e[0] for e in ext] == [512] * 4
    assert all(e[2] == 2 and e[3] == 2 for e in ext)


def test_argument_errors_before_launch(hc):
    d = hc.desc(P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4))
    # null tensors
    assert hc.hc_conv2d_fwd(d, None, None, None, None) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_conv2d_bwd(d, None, None, None, None, None, None) == hc.HC_ERR_INVALID_ARG
    # misaligned pointers (never dereferenced: the check comes first)
    assert hc.hc_conv2d_fwd(d, 4, 16, None, 32) == hc.HC_ERR_INVALID_ARG
    # invalid descs
    for bad in (dict(N=0), dict(groups=3), dict(stride=0), dict(padding=-1), dict(num_shards=0), dict(kh=40)):
        dd = hc.desc(dict(P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4), **bad))
        assert hc.hc_conv2d_fwd(dd, 256, 256, None, 256) == hc.HC_ERR_INVALID_ARG, bad
        assert hc.hc_shard_plan(dd)[0] == hc.HC_ERR_INVALID_ARG, bad
    # unsupported plans
    for bad in (dict(num_shards=3), dict(W=10, num_shards=5, kh=7, kw=7, padding=3)):
        dd = hc.desc(dict(P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4), **bad))
        assert hc.hc_conv2d_fwd(dd, 256, 256, None, 256) == hc.HC_ERR_UNSUPPORTED, bad
    # an algorithm that does not cover the desc
    assert hc.hc_conv2d_fwd(d, 256, 256, None, 256, algo=hc.HC_ALGO_DEPTHWISE) == hc.HC_ERR_UNSUPPORTED
    # too small a workspace for the backward pass
    st, nb = hc.hc_conv2d_workspace_size(d, 1)
    assert st == 0 and nb > 0
    assert hc.hc_conv2d_bwd(d, 256, 256, 256, 256, 256, 256, None, None, 256, nb - 1) == hc.HC_ERR_WORKSPACE
    # maximum sizes: 10^12 elements and more are refused, as are more than 1024 shards
    huge = hc.desc(P.cfg_of(1000, 1000, 1000, 1024, 4, 3, 1, 1, 1, 4))
    assert hc.hc_conv2d_fwd(huge, 256, 256, None, 256) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_shard_plan(huge)[0] == hc.HC_ERR_INVALID_ARG
    many = hc.desc(P.cfg_of(1, 1, 4, 4096, 1, 1, 1, 0, 1, 2048))
    assert hc.hc_shard_plan(many)[0] == hc.HC_ERR_UNSUPPORTED
    # the residual backward: a residual is required, 16-byte aligned and not gx itself; gx is required
    args = (d, 256, 256, 256)
    assert hc.hc_conv2d_bwd_residual(*args, None, 512, 256, 256, ws=256, ws_bytes=nb) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_conv2d_bwd_residual(*args, 512, 512, 256, 256, ws=256, ws_bytes=nb) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_conv2d_bwd_residual(*args, 520, 512, 256, 256, ws=256, ws_bytes=nb) == hc.HC_ERR_INVALID_ARG
    assert hc.hc_conv2d_bwd_residual(*args, 512, None, 256, 256, ws=256, ws_bytes=nb) == hc.HC_ERR_INVALID_ARG


def test_algorithm_choice(hc):
    dw = hc.desc(P.cfg_of(7, 256, 128, 512, 256, 7, 1, 3, 256, 4))
    assert hc.hc_conv2d_select(dw, 0) == (0, hc.HC_ALGO_DEPTHWISE)
    assert hc.hc_conv2d_select(dw, 1) == (0, hc.HC_ALGO_DEPTHWISE)
    small = hc.desc(P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1, 4))
    st, a = hc.hc_conv2d_select(small, 0)
    assert st == 0 and a in (hc.HC_ALGO_DIRECT, hc.HC_ALGO_TC_3XTF32)
    # depthwise tiles are 128 columns inside a shard: 64-column shards fall back
    odd = hc.desc(P.cfg_of(1, 8, 16, 256, 8, 7, 1, 3, 8, 4))
    assert hc.hc_conv2d_select(odd, 0) == (0, hc.HC_ALGO_DIRECT)


def test_bwd_reuse_arguments(hc):
    """The reusing backward pass checks the forward workspace it is handed and
    needs a smaller workspace of its own (no copy of x) for the bf16-piece GEMM;
    other algorithms keep nothing, so their pass-2 size is the pass-1 size."""
    pw = hc.desc(P.cfg_of(2, 256, 8, 256, 256, 1, 1, 0, 1, 2))
    bf = hc.HC_ALGO_TC_BF16X6
    st1, b1 = hc.hc_conv2d_workspace_size(pw, 1, bf)
    st2, b2 = hc.hc_conv2d_workspace_size(pw, 2, bf)
    st0, b0 = hc.hc_conv2d_workspace_size(pw, 0, bf)
    assert st0 == st1 == st2 == 0 and b2 < b1 and b1 - b2 >= 6 * 2 * 256 * 8 * 256
    assert hc.hc_conv2d_workspace_size(pw, 3, bf)[0] == hc.HC_ERR_INVALID_ARG
    dense = hc.desc(P.cfg_of(1, 128, 8, 256, 128, 5, 1, 2, 1, 2))
    assert hc.hc_conv2d_workspace_size(dense, 2)[1] == hc.hc_conv2d_workspace_size(dense, 1)[1]
    call = lambda fws, fnb: hc.hc_conv2d_bwd_reuse(pw, 256, 256, 256, 256, 256, 256, None, None, 256, b2, fws, fnb,
                                                   algo=bf)
    assert call(None, b0) == hc.HC_ERR_INVALID_ARG      # no forward workspace
    assert call(256 + 128, b0) == hc.HC_ERR_INVALID_ARG  # not 256-byte aligned
    assert call(256, b0 - 1) == hc.HC_ERR_WORKSPACE     # too small
    assert hc.hc_conv2d_bwd_reuse(pw, 256, 256, 256, 256, 256, 256, None, None, 256, b2 - 1, 256, b0,
                                  algo=bf) == hc.HC_ERR_WORKSPACE


def test_gelu_input_support(hc):
    """A folded GELU is a bf16-piece 1x1 feature: other algorithms, kernels and
    strides refuse it before launching anything."""
    act = hc.HC_ACT_GELU_INPUT
    pw = hc.desc(P.cfg_of(1, 256, 8, 256, 256, 1, 1, 0, 1, 2))
    _, nb = hc.hc_conv2d_workspace_size(pw, 0, hc.HC_ALGO_TC_3XTF32)
    assert hc.hc_conv2d_fwd_act(pw, 256, 256, None, 256, 256, nb, algo=hc.HC_ALGO_TC_3XTF32,
                                act=act) == hc.HC_ERR_UNSUPPORTED
    for cfg in (P.cfg_of(1, 128, 8, 256, 128, 5, 1, 2, 1, 2), P.cfg_of(1, 128, 8, 256, 128, 2, 2, 0, 1, 2)):
        d = hc.desc(cfg)
        _, nb = hc.hc_conv2d_workspace_size(d, 0)
        assert hc.hc_conv2d_fwd_act(d, 256, 256, None, 256, 256, nb, act=act) == hc.HC_ERR_UNSUPPORTED, cfg
        _, nb1 = hc.hc_conv2d_workspace_size(d, 1)
        assert hc.hc_conv2d_bwd_act(d, 256, 256, 256, 256, 256, 256, None, None, 256, nb1,
                                    act=act) == hc.HC_ERR_UNSUPPORTED, cfg
    # a GELU on the output needs its pre-activation
    _, nb1 = hc.hc_conv2d_workspace_size(pw, 1)
    assert hc.hc_conv2d_bwd_act(pw, 256, 256, 256, 256, 256, 256, None, None, 256, nb1,
                                act=hc.HC_ACT_GELU_OUTPUT) == hc.HC_ERR_INVALID_ARG


def test_pointwise_algorithm_choice(hc):
    """1x1 convs with 128-multiple channels go to the bf16-piece GEMM; its
    operand copies take 6 bytes per element against 8 for tf32 hi / lo."""
    for ci, co in ((256, 1024), (1024, 256)):
        d = hc.desc(P.cfg_of(7, ci, 128, 1024, co, 1, 1, 0, 1, 8))
        assert hc.hc_conv2d_select(d, 0) == (0, hc.HC_ALGO_TC_BF16X6)
        assert hc.hc_conv2d_select(d, 1) == (0, hc.HC_ALGO_TC_BF16X6)
        st6, b6 = hc.hc_conv2d_workspace_size(d, 0, hc.HC_ALGO_TC_BF16X6)
        st3, b3 = hc.hc_conv2d_workspace_size(d, 0, hc.HC_ALGO_TC_3XTF32)
        assert st6 == 0 and st3 == 0 and b6 < b3
        assert b6 >= 6 * 7 * ci * 128 * 1024
    # the block's stem (4x4/s4, 3 -> 256) and a 2x2/s2 downsample: space-to-depth GEMMs
    for cfg in (P.cfg_of(7, 3, 512, 4096, 256, 4, 4, 0, 1, 8), P.cfg_of(7, 256, 128, 2048, 512, 2, 2, 0, 1, 8)):
        assert hc.hc_conv2d_select(hc.desc(cfg), 1) == (0, hc.HC_ALGO_TC_BF16X6)
    # not a 1x1 / stride-1 / unpadded conv, or shard columns not whole 32-pixel chunks
    for cfg in (P.cfg_of(1, 128, 8, 256, 128, 3, 1, 1, 1, 2), P.cfg_of(1, 128, 8, 256, 128, 1, 1, 0, 1, 16),
                P.cfg_of(1, 96, 8, 256, 128, 1, 1, 0, 1, 2), P.cfg_of(1, 128, 8, 256, 96, 2, 2, 0, 1, 2),
                P.cfg_of(1, 128, 8, 256, 128, 2, 2, 1, 1, 2), P.cfg_of(1, 3, 8, 256, 128, 2, 2, 0, 1, 2)):
        d = hc.desc(cfg)
        assert hc.hc_conv2d_workspace_size(d, 0, hc.HC_ALGO_TC_BF16X6)[0] == hc.HC_ERR_UNSUPPORTED, cfg
        assert hc.hc_conv2d_select(d, 0)[1] != hc.HC_ALGO_TC_BF16X6
