"""The bench's accounting, without a GPU: the algorithmic bytes and FLOPs per
step that its throughput and roofline figures divide by, the peaks it divides
them into, and the check that ties a DRAM-traffic record to the source it was
taken on.

Each expected figure is worked out here from the workload's own definition
(tensor shapes, kernel taps, which passes a step runs), not by calling the
bench's helpers: a dropped pass, a wrong element count or a transposed
dimension in the bench shows up as a mismatch.
"""
import hashlib
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_depthwise_bytes_and_flops(bench):
    """Depthwise 7x7 on (7,256,128,512): a step moves five fp32 tensors of that
    shape (forward reads x and writes y; backward reads x and grad_output and
    writes grad_input) and runs three stencil passes of 49 MACs per element."""
    wl = bench.make_workload("dw7")
    E = 7 * 256 * 128 * 512
    assert E == 117_440_512
    assert wl.bytes == (2 + 3) * 4 * E == 2_348_810_240
    assert wl.flops == 3 * 49 * 2 * E
    assert abs(wl.flops - 34.53e9) < 0.01e9
    # throughput unit: GB/s of those bytes
    assert wl.value(1.0) == pytest.approx(2_348_810_240 / 1e-3 / 1e9)
    # per-kernel work: the forward one pass (x in, y out), the backward two
    # (grad_input and the weight correlation; x and grad_output in, grad_input out)
    kw = wl.kernel_work()
    assert kw["dw_fwd_kernel"] == ("alu", 49 * 2 * E, 8 * E)
    assert kw["dw_bwd_kernel"] == ("alu", 2 * 49 * 2 * E, 12 * E)


def test_dense_flops(bench):
    """Dense 5x5 128 -> 128 on (7,128,128,1024), stride 1, padding 2: each
    output pixel of each output channel takes 128 * 25 MACs; forward,
    grad_input and grad_weight each do that many."""
    wl = bench.make_workload("dense5x5")
    per_pass = 2 * (7 * 128 * 1024) * 128 * (128 * 25)
    assert per_pass == 751_619_276_800
    assert wl.flops == 3 * per_pass
    kw = wl.kernel_work()
    assert kw["tc_conv_kernel 3xTF32 conv pass"] == ("tensor_tf32", 2 * per_pass, None)
    assert kw["tc_conv_kernel bf16x6 weight-gradient pass"] == ("tensor", per_pass, None)


def test_small_dense_flops(bench):
    """The (1,4,16,32) 5x5 case: 512 output pixels x 4 channels x 100 MACs per pass."""
    wl = bench.make_workload("config1")
    assert wl.flops == 3 * 2 * (16 * 32) * 4 * (4 * 25) == 1_228_800


def test_block_flops(bench):
    """ConvNeXt-XL stage-1 block on a (7,3,512,4096) image: the 4x4/s4 stem
    (3 -> 256, 48 MACs per output), the depthwise 7x7, the 1x1 convs 256 -> 1024
    and 1024 -> 256 on 128 x 1024 pixels.  A step runs every conv forward, the
    stem's weight gradient only (the image needs no gradient) and both
    gradients of the other three."""
    wl = bench.make_workload("block")
    px = 7 * 128 * 1024
    stem = 2 * px * 256 * 48
    dw = 2 * px * 256 * 49
    pw = 2 * px * 1024 * 256
    assert abs(stem - 2.25e10) < 0.01e10 and abs(dw - 2.30e10) < 0.01e10 and abs(pw - 4.81e11) < 0.01e11
    assert wl.flops == (stem + dw + 2 * pw) + (stem + 2 * dw + 4 * pw)
    kw = wl.kernel_work()
    # the bf16-piece GEMM: stem forward, each 1x1 conv forward and grad_input; its weight gradients
    assert kw["tc_conv_kernel bf16x6 conv pass"][1] == stem + 4 * pw
    assert kw["tc_conv_kernel bf16x6 weight-gradient pass"][1] == 2 * pw
    assert kw["patchify_wgrad_kernel"][1] == stem
    # stem bytes: the image and the 256-channel stem output, once each
    assert wl.stem_bytes() == 4 * (7 * 3 * 512 * 4096 + 7 * 256 * 128 * 1024)
    ow = wl.op_work()
    E = 7 * 256 * 128 * 1024
    assert ow["ls_fwd"] == ("hbm", 12 * E)  # residual and branch in, sum out


def test_depthwise_downsample_flops(bench):
    """Depthwise 7x7 on (7,256,128,2048) then a 2x2/s2 conv 256 -> 512: the
    downsample has 64 x 1024 output pixels, each of 512 channels taking 256 * 4
    MACs; three passes of each."""
    wl = bench.make_workload("dwdown")
    dw = 2 * (7 * 256 * 128 * 2048) * 49
    ds = 2 * (7 * 64 * 1024) * 512 * (256 * 4)
    assert abs(3 * dw - 138e9) < 1e9 and abs(3 * ds - 1.44e12) < 0.01e12
    assert wl.flops == 3 * (dw + ds)


def test_peaks(bench):
    """The FP32 peak is 152 SMs x 128 FMA lanes x 2 FLOP x the clock; the
    fp32-equivalent tensor peaks divide the measured bf16 rate by the passes
    one fp32 product costs."""
    assert bench.alu_peak({"sm_max_mhz": 2070.0}, 152) == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    assert bench.alu_peak({"sm_max_mhz": 2070.0}, 152) == pytest.approx(80.54784)
    assert bench.tc_peak({"bf16": 1922.0}) == pytest.approx(1922.0 * 1.1 / 2.25 / 3)
    assert bench.bf16x6_peak({"bf16": 1922.0}) == pytest.approx(1922.0 / 6)


def test_kernel_rooflines_arithmetic(bench):
    """A kernel's achieved rate is its work per step over its device time per
    step; the line's fraction is that over the kernel's own peak."""
    peaks = {"hbm": 6771.5, "bf16": 1922.0, "sm_max_mhz": 2070.0, "src": "measured"}
    table = bench.kernel_table({"dw_bwd_kernel": (2, 0.8), "dw_fwd_kernel": (2, 0.4)}, steps=2)
    assert table["dw_bwd_kernel"]["ms_per_launch"] == pytest.approx(0.4)
    assert table["dw_bwd_kernel"]["share"] == pytest.approx(2 / 3)
    work = {"dw_bwd_kernel": ("alu", 2.0e10, 1.0e9), "dw_fwd_kernel": ("alu", 1.0e10, None)}
    r = bench.kernel_rooflines(table, work, peaks, 152)
    bwd = r["dw_bwd_kernel"]
    assert bwd["achieved"] == pytest.approx(2.0e10 / 0.4e-3 / 1e12)  # 50 TFLOP/s
    assert bwd["frac"] == pytest.approx(50.0 / 80.54784)
    assert bwd["hbm"]["achieved"] == pytest.approx(1.0e9 / 0.4e-3 / 1e9)  # 2500 GB/s
    assert bwd["traffic"] is None  # no record asked for
    o = bench.op_rooflines({"ls_fwd": 0.5}, {"ls_fwd": ("hbm", 3.0e9)}, peaks, 152)
    assert o["ls_fwd"]["achieved"] == pytest.approx(6000.0) and o["ls_fwd"]["unit"] == "GB/s"


def test_traffic_records_match_their_sources(bench):
    """Every committed DRAM-traffic record names a traced kernel whose source
    file exists; the bench reports a record only while the file's hash is the
    one the record was taken on."""
    recs = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert recs
    for wl, kernels in recs.items():
        for k, d in kernels.items():
            src = bench.kernel_src(k)
            assert src and os.path.exists(src), (wl, k)
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            got = bench.traffic_for(wl, k, src)
            assert got == (d["bytes_per_launch"] if d["source_sha"] == h else None), (wl, k)
            assert d["bytes_per_launch"] > 0
