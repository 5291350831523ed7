"""Benchmark of the width-sharded (halo-exchange) Conv2d, forward + backward.

One step = one pass of the whole hot path over one batch, through the C ABI on
the current CUDA stream: hc_conv2d_fwd (shard plan, halo exchange + concat,
local conv, crop) then hc_conv2d_bwd (grad_output halo, grad_input, per-shard
_Partial grad_weight / grad_bias, fixed-order reduction).

Workloads (--workload):
  dw7       (default) ConvNeXt depthwise 7x7, padding 3, groups = C, fp32,
            x (7,256,128,512) N(0,1), weight (256,1,7,7) trunc-normal std 0.02,
            bias 0, grad_output N(0,1), 4 W-shards of width 128.  Metric:
            algorithmic HBM bytes per step (x + y forward; x + grad_output +
            grad_input backward) over the step time, GB/s.
  dense5x5  dense 5x5 conv 128->128 (3xTF32 tensor cores), x (7,128,128,1024),
            4 W-shards of width 256; TFLOP/s of the fp32 convolution FLOPs.
  block     ConvNeXt-XL stage-1 block on the stem output of a (7,3,512,4096)
            U[0,1] image, 8 W-shards: 4x4/s4 stem 3->256, depthwise 7x7,
            LayerNorm over C, 1x1 256->1024, GELU, 1x1 1024->256, layer scale
            1e-6 + residual; forward + backward; TFLOP/s of the conv FLOPs
            (stem and 1x1 convs on the bf16-piece tensor-core GEMM; the GELU
            folded into the 1x1 convs' operand splits, forward and backward).
  dwdown    depthwise 7x7 then 2x2/s2 downsample 256->512 on x
            (7,256,128,2048), 8 W-shards; forward + backward; TFLOP/s.
All inputs are larger than the 129 MB L2, so no flush is needed between steps.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload ...]
For N > 1 it runs under torch.distributed.run, one replica per GPU (each rank
its own batch; no data-path collective), and reports the whole-job total.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "halo-tiled conv fwd+bwd: HBM GB/s (depthwise) / TFLOP/s (dense), % roofline"
FP32_LANES_PER_SM = 128  # Blackwell: 128 FP32 FMA lanes per SM


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]), sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, sm_max_mhz=2070.0, src="fallback")


def conv_cfg(N, Ci, H, W, Co, k, s, p, g, S):
    return dict(N=N, C_in=Ci, H=H, W=W, C_out=Co, kh=k, kw=k, stride=s, padding=p, groups=g, num_shards=S)


def conv_flops(cfg):
    Ho = (cfg["H"] + 2 * cfg["padding"] - cfg["kh"]) // cfg["stride"] + 1
    Wo = (cfg["W"] + 2 * cfg["padding"] - cfg["kw"]) // cfg["stride"] + 1
    return 2.0 * cfg["N"] * Ho * Wo * cfg["C_out"] * (cfg["C_in"] // cfg["groups"]) * cfg["kh"] * cfg["kw"]


def tc_peak(peaks):
    """3xTF32 peak (fp32-equivalent): measured bf16 dense rate x the nominal
    tf32/bf16 ratio (1.1 / 2.25 PFLOP/s), / 3 for the three TF32 passes."""
    return peaks["bf16"] * (1.1 / 2.25) / 3


def bf16x6_peak(peaks):
    """Peak of the bf16-piece GEMMs (fp32-equivalent): measured bf16 dense rate
    / 6, the six bf16 products that stand for one fp32 product."""
    return peaks["bf16"] / 6


def op_rooflines(ops_ms, work, peaks, sms):
    """Per-op rates against each op's own bound.  work: op -> (bound, amount[,
    hbm bytes]) with bound "tensor" (fp32 FLOPs on the bf16-piece GEMM), "alu"
    (FP32 FLOPs) or "hbm" (algorithmic bytes); a compute-bound op may also give
    its algorithmic HBM bytes, reported beside; ops without an entry are left out."""
    out = {}
    for op, ms in ops_ms.items():
        if op not in work or ms <= 0:
            continue
        bound, amount = work[op][:2]
        if bound == "hbm":
            a, peak, unit = amount / (ms * 1e-3) / 1e9, peaks["hbm"], "GB/s"
        else:
            a = amount / (ms * 1e-3) / 1e12
            peak, unit = (bf16x6_peak(peaks), "TFLOP/s") if bound == "tensor" else (alu_peak(peaks, sms), "TFLOP/s")
        out[op] = {"bound": bound, "achieved": a, "unit": unit, "peak": peak, "frac": a / peak}
        if len(work[op]) > 2 and work[op][2]:
            hb = work[op][2] / (ms * 1e-3) / 1e9
            out[op]["hbm"] = {"achieved": hb, "peak": peaks["hbm"], "unit": "GB/s", "frac": hb / peaks["hbm"]}
    return out


def alu_peak(peaks, sms):
    return sms * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12


# Source file of each traced kernel (a DRAM-traffic record applies only to the source it was taken on).
KERNEL_SRC = {"dw_": "dw.cu", "tc_conv_kernel": "tc.cu", "ln_": "pointwise.cu", "ls_": "pointwise.cu",
              "bias_rows": "reduce.cu", "direct_": "direct.cu", "patchify_": "patchify.cu"}


def kernel_src(name):
    for pre, f in KERNEL_SRC.items():
        if name.startswith(pre):
            return os.path.join(ROOT, "spatially_sharded_cnn_gb300", "csrc", f)
    return None


def kernel_table(trace, steps):
    """Traced kernels: launches per step, device ms per launch and share of the traced time."""
    tot = sum(ms for _, ms in trace.values()) or 1.0
    return {k: {"launches_per_step": n / steps, "ms_per_launch": ms / n, "ms_per_step": ms / steps,
                "share": ms / tot}
            for k, (n, ms) in sorted(trace.items(), key=lambda kv: -kv[1][1])}


def peak_of(bound, peaks, sms):
    if bound == "alu":
        return alu_peak(peaks, sms), "TFLOP/s", \
            f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz"
    if bound == "tensor_tf32":
        return tc_peak(peaks), "TFLOP/s (fp32-equivalent, 3xTF32)", \
            f"measured bf16 {peaks['bf16']:.0f} TFLOP/s x 1.1/2.25 (nominal tf32/bf16) / 3 (3xTF32 passes)"
    if bound == "tensor":
        return bf16x6_peak(peaks), "TFLOP/s (fp32-equivalent, six bf16 products)", \
            f"measured bf16 {peaks['bf16']:.0f} TFLOP/s / 6 (bf16 products per fp32 product)"
    return peaks["hbm"], "GB/s", f"{peaks['src']} HBM copy bandwidth"


def kernel_rooflines(table, work, peaks, sms, traffic_key=None):
    """Each traced kernel with a work entry, against its own bound; the dominant
    one (largest device time per step) is the line's roofline."""
    out = {}
    for k, row in table.items():
        if k not in work:
            continue
        bound, amount, nbytes = work[k]
        t = row["ms_per_step"] * 1e-3
        peak, unit, src = peak_of(bound, peaks, sms)
        a = amount / t / (1e9 if bound == "hbm" else 1e12)
        r = {"bound": bound if bound in ("alu", "hbm") else "tensor", "kernel": k, "achieved": a, "peak": peak,
             "unit": unit, "frac": a / peak, "peak_source": src, "ms_per_launch": row["ms_per_launch"],
             "launches_per_step": row["launches_per_step"], "share": row["share"]}
        if nbytes:
            gbs = nbytes / t / 1e9
            r["hbm"] = {"achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                        "peak_source": peaks["src"]}
        src_file = kernel_src(k)
        r["traffic"] = traffic_for(traffic_key, k, src_file) if src_file and traffic_key else None
        out[k] = r
    return out


class Runner:
    """Device state shared by the workloads: the C ABI, a stream, a workspace
    shared by the backward passes and the pointwise ops, each conv's forward
    workspace, and per-op CUDA events for the op breakdown."""

    def __init__(self, hc, torch, dev, stream):
        self.hc, self.torch, self.dev, self.stream = hc, torch, dev, stream
        self.ws = None
        self.ws_bytes = 0
        self.fws = {}  # each conv's own forward workspace, kept for its backward pass
        self.mark = None  # when set: list collecting (name, start event, end event)

    def empty(self, shape):
        return self.torch.empty(shape, dtype=self.torch.float32, device=self.dev)

    def upload(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def reserve(self, nbytes):
        if nbytes > self.ws_bytes:
            self.ws = self.torch.empty(nbytes // 4 + 64, dtype=self.torch.float32, device=self.dev)
            self.ws_bytes = nbytes

    def op(self, name, fn):
        if self.mark is None:
            fn()
            return
        e0, e1 = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        fn()
        e1.record(self.stream)
        self.mark.append((name, e0, e1))

    def conv_fwd(self, d, x, w, b, y):
        fws, fnb = self.fws[id(d)]
        self.hc.check(self.hc.hc_conv2d_fwd(d, x, w, b, y, fws, fnb, self.stream), "fwd")

    def conv_bwd(self, d, x, w, gy, gx, gw, gb):
        # reads x's operand copy from the forward workspace (where the algorithm keeps one)
        fws, fnb = self.fws[id(d)]
        self.hc.check(self.hc.hc_conv2d_bwd_reuse(d, x, w, gy, gx, gw, gb, None, None, self.ws, self.ws_bytes, fws,
                                                  fnb, self.stream), "bwd")

    def conv_bwd_residual(self, d, x, w, gy, res, gx, gw, gb):
        """Backward whose grad_input also receives res, the gradient along a skip connection."""
        self.hc.check(self.hc.hc_conv2d_bwd_residual(d, x, w, gy, res, gx, gw, gb, ws=self.ws, ws_bytes=self.ws_bytes,
                                                     stream=self.stream), "bwd residual")

    def conv_fwd_gelu(self, d, x, w, b, y):
        """The conv of GELU(x), GELU applied as x's operand pieces are made."""
        fws, fnb = self.fws[id(d)]
        self.hc.check(self.hc.hc_conv2d_fwd_act(d, x, w, b, y, fws, fnb, self.stream, act=self.hc.HC_ACT_GELU_INPUT),
                      "fwd gelu")

    def conv_bwd_gelu(self, d, x, w, gy, gx, gw, gb):
        """Backward of conv_fwd_gelu: gx is the gradient with respect to GELU(x)."""
        fws, fnb = self.fws[id(d)]
        self.hc.check(self.hc.hc_conv2d_bwd_act(d, x, w, gy, gx, gw, gb, None, None, self.ws, self.ws_bytes, fws, fnb,
                                                self.stream, act=self.hc.HC_ACT_GELU_INPUT), "bwd gelu in")

    def conv_bwd_gelu_out(self, d, x, w, gy, y_pre, gx, gw, gb):
        """Backward of a conv whose output y_pre feeds a GELU; gy is the gradient of GELU(y_pre)."""
        fws, fnb = self.fws[id(d)]
        self.hc.check(self.hc.hc_conv2d_bwd_act(d, x, w, gy, gx, gw, gb, None, None, self.ws, self.ws_bytes, fws, fnb,
                                                self.stream, act=self.hc.HC_ACT_GELU_OUTPUT, y_pre=y_pre),
                      "bwd gelu out")

    def conv_ws(self, d):
        """Allocates the conv's forward workspace; returns the bytes its backward
        pass needs from the shared workspace."""
        st, a = self.hc.hc_conv2d_workspace_size(d, 0)
        self.hc.check(st, "ws")
        st, b = self.hc.hc_conv2d_workspace_size(d, 2)
        self.hc.check(st, "ws")
        self.fws[id(d)] = (self.torch.empty(max(a, 16) // 4 + 64, dtype=self.torch.float32, device=self.dev), a)
        return max(b, 16)


class ConvWorkload:
    """A single sharded convolution, forward + backward."""

    def __init__(self, name, cfg, gen, unit, desc):
        self.name, self.cfg, self.gen, self.unit, self.desc = name, cfg, gen, unit, desc
        self.E = cfg["N"] * cfg["C_in"] * cfg["H"] * cfg["W"]
        self.flops = 3 * conv_flops(cfg)
        self.bytes = 5 * 4 * self.E
        self.dense = cfg["groups"] == 1

    def describe(self):
        c = self.cfg
        return {"workload": self.desc, "shape": [c["N"], c["C_in"], c["H"], c["W"]], "kernel": [c["kh"], c["kw"]],
                "padding": c["padding"], "groups": c["groups"], "num_shards": c["num_shards"],
                "num_shards_h": c.get("num_shards_h", 1),
                "l2": "inputs (470 MB each) larger than L2; no flush" if self.name != "config1" else
                      "inputs L2-resident (8 KB); launch-latency bound, no flush"}

    def setup(self, R):
        self.R = R
        self.host = self.gen()
        x, w, b, gy = self.host
        self.x, self.w, self.b, self.gy = (R.upload(a) for a in (x, w, b, gy))
        self.y, self.gx = R.torch.empty_like(self.x), R.torch.empty_like(self.x)
        self.gw, self.gb = R.torch.empty_like(self.w), R.torch.empty_like(self.b)
        self.d = R.hc.desc(self.cfg)
        R.reserve(R.conv_ws(self.d))

    def fwd(self):
        self.R.op("conv_fwd", lambda: self.R.conv_fwd(self.d, self.x, self.w, self.b, self.y))

    def bwd(self):
        self.R.op("conv_bwd", lambda: self.R.conv_bwd(self.d, self.x, self.w, self.gy, self.gx, self.gw, self.gb))

    def make_graph(self):
        """Capture this workload's fwd + bwd step as one CUDA graph; returns (handle, kernels in it)."""
        R = self.R
        n0 = R.hc.hc_launch_count()
        fws, fnb = R.fws[id(self.d)]
        st, g = R.hc.hc_conv2d_step_graph_create(self.d, self.x, self.w, self.b, self.y, self.gy, self.gx, self.gw,
                                                 self.gb, fws, fnb, R.ws, R.ws_bytes)
        R.hc.check(st, "graph create")
        return g, R.hc.hc_launch_count() - n0

    def host_io(self):
        t = self.R.torch
        x, w, b, gy = self.host
        self.h_in = [(d, t.from_numpy(h).pin_memory()) for d, h in ((self.x, x), (self.w, w), (self.b, b), (self.gy, gy))]
        self.h_out = [(o, t.empty_like(o, device="cpu").pin_memory()) for o in (self.y, self.gx, self.gw, self.gb)]

    def kernel_work(self):
        """Algorithmic work per step of each compute kernel, by trace name:
        (bound, amount, HBM bytes or None)."""
        F = conv_flops(self.cfg)
        if self.name == "dw7":
            return {"dw_fwd_kernel": ("alu", F, 8 * self.E), "dw_bwd_kernel": ("alu", 2 * F, 12 * self.E)}
        if self.name == "dense5x5":
            # conv passes on 3xTF32; the weight gradient on bf16 pieces (six products)
            return {"tc_conv_kernel 3xTF32 conv pass": ("tensor_tf32", 2 * F, None),
                    "tc_conv_kernel bf16x6 weight-gradient pass": ("tensor", F, None)}
        return {}

    def oracle_sample(self, orc):
        """One bounded sample of this workload for the oracle, fwd + bwd: config1
        whole; the others one image and a band of rows (the same kernel, channels
        and width).  Returns (run: the oracle calls on inputs made here, units of
        the metric one run does, description)."""
        from spatially_sharded_cnn_gb300 import synth
        c = dict(self.cfg)
        c.pop("num_shards_h", None)
        if self.name != "config1":
            c["N"], c["H"] = 1, (32 if self.name == "dw7" else 4)
        x = synth.normal((c["N"], c["C_in"], c["H"], c["W"]), 1.0, 0, 1)
        w = synth.normal((c["C_out"], c["C_in"] // c["groups"], c["kh"], c["kw"]), 0.02, 0, 2)
        b = synth.normal((c["C_out"],), 0.01, 0, 3)
        Ho = (c["H"] + 2 * c["padding"] - c["kh"]) // c["stride"] + 1
        Wo = (c["W"] + 2 * c["padding"] - c["kw"]) // c["stride"] + 1
        gy = synth.normal((c["N"], c["C_out"], Ho, Wo), 1.0, 0, 4)

        def run():
            orc.conv2d_fwd(c, x, w, b)
            orc.conv2d_bwd_input(c, w, gy)
            orc.conv2d_bwd_weight(c, x, gy)
            orc.conv2d_bwd_bias(c, gy)
        units = 5 * 4 * x.size / 1e9 if not self.dense else 3 * conv_flops(c) / 1e12
        return run, units, (f"{c['N']} image(s) x {c['H']} of {self.cfg['H']} rows of the {self.desc.split(', x ')[0]} "
                       f"workload (shape {[c['N'], c['C_in'], c['H'], c['W']]}), fwd+bwd")

    def value(self, ms):
        return self.flops / (ms * 1e-3) / 1e12 if self.dense else self.bytes / (ms * 1e-3) / 1e9

    def roofline(self, ops_ms, peaks, sms):
        if self.name == "config1":  # a few kernels of microseconds: launch latency, not a unit, bounds it
            alu = alu_peak(peaks, sms)
            ms = sum(ops_ms.values())
            a = self.flops / (ms * 1e-3) / 1e12
            return {"bound": "alu", "kernel": "direct conv kernels (launch-latency bound)", "achieved": a, "peak": alu,
                    "unit": "TFLOP/s", "frac": a / alu, "traffic": None,
                    "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                    "ms_per_launch": ms}
        if "step_graph" in ops_ms:  # graph replay: one timed op, the whole step
            ms = ops_ms["step_graph"]
            if self.dense:
                peak, a = tc_peak(peaks), self.flops / (ms * 1e-3) / 1e12
                return {"bound": "tensor", "kernel": "whole fwd+bwd step (graph replay)", "achieved": a, "peak": peak,
                        "unit": "TFLOP/s (fp32-equivalent, 3xTF32)", "frac": a / peak, "traffic": None,
                        "peak_source": f"measured bf16 {peaks['bf16']:.0f} TFLOP/s x 1.1/2.25 (tf32) / 3",
                        "ms_per_launch": ms}
            alu = alu_peak(peaks, sms)
            a = 3 * conv_flops(self.cfg) / (ms * 1e-3) / 1e12
            return {"bound": "alu", "kernel": "whole fwd+bwd step (graph replay)", "achieved": a, "peak": alu,
                    "unit": "TFLOP/s", "frac": a / alu, "traffic": None,
                    "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                    "ms_per_launch": ms}
        return None  # the dominant traced kernel's roofline (kernel_roofline) applies


def gen_dw7(N=7, seed=0):
    from spatially_sharded_cnn_gb300 import synth
    x = synth.normal((N, 256, 128, 512), 1.0, seed, 1)
    w = synth.trunc_normal((256, 1, 7, 7), 0.02, seed, 2)
    b = np.zeros((256,), np.float32)
    gy = synth.normal((N, 256, 128, 512), 1.0, seed, 4)
    return x, w, b, gy


def gen_config1(seed=0):
    """The small dense case: x U[-1,1], w N(0,0.1), b N(0,0.1), gy N(0,1)."""
    from spatially_sharded_cnn_gb300 import synth
    x = synth.uniform((1, 4, 16, 32), -1.0, 1.0, seed, 1)
    w = synth.normal((4, 4, 5, 5), 0.1, seed, 2)
    b = synth.normal((4,), 0.1, seed, 3)
    gy = synth.normal((1, 4, 16, 32), 1.0, seed, 4)
    return x, w, b, gy


def gen_dense5x5(N=7, seed=0):
    from spatially_sharded_cnn_gb300 import synth
    x = synth.normal((N, 128, 128, 1024), 1.0, seed, 1)
    w = synth.kaiming_normal((128, 128, 5, 5), 128 * 25, seed, 2)
    b = synth.normal((128,), 0.01, seed, 3)
    gy = synth.normal((N, 128, 128, 1024), 1.0, seed, 4)
    return x, w, b, gy


class BlockWorkload:
    """ConvNeXt-XL stage-1 block on the stem output of a (7,3,512,4096) image, 8 W-shards."""

    unit = "TFLOP/s"

    def __init__(self, drop_path=0.0, N=7):
        S = 8
        self.N, self.S = N, S
        self.drop_path, self.steps_drawn = float(drop_path), 0
        self.stem = conv_cfg(N, 3, 512, 4096, 256, 4, 4, 0, 1, S)
        self.dw = conv_cfg(N, 256, 128, 1024, 256, 7, 1, 3, 256, S)
        self.pw1 = conv_cfg(N, 256, 128, 1024, 1024, 1, 1, 0, 1, S)
        self.pw2 = conv_cfg(N, 1024, 128, 1024, 256, 1, 1, 0, 1, S)
        self.HW = 128 * 1024
        fwd = sum(conv_flops(c) for c in (self.stem, self.dw, self.pw1, self.pw2))
        # backward: grad_input and grad_weight of dw / pw1 / pw2, grad_weight of the stem
        bwd = conv_flops(self.stem) + 2 * sum(conv_flops(c) for c in (self.dw, self.pw1, self.pw2))
        self.flops = fwd + bwd

    def describe(self):
        return {"workload": "ConvNeXt-XL stage-1 block fwd+bwd on the stem output of a (7,3,512,4096) U[0,1] image: "
                            "4x4/s4 stem 3->256, depthwise 7x7, LayerNorm(C), 1x1 256->1024, GELU, 1x1 1024->256, "
                            "layer scale 1e-6 + residual" + (f", DropPath {self.drop_path}" if self.drop_path else "") +
                            f"; fp32; 8 W-shards" + (f"; batch {self.N}" if self.N != 7 else ""),
                "shape": [self.N, 3, 512, 4096], "num_shards": 8,
                "l2": "activations (0.13-0.54 GB per image) larger than L2; no flush"}

    def setup(self, R):
        from spatially_sharded_cnn_gb300 import synth
        self.R = R
        hc, t = R.hc, R.torch
        N, HW = self.N, self.HW
        self.h_img = synth.uniform((N, 3, 512, 4096), 0.0, 1.0, 0, 1)
        self.h_gy = synth.normal((N, 256, 128, 1024), 1.0, 0, 9)
        self.img, self.gy = R.upload(self.h_img), R.upload(self.h_gy)
        self.w_stem = R.upload(synth.trunc_normal((256, 3, 4, 4), 0.02, 0, 2))
        self.w_dw = R.upload(synth.trunc_normal((256, 1, 7, 7), 0.02, 0, 3))
        self.w1 = R.upload(synth.trunc_normal((1024, 256, 1, 1), 0.02, 0, 4))
        self.w2 = R.upload(synth.trunc_normal((256, 1024, 1, 1), 0.02, 0, 5))
        self.b256, self.b1024 = t.zeros(256, device=R.dev), t.zeros(1024, device=R.dev)
        self.ln_g, self.ln_b = t.ones(256, device=R.dev), t.zeros(256, device=R.dev)
        self.ls_g = t.full((256,), 1e-6, device=R.dev)
        self.mask = t.empty(N, device=R.dev) if self.drop_path else None
        a256, a1024 = (N, 256, 128, 1024), (N, 1024, 128, 1024)
        self.s, self.dwo, self.ln, self.b2, self.out = (R.empty(a256) for _ in range(5))
        self.mean, self.rstd = R.empty((N, HW)), R.empty((N, HW))
        self.h = R.empty(a1024)  # the 1x1 256->1024 output; GELU(h) is never stored
        self.g_b2, self.g_l, self.g_d, self.g_s = (R.empty(a256) for _ in range(4))
        self.g_a = R.empty(a1024)
        self.gw_stem, self.gb_stem = t.empty_like(self.w_stem), t.empty(256, device=R.dev)
        self.gw_dw, self.gb_dw = t.empty_like(self.w_dw), t.empty(256, device=R.dev)
        self.gw1, self.gb1 = t.empty_like(self.w1), t.empty(1024, device=R.dev)
        self.gw2, self.gb2 = t.empty_like(self.w2), t.empty(256, device=R.dev)
        self.g_lng, self.g_lnb, self.g_ls = (t.empty(256, device=R.dev) for _ in range(3))
        self.d = {k: hc.desc(getattr(self, k)) for k in ("stem", "dw", "pw1", "pw2")}
        st, pwb = hc.hc_pointwise_workspace_size(N, 1024, HW)
        hc.check(st)
        R.reserve(max([R.conv_ws(d) for d in self.d.values()] + [pwb]))

    def fwd(self):
        R, hc, N, HW = self.R, self.R.hc, self.N, self.HW
        R.op("stem_fwd", lambda: R.conv_fwd(self.d["stem"], self.img, self.w_stem, self.b256, self.s))
        R.op("dw_fwd", lambda: R.conv_fwd(self.d["dw"], self.s, self.w_dw, self.b256, self.dwo))
        R.op("ln_fwd", lambda: hc.check(hc.hc_layernorm_c_fwd(N, 256, HW, self.dwo, self.ln_g, self.ln_b, 1e-6, self.ln,
                                                              self.mean, self.rstd, R.stream)))
        R.op("pw1_fwd", lambda: R.conv_fwd(self.d["pw1"], self.ln, self.w1, self.b1024, self.h))
        # GELU goes into the 1x1 1024->256's operand split (hc_conv2d_fwd_act)
        R.op("gelu_pw2_fwd", lambda: R.conv_fwd_gelu(self.d["pw2"], self.h, self.w2, self.b256, self.b2))
        if self.drop_path:  # a fresh per-sample draw each step: offset = samples drawn so far
            R.op("drop_path_mask", lambda: hc.check(hc.hc_drop_path_mask(N, self.drop_path, 2024, self.steps_drawn * N,
                                                                         self.mask, R.stream)))
            self.steps_drawn += 1
        R.op("ls_fwd", lambda: hc.check(hc.hc_layerscale_droppath_fwd(N, 256, HW, self.s, self.b2, self.ls_g, self.mask,
                                                                      self.out, R.stream)))

    def bwd(self):
        R, hc, N, HW = self.R, self.R.hc, self.N, self.HW
        R.op("ls_bwd", lambda: hc.check(hc.hc_layerscale_droppath_bwd(N, 256, HW, self.b2, self.ls_g, self.mask,
                                                                      self.gy, self.g_b2, self.g_ls, R.ws, R.ws_bytes,
                                                                      R.stream)))
        # the 1x1 1024->256's grad_input is the gradient with respect to GELU(h); the
        # 1x1 256->1024's backward runs on it times GELU'(h), formed as it is read
        R.op("pw2_bwd", lambda: R.conv_bwd_gelu(self.d["pw2"], self.h, self.w2, self.g_b2, self.g_a, self.gw2,
                                                self.gb2))
        R.op("gelu_pw1_bwd", lambda: R.conv_bwd_gelu_out(self.d["pw1"], self.ln, self.w1, self.g_a, self.h, self.g_l,
                                                         self.gw1, self.gb1))
        R.op("ln_bwd", lambda: hc.check(hc.hc_layernorm_c_bwd(N, 256, HW, self.dwo, self.ln_g, self.mean, self.rstd,
                                                              self.g_l, self.g_d, self.g_lng, self.g_lnb, R.ws,
                                                              R.ws_bytes, R.stream)))
        # the depthwise conv's grad_input plus the residual's gradient gy, added in its epilogue
        R.op("dw_bwd", lambda: R.conv_bwd_residual(self.d["dw"], self.s, self.w_dw, self.g_d, self.gy, self.g_s,
                                                   self.gw_dw, self.gb_dw))
        R.op("stem_bwd", lambda: R.conv_bwd(self.d["stem"], self.img, self.w_stem, self.g_s, None, self.gw_stem,
                                            self.gb_stem))

    def host_io(self):
        t = self.R.torch
        ins = (self.img, self.gy, self.w_stem, self.w_dw, self.w1, self.w2, self.b256, self.b1024, self.ln_g, self.ln_b,
               self.ls_g)
        self.h_in = [(d, d.cpu().pin_memory()) for d in ins]
        outs = (self.out, self.gw_stem, self.gb_stem, self.gw_dw, self.gw1, self.gw2, self.g_lng, self.g_lnb, self.g_ls)
        self.h_out = [(o, t.empty_like(o, device="cpu").pin_memory()) for o in outs]

    def kernel_work(self):
        """Algorithmic work per step of the compute kernels, by trace name: the
        bf16-piece GEMM passes (stem forward; 1x1 256->1024 and 1024->256 forward,
        grad_input and weight gradient), the depthwise stencil and the stem's
        weight gradient (FP32 reduction reading the image and grad_output once)."""
        st, dw, p1, p2 = (conv_flops(c) for c in (self.stem, self.dw, self.pw1, self.pw2))
        E = self.N * 256 * self.HW
        return {"tc_conv_kernel bf16x6 conv pass": ("tensor", st + 2 * p1 + 2 * p2, None),
                "tc_conv_kernel bf16x6 weight-gradient pass": ("tensor", p1 + p2, None),
                "dw_fwd_kernel": ("alu", dw, 8 * E), "dw_bwd_kernel": ("alu", 2 * dw, 16 * E),
                "patchify_wgrad_kernel": ("alu", st, self.stem_bytes())}

    def stem_bytes(self):
        """The stem's algorithmic HBM bytes: the image and the 256-channel stem
        output (written forward, grad_output read backward) once each."""
        return 4 * (self.N * 3 * 512 * 4096 + self.N * 256 * self.HW)

    def oracle_sample(self, orc):
        """The block's chain for the oracle, forward and backward, on one image
        and a band of 8 of its 512 input rows (2 rows of the stem output)."""
        from spatially_sharded_cnn_gb300 import synth
        f32 = lambda a: np.ascontiguousarray(a, np.float32)
        img = synth.uniform((1, 3, 8, 4096), 0.0, 1.0, 0, 1)
        cs = dict(self.stem, N=1, H=8)
        cd = dict(self.dw, N=1, H=2)
        c1 = dict(self.pw1, N=1, H=2)
        c2 = dict(self.pw2, N=1, H=2)
        for c in (cs, cd, c1, c2):
            c.pop("num_shards_h", None)
        ws = synth.trunc_normal((256, 3, 4, 4), 0.02, 0, 2)
        wd = synth.trunc_normal((256, 1, 7, 7), 0.02, 0, 3)
        w1 = synth.trunc_normal((1024, 256, 1, 1), 0.02, 0, 4)
        w2 = synth.trunc_normal((256, 1024, 1, 1), 0.02, 0, 5)
        z256, z1024 = np.zeros(256, np.float32), np.zeros(1024, np.float32)
        g, bt, ls = np.ones(256), np.zeros(256), np.full(256, 1e-6)
        gy = synth.normal((1, 256, 2, 1024), 1.0, 0, 9)
        flops = sum(conv_flops(c) for c in (cs, cd, c1, c2)) + conv_flops(cs) + 2 * sum(conv_flops(c) for c in (cd, c1, c2))
        return lambda: self._oracle_chain(orc, img, ws, wd, w1, w2, z256, z1024, g, bt, ls, gy, cs, cd, c1, c2), \
            flops / 1e12, ("the block's chain (stem, depthwise, LayerNorm, 1x1, GELU, 1x1, layer scale + residual), "
                           "fwd+bwd, on 1 image x 8 of 512 input rows of the (7,3,512,4096) batch")

    @staticmethod
    def _oracle_chain(orc, img, ws, wd, w1, w2, z256, z1024, g, bt, ls, gy, cs, cd, c1, c2):
        f32 = lambda a: np.ascontiguousarray(a, np.float32)
        s = f32(orc.conv2d_fwd(cs, img, ws, z256))
        d = f32(orc.conv2d_fwd(cd, s, wd, z256))
        ln, _, _ = orc.layernorm_c_fwd(d, g, bt, 1e-6)
        h = orc.conv2d_fwd(c1, f32(ln), w1, z1024)
        a = f32(orc.gelu_fwd(h))
        b2 = orc.conv2d_fwd(c2, a, w2, z256)
        orc.layerscale_residual_fwd(s, b2, ls)
        _, g_b2, _ = orc.layerscale_residual_bwd(b2, ls, gy)
        g_b2 = f32(g_b2)
        g_a = f32(orc.conv2d_bwd_input(c2, w2, g_b2))
        orc.conv2d_bwd_weight(c2, a, g_b2)
        orc.conv2d_bwd_bias(c2, g_b2)
        g_h = f32(orc.gelu_bwd(h, g_a))
        g_l = orc.conv2d_bwd_input(c1, w1, g_h)
        orc.conv2d_bwd_weight(c1, f32(ln), g_h)
        orc.conv2d_bwd_bias(c1, g_h)
        g_d, _, _ = orc.layernorm_c_bwd(d, g, g_l, 1e-6)
        g_d = f32(g_d)
        g_s = f32(orc.conv2d_bwd_input(cd, wd, g_d) + gy)
        orc.conv2d_bwd_weight(cd, s, g_d)
        orc.conv2d_bwd_bias(cd, g_d)
        orc.conv2d_bwd_weight(cs, img, g_s)
        orc.conv2d_bwd_bias(cs, g_s)

    def value(self, ms):
        return self.flops / (ms * 1e-3) / 1e12

    def op_work(self):
        """Each op's bound and algorithmic work: conv FLOPs (tensor: the bf16-piece
        GEMMs; alu: the depthwise stencil and the stem's weight gradient) or HBM
        bytes of the stem forward and the pointwise ops (E = elements of a
        256-channel activation)."""
        E = self.N * 256 * self.HW
        st, dw, p1, p2 = (conv_flops(c) for c in (self.stem, self.dw, self.pw1, self.pw2))
        # the stem: forward bound by its output write (48-deep K, 256 wide), backward
        # (weight and bias gradients only) by the FP32 reduction, HBM bytes beside
        return {"stem_fwd": ("hbm", self.stem_bytes()), "dw_fwd": ("alu", dw), "pw1_fwd": ("tensor", p1),
                "gelu_pw2_fwd": ("tensor", p2), "pw2_bwd": ("tensor", 2 * p2), "gelu_pw1_bwd": ("tensor", 2 * p1),
                "dw_bwd": ("alu", 2 * dw), "stem_bwd": ("alu", st, self.stem_bytes()),
                "ln_fwd": ("hbm", 8 * E + 8 * self.N * self.HW), "ln_bwd": ("hbm", 12 * E + 8 * self.N * self.HW),
                "ls_fwd": ("hbm", 12 * E), "ls_bwd": ("hbm", 12 * E)}

    def roofline(self, ops_ms, peaks, sms):
        return None  # the dominant traced kernel's roofline applies


class DwDownWorkload:
    """Depthwise 7x7 then 2x2/s2 downsample 256->512 on (7,256,128,2048), 8 W-shards."""

    unit = "TFLOP/s"

    def __init__(self, N=7):
        self.N = N
        self.dw = conv_cfg(N, 256, 128, 2048, 256, 7, 1, 3, 256, 8)
        self.down = conv_cfg(N, 256, 128, 2048, 512, 2, 2, 0, 1, 8)
        self.flops = 3 * (conv_flops(self.dw) + conv_flops(self.down))

    def describe(self):
        return {"workload": "depthwise 7x7 (p3, groups=C) then 2x2/s2 downsample 256->512 fwd+bwd on x "
                            f"({self.N},256,128,2048) fp32, 8 W-shards of width 256",
                "shape": [self.N, 256, 128, 2048], "num_shards": 8,
                "l2": "activations (0.27 GB per image) larger than L2; no flush"}

    def setup(self, R):
        from spatially_sharded_cnn_gb300 import synth
        self.R = R
        hc, t = R.hc, R.torch
        self.h_x = synth.normal((self.N, 256, 128, 2048), 1.0, 0, 1)
        self.h_gz = synth.normal((self.N, 512, 64, 1024), 1.0, 0, 9)
        self.x, self.gz = R.upload(self.h_x), R.upload(self.h_gz)
        self.w_dw = R.upload(synth.trunc_normal((256, 1, 7, 7), 0.02, 0, 2))
        self.w_dn = R.upload(synth.trunc_normal((512, 256, 2, 2), 0.02, 0, 3))
        self.b256, self.b512 = t.zeros(256, device=R.dev), t.zeros(512, device=R.dev)
        self.dwo, self.gd, self.gx = (t.empty_like(self.x) for _ in range(3))
        self.z = t.empty_like(self.gz)
        self.gw_dw, self.gb_dw = t.empty_like(self.w_dw), t.empty(256, device=R.dev)
        self.gw_dn, self.gb_dn = t.empty_like(self.w_dn), t.empty(512, device=R.dev)
        self.d = {k: hc.desc(getattr(self, k)) for k in ("dw", "down")}
        R.reserve(max(R.conv_ws(d) for d in self.d.values()))

    def fwd(self):
        R = self.R
        R.op("dw_fwd", lambda: R.conv_fwd(self.d["dw"], self.x, self.w_dw, self.b256, self.dwo))
        R.op("down_fwd", lambda: R.conv_fwd(self.d["down"], self.dwo, self.w_dn, self.b512, self.z))

    def bwd(self):
        R = self.R
        R.op("down_bwd", lambda: R.conv_bwd(self.d["down"], self.dwo, self.w_dn, self.gz, self.gd, self.gw_dn,
                                            self.gb_dn))
        R.op("dw_bwd", lambda: R.conv_bwd(self.d["dw"], self.x, self.w_dw, self.gd, self.gx, self.gw_dw, self.gb_dw))

    def host_io(self):
        t = self.R.torch
        ins = (self.x, self.gz, self.w_dw, self.w_dn, self.b256, self.b512)
        self.h_in = [(d, d.cpu().pin_memory()) for d in ins]
        outs = (self.z, self.gx, self.gw_dw, self.gb_dw, self.gw_dn, self.gb_dn)
        self.h_out = [(o, t.empty_like(o, device="cpu").pin_memory()) for o in outs]

    def kernel_work(self):
        """Algorithmic work per step by trace name: the depthwise stencil (FP32
        ALU) and the downsample's bf16-piece GEMM passes."""
        dw, dn = conv_flops(self.dw), conv_flops(self.down)
        E = self.N * 256 * 128 * 2048
        return {"dw_fwd_kernel": ("alu", dw, 8 * E), "dw_bwd_kernel": ("alu", 2 * dw, 12 * E),
                "tc_conv_kernel bf16x6 conv pass": ("tensor", 2 * dn, None),
                "tc_conv_kernel bf16x6 weight-gradient pass": ("tensor", dn, None)}

    def oracle_sample(self, orc):
        """Depthwise then downsample for the oracle, forward and backward, on one
        image and 4 of its 128 rows."""
        from spatially_sharded_cnn_gb300 import synth
        f32 = lambda a: np.ascontiguousarray(a, np.float32)
        cd, cn = dict(self.dw, N=1, H=4), dict(self.down, N=1, H=4)
        x = synth.normal((1, 256, 4, 2048), 1.0, 0, 1)
        wd = synth.trunc_normal((256, 1, 7, 7), 0.02, 0, 2)
        wn = synth.trunc_normal((512, 256, 2, 2), 0.02, 0, 3)
        z = np.zeros(512, np.float32)
        gz = synth.normal((1, 512, 2, 1024), 1.0, 0, 9)

        def run():
            d = f32(orc.conv2d_fwd(cd, x, wd, z[:256]))
            orc.conv2d_fwd(cn, d, wn, z)
            gd = f32(orc.conv2d_bwd_input(cn, wn, gz))
            orc.conv2d_bwd_weight(cn, d, gz)
            orc.conv2d_bwd_bias(cn, gz)
            orc.conv2d_bwd_input(cd, wd, gd)
            orc.conv2d_bwd_weight(cd, x, gd)
            orc.conv2d_bwd_bias(cd, gd)
        return run, 3 * (conv_flops(cd) + conv_flops(cn)) / 1e12, \
            "depthwise 7x7 + 2x2/s2 downsample, fwd+bwd, on 1 image x 4 of 128 rows of the (7,256,128,2048) batch"

    def value(self, ms):
        return self.flops / (ms * 1e-3) / 1e12

    def op_work(self):
        """Each op's bound and FLOPs: the depthwise stencil on the FP32 ALU, the
        downsample on the bf16-piece GEMM (backward: grad_input and grad_weight)."""
        dw, dn = conv_flops(self.dw), conv_flops(self.down)
        return {"dw_fwd": ("alu", dw), "dw_bwd": ("alu", 2 * dw), "down_fwd": ("tensor", dn),
                "down_bwd": ("tensor", 2 * dn)}

    def roofline(self, ops_ms, peaks, sms):
        return None  # the dominant traced kernel's roofline applies


def make_workload(name, batch=None, drop_path=0.0, shards_h=1):
    """batch overrides N of every workload but config1 (smaller cases for profiling);
    shards_h > 1 also splits their rows (a row x column shard grid)."""
    N = batch or 7
    wl = _make_workload(name, N, drop_path)
    if shards_h > 1:
        if not isinstance(wl, ConvWorkload):
            raise SystemExit("--shards-h applies to the single-conv workloads")
        wl.cfg = dict(wl.cfg, num_shards_h=shards_h)
        wl.desc += f", {shards_h} H-shards (a {shards_h} x {wl.cfg['num_shards']} shard grid)"
    return wl


def _make_workload(name, N, drop_path):
    if name == "dw7":
        return ConvWorkload("dw7", conv_cfg(N, 256, 128, 512, 256, 7, 1, 3, 256, 4), lambda: gen_dw7(N), "GB/s",
                            f"depthwise 7x7 conv fwd+bwd, x ({N},256,128,512) fp32, 4 W-shards of width 128")
    if name == "dense5x5":
        return ConvWorkload("dense5x5", conv_cfg(N, 128, 128, 1024, 128, 5, 1, 2, 1, 4), lambda: gen_dense5x5(N),
                            "TFLOP/s", f"dense 5x5 conv 128->128 fwd+bwd, x ({N},128,128,1024) fp32 (3xTF32 tensor "
                            "cores), 4 W-shards of width 256")
    if name == "config1":
        return ConvWorkload("config1", conv_cfg(1, 4, 16, 32, 4, 5, 1, 2, 1, 4), gen_config1, "TFLOP/s",
                            "dense 5x5 conv 4->4 fwd+bwd, x (1,4,16,32) fp32, 4 W-shards of width 8")
    if name == "block":
        return BlockWorkload(drop_path, N)
    if name == "dwdown":
        return DwDownWorkload(N)
    raise ValueError(name)


WORKLOADS = ["dw7", "dense5x5", "block", "dwdown", "config1"]


# ---------------------------------------------------------------------------
# clocks during the timed region
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,utilization.gpu,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 10]
        sm, smax, busy, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
                util = float(r[4])
            except ValueError:
                continue
            for nm, val in zip(names, r[7:11]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
            if util > 0:
                busy.append(sm[-1])
        use = busy or sm
        return {"sm_mhz": float(np.median(use)) if use else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_busy": len(busy)}


# ---------------------------------------------------------------------------
def traffic_for(workload: str, kernel: str, src_file: str):
    """DRAM bytes per launch of `kernel` in the default-size `workload` from a
    committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload, {}).get(kernel)
    if not d:
        return None
    h = hashlib.sha256(open(src_file, "rb").read()).hexdigest()[:16]
    return d["bytes_per_launch"] if d.get("source_sha") == h else None


def oracle_sample(wl, max_seconds=20.0, reps_max=4):
    """The oracle as it stands, on this host's cores, on a bounded sample of the
    workload (its oracle_sample: one image and a band of rows; config1 whole),
    forward + backward, repeated while time remains (inputs made outside the
    timing).  Returns (the metric's rate on the sample, threads, description,
    seconds per repetition)."""
    import oracle
    orc = oracle.load()
    run, units, desc = wl.oracle_sample(orc)
    t0 = time.perf_counter()
    reps = 0
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 > max_seconds / 2 or reps >= reps_max:
            break
    dt = (time.perf_counter() - t0) / reps
    return units / dt, orc.num_threads(), f"{desc}, {reps} rep(s)", dt


def run_reference(args):
    """Reference arm: the CPU oracle timed on the host cores on the chosen
    workload's config and metric, each step one bounded sample of it."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import oracle
    wl = make_workload(args.workload, args.batch, args.drop_path, args.shards_h)
    orc = oracle.load()
    run, units, desc = wl.oracle_sample(orc)
    for _ in range(args.warmup):
        run()
    steps = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        steps.append(time.perf_counter() - t0)
    dt = float(np.mean(steps)) if steps else float("nan")
    v = units / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": wl.unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": wl.describe(),
            "cpu_baseline": {"value": v, "unit": wl.unit, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": desc + " per step"},
            "e2e": {"value": v, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_peaks(args):
    """--workload peaks: the measured ceilings the rooflines are read against.
    FP32 FMA loops (two loop-invariant operands, packed f32x2 pairs, three
    distinct registers), the depthwise stencil and weight-gradient correlation
    with their tiles in shared memory, and tcgen05 MMA loops (kind::tf32,
    kind::f16 bf16) -- each the best of 5 CUDA-event timed launches after one
    warm-up, with the SM clock sampled meanwhile."""
    import ctypes as C
    import torch
    from spatially_sharded_cnn_gb300 import build
    build.build()
    lib = C.CDLL(build.PEAKS_LIB)
    lib.hcp_out_floats.restype = C.c_longlong
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty(int(lib.hcp_out_floats()), device=dev)
    src = torch.rand(64, device=dev) * 0.5 + 0.25
    w = torch.randn(128 * 49, device=dev) * 0.02
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    P = lambda t: C.c_void_p(t.data_ptr())
    S = C.c_void_p(st.cuda_stream)

    def best(launch):
        fl = C.c_double(0)
        assert launch(C.byref(fl)) == 0
        torch.cuda.synchronize()
        ms = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            assert launch(C.byref(fl)) == 0
            e1.record(st)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return fl.value / (min(ms) * 1e-3) / 1e12, min(ms)

    clocks = ClockSampler(0)
    clocks.start()
    res = {}
    for kind, name in ((0, "ffma_two_invariant_operands"), (1, "ffma2_packed_pairs"), (2, "ffma_three_registers")):
        tf, ms = best(lambda fl: lib.hcp_fp32_loop(kind, 4000, 8, P(out), P(src), S, fl))
        res[name] = {"tflops": tf, "ms": ms}
    for kind, name in ((0, "depthwise7x7_stencil_smem"), (1, "depthwise7x7_weight_correlation_smem")):
        tf, ms = best(lambda fl: lib.hcp_stencil(kind, 1000, P(w), P(out), S, fl))
        res[name] = {"tflops": tf, "ms": ms}
    for kind, name in ((0, "tcgen05_tf32_m128n256k8"), (1, "tcgen05_bf16_m128n256k16"),
                       (2, "tcgen05_tf32_m128n16k8_2cta_per_sm")):
        tf, ms = best(lambda fl: lib.hcp_mma(kind, 20000, C.cast(P(status), C.POINTER(C.c_int)), S, fl))
        res[name] = {"tflops": tf, "ms": ms}
        if kind == 2:  # time per MMA per SM: the floor a narrow (N <= 32) MMA pays
            res[name]["ns_per_mma_per_sm"] = ms * 1e6 / (20000 * 2)
    clk = clocks.stop()
    if int(status.item()):
        raise SystemExit("an MMA loop CTA gave up waiting for its MMAs")
    peaks = load_peaks()
    line = {"workload": "peaks", "sms": sms, "unit": "TFLOP/s", "results": res,
            "fp32_derived_peak": alu_peak(peaks, sms), "clocks": clk,
            "note": "FP32 derived peak = SMs x 128 lanes x 2 x max SM clock; tensor rates per MMA loop of one CTA "
                    "per SM (M 128, N 256, operands zero, from shared memory); the N 16 loop runs two CTAs per SM "
                    "and gives the tensor pipe's time per narrow MMA"}
    print(json.dumps(line), flush=True)
    return 0


def run_exchange(args):
    """--exchange (N ranks under torchrun): the pages' multi-device form of the
    depthwise workload.  Rank r holds column block r (N,256,128,512) of an
    (N,256,128,512*ranks) image in the halo-padded layout, exchanges its edge
    columns with its neighbours (NCCL on device tensors when every rank has a
    device of its own; else gloo through host memory -- ranks that share a
    device run independent kernels, none waits on another) while its interior
    column tiles run, then its edge tiles; the _Partial weight and bias
    gradients are gathered and summed in rank order on every rank
    (spatially_sharded_cnn_gb300.exchange).  Weak scaling: value = the
    algorithmic bytes of all ranks (20 B per element of a block) / the slowest
    rank's step time.  --check compares every rank's block with the one-device
    call on the whole image: forward and grad_input bit for bit, weight and
    bias gradients within 1e-5 (the rank-order sum splits the partials at other
    points than the shard-order sum)."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world < 2:
        raise SystemExit("--exchange needs two or more ranks (torchrun)")
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    ndev = torch.cuda.device_count()
    backend = "nccl" if ndev >= world else "gloo"
    torch.cuda.set_device(local % ndev)
    dev = torch.device("cuda", local % ndev)
    if backend == "nccl":
        dist.init_process_group("nccl", device_id=dev)
    else:
        dist.init_process_group("gloo")
    from spatially_sharded_cnn_gb300 import hc
    from spatially_sharded_cnn_gb300.exchange import RankConv, padded_shape, HALO
    N, C, H, Wl, K = (args.batch or 7), 256, 128, 512, 7
    cfg = dict(N=N, C_in=C, H=H, W=Wl * world, C_out=C, kh=K, kw=K, stride=1, padding=3, groups=C,
               num_shards=world)
    d = hc.desc(cfg)
    conv = RankConv(cfg)
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)  # this rank's block of the synthetic image and of grad_output
    x_pad = torch.zeros(padded_shape(cfg), device=dev)
    gy_pad = torch.zeros(padded_shape(cfg), device=dev)
    x_pad[..., HALO:HALO + Wl] = torch.randn((N, C, H, Wl), generator=g, device=dev)
    gy_pad[..., HALO:HALO + Wl] = torch.randn((N, C, H, Wl), generator=g, device=dev)
    gw0 = torch.Generator(device=dev)
    gw0.manual_seed(7)  # replicated weights: the same on every rank
    w = torch.randn((C, 1, K, K), generator=gw0, device=dev) * 0.02
    b = torch.randn((C,), generator=gw0, device=dev) * 0.01
    y = torch.empty((N, C, H, Wl), device=dev)
    gx = torch.empty_like(y)
    gwt, gbt = torch.empty_like(w), torch.empty_like(b)
    st, nb = hc.hc_conv2d_workspace_size_rank(d)
    hc.check(st, "rank workspace")
    ws = torch.empty(nb // 4 + 64, device=dev)

    def step():
        conv.forward(x_pad, w, b, y, stream)
        conv.backward(x_pad, w, gy_pad, gx, gwt, gbt, ws, nb, stream)

    def slowest(ms):
        t = torch.tensor([ms], dtype=torch.float64, device=dev if backend == "nccl" else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    for _ in range(args.warmup):
        step()
    hc.check(hc.hc_sync_check(stream), "warmup")
    clocks = ClockSampler(local % ndev)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    n0 = hc.hc_launch_count()
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3
    dist.barrier()
    launches = hc.hc_launch_count() - n0
    clk = clocks.stop()
    hc.check(hc.hc_sync_check(stream), "timed region")
    # the exchange waits on the host (gloo) or in NCCL's streams, so a rank's step is
    # its wall time; the device events give the same on the NCCL path
    ms_step = slowest(max(e0.elapsed_time(e1), wall_ms) / args.steps)
    E = N * C * H * Wl
    value = world * 20.0 * E / (ms_step * 1e-3) / 1e9
    check = None
    if args.check:
        def gather(t):  # every rank's block, concatenated along W on every rank
            part = t.contiguous().to("cpu")
            parts = [torch.empty_like(part) for _ in range(world)]
            dist.all_gather(parts, part)
            return torch.cat(parts, dim=3).to(dev)
        xf, gyf = gather(x_pad[..., HALO:HALO + Wl]), gather(gy_pad[..., HALO:HALO + Wl])
        yf, gxf = gather(y), gather(gx)
        y1, gx1 = torch.empty_like(yf), torch.empty_like(gxf)
        gw1, gb1 = torch.empty_like(w), torch.empty_like(b)
        st1, nb1 = hc.hc_conv2d_workspace_size(d, 1)
        hc.check(st1, "workspace")
        ws1 = torch.empty(nb1 // 4 + 64, device=dev)
        hc.check(hc.hc_conv2d_fwd(d, xf, w, b, y1, None, 0, stream), "one-device fwd")
        hc.check(hc.hc_conv2d_bwd(d, xf, w, gyf, gx1, gw1, gb1, None, None, ws1, nb1, stream), "one-device bwd")
        hc.check(hc.hc_sync_check(stream), "check")
        nw = lambda a, r: float((a - r).abs().max() / r.abs().max())
        check = {"y_bit_identical": bool(torch.equal(yf, y1)), "gx_bit_identical": bool(torch.equal(gxf, gx1)),
                 "gw_normwise": nw(gwt, gw1), "gb_normwise": nw(gbt, gb1)}
    if rank == 0:
        peaks = load_peaks()
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": min(world, ndev), "ranks": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": f"depthwise 7x7 p3 groups=C fwd+bwd, {world} ranks each holding one column "
                                       f"block ({N},{C},{H},{Wl}) of a ({N},{C},{H},{Wl * world}) image; halo "
                                       f"exchange over {backend} with the interior tiles during the transfer; "
                                       "partials gathered and summed in rank order",
                           "exchange": backend, "shape_per_rank": [N, C, H, Wl],
                           "l2": "inputs (470 MB each per rank at N = 7) larger than L2; no flush"},
                "hbm_frac": value / min(world, ndev) / peaks["hbm"], "e2e": None,
                "e2e_note": "device-resident inputs only in this mode",
                "gpu_launches": launches, "clocks": clk}
        if check is not None:
            line["check"] = check
        print(json.dumps(line), flush=True)
    dist.barrier()
    dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="end-to-end steps (two buffer sets in turn: more steps amortise the first copy-in and the last copy-out)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=WORKLOADS + ["peaks"], default="dw7")
    ap.add_argument("--shards-h", type=int, default=1,
                    help="single-conv workloads: also split the rows into this many shards")
    ap.add_argument("--drop-path", type=float, default=0.0,
                    help="block workload: DropPath probability (per-sample, shard-consistent draw each step)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each fwd+bwd step from one captured CUDA graph (single-conv workloads)")
    ap.add_argument("--batch", type=int, default=None, help="batch size of every workload but config1 (default 7)")
    ap.add_argument("--exchange", action="store_true",
                    help="with N ranks under torchrun: the depthwise workload W-sharded across the ranks, halo "
                         "exchange and rank-order partial sums (default: N independent replicas)")
    ap.add_argument("--check", action="store_true",
                    help="--exchange: compare every rank's block with the one-device call on the whole image")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.workload == "peaks":
        return run_peaks(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.exchange:
        return run_exchange(args)
    wl = make_workload(args.workload, args.batch, args.drop_path, args.shards_h)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    from spatially_sharded_cnn_gb300 import hc

    peaks = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    R = Runner(hc, torch, dev, stream)
    wl.setup(R)

    graph, graph_kernels = None, 0
    if args.graph:
        if not hasattr(wl, "make_graph"):
            raise SystemExit("--graph applies to the single-conv workloads")
        graph, graph_kernels = wl.make_graph()

    def step():
        if graph is not None:
            R.op("step_graph", lambda: hc.check(hc.hc_step_graph_launch(graph, stream), "graph launch"))
            return
        wl.fwd()
        wl.bwd()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    hc.check(hc.hc_sync_check(stream), "warmup")

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    marks = []
    trace = graph is None and args.workload != "config1"  # config1's few-microsecond kernels: no per-launch events
    # per-op events inside the timed region: the multi-op workloads' phases (several kernels
    # each), config 1 and graph replays; a traced single conv's two ops are its kernels,
    # which the library's own trace times, so no extra events go into its step
    R.mark = None if trace and isinstance(wl, ConvWorkload) else marks
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    n0 = hc.hc_launch_count()
    if trace:
        hc.hc_trace_collect()  # drop anything recorded before
        hc.hc_trace_enable(True)
    start.record(stream)
    for _ in range(K):
        step()
    end.record(stream)
    barrier()
    R.mark = None
    ktable = None
    if trace:
        hc.hc_trace_enable(False)
        st_tr, tr = hc.hc_trace_collect()
        hc.check(st_tr, "trace collect")
        ktable = kernel_table(tr, K)
    launches = hc.hc_launch_count() - n0 + K * graph_kernels  # a replay runs the captured kernels
    clk = clocks.stop()
    hc.check(hc.hc_sync_check(stream), "timed region")
    elapsed_ms = start.elapsed_time(end)
    ops = {}
    for name, e0, e1 in marks:
        ops.setdefault(name, []).append(e0.elapsed_time(e1))
    ops_ms = {k: float(np.mean(v)) for k, v in ops.items()}
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_step = elapsed_ms / K
    value = world * wl.value(ms_step)

    # end to end: host buffers, every step's inputs copied in from pinned host
    # memory and its outputs copied out, inside the timed region.  Three streams
    # ordered by events and two sets of device input / output buffers used in
    # turn: step k+1's inputs upload while step k computes and step k-1's
    # outputs download (both copy directions and the kernels run at once).  A
    # set's inputs are overwritten only after the step two back has used them,
    # and its outputs only after they have been copied out.  (A captured graph
    # keeps its one set of buffers.)
    wl.host_io()
    E2 = max(1, args.e2e_steps)
    sets = [{}]  # per set: attribute name -> device tensor (set 0: the workload's own)
    names = {id(v): k for k, v in vars(wl).items() if isinstance(v, torch.Tensor)}
    io = [names[id(d_t)] for d_t, _ in wl.h_in + wl.h_out]
    sets[0] = {a: getattr(wl, a) for a in io}
    if graph is None and E2 > 1:
        sets.append({a: torch.empty_like(t) for a, t in sets[0].items()})
    h_in = [(names[id(d_t)], h_t) for d_t, h_t in wl.h_in]
    h_out = [(names[id(d_t)], h_t) for d_t, h_t in wl.h_out]
    barrier()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    done_in, done_step, done_out = [ev() for _ in range(E2)], [ev() for _ in range(E2)], [ev() for _ in range(E2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_in.wait_stream(stream)
    e0.record(s_in)
    B = len(sets)
    for k in range(E2):
        cur = sets[k % B]
        with torch.cuda.stream(s_in):
            if k >= B:  # the step that last used this set is done with its inputs
                s_in.wait_event(done_step[k - B])
            for a, h_t in h_in:
                cur[a].copy_(h_t, non_blocking=True)
            done_in[k].record(s_in)
        stream.wait_event(done_in[k])
        if k >= B:  # this set's previous outputs have been copied out
            stream.wait_event(done_out[k - B])
        for a, t in cur.items():
            setattr(wl, a, t)
        step()
        done_step[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done_step[k])
            for a, h_t in h_out:
                h_t.copy_(cur[a], non_blocking=True)
            done_out[k].record(s_out)
    e1.record(s_out)
    barrier()
    for a, t in sets[0].items():
        setattr(wl, a, t)
    e2e_ms = e0.elapsed_time(e1) / E2
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    h2d = sum(h.numel() * 4 for _, h in wl.h_in)
    d2h = sum(h.numel() * 4 for _, h in wl.h_out)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    roof = wl.roofline(ops_ms, peaks, sms)
    k_roofs = None
    if ktable is not None and hasattr(wl, "kernel_work"):
        # DRAM traffic records hold for the default batch of each workload
        k_roofs = kernel_rooflines(ktable, wl.kernel_work(), peaks, sms,
                                   args.workload if args.batch in (None, 7) else None)
        if roof is None and k_roofs:  # the dominant kernel: the largest device time per step
            roof = dict(max(k_roofs.values(), key=lambda r: r["ms_per_launch"] * r["launches_per_step"]))
    op_roofs = op_rooflines(ops_ms, wl.op_work(), peaks, sms) if hasattr(wl, "op_work") else None
    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": wl.describe(),
                "hbm_frac": value / world / peaks["hbm"] if wl.unit == "GB/s" else None,
                "ops_ms": ops_ms,
                "e2e": {"value": world * wl.value(e2e_ms), "unit": wl.unit, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": E2,
                        "copies": "every step: inputs in from pinned host memory, all outputs out; two device "
                                  "buffer sets in turn, so step k+1's copy-in overlaps step k's kernels and step "
                                  "k-1's copy-out"},
                "gpu_launches": launches, "roofline": roof, "clocks": clk}
        if op_roofs:
            line["ops_roofline"] = op_roofs
        if ktable is not None:
            line["kernels"] = ktable
            line["kernels_note"] = ("device time per kernel from CUDA events the library records on the launch "
                                    "stream around every launch (hc_trace_enable) during the timed region")
        if k_roofs:
            line["kernels_roofline"] = k_roofs
        if graph is not None:
            line["config"]["cuda_graph"] = f"each step one graph replay of {graph_kernels} kernels"
        if world == 1 and not args.no_cpu_baseline:
            v, cores, sample, _ = oracle_sample(wl, max_seconds=20.0)
            line["cpu_baseline"] = {"value": v, "unit": wl.unit, "cores": cores, "kind": "oracle", "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
