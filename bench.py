"""Benchmark of the width-sharded (halo-exchange) Conv2d, forward + backward.

One step = one pass of the whole hot path over one batch: hc_conv2d_fwd (shard
plan, halo exchange + concat, local conv, crop) then hc_conv2d_bwd (grad_output
halo, grad_input, per-shard _Partial grad_weight / grad_bias, fixed-order
reduction), through the C ABI on the current CUDA stream.

Default workload: ConvNeXt depthwise 7x7, padding 3, groups = C, fp32,
x (7,256,128,512) N(0,1), weight (256,1,7,7) trunc-normal std 0.02, bias 0,
grad_output N(0,1), 4 W-shards of width 128; seed 0.  Metric: algorithmic HBM
bytes per step (x + y forward; x + grad_output + grad_input backward) over the
step time, in GB/s.  Inputs are 470 MB each, larger than the 129 MB L2, so no
L2 flush is needed between steps.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 it runs under torch.distributed.run, one replica per GPU (each rank
its own batch; no data-path collective), and reports the whole-job total.
"""
from __future__ import annotations

import argparse
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


class DepthwiseWorkload:
    name = "convnext_dw7x7_fwd_bwd"

    def __init__(self, N=7, C=256, H=128, W=512, K=7, S=4, seed=0):
        self.cfg = dict(N=N, C_in=C, H=H, W=W, C_out=C, kh=K, kw=K, stride=1, padding=(K - 1) // 2, groups=C,
                        num_shards=S)
        self.K = K
        self.E = N * C * H * W
        self.seed = seed
        # algorithmic bytes: forward reads x, writes y; backward reads x and gy, writes gx
        self.bytes_fwd = 2 * 4 * self.E
        self.bytes_bwd = 3 * 4 * self.E
        self.bytes = self.bytes_fwd + self.bytes_bwd
        self.flops_bwd = 2 * 2 * K * K * self.E
        self.flops = 3 * 2 * K * K * self.E

    def describe(self):
        c = self.cfg
        return {"workload": f"depthwise {self.K}x{self.K} conv fwd+bwd, x ({c['N']},{c['C_in']},{c['H']},{c['W']}) "
                            f"fp32, {c['num_shards']} W-shards of width {c['W'] // c['num_shards']}",
                "shape": [c["N"], c["C_in"], c["H"], c["W"]], "kernel": [self.K, self.K],
                "padding": c["padding"], "groups": c["groups"], "num_shards": c["num_shards"],
                "l2": "inputs (470 MB each) larger than L2; no flush"}

    def inputs(self):
        from spatially_sharded_cnn_gb300 import synth
        c = self.cfg
        x = synth.normal((c["N"], c["C_in"], c["H"], c["W"]), 1.0, self.seed, 1)
        w = synth.trunc_normal((c["C_out"], 1, self.K, self.K), 0.02, self.seed, 2)
        b = np.zeros((c["C_out"],), np.float32)
        gy = synth.normal((c["N"], c["C_out"], c["H"], c["W"]), 1.0, self.seed, 4)
        return x, w, b, gy


class DenseWorkload:
    """Dense 5x5 conv 128->128, stride 1, padding 2, fp32 via 3xTF32 on the tensor
    cores, x (7,128,128,1024) N(0,1), weight Kaiming-normal, bias N(0,0.01),
    grad_output N(0,1), 4 W-shards of width 256."""
    name = "dense5x5_fwd_bwd"

    def __init__(self, N=7, C=128, H=128, W=1024, K=5, S=4, seed=0):
        self.cfg = dict(N=N, C_in=C, H=H, W=W, C_out=C, kh=K, kw=K, stride=1, padding=(K - 1) // 2, groups=1,
                        num_shards=S)
        self.K = K
        self.E = N * C * H * W
        self.seed = seed
        self.flops_pass = 2.0 * N * H * W * C * C * K * K   # one of forward / grad_input / grad_weight
        self.flops = 3 * self.flops_pass
        self.flops_bwd = 2 * self.flops_pass
        self.bytes = 5 * 4 * self.E
        self.bytes_bwd = 3 * 4 * self.E

    def describe(self):
        c = self.cfg
        return {"workload": f"dense {self.K}x{self.K} conv {c['C_in']}->{c['C_out']} fwd+bwd, x ({c['N']},{c['C_in']},"
                            f"{c['H']},{c['W']}) fp32 (3xTF32 tensor cores), {c['num_shards']} W-shards of width "
                            f"{c['W'] // c['num_shards']}",
                "shape": [c["N"], c["C_in"], c["H"], c["W"]], "kernel": [self.K, self.K], "padding": c["padding"],
                "groups": 1, "num_shards": c["num_shards"], "l2": "inputs (470 MB each) larger than L2; no flush"}

    def inputs(self):
        from spatially_sharded_cnn_gb300 import synth
        c = self.cfg
        x = synth.normal((c["N"], c["C_in"], c["H"], c["W"]), 1.0, self.seed, 1)
        w = synth.kaiming_normal((c["C_out"], c["C_in"], self.K, self.K), c["C_in"] * self.K * self.K, self.seed, 2)
        b = synth.normal((c["C_out"],), 0.01, self.seed, 3)
        gy = synth.normal((c["N"], c["C_out"], c["H"], c["W"]), 1.0, self.seed, 4)
        return x, w, b, gy


WORKLOADS = {"dw7": DepthwiseWorkload, "dense5x5": DenseWorkload}


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
def traffic_for(kernel: str, src_file: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current source."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    h = hashlib.sha256(open(src_file, "rb").read()).hexdigest()[:16]
    return d["bytes_per_launch"] if d.get("source_sha") == h else None


def cpu_oracle_sample(wl, max_seconds=20.0):
    """The oracle as it stands on this host's cores, on a bounded sample of the
    workload (one image, all channels: 1/N of the batch), repeated while time
    remains.  Returns (GB/s of algorithmic bytes, threads, description)."""
    import oracle
    orc = oracle.load()
    x, w, b, gy = wl.inputs_small
    cfg = dict(wl.cfg, N=1)
    t0 = time.perf_counter()
    reps = 0
    while True:
        orc.conv2d_fwd(cfg, x, w, b)
        orc.conv2d_bwd_input(cfg, w, gy)
        orc.conv2d_bwd_weight(cfg, x, gy)
        orc.conv2d_bwd_bias(cfg, gy)
        reps += 1
        if time.perf_counter() - t0 > max_seconds / 2 or reps >= 4:
            break
    dt = (time.perf_counter() - t0) / reps
    sample_bytes = wl.bytes / wl.cfg["N"]
    return sample_bytes / dt / 1e9, orc.num_threads(), f"1 of {wl.cfg['N']} images, all channels, fwd+bwd, {reps} rep(s)"


def run_reference(args, wl):
    """Reference arm: the CPU oracle timed on the host cores, on the same config
    and metric, each step a bounded sample (1 image x 16 channels)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    orc = oracle.load()
    from spatially_sharded_cnn_gb300 import synth
    c = wl.cfg
    Cs = 16
    cfg = dict(c, N=1, C_in=Cs, C_out=Cs, groups=Cs)
    x = synth.normal((1, Cs, c["H"], c["W"]), 1.0, 0, 1)
    w = synth.trunc_normal((Cs, 1, wl.K, wl.K), 0.02, 0, 2)
    b = np.zeros((Cs,), np.float32)
    gy = synth.normal((1, Cs, c["H"], c["W"]), 1.0, 0, 4)

    def step():
        orc.conv2d_fwd(cfg, x, w, b)
        orc.conv2d_bwd_input(cfg, w, gy)
        orc.conv2d_bwd_weight(cfg, x, gy)
        orc.conv2d_bwd_bias(cfg, gy)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    sample_bytes = 5 * 4 * Cs * c["H"] * c["W"]
    v = sample_bytes / dt / 1e9
    sample = f"1 image x {Cs} of {c['C_in']} channels per step ({Cs * c['H'] * c['W']} elements)"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wl.describe(),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dw7")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    wl = WORKLOADS[args.workload]()
    if args.impl == "reference":
        return run_reference(args, wl)

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
    x, w, b, gy = wl.inputs()
    wl.inputs_small = (np.ascontiguousarray(x[:1]), w, b, np.ascontiguousarray(gy[:1]))
    dev = torch.device("cuda", torch.cuda.current_device())
    xd, wd, bd, gyd = (torch.from_numpy(a).to(dev) for a in (x, w, b, gy))
    yd = torch.empty_like(xd)
    gxd = torch.empty_like(xd)
    gwd = torch.empty_like(wd)
    gbd = torch.empty_like(bd)
    d = hc.desc(wl.cfg)
    st, ws_bytes = hc.hc_conv2d_workspace_size(d, 1)
    hc.check(st, "workspace")
    st, ws_fwd = hc.hc_conv2d_workspace_size(d, 0)
    hc.check(st, "workspace")
    ws_bytes = max(ws_bytes, ws_fwd)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def fwd():
        hc.check(hc.hc_conv2d_fwd(d, xd, wd, bd, yd, ws, ws_bytes, stream), "fwd")

    def bwd():
        hc.check(hc.hc_conv2d_bwd(d, xd, wd, gyd, gxd, gwd, gbd, None, None, ws, ws_bytes, stream), "bwd")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        fwd()
        bwd()
    hc.check(hc.hc_sync_check(stream), "warmup")

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    n0 = hc.hc_launch_count()
    start.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        fwd()
        ev[k][1].record(stream)
        bwd()
        ev[k][2].record(stream)
    end.record(stream)
    barrier()
    launches = hc.hc_launch_count() - n0
    clk = clocks.stop()
    hc.check(hc.hc_sync_check(stream), "timed region")
    elapsed_ms = start.elapsed_time(end)
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_step = elapsed_ms / K
    dense = isinstance(wl, DenseWorkload)
    if dense:
        value = world * wl.flops / (ms_step * 1e-3) / 1e12
        unit = "TFLOP/s"
    else:
        value = world * wl.bytes / (ms_step * 1e-3) / 1e9
        unit = "GB/s"

    # end to end: host buffers, copies inside the timed region
    xh = torch.from_numpy(x).pin_memory()
    gyh = torch.from_numpy(gy).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    gxh = torch.empty_like(xh).pin_memory()
    gwh = torch.empty_like(wd, device="cpu").pin_memory()
    gbh = torch.empty_like(bd, device="cpu").pin_memory()
    E2 = max(1, args.e2e_steps)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E2):
        xd.copy_(xh, non_blocking=True)
        gyd.copy_(gyh, non_blocking=True)
        fwd()
        bwd()
        yh.copy_(yd, non_blocking=True)
        gxh.copy_(gxd, non_blocking=True)
        gwh.copy_(gwd, non_blocking=True)
        gbh.copy_(gbd, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / E2
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    h2d = (xh.numel() + gyh.numel()) * 4
    d2h = (yh.numel() + gxh.numel() + gwh.numel() + gbh.numel()) * 4

    # roofline of the dominant kernel (the fused depthwise backward, one launch
    # per hc_conv2d_bwd call plus two tiny fixed-order reductions)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    e2e_value = world * (wl.flops / 1e12 if dense else wl.bytes / 1e9) / (e2e_ms * 1e-3)
    alu_peak = sms * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
    bwd_tflops = wl.flops_bwd / (bwd_ms * 1e-3) / 1e12
    bwd_gbs = wl.bytes_bwd / (bwd_ms * 1e-3) / 1e9
    if dense:
        # forward call = operand preparation + one tensor-core GEMM pass; the peak is the
        # measured bf16 dense rate x the nominal tf32/bf16 ratio (1.1 / 2.25), / 3 for 3xTF32
        tf32_peak = peaks["bf16"] * (1.1 / 2.25)
        fwd_tflops = wl.flops_pass / (fwd_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "tc_conv_kernel (forward call incl. operand prep)",
                "achieved": fwd_tflops, "peak": tf32_peak / 3, "unit": "TFLOP/s (fp32-equivalent, 3xTF32)",
                "frac": fwd_tflops / (tf32_peak / 3), "traffic": None,
                "peak_source": f"measured bf16 {peaks['bf16']:.0f} TFLOP/s x 1.1/2.25 (tf32) / 3 (3xTF32 passes)",
                "ms_per_launch": fwd_ms}
    else:
        roof = {"bound": "alu", "kernel": "dw_bwd_kernel<7>", "achieved": bwd_tflops, "peak": alu_peak,
                "unit": "TFLOP/s", "frac": bwd_tflops / alu_peak,
                "traffic": traffic_for("dw_bwd_kernel<7>", os.path.join(ROOT, "spatially_sharded_cnn_gb300", "csrc",
                                                                        "dw.cu")),
                "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                "hbm": {"achieved": bwd_gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": bwd_gbs / peaks["hbm"],
                        "peak_source": peaks["src"]},
            "ms_per_launch": bwd_ms}
    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": wl.describe(),
                "hbm_frac": None if dense else value / world / peaks["hbm"],
                "phases_ms": {"fwd": fwd_ms, "bwd": bwd_ms},
                "e2e": {"value": e2e_value, "unit": unit,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "gpu_launches": launches, "roofline": roof, "clocks": clk}
        if world == 1 and not args.no_cpu_baseline and not dense:
            v, cores, sample = cpu_oracle_sample(wl)
            line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
