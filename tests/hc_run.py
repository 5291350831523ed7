"""Drive the C ABI from numpy inputs (tests and the smoke check).

Allocates device buffers with torch, calls hc_conv2d_fwd / hc_conv2d_bwd
through the ctypes binding, and returns numpy outputs.  Outputs are
pre-filled with NaN so an element a kernel forgets to write shows up, and
each buffer carries guard words before and after it that must stay intact.
"""
from __future__ import annotations

import numpy as np
import torch

from spatially_sharded_cnn_gb300 import hc

GUARD = 64  # floats of canary on each side of an output
CANARY = 12345.678


def out_hw(cfg):
    Ho = (cfg["H"] + 2 * cfg["padding"] - cfg["kh"]) // cfg["stride"] + 1
    Wo = (cfg["W"] + 2 * cfg["padding"] - cfg["kw"]) // cfg["stride"] + 1
    return Ho, Wo


class Guarded:
    """A device fp32 buffer of `shape` with canaries around it, NaN-filled."""

    def __init__(self, shape, fill=float("nan")):
        self.shape = tuple(shape)
        n = int(np.prod(self.shape))
        self.buf = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.float32, device="cuda")
        self.buf[GUARD:GUARD + n].fill_(fill)
        self.view = self.buf[GUARD:GUARD + n].view(self.shape)

    def numpy(self):
        b = self.buf.cpu().numpy()
        assert np.all(b[:GUARD] == np.float32(CANARY)) and np.all(b[-GUARD:] == np.float32(CANARY)), \
            "a kernel wrote outside its output buffer"
        return b[GUARD:-GUARD].reshape(self.shape)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def workspace(d, pass_, algo=None):
    st, nbytes = hc.hc_conv2d_workspace_size(d, pass_, algo)
    hc.check(st, "workspace size")
    return torch.empty(max(nbytes, 16) // 4 + 64, dtype=torch.float32, device="cuda"), nbytes


def fwd(cfg, x, w, b, algo=None):
    d = hc.desc(cfg)
    Ho, Wo = out_hw(cfg)
    y = Guarded((cfg["N"], cfg["C_out"], Ho, Wo))
    ws, nb = workspace(d, 0, algo)
    xd, wd = dev(x), dev(w)
    bd = dev(b) if b is not None else None
    hc.check(hc.hc_conv2d_fwd(d, xd, wd, bd, y.view, ws, nb, algo=algo), "fwd")
    hc.check(hc.hc_sync_check(), "fwd sync")
    return y.numpy()


def num_partials(cfg):
    """Grid shards Q = num_shards * num_shards_h (the partial count)."""
    return cfg["num_shards"] * max(1, int(cfg.get("num_shards_h", 1)))


def bwd(cfg, x, w, gy, algo=None, partials=True):
    d = hc.desc(cfg)
    S = num_partials(cfg)
    wshape = (cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"])
    gx = Guarded(x.shape)
    gw = Guarded(wshape)
    gb = Guarded((cfg["C_out"],))
    gwp = Guarded((S,) + wshape) if partials else None
    gbp = Guarded((S, cfg["C_out"])) if partials else None
    ws, nb = workspace(d, 1, algo)
    hc.check(hc.hc_conv2d_bwd(d, dev(x), dev(w), dev(gy), gx.view, gw.view, gb.view,
                              gwp.view if gwp else None, gbp.view if gbp else None, ws, nb, algo=algo), "bwd")
    hc.check(hc.hc_sync_check(), "bwd sync")
    out = dict(gx=gx.numpy(), gw=gw.numpy(), gb=gb.numpy())
    if partials:
        out["gw_partials"] = gwp.numpy()
        out["gb_partials"] = gbp.numpy()
    return out


def bwd_subset(cfg, x, w, gy, want, algo=None):
    """Backward with only the outputs named in `want` (subset of gx, gw, gb,
    gw_partials, gb_partials); the others are passed as NULL."""
    d = hc.desc(cfg)
    S = num_partials(cfg)
    wshape = (cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"])
    shapes = dict(gx=x.shape, gw=wshape, gb=(cfg["C_out"],), gw_partials=(S,) + wshape,
                  gb_partials=(S, cfg["C_out"]))
    bufs = {k: Guarded(shapes[k]) for k in want}
    ws, nb = workspace(d, 1, algo)
    view = lambda k: bufs[k].view if k in bufs else None
    hc.check(hc.hc_conv2d_bwd(d, dev(x), dev(w), dev(gy), view("gx"), view("gw"), view("gb"), view("gw_partials"),
                              view("gb_partials"), ws, nb, algo=algo), "bwd subset")
    hc.check(hc.hc_sync_check(), "bwd subset sync")
    return {k: v.numpy() for k, v in bufs.items()}


def normwise(got, ref):
    """max |got - ref| / max |ref| (normwise maximum relative error)."""
    ref = np.asarray(ref, np.float64)
    den = float(np.abs(ref).max())
    return float(np.abs(np.asarray(got, np.float64) - ref).max()) / (den if den > 0 else 1.0)
