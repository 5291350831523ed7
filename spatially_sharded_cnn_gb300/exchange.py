"""One rank of the pages' multi-device Shard(3) convolution.

The NVIDIA blog "Perception model training for autonomous vehicles with
tensor parallelism" (design section and Figure 1) and its write-up at kwkr.cn
news/18980 (sections 2.2 and 5.2) put each column block of the activations on
its own device: a device sends the edge columns its neighbours need, receives
their edge columns as its halo, concatenates, runs the local convolution and
crops; in backward it does the same with grad_output, and the per-device
_Partial grad_weight / grad_bias are summed across the devices.  The region
away from the block edges needs no halo and can be computed while the halo is
in flight.

Here a rank keeps its block in the halo-padded layout of the C ABI
([N][C][H][Wl + 2 * HC_HALO_COLS], own columns at offset HC_HALO_COLS), so the
concat is the layout itself and the exchange only moves HC_HALO_COLS columns
each way:

* device tensors: the library packs / unpacks the columns (hc_halo_pack /
  hc_halo_unpack) and torch.distributed (NCCL) carries them; the interior
  column tiles run (hc_conv2d_*_rank, HC_TILES_INTERIOR) while the transfer is
  in flight, the edge tiles after it;
* host tensors (a gloo group, e.g. CPU ranks): the same messages, packed and
  unpacked on the host;
* device tensors in a gloo group (ranks that share a device, or a host without
  NCCL): packed and unpacked by the library, the messages staged through host
  memory.

The partial gradients are gathered from every rank and summed in rank order
(hc_sum_partials on the device), so every rank holds the same, deterministic
full gradient.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

HALO = 4  # HC_HALO_COLS: columns exchanged each way (the margin of the padded layout)


def padded_shape(cfg):
    """Shape of one rank's halo-padded block for the global conv cfg."""
    Wl = cfg["W"] // cfg["num_shards"]
    return (cfg["N"], cfg["C_in"], cfg["H"], Wl + 2 * HALO)


class RankHalo:
    """The halo exchange and partial-gradient reduction of one rank.

    cfg: the global conv (W the full width, num_shards = the group's size);
    the rank's block is column block `rank` of it.
    """

    def __init__(self, cfg, group=None):
        self.cfg, self.group = dict(cfg), group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        if cfg["num_shards"] != self.world:
            raise ValueError(f"num_shards {cfg['num_shards']} != ranks {self.world}")
        if cfg["W"] % self.world or (cfg["W"] // self.world) % HALO:
            raise ValueError("each rank's block must be a multiple of 4 columns wide")
        self.Wl = cfg["W"] // self.world
        self.rows = cfg["N"] * cfg["C_in"] * cfg["H"]
        self._hc = None
        self.gloo = dist.get_backend(group) == "gloo"  # device messages go through host memory

    # -- peers ------------------------------------------------------------
    def _peer(self, r):
        return r if self.group is None else dist.get_global_rank(self.group, r)

    def _lib(self):
        if self._hc is None:
            from . import hc
            self._hc = hc
        return self._hc

    @staticmethod
    def _st(t, stream):
        """The stream of a device call: the given one, else torch's current one."""
        return stream if stream is not None or not t.is_cuda else torch.cuda.current_stream(t.device)

    # -- packing ------------------------------------------------------------
    def _pack(self, t_pad, side, stream):
        if t_pad.is_cuda:
            hc = self._lib()
            buf = torch.empty((self.rows, HALO), dtype=torch.float32, device=t_pad.device)
            hc.check(hc.hc_halo_pack(hc.desc(self.cfg), t_pad, side, buf, self._st(t_pad, stream)), "halo pack")
            return buf
        cols = slice(HALO, 2 * HALO) if side == 0 else slice(self.Wl, self.Wl + HALO)
        return t_pad[..., cols].reshape(self.rows, HALO).contiguous()

    def _unpack(self, buf, side, t_pad, stream):
        if t_pad.is_cuda:
            hc = self._lib()
            hc.check(hc.hc_halo_unpack(hc.desc(self.cfg), buf, side, t_pad, self._st(t_pad, stream)), "halo unpack")
            return
        cols = slice(0, HALO) if side == 0 else slice(self.Wl + HALO, self.Wl + 2 * HALO)
        if buf is None:
            t_pad[..., cols] = 0.0
        else:
            t_pad[..., cols] = buf.reshape(t_pad.shape[:-1] + (HALO,))

    # -- the exchange ----------------------------------------------------------
    def start(self, t_pad, stream=None):
        """Pack this block's edge columns and post the sends to, and receives
        from, both neighbours.  Returns the pending exchange for finish()."""
        ops, recv = [], {}
        staged = self.gloo and t_pad.is_cuda
        if staged:
            stream = self._st(t_pad, stream)
        for side, nb in ((0, self.rank - 1), (1, self.rank + 1)):
            if 0 <= nb < self.world:
                send = self._pack(t_pad, side, stream)
                if staged:  # the packed columns to the host (the pack must finish first)
                    with torch.cuda.stream(stream):
                        send = send.to("cpu")
                rbuf = torch.empty((self.rows, HALO), dtype=torch.float32, device="cpu" if staged else t_pad.device)
                ops.append(dist.P2POp(dist.isend, send, self._peer(nb), self.group))
                ops.append(dist.P2POp(dist.irecv, rbuf, self._peer(nb), self.group))
                recv[side] = (send, rbuf)
        works = dist.batch_isend_irecv(ops) if ops else []
        return works, recv

    def finish(self, pending, t_pad, stream=None):
        """Wait for the pending exchange (on a device: the stream waits, the host
        does not) and write the halos into t_pad's margins (zeros at the image
        edges)."""
        works, recv = pending
        for w in works:
            w.wait()
        staged = self.gloo and t_pad.is_cuda
        if staged:
            stream = self._st(t_pad, stream)
        for side in (0, 1):
            buf = recv[side][1] if side in recv else None
            if staged and buf is not None:
                with torch.cuda.stream(stream):
                    buf = buf.to(t_pad.device)
            if staged and buf is None:  # the image edge: zeros into the margin
                buf = torch.zeros((self.rows, HALO), dtype=torch.float32, device=t_pad.device)
            self._unpack(buf, side, t_pad, stream)

    def exchange(self, t_pad, stream=None):
        self.finish(self.start(t_pad, stream), t_pad, stream)

    # -- the _Partial reduction ------------------------------------------------
    def reduce_partials(self, part, out=None, stream=None):
        """The full gradient from every rank's _Partial one: gathered, then
        summed in rank order (the same sum on every rank); into `out` if given."""
        flat = part.reshape(-1).contiguous()
        if out is None:
            out = torch.empty_like(part)
        if flat.is_cuda and self.gloo:  # gathered through host memory, summed on the device
            stream = self._st(flat, stream)
            with torch.cuda.stream(stream):
                host = flat.to("cpu")
            g_host = torch.empty((self.world, flat.numel()), dtype=flat.dtype)
            dist.all_gather(list(g_host.unbind(0)), host, group=self.group)
            with torch.cuda.stream(stream):
                gathered = g_host.to(flat.device)
            hc = self._lib()
            hc.check(hc.hc_sum_partials(gathered, self.world, flat.numel(), out, stream), "sum partials")
            return out
        gathered = torch.empty((self.world, flat.numel()), dtype=flat.dtype, device=flat.device)
        dist.all_gather_into_tensor(gathered, flat, group=self.group) if flat.is_cuda else \
            dist.all_gather(list(gathered.unbind(0)), flat, group=self.group)
        if flat.is_cuda:
            hc = self._lib()
            hc.check(hc.hc_sum_partials(gathered, self.world, flat.numel(), out, self._st(out, stream)),
                     "sum partials")
            return out
        g = gathered.numpy()
        acc = g[0].copy()
        for r in range(1, self.world):  # rank order, fp32, as hc_sum_partials
            acc = (acc + g[r]).astype(np.float32)
        out.copy_(torch.from_numpy(acc).reshape(part.shape))
        return out


class RankConv(RankHalo):
    """The depthwise convolution of one rank on device tensors: forward and
    backward with the halo exchange overlapped with the interior column tiles."""

    def forward(self, x_pad, w, bias, y, stream=None):
        """y (the block's output columns) from x_pad, whose own columns are set;
        its margins are exchanged here."""
        hc = self._lib()
        d = hc.desc(self.cfg)
        stream = self._st(x_pad, stream)
        pending = self.start(x_pad, stream)
        hc.check(hc.hc_conv2d_fwd_rank(d, x_pad, w, bias, y, hc.HC_TILES_INTERIOR, stream), "fwd interior")
        self.finish(pending, x_pad, stream)
        hc.check(hc.hc_conv2d_fwd_rank(d, x_pad, w, bias, y, hc.HC_TILES_EDGE, stream), "fwd edge")

    def backward(self, x_pad, w, gy_pad, gx, gw, gb, ws, ws_bytes, stream=None):
        """gx (the block's grad_input) and the full gw / gb (summed over the
        ranks) from x_pad (margins exchanged by forward) and gy_pad, whose own
        columns are set; its margins are exchanged here."""
        hc = self._lib()
        d = hc.desc(self.cfg)
        stream = self._st(x_pad, stream)
        gw_part, gb_part = torch.empty_like(gw), torch.empty_like(gb)
        pending = self.start(gy_pad, stream)
        hc.check(hc.hc_conv2d_bwd_rank(d, x_pad, w, gy_pad, gx, gw_part, gb_part, ws, ws_bytes,
                                       hc.HC_TILES_INTERIOR, stream), "bwd interior")
        self.finish(pending, gy_pad, stream)
        hc.check(hc.hc_conv2d_bwd_rank(d, x_pad, w, gy_pad, gx, gw_part, gb_part, ws, ws_bytes,
                                       hc.HC_TILES_EDGE, stream), "bwd edge")
        self.reduce_partials(gw_part, gw, stream)
        self.reduce_partials(gb_part, gb, stream)
