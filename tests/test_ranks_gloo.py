"""The pages' multi-device protocol, run as CPU ranks over gloo.

Each rank owns one Shard(3) column block.  Forward: send the edge columns to
the neighbours, receive their halos, concat, local conv (oracle), crop.
Backward: zero-pad the local grad_output, local grad_input / grad_weight /
grad_bias (oracle), send the halo part of the local grad_input back to the
neighbour that owns those columns, and all-reduce the _Partial weight and bias
gradients (NVIDIA blog "Perception model training for autonomous vehicles with
tensor parallelism", design section and Figures 1-2; kwkr.cn news/18980,
sections 2.2 and 3.2).  The gathered result must equal the unsharded oracle.

Every halo message is preceded by a header (sender, step, column count); a
receiver that sees a header it does not expect, or no message within the
timeout, raises -- the tests below drop and duplicate messages on the host to
check that.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle_pins as P


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


class HaloError(RuntimeError):
    pass


_pending = []


def _send(t, dst, step, fault):
    """Post the header and payload without blocking; _flush() waits for them."""
    hdr = torch.tensor([dist.get_rank(), step, t.shape[-1]], dtype=torch.int64)
    if fault == "drop":
        return
    for _ in range(2 if fault == "dup" else 1):
        for m in (hdr, t.contiguous()):
            _pending.append((dist.isend(m, dst), m))


def _flush():
    while _pending:
        w, _ = _pending.pop(0)
        w.wait()


def _recv(shape, src, step, timeout_s=3.0, dtype=torch.float32):
    def wait(t, what):
        try:
            ok = dist.irecv(t, src).wait(timeout=datetime.timedelta(seconds=timeout_s))
        except RuntimeError as ex:          # gloo reports a timeout by raising
            raise HaloError(f"no halo {what} from rank {src} at step {step}: {ex}") from None
        if ok is False:
            raise HaloError(f"no halo {what} from rank {src} at step {step}")

    hdr = torch.empty(3, dtype=torch.int64)
    wait(hdr, "header")
    if hdr.tolist() != [src, step, shape[-1]]:
        raise HaloError(f"unexpected halo header {hdr.tolist()} from rank {src} at step {step}")
    buf = torch.empty(shape, dtype=dtype)
    wait(buf, "payload")
    return buf


def _exchange(local, pL, pR, step, fault=None):
    """Return [left halo | local | right halo] along the last dim, zeros at the image edges."""
    r, S = dist.get_rank(), dist.get_world_size()
    sh = list(local.shape)
    def sends():
        if r > 0 and pR:
            _send(local[..., :pR], r - 1, step, fault)
        if r < S - 1 and pL:
            _send(local[..., -pL:], r + 1, step, None)

    def recvs():
        left = torch.zeros(sh[:-1] + [pL])
        right = torch.zeros(sh[:-1] + [pR])
        if r > 0 and pL:
            left = _recv(sh[:-1] + [pL], r - 1, step)
        if r < S - 1 and pR:
            right = _recv(sh[:-1] + [pR], r + 1, step)
        return left, right

    sends()
    left, right = recvs()
    _flush()
    return torch.cat([left, local, right], dim=-1)


def _return_halo_grads(gxe, pL, pR, Wl, step):
    """Send the halo columns of the local grad_input to their owners; add what comes back."""
    r, S = dist.get_rank(), dist.get_world_size()
    own = gxe[..., pL:pL + Wl].clone()
    sh = list(own.shape)

    def sends():
        if r > 0 and pL:
            _send(gxe[..., :pL], r - 1, step, None)
        if r < S - 1 and pR:
            _send(gxe[..., pL + Wl:], r + 1, step, None)

    def recvs():
        if r > 0 and pL:
            # left neighbour's right-halo grads land on my first pL columns
            own[..., :pL] += _recv(sh[:-1] + [pL], r - 1, step, dtype=gxe.dtype)
        if r < S - 1 and pR:
            own[..., -pR:] += _recv(sh[:-1] + [pR], r + 1, step, dtype=gxe.dtype)

    sends()
    recvs()
    _flush()
    return own


def _worker(rank, world, port, cfg, fault, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=30))
    try:
        import oracle
        orc = oracle.load()
        cfg = dict(cfg, num_shards=world)
        x, w, b, gy = P.rand_case(cfg, 77)
        rc, plan, Ho, Wo = orc.shard_plan(cfg)
        e = plan[rank]
        Wl = e[1] - e[0]
        pL, pR = e[2], e[3]
        s, p = cfg["stride"], cfg["padding"]
        xe = _exchange(torch.from_numpy(np.ascontiguousarray(x[..., e[0]:e[1]])), pL, pR, 0, fault if rank == 1 else None)
        xe = np.ascontiguousarray(xe.numpy())
        lcfg = dict(cfg, W=xe.shape[-1])
        yl = orc.conv2d_fwd(lcfg, xe, w, b)
        crop = p // s
        n_own = e[5] - e[4]
        y_own = yl[..., crop:crop + n_own]
        # backward: zero-pad grad_output back to the local conv's width
        gyl = np.zeros(yl.shape, np.float32)
        gyl[..., crop:crop + n_own] = gy[..., e[4]:e[5]]
        gxe = torch.from_numpy(orc.conv2d_bwd_input(lcfg, w, gyl).astype(np.float64))
        gx_own = _return_halo_grads(gxe, pL, pR, Wl, 1)
        gw = torch.from_numpy(orc.conv2d_bwd_weight(lcfg, xe, gyl))
        gb = torch.from_numpy(orc.conv2d_bwd_bias(lcfg, gyl))
        dist.all_reduce(gw)
        dist.all_reduce(gb)
        q.put((rank, "ok", y_own, gx_own.numpy(), gw.numpy(), gb.numpy()))
    except HaloError as ex:
        q.put((rank, "halo_error", str(ex), None, None, None))
    except Exception as ex:                 # e.g. the peer left after its own halo error
        q.put((rank, "error", repr(ex), None, None, None))
    finally:
        dist.destroy_process_group()


def _run(cfg, world=2, fault=None):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cfg, fault, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    out = {}
    for _ in range(world):
        item = q.get(timeout=60)
        out[item[0]] = item[1:]
    for pr in procs:
        pr.join(timeout=60)
    return out


@pytest.mark.parametrize("cfg", [P.cfg_of(1, 4, 16, 32, 4, 5, 1, 2, 1), P.cfg_of(2, 3, 6, 24, 3, 7, 1, 3, 3),
                                 P.cfg_of(1, 2, 6, 16, 4, 2, 2, 0, 1)],
                         ids=["dense5x5", "depthwise7x7", "down2x2s2"])
def test_two_ranks_match_unsharded(orc, cfg):
    out = _run(cfg)
    x, w, b, gy = P.rand_case(dict(cfg, num_shards=2), 77)
    y = orc.conv2d_fwd(cfg, x, w, b)
    gx = orc.conv2d_bwd_input(cfg, w, gy)
    gw = orc.conv2d_bwd_weight(cfg, x, gy)
    gb = orc.conv2d_bwd_bias(cfg, gy)
    assert all(v[0] == "ok" for v in out.values()), out
    y_s = np.concatenate([out[r][1] for r in range(2)], axis=-1)
    gx_s = np.concatenate([out[r][2] for r in range(2)], axis=-1)
    assert np.abs(y_s - y).max() <= 1e-12
    assert np.abs(gx_s - gx).max() <= 1e-12
    for r in range(2):
        assert np.abs(out[r][3] - gw).max() <= 1e-12 * max(1, np.abs(gw).max())
        assert np.abs(out[r][4] - gb).max() <= 1e-12 * max(1, np.abs(gb).max())


@pytest.mark.parametrize("fault", ["drop", "dup"])
def test_halo_fault_is_detected(fault):
    out = _run(P.cfg_of(1, 2, 4, 16, 2, 5, 1, 2, 1), fault=fault)
    # rank 1 dropped (or duplicated) the halo it owes rank 0: rank 0 must notice
    assert out[0][0] == "halo_error", out[0]


# ---- the library's rank path (spatially_sharded_cnn_gb300.exchange) on CPU ranks ----
def _exchange_worker(rank, world, port, cfg, q):
    """One rank of RankHalo on host tensors: pad, exchange x's and grad_output's
    margins, then the local conv on the exchanged block (the oracle standing in
    for the device kernels) and the rank-order reduction of the partials."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=30))
    try:
        import oracle
        from spatially_sharded_cnn_gb300.exchange import HALO, RankHalo, padded_shape
        orc = oracle.load()
        cfg = dict(cfg, num_shards=world)
        x, w, b, gy = P.rand_case(cfg, 91)
        ex = RankHalo(cfg)
        Wl = ex.Wl
        pads = {}
        for name, t in (("x", x), ("gy", gy)):
            tp = torch.full(padded_shape(cfg), float("nan"))
            tp[..., HALO:HALO + Wl] = torch.from_numpy(np.ascontiguousarray(t[..., rank * Wl:(rank + 1) * Wl]))
            ex.exchange(tp)
            pads[name] = tp.numpy()
        p = cfg["padding"]
        xe = np.ascontiguousarray(pads["x"][..., HALO - p:HALO + Wl + p])
        # the local conv on the exchanged block (stride 1, "same"): padding p, then the crop
        lcfg = dict(cfg, W=Wl + 2 * p, num_shards=1)
        y_own = orc.conv2d_fwd(lcfg, xe, w, b)[..., p:p + Wl]
        # this rank's _Partial gradients (the sharded oracle's), reduced across the ranks in rank order
        _, gwp, gbp = orc.sharded_bwd(cfg, x, w, gy)
        gw = ex.reduce_partials(torch.from_numpy(gwp[rank].astype(np.float32)))
        gb = ex.reduce_partials(torch.from_numpy(gbp[rank].astype(np.float32)))
        q.put((rank, "ok", pads["x"], pads["gy"], y_own, gw.numpy(), gb.numpy()))
    except Exception as ex_:
        q.put((rank, "error", repr(ex_), None, None, None, None))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_rank_halo_exchange_on_cpu_ranks(orc, world):
    cfg = P.cfg_of(2, 3, 6, 8 * world, 3, 7, 1, 3, 3)   # depthwise 7x7, 8 columns per rank
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_worker, args=(r, world, port, cfg, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    out = {}
    for _ in range(world):
        item = q.get(timeout=60)
        out[item[0]] = item[1:]
    for pr in procs:
        pr.join(timeout=60)
    assert all(v[0] == "ok" for v in out.values()), out
    c = dict(cfg, num_shards=world)
    x, w, b, gy = P.rand_case(c, 91)
    Wl, p = 8, 3
    for r in range(world):
        # the margins: the neighbours' edge columns (zeros past the image edge), bit for bit
        assert np.array_equal(out[r][1][..., 4 - p:4 + Wl + p], orc.halo_extend(c, r, x)[..., :Wl + 2 * p]), r
        assert np.array_equal(out[r][2][..., 4 - p:4 + Wl + p], orc.halo_extend(c, r, gy)[..., :Wl + 2 * p]), r
    y = orc.conv2d_fwd(c, x, w, b)
    assert np.abs(np.concatenate([out[r][3] for r in range(world)], axis=-1) - y).max() <= 1e-12
    gw, gb = orc.conv2d_bwd_weight(c, x, gy), orc.conv2d_bwd_bias(c, gy)
    for r in range(world):  # every rank holds the same reduced gradient
        assert np.array_equal(out[r][4], out[0][4]) and np.array_equal(out[r][5], out[0][5])
        assert np.abs(out[r][4] - gw).max() <= 1e-6 * np.abs(gw).max()
        assert np.abs(out[r][5] - gb).max() <= 1e-6 * np.abs(gb).max()
