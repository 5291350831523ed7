"""Per-kernel device timing (hc_trace_enable / hc_trace_collect) on the GPU:
every launch of a call is recorded under its kernel's name, the intervals are
positive and add up to at most the wall time of the traced calls, launches
into a capturing stream are left out, and tracing changes no result."""
import numpy as np
import pytest
import torch

import hc_run as R

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    from spatially_sharded_cnn_gb300 import hc as mod
    return mod


def _dw_case():
    from spatially_sharded_cnn_gb300 import synth
    cfg = dict(N=2, C_in=16, H=64, W=512, C_out=16, kh=7, kw=7, stride=1, padding=3, groups=16, num_shards=4)
    x = synth.normal((2, 16, 64, 512), 1.0, 5, 1)
    w = synth.trunc_normal((16, 1, 7, 7), 0.02, 5, 2)
    b = synth.normal((16,), 0.1, 5, 3)
    gy = synth.normal((2, 16, 64, 512), 1.0, 5, 4)
    return cfg, x, w, b, gy


def test_trace_names_and_times(hc):
    cfg, x, w, b, gy = _dw_case()
    d = hc.desc(cfg)
    xd, wd, bd, gyd = (R.dev(a) for a in (x, w, b, gy))
    y, gx, gw, gb = torch.empty_like(xd), torch.empty_like(xd), torch.empty_like(wd), torch.empty_like(bd)
    st, nb = hc.hc_conv2d_workspace_size(d, 1)
    ws = torch.empty(nb // 4 + 64, device="cuda")
    run = lambda: (hc.check(hc.hc_conv2d_fwd(d, xd, wd, bd, y)),
                   hc.check(hc.hc_conv2d_bwd(d, xd, wd, gyd, gx, gw, gb, None, None, ws, nb)))
    run()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (y, gx, gw, gb)]
    hc.hc_trace_collect()
    hc.check(hc.hc_trace_enable(True))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        run()
    e1.record()
    hc.check(hc.hc_trace_enable(False))
    torch.cuda.synchronize()
    st, table = hc.hc_trace_collect()
    hc.check(st, "collect")
    assert set(table) == {"dw_fwd_kernel", "dw_bwd_kernel", "dw_shard_partials_kernel"}, table
    for name, (n, ms) in table.items():
        assert n == 3 and ms > 0, (name, n, ms)
    assert sum(ms for _, ms in table.values()) <= e0.elapsed_time(e1) * 1.01
    for a, r in zip((y, gx, gw, gb), ref):
        assert torch.equal(a, r)
    # a second collect finds nothing new
    assert hc.hc_trace_collect()[1] == {}


def test_trace_skips_capture(hc):
    cfg, x, w, b, gy = _dw_case()
    d = hc.desc(cfg)
    xd, wd, bd = (R.dev(a) for a in (x, w, b))
    y = torch.empty_like(xd)
    hc.check(hc.hc_conv2d_fwd(d, xd, wd, bd, y))  # kernel attributes set outside the capture
    torch.cuda.synchronize()
    hc.hc_trace_collect()
    hc.check(hc.hc_trace_enable(True))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hc.check(hc.hc_conv2d_fwd(d, xd, wd, bd, y, stream=s))
    hc.check(hc.hc_trace_enable(False))
    g.replay()
    torch.cuda.synchronize()
    st, table = hc.hc_trace_collect()
    assert table == {}, table
    ref = R.fwd(cfg, x, w, b)
    assert np.array_equal(y.cpu().numpy(), ref)
