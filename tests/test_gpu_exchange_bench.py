"""bench.py --exchange: the W-sharded multi-rank depthwise step, run as two
ranks under torchrun.

With one visible device both ranks share it and exchange their halo columns
and partial gradients over gloo through host memory (each rank's kernels are
independent; none waits on the other).  The bench's --check gathers every
rank's block and compares it with the one-device call on the whole image:
forward and grad_input bit for bit, weight and bias gradients within 1e-5.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_exchange_bench_two_ranks_matches_one_device():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--exchange", "--check", "--batch", "1",
           "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    line = json.loads(lines[0])
    assert line["ranks"] == 2 and line["scaling"] == "weak" and line["value"] > 0
    assert line["gpu_launches"] > 0
    c = line["check"]
    assert c["y_bit_identical"] and c["gx_bit_identical"], c
    assert c["gw_normwise"] <= 1e-5 and c["gb_normwise"] <= 1e-5, c
