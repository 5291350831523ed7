"""ctypes binding of the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
bench's CPU-baseline leg, never by the product path.  The oracle shares no code
with the CUDA library.

``Oracle(path)`` wraps one compiled copy of the oracle; ``load()`` builds (if
needed) and returns the default one.  A test can compile a modified copy of
oracle.c elsewhere and wrap it the same way.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")


def compile_oracle(src: str = SRC, out: str = LIB, openmp: bool = True) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP if available)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-o", out, src, "-lm"]
    if openmp:
        r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
        if r.returncode == 0:
            return out
    r = subprocess.run(base, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    return out


class Desc(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("N", "C_in", "H", "W", "C_out", "kh", "kw", "stride", "padding", "groups", "num_shards",
                 "num_shards_h")]


class Extent(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("in_begin", "in_end", "halo_left", "halo_right", "out_begin", "out_end")]


def make_desc(cfg: dict) -> Desc:
    return Desc(*(int(cfg.get(k, 1) if k == "num_shards_h" else cfg[k]) for k, _ in Desc._fields_))


_F = C.POINTER(C.c_float)
_D = C.POINTER(C.c_double)


def _f(a):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(_F)


def _d(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def out_size(n, k, s, p):
    return (n + 2 * p - k) // s + 1


class Oracle:
    def __init__(self, path: str = LIB):
        L = C.CDLL(path)
        self.lib = L
        P = C.POINTER(Desc)
        L.or_num_threads.restype = C.c_int
        L.or_out_size.argtypes = [C.c_int] * 4
        L.or_out_size.restype = C.c_int
        for name, args in {
            "or_conv2d_fwd": [P, _F, _F, _F, _D],
            "or_conv2d_bwd_input": [P, _F, _F, _D],
            "or_conv2d_bwd_weight": [P, _F, _F, _D],
            "or_conv2d_bwd_bias": [P, _F, _D],
            "or_shard_plan": [P, C.POINTER(Extent), C.POINTER(C.c_int), C.POINTER(C.c_int)],
            "or_shard_plan_h": [P, C.POINTER(Extent)],
            "or_halo_extend": [P, C.c_int, _F, _F],
            "or_sharded_fwd": [P, _F, _F, _F, _D],
            "or_sharded_bwd": [P, _F, _F, _F, _D, _D, _D],
        }.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = C.c_int
        L.or_conv2d_fwd_at.argtypes = [P, _F, _F, _F] + [C.c_int] * 4
        L.or_conv2d_gx_at.argtypes = [P, _F, _F] + [C.c_int] * 4
        L.or_conv2d_gw_at.argtypes = [P, _F, _F] + [C.c_int] * 8
        L.or_conv2d_gb_at.argtypes = [P, _F] + [C.c_int] * 3
        for n in ("or_conv2d_fwd_at", "or_conv2d_gx_at", "or_conv2d_gw_at", "or_conv2d_gb_at"):
            getattr(L, n).restype = C.c_double
        I64 = C.c_int64
        L.or_layernorm_c_fwd.argtypes = [C.c_int, C.c_int, I64, _D, _D, _D, C.c_double, _D, _D, _D]
        L.or_layernorm_c_bwd.argtypes = [C.c_int, C.c_int, I64, _D, _D, _D, C.c_double, _D, _D, _D]
        L.or_gelu_fwd.argtypes = [I64, _D, _D]
        L.or_gelu_bwd.argtypes = [I64, _D, _D, _D]
        L.or_layerscale_residual_fwd.argtypes = [C.c_int, C.c_int, I64, _D, _D, _D, _D]
        L.or_layerscale_residual_bwd.argtypes = [C.c_int, C.c_int, I64, _D, _D, _D, _D, _D, _D]
        L.or_layerscale_droppath_fwd.argtypes = [C.c_int, C.c_int, I64, _D, _D, _D, _D, _D]
        L.or_layerscale_droppath_bwd.argtypes = [C.c_int, C.c_int, I64, _D, _D, _D, _D, _D, _D, _D]
        for n in ("or_layernorm_c_fwd", "or_layernorm_c_bwd", "or_gelu_fwd", "or_gelu_bwd",
                  "or_layerscale_residual_fwd", "or_layerscale_residual_bwd", "or_layerscale_droppath_fwd",
                  "or_layerscale_droppath_bwd"):
            getattr(L, n).restype = None
        L.or_splitmix64.argtypes = [C.c_uint64, C.c_uint64]
        L.or_splitmix64.restype = C.c_uint64
        L.or_drop_path_mask.argtypes = [C.c_int, C.c_float, C.c_uint64, C.c_uint64, _F]
        L.or_drop_path_mask.restype = C.c_int

    # -- sizes -------------------------------------------------------------
    def num_threads(self) -> int:
        return self.lib.or_num_threads()

    def out_size(self, n, k, s, p) -> int:
        return self.lib.or_out_size(n, k, s, p)

    @staticmethod
    def _shapes(cfg):
        Ho = out_size(cfg["H"], cfg["kh"], cfg["stride"], cfg["padding"])
        Wo = out_size(cfg["W"], cfg["kw"], cfg["stride"], cfg["padding"])
        return Ho, Wo

    # -- unsharded conv ----------------------------------------------------
    def conv2d_fwd(self, cfg, x, w, b=None):
        Ho, Wo = self._shapes(cfg)
        y = np.empty((cfg["N"], cfg["C_out"], Ho, Wo), np.float64)
        rc = self.lib.or_conv2d_fwd(C.byref(make_desc(cfg)), _f(x), _f(w), _f(b), _d(y))
        assert rc == 0, rc
        return y

    def conv2d_bwd_input(self, cfg, w, gy):
        gx = np.empty((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), np.float64)
        rc = self.lib.or_conv2d_bwd_input(C.byref(make_desc(cfg)), _f(w), _f(gy), _d(gx))
        assert rc == 0, rc
        return gx

    def conv2d_bwd_weight(self, cfg, x, gy):
        gw = np.empty((cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"]), np.float64)
        rc = self.lib.or_conv2d_bwd_weight(C.byref(make_desc(cfg)), _f(x), _f(gy), _d(gw))
        assert rc == 0, rc
        return gw

    def conv2d_bwd_bias(self, cfg, gy):
        gb = np.empty((cfg["C_out"],), np.float64)
        rc = self.lib.or_conv2d_bwd_bias(C.byref(make_desc(cfg)), _f(gy), _d(gb))
        assert rc == 0, rc
        return gb

    # -- single elements -----------------------------------------------------
    def fwd_at(self, cfg, x, w, b, n, co, i, j):
        return self.lib.or_conv2d_fwd_at(C.byref(make_desc(cfg)), _f(x), _f(w), _f(b), n, co, i, j)

    def gx_at(self, cfg, w, gy, n, ci, h, c):
        return self.lib.or_conv2d_gx_at(C.byref(make_desc(cfg)), _f(w), _f(gy), n, ci, h, c)

    def gw_at(self, cfg, x, gy, co, cl, u, v, j0, j1, i0=0, i1=1 << 30):
        """grad_weight[co, cl, u, v] restricted to output columns [j0, j1) and rows [i0, i1)."""
        return self.lib.or_conv2d_gw_at(C.byref(make_desc(cfg)), _f(x), _f(gy), co, cl, u, v, j0, j1, i0, i1)

    def gb_at(self, cfg, gy, co, j0, j1):
        return self.lib.or_conv2d_gb_at(C.byref(make_desc(cfg)), _f(gy), co, j0, j1)

    # -- the sharded method --------------------------------------------------
    def shard_plan(self, cfg):
        S = cfg["num_shards"]
        ext = (Extent * S)()
        Ho, Wo = C.c_int(0), C.c_int(0)
        rc = self.lib.or_shard_plan(C.byref(make_desc(cfg)), ext, C.byref(Ho), C.byref(Wo))
        if rc:
            return rc, None, None, None
        rows = [tuple(getattr(e, f) for f, _ in Extent._fields_) for e in ext]
        return 0, rows, Ho.value, Wo.value

    def shard_plan_h(self, cfg):
        """Row-shard extents (num_shards_h of them, or one covering every row)."""
        Sh = max(1, int(cfg.get("num_shards_h", 1)))
        ext = (Extent * Sh)()
        rc = self.lib.or_shard_plan_h(C.byref(make_desc(cfg)), ext)
        if rc:
            return rc, None
        return 0, [tuple(getattr(e, f) for f, _ in Extent._fields_) for e in ext]

    def halo_extend(self, cfg, q, x):
        """Extended tile of grid shard q = a * num_shards + b: [N][C][He][We]."""
        rc, plan, _, _ = self.shard_plan(cfg)
        assert rc == 0, rc
        rc, plan_h = self.shard_plan_h(cfg)
        assert rc == 0, rc
        e, f = plan[q % cfg["num_shards"]], plan_h[q // cfg["num_shards"]]
        We = e[2] + (e[1] - e[0]) + e[3]
        He = f[2] + (f[1] - f[0]) + f[3]
        xe = np.empty((cfg["N"], cfg["C_in"], He, We), np.float32)
        rc = self.lib.or_halo_extend(C.byref(make_desc(cfg)), q, _f(x), _f(xe))
        assert rc == 0, rc
        return xe

    def sharded_fwd(self, cfg, x, w, b=None):
        Ho, Wo = self._shapes(cfg)
        y = np.full((cfg["N"], cfg["C_out"], Ho, Wo), np.nan)
        rc = self.lib.or_sharded_fwd(C.byref(make_desc(cfg)), _f(x), _f(w), _f(b), _d(y))
        assert rc == 0, rc
        return y

    def sharded_bwd(self, cfg, x, w, gy):
        S = cfg["num_shards"] * max(1, int(cfg.get("num_shards_h", 1)))
        gx = np.empty((cfg["N"], cfg["C_in"], cfg["H"], cfg["W"]), np.float64)
        gwp = np.empty((S, cfg["C_out"], cfg["C_in"] // cfg["groups"], cfg["kh"], cfg["kw"]), np.float64)
        gbp = np.empty((S, cfg["C_out"]), np.float64)
        rc = self.lib.or_sharded_bwd(C.byref(make_desc(cfg)), _f(x), _f(w), _f(gy), _d(gx), _d(gwp), _d(gbp))
        assert rc == 0, rc
        return gx, gwp, gbp

    # -- pointwise ops (inputs converted to float64) --------------------------
    def layernorm_c_fwd(self, x, gamma, beta, eps):
        x = np.ascontiguousarray(x, np.float64)
        N, Cc = x.shape[:2]
        HW = int(np.prod(x.shape[2:]))
        y = np.empty_like(x)
        mean = np.empty((N, HW))
        rstd = np.empty((N, HW))
        self.lib.or_layernorm_c_fwd(N, Cc, HW, _d(x), _d(np.ascontiguousarray(gamma, np.float64)),
                                    _d(np.ascontiguousarray(beta, np.float64)), eps, _d(y), _d(mean), _d(rstd))
        return y, mean, rstd

    def layernorm_c_bwd(self, x, gamma, gy, eps):
        x = np.ascontiguousarray(x, np.float64)
        gy = np.ascontiguousarray(gy, np.float64)
        N, Cc = x.shape[:2]
        HW = int(np.prod(x.shape[2:]))
        gx = np.empty_like(x)
        gg = np.empty(Cc)
        gbt = np.empty(Cc)
        self.lib.or_layernorm_c_bwd(N, Cc, HW, _d(x), _d(np.ascontiguousarray(gamma, np.float64)), _d(gy), eps,
                                    _d(gx), _d(gg), _d(gbt))
        return gx, gg, gbt

    def gelu_fwd(self, x):
        x = np.ascontiguousarray(x, np.float64)
        y = np.empty_like(x)
        self.lib.or_gelu_fwd(x.size, _d(x), _d(y))
        return y

    def gelu_bwd(self, x, gy):
        x = np.ascontiguousarray(x, np.float64)
        gy = np.ascontiguousarray(gy, np.float64)
        gx = np.empty_like(x)
        self.lib.or_gelu_bwd(x.size, _d(x), _d(gy), _d(gx))
        return gx

    def layerscale_residual_fwd(self, res, branch, gamma):
        res = np.ascontiguousarray(res, np.float64)
        branch = np.ascontiguousarray(branch, np.float64)
        N, Cc = res.shape[:2]
        HW = int(np.prod(res.shape[2:]))
        out = np.empty_like(res)
        self.lib.or_layerscale_residual_fwd(N, Cc, HW, _d(res), _d(branch),
                                            _d(np.ascontiguousarray(gamma, np.float64)), _d(out))
        return out

    def layerscale_residual_bwd(self, branch, gamma, gy):
        branch = np.ascontiguousarray(branch, np.float64)
        gy = np.ascontiguousarray(gy, np.float64)
        N, Cc = branch.shape[:2]
        HW = int(np.prod(branch.shape[2:]))
        gres = np.empty_like(gy)
        gbr = np.empty_like(gy)
        gg = np.empty(Cc)
        self.lib.or_layerscale_residual_bwd(N, Cc, HW, _d(branch), _d(np.ascontiguousarray(gamma, np.float64)),
                                            _d(gy), _d(gres), _d(gbr), _d(gg))
        return gres, gbr, gg


    # -- DropPath ------------------------------------------------------------
    def splitmix64(self, seed, i) -> int:
        return int(self.lib.or_splitmix64(seed, i))

    def drop_path_mask(self, N, p, seed, offset=0):
        mask = np.empty(N, np.float32)
        if self.lib.or_drop_path_mask(N, float(p), seed, offset, _f(mask)):
            raise ValueError("drop probability must be in [0, 1)")
        return mask

    def layerscale_droppath_fwd(self, res, branch, gamma, mask):
        res = np.ascontiguousarray(res, np.float64)
        branch = np.ascontiguousarray(branch, np.float64)
        N, Cc = res.shape[:2]
        HW = int(np.prod(res.shape[2:]))
        out = np.empty_like(res)
        self.lib.or_layerscale_droppath_fwd(N, Cc, HW, _d(res), _d(branch), _d(np.ascontiguousarray(gamma, np.float64)),
                                            _d(np.ascontiguousarray(mask, np.float64)), _d(out))
        return out

    def layerscale_droppath_bwd(self, branch, gamma, mask, gy):
        branch = np.ascontiguousarray(branch, np.float64)
        gy = np.ascontiguousarray(gy, np.float64)
        N, Cc = branch.shape[:2]
        HW = int(np.prod(branch.shape[2:]))
        gres, gbr, gg = np.empty_like(gy), np.empty_like(gy), np.empty(Cc)
        self.lib.or_layerscale_droppath_bwd(N, Cc, HW, _d(branch), _d(np.ascontiguousarray(gamma, np.float64)),
                                            _d(np.ascontiguousarray(mask, np.float64)), _d(gy), _d(gres), _d(gbr),
                                            _d(gg))
        return gres, gbr, gg


_lock = threading.Lock()
_default = None


def load() -> Oracle:
    """Build the oracle if its library is missing or older than its source, and load it."""
    global _default
    with _lock:
        if _default is None:
            if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
                compile_oracle()
            _default = Oracle(LIB)
        return _default
