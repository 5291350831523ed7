"""Thin ctypes binding of libhc.so (include/hc.h), same names as the C ABI.

Argument marshalling only: tensors may be given as torch tensors (their
``data_ptr()`` is passed), as integer device addresses, or as None for a NULL
pointer; a ``torch.cuda.Stream`` or an integer cudaStream_t selects the
stream.  Every computation runs in the library's CUDA kernels; there is no
fallback.  Importing this module raises ImportError when the library has not
been built.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libhc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with spatially_sharded_cnn_gb300.build.build() "
                      "(nvcc, sm_103a); there is no CPU fallback")

_lib = C.CDLL(LIB_PATH)

HC_OK, HC_ERR_INVALID_ARG, HC_ERR_UNSUPPORTED, HC_ERR_WORKSPACE, HC_ERR_CUDA, HC_ERR_TIMEOUT = range(6)
HC_ALGO_AUTO, HC_ALGO_DIRECT, HC_ALGO_DEPTHWISE, HC_ALGO_TC_3XTF32, HC_ALGO_TC_BF16X6 = range(5)
HC_ACT_NONE, HC_ACT_GELU_INPUT, HC_ACT_GELU_OUTPUT = range(3)
HC_TILES_ALL, HC_TILES_INTERIOR, HC_TILES_EDGE = range(3)
HC_HALO_COLS = 4


class hc_conv_desc(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("N", "C_in", "H", "W", "C_out", "kh", "kw", "stride", "padding", "groups", "num_shards",
                 "num_shards_h")]


class hc_shard_extent(C.Structure):
    _fields_ = [(n, C.c_int) for n in
                ("in_begin", "in_end", "halo_left", "halo_right", "out_begin", "out_end")]


class HcError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {hc_status_string(status)} ({status})")
        self.status = status


def desc(cfg: dict) -> hc_conv_desc:
    """hc_conv_desc from a dict with the field names of the C struct (num_shards_h defaults to 1)."""
    return hc_conv_desc(*(int(cfg.get(k, 1) if k == "num_shards_h" else cfg[k]) for k, _ in hc_conv_desc._fields_))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return C.c_void_p(t)
    return C.c_void_p(t.data_ptr())


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return C.c_void_p(s)
    return C.c_void_p(s.cuda_stream)


_P = C.c_void_p
_D = C.POINTER(hc_conv_desc)
_lib.hc_shard_plan.argtypes = [_D, C.POINTER(hc_shard_extent), C.POINTER(C.c_int), C.POINTER(C.c_int)]
_lib.hc_shard_plan_rows.argtypes = [_D, C.POINTER(hc_shard_extent)]
_lib.hc_conv2d_workspace_size.argtypes = [_D, C.c_int, C.POINTER(C.c_size_t)]
_lib.hc_conv2d_workspace_size_algo.argtypes = [_D, C.c_int, C.c_int, C.POINTER(C.c_size_t)]
_lib.hc_conv2d_select.argtypes = [_D, C.c_int, C.POINTER(C.c_int)]
_lib.hc_conv2d_fwd.argtypes = [_D, _P, _P, _P, _P, _P, C.c_size_t, _P]
_lib.hc_conv2d_fwd_algo.argtypes = [_D, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_int]
_lib.hc_conv2d_bwd.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]
_lib.hc_conv2d_bwd_algo.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_int]
_lib.hc_conv2d_bwd_reuse.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_size_t, _P, C.c_int]
_lib.hc_conv2d_bwd_residual.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_int]
_lib.hc_conv2d_fwd_act.argtypes = [_D, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_int, C.c_int]
_lib.hc_conv2d_bwd_act.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_size_t, _P, C.c_int,
                                   C.c_int, _P]
_lib.hc_halo_gather.argtypes = [_D, _P, _P, _P]
_lib.hc_conv2d_bwd_depthwise_noalloc.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P]
_lib.hc_conv2d_bwd_depthwise_noalloc.restype = C.c_int
_I, _L, _F = C.c_int, C.c_longlong, C.c_float
_lib.hc_pointwise_workspace_size.argtypes = [_I, _I, _L, C.POINTER(C.c_size_t)]
_lib.hc_layernorm_c_fwd.argtypes = [_I, _I, _L, _P, _P, _P, _F, _P, _P, _P, _P]
_lib.hc_layernorm_c_bwd.argtypes = [_I, _I, _L, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]
_lib.hc_gelu_fwd.argtypes = [_L, _P, _P, _P]
_lib.hc_add_inplace.argtypes = [_L, _P, _P, _P]
_lib.hc_gelu_bwd.argtypes = [_L, _P, _P, _P, _P]
_lib.hc_layerscale_residual_fwd.argtypes = [_I, _I, _L, _P, _P, _P, _P, _P]
_lib.hc_layerscale_residual_bwd.argtypes = [_I, _I, _L, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]
for _n in ("hc_add_inplace", "hc_pointwise_workspace_size", "hc_layernorm_c_fwd", "hc_layernorm_c_bwd", "hc_gelu_fwd", "hc_gelu_bwd",
           "hc_layerscale_residual_fwd", "hc_layerscale_residual_bwd"):
    getattr(_lib, _n).restype = C.c_int
_lib.hc_drop_path_mask.argtypes = [_I, _F, C.c_ulonglong, C.c_ulonglong, _P, _P]
_lib.hc_drop_path_mask.restype = C.c_int
_lib.hc_layerscale_droppath_fwd.argtypes = [_I, _I, _L, _P, _P, _P, _P, _P, _P]
_lib.hc_layerscale_droppath_fwd.restype = C.c_int
_lib.hc_layerscale_droppath_bwd.argtypes = [_I, _I, _L, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]
_lib.hc_layerscale_droppath_bwd.restype = C.c_int
_lib.hc_conv2d_step_graph_create.argtypes = [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, C.c_size_t,
                                             C.POINTER(C.c_void_p)]
_lib.hc_conv2d_step_graph_create.restype = C.c_int
_lib.hc_step_graph_launch.argtypes = [C.c_void_p, _P]
_lib.hc_step_graph_launch.restype = C.c_int
_lib.hc_step_graph_destroy.argtypes = [C.c_void_p]
_lib.hc_step_graph_destroy.restype = C.c_int
_lib.hc_sync_check.argtypes = [_P]
_lib.hc_selftest_timeout.argtypes = [C.c_int, _P]
_lib.hc_selftest_timeout.restype = C.c_int
_lib.hc_status_string.argtypes = [C.c_int]
_lib.hc_status_string.restype = C.c_char_p
_lib.hc_launch_count.restype = C.c_ulonglong
for _n in ("hc_shard_plan", "hc_shard_plan_rows", "hc_conv2d_workspace_size", "hc_conv2d_workspace_size_algo",
           "hc_conv2d_select",
           "hc_conv2d_fwd", "hc_conv2d_fwd_algo", "hc_conv2d_bwd", "hc_conv2d_bwd_algo", "hc_halo_gather",
           "hc_sync_check"):
    getattr(_lib, _n).restype = C.c_int

EXPORTS = [
    "hc_shard_plan", "hc_conv2d_workspace_size", "hc_conv2d_workspace_size_algo", "hc_conv2d_select",
    "hc_conv2d_fwd", "hc_conv2d_fwd_algo", "hc_conv2d_bwd", "hc_conv2d_bwd_algo", "hc_halo_gather",
    "hc_sync_check", "hc_status_string", "hc_launch_count", "hc_conv2d_bwd_depthwise_noalloc",
    "hc_pointwise_workspace_size", "hc_layernorm_c_fwd", "hc_layernorm_c_bwd", "hc_gelu_fwd", "hc_gelu_bwd",
    "hc_layerscale_residual_fwd", "hc_layerscale_residual_bwd", "hc_add_inplace", "hc_selftest_timeout",
    "hc_conv2d_step_graph_create", "hc_step_graph_launch", "hc_step_graph_destroy", "hc_drop_path_mask",
    "hc_layerscale_droppath_fwd", "hc_layerscale_droppath_bwd", "hc_shard_plan_rows", "hc_conv2d_bwd_reuse",
    "hc_conv2d_fwd_act", "hc_conv2d_bwd_act", "hc_conv2d_bwd_residual", "hc_trace_enable", "hc_trace_collect",
    "hc_halo_pad", "hc_halo_pack", "hc_halo_unpack", "hc_conv2d_fwd_rank", "hc_conv2d_bwd_rank",
    "hc_conv2d_workspace_size_rank", "hc_sum_partials", "hc_set_sm_count",
]


def hc_status_string(status: int) -> str:
    return _lib.hc_status_string(int(status)).decode()


def hc_shard_plan(d: hc_conv_desc):
    """Returns (status, [extent tuples], H_out, W_out)."""
    ext = (hc_shard_extent * max(1, d.num_shards))()
    ho, wo = C.c_int(0), C.c_int(0)
    st = _lib.hc_shard_plan(C.byref(d), ext, C.byref(ho), C.byref(wo))
    if st:
        return st, None, None, None
    return st, [tuple(getattr(e, f) for f, _ in hc_shard_extent._fields_) for e in ext[:d.num_shards]], ho.value, wo.value


def hc_shard_plan_rows(d: hc_conv_desc):
    """Returns (status, [row extent tuples])."""
    Sh = max(1, d.num_shards_h)
    ext = (hc_shard_extent * Sh)()
    st = _lib.hc_shard_plan_rows(C.byref(d), ext)
    if st:
        return st, None
    return st, [tuple(getattr(e, f) for f, _ in hc_shard_extent._fields_) for e in ext]


def hc_conv2d_workspace_size(d: hc_conv_desc, pass_: int, algo: int | None = None):
    """Returns (status, bytes)."""
    b = C.c_size_t(0)
    if algo is None:
        st = _lib.hc_conv2d_workspace_size(C.byref(d), pass_, C.byref(b))
    else:
        st = _lib.hc_conv2d_workspace_size_algo(C.byref(d), pass_, int(algo), C.byref(b))
    return st, b.value


def hc_conv2d_select(d: hc_conv_desc, pass_: int):
    a = C.c_int(0)
    st = _lib.hc_conv2d_select(C.byref(d), pass_, C.byref(a))
    return st, a.value


def hc_conv2d_fwd(d, x, w, bias, y, ws=None, ws_bytes=0, stream=None, algo=None) -> int:
    if algo is None:
        return _lib.hc_conv2d_fwd(C.byref(d), _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(ws), int(ws_bytes),
                                  _stream(stream))
    return _lib.hc_conv2d_fwd_algo(C.byref(d), _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(ws), int(ws_bytes),
                                   _stream(stream), int(algo))


def hc_conv2d_bwd(d, x, w, gy, gx, gw, gb, gw_partials=None, gb_partials=None, ws=None, ws_bytes=0, stream=None,
                  algo=None) -> int:
    args = [C.byref(d), _ptr(x), _ptr(w), _ptr(gy), _ptr(gx), _ptr(gw), _ptr(gb), _ptr(gw_partials),
            _ptr(gb_partials), _ptr(ws), int(ws_bytes), _stream(stream)]
    if algo is None:
        return _lib.hc_conv2d_bwd(*args)
    return _lib.hc_conv2d_bwd_algo(*args, int(algo))


def hc_conv2d_bwd_reuse(d, x, w, gy, gx, gw, gb, gw_partials=None, gb_partials=None, ws=None, ws_bytes=0,
                        fwd_ws=None, fwd_ws_bytes=0, stream=None, algo=None) -> int:
    """Backward pass reading x's operand copy from the forward workspace fwd_ws."""
    return _lib.hc_conv2d_bwd_reuse(C.byref(d), _ptr(x), _ptr(w), _ptr(gy), _ptr(gx), _ptr(gw), _ptr(gb),
                                    _ptr(gw_partials), _ptr(gb_partials), _ptr(ws), int(ws_bytes), _ptr(fwd_ws),
                                    int(fwd_ws_bytes), _stream(stream), int(algo or HC_ALGO_AUTO))


def hc_conv2d_bwd_residual(d, x, w, gy, residual, gx, gw, gb, gw_partials=None, gb_partials=None, ws=None,
                           ws_bytes=0, stream=None, algo=None) -> int:
    """Backward pass whose grad_input also receives a residual gradient: gx = grad_input + residual."""
    return _lib.hc_conv2d_bwd_residual(C.byref(d), _ptr(x), _ptr(w), _ptr(gy), _ptr(residual), _ptr(gx), _ptr(gw),
                                       _ptr(gb), _ptr(gw_partials), _ptr(gb_partials), _ptr(ws), int(ws_bytes),
                                       _stream(stream), int(algo or HC_ALGO_AUTO))


def hc_conv2d_fwd_act(d, x, w, b, y, ws=None, ws_bytes=0, stream=None, algo=None, act=HC_ACT_NONE) -> int:
    """Forward pass on act(x) (HC_ACT_GELU_INPUT: conv of GELU(x))."""
    return _lib.hc_conv2d_fwd_act(C.byref(d), _ptr(x), _ptr(w), _ptr(b), _ptr(y), _ptr(ws), int(ws_bytes),
                                  _stream(stream), int(algo or HC_ALGO_AUTO), int(act))


def hc_conv2d_bwd_act(d, x, w, gy, gx, gw, gb, gw_partials=None, gb_partials=None, ws=None, ws_bytes=0,
                      fwd_ws=None, fwd_ws_bytes=0, stream=None, algo=None, act=HC_ACT_NONE, y_pre=None) -> int:
    """Backward pass with a GELU on the input (gx w.r.t. GELU(x)) or on the output
    (gy w.r.t. GELU(y_pre); the pass runs on gy * GELU'(y_pre))."""
    return _lib.hc_conv2d_bwd_act(C.byref(d), _ptr(x), _ptr(w), _ptr(gy), _ptr(gx), _ptr(gw), _ptr(gb),
                                  _ptr(gw_partials), _ptr(gb_partials), _ptr(ws), int(ws_bytes), _ptr(fwd_ws),
                                  int(fwd_ws_bytes), _stream(stream), int(algo or HC_ALGO_AUTO), int(act),
                                  _ptr(y_pre))


def hc_conv2d_bwd_depthwise_noalloc(d, x, w, gy, gx, gw, gb, gw_partials=None, gb_partials=None,
                                    stream=None) -> int:
    """Depthwise backward with library-owned scratch: no workspace argument."""
    return _lib.hc_conv2d_bwd_depthwise_noalloc(C.byref(d), _ptr(x), _ptr(w), _ptr(gy), _ptr(gx), _ptr(gw),
                                                _ptr(gb), _ptr(gw_partials), _ptr(gb_partials), _stream(stream))


def hc_conv2d_step_graph_create(d, x, w, bias, y, gy, gx, gw, gb, ws_fwd, ws_fwd_bytes, ws_bwd, ws_bwd_bytes):
    """Returns (status, handle): one fwd + bwd step captured as a CUDA graph."""
    h = C.c_void_p(None)
    st = _lib.hc_conv2d_step_graph_create(C.byref(d), _ptr(x), _ptr(w), _ptr(bias), _ptr(y), _ptr(gy), _ptr(gx),
                                          _ptr(gw), _ptr(gb), _ptr(ws_fwd), int(ws_fwd_bytes), _ptr(ws_bwd),
                                          int(ws_bwd_bytes), C.byref(h))
    return st, h


def hc_step_graph_launch(h, stream=None) -> int:
    return _lib.hc_step_graph_launch(h, _stream(stream))


def hc_step_graph_destroy(h) -> int:
    return _lib.hc_step_graph_destroy(h)


def hc_drop_path_mask(N, drop_prob, seed, offset, mask, stream=None) -> int:
    return _lib.hc_drop_path_mask(int(N), float(drop_prob), int(seed), int(offset), _ptr(mask), _stream(stream))


def hc_layerscale_droppath_fwd(N, C_, HW, res, branch, gamma, mask, out, stream=None) -> int:
    return _lib.hc_layerscale_droppath_fwd(int(N), int(C_), int(HW), _ptr(res), _ptr(branch), _ptr(gamma), _ptr(mask),
                                           _ptr(out), _stream(stream))


def hc_layerscale_droppath_bwd(N, C_, HW, branch, gamma, mask, gy, gbranch, ggamma, ws, ws_bytes, stream=None) -> int:
    return _lib.hc_layerscale_droppath_bwd(int(N), int(C_), int(HW), _ptr(branch), _ptr(gamma), _ptr(mask), _ptr(gy),
                                           _ptr(gbranch), _ptr(ggamma), _ptr(ws), int(ws_bytes), _stream(stream))


def hc_halo_gather(d, x, x_ext, stream=None) -> int:
    return _lib.hc_halo_gather(C.byref(d), _ptr(x), _ptr(x_ext), _stream(stream))


def hc_pointwise_workspace_size(N, C_, HW):
    b = C.c_size_t(0)
    st = _lib.hc_pointwise_workspace_size(int(N), int(C_), int(HW), C.byref(b))
    return st, b.value


def hc_layernorm_c_fwd(N, C_, HW, x, gamma, beta, eps, y, mean=None, rstd=None, stream=None) -> int:
    return _lib.hc_layernorm_c_fwd(int(N), int(C_), int(HW), _ptr(x), _ptr(gamma), _ptr(beta), float(eps), _ptr(y),
                                   _ptr(mean), _ptr(rstd), _stream(stream))


def hc_layernorm_c_bwd(N, C_, HW, x, gamma, mean, rstd, gy, gx, ggamma=None, gbeta=None, ws=None, ws_bytes=0,
                       stream=None) -> int:
    return _lib.hc_layernorm_c_bwd(int(N), int(C_), int(HW), _ptr(x), _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(gy),
                                   _ptr(gx), _ptr(ggamma), _ptr(gbeta), _ptr(ws), int(ws_bytes), _stream(stream))


def hc_add_inplace(n, y, x, stream=None) -> int:
    return _lib.hc_add_inplace(int(n), _ptr(y), _ptr(x), _stream(stream))


def hc_gelu_fwd(n, x, y, stream=None) -> int:
    return _lib.hc_gelu_fwd(int(n), _ptr(x), _ptr(y), _stream(stream))


def hc_gelu_bwd(n, x, gy, gx, stream=None) -> int:
    return _lib.hc_gelu_bwd(int(n), _ptr(x), _ptr(gy), _ptr(gx), _stream(stream))


def hc_layerscale_residual_fwd(N, C_, HW, res, branch, gamma, out, stream=None) -> int:
    return _lib.hc_layerscale_residual_fwd(int(N), int(C_), int(HW), _ptr(res), _ptr(branch), _ptr(gamma), _ptr(out),
                                           _stream(stream))


def hc_layerscale_residual_bwd(N, C_, HW, branch, gamma, gy, gbranch, ggamma, ws, ws_bytes, stream=None) -> int:
    return _lib.hc_layerscale_residual_bwd(int(N), int(C_), int(HW), _ptr(branch), _ptr(gamma), _ptr(gy),
                                           _ptr(gbranch), _ptr(ggamma), _ptr(ws), int(ws_bytes), _stream(stream))


def hc_selftest_timeout(wait_us, stream=None) -> int:
    return _lib.hc_selftest_timeout(int(wait_us), _stream(stream))


def hc_sync_check(stream=None) -> int:
    return _lib.hc_sync_check(_stream(stream))


def hc_launch_count() -> int:
    return int(_lib.hc_launch_count())


_lib.hc_set_sm_count.argtypes = [C.c_int]
_lib.hc_set_sm_count.restype = C.c_int


def hc_set_sm_count(sms: int) -> int:
    return _lib.hc_set_sm_count(int(sms))


# ---- one rank of a multi-device layout (halo-padded blocks) -----------------
for _n, _a in (("hc_halo_pad", [_D, _P, _P, _P]), ("hc_halo_pack", [_D, _P, C.c_int, _P, _P]),
               ("hc_halo_unpack", [_D, _P, C.c_int, _P, _P]),
               ("hc_conv2d_fwd_rank", [_D, _P, _P, _P, _P, C.c_int, _P]),
               ("hc_conv2d_bwd_rank", [_D, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, C.c_int, _P]),
               ("hc_conv2d_workspace_size_rank", [_D, C.POINTER(C.c_size_t)]),
               ("hc_sum_partials", [_P, C.c_int, C.c_longlong, _P, _P])):
    getattr(_lib, _n).argtypes = _a
    getattr(_lib, _n).restype = C.c_int


def hc_halo_pad(d, x_local, x_pad, stream=None) -> int:
    return _lib.hc_halo_pad(C.byref(d), _ptr(x_local), _ptr(x_pad), _stream(stream))


def hc_halo_pack(d, x_pad, side, buf, stream=None) -> int:
    return _lib.hc_halo_pack(C.byref(d), _ptr(x_pad), int(side), _ptr(buf), _stream(stream))


def hc_halo_unpack(d, buf, side, x_pad, stream=None) -> int:
    return _lib.hc_halo_unpack(C.byref(d), _ptr(buf), int(side), _ptr(x_pad), _stream(stream))


def hc_conv2d_fwd_rank(d, x_pad, w, bias, y, tiles=HC_TILES_ALL, stream=None) -> int:
    return _lib.hc_conv2d_fwd_rank(C.byref(d), _ptr(x_pad), _ptr(w), _ptr(bias), _ptr(y), int(tiles), _stream(stream))


def hc_conv2d_workspace_size_rank(d):
    n = C.c_size_t(0)
    st = _lib.hc_conv2d_workspace_size_rank(C.byref(d), C.byref(n))
    return st, n.value


def hc_conv2d_bwd_rank(d, x_pad, w, gy_pad, gx, gw_part, gb_part, ws=None, ws_bytes=0, tiles=HC_TILES_ALL,
                       stream=None) -> int:
    return _lib.hc_conv2d_bwd_rank(C.byref(d), _ptr(x_pad), _ptr(w), _ptr(gy_pad), _ptr(gx), _ptr(gw_part),
                                   _ptr(gb_part), _ptr(ws), int(ws_bytes), int(tiles), _stream(stream))


def hc_sum_partials(parts, count, n, out, stream=None) -> int:
    return _lib.hc_sum_partials(_ptr(parts), int(count), int(n), _ptr(out), _stream(stream))


class hc_trace_entry(C.Structure):
    _fields_ = [("name", C.c_char * 48), ("launches", C.c_int), ("total_ms", C.c_double)]


_lib.hc_trace_enable.argtypes = [C.c_int]
_lib.hc_trace_enable.restype = C.c_int
_lib.hc_trace_collect.argtypes = [C.POINTER(hc_trace_entry), C.c_int, C.POINTER(C.c_int)]
_lib.hc_trace_collect.restype = C.c_int


def hc_trace_enable(on: bool) -> int:
    return _lib.hc_trace_enable(1 if on else 0)


def hc_trace_collect(max_entries: int = 256):
    """(status, {kernel name: (launches, total device ms)}) since the last collect."""
    arr = (hc_trace_entry * max_entries)()
    n = C.c_int(0)
    st = _lib.hc_trace_collect(arr, max_entries, C.byref(n))
    return st, {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(n.value)}


def check(status: int, what: str = "hc call") -> None:
    """Raise HcError unless status is HC_OK."""
    if status != HC_OK:
        raise HcError(status, what)
