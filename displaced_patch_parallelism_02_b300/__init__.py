"""Python binding of libdpp.so, the displaced-patch-parallelism hot path on one B300.

Argument marshalling only: every entry point has the name and argument order
of the C ABI in include/dpp.h and forwards to it through ctypes.  Tensor
arguments may be torch tensors (their data_ptr() is passed) or raw integer
device pointers; ``stream`` defaults to torch's current CUDA stream.  All
compute runs in the library's CUDA kernels.  There is no other code path:
importing this package fails when libdpp.so has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdpp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python displaced_patch_parallelism_02_b300/build.py` (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------------ enums
DPP_OK = 0
DPP_ERR_INVALID_ARG = 1
DPP_ERR_UNSUPPORTED = 2
DPP_ERR_ALIAS = 3
DPP_ERR_WORKSPACE = 4
DPP_ERR_CUDA = 5
DPP_ERR_TIMEOUT = 6
DPP_ERR_ALIGN = 7
DPP_ERR_RANGE = 8

DPP_F32 = 0
DPP_BF16 = 1

DPP_HALO_STALE = 0
DPP_HALO_FRESH = 1
DPP_HALO_ZERO = 2

DPP_ACT_NONE = 0
DPP_ACT_SILU = 1

DPP_EPI_NONE = 0
DPP_EPI_GEGLU = 1

DPP_OP_CONV3X3 = 0
DPP_OP_GROUPNORM = 1
DPP_OP_SELF_ATTN = 2
DPP_OP_CROSS_ATTN = 3
DPP_OP_CFG_COMBINE = 4
DPP_OP_REFRESH_STALE = 5


class DppError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dpp_status_string(status)}")


# ------------------------------------------------------------ descriptors
class dpp_conv_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("C_in", ctypes.c_int), ("C_out", ctypes.c_int), ("P", ctypes.c_int),
                ("dtype", ctypes.c_int), ("halo", ctypes.c_int), ("accumulate", ctypes.c_int)]


class dpp_gn_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("C", ctypes.c_int), ("G", ctypes.c_int), ("P", ctypes.c_int),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int), ("band_local", ctypes.c_int),
                ("act", ctypes.c_int)]


class dpp_attn_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("C", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("P", ctypes.c_int), ("n_ctx", ctypes.c_int), ("c_ctx", ctypes.c_int),
                ("dtype", ctypes.c_int), ("band_local", ctypes.c_int),
                ("accumulate", ctypes.c_int)]


class dpp_ln_desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("C", ctypes.c_int), ("eps", ctypes.c_float),
                ("dtype", ctypes.c_int)]


class dpp_linear_desc(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("K", ctypes.c_int), ("N", ctypes.c_int),
                ("dtype", ctypes.c_int), ("epilogue", ctypes.c_int), ("accumulate", ctypes.c_int)]


class dpp_switch_state(ctypes.Structure):
    _fields_ = [("flat_tol", ctypes.c_double), ("rise_tol", ctypes.c_double),
                ("patience", ctypes.c_int), ("stage", ctypes.c_int), ("run", ctypes.c_int),
                ("steps", ctypes.c_int), ("prev", ctypes.c_double), ("min_d", ctypes.c_double)]


DPP_STAGE_WARMUP = 0
DPP_STAGE_PARALLEL = 1
DPP_STAGE_FULLY_CONNECTING = 2

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_st = ctypes.c_int

_SIGNATURES = {
    "dpp_conv3x3": (_st, [ctypes.POINTER(dpp_conv_desc), _vp, _vp, _vp, _vp, _vp, _vp]),
    "dpp_groupnorm": (_st, [ctypes.POINTER(dpp_gn_desc), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _sz, _vp]),
    "dpp_groupnorm_workspace_bytes": (_sz, [ctypes.POINTER(dpp_gn_desc)]),
    "dpp_conv3x3_gn": (_st, [ctypes.POINTER(dpp_conv_desc), _vp, _vp, _vp, _vp, _vp,
                             ctypes.c_int, _vp, _vp]),
    "dpp_groupnorm_apply": (_st, [ctypes.POINTER(dpp_gn_desc), _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp]),
    "dpp_groupnorm_static": (_st, [ctypes.POINTER(dpp_gn_desc), _vp, _vp, _vp, _vp, _vp, _vp,
                                   _vp]),
    "dpp_groupnorm_sums": (_st, [ctypes.POINTER(dpp_gn_desc), _vp, _vp, _vp]),
    "dpp_groupnorm_affine": (_st, [ctypes.POINTER(dpp_gn_desc), _vp, _vp, _vp, _vp, _vp, _vp,
                                   _vp]),
    "dpp_conv3x3_norm": (_st, [ctypes.POINTER(dpp_conv_desc), _vp, _vp, _vp, _vp, ctypes.c_int,
                               _vp, _vp, _vp, ctypes.c_int, _vp, _vp]),
    "dpp_self_attn": (_st, [ctypes.POINTER(dpp_attn_desc), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp, _vp, _sz, _vp]),
    "dpp_self_attn_workspace_bytes": (_sz, [ctypes.POINTER(dpp_attn_desc)]),
    "dpp_cross_attn": (_st, [ctypes.POINTER(dpp_attn_desc), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                             _vp, _sz, _vp]),
    "dpp_cross_attn_workspace_bytes": (_sz, [ctypes.POINTER(dpp_attn_desc)]),
    "dpp_cross_attn_kv": (_st, [ctypes.POINTER(dpp_attn_desc), _vp, _vp, _vp, _vp, _vp]),
    "dpp_cross_attn_cached": (_st, [ctypes.POINTER(dpp_attn_desc), _vp, _vp, _vp, _vp, _vp, _vp,
                                    _sz, _vp]),
    "dpp_cross_attn_cached_workspace_bytes": (_sz, [ctypes.POINTER(dpp_attn_desc)]),
    "dpp_cfg_combine": (_st, [_vp, _vp, ctypes.c_float, _sz, _vp, _vp, _vp, _sz, _vp]),
    "dpp_cfg_workspace_bytes": (_sz, [_sz]),
    "dpp_refresh_stale": (_st, [_vp, _vp, _sz, _sz, _sz, ctypes.c_int, ctypes.c_uint64, _vp]),
    "dpp_refresh_halo": (_st, [_vp, _vp, _sz, _sz, _sz, ctypes.c_int, _vp]),
    "dpp_device_status": (_st, [_vp]),
    "dpp_status_string": (ctypes.c_char_p, [_st]),
    "dpp_version": (ctypes.c_int, []),
    "dpp_source_hash": (ctypes.c_char_p, []),
    "dpp_launch_count": (ctypes.c_uint64, []),
    "dpp_set_attn_core_events": (None, [_vp, _vp]),
    "dpp_workspace_bytes": (_sz, [ctypes.c_int, _vp]),
    "dpp_wait_selftest": (_st, [ctypes.c_int, _vp, _vp]),
    "dpp_layernorm": (_st, [ctypes.POINTER(dpp_ln_desc), _vp, _vp, _vp, _vp, _vp]),
    "dpp_linear": (_st, [ctypes.POINTER(dpp_linear_desc), _vp, _vp, _vp, _vp, _vp]),
    "dpp_switch_init": (None, [ctypes.POINTER(dpp_switch_state), ctypes.c_double,
                               ctypes.c_double, ctypes.c_int]),
    "dpp_switch_update": (ctypes.c_int, [ctypes.POINTER(dpp_switch_state), ctypes.c_double]),
}

for _name, (_res, _args) in _SIGNATURES.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


# ---------------------------------------------------------------- helpers
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t or None
    return t.data_ptr() or None


def _stream(stream):
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream or None
        return None
    if isinstance(stream, int):
        return stream or None
    return getattr(stream, "cuda_stream", stream) or None


def _check(status: int, where: str, raise_on_error: bool):
    if raise_on_error and status != DPP_OK:
        raise DppError(status, where)
    return status


def dpp_status_string(status: int) -> str:
    return lib.dpp_status_string(int(status)).decode()


def dpp_version() -> int:
    return lib.dpp_version()


def dpp_source_hash() -> str:
    return lib.dpp_source_hash().decode()


def dpp_launch_count() -> int:
    return lib.dpp_launch_count()


def dpp_set_attn_core_events(start, stop) -> None:
    """start/stop: torch.cuda.Event (recorded by the library) or None."""
    lib.dpp_set_attn_core_events(None if start is None else start.cuda_event,
                                 None if stop is None else stop.cuda_event)


def dpp_switch_init(state: dpp_switch_state, flat_tol: float, rise_tol: float,
                    patience: int) -> None:
    lib.dpp_switch_init(ctypes.byref(state), float(flat_tol), float(rise_tol), int(patience))


def dpp_switch_update(state: dpp_switch_state, d: float) -> int:
    return lib.dpp_switch_update(ctypes.byref(state), float(d))


def dpp_device_status(stream=None) -> int:
    return lib.dpp_device_status(_stream(stream))


# ------------------------------------------------------------ entry points
def dpp_conv3x3(desc: dpp_conv_desc, x, stale_prev, w, bias, y, stream=None,
                raise_on_error: bool = True) -> int:
    return _check(lib.dpp_conv3x3(ctypes.byref(desc), _ptr(x), _ptr(stale_prev), _ptr(w),
                                  _ptr(bias), _ptr(y), _stream(stream)),
                  "dpp_conv3x3", raise_on_error)


def dpp_conv3x3_gn(desc: dpp_conv_desc, x, stale_prev, w, bias, y, G: int, gn_sums,
                   stream=None, raise_on_error: bool = True) -> int:
    return _check(lib.dpp_conv3x3_gn(ctypes.byref(desc), _ptr(x), _ptr(stale_prev), _ptr(w),
                                     _ptr(bias), _ptr(y), int(G), _ptr(gn_sums),
                                     _stream(stream)),
                  "dpp_conv3x3_gn", raise_on_error)


def dpp_groupnorm_apply(desc: dpp_gn_desc, x, stats_prev, gn_sums, stats_next, gamma, beta, y,
                        stream=None, raise_on_error: bool = True) -> int:
    return _check(lib.dpp_groupnorm_apply(ctypes.byref(desc), _ptr(x), _ptr(stats_prev),
                                          _ptr(gn_sums), _ptr(stats_next), _ptr(gamma),
                                          _ptr(beta), _ptr(y), _stream(stream)),
                  "dpp_groupnorm_apply", raise_on_error)


def dpp_groupnorm_sums(desc: dpp_gn_desc, x, gn_sums, stream=None,
                       raise_on_error: bool = True) -> int:
    return _check(lib.dpp_groupnorm_sums(ctypes.byref(desc), _ptr(x), _ptr(gn_sums),
                                         _stream(stream)),
                  "dpp_groupnorm_sums", raise_on_error)


def dpp_groupnorm_affine(desc: dpp_gn_desc, gn_sums, stats_prev, stats_next, gamma, beta,
                         affine, stream=None, raise_on_error: bool = True) -> int:
    return _check(lib.dpp_groupnorm_affine(ctypes.byref(desc), _ptr(gn_sums), _ptr(stats_prev),
                                           _ptr(stats_next), _ptr(gamma), _ptr(beta),
                                           _ptr(affine), _stream(stream)),
                  "dpp_groupnorm_affine", raise_on_error)


def dpp_conv3x3_norm(desc: dpp_conv_desc, x, stale_prev, affine, affine_prev, act: int, w, bias,
                     y, G: int = 0, gn_sums=None, stream=None,
                     raise_on_error: bool = True) -> int:
    return _check(lib.dpp_conv3x3_norm(ctypes.byref(desc), _ptr(x), _ptr(stale_prev),
                                       _ptr(affine), _ptr(affine_prev), int(act), _ptr(w),
                                       _ptr(bias), _ptr(y), int(G), _ptr(gn_sums),
                                       _stream(stream)),
                  "dpp_conv3x3_norm", raise_on_error)


def dpp_wait_selftest(kind: int, scratch=None, stream=None, raise_on_error: bool = True) -> int:
    return _check(lib.dpp_wait_selftest(int(kind), _ptr(scratch), _stream(stream)),
                  "dpp_wait_selftest", raise_on_error)


def dpp_workspace_bytes(op: int, desc) -> int:
    """desc: the op's descriptor (a ctypes structure) or, for
    DPP_OP_CFG_COMBINE, the element count n."""
    if isinstance(desc, int):
        arg = ctypes.byref(ctypes.c_size_t(desc))
    else:
        arg = ctypes.byref(desc)
    return lib.dpp_workspace_bytes(int(op), ctypes.cast(arg, _vp))


def dpp_layernorm(desc: dpp_ln_desc, x, gamma, beta, y, stream=None,
                  raise_on_error: bool = True) -> int:
    return _check(lib.dpp_layernorm(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(beta),
                                    _ptr(y), _stream(stream)),
                  "dpp_layernorm", raise_on_error)


def dpp_linear(desc: dpp_linear_desc, x, w, bias, y, stream=None,
               raise_on_error: bool = True) -> int:
    return _check(lib.dpp_linear(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(y),
                                 _stream(stream)),
                  "dpp_linear", raise_on_error)


def dpp_groupnorm_workspace_bytes(desc: dpp_gn_desc) -> int:
    return lib.dpp_groupnorm_workspace_bytes(ctypes.byref(desc))


def dpp_groupnorm(desc: dpp_gn_desc, x, stats_prev, stats_next, gamma, beta, y, ws, ws_bytes,
                  stream=None, raise_on_error: bool = True) -> int:
    return _check(lib.dpp_groupnorm(ctypes.byref(desc), _ptr(x), _ptr(stats_prev),
                                    _ptr(stats_next), _ptr(gamma), _ptr(beta), _ptr(y),
                                    _ptr(ws), int(ws_bytes), _stream(stream)),
                  "dpp_groupnorm", raise_on_error)


DPP_GN_STATIC_SCRATCH_BYTES = 1 << 20


def dpp_groupnorm_static(desc: dpp_gn_desc, x, stats_prev, stats_next, gamma, beta, y,
                         stream=None, raise_on_error: bool = True) -> int:
    """dpp_groupnorm with its scratch in the library's static device array
    (for callers that cannot allocate; see include/dpp.h)."""
    return _check(lib.dpp_groupnorm_static(ctypes.byref(desc), _ptr(x), _ptr(stats_prev),
                                           _ptr(stats_next), _ptr(gamma), _ptr(beta), _ptr(y),
                                           _stream(stream)),
                  "dpp_groupnorm_static", raise_on_error)


def dpp_self_attn_workspace_bytes(desc: dpp_attn_desc) -> int:
    return lib.dpp_self_attn_workspace_bytes(ctypes.byref(desc))


def dpp_self_attn(desc: dpp_attn_desc, x, wq, wk, wv, wo, kv_prev, kv_next, y, ws, ws_bytes,
                  stream=None, raise_on_error: bool = True) -> int:
    return _check(lib.dpp_self_attn(ctypes.byref(desc), _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv),
                                    _ptr(wo), _ptr(kv_prev), _ptr(kv_next), _ptr(y), _ptr(ws),
                                    int(ws_bytes), _stream(stream)),
                  "dpp_self_attn", raise_on_error)


def dpp_cross_attn_workspace_bytes(desc: dpp_attn_desc) -> int:
    return lib.dpp_cross_attn_workspace_bytes(ctypes.byref(desc))


def dpp_cross_attn(desc: dpp_attn_desc, x, ctx, wq, wk, wv, wo, y, ws, ws_bytes, stream=None,
                   raise_on_error: bool = True) -> int:
    return _check(lib.dpp_cross_attn(ctypes.byref(desc), _ptr(x), _ptr(ctx), _ptr(wq),
                                     _ptr(wk), _ptr(wv), _ptr(wo), _ptr(y), _ptr(ws),
                                     int(ws_bytes), _stream(stream)),
                  "dpp_cross_attn", raise_on_error)


def dpp_cross_attn_kv(desc: dpp_attn_desc, ctx, wk, wv, kv_ctx, stream=None,
                      raise_on_error: bool = True) -> int:
    return _check(lib.dpp_cross_attn_kv(ctypes.byref(desc), _ptr(ctx), _ptr(wk), _ptr(wv),
                                        _ptr(kv_ctx), _stream(stream)),
                  "dpp_cross_attn_kv", raise_on_error)


def dpp_cross_attn_cached_workspace_bytes(desc: dpp_attn_desc) -> int:
    return lib.dpp_cross_attn_cached_workspace_bytes(ctypes.byref(desc))


def dpp_cross_attn_cached(desc: dpp_attn_desc, x, kv_ctx, wq, wo, y, ws, ws_bytes, stream=None,
                          raise_on_error: bool = True) -> int:
    return _check(lib.dpp_cross_attn_cached(ctypes.byref(desc), _ptr(x), _ptr(kv_ctx), _ptr(wq),
                                            _ptr(wo), _ptr(y), _ptr(ws), int(ws_bytes),
                                            _stream(stream)),
                  "dpp_cross_attn_cached", raise_on_error)


def dpp_cfg_workspace_bytes(n: int) -> int:
    return lib.dpp_cfg_workspace_bytes(int(n))


def dpp_cfg_combine(eps_u, eps_c, scale: float, n: int, out, sums3, ws, ws_bytes, stream=None,
                    raise_on_error: bool = True) -> int:
    return _check(lib.dpp_cfg_combine(_ptr(eps_u), _ptr(eps_c), float(scale), int(n), _ptr(out),
                                      _ptr(sums3), _ptr(ws), int(ws_bytes), _stream(stream)),
                  "dpp_cfg_combine", raise_on_error)


def dpp_refresh_stale(fresh, stale, outer: int, rows: int, row_bytes: int, P: int,
                      patch_mask: int = (1 << 64) - 1, stream=None,
                      raise_on_error: bool = True) -> int:
    return _check(lib.dpp_refresh_stale(_ptr(fresh), _ptr(stale), int(outer), int(rows),
                                        int(row_bytes), int(P), int(patch_mask) & ((1 << 64) - 1),
                                        _stream(stream)),
                  "dpp_refresh_stale", raise_on_error)


def dpp_refresh_halo(fresh, stale, outer: int, rows: int, row_bytes: int, P: int, stream=None,
                     raise_on_error: bool = True) -> int:
    return _check(lib.dpp_refresh_halo(_ptr(fresh), _ptr(stale), int(outer), int(rows),
                                       int(row_bytes), int(P), _stream(stream)),
                  "dpp_refresh_halo", raise_on_error)


__all__ = [n for n in dir() if n.startswith(("dpp_", "DPP_"))] + ["DppError", "lib", "LIB_PATH"]
