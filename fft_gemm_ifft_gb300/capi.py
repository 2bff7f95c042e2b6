"""ctypes binding of the C ABI in ``include/fno.h`` -- argument marshalling only.

Every function here has the name of the C entry point it calls and returns
the raw ``fno_status_t`` (plus any out-parameters).  No arithmetic of the layer
happens in Python: the library's kernels do all of it.  If ``libfno.so`` has
not been built this module raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FNO_OK = 0
FNO_ERR_INVALID_ARG = 1
FNO_ERR_UNSUPPORTED = 2
FNO_ERR_MISALIGNED = 3
FNO_ERR_OUT_OF_MEMORY = 4
FNO_ERR_CUDA = 5
FNO_ERR_DEVICE_TIMEOUT = 6
FNO_ERR_DEVICE_BOUNDS = 7
FNO_ERR_ALIASING = 8

FNO_F32 = 0
FNO_F16 = 1
FNO_BF16 = 2
DTYPE_CODES = {"f32": FNO_F32, "f16": FNO_F16, "bf16": FNO_BF16}

FNO_PLAN_DEFAULT = 0
FNO_PLAN_UNFUSED = 1
FNO_PLAN_TRACE = 2
FNO_PLAN_PERSISTENT = 8
FNO_PLAN_BACKWARD = 16
FNO_PLAN_SIMT_MIX = 32
FNO_PLAN_SIMT_TRANSFORM = 64
FNO_PLAN_PACKED_WEIGHTS = 128
FNO_PLAN_TENSOR_EXTRA = 256
FNO_PLAN_SPLIT_LAYER = 512

# Every symbol include/fno.h declares.
EXPORTS = (
    "fno_status_string", "fno_version",
    "fno_spectral_conv_query", "fno_spectral_conv_plan",
    "fno_spectral_conv_query_padded", "fno_spectral_conv_plan_padded",
    "fno_spectral_conv_workspace_size", "fno_spectral_conv_kernel_count",
    "fno_spectral_conv_forward", "fno_plan_get_device_error", "fno_plan_destroy",
    "fno_spectral_conv_forward_static", "fno_plan_get_trace", "fno_spectral_conv_backward",
    "fno_spectral_conv_pack_weights", "fno_plan_check_bounded_wait",
    "fno_model_plan", "fno_model_workspace_size", "fno_model_kernel_count",
    "fno_forward", "fno_model_get_device_error", "fno_model_destroy",
)

_vp = ctypes.c_void_p
_st = ctypes.c_int


class fno_model_desc_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("cin_lift", ctypes.c_int32),
                ("width", ctypes.c_int32), ("nlayers", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("cout", ctypes.c_int32),
                ("h", ctypes.c_int64), ("w", ctypes.c_int64),
                ("modes", ctypes.c_int32 * 2), ("dtype", ctypes.c_int),
                ("flags", ctypes.c_uint32)]


class fno_trace_record_t(ctypes.Structure):
    _fields_ = [("item", ctypes.c_uint32), ("worker", ctypes.c_uint32),
                ("t_start", ctypes.c_uint64), ("t_ready", ctypes.c_uint64),
                ("t_compute", ctypes.c_uint64), ("t_end", ctypes.c_uint64)]


class fno_model_params_t(ctypes.Structure):
    _fields_ = [(name, _vp) for name in
                ("lift_w", "lift_b", "spec_w", "pw_w", "pw_b", "proj1_w", "proj1_b",
                 "proj2_w", "proj2_b")]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """libfno.so, or the index-checking build libfno_bounds.so when the
    environment sets FNO_LIBRARY=bounds (read once, at the first load)."""
    return _build.BOUNDS_LIB_PATH if os.environ.get("FNO_LIBRARY") == "bounds" else _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libfno.so (raises if it is missing; there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built; run fft_gemm_ifft_gb300.build.build() "
                    "(the CUDA library is required, there is no CPU path)")
            L = ctypes.CDLL(path)
            L.fno_status_string.argtypes = [_st]
            L.fno_status_string.restype = ctypes.c_char_p
            L.fno_version.restype = ctypes.c_int
            pi64, pi32, psz = (ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32),
                               ctypes.POINTER(ctypes.c_size_t))
            L.fno_spectral_conv_query.argtypes = [ctypes.c_int, pi64, pi32, ctypes.c_int64,
                                                  ctypes.c_int32, ctypes.c_int32, _st,
                                                  ctypes.c_uint32, psz, psz]
            L.fno_spectral_conv_plan.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, pi64, pi32,
                                                 ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                 _st, ctypes.c_uint32]
            L.fno_spectral_conv_query_padded.argtypes = [
                ctypes.c_int, pi64, pi64, pi32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                _st, ctypes.c_uint32, psz, psz]
            L.fno_spectral_conv_plan_padded.argtypes = [
                ctypes.POINTER(_vp), ctypes.c_int, pi64, pi64, pi32, ctypes.c_int64,
                ctypes.c_int32, ctypes.c_int32, _st, ctypes.c_uint32]
            L.fno_spectral_conv_workspace_size.argtypes = [_vp, psz]
            L.fno_spectral_conv_kernel_count.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
            L.fno_spectral_conv_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp]
            L.fno_spectral_conv_forward_static.argtypes = [
                ctypes.c_int, pi64, pi32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _st,
                _vp, _vp, _vp, _vp]
            L.fno_spectral_conv_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
            L.fno_spectral_conv_pack_weights.argtypes = [_vp, _vp, _vp, _vp]
            L.fno_plan_get_trace.argtypes = [_vp, ctypes.POINTER(fno_trace_record_t),
                                             ctypes.c_size_t, psz]
            L.fno_plan_get_device_error.argtypes = [_vp, _vp]
            L.fno_plan_check_bounded_wait.argtypes = [_vp, ctypes.c_int, _vp]
            L.fno_plan_destroy.argtypes = [_vp]
            L.fno_model_plan.argtypes = [ctypes.POINTER(_vp), ctypes.POINTER(fno_model_desc_t)]
            L.fno_model_workspace_size.argtypes = [_vp, psz]
            L.fno_model_kernel_count.argtypes = [_vp, ctypes.POINTER(ctypes.c_int)]
            L.fno_forward.argtypes = [_vp, _vp, ctypes.POINTER(fno_model_params_t), _vp, _vp, _vp]
            L.fno_model_get_device_error.argtypes = [_vp, _vp]
            L.fno_model_destroy.argtypes = [_vp]
            for name in EXPORTS[2:]:
                getattr(L, name).restype = _st
            _lib = L
    return _lib


def _arr(ctype, vals):
    vals = [int(v) for v in vals]
    return (ctype * max(1, len(vals)))(*vals)


def fno_status_string(status: int) -> str:
    return lib().fno_status_string(int(status)).decode()


def fno_version() -> int:
    return lib().fno_version()


def fno_spectral_conv_query(ndim, n, modes, batch, cin, cout, dtype, flags=0):
    ws, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib().fno_spectral_conv_query(int(ndim), _arr(ctypes.c_int64, n),
                                       _arr(ctypes.c_int32, modes), int(batch), int(cin),
                                       int(cout), int(dtype), int(flags),
                                       ctypes.byref(ws), ctypes.byref(wb))
    return st, ws.value, wb.value


def fno_spectral_conv_plan(ndim, n, modes, batch, cin, cout, dtype, flags=0):
    h = _vp(0)
    st = lib().fno_spectral_conv_plan(ctypes.byref(h), int(ndim), _arr(ctypes.c_int64, n),
                                      _arr(ctypes.c_int32, modes), int(batch), int(cin),
                                      int(cout), int(dtype), int(flags))
    return st, h.value


def fno_spectral_conv_query_padded(ndim, n, pad, modes, batch, cin, cout, dtype, flags=0):
    ws, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib().fno_spectral_conv_query_padded(
        int(ndim), _arr(ctypes.c_int64, n), None if pad is None else _arr(ctypes.c_int64, pad),
        _arr(ctypes.c_int32, modes), int(batch), int(cin), int(cout), int(dtype), int(flags),
        ctypes.byref(ws), ctypes.byref(wb))
    return st, ws.value, wb.value


def fno_spectral_conv_plan_padded(ndim, n, pad, modes, batch, cin, cout, dtype, flags=0):
    h = _vp(0)
    st = lib().fno_spectral_conv_plan_padded(
        ctypes.byref(h), int(ndim), _arr(ctypes.c_int64, n),
        None if pad is None else _arr(ctypes.c_int64, pad), _arr(ctypes.c_int32, modes),
        int(batch), int(cin), int(cout), int(dtype), int(flags))
    return st, h.value


def fno_spectral_conv_workspace_size(plan):
    v = ctypes.c_size_t(0)
    return lib().fno_spectral_conv_workspace_size(plan, ctypes.byref(v)), v.value


def fno_spectral_conv_kernel_count(plan):
    v = ctypes.c_int(0)
    return lib().fno_spectral_conv_kernel_count(plan, ctypes.byref(v)), v.value


def fno_spectral_conv_forward(plan, x_ptr, w_ptr, y_ptr, ws_ptr, stream):
    return lib().fno_spectral_conv_forward(plan, x_ptr, w_ptr, y_ptr, ws_ptr, stream)


def fno_spectral_conv_backward(plan, x_ptr, w_ptr, dy_ptr, dx_ptr, dw_ptr, ws_ptr, stream):
    return lib().fno_spectral_conv_backward(plan, x_ptr, w_ptr, dy_ptr, dx_ptr, dw_ptr, ws_ptr,
                                            stream)


def fno_spectral_conv_pack_weights(plan, w_ptr, wp_ptr, stream):
    return lib().fno_spectral_conv_pack_weights(plan, w_ptr, wp_ptr, stream)


def fno_spectral_conv_forward_static(ndim, n, modes, batch, cin, cout, dtype, x_ptr, w_ptr,
                                     y_ptr, stream):
    return lib().fno_spectral_conv_forward_static(
        int(ndim), _arr(ctypes.c_int64, n), _arr(ctypes.c_int32, modes), int(batch), int(cin),
        int(cout), int(dtype), x_ptr, w_ptr, y_ptr, stream)


def fno_plan_get_trace(plan, capacity=1 << 16):
    """Returns (status, list of (phase, group, index, worker, t_start, t_ready,
    t_compute, t_end))."""
    buf = (fno_trace_record_t * max(1, capacity))()
    n = ctypes.c_size_t(0)
    st = lib().fno_plan_get_trace(plan, buf, capacity, ctypes.byref(n))
    recs = []
    if st == FNO_OK:
        for r in buf[:min(n.value, capacity)]:
            recs.append((r.item >> 24, (r.item >> 16) & 0xFF, r.item & 0xFFFF, r.worker,
                         r.t_start, r.t_ready, r.t_compute, r.t_end))
    return st, recs


def fno_plan_get_device_error(plan, stream):
    return lib().fno_plan_get_device_error(plan, stream)


def fno_plan_check_bounded_wait(plan, which, stream):
    return lib().fno_plan_check_bounded_wait(plan, int(which), stream)


def fno_plan_destroy(plan):
    return lib().fno_plan_destroy(plan)


def fno_model_plan(desc: fno_model_desc_t):
    h = _vp(0)
    st = lib().fno_model_plan(ctypes.byref(h), ctypes.byref(desc))
    return st, h.value


def fno_model_workspace_size(model):
    v = ctypes.c_size_t(0)
    return lib().fno_model_workspace_size(model, ctypes.byref(v)), v.value


def fno_model_kernel_count(model):
    v = ctypes.c_int(0)
    return lib().fno_model_kernel_count(model, ctypes.byref(v)), v.value


def fno_forward(model, x_ptr, params: fno_model_params_t, out_ptr, ws_ptr, stream):
    return lib().fno_forward(model, x_ptr, ctypes.byref(params), out_ptr, ws_ptr, stream)


def fno_model_get_device_error(model, stream):
    return lib().fno_model_get_device_error(model, stream)


def fno_model_destroy(model):
    return lib().fno_model_destroy(model)
