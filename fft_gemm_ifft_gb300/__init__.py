"""GB300 (sm_103a) Fourier Neural Operator spectral-convolution library.

The compute lives in ``libfno.so`` (hand-written CUDA, C ABI in
``include/fno.h``).  This package only marshals arguments: ``capi`` mirrors
the C entry points one to one, and the two small classes below hold a plan
plus a torch-allocated workspace and pass tensor pointers and the current
stream to the library.  PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

from . import capi
from .capi import (FNO_BF16, FNO_F16, FNO_F32, FNO_PLAN_DEFAULT,  # noqa: F401
                   FNO_PLAN_UNFUSED, fno_status_string)

__all__ = ["capi", "FnoError", "SpectralConv", "FnoModel", "check"]


class FnoError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {fno_status_string(status)}" if what
                         else fno_status_string(status))


def check(status: int, what: str = "") -> None:
    if status != capi.FNO_OK:
        raise FnoError(status, what)


def _stream_handle(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _require(t, dtype, shape, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class SpectralConv:
    """One spectral-convolution plan and its workspace on the current device.

    ``w`` is passed as the real view of the interleaved complex weights,
    shape (nblk, cin, cout, m..., 2), in the storage dtype.  ``pad`` (one
    entry per axis) makes the layer non-periodic: x is read as if followed by
    that many zeros per axis, the transform runs over n + pad points and y
    keeps the first n (``fno_spectral_conv_plan_padded``).
    """

    def __init__(self, n, modes, batch, cin, cout, dtype="f32", flags=0, pad=None):
        import torch
        self.n, self.modes = tuple(int(v) for v in n), tuple(int(v) for v in modes)
        self.batch, self.cin, self.cout = int(batch), int(cin), int(cout)
        self.dtype = dtype
        self.pad = None if pad is None else tuple(int(v) for v in pad)
        self.torch_dtype = {"f32": torch.float32, "f16": torch.float16,
                            "bf16": torch.bfloat16}[dtype]
        code = capi.DTYPE_CODES[dtype]
        if self.pad is None:
            st, self.handle = capi.fno_spectral_conv_plan(len(self.n), self.n, self.modes,
                                                          batch, cin, cout, code, flags)
        else:
            st, self.handle = capi.fno_spectral_conv_plan_padded(
                len(self.n), self.n, self.pad, self.modes, batch, cin, cout, code, flags)
        check(st, "fno_spectral_conv_plan")
        st, self.workspace_bytes = capi.fno_spectral_conv_workspace_size(self.handle)
        check(st)
        st, self.kernel_count = capi.fno_spectral_conv_kernel_count(self.handle)
        check(st)
        self.workspace = (torch.empty(self.workspace_bytes, dtype=torch.uint8, device="cuda")
                          if self.workspace_bytes else None)
        nblk = 2 ** (len(self.n) - 1)
        self.x_shape = (self.batch, self.cin) + self.n
        self.y_shape = (self.batch, self.cout) + self.n
        self.w_shape = (nblk, self.cin, self.cout) + self.modes + (2,)

    def forward(self, x, w, y=None, stream=None):
        import torch
        _require(x, self.torch_dtype, self.x_shape, "x")
        _require(w, self.torch_dtype, self.w_shape, "w")
        if y is None:
            y = torch.empty(self.y_shape, dtype=self.torch_dtype, device=x.device)
        _require(y, self.torch_dtype, self.y_shape, "y")
        ws = self.workspace.data_ptr() if self.workspace is not None else None
        check(capi.fno_spectral_conv_forward(self.handle, x.data_ptr(), w.data_ptr(),
                                             y.data_ptr(), ws, _stream_handle(stream)),
              "fno_spectral_conv_forward")
        return y

    __call__ = forward

    def pack_weights(self, w, out=None, stream=None):
        """The packed copy of w for a plan made with FNO_PLAN_PACKED_WEIGHTS
        (pass it to forward in place of w)."""
        import torch
        _require(w, self.torch_dtype, self.w_shape, "w")
        if out is None:
            out = torch.empty_like(w)
        _require(out, self.torch_dtype, self.w_shape, "out")
        check(capi.fno_spectral_conv_pack_weights(self.handle, w.data_ptr(), out.data_ptr(),
                                                  _stream_handle(stream)),
              "fno_spectral_conv_pack_weights")
        return out

    def backward(self, x, w, dy, need_dx=True, need_dw=True, dx=None, dw=None, stream=None):
        """Gradients (dx, dw) of a real loss given dy = dL/dy; the plan must have
        been made with FNO_PLAN_BACKWARD.  dw is dL/dRe(w) + i dL/dIm(w) in w's
        interleaved layout.  Either may be skipped (returned as None)."""
        import torch
        _require(dy, self.torch_dtype, self.y_shape, "dy")
        if need_dx:
            _require(w, self.torch_dtype, self.w_shape, "w")
            if dx is None:
                dx = torch.empty(self.x_shape, dtype=self.torch_dtype, device=dy.device)
            _require(dx, self.torch_dtype, self.x_shape, "dx")
        if need_dw:
            _require(x, self.torch_dtype, self.x_shape, "x")
            if dw is None:
                dw = torch.empty(self.w_shape, dtype=self.torch_dtype, device=dy.device)
            _require(dw, self.torch_dtype, self.w_shape, "dw")
        ptr = lambda t: t.data_ptr() if t is not None else None
        ws = self.workspace.data_ptr() if self.workspace is not None else None
        check(capi.fno_spectral_conv_backward(
            self.handle, ptr(x) if need_dw else None, ptr(w) if need_dx else None, dy.data_ptr(),
            ptr(dx) if need_dx else None, ptr(dw) if need_dw else None, ws,
            _stream_handle(stream)), "fno_spectral_conv_backward")
        return (dx if need_dx else None), (dw if need_dw else None)

    def device_error(self, stream=None) -> int:
        return capi.fno_plan_get_device_error(self.handle, _stream_handle(stream))

    def close(self):
        if getattr(self, "handle", None):
            check(capi.fno_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class FnoModel:
    """The 2-D FNO forward stack (lift, spectral layers, projection)."""

    PARAM_NAMES = ("lift_w", "lift_b", "spec_w", "pw_w", "pw_b", "proj1_w", "proj1_b",
                   "proj2_w", "proj2_b")

    def __init__(self, batch, h, w, modes=(16, 16), cin_lift=3, width=64, nlayers=4,
                 hidden=128, cout=1, flags=0, dtype="f32"):
        import torch
        d = capi.fno_model_desc_t()
        d.batch, d.cin_lift, d.width, d.nlayers = batch, cin_lift, width, nlayers
        d.hidden, d.cout, d.h, d.w = hidden, cout, h, w
        d.modes[0], d.modes[1] = modes
        d.dtype, d.flags = capi.DTYPE_CODES[dtype], flags
        self.dtype = dtype
        # x, the activations, spec_w and out in the storage type; 1x1 weights float32
        self.torch_dtype = {"f32": torch.float32, "f16": torch.float16,
                            "bf16": torch.bfloat16}[dtype]
        self.desc = d
        st, self.handle = capi.fno_model_plan(d)
        check(st, "fno_model_plan")
        st, self.workspace_bytes = capi.fno_model_workspace_size(self.handle)
        check(st)
        st, self.kernel_count = capi.fno_model_kernel_count(self.handle)
        check(st)
        self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device="cuda")
        self.x_shape = (batch, cin_lift, h, w)
        self.y_shape = (batch, cout, h, w)
        self.shapes = {
            "lift_w": (width, cin_lift), "lift_b": (width,),
            "spec_w": (nlayers, 2, width, width) + tuple(modes) + (2,),
            "pw_w": (nlayers, width, width), "pw_b": (nlayers, width),
            "proj1_w": (hidden, width), "proj1_b": (hidden,),
            "proj2_w": (cout, hidden), "proj2_b": (cout,),
        }

    def forward(self, x, params: dict, out=None, stream=None):
        import torch
        _require(x, self.torch_dtype, self.x_shape, "x")
        p = capi.fno_model_params_t()
        for k in self.PARAM_NAMES:
            want = self.torch_dtype if k == "spec_w" else torch.float32
            _require(params[k], want, self.shapes[k], k)
            setattr(p, k, params[k].data_ptr())
        if out is None:
            out = torch.empty(self.y_shape, dtype=self.torch_dtype, device=x.device)
        _require(out, self.torch_dtype, self.y_shape, "out")
        check(capi.fno_forward(self.handle, x.data_ptr(), p, out.data_ptr(),
                               self.workspace.data_ptr(), _stream_handle(stream)), "fno_forward")
        return out

    __call__ = forward

    def device_error(self, stream=None) -> int:
        return capi.fno_model_get_device_error(self.handle, _stream_handle(stream))

    def close(self):
        if getattr(self, "handle", None):
            check(capi.fno_model_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
