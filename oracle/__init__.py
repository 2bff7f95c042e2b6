"""Float64 CPU oracle for the FNO spectral-convolution layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline / reference arm may import this package.  It shares no code with the
CUDA library in ``fft_gemm_ifft_gb300``; the two meet only in the seeded input
generators of ``fft_gemm_ifft_gb300.workloads`` (which hold no FFT or mixing
arithmetic).

The arithmetic lives in ``fno_oracle.c`` (plain C, double precision, libm
cos/sin/erf, OpenMP over independent images).  This module compiles it with
gcc and marshals numpy arrays into it.  What each function follows in the
TurboFNO article (gsyq.cn/news/457482):

* ``forward_modes``  -- §2.1, real FFT over the spatial axes, truncated to the
  kept modes (low and high rows on full axes, low bins on the half axis);
* ``mix``            -- §2.2, per-mode complex contraction over input channels;
* ``inverse_modes``  -- §2.3 / §3.3, zero-padded inverse real FFT;
* ``spectral_conv``  -- the three in order;
* ``spectral_conv_padded`` -- §2.3 / §3.3, the layer on a zero-padded domain
  with the output cropped back to the input's extents;
* ``spectral_conv_backward`` -- dL/dx and dL/dw of the layer for a real loss,
  the derivatives of the three steps above (the pages print no backward pass);
* ``adjoint_modes``  -- the adjoint of ``forward_modes`` (used by the above);
* ``fno_forward``    -- the lift / 4 x (spectral conv + 1x1 linear, GELU) /
  projection stack of the 2-D FNO workload.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
brute-force DFTs, closed forms, numpy.fft and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fno_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE double, no fast-math) and return the path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.fno_oracle_fft.argtypes = [_f64p, _f64p, ctypes.c_int64, ctypes.c_int]
            lib.fno_oracle_fft.restype = None
            sig = [ctypes.c_int, _i64p, _i32p]
            lib.fno_oracle_forward_modes.argtypes = sig + [ctypes.c_int64, _f64p, _f64p]
            lib.fno_oracle_inverse_modes.argtypes = sig + [ctypes.c_int64, _f64p, _f64p]
            lib.fno_oracle_mix.argtypes = sig + [ctypes.c_int64] * 3 + [_f64p] * 3
            lib.fno_oracle_spectral_conv.argtypes = sig + [ctypes.c_int64] * 3 + [_f64p] * 3
            lib.fno_oracle_fno_forward.argtypes = (
                [ctypes.c_int64] * 3 + [_i32p] + [ctypes.c_int64] * 5 + [_f64p] * 11)
            lib.fno_oracle_adjoint_modes.argtypes = sig + [ctypes.c_int64, _f64p, _f64p]
            lib.fno_oracle_spectral_conv_backward.argtypes = (
                sig + [ctypes.c_int64] * 3 + [_f64p] * 5)
            for f in ("forward_modes", "inverse_modes", "mix", "spectral_conv", "fno_forward",
                      "adjoint_modes", "spectral_conv_backward"):
                getattr(lib, "fno_oracle_" + f).restype = ctypes.c_int
            lib.fno_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.fno_oracle_get_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _d(a: np.ndarray):
    return a.ctypes.data_as(_f64p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _geom(n, modes):
    n = np.ascontiguousarray(n, dtype=np.int64)
    m = np.ascontiguousarray(modes, dtype=np.int32)
    if n.shape != m.shape or not 1 <= n.size <= 3:
        raise ValueError("n and modes must have the same length 1..3")
    return n, m


def kept_shape(n, modes):
    """Extent of the kept-mode array per axis: 2m on full axes, m on the half axis."""
    n, m = _geom(n, modes)
    return tuple(int(2 * v) for v in m[:-1]) + (int(m[-1]),)


def set_threads(nthreads: int) -> None:
    _load().fno_oracle_set_threads(int(nthreads))


def get_threads() -> int:
    return int(_load().fno_oracle_get_threads())


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def fft(z: np.ndarray, inverse: bool = False) -> np.ndarray:
    """1-D radix-2 complex FFT (unnormalised both ways) of a complex vector."""
    z = np.asarray(z, dtype=np.complex128)
    re = np.ascontiguousarray(z.real.copy())
    im = np.ascontiguousarray(z.imag.copy())
    _load().fno_oracle_fft(_d(re), _d(im), re.size, 1 if inverse else -1)
    return re + 1j * im


def forward_modes(x: np.ndarray, modes) -> np.ndarray:
    """x (..., N_0..N_{d-1}) real -> kept modes (..., K_0..K_{d-1}) complex128."""
    d = len(modes)
    x = _f64(x)
    n, m = _geom(x.shape[-d:], modes)
    lead = x.shape[:-d]
    nimg = int(np.prod(lead, dtype=np.int64))
    kshape = kept_shape(n, m)
    out = np.empty((nimg,) + kshape + (2,), dtype=np.float64)
    _check(_load().fno_oracle_forward_modes(
        d, n.ctypes.data_as(_i64p), m.ctypes.data_as(_i32p), nimg, _d(x), _d(out)),
        "forward_modes")
    return (out[..., 0] + 1j * out[..., 1]).reshape(lead + kshape)


def _split(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.complex128)
    return np.ascontiguousarray(np.stack([z.real, z.imag], axis=-1))


def mix(X: np.ndarray, w: np.ndarray, n, modes) -> np.ndarray:
    """X (B, Cin, K...) complex, w (nblk, Cin, Cout, m...) complex -> Y (B, Cout, K...)."""
    n, m = _geom(n, modes)
    d = m.size
    B, cin = X.shape[:2]
    cout = w.shape[2]
    kshape = kept_shape(n, m)
    Xs = _split(X)
    ws = _split(w)
    Y = np.empty((B, cout) + kshape + (2,), dtype=np.float64)
    _check(_load().fno_oracle_mix(d, n.ctypes.data_as(_i64p), m.ctypes.data_as(_i32p),
                                  B, cin, cout, _d(Xs), _d(ws), _d(Y)), "mix")
    return Y[..., 0] + 1j * Y[..., 1]


def inverse_modes(Y: np.ndarray, n, modes) -> np.ndarray:
    """Kept modes (..., K...) complex -> real grid (..., N...)."""
    n, m = _geom(n, modes)
    d = m.size
    lead = Y.shape[:-d]
    nimg = int(np.prod(lead, dtype=np.int64))
    Ys = _split(Y)
    out = np.empty(lead + tuple(int(v) for v in n), dtype=np.float64)
    _check(_load().fno_oracle_inverse_modes(d, n.ctypes.data_as(_i64p),
                                            m.ctypes.data_as(_i32p), nimg, _d(Ys), _d(out)),
           "inverse_modes")
    return out


def spectral_conv(x: np.ndarray, w: np.ndarray, modes) -> np.ndarray:
    """x (B, Cin, N...) real, w (nblk, Cin, Cout, m...) complex -> y (B, Cout, N...)."""
    d = len(modes)
    x = _f64(x)
    n, m = _geom(x.shape[-d:], modes)
    B, cin = x.shape[:2]
    if w.shape[1] != cin:
        raise ValueError("weight Cin does not match x")
    cout = w.shape[2]
    ws = _split(w)
    y = np.empty((B, cout) + tuple(int(v) for v in n), dtype=np.float64)
    _check(_load().fno_oracle_spectral_conv(d, n.ctypes.data_as(_i64p),
                                            m.ctypes.data_as(_i32p), B, cin, cout,
                                            _d(x), _d(ws), _d(y)), "spectral_conv")
    return y


def spectral_conv_padded(x: np.ndarray, w: np.ndarray, modes, pad) -> np.ndarray:
    """The layer on a non-periodic domain (TurboFNO §2.3, §3.3): every spatial
    axis a of x (B, Cin, N...) is extended with pad[a] zeros after its last
    sample, the layer runs at the extents L = N + pad (modes counted on L),
    and the output is cropped back to its first N samples per axis."""
    d = len(modes)
    x = _f64(x)
    n = x.shape[-d:]
    pad = tuple(int(p) for p in pad)
    if len(pad) != d or min(pad) < 0:
        raise ValueError("pad needs one non-negative entry per spatial axis")
    xp = np.zeros(x.shape[:2] + tuple(na + pa for na, pa in zip(n, pad)), dtype=np.float64)
    xp[(slice(None), slice(None)) + tuple(slice(0, na) for na in n)] = x
    yp = spectral_conv(xp, w, modes)
    return np.ascontiguousarray(yp[(slice(None), slice(None)) + tuple(slice(0, na) for na in n)])


def adjoint_modes(dX: np.ndarray, n, modes) -> np.ndarray:
    """Kept-mode gradients (..., K...) complex -> dx (..., N...) real, the
    adjoint of ``forward_modes``: dx_n = sum over kept k of Re(dX_k e^{+2 pi i k.n/N})."""
    n, m = _geom(n, modes)
    d = m.size
    lead = dX.shape[:-d]
    nimg = int(np.prod(lead, dtype=np.int64))
    Gs = _split(dX)
    out = np.empty(lead + tuple(int(v) for v in n), dtype=np.float64)
    _check(_load().fno_oracle_adjoint_modes(d, n.ctypes.data_as(_i64p),
                                            m.ctypes.data_as(_i32p), nimg, _d(Gs), _d(out)),
           "adjoint_modes")
    return out


def spectral_conv_backward(x: np.ndarray, w: np.ndarray, dy: np.ndarray, modes):
    """Gradients of a real loss through the layer, given dy = dL/dy:
    returns (dx, dw) with dx (B, Cin, N...) real and dw (nblk, Cin, Cout, m...)
    complex = dL/dRe(w) + i dL/dIm(w)."""
    d = len(modes)
    x = _f64(x)
    dy = _f64(dy)
    n, m = _geom(x.shape[-d:], modes)
    B, cin = x.shape[:2]
    cout = w.shape[2]
    if w.shape[1] != cin or dy.shape != (B, cout) + tuple(int(v) for v in n):
        raise ValueError("x, w and dy shapes do not agree")
    ws = _split(w)
    dx = np.empty(x.shape, dtype=np.float64)
    dw = np.empty(w.shape + (2,), dtype=np.float64)
    _check(_load().fno_oracle_spectral_conv_backward(
        d, n.ctypes.data_as(_i64p), m.ctypes.data_as(_i32p), B, cin, cout,
        _d(x), _d(ws), _d(dy), _d(dx), _d(dw)), "spectral_conv_backward")
    return dx, dw[..., 0] + 1j * dw[..., 1]


def fno_forward(x: np.ndarray, params: dict, modes) -> np.ndarray:
    """2-D FNO stack.  params holds float64/complex arrays:
    lift_w (W, Cl), lift_b (W,), spec_w (L, 2, W, W, m0, m1) complex,
    pw_w (L, W, W), pw_b (L, W), proj1_w (H, W), proj1_b (H,),
    proj2_w (Co, H), proj2_b (Co,)."""
    x = _f64(x)
    B, cl, h, wd = x.shape
    width = params["lift_w"].shape[0]
    nlayers = params["pw_w"].shape[0]
    hidden = params["proj1_w"].shape[0]
    cout = params["proj2_w"].shape[0]
    m = np.ascontiguousarray(modes, dtype=np.int32)
    out = np.empty((B, cout, h, wd), dtype=np.float64)
    arrs = [_f64(params[k]) for k in ("lift_w", "lift_b")]
    arrs.append(_split(params["spec_w"]))
    arrs += [_f64(params[k]) for k in ("pw_w", "pw_b", "proj1_w", "proj1_b",
                                       "proj2_w", "proj2_b")]
    _check(_load().fno_oracle_fno_forward(
        B, h, wd, m.ctypes.data_as(_i32p), cl, width, nlayers, hidden, cout,
        _d(x), *[_d(a) for a in arrs], _d(out)), "fno_forward")
    return out
