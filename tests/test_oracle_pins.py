"""Pins for the float64 oracle, against facts fixed by the mathematics.

Each test would fail under a plausible mistake in the oracle: a wrong twiddle
sign or index (brute force, textbook values, shift theorem), a dropped
normalisation (impulse, Parseval, round trip), a wrong half-spectrum weight at
DC or Nyquist (closed forms, Nyquist round trip), a swapped low/high block or
block order (one-hot blocks), a transposed mixing operand (Cin != Cout einsum),
and a wrong activation or layer order in the FNO stack (reductions to a
per-pixel MLP and to composed spectral convolutions).
"""
import math
import os

import numpy as np
import pytest
from scipy.special import erf

from fft_gemm_ifft_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_dft(z, sign=-1):
    """O(N^2) DFT straight from the definition (independent of the oracle)."""
    z = np.asarray(z, dtype=np.complex128)
    n = z.shape[0]
    k = np.arange(n)
    mat = np.exp(sign * 2j * np.pi * np.outer(k, k) / n)
    return mat @ z


def brute_dftn(x, sign=-1):
    """Multi-dimensional DFT from the definition, one explicit matrix per axis."""
    out = np.asarray(x, dtype=np.complex128)
    for ax in range(out.ndim):
        n = out.shape[ax]
        k = np.arange(n)
        mat = np.exp(sign * 2j * np.pi * np.outer(k, k) / n)
        out = np.moveaxis(np.tensordot(mat, np.moveaxis(out, ax, 0), axes=(1, 0)), 0, ax)
    return out


def kept_freqs(n, modes):
    """Frequencies of the kept set per axis: low then high rows on full axes."""
    per_axis = []
    for a, (na, ma) in enumerate(zip(n, modes)):
        if a < len(n) - 1:
            per_axis.append(list(range(ma)) + list(range(na - ma, na)))
        else:
            per_axis.append(list(range(ma)))
    return per_axis


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# 1-D radix-2 FFT
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 256, 3, 6, 12, 15, 100])
@pytest.mark.parametrize("inverse", [False, True])
def test_fft_matches_brute_force(oracle_mod, n, inverse):
    r = rng(n)
    z = r.standard_normal(n) + 1j * r.standard_normal(n)
    got = oracle_mod.fft(z, inverse=inverse)
    want = brute_dft(z, sign=+1 if inverse else -1)
    assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))


def test_fft_textbook_values(oracle_mod):
    with open(os.path.join(GOLDEN, "dft_textbook.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert rows
    for row in rows:
        n_s, x_s, X_s = [p.strip() for p in row.split("|")]
        x = np.array([float(v) for v in x_s.split()])
        want = np.array([complex(float(a), float(b)) for a, b in
                         (p.split(":") for p in X_s.split())])
        assert x.size == int(n_s) == want.size
        got = oracle_mod.fft(x)
        assert np.max(np.abs(got - want)) < 1e-12


def test_fft_impulse_is_all_ones(oracle_mod):
    for n in (8, 64):
        z = np.zeros(n, dtype=complex)
        z[0] = 1.0
        assert np.max(np.abs(oracle_mod.fft(z) - 1.0)) < 1e-14


def test_fft_parseval_linearity_shift(oracle_mod):
    r = rng(7)
    n = 128
    a = r.standard_normal(n) + 1j * r.standard_normal(n)
    b = r.standard_normal(n) + 1j * r.standard_normal(n)
    A, B = oracle_mod.fft(a), oracle_mod.fft(b)
    # Parseval: sum |x|^2 = (1/N) sum |X|^2
    assert abs(np.sum(abs(a) ** 2) - np.sum(abs(A) ** 2) / n) < 1e-10 * np.sum(abs(a) ** 2)
    # linearity
    al, be = 0.3 - 1.1j, -2.5 + 0.25j
    assert np.max(np.abs(oracle_mod.fft(al * a + be * b) - (al * A + be * B))) < 1e-11
    # shift theorem: x[n - s] <-> X[k] e^{-2 pi i k s / N}
    s = 5
    k = np.arange(n)
    assert np.max(np.abs(oracle_mod.fft(np.roll(a, s)) - A * np.exp(-2j * np.pi * k * s / n))) < 1e-11
    # inverse of forward is N times the input (unnormalised both ways)
    assert np.max(np.abs(oracle_mod.fft(A, inverse=True) / n - a)) < 1e-13


# ---------------------------------------------------------------------------
# Truncated forward transform (step a1)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,modes", [
    ((16,), (5,)), ((16,), (9,)), ((8, 8), (2, 3)), ((8, 16), (4, 9)),
    ((4, 4, 8), (1, 2, 3)), ((4, 8, 8), (2, 1, 5)),
    ((12,), (7,)), ((6, 10), (2, 4)), ((5, 6, 7), (2, 3, 4)),      # any extent
])
def test_forward_modes_brute_force(oracle_mod, n, modes):
    r = rng(sum(n) + sum(modes))
    x = r.standard_normal((2, 3) + n)
    got = oracle_mod.forward_modes(x, modes)
    full = np.stack([brute_dftn(img) for img in x.reshape((-1,) + n)]).reshape(x.shape)
    idx = np.ix_(*kept_freqs(n, modes))
    want = full[(slice(None), slice(None)) + idx]
    assert got.shape == want.shape
    assert np.max(np.abs(got - want)) < 1e-11 * max(1.0, np.max(np.abs(want)))


def test_forward_modes_vs_numpy_rfftn(oracle_mod):
    r = rng(11)
    n, modes = (32, 16, 64), (5, 3, 7)
    x = r.standard_normal((2,) + n)
    got = oracle_mod.forward_modes(x, modes)
    full = np.fft.rfftn(x, axes=(1, 2, 3))
    want = full[(slice(None),) + np.ix_(*kept_freqs(n, modes))]
    assert np.max(np.abs(got - want)) < 1e-10


def test_forward_modes_high_rows_are_negative_frequencies(oracle_mod):
    # x = exp(-2 pi i * 3 r / 16) has its energy at row frequency -3 = 13,
    # which is the 3rd-from-last high row: index 2m - 3 of the kept axis.
    n, m = 16, 4
    r_ = np.arange(n)[:, None]
    c_ = np.arange(8)[None, :]
    x = np.cos(2 * np.pi * (-3 * r_ / n + 2 * c_ / 8))
    X = oracle_mod.forward_modes(x[None], (m, 3))[0]
    k = np.argmax(np.abs(X).ravel())
    assert np.unravel_index(k, X.shape) == (2 * m - 3, 2)
    assert abs(X[2 * m - 3, 2] - n * 8 / 2) < 1e-10


# ---------------------------------------------------------------------------
# Inverse transform (step a3)
# ---------------------------------------------------------------------------

def inverse_brute(Y, n, modes):
    """y[n] = (1/prod N) sum_{k kept} c(k_last) Re(Y[k] e^{+2 pi i k.n/N})."""
    d = len(n)
    freqs = kept_freqs(n, modes)
    grids = np.meshgrid(*[np.arange(v) for v in n], indexing="ij")
    y = np.zeros(n)
    for kidx in np.ndindex(*[len(f) for f in freqs]):
        fk = [freqs[a][kidx[a]] for a in range(d)]
        kl = fk[-1]
        c = 1.0 if (kl == 0 or 2 * kl == n[-1]) else 2.0
        phase = sum(fk[a] * grids[a] / n[a] for a in range(d))
        y += c * np.real(Y[kidx] * np.exp(2j * np.pi * phase))
    return y / np.prod(n)


@pytest.mark.parametrize("n,modes", [((16,), (9,)), ((8, 8), (2, 5)), ((4, 4, 8), (2, 1, 3)),
                                     ((12,), (7,)), ((6, 9), (3, 5)), ((5, 6, 7), (2, 2, 4))])
def test_inverse_modes_brute_force_and_numpy(oracle_mod, n, modes):
    r = rng(3 + len(n))
    kshape = oracle_mod.kept_shape(n, modes)
    Y = r.standard_normal(kshape) + 1j * r.standard_normal(kshape)
    got = oracle_mod.inverse_modes(Y[None], n, modes)[0]
    want = inverse_brute(Y, n, modes)
    assert np.max(np.abs(got - want)) < 1e-12
    # numpy's irfftn applies the same half-spectrum convention (real part of
    # the DC / Nyquist bins along the last axis) to a zero-filled half spectrum
    half = np.zeros(n[:-1] + (n[-1] // 2 + 1,), dtype=complex)
    half[np.ix_(*kept_freqs(n, modes))] = Y
    ref = np.fft.irfftn(half, s=n, axes=tuple(range(len(n))))
    assert np.max(np.abs(got - ref)) < 1e-12


def test_inverse_weights_at_dc_and_nyquist(oracle_mod):
    # A lone DC bin of value a + ib gives a/N everywhere (imaginary part dropped,
    # weight 1); a lone Nyquist bin gives (a/N)(-1)^n; bin 1 gives weight 2.
    n = 8
    for kb, want in [(0, np.full(n, 2.0 / n)),
                     (4, 2.0 / n * (-1.0) ** np.arange(n)),
                     (1, 2 * (2.0 * np.cos(2 * np.pi * np.arange(n) / n)
                              - 3.0 * np.sin(2 * np.pi * np.arange(n) / n)) / n)]:
        Y = np.zeros(5, dtype=complex)
        Y[kb] = 2.0 + 3.0j
        got = oracle_mod.inverse_modes(Y[None], (n,), (5,))[0]
        assert np.max(np.abs(got - want)) < 1e-14, kb


# ---------------------------------------------------------------------------
# Whole layer (a1 -> a2 -> a3)
# ---------------------------------------------------------------------------

def identity_weights(cin, nblk, modes):
    w = np.zeros((nblk, cin, cin) + tuple(modes), dtype=complex)
    for i in range(cin):
        w[:, i, i] = 1.0
    return w


@pytest.mark.parametrize("n", [(8,), (16,), (8, 8), (8, 16), (4, 4, 8), (4, 8, 4)])
def test_all_modes_identity_reproduces_input(oracle_mod, n):
    modes = tuple(v // 2 for v in n[:-1]) + (n[-1] // 2 + 1,)
    cin = 3
    x = rng(5).standard_normal((2, cin) + n)
    w = identity_weights(cin, 2 ** (len(n) - 1), modes)
    y = oracle_mod.spectral_conv(x, w, modes)
    assert np.max(np.abs(y - x)) < 1e-12


def test_constant_input_closed_form(oracle_mod):
    # x[b,i] = a_i everywhere -> y[b,o] = sum_i a_i Re(W[0,i,o,0,..,0])
    n, modes = (16, 8), (3, 2)
    cin, cout = 4, 3
    r = rng(9)
    a = r.standard_normal(cin)
    x = np.broadcast_to(a[None, :, None, None], (1, cin) + n).copy()
    w = r.standard_normal((2, cin, cout) + modes) + 1j * r.standard_normal((2, cin, cout) + modes)
    y = oracle_mod.spectral_conv(x, w, modes)
    want = np.einsum("i,io->o", a, w[0, :, :, 0, 0].real)
    assert np.max(np.abs(y[0] - want[:, None, None])) < 1e-12


def test_cosine_closed_forms(oracle_mod):
    n, m, k0 = 32, 8, 3
    t = np.arange(n)
    x = np.cos(2 * np.pi * k0 * t / n)[None, None]
    w1 = np.ones((1, 1, 1, m), dtype=complex)
    assert np.max(np.abs(oracle_mod.spectral_conv(x, w1, (m,))[0, 0] - x[0, 0])) < 1e-13
    wi = 1j * np.ones((1, 1, 1, m))
    want = -np.sin(2 * np.pi * k0 * t / n)
    assert np.max(np.abs(oracle_mod.spectral_conv(x, wi, (m,))[0, 0] - want)) < 1e-13
    # a frequency outside the kept set is removed
    x_hi = np.cos(2 * np.pi * (m + 1) * t / n)[None, None]
    assert np.max(np.abs(oracle_mod.spectral_conv(x_hi, w1, (m,)))) < 1e-13


def test_nyquist_round_trip_pins_weight_one(oracle_mod):
    n = 8
    x = ((-1.0) ** np.arange(n) * 1.5 + 0.25)[None, None]
    w = np.ones((1, 1, 1, n // 2 + 1), dtype=complex)
    y = oracle_mod.spectral_conv(x, w, (n // 2 + 1,))
    assert np.max(np.abs(y - x)) < 1e-14


def test_block_order_2d(oracle_mod):
    # cos at row frequency +2 lives in block 0 (low rows); at -2 in block 1.
    n, modes = (16, 16), (4, 4)
    r_, c_ = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    for f0, live in [(2, 0), (14, 1)]:
        x = np.cos(2 * np.pi * (f0 * r_ / 16 + 1 * c_ / 16))[None, None]
        for blk in (0, 1):
            w = np.zeros((2, 1, 1) + modes, dtype=complex)
            w[blk] = 1.0
            y = oracle_mod.spectral_conv(x, w, modes)
            want = x if blk == live else np.zeros_like(x)
            assert np.max(np.abs(y - want)) < 1e-12, (f0, blk)


def test_block_order_3d(oracle_mod):
    # block index = (axis-0 high) + 2 * (axis-1 high)
    n, modes = (8, 8, 8), (2, 2, 2)
    g = np.meshgrid(*[np.arange(8)] * 3, indexing="ij")
    for f0, f1, live in [(1, 1, 0), (7, 1, 1), (1, 7, 2), (7, 7, 3)]:
        x = np.cos(2 * np.pi * (f0 * g[0] + f1 * g[1] + 1 * g[2]) / 8)[None, None]
        for blk in range(4):
            w = np.zeros((4, 1, 1) + modes, dtype=complex)
            w[blk] = 1.0
            y = oracle_mod.spectral_conv(x, w, modes)
            want = x if blk == live else np.zeros_like(x)
            assert np.max(np.abs(y - want)) < 1e-12, (f0, f1, blk)


def test_mixing_matches_independent_einsum(oracle_mod):
    n, modes = (16, 8), (3, 4)
    B, cin, cout = 2, 3, 5
    r = rng(21)
    ks = oracle_mod.kept_shape(n, modes)
    X = r.standard_normal((B, cin) + ks) + 1j * r.standard_normal((B, cin) + ks)
    w = r.standard_normal((2, cin, cout) + modes) + 1j * r.standard_normal((2, cin, cout) + modes)
    Y = oracle_mod.mix(X, w, n, modes)
    wk = np.concatenate([w[0], w[1]], axis=2)          # (cin, cout, 2m0, m1)
    want = np.einsum("bikl,iokl->bokl", X, wk)
    assert np.max(np.abs(Y - want)) < 1e-12
    # and through the whole layer: conv = irfft(einsum(rfft(x)))
    x = r.standard_normal((B, cin) + n)
    y = oracle_mod.spectral_conv(x, w, modes)
    Xb = np.fft.rfft2(x)[:, :, np.r_[0:3, 13:16], :4]
    half = np.zeros((B, cout, 16, 5), dtype=complex)
    half[:, :, np.r_[0:3, 13:16], :4] = np.einsum("bikl,iokl->bokl", Xb, wk)
    assert np.max(np.abs(y - np.fft.irfft2(half, s=n))) < 1e-12


def test_layer_is_linear(oracle_mod):
    n, modes = (8, 8, 8), (2, 3, 3)
    r = rng(31)
    x1, x2 = r.standard_normal((2, 1, 2) + n)
    w = r.standard_normal((4, 2, 2) + modes) + 1j * r.standard_normal((4, 2, 2) + modes)
    y1 = oracle_mod.spectral_conv(x1, w, modes)
    y2 = oracle_mod.spectral_conv(x2, w, modes)
    y12 = oracle_mod.spectral_conv(0.5 * x1 - 3.0 * x2, w, modes)
    assert np.max(np.abs(y12 - (0.5 * y1 - 3.0 * y2))) < 1e-12


def test_rfft_parseval_with_half_weights(oracle_mod):
    n = 64
    x = rng(41).standard_normal(n)
    X = oracle_mod.forward_modes(x[None], (n // 2 + 1,))[0]
    c = np.full(n // 2 + 1, 2.0)
    c[0] = c[-1] = 1.0
    assert abs(np.sum(x ** 2) - np.sum(c * np.abs(X) ** 2) / n) < 1e-10


# ---------------------------------------------------------------------------
# FNO stack (a5)
# ---------------------------------------------------------------------------

def gelu_ref(v):
    return 0.5 * v * (1.0 + erf(v / math.sqrt(2.0)))


def small_fno_params(r, cl=3, width=4, nlayers=2, hidden=5, cout=2, modes=(2, 3)):
    p = {
        "lift_w": r.standard_normal((width, cl)), "lift_b": r.standard_normal(width),
        "spec_w": (r.standard_normal((nlayers, 2, width, width) + modes)
                   + 1j * r.standard_normal((nlayers, 2, width, width) + modes)) * 0.2,
        "pw_w": r.standard_normal((nlayers, width, width)) * 0.5,
        "pw_b": r.standard_normal((nlayers, width)),
        "proj1_w": r.standard_normal((hidden, width)), "proj1_b": r.standard_normal(hidden),
        "proj2_w": r.standard_normal((cout, hidden)), "proj2_b": r.standard_normal(cout),
    }
    return p


def test_gelu_value_pin():
    # GELU(1) = Phi(1) = 0.841344746068542948585...; GELU(-1) = -(1 - Phi(1))
    assert abs(gelu_ref(1.0) - 0.8413447460685429) < 1e-15
    assert abs(gelu_ref(-1.0) + 0.15865525393145707) < 1e-15


def test_fno_zero_spectral_is_pointwise_mlp(oracle_mod):
    r = rng(51)
    p = small_fno_params(r)
    p["spec_w"] = np.zeros_like(p["spec_w"])
    x = r.standard_normal((2, 3, 8, 8))
    got = oracle_mod.fno_forward(x, p, (2, 3))
    a = np.einsum("ci,bihw->bchw", p["lift_w"], x) + p["lift_b"][None, :, None, None]
    L = p["pw_w"].shape[0]
    for l in range(L):
        t = np.einsum("ci,bihw->bchw", p["pw_w"][l], a) + p["pw_b"][l][None, :, None, None]
        a = t if l == L - 1 else gelu_ref(t)
    h = gelu_ref(np.einsum("ci,bihw->bchw", p["proj1_w"], a) + p["proj1_b"][None, :, None, None])
    want = np.einsum("ci,bihw->bchw", p["proj2_w"], h) + p["proj2_b"][None, :, None, None]
    assert np.max(np.abs(got - want)) < 1e-12


def test_fno_zero_pointwise_is_composed_spectral(oracle_mod):
    r = rng(52)
    modes = (2, 3)
    p = small_fno_params(r, modes=modes)
    p["pw_w"] = np.zeros_like(p["pw_w"])
    p["pw_b"] = np.zeros_like(p["pw_b"])
    x = r.standard_normal((2, 3, 8, 8))
    got = oracle_mod.fno_forward(x, p, modes)
    a = np.einsum("ci,bihw->bchw", p["lift_w"], x) + p["lift_b"][None, :, None, None]
    L = p["pw_w"].shape[0]
    for l in range(L):
        s = oracle_mod.spectral_conv(a, p["spec_w"][l], modes)
        a = s if l == L - 1 else gelu_ref(s)
    h = gelu_ref(np.einsum("ci,bihw->bchw", p["proj1_w"], a) + p["proj1_b"][None, :, None, None])
    want = np.einsum("ci,bihw->bchw", p["proj2_w"], h) + p["proj2_b"][None, :, None, None]
    assert np.max(np.abs(got - want)) < 1e-12


def test_fno_single_spectral_layer_against_numpy_fft(oracle_mod):
    # One layer, no pointwise term: out = Q2 gelu(Q1 SpecConv(L x + l) + q1) + q2
    # with SpecConv written independently via numpy.fft.
    r = rng(53)
    modes = (2, 3)
    p = small_fno_params(r, nlayers=1, modes=modes)
    p["pw_w"][:] = 0
    p["pw_b"][:] = 0
    x = r.standard_normal((1, 3, 8, 8))
    got = oracle_mod.fno_forward(x, p, modes)
    a = np.einsum("ci,bihw->bchw", p["lift_w"], x) + p["lift_b"][None, :, None, None]
    Xf = np.fft.rfft2(a)
    rows = np.r_[0:2, 6:8]
    wk = np.concatenate([p["spec_w"][0, 0], p["spec_w"][0, 1]], axis=2)
    half = np.zeros(a.shape[:2] + (8, 5), dtype=complex)
    half[:, :, rows, :3] = np.einsum("bikl,iokl->bokl", Xf[:, :, rows, :3], wk)
    s = np.fft.irfft2(half, s=(8, 8))
    h = gelu_ref(np.einsum("ci,bihw->bchw", p["proj1_w"], s) + p["proj1_b"][None, :, None, None])
    want = np.einsum("ci,bihw->bchw", p["proj2_w"], h) + p["proj2_b"][None, :, None, None]
    assert np.max(np.abs(got - want)) < 1e-12


def _numpy_spectral_conv(a, w, modes):
    """The layer written independently with numpy.fft: rfft2, the two corner
    blocks (low rows, then high rows) mixed by einsum, irfft2."""
    h, wd = a.shape[-2:]
    m0, m1 = modes
    Xf = np.fft.rfft2(a)
    rows = np.r_[0:m0, h - m0:h]
    wk = np.concatenate([w[0], w[1]], axis=2)
    half = np.zeros(a.shape[:1] + (w.shape[2], h, wd // 2 + 1), dtype=complex)
    half[:, :, rows, :m1] = np.einsum("bikl,iokl->bokl", Xf[:, :, rows, :m1], wk)
    return np.fft.irfft2(half, s=(h, wd))


def _numpy_fno(x, p, modes):
    """The whole stack with both branches live: a_{l+1} = GELU(S_l(a_l) + P_l a_l
    + b_l), no GELU after the last layer, then the two-layer head."""
    lin = lambda wt, b, v: np.einsum("ci,bihw->bchw", wt, v) + b[None, :, None, None]
    a = lin(p["lift_w"], p["lift_b"], x)
    L = p["pw_w"].shape[0]
    for l in range(L):
        t = _numpy_spectral_conv(a, p["spec_w"][l], modes) + lin(p["pw_w"][l], p["pw_b"][l], a)
        a = t if l == L - 1 else gelu_ref(t)
    return lin(p["proj2_w"], p["proj2_b"], gelu_ref(lin(p["proj1_w"], p["proj1_b"], a)))


@pytest.mark.parametrize("nlayers", [2, 3])
def test_fno_both_branches_against_numpy(oracle_mod, nlayers):
    # Spectral and pointwise weights and all biases non-zero together: pins that
    # the two branches are summed before the GELU (gelu(s) + gelu(t) agrees with
    # both one-branch reductions above, because gelu(0) = 0), that the pointwise
    # term reads the same layer's input as the spectral one, and that the last
    # layer has no GELU.  Rectangular grid (8 x 16) so that a swapped axis fails.
    r = rng(54 + nlayers)
    modes = (2, 3)
    p = small_fno_params(r, width=5, nlayers=nlayers, modes=modes)
    x = r.standard_normal((2, 3, 8, 16))
    got = oracle_mod.fno_forward(x, p, modes)
    want = _numpy_fno(x, p, modes)
    assert np.max(np.abs(want)) > 1.0
    assert np.max(np.abs(got - want)) < 1e-12 * max(1.0, np.max(np.abs(want)))
    # the plausible mistakes named above all move the result well past that bound
    lin = lambda wt, b, v: np.einsum("ci,bihw->bchw", wt, v) + b[None, :, None, None]
    a = lin(p["lift_w"], p["lift_b"], x)
    for l in range(nlayers):
        s = _numpy_spectral_conv(a, p["spec_w"][l], modes)
        t = lin(p["pw_w"][l], p["pw_b"][l], a)
        a = s + t if l == nlayers - 1 else gelu_ref(s) + gelu_ref(t)
    wrong = lin(p["proj2_w"], p["proj2_b"], gelu_ref(lin(p["proj1_w"], p["proj1_b"], a)))
    assert np.max(np.abs(got - wrong)) > 1e-3


# ---------------------------------------------------------------------------
# Backward pass: pinned to the (pinned) forward by the identities a gradient
# of a real loss must satisfy.  The layer is linear in x and in w, so with
# L = <dy, y> the gradients are the adjoints: <dx, u> = <dy, S_w(u)> for every
# real u, and sum Re(conj(dw) V) = <dy, S_V(x)> for every complex V.  A dropped
# half-spectrum weight, a wrong scale, a missing conjugate or a transposed
# weight (Cin != Cout) breaks them.  Finite differences (exact here because L
# is linear) pin single entries, including the Nyquist bin.
# ---------------------------------------------------------------------------

BACKWARD_SHAPES = [
    ((16,), (9,), 2, 3, 4),            # 1-D with the Nyquist bin kept
    ((6, 9), (2, 5), 2, 2, 3),         # extents that are not powers of two
    ((8, 16), (3, 5), 2, 3, 2),        # 2-D, two blocks
    ((8, 8), (4, 5), 1, 2, 3),         # 2-D, touching blocks, Nyquist kept
    ((4, 8, 8), (2, 3, 4), 2, 2, 3),   # 3-D, four blocks
]


def _rand_case(r, n, modes, b, ci, co):
    nblk = 2 ** (len(n) - 1)
    x = r.standard_normal((b, ci) + n)
    w = r.standard_normal((nblk, ci, co) + modes) + 1j * r.standard_normal((nblk, ci, co) + modes)
    dy = r.standard_normal((b, co) + n)
    return x, w, dy


@pytest.mark.parametrize("shape", BACKWARD_SHAPES)
def test_backward_dx_is_the_adjoint(oracle_mod, shape):
    n, modes, b, ci, co = shape
    r = np.random.default_rng(41)
    x, w, dy = _rand_case(r, n, modes, b, ci, co)
    dx, _ = oracle_mod.spectral_conv_backward(x, w, dy, modes)
    for _ in range(3):
        u = r.standard_normal(x.shape)
        lhs = float(np.sum(dx * u))
        rhs = float(np.sum(dy * oracle_mod.spectral_conv(u, w, modes)))
        assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(rhs))


@pytest.mark.parametrize("shape", BACKWARD_SHAPES)
def test_backward_dw_is_the_adjoint(oracle_mod, shape):
    n, modes, b, ci, co = shape
    r = np.random.default_rng(43)
    x, w, dy = _rand_case(r, n, modes, b, ci, co)
    _, dw = oracle_mod.spectral_conv_backward(x, w, dy, modes)
    assert dw.shape == w.shape
    for _ in range(3):
        v = r.standard_normal(w.shape) + 1j * r.standard_normal(w.shape)
        lhs = float(np.sum((np.conj(dw) * v).real))
        rhs = float(np.sum(dy * oracle_mod.spectral_conv(x, v, modes)))
        assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(rhs))


def test_backward_finite_differences(oracle_mod):
    # L(x, w) = <dy, S_w(x)> is linear in x and in (Re w, Im w): a unit step
    # gives the derivative exactly
    n, modes = (8,), (5,)                      # bin 4 = N/2 is kept
    r = np.random.default_rng(47)
    x, w, dy = _rand_case(r, n, modes, 2, 2, 3)
    dx, dw = oracle_mod.spectral_conv_backward(x, w, dy, modes)
    L = lambda xx, ww: float(np.sum(dy * oracle_mod.spectral_conv(xx, ww, modes)))
    base = L(x, w)
    for idx in [(0, 0, 0), (1, 1, 5), (0, 1, 7)]:
        e = np.zeros_like(x)
        e[idx] = 1.0
        assert abs((L(x + e, w) - base) - dx[idx]) < 1e-11
    for idx in [(0, 0, 0, 0), (0, 1, 2, 4), (0, 0, 1, 2)]:
        e = np.zeros(w.shape, dtype=complex)
        e[idx] = 1.0
        assert abs((L(x, w + e) - base) - dw[idx].real) < 1e-11
        assert abs((L(x, w + 1j * e) - base) - dw[idx].imag) < 1e-11


def test_adjoint_modes_of_unit_mode(oracle_mod):
    # one kept mode with gradient 1 at frequency (f0, k) gives cos(2 pi (f0 n0/N0 + k n1/N1))
    n, modes = (8, 8), (2, 3)
    dX = np.zeros((1, 4, 3), dtype=complex)
    dX[0, 3, 2] = 1.0                          # high row 3 -> f0 = 8 - 4 + 3 = 7, k = 2
    got = oracle_mod.adjoint_modes(dX, n, modes)
    n0, n1 = np.meshgrid(np.arange(8), np.arange(8), indexing="ij")
    want = np.cos(2 * np.pi * (7 * n0 / 8 + 2 * n1 / 8))
    assert np.max(np.abs(got[0] - want)) < 1e-13


# ---------------------------------------------------------------------------
# Workload generators: shapes and determinism only (no arithmetic to pin)
# ---------------------------------------------------------------------------

def test_workload_generators_deterministic():
    c = workloads.CASES["2d_f32"]
    a, b = workloads.make_w(c), workloads.make_w(c)
    assert a.shape == c.weight_shape + (2,) and a.dtype == np.float32
    assert np.array_equal(a, b)
    assert 0 <= a.min() and a.max() < 1.0 / (c.cin * c.cout)
    x = workloads.make_x(workloads.small_case((8, 8), (2, 2), 2, 3, 3))
    assert x.shape == (2, 3, 8, 8)
    fx = workloads.make_fno_inputs(batch=2)
    assert fx.shape == (2, 3, 128, 128)
    assert fx[0, 1, 0, 0] == 0.0 and fx[0, 1, -1, 0] == 1.0 and fx[0, 2, 0, -1] == 1.0


# ---------------------------------------------------------------------------
# Zero padding for non-periodic domains and output cropping (TurboFNO §2.3,
# §3.3): x extended with zeros to L = N + pad per axis, the layer at L, the
# output cropped to N.
# ---------------------------------------------------------------------------

def _numpy_padded_layer(x, w, modes, pad):
    """pad -> rfftn -> per-block mixing -> irfftn -> crop, written with numpy."""
    d = len(modes)
    n = x.shape[-d:]
    L = tuple(a + b for a, b in zip(n, pad))
    xp = np.zeros(x.shape[:2] + L)
    xp[(slice(None), slice(None)) + tuple(slice(0, a) for a in n)] = x
    X = np.fft.rfftn(xp, axes=tuple(range(2, 2 + d)))
    half = np.zeros(x.shape[:1] + (w.shape[2],) + X.shape[2:], dtype=complex)
    for blk in range(w.shape[0]):
        sl = []
        for a in range(d - 1):
            hi = (blk >> a) & 1
            sl.append(slice(L[a] - modes[a], L[a]) if hi else slice(0, modes[a]))
        sl.append(slice(0, modes[-1]))
        idx = (slice(None), slice(None)) + tuple(sl)
        half[idx] = np.einsum("bi...,io...->bo...", X[idx], w[blk])
    y = np.fft.irfftn(half, s=L, axes=tuple(range(2, 2 + d)))
    return y[(slice(None), slice(None)) + tuple(slice(0, a) for a in n)]


PADDED_SHAPES = [
    ((12,), (4,), (4,)),              # L = 16, power of two
    ((10,), (6,), (5,)),              # L = 15: odd, the DFT fallback, no Nyquist bin
    ((6,), (2,), (5,)),               # L = 8 with the Nyquist bin kept
    ((6, 10), (2, 6), (2, 4)),        # 2-D, L = (8, 16)
    ((5, 7), (3, 1), (2, 3)),         # 2-D, L = (8, 8)
    ((3, 4, 6), (1, 4, 2), (2, 2, 3)),  # 3-D, L = (4, 8, 8)
]


@pytest.mark.parametrize("n,pad,modes", PADDED_SHAPES)
def test_padded_layer_against_numpy(oracle_mod, n, pad, modes):
    r = rng(600 + sum(n) + sum(pad))
    nblk = 2 ** (len(n) - 1)
    x = r.standard_normal((2, 3) + n)
    w = (r.standard_normal((nblk, 3, 4) + modes) + 1j * r.standard_normal((nblk, 3, 4) + modes))
    got = oracle_mod.spectral_conv_padded(x, w, modes, pad)
    assert got.shape == (2, 4) + n
    want = _numpy_padded_layer(x, w, modes, pad)
    assert np.max(np.abs(got - want)) < 1e-12 * max(1.0, np.max(np.abs(want)))


def test_padded_layer_brute_force_1d(oracle_mod):
    # direct sums from the definition: X[k] = sum_{n<N} x[n] e^{-2 pi i k n / L}
    # (the appended zeros add nothing), y[n] = (1/L) sum_k c(k) Re(Y[k] e^{+2 pi i k n / L})
    # for n < N only
    r = rng(610)
    N, P, m = 7, 5, 4
    L = N + P
    x = r.standard_normal((1, 2, N))
    w = r.standard_normal((1, 2, 3, m)) + 1j * r.standard_normal((1, 2, 3, m))
    got = oracle_mod.spectral_conv_padded(x, w, (m,), (P,))
    want = np.zeros((1, 3, N))
    for o in range(3):
        for t in range(N):
            acc = 0.0
            for k in range(m):
                Xk = [sum(x[0, i, s] * np.exp(-2j * np.pi * k * s / L) for s in range(N))
                      for i in range(2)]
                Yk = sum(Xk[i] * w[0, i, o, k] for i in range(2))
                c = 1.0 if (k == 0 or 2 * k == L) else 2.0
                acc += c * (Yk * np.exp(2j * np.pi * k * t / L)).real
            want[0, o, t] = acc / L
    assert np.max(np.abs(got - want)) < 1e-12


def test_padded_identity_all_modes_reproduces_input(oracle_mod):
    # identity weights with every mode of the padded extents kept: the layer is
    # the identity on the padded field, so the cropped output is x itself
    r = rng(611)
    n, pad = (6, 10), (2, 6)
    L = (8, 16)
    modes = (L[0] // 2, L[1] // 2 + 1)
    x = r.standard_normal((2, 3) + n)
    eye = np.eye(3)[None, :, :, None, None] * np.ones((2, 1, 1) + modes)
    got = oracle_mod.spectral_conv_padded(x, eye.astype(complex), modes, pad)
    assert np.max(np.abs(got - x)) < 1e-12


def test_padded_zero_pad_is_the_periodic_layer(oracle_mod):
    r = rng(612)
    x = r.standard_normal((2, 3, 8, 16))
    w = r.standard_normal((2, 3, 2, 2, 3)) + 1j * r.standard_normal((2, 3, 2, 2, 3))
    a = oracle_mod.spectral_conv_padded(x, w, (2, 3), (0, 0))
    b = oracle_mod.spectral_conv(x, w, (2, 3))
    assert np.max(np.abs(a - b)) == 0.0
    # and padding changes the result (the domain is no longer periodic)
    c = oracle_mod.spectral_conv_padded(x, w, (2, 3), (8, 0))
    assert np.max(np.abs(c - b)) > 1e-3
