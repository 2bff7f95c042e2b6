"""The index splits that the column transforms of the kernels rest on, checked
in float64 against the direct sums over the kept rows (no GPU needed).

A full axis of N rows keeps the rows j < M (frequency g = j) and j >= M
(g = j - 2M).  Writing g = g1 + G1*g2 (0 <= g1 < G1) and t = t1 + T1*t2 with
T1 = N / G1, exp(+-2 pi i g t / N) = exp(+-2 pi i g t1 / N) * exp(+-2 pi i g1 t2 / G1),
so a column transform is a short sum over g2 (or t1) and one G1-point DFT."""
import numpy as np
import pytest

# (N rows, M kept per side, G1): the fp32 128^2 inverse, the 16-bit 256^2
# forward and inverse, the 64-row planes of the 3-D inverse
SPLITS = [(128, 16, 8), (256, 32, 32), (64, 16, 8)]


def kept_freq(j, m):
    return j if j < m else j - 2 * m


def direct_inverse(v, n, m):
    t = np.arange(n)[:, None]
    g = np.array([kept_freq(j, m) for j in range(2 * m)])[None, :]
    return np.exp(2j * np.pi * g * t / n) @ v


def split_inverse(v, n, m, g1n):
    t1n = n // g1n
    out = np.zeros((n,) + v.shape[1:], complex)
    for t1 in range(t1n):
        u = np.zeros((g1n,) + v.shape[1:], complex)
        for j in range(2 * m):
            g = kept_freq(j, m)
            u[g % g1n] += v[j] * np.exp(2j * np.pi * g * t1 / n)
        z = np.fft.ifft(u, axis=0) * g1n          # sum_g1 U[g1] e^{+2 pi i g1 t2 / G1}
        for t2 in range(g1n):
            out[t1 + t1n * t2] = z[t2]
    return out


def direct_forward(z, n, m):
    g = np.array([kept_freq(j, m) for j in range(2 * m)])[:, None]
    t = np.arange(n)[None, :]
    return np.exp(-2j * np.pi * g * t / n) @ z


def split_forward(z, n, m, g1n):
    t1n = n // g1n
    f = np.stack([np.fft.fft(z[t1::t1n], axis=0) for t1 in range(t1n)])  # [t1][g1]
    x = np.zeros((2 * m,) + z.shape[1:], complex)
    for j in range(2 * m):
        g = kept_freq(j, m)
        for t1 in range(t1n):
            x[j] += np.exp(-2j * np.pi * g * t1 / n) * f[t1][g % g1n]
    return x


@pytest.mark.parametrize("n,m,g1n", SPLITS)
def test_inverse_split_matches_direct_sum(n, m, g1n):
    rng = np.random.default_rng(n + m)
    v = rng.standard_normal((2 * m, 5)) + 1j * rng.standard_normal((2 * m, 5))
    ref = direct_inverse(v, n, m)
    got = split_inverse(v, n, m, g1n)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
    # each U[g1] takes 2M / G1 terms: four, two and four for the kernels above
    assert (2 * m) % g1n == 0


@pytest.mark.parametrize("n,m,g1n", SPLITS)
def test_forward_split_matches_direct_sum(n, m, g1n):
    rng = np.random.default_rng(2 * n + m)
    z = rng.standard_normal((n, 3)) + 1j * rng.standard_normal((n, 3))
    ref = direct_forward(z, n, m)
    got = split_forward(z, n, m, g1n)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_a_wrong_split_fails():
    # t = t1 * G1 + t2 (transposed roles) is not the split the kernels use
    n, m, g1n = 64, 16, 8
    rng = np.random.default_rng(7)
    v = rng.standard_normal((2 * m, 2)) + 1j * rng.standard_normal((2 * m, 2))
    ref = direct_inverse(v, n, m)
    got = split_inverse(v, n, m, g1n)
    wrong = got.reshape(n // g1n, g1n, -1).transpose(1, 0, 2).reshape(n, -1)
    assert np.max(np.abs(wrong - ref)) > 1e-3 * np.max(np.abs(ref))


def test_plane_kept_modes_by_two_8_point_ffts():
    # the 64-row plane of the 3-D forward transform: S[t1][q] = sum_t2 Z[t1 + 8 t2]
    # W_8^{q t2}, then per (q, k) one more 8-point FFT over t1 after the twiddle
    # W_64^{q t1}; output f2 is frequency f = q + 8 f2, and the kept rows
    # j = q + 8 m (m = 0..3) are f2 = 0, 1, 6, 7
    n, m = 64, 16
    rng = np.random.default_rng(11)
    z = rng.standard_normal((n, 4)) + 1j * rng.standard_normal((n, 4))
    ref = direct_forward(z, n, m)                               # [32 kept rows][4]
    s = np.stack([np.fft.fft(z[t1::8], axis=0) for t1 in range(8)])   # [t1][q][k]
    got = np.zeros_like(ref)
    for q in range(8):
        u = s[:, q, :] * np.exp(-2j * np.pi * q * np.arange(8) / n)[:, None]
        x = np.fft.fft(u, axis=0)                               # [f2][k]
        for mm, f2 in enumerate((0, 1, 6, 7)):
            j = q + 8 * mm
            assert (q + 8 * f2) % n == kept_freq(j, m) % n
            got[j] = x[f2]
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_eighth_roots_as_adds():
    # acc += v W_8^m for the eight m, W_8 = exp(-2 pi i / 8): the even powers
    # as swaps and signs, the odd ones from s = (re + im)/sqrt 2 and
    # d = (im - re)/sqrt 2, as the fold of the 3-D forward transform applies them
    rng = np.random.default_rng(3)
    v = complex(rng.standard_normal(), rng.standard_normal())
    s, d = (v.real + v.imag) / np.sqrt(2), (v.imag - v.real) / np.sqrt(2)
    table = {0: (v.real, v.imag), 1: (s, d), 2: (v.imag, -v.real), 3: (d, -s),
             4: (-v.real, -v.imag), 5: (-s, -d), 6: (-v.imag, v.real), 7: (-d, s)}
    for mm in range(8):
        ref = v * np.exp(-2j * np.pi * mm / 8)
        assert abs(complex(*table[mm]) - ref) <= 1e-12 * abs(v)
