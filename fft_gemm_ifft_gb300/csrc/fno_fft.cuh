// fno_fft.cuh -- register-resident FFT building blocks for the fused kernels.
//
// The TurboFNO article (gsyq.cn/news/457482, §3.1) computes its transform as
// radix-2 butterfly stages on small tiles held on chip with precomputed
// twiddle factors.  Here each thread holds a short line (8..64 points) in
// registers and runs a fully unrolled radix-2 decimation-in-frequency FFT on
// it; the twiddles are compile-time constants (exp(+-2 pi i k / n) evaluated
// by a constexpr Taylor series in double, rounded once to float), so no
// table is read.  Everything here is __host__ __device__ so the codelets can
// be checked on the CPU against a brute-force DFT.
#pragma once

#include <cuda_runtime.h>

namespace fno {
namespace fft {

// ---------------------------------------------------------------------------
// complex float helpers
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ float2 c2(float x, float y) { return make_float2(x, y); }
__host__ __device__ __forceinline__ float2 cadd(float2 a, float2 b) { return c2(a.x + b.x, a.y + b.y); }
__host__ __device__ __forceinline__ float2 csub(float2 a, float2 b) { return c2(a.x - b.x, a.y - b.y); }
__host__ __device__ __forceinline__ float2 cscale(float2 a, float s) { return c2(a.x * s, a.y * s); }
__host__ __device__ __forceinline__ float2 cconj(float2 a) { return c2(a.x, -a.y); }
__host__ __device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return c2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// a * conj(b)
__host__ __device__ __forceinline__ float2 cmulc(float2 a, float2 b) {
    return c2(fmaf(a.x, b.x, a.y * b.y), fmaf(a.y, b.x, -a.x * b.y));
}
// acc += a * b
__host__ __device__ __forceinline__ void cmac(float2 &acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, acc.x);
    acc.x = fmaf(-a.y, b.y, acc.x);
    acc.y = fmaf(a.x, b.y, acc.y);
    acc.y = fmaf(a.y, b.x, acc.y);
}

// ---------------------------------------------------------------------------
// compile-time twiddles
// ---------------------------------------------------------------------------
constexpr double kPi = 3.14159265358979323846264338327950288;

// Taylor series, |x| <= pi: 24 terms reach double precision there.
__host__ __device__ constexpr double ct_sin(double x) {
    double term = x, sum = x;
    for (int i = 1; i < 24; ++i) {
        term *= -x * x / ((2.0 * i) * (2.0 * i + 1.0));
        sum += term;
    }
    return sum;
}
__host__ __device__ constexpr double ct_cos(double x) {
    double term = 1.0, sum = 1.0;
    for (int i = 1; i < 24; ++i) {
        term *= -x * x / ((2.0 * i - 1.0) * (2.0 * i));
        sum += term;
    }
    return sum;
}
// angle 2 pi k / n reduced exactly (integers) to [-pi, pi]
__host__ __device__ constexpr double ct_angle(long k, long n) {
    long r = k % n;
    if (r < 0) r += n;
    if (2 * r > n) r -= n;
    return 2.0 * kPi * (double)r / (double)n;
}
// exp(sign * 2 pi i k / n), exact for the axis-aligned and diagonal points
__host__ __device__ constexpr double tw_re(long k, long n) {
    long r = ((k % n) + n) % n;
    if (r == 0) return 1.0;
    if (4 * r == n || 4 * r == 3 * n) return 0.0;
    if (2 * r == n) return -1.0;
    return ct_cos(ct_angle(k, n));
}
__host__ __device__ constexpr double tw_im(long k, long n, int sign) {
    long r = ((k % n) + n) % n;
    if (r == 0 || 2 * r == n) return 0.0;
    if (4 * r == n) return (double)sign;
    if (4 * r == 3 * n) return -(double)sign;
    return (double)sign * ct_sin(ct_angle(k, n));
}

template <int I> struct ic { static constexpr int value = I; };

template <int B, int E, typename F>
__host__ __device__ __forceinline__ void unroll(F &&f) {
    if constexpr (B < E) {
        f(ic<B>{});
        unroll<B + 1, E>(f);
    }
}

__host__ __device__ constexpr int ilog2(int n) { return n <= 1 ? 0 : 1 + ilog2(n >> 1); }
__host__ __device__ constexpr int bitrev(int v, int bits) {
    int r = 0;
    for (int i = 0; i < bits; ++i) r |= ((v >> i) & 1) << (bits - 1 - i);
    return r;
}

// d * exp(SIGN * 2 pi i K / LEN), with the trivial cases folded at compile time
template <int K, int LEN, int SIGN>
__host__ __device__ __forceinline__ float2 twiddle(float2 d) {
    constexpr long r = ((long)K % LEN + LEN) % LEN;
    if constexpr (r == 0) {
        return d;
    } else if constexpr (2 * r == LEN) {
        return c2(-d.x, -d.y);
    } else if constexpr (4 * r == LEN) {          // multiply by SIGN * i
        return SIGN < 0 ? c2(d.y, -d.x) : c2(-d.y, d.x);
    } else if constexpr (4 * r == 3 * LEN) {      // multiply by -SIGN * i
        return SIGN < 0 ? c2(-d.y, d.x) : c2(d.y, -d.x);
    } else {
        constexpr float wr = (float)tw_re(K, LEN);
        constexpr float wi = (float)tw_im(K, LEN, SIGN);
        if constexpr (8 * r == LEN || 8 * r == 3 * LEN || 8 * r == 5 * LEN ||
                      8 * r == 7 * LEN) {
            // |wr| == |wi| == sqrt(1/2): 2 multiplies + 2 adds
            constexpr float h = wr;
            constexpr float s = (wi == wr) ? 1.f : -1.f;
            return c2(h * (d.x - s * d.y), h * (d.y + s * d.x));
        } else {
            return c2(fmaf(d.x, wr, -d.y * wi), fmaf(d.x, wi, d.y * wr));
        }
    }
}

// In-place radix-2 decimation-in-frequency FFT of N points in registers.
// Input in natural order; on return v[j] holds bin bitrev(j).
// SIGN = -1: forward kernel e^{-2 pi i k n / N}; +1: inverse (unnormalised).
template <int N, int SIGN>
__host__ __device__ __forceinline__ void fft_dif(float2 (&v)[N]) {
    constexpr int S = ilog2(N);
    unroll<0, S>([&](auto st) {
        constexpr int len = N >> decltype(st)::value;
        constexpr int half = len / 2;
        unroll<0, N / len>([&](auto bl) {
            unroll<0, half>([&](auto kk) {
                constexpr int k = decltype(kk)::value;
                constexpr int a = decltype(bl)::value * len + k;
                constexpr int b = a + half;
                const float2 u = v[a], w = v[b];
                v[a] = cadd(u, w);
                v[b] = twiddle<k, len, SIGN>(csub(u, w));
            });
        });
    });
}

// Bin q of a transform left in bit-reversed order by fft_dif.
template <int N, int Q>
__host__ __device__ __forceinline__ float2 bin(const float2 (&v)[N]) {
    return v[bitrev(Q, ilog2(N))];
}

// Two real sequences a, b of length N packed as z = a + i b and transformed
// by fft_dif<N,-1>: A[q] = (Z[q] + conj Z[N-q]) / 2, B[q] = (Z[q] - conj Z[N-q]) / (2i).
template <int N, int Q>
__host__ __device__ __forceinline__ void split_real_pair(const float2 (&z)[N], float2 &A,
                                                         float2 &B) {
    const float2 p = bin<N, Q>(z);
    const float2 m = bin<N, (N - Q) % N>(z);
    A = c2(0.5f * (p.x + m.x), 0.5f * (p.y - m.y));
    B = c2(0.5f * (p.y + m.y), 0.5f * (m.x - p.x));
}

// The same split without the factor 1/2 (2A and 2B), for callers that fold
// the 1/2 into a twiddle they multiply by anyway.
template <int N, int Q>
__host__ __device__ __forceinline__ void split_real_pair2(const float2 (&z)[N], float2 &A2,
                                                          float2 &B2) {
    const float2 p = bin<N, Q>(z);
    const float2 m = bin<N, (N - Q) % N>(z);
    A2 = c2(p.x + m.x, p.y - m.y);
    B2 = c2(p.y + m.y, m.x - p.x);
}

}  // namespace fft
}  // namespace fno
