// Host-side check of the register FFT codelets (fno_fft.cuh): every codelet
// runs on the CPU here and is compared with an O(N^2) double-precision DFT.
// Prints one line per case: "<name> <max abs error> <max |X|>".
#include <cmath>
#include <cstdio>
#include <cstdint>

#include "fno_fft.cuh"

using namespace fno::fft;

static uint64_t state = 88172645463325252ull;
static double urand() {  // xorshift64, uniform in [-1, 1)
    state ^= state << 13;
    state ^= state >> 7;
    state ^= state << 17;
    return (double)(state >> 11) / (double)(1ull << 52) - 1.0;
}

template <int N, int SIGN>
static void check_fft() {
    float2 v[N];
    double re[N], im[N];
    for (int i = 0; i < N; ++i) {
        re[i] = urand();
        im[i] = urand();
        v[i] = make_float2((float)re[i], (float)im[i]);
        re[i] = v[i].x;
        im[i] = v[i].y;
    }
    fft_dif<N, SIGN>(v);
    double err = 0, mx = 0;
    for (int q = 0; q < N; ++q) {
        double sr = 0, si = 0;
        for (int n = 0; n < N; ++n) {
            double a = SIGN * 2.0 * M_PI * (double)q * n / N;
            sr += re[n] * cos(a) - im[n] * sin(a);
            si += re[n] * sin(a) + im[n] * cos(a);
        }
        float2 g = v[bitrev(q, ilog2(N))];
        err = fmax(err, fmax(fabs(g.x - sr), fabs(g.y - si)));
        mx = fmax(mx, hypot(sr, si));
    }
    printf("fft_dif<%d,%d> %.3e %.3e\n", N, SIGN, err, mx);
}

template <int N, int Q>
static void check_split() {
    float2 v[N];
    double a[N], b[N];
    for (int i = 0; i < N; ++i) {
        v[i] = make_float2((float)urand(), (float)urand());
        a[i] = v[i].x;
        b[i] = v[i].y;
    }
    fft_dif<N, -1>(v);
    float2 A, B;
    split_real_pair<N, Q>(v, A, B);
    double ar = 0, ai = 0, br = 0, bi = 0;
    for (int n = 0; n < N; ++n) {
        double t = -2.0 * M_PI * (double)Q * n / N;
        ar += a[n] * cos(t); ai += a[n] * sin(t);
        br += b[n] * cos(t); bi += b[n] * sin(t);
    }
    double err = fmax(fmax(fabs(A.x - ar), fabs(A.y - ai)), fmax(fabs(B.x - br), fabs(B.y - bi)));
    // the unscaled split returns exactly twice the scaled one
    float2 A2, B2;
    split_real_pair2<N, Q>(v, A2, B2);
    if (A2.x != 2.f * A.x || A2.y != 2.f * A.y || B2.x != 2.f * B.x || B2.y != 2.f * B.y) err = 1.0;
    printf("split<%d,%d> %.3e %.3e\n", N, Q, err, hypot(ar, ai) + hypot(br, bi));
}

int main() {
    check_fft<2, -1>(); check_fft<4, -1>(); check_fft<8, -1>(); check_fft<16, -1>();
    check_fft<32, -1>(); check_fft<64, -1>();
    check_fft<2, 1>(); check_fft<4, 1>(); check_fft<8, 1>(); check_fft<16, 1>();
    check_fft<32, 1>(); check_fft<64, 1>();
    check_split<16, 0>(); check_split<16, 3>(); check_split<16, 8>(); check_split<16, 13>();
    check_split<32, 5>(); check_split<8, 4>();
    // compile-time twiddles against libm
    double terr = 0;
    for (int n = 2; n <= 1024; n *= 2)
        for (int k = -n; k < 2 * n; ++k) {
            terr = fmax(terr, fabs(tw_re(k, n) - cos(2 * M_PI * k / n)));
            terr = fmax(terr, fabs(tw_im(k, n, -1) + sin(2 * M_PI * k / n)));
        }
    printf("twiddles %.3e 1\n", terr);
    return 0;
}
