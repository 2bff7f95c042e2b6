/*
 * fno_oracle.c -- plain float64 CPU oracle for the FNO spectral-convolution
 * layer and the FNO forward stack.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no code, table or header with the CUDA library under fft_gemm_ifft_gb300/.
 *
 * What it computes follows the TurboFNO article (gsyq.cn/news/457482):
 *   - §2.1: the layer starts with a real FFT over the spatial axes of an NCHW
 *     real tensor (torch.fft.rfft2/rfftn with the default normalisation:
 *     forward kernel e^{-2 pi i k n / N}, unnormalised);
 *   - §2.2: only the retained low-frequency modes are multiplied by a learned
 *     complex weight per mode, contracting the input channels, using the plain
 *     complex product (a+bi)(c+di) = (ac-bd) + (ad+bc)i;
 *   - §2.3 / §3.3: the discarded modes are zero and an inverse real FFT
 *     (conjugate twiddles, scale 1/prod(N)) returns to the grid.
 *
 * Readings taken where the article is silent (each is listed in the design
 * notes): kept modes on a full (non-last) axis are the low rows 0..m-1 and the
 * high rows N-m..N-1; on the last (half) axis the bins 0..m-1; weight blocks
 * are ordered low/high with axis 0 varying fastest; the inverse applies the
 * half-spectrum weight c(k)=1 at k=0 and k=N/2 (else 2) and keeps the real part.
 *
 * Method, in the order the pages give it:
 *   1. complex radix-2 FFT (bit reversal + butterflies, twiddles from libm
 *      cos/sin in double) along every axis of each (batch, channel) image;
 *      an axis whose length is not a power of two takes the plain O(N^2)
 *      DFT sum instead;
 *   2. explicit loops pick the kept modes block by block;
 *   3. explicit triple loop for the per-mode mixing;
 *   4. scatter the mixed modes into a zero full spectrum with the c(k)
 *      weights, inverse radix-2 FFT along every axis, real part / prod(N).
 *
 * Layouts (all row-major, complex = interleaved (re, im) doubles):
 *   x  : (nimg, N_0, .., N_{d-1}) real
 *   X  : (nimg, K_0, .., K_{d-1}) complex, K_a = 2 m_a for a < d-1, K_{d-1} = m_{d-1}
 *   w  : (nblk, cin, cout, m_0, .., m_{d-1}) complex, nblk = 2^(d-1)
 *   y  : (nimg, N_0, .., N_{d-1}) real
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PI 3.14159265358979323846264338327950288

/* ------------------------------------------------------------------------ */
/* 1-D complex radix-2 FFT, in place.  sign = -1: forward kernel
 * e^{-2 pi i k n/N}; sign = +1: inverse kernel, no normalisation.           */
static void direct_dft(double *re, double *im, int64_t n, int sign)
{
    double *tr = malloc(sizeof(double) * n), *ti = malloc(sizeof(double) * n);
    if (!tr || !ti) { free(tr); free(ti); return; }
    for (int64_t k = 0; k < n; ++k) {
        double sr = 0.0, si = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            /* angle of (j k mod n) / n: the product is reduced exactly first */
            double ang = (double)sign * 2.0 * ORACLE_PI * (double)((j * k) % n) / (double)n;
            double c = cos(ang), s = sin(ang);
            sr += re[j] * c - im[j] * s;
            si += re[j] * s + im[j] * c;
        }
        tr[k] = sr;
        ti[k] = si;
    }
    memcpy(re, tr, sizeof(double) * n);
    memcpy(im, ti, sizeof(double) * n);
    free(tr);
    free(ti);
}

void fno_oracle_fft(double *re, double *im, int64_t n, int sign)
{
    if (n & (n - 1)) {          /* not a power of two */
        direct_dft(re, im, n, sign);
        return;
    }
    /* bit-reversal permutation */
    int64_t j = 0;
    for (int64_t i = 1; i < n; ++i) {
        int64_t bit = n >> 1;
        while (j & bit) {
            j ^= bit;
            bit >>= 1;
        }
        j ^= bit;
        if (i < j) {
            double t = re[i]; re[i] = re[j]; re[j] = t;
            t = im[i]; im[i] = im[j]; im[j] = t;
        }
    }
    /* butterflies: spans of length len combine two halves of length len/2 */
    for (int64_t len = 2; len <= n; len <<= 1) {
        int64_t half = len >> 1;
        for (int64_t k = 0; k < half; ++k) {
            double ang = (double)sign * 2.0 * ORACLE_PI * (double)k / (double)len;
            double wr = cos(ang), wi = sin(ang);
            for (int64_t s = 0; s < n; s += len) {
                int64_t a = s + k, b = s + k + half;
                double tr = re[b] * wr - im[b] * wi;
                double ti = re[b] * wi + im[b] * wr;
                re[b] = re[a] - tr;
                im[b] = im[a] - ti;
                re[a] += tr;
                im[a] += ti;
            }
        }
    }
}

/* FFT of every line along `axis` of a d-dimensional complex array. */
static void fft_axis(double *re, double *im, int d, const int64_t *n, int axis,
                     int sign, double *lre, double *lim)
{
    int64_t outer = 1, inner = 1;
    for (int a = 0; a < axis; ++a) outer *= n[a];
    for (int a = axis + 1; a < d; ++a) inner *= n[a];
    int64_t len = n[axis];
    for (int64_t o = 0; o < outer; ++o) {
        for (int64_t q = 0; q < inner; ++q) {
            int64_t base = o * len * inner + q;
            for (int64_t t = 0; t < len; ++t) {
                lre[t] = re[base + t * inner];
                lim[t] = im[base + t * inner];
            }
            fno_oracle_fft(lre, lim, len, sign);
            for (int64_t t = 0; t < len; ++t) {
                re[base + t * inner] = lre[t];
                im[base + t * inner] = lim[t];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Geometry of the kept-mode set.                                            */
typedef struct {
    int d;
    int64_t n[3];
    int64_t m[3];
    int64_t kdim[3];   /* extent of each kept axis: 2m (full axes), m (last) */
    int64_t nkept;     /* number of kept modes                               */
    int64_t npix;      /* prod n                                             */
    int64_t nblk;      /* number of weight blocks, 2^(d-1)                   */
    int64_t mblk;      /* modes per block, prod m                            */
} geom_t;

static int make_geom(geom_t *g, int d, const int64_t *n, const int32_t *m)
{
    if (d < 1 || d > 3) return -1;
    g->d = d;
    g->nkept = 1; g->npix = 1; g->mblk = 1; g->nblk = 1;
    for (int a = 0; a < d; ++a) {
        g->n[a] = n[a];
        g->m[a] = m[a];
        if (n[a] < 1) return -2;
        if (a < d - 1) {
            if (m[a] < 1 || 2 * (int64_t)m[a] > n[a]) return -3;
            g->kdim[a] = 2 * (int64_t)m[a];
            g->nblk *= 2;
        } else {
            if (m[a] < 1 || (int64_t)m[a] > n[a] / 2 + 1) return -3;
            g->kdim[a] = m[a];
        }
        g->nkept *= g->kdim[a];
        g->npix *= n[a];
        g->mblk *= m[a];
    }
    return 0;
}

/* For kept-mode flat index kk: the flat spatial-frequency index in the full
 * spectrum, the weight block and the index inside the block.               */
static void kept_mode(const geom_t *g, int64_t kk, int64_t *freq_flat,
                      int64_t *blk, int64_t *local, int64_t *last_bin)
{
    int64_t r[3];
    int64_t rem = kk;
    for (int a = g->d - 1; a >= 0; --a) {
        r[a] = rem % g->kdim[a];
        rem /= g->kdim[a];
    }
    int64_t f = 0, b = 0, l = 0;
    for (int a = 0; a < g->d; ++a) {
        int64_t fa, la;
        if (a < g->d - 1) {
            int hi = r[a] >= g->m[a];
            fa = hi ? g->n[a] - 2 * g->m[a] + r[a] : r[a];
            la = hi ? r[a] - g->m[a] : r[a];
            b |= (int64_t)hi << a;
        } else {
            fa = r[a];
            la = r[a];
        }
        f = f * g->n[a] + fa;
        l = l * g->m[a] + la;
    }
    *freq_flat = f;
    *blk = b;
    *local = l;
    *last_bin = r[g->d - 1];
}

/* ------------------------------------------------------------------------ */
/* Step a1: truncated forward real FFT of nimg images -> kept modes.         */
int fno_oracle_forward_modes(int d, const int64_t *n, const int32_t *m,
                             int64_t nimg, const double *x, double *X)
{
    geom_t g;
    if (make_geom(&g, d, n, m)) return -1;
    int64_t maxn = 1;
    for (int a = 0; a < d; ++a) if (n[a] > maxn) maxn = n[a];
    int err = 0;
#pragma omp parallel
    {
        double *re = malloc(sizeof(double) * g.npix);
        double *im = malloc(sizeof(double) * g.npix);
        double *lre = malloc(sizeof(double) * maxn);
        double *lim = malloc(sizeof(double) * maxn);
        if (!re || !im || !lre || !lim) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t img = 0; img < nimg; ++img) {
                const double *xi = x + img * g.npix;
                for (int64_t p = 0; p < g.npix; ++p) { re[p] = xi[p]; im[p] = 0.0; }
                for (int a = d - 1; a >= 0; --a) fft_axis(re, im, d, g.n, a, -1, lre, lim);
                double *Xi = X + img * g.nkept * 2;
                for (int64_t kk = 0; kk < g.nkept; ++kk) {
                    int64_t f, b, l, kb;
                    kept_mode(&g, kk, &f, &b, &l, &kb);
                    Xi[2 * kk] = re[f];
                    Xi[2 * kk + 1] = im[f];
                }
            }
        }
        free(re); free(im); free(lre); free(lim);
    }
    return err ? -4 : 0;
}

/* Step a2: Y[b,o,k] = sum_i X[b,i,k] * W[blk(k), i, o, local(k)].           */
int fno_oracle_mix(int d, const int64_t *n, const int32_t *m, int64_t batch,
                   int64_t cin, int64_t cout, const double *X, const double *w,
                   double *Y)
{
    geom_t g;
    if (make_geom(&g, d, n, m)) return -1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t o = 0; o < cout; ++o) {
            for (int64_t kk = 0; kk < g.nkept; ++kk) {
                int64_t f, blk, l, kb;
                kept_mode(&g, kk, &f, &blk, &l, &kb);
                double ar = 0.0, ai = 0.0;
                for (int64_t i = 0; i < cin; ++i) {
                    const double *xv = X + ((b * cin + i) * g.nkept + kk) * 2;
                    const double *wv = w + (((blk * cin + i) * cout + o) * g.mblk + l) * 2;
                    ar += xv[0] * wv[0] - xv[1] * wv[1];
                    ai += xv[0] * wv[1] + xv[1] * wv[0];
                }
                double *yv = Y + ((b * cout + o) * g.nkept + kk) * 2;
                yv[0] = ar;
                yv[1] = ai;
            }
        }
    }
    return 0;
}

/* Step a3: zero-fill the discarded modes, inverse real FFT.  The half axis
 * carries weight c = 1 at bin 0 and bin N/2, 2 elsewhere; the real part of
 * the inverse complex FFT divided by prod(N) is the output.                */
int fno_oracle_inverse_modes(int d, const int64_t *n, const int32_t *m,
                             int64_t nimg, const double *Y, double *y)
{
    geom_t g;
    if (make_geom(&g, d, n, m)) return -1;
    int64_t maxn = 1;
    for (int a = 0; a < d; ++a) if (n[a] > maxn) maxn = n[a];
    int64_t nlast = n[d - 1];
    int err = 0;
#pragma omp parallel
    {
        double *re = malloc(sizeof(double) * g.npix);
        double *im = malloc(sizeof(double) * g.npix);
        double *lre = malloc(sizeof(double) * maxn);
        double *lim = malloc(sizeof(double) * maxn);
        if (!re || !im || !lre || !lim) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t img = 0; img < nimg; ++img) {
                memset(re, 0, sizeof(double) * g.npix);
                memset(im, 0, sizeof(double) * g.npix);
                const double *Yi = Y + img * g.nkept * 2;
                for (int64_t kk = 0; kk < g.nkept; ++kk) {
                    int64_t f, b, l, kb;
                    kept_mode(&g, kk, &f, &b, &l, &kb);
                    double c = (kb == 0 || 2 * kb == nlast) ? 1.0 : 2.0;
                    re[f] = c * Yi[2 * kk];
                    im[f] = c * Yi[2 * kk + 1];
                }
                for (int a = 0; a < d; ++a) fft_axis(re, im, d, g.n, a, +1, lre, lim);
                double *yi = y + img * g.npix;
                double scale = 1.0 / (double)g.npix;
                for (int64_t p = 0; p < g.npix; ++p) yi[p] = re[p] * scale;
            }
        }
        free(re); free(im); free(lre); free(lim);
    }
    return err ? -4 : 0;
}

/* The whole layer: a1 -> a2 -> a3. */
int fno_oracle_spectral_conv(int d, const int64_t *n, const int32_t *m,
                             int64_t batch, int64_t cin, int64_t cout,
                             const double *x, const double *w, double *y)
{
    geom_t g;
    if (make_geom(&g, d, n, m)) return -1;
    double *X = malloc(sizeof(double) * 2 * batch * cin * g.nkept);
    double *Y = malloc(sizeof(double) * 2 * batch * cout * g.nkept);
    int rc = (X && Y) ? 0 : -4;
    if (!rc) rc = fno_oracle_forward_modes(d, n, m, batch * cin, x, X);
    if (!rc) rc = fno_oracle_mix(d, n, m, batch, cin, cout, X, w, Y);
    if (!rc) rc = fno_oracle_inverse_modes(d, n, m, batch * cout, Y, y);
    free(X);
    free(Y);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Gradients of the layer for a real loss L, given dy = dL/dy.  The pages print
 * no backward pass; these are the derivatives of the forward definition above,
 * with the usual convention for a complex quantity z: dz = dL/dRe(z) + i dL/dIm(z).
 *   y = (1/prod N) sum_k c(k_last) Re(Y_k e^{+i theta})      (step a3)
 *       => dY_k = (c(k_last)/prod N) sum_n dy_n e^{-i theta}  (the forward DFT of dy)
 *   Y[b,o,k] = sum_i X[b,i,k] W[i,o,k]                        (step a2)
 *       => dX[b,i,k] = sum_o dY[b,o,k] conj(W[i,o,k])
 *          dW[i,o,k] = sum_b dY[b,o,k] conj(X[b,i,k])
 *   X_k = sum_n x_n e^{-i theta}                              (step a1)
 *       => dx_n = sum_{k kept} Re(dX_k e^{+i theta})
 * dx is the real part of the unnormalised inverse complex FFT of the full
 * spectrum that holds dX at the kept positions and zero elsewhere (each kept
 * mode once, no half-spectrum weight).                                      */

/* dx of nimg images from their kept-mode gradients dX.                      */
int fno_oracle_adjoint_modes(int d, const int64_t *n, const int32_t *m,
                             int64_t nimg, const double *dX, double *dx)
{
    geom_t g;
    if (make_geom(&g, d, n, m)) return -1;
    int64_t maxn = 1;
    for (int a = 0; a < d; ++a) if (n[a] > maxn) maxn = n[a];
    int err = 0;
#pragma omp parallel
    {
        double *re = malloc(sizeof(double) * g.npix);
        double *im = malloc(sizeof(double) * g.npix);
        double *lre = malloc(sizeof(double) * maxn);
        double *lim = malloc(sizeof(double) * maxn);
        if (!re || !im || !lre || !lim) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t img = 0; img < nimg; ++img) {
                memset(re, 0, sizeof(double) * g.npix);
                memset(im, 0, sizeof(double) * g.npix);
                const double *Gi = dX + img * g.nkept * 2;
                for (int64_t kk = 0; kk < g.nkept; ++kk) {
                    int64_t f, b, l, kb;
                    kept_mode(&g, kk, &f, &b, &l, &kb);
                    re[f] = Gi[2 * kk];
                    im[f] = Gi[2 * kk + 1];
                }
                for (int a = 0; a < d; ++a) fft_axis(re, im, d, g.n, a, +1, lre, lim);
                double *o = dx + img * g.npix;
                for (int64_t p = 0; p < g.npix; ++p) o[p] = re[p];
            }
        }
        free(re); free(im); free(lre); free(lim);
    }
    return err ? -4 : 0;
}

/* The layer's gradients: dx (B, cin, N...) and dw (nblk, cin, cout, m...)
 * complex from x, w and dy (B, cout, N...).  Either output may be NULL.    */
int fno_oracle_spectral_conv_backward(int d, const int64_t *n, const int32_t *m,
                                      int64_t batch, int64_t cin, int64_t cout,
                                      const double *x, const double *w, const double *dy,
                                      double *dx, double *dw)
{
    geom_t g;
    if (make_geom(&g, d, n, m)) return -1;
    const int64_t nlast = n[d - 1];
    double *dY = malloc(sizeof(double) * 2 * batch * cout * g.nkept);
    double *X = malloc(sizeof(double) * 2 * batch * cin * g.nkept);
    int rc = (dY && X) ? 0 : -4;
    /* dY = c(k_last) / prod N * (forward DFT of dy at the kept modes) */
    if (!rc) rc = fno_oracle_forward_modes(d, n, m, batch * cout, dy, dY);
    if (!rc) {
        for (int64_t r = 0; r < batch * cout; ++r)
            for (int64_t kk = 0; kk < g.nkept; ++kk) {
                int64_t f, b, l, kb;
                kept_mode(&g, kk, &f, &b, &l, &kb);
                double c = (kb == 0 || 2 * kb == nlast) ? 1.0 : 2.0;
                dY[(r * g.nkept + kk) * 2] *= c / (double)g.npix;
                dY[(r * g.nkept + kk) * 2 + 1] *= c / (double)g.npix;
            }
    }
    if (!rc && dx) {
        /* dX[b,i,k] = sum_o dY[b,o,k] conj(W[blk,i,o,l]); dx = adjoint of the DFT */
#pragma omp parallel for collapse(2) schedule(static)
        for (int64_t b = 0; b < batch; ++b) {
            for (int64_t i = 0; i < cin; ++i) {
                for (int64_t kk = 0; kk < g.nkept; ++kk) {
                    int64_t f, blk, l, kb;
                    kept_mode(&g, kk, &f, &blk, &l, &kb);
                    double ar = 0.0, ai = 0.0;
                    for (int64_t o = 0; o < cout; ++o) {
                        const double *gv = dY + ((b * cout + o) * g.nkept + kk) * 2;
                        const double *wv = w + (((blk * cin + i) * cout + o) * g.mblk + l) * 2;
                        ar += gv[0] * wv[0] + gv[1] * wv[1];
                        ai += gv[1] * wv[0] - gv[0] * wv[1];
                    }
                    X[((b * cin + i) * g.nkept + kk) * 2] = ar;
                    X[((b * cin + i) * g.nkept + kk) * 2 + 1] = ai;
                }
            }
        }
        rc = fno_oracle_adjoint_modes(d, n, m, batch * cin, X, dx);
    }
    if (!rc && dw) {
        /* dW[blk,i,o,l] = sum_b dY[b,o,k] conj(X[b,i,k]), X the forward modes of x */
        rc = fno_oracle_forward_modes(d, n, m, batch * cin, x, X);
        if (!rc) {
#pragma omp parallel for collapse(2) schedule(static)
            for (int64_t i = 0; i < cin; ++i) {
                for (int64_t o = 0; o < cout; ++o) {
                    for (int64_t kk = 0; kk < g.nkept; ++kk) {
                        int64_t f, blk, l, kb;
                        kept_mode(&g, kk, &f, &blk, &l, &kb);
                        double ar = 0.0, ai = 0.0;
                        for (int64_t b = 0; b < batch; ++b) {
                            const double *gv = dY + ((b * cout + o) * g.nkept + kk) * 2;
                            const double *xv = X + ((b * cin + i) * g.nkept + kk) * 2;
                            ar += gv[0] * xv[0] + gv[1] * xv[1];
                            ai += gv[1] * xv[0] - gv[0] * xv[1];
                        }
                        double *wv = dw + (((blk * cin + i) * cout + o) * g.mblk + l) * 2;
                        wv[0] = ar;
                        wv[1] = ai;
                    }
                }
            }
        }
    }
    free(dY);
    free(X);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* FNO forward stack (2-D grid), channels-first:
 *   a_0 = L x + l_b                              (1x1 lift, cin_lift -> width)
 *   t_l = SpecConv_l(a_l) + P_l a_l + p_l         (l = 0 .. nlayers-1)
 *   a_{l+1} = gelu(t_l) for l < nlayers-1, t_l for the last layer
 *   h = gelu(Q1 a_L + q1)                         (width -> hidden)
 *   out = Q2 h + q2                               (hidden -> cout_proj)
 * Linear weights are (out, in) row-major.  gelu(v) = v/2 (1 + erf(v/sqrt 2)).
 * spec_w holds nlayers consecutive spectral weights, each (nblk, width,
 * width, m0, m1) complex.                                                   */
static double gelu(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

static void pointwise(int64_t batch, int64_t cin, int64_t cout, int64_t npix,
                      const double *a, const double *W, const double *bias,
                      double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t o = 0; o < cout; ++o) {
            double *dst = out + (b * cout + o) * npix;
            for (int64_t p = 0; p < npix; ++p) dst[p] = bias[o];
            for (int64_t i = 0; i < cin; ++i) {
                double wv = W[o * cin + i];
                const double *src = a + (b * cin + i) * npix;
                for (int64_t p = 0; p < npix; ++p) dst[p] += wv * src[p];
            }
        }
    }
}

int fno_oracle_fno_forward(int64_t batch, int64_t h, int64_t wdt,
                           const int32_t *modes, int64_t cin_lift,
                           int64_t width, int64_t nlayers, int64_t hidden,
                           int64_t cout_proj, const double *x,
                           const double *lift_w, const double *lift_b,
                           const double *spec_w, const double *pw_w,
                           const double *pw_b, const double *proj1_w,
                           const double *proj1_b, const double *proj2_w,
                           const double *proj2_b, double *out)
{
    int64_t n[2] = {h, wdt};
    geom_t g;
    if (make_geom(&g, 2, n, modes)) return -1;
    int64_t npix = h * wdt;
    int64_t act = batch * width * npix;
    double *a = malloc(sizeof(double) * act);
    double *s = malloc(sizeof(double) * act);
    double *t = malloc(sizeof(double) * act);
    double *hb = malloc(sizeof(double) * batch * hidden * npix);
    int rc = (a && s && t && hb) ? 0 : -4;
    if (!rc) pointwise(batch, cin_lift, width, npix, x, lift_w, lift_b, a);
    int64_t spec_stride = 2 * g.nblk * width * width * g.mblk;
    for (int64_t l = 0; l < nlayers && !rc; ++l) {
        rc = fno_oracle_spectral_conv(2, n, modes, batch, width, width, a,
                                      spec_w + l * spec_stride, s);
        if (rc) break;
        pointwise(batch, width, width, npix, a, pw_w + l * width * width,
                  pw_b + l * width, t);
        int last = (l == nlayers - 1);
        for (int64_t e = 0; e < act; ++e) {
            double v = s[e] + t[e];
            a[e] = last ? v : gelu(v);
        }
    }
    if (!rc) {
        pointwise(batch, width, hidden, npix, a, proj1_w, proj1_b, hb);
        for (int64_t e = 0; e < batch * hidden * npix; ++e) hb[e] = gelu(hb[e]);
        pointwise(batch, hidden, cout_proj, npix, hb, proj2_w, proj2_b, out);
    }
    free(a); free(s); free(t); free(hb);
    return rc;
}

/* Threads the oracle runs with (0 = library default). */
void fno_oracle_set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int fno_oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
