// fno_unfused.cu -- the layer as separate kernels, one per transform axis,
// one for the mixing, through the workspace.
//
// This is the "separate kernels" arrangement that the TurboFNO article
// (gsyq.cn/news/457482) measures against its fused kernel (§5.2 note): each
// step of §2.1-§2.3 is its own launch and the intermediates round-trip
// through device memory.  Every axis pass is a direct (dense) DFT over the
// kept frequencies only, so it is exact up to float rounding for any
// extent; it serves as the ablation baseline and covers shapes
// the fused kernels are not specialised for.
#include <algorithm>

#include "fno_fused.cuh"
#include "fno_internal.cuh"

namespace fno {
namespace {

constexpr int kThreads = 256;

struct KeptGeom {            // by-value kernel argument
    int d;
    int64_t kdim[FNO_MAX_NDIM];
    int32_t m[FNO_MAX_NDIM];
    int64_t nkept, mblk;
};

// (k n) mod N for a twiddle-table index: a mask for power-of-two N, else a
// remainder (the product stays below 2^31 for N <= 4096)
__device__ __forceinline__ int tw_idx(int prod, int N) {
    return (N & (N - 1)) == 0 ? (prod & (N - 1)) : (prod % N);
}

// Frequency of kept row r on a full axis: low rows 0..m-1, then high rows
// N-m..N-1 (TurboFNO §2.2 keeps the low-frequency modes; the high rows are
// the negative frequencies -m..-1 of the two-sided full axis).
__device__ __forceinline__ int kept_freq(int r, int m, int n) {
    return r < m ? r : n - 2 * m + r;
}

// Step a1, last axis: out[line][k] = sum_n x[line][n] e^{-2 pi i k n / N}, k < M,
// over the E <= N stored samples of a line (a padded line's other N - E
// samples are zeros and add nothing).
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_fwd_last(const T *__restrict__ x, float2 *__restrict__ out, int64_t nlines, int N, int E,
           int M, const float2 *__restrict__ tw, int *err) {
    const int64_t total = nlines * M;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t line = idx / M;
        const int k = (int)(idx - line * M);
        const T *src = x + line * E;
        float2 acc = make_float2(0.f, 0.f);
        if (!in_bounds(line * E + E - 1, nlines * E, err)) continue;
        for (int n = 0; n < E; ++n) {
            const float v = Storage<T>::load(src + n);
            const float2 w = tw[tw_idx(k * n, N)];
            acc.x = fmaf(v, w.x, acc.x);
            acc.y = fmaf(v, w.y, acc.y);
        }
        out[idx] = acc;
    }
}

// Step a1, one full axis: out[o][r][q] = sum_n in[o][n][q] e^{-2 pi i f(r) n / N},
// over the E <= N stored rows n (the others are zero padding).
__global__ void __launch_bounds__(kThreads)
k_fwd_full(const float2 *__restrict__ in, float2 *__restrict__ out, int64_t outer, int N,
           int E, int64_t inner, int m, const float2 *__restrict__ tw, int *err) {
    const int K = 2 * m;
    const int64_t total = outer * K * inner;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = idx % inner;
        const int64_t t = idx / inner;
        const int r = (int)(t % K);
        const int64_t o = t / K;
        const int f = kept_freq(r, m, N);
        const float2 *src = in + o * E * inner + q;
        float2 acc = make_float2(0.f, 0.f);
        if (!in_bounds(o * E * inner + q + (int64_t)(E - 1) * inner, outer * E * inner, err))
            continue;
        for (int n = 0; n < E; ++n) cfma(acc, src[n * inner], tw[tw_idx(f * n, N)]);
        out[idx] = acc;
    }
}

// Step a2: Y[b][o][k] = sum_i X[b][i][k] W[blk(k)][i][o][local(k)].
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_mix(const float2 *__restrict__ X, const T *__restrict__ w, float2 *__restrict__ Y,
      int64_t batch, int cin, int cout, KeptGeom g, int packed, int *err) {
    const int64_t total = batch * cout * g.nkept;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t kk = idx % g.nkept;
        const int64_t t = idx / g.nkept;
        const int o = (int)(t % cout);
        const int64_t b = t / cout;
        int64_t rem = kk, local = 0, stride = 1;
        int blk = 0;
        for (int a = g.d - 1; a >= 0; --a) {
            const int64_t r = rem % g.kdim[a];
            rem /= g.kdim[a];
            int64_t l = r;
            if (a < g.d - 1 && r >= g.m[a]) {
                l = r - g.m[a];
                blk |= 1 << a;
            }
            local += l * stride;
            stride *= g.m[a];
        }
        const float2 *xs = X + b * cin * g.nkept + kk;
        const T *ws = packed ? w + packed_index(kk, 0, o, cin, cout) * 2
                             : w + ((((int64_t)blk * cin) * cout + o) * g.mblk + local) * 2;
        const int64_t wstride = packed ? (int64_t)cout * 4 * 2 : (int64_t)cout * g.mblk * 2;
        float2 acc = make_float2(0.f, 0.f);
        const int64_t wl = (int64_t)g.nkept * cin * cout * 2;       // weight elements
        if (!in_bounds(b * cin * g.nkept + kk + (int64_t)(cin - 1) * g.nkept, batch * cin * g.nkept,
                       err) ||
            !in_bounds((ws - w) + (int64_t)(cin - 1) * wstride + 1, wl, err))
            continue;
        for (int i = 0; i < cin; ++i)
            cfma(acc, xs[(int64_t)i * g.nkept], Storage<T>::load2(ws + i * wstride));
        Y[idx] = acc;
    }
}

// Step a3, one full axis: out[o][n][q] = sum_r in[o][r][q] e^{+2 pi i f(r) n / N},
// for the first E <= N rows n only (the output crop of a padded axis).
__global__ void __launch_bounds__(kThreads)
k_inv_full(const float2 *__restrict__ in, float2 *__restrict__ out, int64_t outer, int N,
           int E, int64_t inner, int m, const float2 *__restrict__ tw, int *err) {
    const int K = 2 * m;
    const int64_t total = outer * E * inner;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = idx % inner;
        const int64_t t = idx / inner;
        const int n = (int)(t % E);
        const int64_t o = t / E;
        const float2 *src = in + o * K * inner + q;
        float2 acc = make_float2(0.f, 0.f);
        if (!in_bounds(o * K * inner + q + (int64_t)(K - 1) * inner, outer * K * inner, err))
            continue;
        for (int r = 0; r < K; ++r) {
            const float2 w = tw[tw_idx(kept_freq(r, m, N) * n, N)];
            cfma(acc, src[r * inner], make_float2(w.x, -w.y));   // conjugate twiddle
        }
        out[idx] = acc;
    }
}

// Step a3, last axis: y[line][n] = scale * sum_{k<M} c(k) Re(Y[k] e^{+2 pi i k n/N}),
// c(0) = c(N/2) = 1, c = 2 otherwise, for the first E <= N samples n of a line:
// the crop of a padded axis is this guarded store (TurboFNO §3.3), not a copy.
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_inv_last(const float2 *__restrict__ in, T *__restrict__ y, int64_t nlines, int N, int E,
           int M, const float2 *__restrict__ tw, float scale, int *err) {
    const int64_t total = nlines * E;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t line = idx / E;
        const int n = (int)(idx - line * E);
        const float2 *src = in + line * M;
        float acc = 0.f;
        if (!in_bounds(line * M + M - 1, nlines * M, err)) continue;
        for (int k = 0; k < M; ++k) {
            const float c = (k == 0 || 2 * k == N) ? 1.f : 2.f;
            const float2 v = src[k];
            const float2 w = tw[tw_idx(k * n, N)];
            // Re(v * conj(w)) with w = e^{-i theta}
            acc = fmaf(c, fmaf(v.x, w.x, v.y * w.y), acc);
        }
        Storage<T>::store(y + idx, acc * scale);
    }
}

int grid_for(int64_t total, int num_sms) {
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms * 16));
}

// Complex-element counts of every intermediate of the sequence.
void stage_sizes(const Geom &g, int64_t batch, int cin, int cout, int64_t *max_elems) {
    const int d = g.d;
    const int64_t ml = g.m[d - 1];
    int64_t best = 0;
    // forward: after the last axis, then after each full axis from d-2 down to 0
    int64_t s0 = batch * cin * ml;
    for (int j = 0; j < d - 1; ++j) s0 *= g.ext[j];
    best = std::max(best, s0);
    for (int a = d - 2; a >= 0; --a) {
        int64_t s = batch * cin * ml;
        for (int j = 0; j < d - 1; ++j) s *= (j < a) ? g.ext[j] : g.kdim[j];
        best = std::max(best, s);
    }
    best = std::max(best, batch * cin * g.nkept);
    best = std::max(best, batch * cout * g.nkept);
    // inverse: after expanding full axis a = 0..d-2
    for (int a = 0; a < d - 1; ++a) {
        int64_t s = batch * cout * ml;
        for (int j = 0; j < d - 1; ++j) s *= (j <= a) ? g.ext[j] : g.kdim[j];
        best = std::max(best, s);
    }
    *max_elems = best;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

size_t unfused_workspace_bytes(const Geom &g, int64_t batch, int cin, int cout) {
    int64_t e = 0;
    stage_sizes(g, batch, cin, cout, &e);
    return 2 * align256((size_t)e * sizeof(float2));
}

int unfused_kernel_count(const Geom &g) { return 2 * g.d + 1; }

template <typename T>
static cudaError_t unfused_forward_t(const Plan &p, const Buffers &bf, cudaStream_t s) {
    const Geom &g = p.g;
    const int d = g.d;
    const int64_t ml = g.m[d - 1];
    int64_t e = 0;
    stage_sizes(g, p.batch, p.cin, p.cout, &e);
    float2 *bufA = reinterpret_cast<float2 *>(bf.ws);
    float2 *bufB = reinterpret_cast<float2 *>(reinterpret_cast<char *>(bf.ws) +
                                              align256((size_t)e * sizeof(float2)));
    const int sms = p.num_sms;

    // a1, last axis (real -> half spectrum, truncated)
    int64_t lines = p.batch * p.cin;
    for (int j = 0; j < d - 1; ++j) lines *= g.ext[j];
    k_fwd_last<T><<<grid_for(lines * ml, sms), kThreads, 0, s>>>(
        reinterpret_cast<const T *>(bf.x), bufA, lines, (int)g.n[d - 1], (int)g.ext[d - 1],
        (int)ml, p.tw[d - 1], p.dev_err);
    float2 *cur = bufA, *nxt = bufB;
    // a1, full axes from d-2 down to 0
    for (int a = d - 2; a >= 0; --a) {
        int64_t outer = p.batch * p.cin, inner = ml;
        for (int j = 0; j < a; ++j) outer *= g.ext[j];
        for (int j = a + 1; j < d - 1; ++j) inner *= g.kdim[j];
        k_fwd_full<<<grid_for(outer * g.kdim[a] * inner, sms), kThreads, 0, s>>>(
            cur, nxt, outer, (int)g.n[a], (int)g.ext[a], inner, g.m[a], p.tw[a], p.dev_err);
        std::swap(cur, nxt);
    }
    // a2, mixing
    KeptGeom kg;
    kg.d = d;
    for (int a = 0; a < FNO_MAX_NDIM; ++a) {
        kg.kdim[a] = a < d ? g.kdim[a] : 1;
        kg.m[a] = a < d ? g.m[a] : 1;
    }
    kg.nkept = g.nkept;
    kg.mblk = g.mblk;
    k_mix<T><<<grid_for(p.batch * p.cout * g.nkept, sms), kThreads, 0, s>>>(
        cur, reinterpret_cast<const T *>(bf.w), nxt, p.batch, p.cin, p.cout, kg,
        (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0, p.dev_err);
    std::swap(cur, nxt);
    // a3, full axes 0..d-2
    for (int a = 0; a < d - 1; ++a) {
        int64_t outer = p.batch * p.cout, inner = ml;
        for (int j = 0; j < a; ++j) outer *= g.ext[j];
        for (int j = a + 1; j < d - 1; ++j) inner *= g.kdim[j];
        k_inv_full<<<grid_for(outer * g.ext[a] * inner, sms), kThreads, 0, s>>>(
            cur, nxt, outer, (int)g.n[a], (int)g.ext[a], inner, g.m[a], p.tw[a], p.dev_err);
        std::swap(cur, nxt);
    }
    // a3, last axis (half spectrum -> real), scale 1/prod(N) over the transform
    lines = p.batch * p.cout;
    for (int j = 0; j < d - 1; ++j) lines *= g.ext[j];
    k_inv_last<T><<<grid_for(lines * g.ext[d - 1], sms), kThreads, 0, s>>>(
        cur, reinterpret_cast<T *>(bf.y), lines, (int)g.n[d - 1], (int)g.ext[d - 1], (int)ml,
        p.tw[d - 1], (float)(1.0 / (double)g.ntr), p.dev_err);
    return cudaGetLastError();
}

int64_t unfused_modes_scratch_elems(const Geom &g, int64_t nch) {
    const int d = g.d;
    const int64_t ml = g.m[d - 1];
    int64_t best = 0;
    if (d > 1) {
        int64_t s0 = nch * ml;
        for (int j = 0; j < d - 1; ++j) s0 *= g.ext[j];
        best = s0;
    }
    // outputs of the full-axis passes a = d-2 .. 1 (the pass a = 0 writes out)
    for (int a = d - 2; a >= 1; --a) {
        int64_t s = nch * ml;
        for (int j = 0; j < d - 1; ++j) s *= (j < a) ? g.ext[j] : g.kdim[j];
        best = std::max(best, s);
    }
    return best;
}

template <typename T>
static cudaError_t forward_modes_t(const Plan &p, const T *x, int64_t nch, float2 *sa,
                                   float2 *sb, float2 *out, cudaStream_t s) {
    const Geom &g = p.g;
    const int d = g.d;
    const int64_t ml = g.m[d - 1];
    int64_t lines = nch;
    for (int j = 0; j < d - 1; ++j) lines *= g.ext[j];
    float2 *cur = d == 1 ? out : sa;
    k_fwd_last<T><<<grid_for(lines * ml, p.num_sms), kThreads, 0, s>>>(
        x, cur, lines, (int)g.n[d - 1], (int)g.ext[d - 1], (int)ml, p.tw[d - 1], p.dev_err);
    for (int a = d - 2; a >= 0; --a) {
        float2 *dst = a == 0 ? out : (cur == sa ? sb : sa);
        int64_t outer = nch, inner = ml;
        for (int j = 0; j < a; ++j) outer *= g.ext[j];
        for (int j = a + 1; j < d - 1; ++j) inner *= g.kdim[j];
        k_fwd_full<<<grid_for(outer * g.kdim[a] * inner, p.num_sms), kThreads, 0, s>>>(
            cur, dst, outer, (int)g.n[a], (int)g.ext[a], inner, g.m[a], p.tw[a], p.dev_err);
        cur = dst;
    }
    return cudaGetLastError();
}

cudaError_t unfused_forward_modes(const Plan &p, const void *x, int64_t nch, float2 *sa,
                                  float2 *sb, float2 *out, cudaStream_t s) {
    return with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        return forward_modes_t<T>(p, static_cast<const T *>(x), nch, sa, sb, out, s);
    });
}

// Packed weights, one destination element per thread (coalesced writes):
// wp[(q cin + i) cout + o][r] = w[blk(k)][i][o][local(k)], k = 4 q + r
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_pack_weights(const T *__restrict__ w, T *__restrict__ wp, int cin, int cout, KeptGeom g) {
    const int64_t total = g.nkept * cin * cout;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(idx & 3);
        int64_t t = idx >> 2;
        const int o = (int)(t % cout);
        t /= cout;
        const int i = (int)(t % cin);
        const int64_t kk = (t / cin) * 4 + r;
        int64_t rem = kk, local = 0, stride = 1;
        int blk = 0;
        for (int a = g.d - 1; a >= 0; --a) {
            const int64_t rr = rem % g.kdim[a];
            rem /= g.kdim[a];
            int64_t l = rr;
            if (a < g.d - 1 && rr >= g.m[a]) {
                l = rr - g.m[a];
                blk |= 1 << a;
            }
            local += l * stride;
            stride *= g.m[a];
        }
        const T *src = w + ((((int64_t)blk * cin + i) * cout + o) * g.mblk + local) * 2;
        wp[idx * 2] = src[0];
        wp[idx * 2 + 1] = src[1];
    }
}

cudaError_t launch_pack_weights(const Plan &p, const void *w, void *wp, cudaStream_t s) {
    const Geom &g = p.g;
    if (p.mix_image)      // the tensor-core mixing's operand images
        return mixtc_pack_image(p.dtype, w, wp, p.cin, p.cout, g.m[0], g.m[1], (int)g.mblk,
                                (int)g.nkept, p.num_sms, s);
    KeptGeom kg;
    kg.d = g.d;
    for (int a = 0; a < FNO_MAX_NDIM; ++a) {
        kg.kdim[a] = a < g.d ? g.kdim[a] : 1;
        kg.m[a] = a < g.d ? g.m[a] : 1;
    }
    kg.nkept = g.nkept;
    kg.mblk = g.mblk;
    const int grid = grid_for(g.nkept * p.cin * p.cout, p.num_sms);
    with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        k_pack_weights<T><<<grid, kThreads, 0, s>>>(static_cast<const T *>(w), static_cast<T *>(wp),
                                                    p.cin, p.cout, kg);
        return 0;
    });
    return cudaGetLastError();
}

cudaError_t launch_axis_forward(const float2 *in, float2 *out, int64_t outer, int n, int64_t inner,
                                int m, const float2 *tw, int num_sms, cudaStream_t s) {
    k_fwd_full<<<grid_for(outer * 2 * m * inner, num_sms), kThreads, 0, s>>>(in, out, outer, n,
                                                                           n, inner, m, tw,
                                                                           nullptr);
    return cudaGetLastError();
}

cudaError_t launch_axis_inverse(const float2 *in, float2 *out, int64_t outer, int n, int64_t inner,
                                int m, const float2 *tw, int num_sms, cudaStream_t s) {
    k_inv_full<<<grid_for(outer * n * inner, num_sms), kThreads, 0, s>>>(in, out, outer, n, n,
                                                                       inner, m, tw, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_mix(const Plan &p, const float2 *X, const void *w, float2 *Y, cudaStream_t s) {
    const Geom &g = p.g;
    KeptGeom kg;
    kg.d = g.d;
    for (int a = 0; a < FNO_MAX_NDIM; ++a) {
        kg.kdim[a] = a < g.d ? g.kdim[a] : 1;
        kg.m[a] = a < g.d ? g.m[a] : 1;
    }
    kg.nkept = g.nkept;
    kg.mblk = g.mblk;
    const int grid = grid_for(p.batch * p.cout * g.nkept, p.num_sms);
    with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        k_mix<T><<<grid, kThreads, 0, s>>>(X, static_cast<const T *>(w), Y, p.batch, p.cin,
                                          p.cout, kg, (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0,
                                          p.dev_err);
        return 0;
    });
    return cudaGetLastError();
}

cudaError_t unfused_forward(const Plan &p, const Buffers &b, cudaStream_t s) {
    return with_storage(p.dtype, [&](auto t) { return unfused_forward_t<decltype(t)>(p, b, s); });
}

}  // namespace fno
