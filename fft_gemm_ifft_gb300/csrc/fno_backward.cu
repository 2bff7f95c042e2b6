// fno_backward.cu -- gradients of the spectral-convolution layer.
//
// The TurboFNO article (gsyq.cn/news/457482) wraps its fused layer in an
// autograd function (§4.3) but prints only the forward pass; the backward here
// is the derivative of the forward definition (§2.1-§2.3) for a real loss L,
// with dz = dL/dRe(z) + i dL/dIm(z) for a complex z:
//
//   dY[b,o,k] = c(k_last) / prod(N) * F(dy)[b,o,k]     F = truncated forward DFT
//   dX[b,i,k] = sum_o dY[b,o,k] conj(W[blk,i,o,l])
//   dx        = sum over kept k of Re(dX_k e^{+2 pi i k.n/N})
//   dW[blk,i,o,l] = sum_b dY[b,o,k] conj(X[b,i,k]),   X = F(x)
//
// dx is exactly the forward layer applied to dy with W'[blk][o][i][l] =
// conj(W[blk][i][o][l]) (Cout inputs -> Cin outputs): the inverse step of the
// forward supplies the c(k)/prod(N) factor.  So dx reuses the fused forward
// kernels through the adjoint plan, after k_adjoint_weights writes W' into the
// workspace.  dW needs the kept modes of x and dy (the forward-transform kernel
// of the three-kernel path where the shape has one, else the per-axis DFT
// kernels) and one reduction over the batch per weight (k_grad_w).
#include <algorithm>

#include "fno_internal.cuh"

namespace fno {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t total, int num_sms) {
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms * 16));
}

struct ModeGeom {            // by-value kernel argument
    int d;
    int32_t m[FNO_MAX_NDIM];
    int64_t kdim[FNO_MAX_NDIM];
    int64_t nkept, mblk, nlast;
};

// W'[blk][o][i][l] = conj(W[blk][i][o][l]); the sign flip is exact in every
// storage type
template <typename T>
__global__ void __launch_bounds__(kThreads)
k_adjoint_weights(const T *__restrict__ w, T *__restrict__ wt, int64_t nblk, int cin, int cout,
                  int64_t mblk) {
    const int64_t total = nblk * cin * cout * mblk;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t l = idx % mblk;
        int64_t t = idx / mblk;
        const int i = (int)(t % cin);
        t /= cin;
        const int o = (int)(t % cout);
        const int64_t blk = t / cout;
        const T *src = w + (((blk * cin + i) * cout + o) * mblk + l) * 2;
        Storage<T>::store(wt + idx * 2, Storage<T>::load(src));
        Storage<T>::store(wt + idx * 2 + 1, -Storage<T>::load(src + 1));
    }
}

// dW[blk][i][o][l] = c / prod(N) sum_b G[b][o][k] conj(X[b][i][k]), k the kept
// mode of (blk, l), G = F(dy), X = F(x).  X and G may each be the sum of
// `parts` partial copies ([parts][images][|K|]).  A thread owns kOB
// consecutive outputs o of one (blk, i, l), so each X value it loads serves
// kOB products; consecutive threads take consecutive l (coalesced).
constexpr int kOB = 8;

template <typename T>
__global__ void __launch_bounds__(kThreads)
k_grad_w(const float2 *__restrict__ X, const float2 *__restrict__ G, int parts,
         T *__restrict__ dw, int64_t batch, int cin, int cout, int64_t nblk, ModeGeom mg,
         float inv_npix) {
    const int nog = (cout + kOB - 1) / kOB;
    const int64_t total = nblk * cin * nog * mg.mblk;
    const int64_t gstride = batch * cout * mg.nkept, xstride = batch * cin * mg.nkept;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t l = idx % mg.mblk;
        int64_t t = idx / mg.mblk;
        const int o0 = (int)(t % nog) * kOB;
        t /= nog;
        const int i = (int)(t % cin);
        const int blk = (int)(t / cin);
        // kept index: local index per axis, plus m_a on the high rows of a full axis
        int64_t rem = l, kk = 0, stride = 1, rlast = 0;
        for (int a = mg.d - 1; a >= 0; --a) {
            int64_t r = rem % mg.m[a];
            rem /= mg.m[a];
            if (a < mg.d - 1 && ((blk >> a) & 1)) r += mg.m[a];
            if (a == mg.d - 1) rlast = r;
            kk += r * stride;
            stride *= mg.kdim[a];
        }
        const float c = (rlast == 0 || 2 * rlast == mg.nlast) ? inv_npix : 2.f * inv_npix;
        const int no = min(kOB, cout - o0);
        float2 acc[kOB];
#pragma unroll
        for (int q = 0; q < kOB; ++q) acc[q] = make_float2(0.f, 0.f);
        for (int64_t b = 0; b < batch; ++b) {
            float2 x = make_float2(0.f, 0.f);
            for (int p = 0; p < parts; ++p) {
                const float2 xp = X[p * xstride + (b * cin + i) * mg.nkept + kk];
                x.x += xp.x;
                x.y += xp.y;
            }
#pragma unroll
            for (int q = 0; q < kOB; ++q) {
                if (q >= no) break;
                float2 g = make_float2(0.f, 0.f);
                for (int p = 0; p < parts; ++p) {
                    const float2 gp = G[p * gstride + (b * cout + o0 + q) * mg.nkept + kk];
                    g.x += gp.x;
                    g.y += gp.y;
                }
                acc[q].x = fmaf(g.x, x.x, fmaf(g.y, x.y, acc[q].x));     // g conj(x)
                acc[q].y = fmaf(g.y, x.x, fmaf(-g.x, x.y, acc[q].y));
            }
        }
#pragma unroll
        for (int q = 0; q < kOB; ++q) {
            if (q >= no) break;
            T *d = dw + ((((int64_t)blk * cin + i) * cout + o0 + q) * mg.mblk + l) * 2;
            Storage<T>::store(d, acc[q].x * c);
            Storage<T>::store(d + 1, acc[q].y * c);
        }
    }
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

BackwardLayout backward_layout(const Geom &g, int64_t batch, int cin, int cout,
                               size_t weight_bytes, size_t adjoint_workspace, int parts) {
    BackwardLayout l;
    const int64_t scratch =
        parts > 0 ? 0 : unfused_modes_scratch_elems(g, batch * std::max(cin, cout));
    const size_t copies = parts > 0 ? (size_t)parts : 1;
    l.wt = 0;
    l.adj = l.wt + align256(weight_bytes);
    l.x = l.adj + align256(adjoint_workspace);
    l.g = l.x + align256(copies * batch * cin * g.nkept * sizeof(float2));
    l.sa = l.g + align256(copies * batch * cout * g.nkept * sizeof(float2));
    l.sb = l.sa + align256((size_t)scratch * sizeof(float2));
    l.total = l.sb + align256((size_t)scratch * sizeof(float2));
    return l;
}

cudaError_t launch_adjoint_weights(const Plan &p, const void *w, void *wt, cudaStream_t s) {
    const int64_t total = p.g.nblk * p.cin * p.cout * p.g.mblk;
    with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        k_adjoint_weights<T><<<grid_for(total, p.num_sms), kThreads, 0, s>>>(
            static_cast<const T *>(w), static_cast<T *>(wt), p.g.nblk, p.cin, p.cout, p.g.mblk);
        return 0;
    });
    return cudaGetLastError();
}

cudaError_t launch_grad_w(const Plan &p, const float2 *X, const float2 *G, int parts, void *dw,
                          cudaStream_t s) {
    ModeGeom mg;
    mg.d = p.g.d;
    for (int a = 0; a < FNO_MAX_NDIM; ++a) {
        mg.m[a] = a < p.g.d ? p.g.m[a] : 1;
        mg.kdim[a] = a < p.g.d ? p.g.kdim[a] : 1;
    }
    mg.nkept = p.g.nkept;
    mg.mblk = p.g.mblk;
    mg.nlast = p.g.n[p.g.d - 1];
    const int64_t total = p.g.nblk * p.cin * ((p.cout + kOB - 1) / kOB) * p.g.mblk;
    const float inv_npix = (float)(1.0 / (double)p.g.ntr);
    with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        k_grad_w<T><<<grid_for(total, p.num_sms), kThreads, 0, s>>>(
            X, G, parts, static_cast<T *>(dw), p.batch, p.cin, p.cout, p.g.nblk, mg, inv_npix);
        return 0;
    });
    return cudaGetLastError();
}

}  // namespace fno
