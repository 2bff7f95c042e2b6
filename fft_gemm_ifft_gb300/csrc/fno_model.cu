// fno_model.cu -- the FNO forward stack on top of the spectral-conv plan.
//
// The stack is the model the TurboFNO article (gsyq.cn/news/457482) runs in
// its §5 tasks: a 1x1 lift, layers of [spectral convolution + 1x1 linear with
// bias, summed, GELU (none after the last layer)], and a two-layer 1x1
// projection with a GELU between.  Each spectral convolution runs through the
// layer plan (fused path); the 1x1 linears, bias, sum and GELU run here.
#include <cstring>
#include <new>

#include "fno_internal.cuh"

using namespace fno;

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCout = 8;

struct Model {
    fno_model_desc_t desc;
    fno_plan_t spec;
    int64_t npix;
    size_t act_bytes;      // one activation buffer (B, width, H, W) float32
    size_t spec_ws_bytes;
    size_t ws_bytes;
    int kernels;
};

__device__ __forceinline__ float gelu(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
}

int grid_for(int64_t total) {
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    return (int)(blocks < 65535 * 16 ? blocks : 65535 * 16);
}

// a[b][c][p] = sum_j W[c][j] x[b][j][p] + bias[c]   (1x1 linear, channels-first)
// optionally + add[b][c][p], optionally followed by GELU.
__global__ void __launch_bounds__(kThreads)
k_linear1x1(const float *__restrict__ x, const float *__restrict__ W,
            const float *__restrict__ bias, const float *__restrict__ add,
            float *__restrict__ out, int64_t batch, int cin, int cout, int64_t npix,
            int apply_gelu) {
    const int64_t total = batch * cout * npix;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = idx % npix;
        const int64_t t = idx / npix;
        const int c = (int)(t % cout);
        const int64_t b = t / cout;
        const float *src = x + b * cin * npix + p;
        const float *wr = W + (int64_t)c * cin;
        float acc = bias[c];
        for (int j = 0; j < cin; ++j) acc = fmaf(wr[j], src[(int64_t)j * npix], acc);
        if (add) acc += add[idx];
        out[idx] = apply_gelu ? gelu(acc) : acc;
    }
}

// out[b][o][p] = sum_k P2[o][k] gelu(sum_c P1[k][c] a[b][c][p] + c1[k]) + c2[o]
__global__ void __launch_bounds__(kThreads)
k_projection(const float *__restrict__ a, const float *__restrict__ P1,
             const float *__restrict__ c1, const float *__restrict__ P2,
             const float *__restrict__ c2, float *__restrict__ out, int64_t batch, int width,
             int hidden, int cout, int64_t npix) {
    const int64_t total = batch * npix;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = idx % npix;
        const int64_t b = idx / npix;
        const float *src = a + b * width * npix + p;
        float acc[kMaxCout];
        for (int o = 0; o < kMaxCout; ++o) acc[o] = o < cout ? c2[o] : 0.f;
        for (int k = 0; k < hidden; ++k) {
            float h = c1[k];
            const float *wr = P1 + (int64_t)k * width;
            for (int c = 0; c < width; ++c) h = fmaf(wr[c], src[(int64_t)c * npix], h);
            h = gelu(h);
#pragma unroll
            for (int o = 0; o < kMaxCout; ++o)
                if (o < cout) acc[o] = fmaf(P2[o * hidden + k], h, acc[o]);
        }
        for (int o = 0; o < cout; ++o) out[(b * cout + o) * npix + p] = acc[o];
    }
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

fno_status_t fno_model_plan(fno_model_t *out, const fno_model_desc_t *d) {
    if (!out) return FNO_ERR_INVALID_ARG;
    *out = nullptr;
    if (!d) return FNO_ERR_INVALID_ARG;
    if (d->batch < 1 || d->cin_lift < 1 || d->width < 1 || d->nlayers < 1 || d->hidden < 1 ||
        d->cout < 1)
        return FNO_ERR_INVALID_ARG;
    if (d->cout > kMaxCout) return FNO_ERR_UNSUPPORTED;
    if (d->dtype != FNO_F32) return FNO_ERR_UNSUPPORTED;
    const int64_t n[2] = {d->h, d->w};
    size_t spec_ws = 0;
    fno_status_t st = fno_spectral_conv_query(2, n, d->modes, d->batch, d->width, d->width,
                                              FNO_F32, d->flags, &spec_ws, nullptr);
    if (st != FNO_OK) return st;
    Model *m = new (std::nothrow) Model();
    if (!m) return FNO_ERR_OUT_OF_MEMORY;
    m->desc = *d;
    st = fno_spectral_conv_plan(&m->spec, 2, n, d->modes, d->batch, d->width, d->width,
                                FNO_F32, d->flags);
    if (st != FNO_OK) {
        delete m;
        return st;
    }
    int spec_kernels = 0;
    fno_spectral_conv_kernel_count(m->spec, &spec_kernels);
    m->npix = d->h * d->w;
    m->act_bytes = align256((size_t)d->batch * d->width * m->npix * sizeof(float));
    m->spec_ws_bytes = spec_ws;
    m->ws_bytes = 3 * m->act_bytes + align256(spec_ws);
    m->kernels = 1 + d->nlayers * (spec_kernels + 1) + 1;
    *out = reinterpret_cast<fno_model_t>(m);
    return FNO_OK;
}

fno_status_t fno_model_workspace_size(fno_model_t model, size_t *bytes) {
    if (!model || !bytes) return FNO_ERR_INVALID_ARG;
    *bytes = reinterpret_cast<Model *>(model)->ws_bytes;
    return FNO_OK;
}

fno_status_t fno_model_kernel_count(fno_model_t model, int *count) {
    if (!model || !count) return FNO_ERR_INVALID_ARG;
    *count = reinterpret_cast<Model *>(model)->kernels;
    return FNO_OK;
}

fno_status_t fno_forward(fno_model_t model, const void *x, const fno_model_params_t *p,
                         void *out, void *workspace, fno_stream_t stream) {
    if (!model || !x || !p || !out || !workspace) return FNO_ERR_INVALID_ARG;
    const Model &m = *reinterpret_cast<Model *>(model);
    const fno_model_desc_t &d = m.desc;
    const void *ptrs[] = {x, out, workspace, p->lift_w, p->lift_b, p->spec_w, p->pw_w,
                          p->pw_b, p->proj1_w, p->proj1_b, p->proj2_w, p->proj2_b};
    for (const void *q : ptrs) {
        if (!q) return FNO_ERR_INVALID_ARG;
        if (!aligned16(q)) return FNO_ERR_MISALIGNED;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    float *A = reinterpret_cast<float *>(ws);
    float *S = reinterpret_cast<float *>(ws + m.act_bytes);
    float *T = reinterpret_cast<float *>(ws + 2 * m.act_bytes);
    void *spec_ws = ws + 3 * m.act_bytes;
    const int64_t act = d.batch * d.width * m.npix;
    const size_t spec_stride = (size_t)2 * d.width * d.width * d.modes[0] * d.modes[1] * 2;

    k_linear1x1<<<grid_for(act), kThreads, 0, s>>>(
        static_cast<const float *>(x), p->lift_w, p->lift_b, nullptr, A, d.batch, d.cin_lift,
        d.width, m.npix, 0);
    if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
    for (int l = 0; l < d.nlayers; ++l) {
        fno_status_t st = fno_spectral_conv_forward(m.spec, A, p->spec_w + l * spec_stride, S,
                                                    m.spec_ws_bytes ? spec_ws : nullptr,
                                                    stream);
        if (st != FNO_OK) return st;
        const int last = (l == d.nlayers - 1);
        k_linear1x1<<<grid_for(act), kThreads, 0, s>>>(
            A, p->pw_w + (size_t)l * d.width * d.width, p->pw_b + (size_t)l * d.width, S, T,
            d.batch, d.width, d.width, m.npix, last ? 0 : 1);
        if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
        float *tmp = A;
        A = T;
        T = tmp;
    }
    k_projection<<<grid_for(d.batch * m.npix), kThreads, 0, s>>>(
        A, p->proj1_w, p->proj1_b, p->proj2_w, p->proj2_b, static_cast<float *>(out), d.batch,
        d.width, d.hidden, d.cout, m.npix);
    if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
    return FNO_OK;
}

fno_status_t fno_model_get_device_error(fno_model_t model, fno_stream_t stream) {
    if (!model) return FNO_ERR_INVALID_ARG;
    return fno_plan_get_device_error(reinterpret_cast<Model *>(model)->spec, stream);
}

fno_status_t fno_model_destroy(fno_model_t model) {
    if (!model) return FNO_OK;
    Model *m = reinterpret_cast<Model *>(model);
    fno_status_t st = fno_plan_destroy(m->spec);
    delete m;
    return st;
}

}  // extern "C"
