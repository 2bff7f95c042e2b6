// fno_model.cu -- the FNO forward stack on top of the spectral-conv plan.
//
// The stack is the model the TurboFNO article (gsyq.cn/news/457482) runs in
// its §5 tasks: a 1x1 lift, layers of [spectral convolution + 1x1 linear with
// bias, summed, GELU (none after the last layer)], and a two-layer 1x1
// projection with a GELU between.  Each spectral convolution runs through the
// layer plan (fused path); the 1x1 linears, bias, sum and GELU run here.
#include <algorithm>
#include <cstring>
#include <new>
#include <type_traits>

#include "fno_internal.cuh"
#include "fno_fused.cuh"
#include "fno_gelu.cuh"
#include "fno_head.cuh"
#include "fno_layer.cuh"
#include "fno_pointwise.cuh"

using namespace fno;

namespace {

constexpr int kMaxCout = 8;

struct Model {
    fno_model_desc_t desc;
    fno_plan_t spec;
    int64_t npix;
    size_t act_bytes;      // one activation buffer (B, width, H, W) in the storage type
    size_t spec_ws_bytes;
    size_t ws_bytes;
    int kernels;
    // which 1x1 linears run on the tensor cores (fno_pointwise.cu; otherwise
    // the register-tiled SIMT kernels below)
    bool lift_simt, lift_tc, layer_tc, head_tc;
    // heads whose shape fits it: the persistent head kernel (fno_head.cu)
    bool head_fast;
    // the float32 128 x 128 layers: the spectral plan's forward transform and
    // mixing, then the column step and ONE GEMM for the inverse row DFT and the
    // 1x1 linear (fno_layer.cu) instead of the inverse kernel and the linear
    bool layer_fused;
    size_t z_off;          // the column step's output in the workspace
    void *row_table;       // the inverse row-DFT operand (model-owned)
    int num_sms;
};

// GELU(v) = v/2 (1 + erf(v / sqrt 2)), erf by Abramowitz & Stegun 7.1.26
// (fno_gelu.cuh; |error of erf| <= 1.5e-7)
__device__ __forceinline__ float gelu(float v) { return gelu_erf(v); }

// ---------------------------------------------------------------------------
// Register-tiled 1x1 linears.  A CTA of kTT threads owns kTP pixels of one
// image and kTO output channels; the input channels are staged kTK at a time
// in shared memory (cp.async, zero-filled past the edges), together with the
// matching weight columns stored transposed.  Thread (og, pg) accumulates 4
// outputs x 8 pixels (pixels pg*4.. and 64+pg*4..), so every k step is one
// float4 weight load (a broadcast: a warp touches two og) and two float4
// activation loads (conflict-free) for 32 FMAs.  The pixel count must be a
// multiple of 4 (the 16-byte copies); channel counts are arbitrary.
// ---------------------------------------------------------------------------
constexpr int kTT = 256;   // threads per CTA
constexpr int kTP = 128;   // pixels per tile
constexpr int kTO = 64;    // output channels per tile
constexpr int kTK = 64;    // input channels per shared-memory chunk

struct TileSmem {
    float a[kTK][kTP];     // activations [k][pixel]
    float w[kTK][kTO];     // weights, transposed [k][output]
    float red[kTT / 16][kTP];   // projection: partial sums of the 16 output groups
};

__device__ __forceinline__ void cp_async16(void *s, const void *g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 ::"r"((unsigned)__cvta_generic_to_shared(s)), "l"(g) : "memory");
}

// Input channels [k0, k0 + kc) of pixels [p0, p0 + kTP) of one image (a_img,
// in the activation storage type; float32 in shared memory), and the weights
// W[o0 + o][k0 + k] (row length cin) of outputs o < no.
template <typename T>
__device__ void load_chunk(TileSmem &s, const T *__restrict__ a_img, int cin, int64_t npix,
                           int64_t p0, int k0, int kc, const float *__restrict__ W, int o0,
                           int no) {
    const int tid = threadIdx.x;
    for (int e = tid; e < kTK * (kTP / 4); e += kTT) {
        const int k = e / (kTP / 4), g = e % (kTP / 4);
        const int64_t px = p0 + 4 * g;
        float *dst = &s.a[k][4 * g];
        const bool in = k < kc && px < npix;
        if constexpr (std::is_same<T, float>::value) {
            if (in)
                cp_async16(dst, a_img + (int64_t)(k0 + k) * npix + px);
            else
                *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            *reinterpret_cast<float4 *>(dst) =
                in ? Storage<T>::load4(a_img + (int64_t)(k0 + k) * npix + px)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    for (int e = tid; e < kTK * kTO; e += kTT) {
        const int k = e / kTO, o = e % kTO;
        s.w[k][o] = (k < kc && o < no) ? W[(int64_t)(o0 + o) * cin + k0 + k] : 0.f;
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
}

// acc[i][j] += sum_k w[k][og*4 + i] a[k][pix(j)], pix(j) = pg*4 + j (j < 4), 64 + pg*4 + j - 4
__device__ __forceinline__ void fma_chunk(const TileSmem &s, int kc, int og, int pg,
                                          float (&acc)[4][8]) {
#pragma unroll 4
    for (int k = 0; k < kc; ++k) {
        const float4 w4 = *reinterpret_cast<const float4 *>(&s.w[k][og * 4]);
        const float4 a0 = *reinterpret_cast<const float4 *>(&s.a[k][pg * 4]);
        const float4 a1 = *reinterpret_cast<const float4 *>(&s.a[k][64 + pg * 4]);
        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(wv[i], av[j], acc[i][j]);
    }
}

// out[b][o][p] = act(sum_j W[o][j] x[b][j][p] + bias[o] (+ add[b][o][p])); x, add
// and out in the activation storage type T, arithmetic in float32
// grid: (pixel tiles, output tiles, batch)
template <typename T>
__global__ void __launch_bounds__(kTT)
k_linear_tiled(const T *__restrict__ x, const float *__restrict__ W,
               const float *__restrict__ bias, const T *__restrict__ add,
               T *__restrict__ out, int cin, int cout, int64_t npix, int apply_gelu) {
    extern __shared__ __align__(16) char smem_raw[];
    TileSmem &s = *reinterpret_cast<TileSmem *>(smem_raw);
    const int64_t p0 = (int64_t)blockIdx.x * kTP;
    const int o0 = blockIdx.y * kTO, no = min(kTO, cout - o0);
    const int64_t b = blockIdx.z;
    const int og = threadIdx.x / 16, pg = threadIdx.x % 16;
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    const T *a_img = x + b * cin * npix;
    for (int k0 = 0; k0 < cin; k0 += kTK) {
        const int kc = min(kTK, cin - k0);
        load_chunk<T>(s, a_img, cin, npix, p0, k0, kc, W, o0, no);
        fma_chunk(s, kc, og, pg, acc);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int o = og * 4 + i;
        if (o >= no) continue;
        const float bo = bias[o0 + o];
        const int64_t row = (b * cout + o0 + o) * npix;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t px = p0 + h * 64 + pg * 4;
            if (px >= npix) continue;
            float4 v = make_float4(acc[i][4 * h] + bo, acc[i][4 * h + 1] + bo,
                                   acc[i][4 * h + 2] + bo, acc[i][4 * h + 3] + bo);
            if (add) {
                float4 q;
                if constexpr (std::is_same<T, float>::value)
                    q = __ldcs(reinterpret_cast<const float4 *>(add + row + px));
                else
                    q = Storage<T>::load4(add + row + px);
                v.x += q.x; v.y += q.y; v.z += q.z; v.w += q.w;
            }
            if (apply_gelu) {
                v.x = gelu(v.x); v.y = gelu(v.y); v.z = gelu(v.z); v.w = gelu(v.w);
            }
            Storage<T>::store4(out + row + px, v);
        }
    }
}

// out[b][o][p] = sum_k P2[o][k] gelu(sum_c P1[k][c] a[b][c][p] + c1[k]) + c2[o], o < cout
// grid: (pixel tiles, batch); the hidden units run in tiles of kTO; kCo >= cout
// partial outputs are held per thread
template <int kCo, typename T>
__global__ void __launch_bounds__(kTT)
k_projection_tiled(const T *__restrict__ a, const float *__restrict__ P1,
                   const float *__restrict__ c1, const float *__restrict__ P2,
                   const float *__restrict__ c2, T *__restrict__ out, int width, int hidden,
                   int cout, int64_t npix) {
    extern __shared__ __align__(16) char smem_raw[];
    TileSmem &s = *reinterpret_cast<TileSmem *>(smem_raw);
    const int64_t p0 = (int64_t)blockIdx.x * kTP;
    const int64_t b = blockIdx.y;
    const int og = threadIdx.x / 16, pg = threadIdx.x % 16;
    const T *a_img = a + b * width * npix;
    float part[kCo][8];
#pragma unroll
    for (int o = 0; o < kCo; ++o)
#pragma unroll
        for (int j = 0; j < 8; ++j) part[o][j] = 0.f;
    for (int h0 = 0; h0 < hidden; h0 += kTO) {
        const int nh = min(kTO, hidden - h0);
        float acc[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
        for (int k0 = 0; k0 < width; k0 += kTK) {
            const int kc = min(kTK, width - k0);
            load_chunk<T>(s, a_img, width, npix, p0, k0, kc, P1, h0, nh);
            fma_chunk(s, kc, og, pg, acc);
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int h = og * 4 + i;
            if (h >= nh) continue;
            const float ch = c1[h0 + h];
#pragma unroll
            for (int o = 0; o < kCo; ++o) {
                if (o >= cout) break;
                const float p2 = P2[(int64_t)o * hidden + h0 + h];
#pragma unroll
                for (int j = 0; j < 8; ++j) part[o][j] = fmaf(p2, gelu(acc[i][j] + ch), part[o][j]);
            }
        }
    }
    // sum the 16 output groups' partials of every pixel
    for (int o = 0; o < cout; ++o) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v = 0.f;
#pragma unroll
            for (int q = 0; q < kCo; ++q)
                if (q == o) v = part[q][j];
            s.red[og][(j < 4 ? 0 : 64) + pg * 4 + (j & 3)] = v;
        }
        __syncthreads();
        if (threadIdx.x < kTP && p0 + threadIdx.x < npix) {
            float v = c2[o];
            for (int g = 0; g < kTT / 16; ++g) v += s.red[g][threadIdx.x];
            Storage<T>::store(out + (b * cout + o) * npix + p0 + threadIdx.x, v);
        }
        __syncthreads();
    }
}


// The lift of a few input channels (the field and its coordinates) to the
// model width: a pure write stream (each output value costs cin FMAs), so a
// thread takes 4 consecutive pixels of one image, reads them once per input
// channel and writes its 4 pixels of every output channel (a warp: 512
// contiguous bytes per channel).
constexpr int kLiftMaxCin = 8;
constexpr int kLiftThreads = 256;
template <typename T>
__global__ void __launch_bounds__(kLiftThreads)
k_lift(const T *__restrict__ x, const float *__restrict__ W, const float *__restrict__ bias,
       T *__restrict__ out, int cin, int cout, int64_t npix) {
    extern __shared__ float s_wb[];                  // W [cout][cin], then bias [cout]
    for (int e = threadIdx.x; e < cout * (cin + 1); e += kLiftThreads)
        s_wb[e] = e < cout * cin ? W[e] : bias[e - cout * cin];
    __syncthreads();
    const int b = blockIdx.y;
    const int64_t p = ((int64_t)blockIdx.x * kLiftThreads + threadIdx.x) * 4;
    if (p >= npix) return;
    float4 xv[kLiftMaxCin];
#pragma unroll
    for (int i = 0; i < kLiftMaxCin; ++i)
        if (i < cin) xv[i] = Storage<T>::load4(x + ((int64_t)b * cin + i) * npix + p);
    T *op = out + (int64_t)b * cout * npix + p;
    for (int o = 0; o < cout; ++o) {
        const float bo = s_wb[cout * cin + o];
        float4 y = make_float4(bo, bo, bo, bo);
#pragma unroll
        for (int i = 0; i < kLiftMaxCin; ++i) {
            if (i < cin) {
                const float w = s_wb[o * cin + i];
                y.x = fmaf(w, xv[i].x, y.x);
                y.y = fmaf(w, xv[i].y, y.y);
                y.z = fmaf(w, xv[i].z, y.z);
                y.w = fmaf(w, xv[i].w, y.w);
            }
        }
        Storage<T>::store4(op + (int64_t)o * npix, y);
    }
}

template <typename T>
using ProjFn = void (*)(const T *, const float *, const float *, const float *,
                        const float *, T *, int, int, int, int64_t);
template <typename T>
ProjFn<T> projection_kernel(int cout) {
    if (cout <= 1) return k_projection_tiled<1, T>;
    if (cout <= 2) return k_projection_tiled<2, T>;
    if (cout <= 4) return k_projection_tiled<4, T>;
    return k_projection_tiled<kMaxCout, T>;
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
    if (d->cout > kMaxCout || d->batch > 65535) return FNO_ERR_UNSUPPORTED;
    // the tiled 1x1 linears move pixel rows in 16-byte copies
    if ((d->h * d->w) % 4 != 0) return FNO_ERR_UNSUPPORTED;
    if (d->dtype != FNO_F32 && d->dtype != FNO_F16 && d->dtype != FNO_BF16)
        return FNO_ERR_INVALID_ARG;
    const int64_t n[2] = {d->h, d->w};
    size_t spec_ws = 0;
    fno_status_t st = fno_spectral_conv_query(2, n, d->modes, d->batch, d->width, d->width,
                                              d->dtype, d->flags, &spec_ws, nullptr);
    if (st != FNO_OK) return st;
    Model *m = new (std::nothrow) Model();
    if (!m) return FNO_ERR_OUT_OF_MEMORY;
    m->desc = *d;
    st = fno_spectral_conv_plan(&m->spec, 2, n, d->modes, d->batch, d->width, d->width,
                                d->dtype, d->flags);
    if (st != FNO_OK) {
        delete m;
        return st;
    }
    const int smem = (int)sizeof(TileSmem);
    const cudaError_t se = with_storage(d->dtype, [&](auto t) {
        using T = decltype(t);
        cudaError_t e = raise_smem_limit(k_linear_tiled<T>, smem);
        return e == cudaSuccess ? raise_smem_limit(projection_kernel<T>(d->cout), smem) : e;
    });
    if (se != cudaSuccess) {
        cudaGetLastError();
        fno_plan_destroy(m->spec);
        delete m;
        return FNO_ERR_CUDA;
    }
    // tensor-core linears where the channel counts fit their tiles
    int dev = 0;
    cudaGetDevice(&dev);
    m->num_sms = 0;
    cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t npix = d->h * d->w;
    // a lift of up to 8 channels is a write stream: its own kernel
    m->lift_simt = d->cin_lift <= kLiftMaxCin &&
                   (size_t)d->width * (d->cin_lift + 1) * sizeof(float) <= (48u << 10);
    m->lift_tc = !m->lift_simt &&
                 pointwise_supported(d->dtype, d->cin_lift, d->width, 0, false, npix);
    m->layer_tc = pointwise_supported(d->dtype, d->width, d->width, 0, false, npix);
    m->head_fast = head_supported(d->dtype, d->width, d->hidden, d->cout, npix);
    m->head_tc = !m->head_fast &&
                 pointwise_supported(d->dtype, d->width, d->hidden, d->cout, true, npix);
    if ((m->lift_tc && pointwise_init(d->dtype, d->cin_lift, d->width, 0, false) != cudaSuccess) ||
        (m->layer_tc && pointwise_init(d->dtype, d->width, d->width, 0, false) != cudaSuccess) ||
        (m->head_tc && pointwise_init(d->dtype, d->width, d->hidden, d->cout, true) != cudaSuccess) ||
        (m->head_fast && head_init(d->dtype, d->width, d->hidden, d->cout) != cudaSuccess)) {
        cudaGetLastError();
        fno_plan_destroy(m->spec);
        delete m;
        return FNO_ERR_CUDA;
    }
    int spec_kernels = 0;
    fno_spectral_conv_kernel_count(m->spec, &spec_kernels);
    m->npix = d->h * d->w;
    m->act_bytes = align256((size_t)d->batch * d->width * m->npix * (d->dtype == FNO_F32 ? 4 : 2));
    m->spec_ws_bytes = spec_ws;
    m->ws_bytes = 3 * m->act_bytes + align256(spec_ws);
    m->layer_fused = !(d->flags & FNO_PLAN_SPLIT_LAYER) && d->h == 128 && d->w == 128 &&
                     d->modes[0] == 16 && d->modes[1] == 16 &&
                     fused_mixed_available(*reinterpret_cast<Plan *>(m->spec)) &&
                     layer_out_supported(d->width, d->batch);
    m->row_table = nullptr;
    if (m->layer_fused) {
        std::vector<unsigned char> img;
        inverse_row_operand_tf32(img);
        cudaError_t e = layer_out_init(d->dtype, d->width);
        if (e == cudaSuccess) e = cudaMalloc(&m->row_table, img.size());
        if (e == cudaSuccess)
            e = cudaMemcpy(m->row_table, img.data(), img.size(), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cudaGetLastError();
            if (m->row_table) cudaFree(m->row_table);
            fno_plan_destroy(m->spec);
            delete m;
            return FNO_ERR_CUDA;
        }
        m->z_off = m->ws_bytes;
        m->ws_bytes += align256(layer_out_z_bytes(d->batch, d->width));
    }
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
    return with_storage(d.dtype, [&](auto t) -> fno_status_t {
        using T = decltype(t);
        char *ws = static_cast<char *>(workspace);
        T *A = reinterpret_cast<T *>(ws);
        T *S = reinterpret_cast<T *>(ws + m.act_bytes);
        T *Tn = reinterpret_cast<T *>(ws + 2 * m.act_bytes);
        void *spec_ws = ws + 3 * m.act_bytes;
        // one layer's spectral weights, in elements of the storage type
        const size_t spec_stride = (size_t)2 * d.width * d.width * d.modes[0] * d.modes[1] * 2;
        const T *spec_w = static_cast<const T *>(p->spec_w);

        const unsigned ptiles = (unsigned)((m.npix + kTP - 1) / kTP);
        int *err = reinterpret_cast<Plan *>(m.spec)->dev_err;
        const dim3 lin_grid(ptiles, (unsigned)((d.width + kTO - 1) / kTO), (unsigned)d.batch);
        const size_t smem = sizeof(TileSmem);
        // a tensor-core linear: out = act(W a + bias (+ add)), or the head
        auto linear_tc = [&](const void *a, int cin, const float *W, const float *bias,
                             const void *add, void *o, int n, int gelu) {
            PointwiseArgs pa{};
            pa.a = a;
            pa.W = W;
            pa.bias = bias;
            pa.add = add;
            pa.out = o;
            pa.cin = cin;
            pa.n = n;
            pa.batch = d.batch;
            pa.npix = m.npix;
            pa.gelu = gelu;
            pa.err = err;
            return pointwise_launch(d.dtype, pa, m.num_sms, s);
        };
        if (m.lift_simt) {
            const dim3 grid((unsigned)((m.npix / 4 + kLiftThreads - 1) / kLiftThreads),
                            (unsigned)d.batch);
            k_lift<T><<<grid, kLiftThreads,
                        (size_t)d.width * (d.cin_lift + 1) * sizeof(float), s>>>(
                static_cast<const T *>(x), p->lift_w, p->lift_b, A, d.cin_lift, d.width, m.npix);
        } else if (m.lift_tc) {
            if (linear_tc(x, d.cin_lift, p->lift_w, p->lift_b, nullptr, A, d.width, 0) !=
                cudaSuccess)
                return FNO_ERR_CUDA;
        } else {
            k_linear_tiled<T><<<lin_grid, kTT, smem, s>>>(static_cast<const T *>(x), p->lift_w,
                                                          p->lift_b, nullptr, A, d.cin_lift,
                                                          d.width, m.npix, 0);
        }
        if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
        for (int l = 0; l < d.nlayers; ++l) {
            const int last = (l == d.nlayers - 1);
            const float *W = p->pw_w + (size_t)l * d.width * d.width;
            const float *bias = p->pw_b + (size_t)l * d.width;
            {
                if (m.layer_fused) {
                    const Plan &sp = *reinterpret_cast<const Plan *>(m.spec);
                    const Buffers b{A, spec_w + l * spec_stride, nullptr, spec_ws};
                    LayerOutArgs la{};
                    if (fused_forward_mixed(sp, b, &la.Y, s) != cudaSuccess) return FNO_ERR_CUDA;
                    la.tw = sp.tw[0];
                    la.Z = reinterpret_cast<float *>(ws + m.z_off);
                    la.x = A;
                    la.W = W;
                    la.bias = bias;
                    la.out = Tn;
                    la.table = m.row_table;
                    la.batch = d.batch;
                    la.dtype = d.dtype;
                    la.width = d.width;
                    la.gelu = last ? 0 : 1;
                    la.err = err;
                    if (layer_out_launch(la, m.num_sms, s) != cudaSuccess) return FNO_ERR_CUDA;
                    T *tmp = A;
                    A = Tn;
                    Tn = tmp;
                    continue;
                }
            }
            fno_status_t st = fno_spectral_conv_forward(m.spec, A, spec_w + l * spec_stride, S,
                                                        m.spec_ws_bytes ? spec_ws : nullptr,
                                                        stream);
            if (st != FNO_OK) return st;
            if (m.layer_tc) {
                if (linear_tc(A, d.width, W, bias, S, Tn, d.width, last ? 0 : 1) != cudaSuccess)
                    return FNO_ERR_CUDA;
            } else {
                k_linear_tiled<T><<<lin_grid, kTT, smem, s>>>(A, W, bias, S, Tn, d.width,
                                                              d.width, m.npix, last ? 0 : 1);
            }
            if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
            T *tmp = A;
            A = Tn;
            Tn = tmp;
        }
        bool head_done = false;
        {
            if (m.head_fast) {
                HeadArgs ha{};
                ha.a = A;
                ha.W = p->proj1_w;
                ha.bias = p->proj1_b;
                ha.P2 = p->proj2_w;
                ha.c2 = p->proj2_b;
                ha.out = out;
                ha.cin = d.width;
                ha.hidden = d.hidden;
                ha.cout2 = d.cout;
                ha.batch = d.batch;
                ha.npix = m.npix;
                ha.dtype = d.dtype;
                ha.err = err;
                if (head_launch(ha, m.num_sms, s) != cudaSuccess) return FNO_ERR_CUDA;
                head_done = true;
            }
        }
        if (head_done) {
        } else if (m.head_tc) {
            PointwiseArgs pa{};
            pa.a = A;
            pa.W = p->proj1_w;
            pa.bias = p->proj1_b;
            pa.P2 = p->proj2_w;
            pa.c2 = p->proj2_b;
            pa.out = out;
            pa.cin = d.width;
            pa.n = d.hidden;
            pa.cout2 = d.cout;
            pa.batch = d.batch;
            pa.npix = m.npix;
            pa.gelu = 1;
            pa.head = 1;
            pa.err = err;
            if (pointwise_launch(d.dtype, pa, m.num_sms, s) != cudaSuccess) return FNO_ERR_CUDA;
        } else {
            projection_kernel<T>(d.cout)<<<dim3(ptiles, (unsigned)d.batch), kTT, smem, s>>>(
                A, p->proj1_w, p->proj1_b, p->proj2_w, p->proj2_b, static_cast<T *>(out),
                d.width, d.hidden, d.cout, m.npix);
        }
        if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
        return FNO_OK;
    });
}

fno_status_t fno_model_get_device_error(fno_model_t model, fno_stream_t stream) {
    if (!model) return FNO_ERR_INVALID_ARG;
    return fno_plan_get_device_error(reinterpret_cast<Model *>(model)->spec, stream);
}

fno_status_t fno_model_destroy(fno_model_t model) {
    if (!model) return FNO_OK;
    Model *m = reinterpret_cast<Model *>(model);
    fno_status_t st = fno_plan_destroy(m->spec);
    if (m->row_table) cudaFree(m->row_table);
    delete m;
    return st;
}

}  // extern "C"
