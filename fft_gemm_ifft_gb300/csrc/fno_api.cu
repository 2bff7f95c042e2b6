// fno_api.cu -- the C ABI: argument validation, plans, dispatch, errors.
//
// The boundary follows §4.3 of the TurboFNO article (gsyq.cn/news/457482): a
// C function in a shared library that receives raw device pointers and runs
// the fused layer on a stream, bypassing any framework dispatch.  Nothing here
// allocates in the forward call, so a forward is capturable in a CUDA graph
// (the article's §2.3 / §3.3 point about a compile-time output size).
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "fno_internal.cuh"
#include "fno_fused.cuh"

using namespace fno;

namespace fno {

cudaError_t raise_smem_limit_fn(const void *fn, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> limit;   // (device, kernel)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t &cur = limit[{dev, fn}];
    if (bytes <= cur) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) cur = bytes;
    return e;
}

}  // namespace fno

namespace {

constexpr int kVersion = 10000;   // 1.0.0
constexpr int64_t kMaxN = 4096;

// Host-side fault injection for the failure-path tests: FNO_FAULT_INJECT names
// one site ("plan_alloc" or "launch") at which the library behaves as if the
// CUDA call there had failed.  No device fault is involved.
bool inject(const char *site) {
    const char *v = std::getenv("FNO_FAULT_INJECT");
    return v && std::strcmp(v, site) == 0;
}


// pad == NULL: a periodic layer; else the transform of axis a runs over
// n[a] + pad[a] points of which the last pad[a] are zeros (and are not stored).
fno_status_t make_geom(Geom *g, int ndim, const int64_t *n, const int32_t *modes,
                       const int64_t *pad = nullptr) {
    if (ndim < 1 || ndim > FNO_MAX_NDIM || !n || !modes) return FNO_ERR_INVALID_ARG;
    std::memset(g, 0, sizeof(*g));
    g->d = ndim;
    g->nkept = g->npix = g->ntr = g->nblk = g->mblk = 1;
    for (int a = 0; a < ndim; ++a) {
        const int64_t p = pad ? pad[a] : 0;
        if (p < 0 || n[a] < 1) return FNO_ERR_INVALID_ARG;
        if (n[a] > kMaxN || p > kMaxN) return FNO_ERR_UNSUPPORTED;
        g->ext[a] = n[a];
        g->padded |= p > 0;
        const int64_t len = n[a] + p;               // transform length
        if (len < 2) return FNO_ERR_INVALID_ARG;
        if (len > kMaxN) return FNO_ERR_UNSUPPORTED;
        const int64_t m = modes[a];
        if (m < 1) return FNO_ERR_INVALID_ARG;
        if (a < ndim - 1) {
            if (2 * m > len) return FNO_ERR_INVALID_ARG;    // corner blocks may not overlap
            g->kdim[a] = 2 * m;
            g->nblk *= 2;
        } else {
            if (m > len / 2 + 1) return FNO_ERR_INVALID_ARG;
            g->kdim[a] = m;
        }
        g->n[a] = len;
        g->m[a] = (int32_t)m;
        g->nkept *= g->kdim[a];
        g->npix *= n[a];
        g->ntr *= len;
        g->mblk *= m;
    }
    return FNO_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fno_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? FNO_OK : FNO_ERR_CUDA; }

size_t elem_bytes(fno_dtype_t t) { return (t == FNO_F16 || t == FNO_BF16) ? 2 : 4; }

// Which kernel sequence a valid description runs on.
int choose_path(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout,
                uint32_t flags) {
    if (flags & FNO_PLAN_UNFUSED) return kPathUnfused;
    if (fused_supported(g, dtype, batch, cin, cout, flags)) return kPathFused;
    return kPathUnfused;
}

struct Sizes {
    size_t workspace, weight, adjoint_workspace;
    int path, kernels, bw_parts;
};

fno_status_t describe(int ndim, const int64_t *n, const int32_t *modes, int64_t batch,
                      int32_t cin, int32_t cout, fno_dtype_t dtype, uint32_t flags,
                      Geom *g, Sizes *sz, const int64_t *pad = nullptr) {
    fno_status_t st = make_geom(g, ndim, n, modes, pad);
    if (st != FNO_OK) return st;
    // a padded layer runs on the separate per-axis kernels (the fused kernels
    // are specialised to periodic power-of-two extents); it has no backward
    if (g->padded) {
        if (flags & FNO_PLAN_BACKWARD) return FNO_ERR_UNSUPPORTED;
        flags |= FNO_PLAN_UNFUSED;
    }
    if (batch < 1 || cin < 1 || cout < 1) return FNO_ERR_INVALID_ARG;
    if (dtype != FNO_F32 && dtype != FNO_F16 && dtype != FNO_BF16) return FNO_ERR_INVALID_ARG;
    if (flags & ~(FNO_PLAN_UNFUSED | FNO_PLAN_TRACE |
                  FNO_PLAN_PERSISTENT | FNO_PLAN_BACKWARD | FNO_PLAN_SIMT_MIX |
                  FNO_PLAN_SIMT_TRANSFORM | FNO_PLAN_PACKED_WEIGHTS | FNO_PLAN_TENSOR_EXTRA |
                  FNO_PLAN_SPLIT_LAYER))
        return FNO_ERR_INVALID_ARG;
    // packed weights: groups of four kept modes; the backward reads the standard layout
    if ((flags & FNO_PLAN_PACKED_WEIGHTS) &&
        (g->nkept % 4 != 0 || (flags & FNO_PLAN_BACKWARD)))
        return FNO_ERR_INVALID_ARG;
    // int64 element counts must not overflow and a tensor must stay addressable
    const double xe = (double)batch * cin * g->npix, ye = (double)batch * cout * g->npix;
    if (xe > 4.0e12 || ye > 4.0e12) return FNO_ERR_UNSUPPORTED;
    sz->path = choose_path(*g, dtype, batch, cin, cout, flags);
    if (sz->path == kPathUnfused) {
        sz->workspace = unfused_workspace_bytes(*g, batch, cin, cout);
        sz->kernels = unfused_kernel_count(*g);
    } else {
        sz->workspace = fused_workspace_bytes(*g, dtype, batch, cin, cout, flags);
        sz->kernels = fused_kernel_count(*g, dtype, batch, cin, cout, flags);
    }
    sz->weight = (size_t)g->nblk * cin * cout * g->mblk * 2 * elem_bytes(dtype);
    sz->adjoint_workspace = 0;
    sz->bw_parts = 0;
    if (flags & FNO_PLAN_BACKWARD) {
        // the adjoint layer (Cout -> Cin) runs dx; its plan never traces
        Geom ga;
        Sizes sa;
        st = describe(ndim, n, modes, batch, cout, cin, dtype,
                      flags & ~(FNO_PLAN_BACKWARD | FNO_PLAN_TRACE), &ga, &sa);
        if (st != FNO_OK) return st;
        sz->adjoint_workspace = sa.workspace;
        sz->bw_parts = sz->path == kPathFused ? fused_modes_parts(*g, dtype, flags) : 0;
        const BackwardLayout bl =
            backward_layout(*g, batch, cin, cout, sz->weight, sa.workspace, sz->bw_parts);
        if (bl.total > sz->workspace) sz->workspace = bl.total;
    }
    return FNO_OK;
}

}  // namespace

extern "C" {

const char *fno_status_string(fno_status_t s) {
    switch (s) {
        case FNO_OK: return "FNO_OK";
        case FNO_ERR_INVALID_ARG: return "FNO_ERR_INVALID_ARG: invalid argument";
        case FNO_ERR_UNSUPPORTED: return "FNO_ERR_UNSUPPORTED: shape not supported";
        case FNO_ERR_MISALIGNED: return "FNO_ERR_MISALIGNED: pointer not 16-byte aligned";
        case FNO_ERR_OUT_OF_MEMORY: return "FNO_ERR_OUT_OF_MEMORY: allocation failed";
        case FNO_ERR_CUDA: return "FNO_ERR_CUDA: CUDA call or launch failed";
        case FNO_ERR_DEVICE_TIMEOUT: return "FNO_ERR_DEVICE_TIMEOUT: device wait gave up";
        case FNO_ERR_DEVICE_BOUNDS: return "FNO_ERR_DEVICE_BOUNDS: device index check failed";
        case FNO_ERR_ALIASING: return "FNO_ERR_ALIASING: output overlaps an input";
    }
    return "FNO_ERR_UNKNOWN: not a status code";
}

int fno_version(void) { return kVersion; }

fno_status_t fno_spectral_conv_query_padded(int ndim, const int64_t *n, const int64_t *pad,
                                            const int32_t *modes, int64_t batch, int32_t cin,
                                            int32_t cout, fno_dtype_t dtype, uint32_t flags,
                                            size_t *workspace_bytes, size_t *weight_bytes) {
    Geom g;
    Sizes sz;
    fno_status_t st = describe(ndim, n, modes, batch, cin, cout, dtype, flags, &g, &sz, pad);
    if (st != FNO_OK) return st;
    if (workspace_bytes) *workspace_bytes = sz.workspace;
    if (weight_bytes) *weight_bytes = sz.weight;
    return FNO_OK;
}

fno_status_t fno_spectral_conv_query(int ndim, const int64_t *n, const int32_t *modes,
                                     int64_t batch, int32_t cin, int32_t cout,
                                     fno_dtype_t dtype, uint32_t flags,
                                     size_t *workspace_bytes, size_t *weight_bytes) {
    return fno_spectral_conv_query_padded(ndim, n, nullptr, modes, batch, cin, cout, dtype,
                                          flags, workspace_bytes, weight_bytes);
}

fno_status_t fno_spectral_conv_plan(fno_plan_t *out, int ndim, const int64_t *n,
                                    const int32_t *modes, int64_t batch, int32_t cin,
                                    int32_t cout, fno_dtype_t dtype, uint32_t flags) {
    return fno_spectral_conv_plan_padded(out, ndim, n, nullptr, modes, batch, cin, cout, dtype,
                                         flags);
}

fno_status_t fno_spectral_conv_plan_padded(fno_plan_t *out, int ndim, const int64_t *n,
                                           const int64_t *pad, const int32_t *modes,
                                           int64_t batch, int32_t cin, int32_t cout,
                                           fno_dtype_t dtype, uint32_t flags) {
    if (!out) return FNO_ERR_INVALID_ARG;
    *out = nullptr;
    Geom g;
    Sizes sz;
    fno_status_t st = describe(ndim, n, modes, batch, cin, cout, dtype, flags, &g, &sz, pad);
    if (st != FNO_OK) return st;
    if (inject("plan_alloc")) return FNO_ERR_OUT_OF_MEMORY;

    Plan *p = new (std::nothrow) Plan();
    if (!p) return FNO_ERR_OUT_OF_MEMORY;
    p->g = g;
    p->batch = batch;
    p->cin = cin;
    p->cout = cout;
    p->dtype = dtype;
    p->flags = flags;
    p->path = sz.path;
    p->kernels_per_forward = sz.kernels;
    p->workspace_bytes = sz.workspace;
    p->weight_bytes = sz.weight;

    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) !=
            cudaSuccess) {
        cudaGetLastError();
        delete p;
        return FNO_ERR_CUDA;
    }

    // Twiddle tables, one per axis: tw[a][j] = exp(-2 pi i j / N_a), computed
    // in double and rounded once to float; then the device error word.
    size_t off[FNO_MAX_NDIM + 1];
    size_t total = 0;
    for (int a = 0; a < g.d; ++a) {
        off[a] = total;
        total += ((size_t)g.n[a] * sizeof(float2) + 255) & ~size_t(255);
    }
    off[g.d] = total;
    total += 256 + ((fused_sync_bytes() + 255) & ~size_t(255));   // error word, counters
    std::vector<unsigned char> host(total, 0);
    for (int a = 0; a < g.d; ++a) {
        float2 *t = reinterpret_cast<float2 *>(host.data() + off[a]);
        for (int64_t j = 0; j < g.n[a]; ++j) {
            const double ang = -2.0 * M_PI * (double)j / (double)g.n[a];
            t[j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    }
    if (cudaMalloc(&p->dev_tables, total) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return FNO_ERR_OUT_OF_MEMORY;
    }
    p->dev_tables_bytes = total;
    unsigned char *base = static_cast<unsigned char *>(p->dev_tables);
    for (int a = 0; a < FNO_MAX_NDIM; ++a)
        p->tw[a] = a < g.d ? reinterpret_cast<float2 *>(base + off[a]) : nullptr;
    p->dev_err = reinterpret_cast<int *>(base + off[g.d]);
    p->sync = base + off[g.d] + 256;
    cudaError_t e = cudaMemcpy(p->dev_tables, host.data(), total, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && p->path != kPathUnfused) e = fused_plan_init(*p);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (p->path != kPathUnfused) fused_plan_release(*p);
        cudaFree(p->dev_tables);
        delete p;
        return FNO_ERR_CUDA;
    }
    if (flags & FNO_PLAN_BACKWARD) {
        st = fno_spectral_conv_plan(&p->adjoint, ndim, n, modes, batch, cout, cin, dtype,
                                    flags & ~(FNO_PLAN_BACKWARD | FNO_PLAN_TRACE));
        if (st != FNO_OK) {
            fno_plan_destroy(reinterpret_cast<fno_plan_t>(p));
            return st;
        }
        const BackwardLayout bl = backward_layout(g, batch, cin, cout, sz.weight,
                                                  sz.adjoint_workspace, sz.bw_parts);
        p->bw_parts = sz.bw_parts;
        p->bw_wt = bl.wt;
        p->bw_adj = bl.adj;
        p->bw_x = bl.x;
        p->bw_g = bl.g;
        p->bw_sa = bl.sa;
        p->bw_sb = bl.sb;
    }
    *out = reinterpret_cast<fno_plan_t>(p);
    return FNO_OK;
}

fno_status_t fno_spectral_conv_workspace_size(fno_plan_t plan, size_t *bytes) {
    if (!plan || !bytes) return FNO_ERR_INVALID_ARG;
    *bytes = reinterpret_cast<Plan *>(plan)->workspace_bytes;
    return FNO_OK;
}

fno_status_t fno_spectral_conv_kernel_count(fno_plan_t plan, int *count) {
    if (!plan || !count) return FNO_ERR_INVALID_ARG;
    *count = reinterpret_cast<Plan *>(plan)->kernels_per_forward;
    return FNO_OK;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

fno_status_t fno_spectral_conv_forward(fno_plan_t plan, const void *x, const void *w,
                                       void *y, void *workspace, fno_stream_t stream) {
    if (!plan || !x || !w || !y) return FNO_ERR_INVALID_ARG;
    const Plan &p = *reinterpret_cast<Plan *>(plan);
    if (p.workspace_bytes && !workspace) return FNO_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(workspace))
        return FNO_ERR_MISALIGNED;
    const size_t eb = elem_bytes(p.dtype);
    const size_t xb = (size_t)p.batch * p.cin * p.g.npix * eb;
    const size_t yb = (size_t)p.batch * p.cout * p.g.npix * eb;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, p.weight_bytes) ||
        overlaps(y, yb, workspace, p.workspace_bytes))
        return FNO_ERR_ALIASING;
    if (inject("launch")) return FNO_ERR_CUDA;
    Buffers b{x, w, y, workspace};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = p.path == kPathUnfused ? unfused_forward(p, b, s) : fused_forward(p, b, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FNO_ERR_CUDA;
    }
    return FNO_OK;
}

fno_status_t fno_spectral_conv_pack_weights(fno_plan_t plan, const void *w, void *w_packed,
                                            fno_stream_t stream) {
    if (!plan || !w || !w_packed) return FNO_ERR_INVALID_ARG;
    const Plan &p = *reinterpret_cast<Plan *>(plan);
    if (!(p.flags & FNO_PLAN_PACKED_WEIGHTS)) return FNO_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(w_packed)) return FNO_ERR_MISALIGNED;
    if (overlaps(w, p.weight_bytes, w_packed, p.weight_bytes)) return FNO_ERR_ALIASING;
    if (inject("launch")) return FNO_ERR_CUDA;
    if (launch_pack_weights(p, w, w_packed, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return FNO_ERR_CUDA;
    }
    return FNO_OK;
}

fno_status_t fno_spectral_conv_backward(fno_plan_t plan, const void *x, const void *w,
                                        const void *dy, void *dx, void *dw, void *workspace,
                                        fno_stream_t stream) {
    if (!plan || !dy || (!dx && !dw)) return FNO_ERR_INVALID_ARG;
    const Plan &p = *reinterpret_cast<Plan *>(plan);
    if (!(p.flags & FNO_PLAN_BACKWARD) || !p.adjoint) return FNO_ERR_INVALID_ARG;
    if ((dx && !w) || (dw && !x) || (p.workspace_bytes && !workspace))
        return FNO_ERR_INVALID_ARG;
    const void *ptrs[] = {x, w, dy, dx, dw, workspace};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return FNO_ERR_MISALIGNED;
    const size_t eb = elem_bytes(p.dtype);
    const size_t xb = (size_t)p.batch * p.cin * p.g.npix * eb;
    const size_t yb = (size_t)p.batch * p.cout * p.g.npix * eb;
    const size_t wb = p.weight_bytes, wsb = p.workspace_bytes;
    if (dx && (overlaps(dx, xb, x, xb) || overlaps(dx, xb, w, wb) || overlaps(dx, xb, dy, yb) ||
               overlaps(dx, xb, dw, wb) || overlaps(dx, xb, workspace, wsb)))
        return FNO_ERR_ALIASING;
    if (dw && (overlaps(dw, wb, x, xb) || overlaps(dw, wb, w, wb) || overlaps(dw, wb, dy, yb) ||
               overlaps(dw, wb, workspace, wsb)))
        return FNO_ERR_ALIASING;
    if (inject("launch")) return FNO_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    if (dx) {
        // dx = the layer applied to dy with W' = conj(W) transposed (Cout -> Cin)
        if (launch_adjoint_weights(p, w, ws + p.bw_wt, s) != cudaSuccess) {
            cudaGetLastError();
            return FNO_ERR_CUDA;
        }
        fno_status_t st = fno_spectral_conv_forward(p.adjoint, dy, ws + p.bw_wt, dx,
                                                    ws + p.bw_adj, stream);
        if (st != FNO_OK) return st;
    }
    if (dw) {
        float2 *X = reinterpret_cast<float2 *>(ws + p.bw_x);
        float2 *G = reinterpret_cast<float2 *>(ws + p.bw_g);
        float2 *sa = reinterpret_cast<float2 *>(ws + p.bw_sa);
        float2 *sb = reinterpret_cast<float2 *>(ws + p.bw_sb);
        cudaError_t e;
        if (p.bw_parts > 0) {
            e = fused_forward_modes(p, x, p.batch * p.cin, X, s);
            if (e == cudaSuccess) e = fused_forward_modes(p, dy, p.batch * p.cout, G, s);
        } else {
            e = unfused_forward_modes(p, x, p.batch * p.cin, sa, sb, X, s);
            if (e == cudaSuccess) e = unfused_forward_modes(p, dy, p.batch * p.cout, sa, sb, G, s);
        }
        if (e == cudaSuccess) e = launch_grad_w(p, X, G, p.bw_parts > 0 ? p.bw_parts : 1, dw, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return FNO_ERR_CUDA;
        }
    }
    return FNO_OK;
}

fno_status_t fno_plan_get_trace(fno_plan_t plan, fno_trace_record_t *records, size_t capacity,
                                size_t *count) {
    if (!plan || !count) return FNO_ERR_INVALID_ARG;
    const Plan &p = *reinterpret_cast<Plan *>(plan);
    if (!p.trace) return FNO_ERR_INVALID_ARG;
    *count = p.trace_records;
    const size_t n = capacity < p.trace_records ? capacity : p.trace_records;
    if (n && !records) return FNO_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        (n && cudaMemcpy(records, p.trace, n * sizeof(fno_trace_record_t),
                         cudaMemcpyDeviceToHost) != cudaSuccess)) {
        cudaGetLastError();
        return FNO_ERR_CUDA;
    }
    return FNO_OK;
}

fno_status_t fno_plan_get_device_error(fno_plan_t plan, fno_stream_t stream) {
    if (!plan) return FNO_ERR_INVALID_ARG;
    const Plan &p = *reinterpret_cast<Plan *>(plan);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(&v, p.dev_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p.dev_err, 0, sizeof(int));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return FNO_ERR_CUDA;
    }
    if (v == kDevTimeout) return FNO_ERR_DEVICE_TIMEOUT;
    if (v == kDevBounds) return FNO_ERR_DEVICE_BOUNDS;
    return FNO_OK;
}

fno_status_t fno_plan_check_bounded_wait(fno_plan_t plan, int which, fno_stream_t stream) {
    if (!plan || (which != 0 && which != 1)) return FNO_ERR_INVALID_ARG;
    const Plan &p = *reinterpret_cast<Plan *>(plan);
    return from_cuda(launch_wait_check(p, which, reinterpret_cast<cudaStream_t>(stream)));
}

fno_status_t fno_plan_destroy(fno_plan_t plan) {
    if (!plan) return FNO_OK;
    Plan *p = reinterpret_cast<Plan *>(plan);
    cudaError_t e = cudaSuccess;
    fno_status_t st = fno_plan_destroy(p->adjoint);
    if (p->path != kPathUnfused) fused_plan_release(*p);
    if (p->dev_tables) e = cudaFree(p->dev_tables);
    delete p;
    return st != FNO_OK ? st : from_cuda(e);
}

}  // extern "C"
