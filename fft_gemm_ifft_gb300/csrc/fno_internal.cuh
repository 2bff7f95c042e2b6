// fno_internal.cuh -- shared definitions of the CUDA library (not installed).
//
// Geometry of the layer (TurboFNO article, gsyq.cn/news/457482, §2.1-§2.3):
// x (B, Cin, N_0..N_{d-1}) real -> kept modes X (B, Cin, K_0..K_{d-1}) complex,
// K_a = 2 m_a on full axes (low rows then high rows), K_{d-1} = m_{d-1};
// Y[b,o,k] = sum_i X[b,i,k] W[blk(k), i, o, local(k)]; y = inverse(Y).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fno.h"

namespace fno {

// Device error word codes (plan-owned int, first error wins).
enum : int { kDevOk = 0, kDevTimeout = 1, kDevBounds = 2 };

// n[a] is the transform length of axis a and ext[a] the extent of x and y
// along it.  They differ only for a zero-padded layer (a non-periodic domain,
// TurboFNO §2.3 / §3.3): x is read as if extended with n - ext zeros per axis
// and y keeps the first ext samples of the inverse; everywhere else ext == n.
struct Geom {
    int d;
    int64_t n[FNO_MAX_NDIM];
    int32_t m[FNO_MAX_NDIM];
    int64_t kdim[FNO_MAX_NDIM];   // kept extent per axis
    int64_t ext[FNO_MAX_NDIM];    // extent of x and y per axis (<= n)
    int64_t nkept;                // |K|
    int64_t npix;                 // prod ext: elements of one x or y image
    int64_t ntr;                  // prod n: points of the transform (scale 1/ntr)
    int64_t nblk;                 // weight blocks 2^(d-1)
    int64_t mblk;                 // modes per block prod m
    bool padded;                  // ext != n on some axis
};

// Host-side plan state.
struct Plan {
    Geom g;
    int64_t batch;
    int32_t cin, cout;
    fno_dtype_t dtype;
    uint32_t flags;
    int device;
    int path;                     // which kernel sequence runs (kPath*)
    int kernels_per_forward;
    size_t workspace_bytes;
    size_t weight_bytes;
    // plan-owned device memory
    float2 *tw[FNO_MAX_NDIM];     // tw[a][j] = exp(-2 pi i j / N_a), j < N_a
    int *dev_err;                 // device error word
    void *sync;                   // fused-path queue counters (256 bytes, zero between launches)
    void *dev_tables;             // single allocation holding the above
    size_t dev_tables_bytes;
    int num_sms;
    // fused path launch shape (set by fused_plan_init)
    int fused_grid;
    size_t fused_smem;
    int fused_ob;
    int fused_bb;
    int fused_bstream;            // > 0: kernel B streams the weights, this many modes a CTA
    void *fused_tables;           // tensor-core path: twiddle operands (plan-owned)
    bool fused_mixtc;             // three-kernel path mixes on the tensor cores
    bool fused_mixtf32;           // fp32 three-kernel path mixes on the tensor cores (3xTF32)
    bool fused_tca;               // three-kernel path transforms (kernel A) on the tensor cores
    bool fused_tcc;               // ... and inverts (kernel C) on the tensor cores
    bool fused_c1pass;            // fp32 kernel C: one-pass column inverse, 3 CTAs per SM
    bool mix_image;               // packed weights are the tensor-core mixing's operand images
    size_t fused_table_c;         // byte offset of kernel C's operand in fused_tables
    fno_trace_record_t *trace;    // FNO_PLAN_TRACE: one record per work item (plan-owned)
    size_t trace_records;         // records one forward call produces
    // FNO_PLAN_BACKWARD: the adjoint layer's plan and the backward workspace map
    fno_plan_t adjoint;
    size_t bw_wt, bw_adj, bw_x, bw_g, bw_sa, bw_sb;   // byte offsets in the workspace
    int bw_parts;                 // partial copies of the kept modes (0: per-axis kernels)
};

// Backward workspace map of a description (offsets and total size).
struct BackwardLayout {
    size_t wt, adj, x, g, sa, sb, total;
};
// parts = partial copies the forward-transform kernel writes, 0 when the
// per-axis kernels (and their scratch) compute the kept modes
BackwardLayout backward_layout(const Geom &g, int64_t batch, int cin, int cout,
                               size_t weight_bytes, size_t adjoint_workspace, int parts);

enum { kPathUnfused = 0, kPathFused = 1 };

// --------------------------------------------------------------------------
// Small device helpers
// --------------------------------------------------------------------------
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
// a * conj(b)
__device__ __forceinline__ float2 cmulc(float2 a, float2 b) {
    return make_float2(a.x * b.x + a.y * b.y, a.y * b.x - a.x * b.y);
}
__device__ __forceinline__ void cfma(float2 &acc, float2 a, float2 b) {
    acc.x = fmaf(a.x, b.x, acc.x);
    acc.x = fmaf(-a.y, b.y, acc.x);
    acc.y = fmaf(a.x, b.y, acc.y);
    acc.y = fmaf(a.y, b.x, acc.y);
}

template <typename T> struct Storage;
template <> struct Storage<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float v) { *p = v; }
    static __device__ __forceinline__ float2 load2(const float *p) {
        return *reinterpret_cast<const float2 *>(p);
    }
    // four consecutive elements (16-byte aligned for float, 8-byte otherwise)
    static __device__ __forceinline__ float4 load4(const float *p) {
        return *reinterpret_cast<const float4 *>(p);
    }
    static __device__ __forceinline__ void store4(float *p, float4 v) {
        *reinterpret_cast<float4 *>(p) = v;
    }
    // read or written once: streaming cache hints
    static __device__ __forceinline__ float load_stream(const float *p) { return __ldcs(p); }
    static __device__ __forceinline__ void store_stream(float *p, float v) { __stcs(p, v); }
};
template <> struct Storage<__half> {
    static __device__ __forceinline__ float load(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void store(__half *p, float v) { *p = __float2half_rn(v); }
    static __device__ __forceinline__ float2 load2(const __half *p) {
        return __half22float2(*reinterpret_cast<const __half2 *>(p));
    }
    static __device__ __forceinline__ float4 load4(const __half *p) {
        const float2 a = load2(p), b = load2(p + 2);
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void store4(__half *p, float4 v) {
        reinterpret_cast<__half2 *>(p)[0] = __floats2half2_rn(v.x, v.y);
        reinterpret_cast<__half2 *>(p)[1] = __floats2half2_rn(v.z, v.w);
    }
    static __device__ __forceinline__ float load_stream(const __half *p) {
        return __half2float(__ldcs(p));
    }
    static __device__ __forceinline__ void store_stream(__half *p, float v) {
        __stcs(p, __float2half_rn(v));
    }
};

template <> struct Storage<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float v) {
        *p = __float2bfloat16_rn(v);
    }
    static __device__ __forceinline__ float2 load2(const __nv_bfloat16 *p) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    }
    static __device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
        const float2 a = load2(p), b = load2(p + 2);
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
        reinterpret_cast<__nv_bfloat162 *>(p)[0] = __floats2bfloat162_rn(v.x, v.y);
        reinterpret_cast<__nv_bfloat162 *>(p)[1] = __floats2bfloat162_rn(v.z, v.w);
    }
    static __device__ __forceinline__ float load_stream(const __nv_bfloat16 *p) {
        return __bfloat162float(__ldcs(p));
    }
    static __device__ __forceinline__ void store_stream(__nv_bfloat16 *p, float v) {
        __stcs(p, __float2bfloat16_rn(v));
    }
};

// Calls f with a value of the storage type of `dt` (float, __half or
// __nv_bfloat16), so that a generic lambda can pick the kernel instance.
template <class F>
decltype(auto) with_storage(fno_dtype_t dt, F &&f) {
    if (dt == FNO_F16) return f(__half());
    if (dt == FNO_BF16) return f(__nv_bfloat16());
    return f(0.0f);
}

// Complex-element index of weight (kept mode kk, input i, output o) in the
// packed mode-major layout: groups of four kept modes, [group][i][o][4].
__host__ __device__ __forceinline__ size_t packed_index(int64_t kk, int i, int o, int cin,
                                                         int cout) {
    return ((((size_t)(kk >> 2) * cin + i) * cout + o) << 2) + (size_t)(kk & 3);
}

// Sets the device error word once (first error wins).
__device__ __forceinline__ void raise_dev_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Index checks of the debug build (compiled with FNO_DEBUG_BOUNDS, the library
// libfno_bounds.so): a global-memory index outside [0, size) records kDevBounds
// in the error word and the access is skipped, so a wrong index shows up as
// FNO_ERR_DEVICE_BOUNDS from fno_plan_get_device_error instead of a fault.  In
// the normal build every check is the constant true and compiles away.
#ifdef FNO_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(int64_t idx, int64_t size, int *err) {
    if (idx >= 0 && idx < size) return true;
    raise_dev_error(err, kDevBounds);
    return false;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(int64_t, int64_t, int *) { return true; }
#endif

// --------------------------------------------------------------------------
// Host-side entry points of the kernel translation units
// --------------------------------------------------------------------------
struct Buffers {
    const void *x;
    const void *w;
    void *y;
    void *ws;
};

// Unfused per-axis path (fno_unfused.cu).
size_t unfused_workspace_bytes(const Geom &g, int64_t batch, int cin, int cout);
int unfused_kernel_count(const Geom &g);
cudaError_t unfused_forward(const Plan &p, const Buffers &b, cudaStream_t s);
// Single steps of the unfused path, for composite sequences: a DFT along one
// full axis over the kept rows (forward) or back to every row (inverse), with
// the (outer, N, inner) view of the tensor; and the per-mode mixing.
cudaError_t launch_axis_forward(const float2 *in, float2 *out, int64_t outer, int n, int64_t inner,
                                int m, const float2 *tw, int num_sms, cudaStream_t s);
cudaError_t launch_axis_inverse(const float2 *in, float2 *out, int64_t outer, int n, int64_t inner,
                                int m, const float2 *tw, int num_sms, cudaStream_t s);
cudaError_t launch_mix(const Plan &p, const float2 *X, const void *w, float2 *Y, cudaStream_t s);
// Standard (nblk, Cin, Cout, m...) weights -> the packed layout.
cudaError_t launch_pack_weights(const Plan &p, const void *w, void *wp, cudaStream_t s);
// A kernel's dynamic shared-memory limit is an attribute of the process (per
// device), not of a plan: plans only ever raise it, so that a plan made later
// with a smaller need cannot break the launches of an earlier, larger one.
cudaError_t raise_smem_limit_fn(const void *fn, size_t bytes);
template <typename F>
cudaError_t raise_smem_limit(F fn, size_t bytes) {
    return raise_smem_limit_fn((const void *)fn, bytes);
}

// one CTA runs a bounded wait that nothing satisfies (which 0: flag, 1: mbarrier)
cudaError_t launch_wait_check(const Plan &p, int which, cudaStream_t s);
// Truncated forward DFT of nch real images x (storage dtype of p) to their
// kept modes out[nch][|K|], through the per-axis kernels; sa, sb hold
// unfused_modes_scratch_elems(g, nch) complex values each.
int64_t unfused_modes_scratch_elems(const Geom &g, int64_t nch);
cudaError_t unfused_forward_modes(const Plan &p, const void *x, int64_t nch, float2 *sa,
                                  float2 *sb, float2 *out, cudaStream_t s);
// Backward kernels (fno_backward.cu).
cudaError_t launch_adjoint_weights(const Plan &p, const void *w, void *wt, cudaStream_t s);
cudaError_t launch_grad_w(const Plan &p, const float2 *X, const float2 *G, int parts, void *dw,
                          cudaStream_t s);

}  // namespace fno
