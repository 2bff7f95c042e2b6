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
#include "fno_gelu.cuh"
#include "fno_tc.cuh"

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
    // tensor-core linears (0 grid: the register-tiled SIMT kernels run instead)
    int layer_tc_grid, head_tc_grid;
    size_t layer_tc_smem, head_tc_smem;
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

// ---------------------------------------------------------------------------
// Tensor-core 1x1 linears (tcgen05, 3xTF32).  A 1x1 linear over a channels-
// first activation is the dense GEMM D[p][o] = sum_i act[i][p] W[o][i] with
// M = 128 pixels per tile, N = the output channels, K = the input channels.
// Both operands are staged K-major with the 128-byte swizzle: the weights once
// per CTA (hi = the value read at tf32 precision, lo = the exact remainder),
// the activation tile transposed on its way into shared memory (each thread
// owns one pixel row and writes 16-byte pieces, conflict-free under the
// swizzle).  Three chains (hi*hi + hi*lo + lo*hi) accumulate in tensor
// memory; the epilogue reads one pixel's N sums per thread (32x32b loads, a
// warp per 32 lanes) and applies bias, the spectral sum and GELU (layer,
// k_linear_tc) or GELU and the second projection (head, k_head_tc, which
// double-buffers the tile and the accumulator).  A CTA walks tiles grid-stride.
// ---------------------------------------------------------------------------
// one activation element as float: streaming load for float32 storage
__device__ __forceinline__ float load_act(const float *p) { return __ldcs(p); }
__device__ __forceinline__ float load_act(const __half *p) { return Storage<__half>::load(p); }
__device__ __forceinline__ float load_act(const __nv_bfloat16 *p) {
    return Storage<__nv_bfloat16>::load(p);
}

namespace lintc {

constexpr int kThreads = 512;            // four threads per pixel row of a tile
constexpr int kParts4 = kThreads / 128;  // threads sharing a pixel (column quarters)
constexpr int kRows = 128;               // M
constexpr uint32_t kChunk = 16384;       // 128 rows x 128 bytes (32 fp32 of K)

struct Smem {                            // offsets from a 1024-aligned base
    uint32_t ahi, alo, whi, wlo, total;
};
__host__ __device__ inline Smem smem_map(int k, int n) {
    const uint32_t kc = (uint32_t)(k / 32);
    const uint32_t wchunk = (uint32_t)n * 128;   // n rows x 128 bytes
    Smem s;
    s.ahi = 0;
    s.alo = kc * kChunk;
    s.whi = 2 * kc * kChunk;
    s.wlo = s.whi + kc * ((wchunk + 1023) / 1024 * 1024);
    s.total = s.wlo + kc * ((wchunk + 1023) / 1024 * 1024) + 1024;   // + alignment slack
    return s;
}

// out[b][o][p] = act(sum_i W[o][i] a[b][i][p] + bias[o] + add[b][o][p])
// KC = input channels / 32, NG = output channels / 16 (fully unrolled, so that
// every load of a tile is in flight before its first use)
template <int KC, int NG, typename T>
__global__ void __launch_bounds__(kThreads, 2)
k_linear_tc(const T *__restrict__ a, const float *__restrict__ W,
            const float *__restrict__ bias, const T *__restrict__ add,
            const float *__restrict__ P2, const float *__restrict__ c2, T *__restrict__ out,
            int cout2, int64_t npix, int64_t ntiles, int apply_gelu, int *err) {
    using namespace tcu;
    (void)P2;
    (void)c2;
    (void)cout2;
    constexpr int cin = 32 * KC, n = 16 * NG;
    static_assert(NG % kParts4 == 0 || NG < kParts4, "column groups split over the threads of a pixel");
    constexpr int kCinT = cin / kParts4;                 // input channels loaded per thread
    constexpr int kGroupsT = NG >= kParts4 ? NG / kParts4 : 1;   // column groups per thread
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    const Smem sm = smem_map(cin, n);
    const int tid = threadIdx.x, warp = tid >> 5;
    // thread -> (pixel row, quarter): warps w, w+4, w+8, w+12 share tensor-memory lanes
    const int row = 32 * (warp & 3) + (tid & 31), quarter = warp >> 2;
    constexpr uint32_t wchunk = ((uint32_t)n * 128 + 1023) / 1024 * 1024;
    // weights, hi and lo, as the B operand (N rows = outputs, K = inputs)
    for (int e = tid; e < n * cin; e += kThreads) {
        const int o = e / cin, i = e % cin;
        const float w = W[(int64_t)o * cin + i];
        const uint32_t off = (uint32_t)(i / 32) * wchunk + sw_off(o, i % 32);
        *reinterpret_cast<float *>(base + sm.whi + off) = w;
        *reinterpret_cast<float *>(base + sm.wlo + off) = tf32_lo(w);
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    constexpr uint32_t ncols = n <= 32 ? 32 : (n <= 64 ? 64 : 128);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(ncols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    constexpr uint32_t idesc = idesc_tf32(n);
    const int64_t ptiles = (npix + kRows - 1) / kRows;
    const int i0 = quarter * kCinT;
    // activation tile, transposed: row = pixel, K = input channel; this thread's
    // quarter of the channels.  The next tile's loads are issued before the
    // current tile's MMAs are waited for, so they land under its epilogue.
    float av[kCinT];
    auto load_tile = [&](int64_t t) {
        const int64_t tb = t / ptiles, tp = (t % ptiles) * kRows + row;
        const bool tin = t < ntiles && tp < npix;
        const T *ab = a + (tb * cin + i0) * npix + tp;
#pragma unroll
        for (int i = 0; i < kCinT; ++i) av[i] = tin ? load_act(ab + (int64_t)i * npix) : 0.f;
    };
    load_tile(blockIdx.x);
    // this thread's output columns: groups quarter, quarter + 4, ...; the
    // biases are read once into shared memory (broadcast reads per tile)
    const bool has_cols = quarter < NG;
    __shared__ float s_bias[16 * 8];
    for (int o = tid; o < n; o += kThreads) s_bias[o] = bias[o];
    __syncthreads();
    uint32_t phase = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t b = tile / ptiles, p0 = (tile % ptiles) * kRows;
        const int64_t p = p0 + row;
        const bool pin = p < npix;
        // pixel p of image b in channel 0; channel o is o * npix further
        const int64_t pix0 = b * n * npix + p;
#pragma unroll
        for (int i4 = 0; i4 < kCinT / 4; ++i4) {
            const int i = i0 + 4 * i4;
            const float4 v = make_float4(av[4 * i4], av[4 * i4 + 1], av[4 * i4 + 2], av[4 * i4 + 3]);
            const uint32_t off = (uint32_t)(i / 32) * kChunk + sw_off(row, i % 32);
            *reinterpret_cast<float4 *>(base + sm.ahi + off) = v;
            *reinterpret_cast<float4 *>(base + sm.alo + off) =
                make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc_after_sync();
            const uint32_t ah = tc_smem_addr(base + sm.ahi), al = tc_smem_addr(base + sm.alo);
            const uint32_t wh = tc_smem_addr(base + sm.whi), wl = tc_smem_addr(base + sm.wlo);
#pragma unroll
            for (int c = 0; c < KC; ++c) {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint32_t ao = c * kChunk + s * 32, bo = c * wchunk + s * 32;
                    mma_tf32(tmem, desc_sw128(ah + ao), desc_sw128(wh + bo), idesc,
                             (c | s) ? 1u : 0u);
                    mma_tf32(tmem, desc_sw128(ah + ao), desc_sw128(wl + bo), idesc, 1u);
                    mma_tf32(tmem, desc_sw128(al + ao), desc_sw128(wh + bo), idesc, 1u);
                }
            }
            mma_commit(&bar);
        }
        load_tile(tile + gridDim.x);    // av is in shared memory: prefetch the next tile
        // the spectral sums of these outputs are fetched while the MMAs run
        float sv[16 * kGroupsT];
#pragma unroll
        for (int gg = 0; gg < kGroupsT; ++gg) {
            const T *ap = add + pix0 + (int64_t)(16 * (quarter + kParts4 * gg)) * npix;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                sv[16 * gg + q] = (add && pin && has_cols) ? load_act(ap) : 0.f;
                ap += npix;
            }
        }
        const bool ok = mbar_wait(&bar, phase++, err);
        tc_after_sync();
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll
        for (int gg = 0; gg < kGroupsT; ++gg) {
            const int g = quarter + kParts4 * gg;
            if (g < NG) {
                float v[16];
                tmem_ld16(lane_addr + 16 * g, v);
                T *op = out + pix0 + (int64_t)(16 * g) * npix;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float r = (ok ? v[q] : 0.f) + s_bias[16 * g + q] + sv[16 * gg + q];
                    if (apply_gelu) r = gelu(r);
                    if (pin) Storage<T>::store(op, r);
                    op += npix;
                }
            }
        }
        tc_before_sync();
        __syncthreads();            // tensor memory and the A tile are reused by the next tile
    }
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(ncols));
    }
}

// Whether a linear with these channel counts runs on the tensor cores.
inline bool eligible(int cin, int n) {
    return (cin == 32 || cin == 64) && (n == 32 || n == 48 || n == 64 || n == 128);
}

template <typename T>
using TcFn = void (*)(const T *, const float *, const float *, const T *, const float *,
                      const float *, T *, int, int64_t, int64_t, int, int *);

template <int KC, typename T>
TcFn<T> pick_n(int n) {
    switch (n) {
        case 32: return k_linear_tc<KC, 2, T>;
        case 48: return k_linear_tc<KC, 3, T>;
        case 64: return k_linear_tc<KC, 4, T>;
        default: return k_linear_tc<KC, 8, T>;
    }
}
template <typename T>
TcFn<T> kernel(int cin, int n) { return cin == 32 ? pick_n<1, T>(n) : pick_n<2, T>(n); }

// The projection head, pipelined over its tiles: two activation-tile buffers
// and two tensor-memory accumulators, so that while the threads run tile k's
// epilogue (a GELU per hidden unit and the second projection) the tensor
// cores already multiply tile k + 1, whose loads and tf32 split ran before
// tile k's product was waited for.  One CTA per SM (the double buffer needs
// most of the shared memory).
__host__ __device__ inline uint32_t head_smem(int k, int n) {
    const uint32_t kc = (uint32_t)(k / 32);
    const uint32_t wchunk = ((uint32_t)n * 128 + 1023) / 1024 * 1024;
    return 2 * (2 * kc * kChunk) + 2 * kc * wchunk + 1024;
}
template <int KC, int NG, typename T>
__global__ void __launch_bounds__(kThreads, 1)
k_head_tc(const T *__restrict__ a, const float *__restrict__ W,
          const float *__restrict__ bias, const T *__restrict__ add,
          const float *__restrict__ P2, const float *__restrict__ c2, T *__restrict__ out,
          int cout2, int64_t npix, int64_t ntiles, int apply_gelu, int *err) {
    using namespace tcu;
    (void)add;
    (void)apply_gelu;
    constexpr int cin = 32 * KC, n = 16 * NG;
    static_assert(NG % kParts4 == 0 || NG < kParts4, "column groups split over the threads of a pixel");
    constexpr int kCinT = cin / kParts4;
    constexpr int kGroupsT = NG >= kParts4 ? NG / kParts4 : 1;
    constexpr uint32_t kBuf = 2 * KC * kChunk;                  // one tile: hi then lo
    constexpr uint32_t wchunk = ((uint32_t)n * 128 + 1023) / 1024 * 1024;
    constexpr uint32_t kW = 2 * kBuf, kWlo = kW + KC * wchunk;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ uint32_t s_tmem;
    __shared__ float s_head[kParts4 * kMaxCout * 128];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = 32 * (warp & 3) + (tid & 31), quarter = warp >> 2;
    for (int e = tid; e < n * cin; e += kThreads) {
        const int o = e / cin, i = e % cin;
        const float w = W[(int64_t)o * cin + i];
        const uint32_t off = (uint32_t)(i / 32) * wchunk + sw_off(o, i % 32);
        *reinterpret_cast<float *>(base + kW + off) = w;
        *reinterpret_cast<float *>(base + kWlo + off) = tf32_lo(w);
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar[0])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar[1])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    constexpr uint32_t ncols = 2 * n <= 64 ? 64 : (2 * n <= 128 ? 128 : 256);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(ncols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    constexpr uint32_t idesc = idesc_tf32(n);
    const int64_t ptiles = (npix + kRows - 1) / kRows;
    const int i0 = quarter * kCinT;
    // tile t's activations, transposed into buffer `buf` as the K-major A operand
    auto load_split = [&](int64_t t, int buf) {
        const int64_t tb = t / ptiles, tp = (t % ptiles) * kRows + row;
        const bool tin = tp < npix;
        const T *ab = a + (tb * cin + i0) * npix + tp;
        float av[kCinT];
#pragma unroll
        for (int i = 0; i < kCinT; ++i) av[i] = tin ? load_act(ab + (int64_t)i * npix) : 0.f;
        char *hi = base + buf * kBuf, *lo = hi + KC * kChunk;
#pragma unroll
        for (int i4 = 0; i4 < kCinT / 4; ++i4) {
            const int i = i0 + 4 * i4;
            const float4 v = make_float4(av[4 * i4], av[4 * i4 + 1], av[4 * i4 + 2], av[4 * i4 + 3]);
            const uint32_t off = (uint32_t)(i / 32) * kChunk + sw_off(row, i % 32);
            *reinterpret_cast<float4 *>(hi + off) = v;
            *reinterpret_cast<float4 *>(lo + off) =
                make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();
    };
    // one thread: the 3xTF32 chains of buffer `buf` into accumulator `buf`
    auto issue = [&](int buf) {
        tc_after_sync();
        const uint32_t ah = tc_smem_addr(base + buf * kBuf), al = ah + KC * kChunk;
        const uint32_t wh = tc_smem_addr(base + kW), wl = tc_smem_addr(base + kWlo);
        const uint32_t d = tmem + buf * n;
#pragma unroll
        for (int c = 0; c < KC; ++c) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t ao = c * kChunk + s * 32, bo = c * wchunk + s * 32;
                mma_tf32(d, desc_sw128(ah + ao), desc_sw128(wh + bo), idesc, (c | s) ? 1u : 0u);
                mma_tf32(d, desc_sw128(ah + ao), desc_sw128(wl + bo), idesc, 1u);
                mma_tf32(d, desc_sw128(al + ao), desc_sw128(wh + bo), idesc, 1u);
            }
        }
        mma_commit(&bar[buf]);
    };
    // the first layer's biases and the second layer's weights, read once
    __shared__ float s_b1[16 * 8], s_p2[kMaxCout * 16 * 8];
    for (int o = tid; o < n; o += kThreads) s_b1[o] = bias[o];
    for (int e = tid; e < cout2 * n; e += kThreads) s_p2[e] = P2[e];
    __syncthreads();
    int64_t tile = blockIdx.x;
    if (tile < ntiles) {
        load_split(tile, 0);
        if (tid == 0) issue(0);
    }
    for (int k = 0; tile < ntiles; tile += gridDim.x, ++k) {
        const int buf = k & 1;
        const int64_t nxt = tile + gridDim.x;
        if (nxt < ntiles) {
            // buffer and accumulator buf ^ 1 were released at the end of tile k - 1
            load_split(nxt, buf ^ 1);
            if (tid == 0) issue(buf ^ 1);
        }
        const bool ok = mbar_wait(&bar[buf], (uint32_t)(k >> 1) & 1u, err);
        tc_after_sync();
        const int64_t b = tile / ptiles, p = (tile % ptiles) * kRows + row;
        const bool pin = p < npix;
        const uint32_t lane_addr = tmem + buf * n + ((uint32_t)(32 * (warp & 3)) << 16);
        float hacc[kMaxCout];
#pragma unroll
        for (int q = 0; q < kMaxCout; ++q) hacc[q] = 0.f;
#pragma unroll
        for (int gg = 0; gg < kGroupsT; ++gg) {
            const int g = quarter + kParts4 * gg;
            if (g < NG) {
                float v[16];
                tmem_ld16(lane_addr + 16 * g, v);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int o = 16 * g + q;
                    const float h = gelu((ok ? v[q] : 0.f) + s_b1[o]);
#pragma unroll
                    for (int c = 0; c < kMaxCout; ++c)
                        if (c < cout2) hacc[c] = fmaf(s_p2[c * n + o], h, hacc[c]);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < kMaxCout; ++c)
            if (c < cout2) s_head[(quarter * kMaxCout + c) * 128 + row] = hacc[c];
        __syncthreads();
        if (quarter == 0 && pin) {
            for (int c = 0; c < cout2; ++c) {
                float v = c2[c];
#pragma unroll
                for (int qq = 0; qq < kParts4; ++qq) v += s_head[(qq * kMaxCout + c) * 128 + row];
                Storage<T>::store(out + (b * cout2 + c) * npix + p, v);
            }
        }
        tc_before_sync();
        __syncthreads();            // accumulator buf and s_head are reused
    }
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(ncols));
    }
}

template <typename T>
TcFn<T> head_kernel(int cin, int n) {
    auto pick = [](auto kc, int nn) -> TcFn<T> {
        constexpr int KC = decltype(kc)::value;
        switch (nn) {
            case 32: return k_head_tc<KC, 2, T>;
            case 48: return k_head_tc<KC, 3, T>;
            case 64: return k_head_tc<KC, 4, T>;
            default: return k_head_tc<KC, 8, T>;
        }
    };
    return cin == 32 ? pick(std::integral_constant<int, 1>{}, n)
                     : pick(std::integral_constant<int, 2>{}, n);
}

}  // namespace lintc

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
    // tensor-core linears where the channel counts fit one K x N tile
    m->layer_tc_grid = m->head_tc_grid = 0;
    const int64_t ntiles = d->batch * ((d->h * d->w + lintc::kRows - 1) / lintc::kRows);
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    auto setup_tc = [&](const void *fn, int cin, int n, size_t sb, int *grid,
                        size_t *smem_bytes) {
        if (!lintc::eligible(cin, n)) return true;
        int per_sm = 0;
        if (raise_smem_limit(fn, (int)sb) !=
                cudaSuccess ||
            cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, lintc::kThreads, sb) !=
                cudaSuccess)
            return false;
        if (per_sm < 1) return true;
        // the occupancy query can under-count here; two CTAs fit when their
        // shared memory (dynamic, static, reserved) and registers do
        cudaFuncAttributes fa;
        int smem_sm = 0, reserved = 0;
        if (cudaFuncGetAttributes(&fa, fn) == cudaSuccess &&
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ==
                cudaSuccess &&
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) ==
                cudaSuccess &&
            2 * (sb + fa.sharedSizeBytes + (size_t)reserved) <= (size_t)smem_sm &&
            2 * fa.numRegs * lintc::kThreads <= 65536)
            per_sm = std::max(per_sm, 2);
        cudaGetLastError();
        const int64_t g = std::min<int64_t>(ntiles, (int64_t)sms * per_sm);
        *grid = (int)g;
        *smem_bytes = sb;
        return true;
    };
    // (16-bit activations convert on load and round once on store)
    const bool f32 = d->dtype == FNO_F32;
    const bool tc_ok = lintc::eligible(d->width, d->width),
               th_ok = lintc::eligible(d->width, d->hidden);
    const bool tc_fail = with_storage(d->dtype, [&](auto t) {
        using T = decltype(t);
        return (tc_ok && !setup_tc((const void *)lintc::kernel<T>(d->width, d->width), d->width,
                                   d->width, lintc::smem_map(d->width, d->width).total,
                                   &m->layer_tc_grid, &m->layer_tc_smem)) ||
               (th_ok && !setup_tc((const void *)lintc::head_kernel<T>(d->width, d->hidden),
                                   d->width, d->hidden, lintc::head_smem(d->width, d->hidden),
                                   &m->head_tc_grid, &m->head_tc_smem));
    });
    if (tc_fail) {
        cudaGetLastError();
        fno_plan_destroy(m->spec);
        delete m;
        return FNO_ERR_CUDA;
    }
    int spec_kernels = 0;
    fno_spectral_conv_kernel_count(m->spec, &spec_kernels);
    m->npix = d->h * d->w;
    m->act_bytes = align256((size_t)d->batch * d->width * m->npix * (f32 ? 4 : 2));
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
        const int64_t ntiles = d.batch * ((m.npix + lintc::kRows - 1) / lintc::kRows);
        int *err = reinterpret_cast<Plan *>(m.spec)->dev_err;
        const dim3 lin_grid(ptiles, (unsigned)((d.width + kTO - 1) / kTO), (unsigned)d.batch);
        const size_t smem = sizeof(TileSmem);
        k_linear_tiled<T><<<lin_grid, kTT, smem, s>>>(static_cast<const T *>(x), p->lift_w,
                                                      p->lift_b, nullptr, A, d.cin_lift, d.width,
                                                      m.npix, 0);
        if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
        for (int l = 0; l < d.nlayers; ++l) {
            fno_status_t st = fno_spectral_conv_forward(m.spec, A, spec_w + l * spec_stride, S,
                                                        m.spec_ws_bytes ? spec_ws : nullptr,
                                                        stream);
            if (st != FNO_OK) return st;
            const int last = (l == d.nlayers - 1);
            if (m.layer_tc_grid)
                lintc::kernel<T>(d.width, d.width)<<<m.layer_tc_grid, lintc::kThreads,
                                                     m.layer_tc_smem, s>>>(
                    A, p->pw_w + (size_t)l * d.width * d.width, p->pw_b + (size_t)l * d.width,
                    S, nullptr, nullptr, Tn, 0, m.npix, ntiles, last ? 0 : 1, err);
            else
                k_linear_tiled<T><<<lin_grid, kTT, smem, s>>>(
                    A, p->pw_w + (size_t)l * d.width * d.width, p->pw_b + (size_t)l * d.width,
                    S, Tn, d.width, d.width, m.npix, last ? 0 : 1);
            if (cudaGetLastError() != cudaSuccess) return FNO_ERR_CUDA;
            T *tmp = A;
            A = Tn;
            Tn = tmp;
        }
        if (m.head_tc_grid)
            lintc::head_kernel<T>(d.width, d.hidden)<<<m.head_tc_grid, lintc::kThreads,
                                                      m.head_tc_smem, s>>>(
                A, p->proj1_w, p->proj1_b, nullptr, p->proj2_w, p->proj2_b,
                static_cast<T *>(out), d.cout, m.npix, ntiles, 1, err);
        else
            projection_kernel<T>(d.cout)<<<dim3(ptiles, (unsigned)d.batch), kTT, smem, s>>>(
                A, p->proj1_w, p->proj1_b, p->proj2_w, p->proj2_b, static_cast<T *>(out),
                d.width, d.hidden, d.cout, m.npix);
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
    delete m;
    return st;
}

}  // extern "C"
