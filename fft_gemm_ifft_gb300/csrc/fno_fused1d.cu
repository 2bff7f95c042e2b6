// fno_fused1d.cu -- the 1-D spectral-convolution layer as one kernel.
//
// The steps of the TurboFNO article (gsyq.cn/news/457482) §2.1-§2.3 on a
// line of N samples: kept bins X[i][k] = sum_n x[i][n] e^{-2 pi i k n / N}
// (k < M), Y[o][k] = sum_i X[i][k] W[i][o][k], and the half-spectrum inverse
// y[o][n] = (1/N) sum_k c(k) Re(Y[o][k] e^{+2 pi i k n / N}) with c(0) =
// c(N/2) = 1, c = 2 otherwise.  A 1-D layer is small (a few KiB per
// sample), so each sample runs on one cluster of kG1 CTAs: CTA r transforms
// the input channels i = r (mod kG1), the cluster gathers every channel's
// bins through distributed shared memory, and CTA r then mixes and inverts the
// output channels o = r (mod kG1).  Bins and twiddles are dense DFT sums
// (N * M terms per channel), which at these sizes costs less than the
// launches an FFT split would add.
#include "fno_fused.cuh"

namespace fno {
namespace {

constexpr int kG1 = 8;                     // CTAs per sample (one cluster)
constexpr int kT1 = 128;                   // threads per CTA
constexpr size_t kSmem1Max = 48u << 10;    // shared memory of one CTA (no opt-in)

size_t smem1_bytes(int n, int m, int cin, int cout) {
    const int own_out = (cout + kG1 - 1) / kG1;
    return ((size_t)n + (size_t)cin * m + (size_t)own_out * m) * sizeof(float2);
}

// grid: batch x kG1 CTAs, clusters of kG1 along x (rank = blockIdx.x % kG1)
template <typename T>
__global__ void __launch_bounds__(kT1)
k_fused1d(const T *__restrict__ x, const T *__restrict__ w, T *__restrict__ y, int cin,
          int cout, int N, int M, const float2 *__restrict__ tw_g, int packed) {
    extern __shared__ __align__(16) float2 sm1[];
    float2 *tw = sm1;                      // [N]      e^{-2 pi i j / N}
    float2 *X = tw + N;                    // [cin][M] bins of every input channel
    float2 *Y = X + (size_t)cin * M;       // [own outputs][M]
    const int r = blockIdx.x % kG1;
    const int64_t b = blockIdx.x / kG1;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int kWarps = kT1 / 32;
    for (int e = threadIdx.x; e < N; e += kT1) tw[e] = tw_g[e];
    __syncthreads();

    // 1. bins of this CTA's input channels: one warp per (channel, bin), lanes
    //    split the samples, then a warp reduction
    const int own_in = cin > r ? (cin - r + kG1 - 1) / kG1 : 0;
    for (int pidx = warp; pidx < own_in * M; pidx += kWarps) {
        const int i = r + kG1 * (pidx / M), k = pidx % M;
        const T *src = x + (b * cin + i) * (int64_t)N;
        float2 acc = make_float2(0.f, 0.f);
        for (int n = lane; n < N; n += 32) {
            const float v = Storage<T>::load(src + n);
            const float2 t = tw[(k * n) & (N - 1)];
            acc.x = fmaf(v, t.x, acc.x);
            acc.y = fmaf(v, t.y, acc.y);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        }
        if (lane == 0) X[(size_t)i * M + k] = acc;
    }

    // 2. gather the other channels' bins from the CTAs that computed them
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
    const uint32_t xs = (uint32_t)__cvta_generic_to_shared(X);
    for (int e = threadIdx.x; e < cin * M; e += kT1) {
        const int i = e / M, src_rank = i % kG1;
        if (src_rank == r) continue;
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                     : "=r"(remote) : "r"(xs + (uint32_t)e * 8), "r"(src_rank));
        float2 v;
        asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                     : "=f"(v.x), "=f"(v.y) : "r"(remote) : "memory");
        X[e] = v;
    }
    // every CTA has its copy before any CTA moves on (and may exit)
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");

    // 3. mixing for this CTA's output channels: Y[o][k] = sum_i X[i][k] W[i][o][k]
    const int own_out = cout > r ? (cout - r + kG1 - 1) / kG1 : 0;
    for (int e = threadIdx.x; e < own_out * M; e += kT1) {
        const int q = e / M, k = e % M, o = r + kG1 * q;
        float2 acc = make_float2(0.f, 0.f);
        for (int i = 0; i < cin; ++i)
            cfma(acc, X[(size_t)i * M + k],
                 Storage<T>::load2(w + (packed ? packed_index(k, i, o, cin, cout)
                                               : ((size_t)i * cout + o) * M + k) * 2));
        Y[e] = acc;
    }
    __syncthreads();

    // 4. inverse of this CTA's output channels, one sample per thread
    const float scale = 1.0f / (float)N;
    for (int e = threadIdx.x; e < own_out * N; e += kT1) {
        const int q = e / N, n = e % N, o = r + kG1 * q;
        const float2 *yq = Y + (size_t)q * M;
        float acc = 0.f;
        for (int k = 0; k < M; ++k) {
            const float c = (k == 0 || 2 * k == N) ? 1.f : 2.f;
            const float2 v = yq[k], t = tw[(k * n) & (N - 1)];
            // Re(v e^{+i theta}) with t = e^{-i theta}
            acc = fmaf(c, fmaf(v.x, t.x, v.y * t.y), acc);
        }
        Storage<T>::store(y + (b * cout + o) * (int64_t)N + n, acc * scale);
    }
}

}  // namespace

bool fused1d_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout) {
    return g.d == 1 && (dtype == FNO_F32 || dtype == FNO_F16 || dtype == FNO_BF16) &&
           g.n[0] <= 1024 && (g.n[0] & (g.n[0] - 1)) == 0 &&
           batch * kG1 < (1ll << 31) &&
           smem1_bytes((int)g.n[0], g.m[0], cin, cout) <= kSmem1Max;
}

cudaError_t fused1d_forward(const Plan &p, const Buffers &b, cudaStream_t s) {
    const int N = (int)p.g.n[0], M = p.g.m[0];
    cudaLaunchAttribute cl;
    cl.id = cudaLaunchAttributeClusterDimension;
    cl.val.clusterDim.x = kG1;
    cl.val.clusterDim.y = 1;
    cl.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.batch * kG1));
    cfg.blockDim = dim3(kT1);
    cfg.dynamicSmemBytes = smem1_bytes(N, M, p.cin, p.cout);
    cfg.stream = s;
    cfg.attrs = &cl;
    cfg.numAttrs = 1;
    const cudaError_t e = with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        return cudaLaunchKernelEx(&cfg, k_fused1d<T>, static_cast<const T *>(b.x),
                                  static_cast<const T *>(b.w), static_cast<T *>(b.y), p.cin,
                                  p.cout, N, M, static_cast<const float2 *>(p.tw[0]),
                                  (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0);
    });
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace fno
