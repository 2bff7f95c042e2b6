// fno_fused.cu -- the spectral-convolution layer as ONE persistent kernel.
//
// The TurboFNO article (gsyq.cn/news/457482) fuses FFT, channel mixing and
// inverse FFT into a single kernel so that the intermediates never make a
// round trip through device memory between launches (§3.4, §1).  On GB300
// the mixing of one mode needs every input channel of a sample, and the
// inverse of one output image needs every mode, so the layer has two
// all-to-all dependencies.  This kernel resolves them inside one launch with
// a ticket-ordered work queue:
//
//   phase A  (image, row chunk)   x rows  -> partial kept modes   (HBM read)
//   phase B  (mode group, o blk)  sum partials, mix with W -> Y   (L2 + W read)
//   phase C  (image, row chunk)   Y -> output rows                (HBM write)
//
// Every CTA takes the next ticket from an atomic counter; tickets are ordered
// A, then B, then C, and a B (C) item waits -- with a bounded spin -- until
// every A (B) item has been counted done.  An item only ever waits on items
// with smaller tickets, which were taken by CTAs already running, so the
// queue cannot deadlock whatever the residency of the grid.  The
// intermediates (partial modes, mixed modes) are a few MiB and stay in L2.
//
// Transforms (the article's §3.1 radix-2 butterflies, re-planned for
// registers): a row of N1 real samples is split n = n1 + P*n2; each thread
// runs a Q-point FFT (Q = N1/P) on two rows at once packed as re/im, then
// the P partial sums of a bin are combined with the twiddle W_N1^{n1 k}
// through a warp-shuffle reduce-scatter.  The rows of one chunk are the
// strided rows r = c + C*t, so the column DFT over a chunk is a full RC-point
// DFT (RC = N0/C rows) followed by the twiddle W_N0^{f c}; it is split as
// RC = A*B2 with B2-point register FFTs.  The inverse runs the same steps
// backwards with conjugate twiddles, applies the half-spectrum weights
// c(0) = 1, c(k) = 2 and the 1/(N0*N1) scale, and stores the rows.
#include <cstdio>
#include <type_traits>

#include "fno_fft.cuh"
#include "fno_fused.cuh"

namespace fno {
namespace {

using fft::cadd;
using fft::cconj;
using fft::cmac;
using fft::cmul;
using fft::cmulc;
using fft::cscale;
using fft::csub;

constexpr int kNT = 128;                       // threads per CTA
constexpr long long kWaitTimeoutNs = 500000000; // bounded device waits: 0.5 s

// Counters shared by the CTAs of one launch (plan-owned, zero between launches).
struct SyncBlock {
    int ticket;      // next work item
    int exited;      // CTAs that have left the queue
    int done_a;      // finished phase-A items
    int done_b;      // finished phase-B items
    int pad[60];
};

template <int N0_, int N1_, int M0_, int M1_, int RC_, int Q_, int B2_>
struct Cfg {
    static constexpr int N0 = N0_, N1 = N1_, M0 = M0_, M1 = M1_;
    static constexpr int K0 = 2 * M0;            // kept rows
    static constexpr int NK = K0 * M1;           // kept modes per image
    static constexpr int RC = RC_;               // rows per chunk
    static constexpr int C = N0 / RC;            // chunks per image
    static constexpr int Q = Q_;                 // row FFT length
    static constexpr int P = N1 / Q;             // row partial sums per bin
    static constexpr int B2 = B2_;               // column FFT length
    static constexpr int A = RC / B2;            // column partial sums
    static constexpr int XS = N1 + 8;            // padded smem row stride (floats)
    static constexpr int PAIRS = RC * P / 2;     // row-FFT work units (2 rows each)
    static constexpr int KB = P / 2;             // bins per reduce-scatter block
    static_assert(N0 % RC == 0 && N1 % Q == 0 && RC % B2 == 0, "tiling");
    static_assert(K0 <= RC, "kept rows must have distinct residues mod the chunk");
    static_assert(M1 <= Q, "row FFT must cover the kept bins");
    static_assert(P >= 2 && P <= 32 && (32 % P) == 0, "P lanes share a row");
    static_assert(M1 % KB == 0, "bins split into reduce-scatter blocks");
    static_assert(PAIRS % 128 == 0, "whole CTAs in the row pass (warp shuffles)");
    // smem floats for each phase
    static constexpr int kSmemA = RC * XS + 2 * RC * M1 + 2 * A * M1 * B2;
    static constexpr int kSmemC = 4 * RC * M1 + 2 * A * M1 * B2;
};

// Frequency of kept row j on axis 0: low rows 0..M0-1, then N0-M0..N0-1.
template <class Cf>
__device__ __forceinline__ int kept_freq(int j) {
    return j < Cf::M0 ? j : Cf::N0 - 2 * Cf::M0 + j;
}

template <typename T> struct Io;
template <> struct Io<float> {
    // 8 consecutive values -> float
    static __device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ float2 w2(const float *p) {
        return *reinterpret_cast<const float2 *>(p);
    }
    static __device__ __forceinline__ void store(float *p, float v) { __stcs(p, v); }
};
template <> struct Io<__half> {
    static __device__ __forceinline__ void load8(const __half *p, float (&v)[8]) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(p));
        const __half2 *h = reinterpret_cast<const __half2 *>(&a);
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(h[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ float2 w2(const __half *p) {
        return __half22float2(*reinterpret_cast<const __half2 *>(p));
    }
    static __device__ __forceinline__ void store(__half *p, float v) {
        *p = __float2half_rn(v);
    }
};

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ long long globaltimer() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Thread 0 waits until *ctr >= target; gives up (sets the error word) after
// kWaitTimeoutNs or as soon as another CTA has reported an error.
__device__ bool wait_count(const int *ctr, int target, int *err) {
    if (ld_acquire(ctr) >= target) return true;
    const long long t0 = globaltimer();
    for (unsigned spin = 0;; ++spin) {
        if (ld_acquire(ctr) >= target) {
            __threadfence();
            return true;
        }
        if (*reinterpret_cast<volatile int *>(err) != 0) return false;
        __nanosleep(64);
        if ((spin & 255u) == 255u && globaltimer() - t0 > kWaitTimeoutNs) {
            raise_dev_error(err, kDevTimeout);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Phase A: one chunk of rows of one input image -> partial kept modes
// ---------------------------------------------------------------------------
template <class Cf, typename T>
__device__ void phase_a(const T *__restrict__ x, float2 *__restrict__ part, int nimg, int img,
                        int c, float *smem, const float2 *tw0, const float2 *tw1) {
    constexpr int N1 = Cf::N1, RC = Cf::RC, C = Cf::C, P = Cf::P, Q = Cf::Q, M1 = Cf::M1;
    constexpr int XS = Cf::XS, A = Cf::A, B2 = Cf::B2, K0 = Cf::K0, NK = Cf::NK;
    float *xs = smem;                                             // [RC][XS]
    float2 *zs = reinterpret_cast<float2 *>(smem + RC * XS);      // [RC][M1]
    float2 *ss = zs + RC * M1;                                    // [A][M1][B2]
    const int tid = threadIdx.x;

    // 1. rows c, c+C, c+2C, ... of the image into shared memory (as float)
    const T *src = x + (size_t)img * Cf::N0 * N1;
    constexpr int kLoads = RC * (N1 / 8) / kNT;
    static_assert(RC * (N1 / 8) % kNT == 0, "whole load rounds");
    float v[kLoads][8];
#pragma unroll
    for (int r = 0; r < kLoads; ++r) {          // all loads in flight before any store
        const int e = tid + r * kNT;
        const int t = e / (N1 / 8), s = e % (N1 / 8);
        Io<T>::load8(src + (size_t)(c + C * t) * N1 + 8 * s, v[r]);
    }
#pragma unroll
    for (int r = 0; r < kLoads; ++r) {
        const int e = tid + r * kNT;
        const int t = e / (N1 / 8), s = e % (N1 / 8);
        float4 *dst = reinterpret_cast<float4 *>(xs + t * XS + 8 * s);
        dst[0] = make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
        dst[1] = make_float4(v[r][4], v[r][5], v[r][6], v[r][7]);
    }
    __syncthreads();

    // 2. row DFT, bins 0..M1-1: Z[t][k] = sum_n1 W_N1^{n1 k} U[t][n1][k], U = Q-point DFT of
    //    x[t][n1 + P n2] over n2.  Lanes P*g .. P*g+P-1 share rows (t, t + RC/2).
    for (int pr = tid; pr < Cf::PAIRS; pr += kNT) {
        const int t = pr / P, n1 = pr % P, t2 = t + RC / 2;
        float2 z[Q];
#pragma unroll
        for (int n2 = 0; n2 < Q; ++n2)
            z[n2] = make_float2(xs[t * XS + n1 + P * n2], xs[t2 * XS + n1 + P * n2]);
        fft::fft_dif<Q, -1>(z);
        const int lane_in_group = n1;   // == lane % P
        fft::unroll<0, M1 / Cf::KB>([&](auto kbi) {
            constexpr int kb = decltype(kbi)::value;
            // contributions of this lane for bins kb*KB .. kb*KB+KB-1 of both rows
            float2 v[2 * Cf::KB];
            fft::unroll<0, Cf::KB>([&](auto qi) {
                constexpr int k = kb * Cf::KB + decltype(qi)::value;
                float2 a, b;
                fft::split_real_pair<Q, k % Q>(z, a, b);
                const float2 w = tw1[(n1 * k) & (N1 - 1)];
                v[decltype(qi)::value] = cmul(a, w);
                v[Cf::KB + decltype(qi)::value] = cmul(b, w);
            });
            // reduce-scatter over the P lanes: lane l ends with element l of v
            fft::unroll<0, fft::ilog2(P)>([&](auto ri) {
                constexpr int half = P >> (decltype(ri)::value + 1);
                const bool upper = (lane_in_group & half) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float2 send = upper ? v[i] : v[i + half];
                    float2 keep = upper ? v[i + half] : v[i];
                    keep.x += __shfl_xor_sync(0xffffffffu, send.x, half);
                    keep.y += __shfl_xor_sync(0xffffffffu, send.y, half);
                    v[i] = keep;
                }
            });
            const int row = lane_in_group < Cf::KB ? t : t2;
            const int k = kb * Cf::KB + (lane_in_group % Cf::KB);
            zs[row * M1 + k] = v[0];
        });
    }
    __syncthreads();

    // 3a. column DFT over the chunk, inner B2-point FFTs: t = t1 + A*t2
    for (int u = tid; u < A * M1; u += kNT) {
        const int t1 = u / M1, k = u % M1;
        float2 z[B2];
#pragma unroll
        for (int i = 0; i < B2; ++i) z[i] = zs[(t1 + A * i) * M1 + k];
        fft::fft_dif<B2, -1>(z);
#pragma unroll
        for (int q = 0; q < B2; ++q) ss[(t1 * M1 + k) * B2 + q] = z[fft::bitrev(q, fft::ilog2(B2))];
    }
    __syncthreads();

    // 3b. X_c[j][k] = W_N0^{f c} sum_t1 W_RC^{f t1} S[t1][k][f mod B2], f = freq of kept row j
    float2 *dst = part + ((size_t)c * nimg + img) * NK;
    constexpr int kRcStep = Cf::N0 / RC;         // W_RC^e = tw0[e * N0/RC]
    for (int o = tid; o < NK; o += kNT) {
        const int j = o / M1, k = o % M1;
        const int f = kept_freq<Cf>(j);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int t1 = 0; t1 < A; ++t1)
            cmac(acc, ss[(t1 * M1 + k) * B2 + (f % B2)],
                 tw0[((f % RC) * t1 * kRcStep) & (Cf::N0 - 1)]);
        __stcg(dst + o, cmul(acc, tw0[(f * c) & (Cf::N0 - 1)]));
    }
    (void)K0;
}

// ---------------------------------------------------------------------------
// Phase B: Y[b][o][mode] = sum_i X[b][i][mode] W[blk][i][o][local], X = sum of partials
// ---------------------------------------------------------------------------
template <class Cf, int G, typename T>
__device__ void phase_b(const float2 *__restrict__ part, const T *__restrict__ w,
                        float2 *__restrict__ Y, int batch, int cin, int cout, int nimg_in,
                        int group, int oblk, int ob, float *smem) {
    constexpr int M0 = Cf::M0, M1 = Cf::M1, NK = Cf::NK, C = Cf::C;
    const int mode0 = group * G;                 // G consecutive bins of one kept row
    const int j = mode0 / M1, k0 = mode0 % M1;
    const int blk = j >= M0 ? 1 : 0, l0 = j - blk * M0;
    const int o0 = oblk * ob;
    const int nob = min(ob, cout - o0);
    float2 *ws = reinterpret_cast<float2 *>(smem);            // [cin][ob][G]
    float2 *xs = ws + (size_t)cin * ob * G;                   // [batch][cin][G]
    const int tid = threadIdx.x;
    const size_t mblk = (size_t)M0 * M1;
    for (int e = tid; e < cin * nob * G; e += kNT) {
        const int g = e % G, r = e / G, o = r % nob, i = r / nob;
        const T *p = w + ((((size_t)blk * cin + i) * cout + o0 + o) * mblk + l0 * M1 + k0 + g) * 2;
        ws[(i * ob + o) * G + g] = Io<T>::w2(p);
    }
    for (int e = tid; e < batch * cin * G; e += kNT) {
        const int g = e % G, r = e / G;            // r = b * cin + i
        float2 acc = __ldcg(part + (size_t)r * NK + mode0 + g);
#pragma unroll
        for (int cc = 1; cc < C; ++cc)
            acc = cadd(acc, __ldcg(part + ((size_t)cc * nimg_in + r) * NK + mode0 + g));
        xs[e] = acc;
    }
    __syncthreads();
    constexpr int BB = 8;                          // batch rows per register block
    for (int u = tid; u < nob * G; u += kNT) {
        const int o = u / G, g = u % G;
        for (int b0 = 0; b0 < batch; b0 += BB) {
            float2 acc[BB];
#pragma unroll
            for (int bb = 0; bb < BB; ++bb) acc[bb] = make_float2(0.f, 0.f);
            for (int i = 0; i < cin; ++i) {
                const float2 wv = ws[(i * ob + o) * G + g];
#pragma unroll
                for (int bb = 0; bb < BB; ++bb)
                    if (b0 + bb < batch) cmac(acc[bb], xs[((b0 + bb) * cin + i) * G + g], wv);
            }
#pragma unroll
            for (int bb = 0; bb < BB; ++bb)
                if (b0 + bb < batch)
                    __stcg(Y + ((size_t)(b0 + bb) * cout + o0 + o) * NK + mode0 + g, acc[bb]);
        }
    }
}

// ---------------------------------------------------------------------------
// Phase C: mixed modes of one output image -> one chunk of its rows
// ---------------------------------------------------------------------------
template <class Cf, typename T>
__device__ void phase_c(const float2 *__restrict__ Y, T *__restrict__ y, int img, int c,
                        float *smem, const float2 *tw0, const float2 *tw1) {
    constexpr int N0 = Cf::N0, N1 = Cf::N1, RC = Cf::RC, C = Cf::C, P = Cf::P, Q = Cf::Q;
    constexpr int M1 = Cf::M1, A = Cf::A, B2 = Cf::B2, K0 = Cf::K0, NK = Cf::NK;
    float2 *vs = reinterpret_cast<float2 *>(smem);            // [RC][M1] residue-ordered
    float2 *ss = vs + RC * M1;                                // [A][M1][B2]
    float2 *zo = ss + A * M1 * B2;                            // [RC][M1]
    const int tid = threadIdx.x;
    const float2 *src = Y + (size_t)img * NK;

    // 1. V[q][k] = Y[j][k] conj(W_N0^{f c}), q = f mod RC (distinct for the kept rows)
    for (int e = tid; e < RC * M1; e += kNT) {
        const int q = e / M1, k = e % M1;
        // kept row j with f(j) == q (mod RC), if any
        int j = -1;
        if (q < Cf::M0) j = q;
        else if (q >= RC - Cf::M0) j = K0 - (RC - q);
        float2 v = make_float2(0.f, 0.f);
        if (j >= 0) {
            const int f = kept_freq<Cf>(j);
            v = cmulc(__ldcg(src + j * M1 + k), tw0[(f * c) & (N0 - 1)]);
        }
        vs[e] = v;
    }
    __syncthreads();
    // 2a. inner B2-point inverse FFTs over q2 (q = q1 + A q2)
    for (int u = tid; u < A * M1; u += kNT) {
        const int q1 = u / M1, k = u % M1;
        float2 z[B2];
#pragma unroll
        for (int i = 0; i < B2; ++i) z[i] = vs[(q1 + A * i) * M1 + k];
        fft::fft_dif<B2, 1>(z);
#pragma unroll
        for (int r = 0; r < B2; ++r) ss[(q1 * M1 + k) * B2 + r] = z[fft::bitrev(r, fft::ilog2(B2))];
    }
    __syncthreads();
    // 2b. Zo[t][k] = sum_q1 W_RC^{-q1 t} S[q1][k][t mod B2]
    constexpr int kRcStep = N0 / RC;
    for (int e = tid; e < RC * M1; e += kNT) {
        const int t = e / M1, k = e % M1;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q1 = 0; q1 < A; ++q1) {
            const float2 wv = tw0[(q1 * t * kRcStep) & (N0 - 1)];
            cmac(acc, ss[(q1 * M1 + k) * B2 + (t % B2)], make_float2(wv.x, -wv.y));
        }
        zo[e] = acc;
    }
    __syncthreads();
    // 3. rows: y[t][n1 + P n2] = s Re sum_k c_k W_N1^{-k n1} Zo[t][k] W_Q^{-k n2}
    const float scale = 1.0f / ((float)N0 * (float)N1);
    T *dst = y + (size_t)img * N0 * N1;
    for (int pr = tid; pr < Cf::PAIRS; pr += kNT) {
        const int t = pr / P, n1 = pr % P, t2 = t + RC / 2;
        float2 ga[Q], gb[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            ga[q] = make_float2(0.f, 0.f);
            gb[q] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < M1; ++k) {
            const float ck = (k == 0 || 2 * k == N1) ? 1.f : 2.f;
            const float2 w = tw1[(k * n1) & (N1 - 1)];
            ga[k % Q] = cadd(ga[k % Q], cscale(cmulc(zo[t * M1 + k], w), ck));
            gb[k % Q] = cadd(gb[k % Q], cscale(cmulc(zo[t2 * M1 + k], w), ck));
        }
        // Hermitian parts, packed: z[q] = Herm(ga)[q] + i Herm(gb)[q]
        float2 z[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int qm = (Q - q) % Q;
            const float2 ha = make_float2(0.5f * (ga[q].x + ga[qm].x), 0.5f * (ga[q].y - ga[qm].y));
            const float2 hb = make_float2(0.5f * (gb[q].x + gb[qm].x), 0.5f * (gb[q].y - gb[qm].y));
            z[q] = make_float2(ha.x - hb.y, ha.y + hb.x);
        }
        fft::fft_dif<Q, 1>(z);
        T *ra = dst + (size_t)(c + C * t) * N1 + n1;
        T *rb = dst + (size_t)(c + C * t2) * N1 + n1;
#pragma unroll
        for (int n2 = 0; n2 < Q; ++n2) {
            const float2 v = z[fft::bitrev(n2, fft::ilog2(Q))];
            Io<T>::store(ra + P * n2, v.x * scale);
            Io<T>::store(rb + P * n2, v.y * scale);
        }
    }
}

// ---------------------------------------------------------------------------
// The persistent kernel
// ---------------------------------------------------------------------------
struct Args {
    const void *x;
    const void *w;
    void *y;
    float2 *part;       // [C][B*Cin][NK]
    float2 *Y;          // [B*Cout][NK]
    SyncBlock *sync;
    const float2 *tw0;  // N0 twiddles
    const float2 *tw1;  // N1 twiddles
    int *err;
    int batch, cin, cout;
    int nA, nB, nC;
    int ob;             // outputs per phase-B item
    int nob;            // phase-B items per mode group
};

template <class Cf, int G, typename T>
__global__ void __launch_bounds__(kNT)
k_fused2d(Args a) {
    extern __shared__ __align__(16) float smem[];
    __shared__ int s_item;
    float2 *tw0 = reinterpret_cast<float2 *>(smem);
    float2 *tw1 = tw0 + Cf::N0;
    float *work = reinterpret_cast<float *>(tw1 + Cf::N1);
    const int tid = threadIdx.x;
    for (int e = tid; e < Cf::N0; e += kNT) tw0[e] = a.tw0[e];
    for (int e = tid; e < Cf::N1; e += kNT) tw1[e] = a.tw1[e];
    const int nimg_in = a.batch * a.cin;
    const int total = a.nA + a.nB + a.nC;
    for (;;) {
        if (tid == 0) s_item = atomicAdd(&a.sync->ticket, 1);
        __syncthreads();
        const int item = s_item;
        __syncthreads();
        if (item >= total) break;
        if (item < a.nA) {
            phase_a<Cf, T>(static_cast<const T *>(a.x), a.part, nimg_in, item / Cf::C,
                           item % Cf::C, work, tw0, tw1);
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                atomicAdd(&a.sync->done_a, 1);
            }
        } else if (item < a.nA + a.nB) {
            const int it = item - a.nA;
            if (tid == 0) s_item = wait_count(&a.sync->done_a, a.nA, a.err) ? 1 : 0;
            __syncthreads();
            const bool ok = s_item != 0;
            __syncthreads();
            if (ok)
                phase_b<Cf, G, T>(a.part, static_cast<const T *>(a.w), a.Y, a.batch, a.cin,
                                  a.cout, nimg_in, it / a.nob, it % a.nob, a.ob, work);
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                atomicAdd(&a.sync->done_b, 1);
            }
        } else {
            const int it = item - a.nA - a.nB;
            if (tid == 0) s_item = wait_count(&a.sync->done_b, a.nB, a.err) ? 1 : 0;
            __syncthreads();
            const bool ok = s_item != 0;
            __syncthreads();
            if (ok)
                phase_c<Cf, T>(a.Y, static_cast<T *>(a.y), it / Cf::C, it % Cf::C, work, tw0,
                               tw1);
        }
        __syncthreads();
    }
    // the last CTA to leave resets the counters for the next launch
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(&a.sync->exited, 1);
        if (prev == (int)gridDim.x - 1) {
            a.sync->ticket = 0;
            a.sync->done_a = 0;
            a.sync->done_b = 0;
            __threadfence();
            a.sync->exited = 0;
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// 128 x 128 grid, 16 x 16 modes per block: chunks of 32 strided rows,
// 16-point row FFTs (8 partial sums per bin), 8-point column FFTs.
using Cfg128 = Cfg<128, 128, 16, 16, 32, 16, 8>;
constexpr int kG128 = 4;   // modes per phase-B item

template <class Cf, int G>
struct Variant {
    static size_t smem_bytes(int cin, int ob, int batch) {
        const size_t tw = (size_t)(Cf::N0 + Cf::N1) * sizeof(float2);
        const size_t a = (size_t)Cf::kSmemA * sizeof(float);
        const size_t c = (size_t)Cf::kSmemC * sizeof(float);
        const size_t b = ((size_t)cin * ob * G + (size_t)batch * cin * G) * sizeof(float2);
        size_t m = a > c ? a : c;
        m = m > b ? m : b;
        return tw + m;
    }
};

bool is_cfg128(const Geom &g) {
    return g.d == 2 && g.n[0] == 128 && g.n[1] == 128 && g.m[0] == 16 && g.m[1] == 16;
}

int pick_ob(int cin, int cout) {
    // outputs per phase-B item: keep the W slab (cin x ob x G complex) <= 32 KiB
    int ob = cout;
    while (ob > 1 && (size_t)cin * ob * kG128 * sizeof(float2) > (32u << 10)) ob = (ob + 1) / 2;
    return ob;
}

struct Layout {
    size_t part_off, y_off, total;
};

Layout layout(const Geom &g, int64_t batch, int cin, int cout) {
    Layout l;
    const size_t C = Cfg128::C;
    l.part_off = 0;
    const size_t part = C * batch * cin * g.nkept * sizeof(float2);
    l.y_off = (part + 255) & ~size_t(255);
    l.total = l.y_off + (((size_t)batch * cout * g.nkept * sizeof(float2) + 255) & ~size_t(255));
    return l;
}

template <typename T>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&k_fused2d<Cfg128, kG128, T>);
}

}  // namespace

bool fused_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout) {
    if (!is_cfg128(g)) return false;
    if (batch * (int64_t)cin * Cfg128::C >= (1 << 30) || batch * (int64_t)cout * Cfg128::C >= (1 << 30))
        return false;
    const int ob = pick_ob(cin, cout);
    return Variant<Cfg128, kG128>::smem_bytes(cin, ob, (int)batch) <= 200 * 1024 &&
           (dtype == FNO_F32 || dtype == FNO_F16);
}

size_t fused_workspace_bytes(const Geom &g, fno_dtype_t, int64_t batch, int cin, int cout) {
    return layout(g, batch, cin, cout).total;
}

int fused_kernel_count(const Geom &, fno_dtype_t, int64_t, int, int) { return 1; }

cudaError_t fused_plan_init(Plan &p) {
    const int ob = pick_ob(p.cin, p.cout);
    const size_t smem = Variant<Cfg128, kG128>::smem_bytes(p.cin, ob, (int)p.batch);
    void *fn = p.dtype == FNO_F32 ? kernel_ptr<float>() : kernel_ptr<__half>();
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kNT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    p.fused_grid = p.num_sms * per_sm;
    p.fused_smem = smem;
    p.fused_ob = ob;
    return cudaMemset(p.sync, 0, sizeof(SyncBlock));
}

void fused_plan_release(Plan &) {}

cudaError_t fused_forward(const Plan &p, const Buffers &b, cudaStream_t s) {
    const Layout l = layout(p.g, p.batch, p.cin, p.cout);
    Args a;
    a.x = b.x;
    a.w = b.w;
    a.y = b.y;
    a.part = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) + l.part_off);
    a.Y = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) + l.y_off);
    a.sync = reinterpret_cast<SyncBlock *>(p.sync);
    a.tw0 = p.tw[0];
    a.tw1 = p.tw[1];
    a.err = p.dev_err;
    a.batch = (int)p.batch;
    a.cin = p.cin;
    a.cout = p.cout;
    a.nA = (int)p.batch * p.cin * Cfg128::C;
    a.ob = p.fused_ob;
    a.nob = (p.cout + a.ob - 1) / a.ob;
    a.nB = (int)(p.g.nkept / kG128) * a.nob;
    a.nC = (int)p.batch * p.cout * Cfg128::C;
    const int grid = p.fused_grid < a.nA + a.nB + a.nC ? p.fused_grid : a.nA + a.nB + a.nC;
    if (p.dtype == FNO_F32)
        k_fused2d<Cfg128, kG128, float><<<grid, kNT, p.fused_smem, s>>>(a);
    else
        k_fused2d<Cfg128, kG128, __half><<<grid, kNT, p.fused_smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace fno
