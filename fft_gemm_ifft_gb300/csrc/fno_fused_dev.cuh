// fno_fused_dev.cuh -- device building blocks shared by the fused layer kernels:
// configuration structs, load/store helpers, the bounded device waits, and
// the three phases of the layer (forward transform of a chunk of rows, the
// per-mode mixing, inverse transform of a chunk of rows) split into steps
// that the 2-D and 3-D kernels compose.
#pragma once

#include <cuda.h>

#include <cmath>
#include <cstring>
#include <type_traits>

#include "fno_fft.cuh"
#include "fno_fused.cuh"

namespace fno {
namespace {

using fft::cadd;
using fft::cmac;
using fft::cmul;
using fft::cmulc;
using fft::cscale;

constexpr int kNT = 128;                        // threads per CTA
constexpr long long kWaitTimeoutNs = 500000000;  // bounded device waits: 0.5 s
constexpr int kG = 2;                           // kept modes per phase-B item
#ifndef FNO_WS_BUDGET
#define FNO_WS_BUDGET 16384
#endif
constexpr size_t kWsBudget = FNO_WS_BUDGET;      // phase-B weight slab (bytes)
constexpr size_t kXpBudget = 24u << 10;         // phase-B partial modes (bytes)

// Counters shared by the CTAs of one launch (plan-owned, zero between
// launches).  Each counter has its own 128-byte line; the end of a phase is
// published as kFlagCopies flags on separate lines so that the CTAs waiting
// for it spread their polling over many L2 lines instead of one.
constexpr int kLine = 32;          // ints per 128-byte line
constexpr int kFlagCopies = 16;
constexpr int kMaxGroups = 16;     // batch groups of one launch
#ifndef FNO_TARGET_GROUPS
#define FNO_TARGET_GROUPS 2
#endif
constexpr int kTargetGroups = FNO_TARGET_GROUPS;   // batch groups the phases pipeline over
#ifndef FNO_WEIGHT_PREFETCH
#define FNO_WEIGHT_PREFETCH 0
#endif
constexpr bool kWeightPrefetch = FNO_WEIGHT_PREFETCH;   // phase-A items prefetch W into L2
struct SyncBlock {
    int ticket[kLine];                         // [0]: next work item
    int exited[kLine];                         // [0]: CTAs that have left the queue
    int done_a[kMaxGroups][kLine];             // [g][0]: finished phase-A items of group g
    int done_b[kMaxGroups][kLine];             // [g][0]: finished phase-B items of group g
    int flag_a[kMaxGroups][kFlagCopies][kLine];  // [g][i][0] = 1: phase A of group g done
    int flag_b[kMaxGroups][kFlagCopies][kLine];  // [g][i][0] = 1: phase B of group g done
};
constexpr size_t kSyncBytes = sizeof(SyncBlock);

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
    // x row stride in shared memory (floats): the P lanes of a row read
    // consecutive samples and a warp's 32 / P rows start P banks apart, so the
    // row DFT's loads are conflict-free
    static constexpr int XS = N1 + P;
    // row stride of raw storage-type rows (the 3-D plane ring): XS where its rows
    // stay 16-byte aligned, else N1 + 8
    template <typename S>
    static constexpr int xs_of() {
        return ((size_t)XS * sizeof(S)) % 16 == 0 ? XS : N1 + 8;
    }
    static constexpr int ZS = M1 + 4;            // Z row stride in smem (float2)
    static constexpr int TS = M1 + 1;            // per-lane twiddle row stride (float2)
    static constexpr int PAIRS = RC * P / 2;     // row-FFT work units (2 rows each)
    static constexpr int KB = P / 2;             // bins per reduce-scatter block
    static_assert(N0 % RC == 0 && N1 % Q == 0 && RC % B2 == 0, "tiling");
    static_assert(K0 <= RC, "kept rows must have distinct residues mod the chunk");
    static_assert(M1 <= Q, "row FFT must cover the kept bins");
    static_assert(P >= 2 && P <= 32 && (32 % P) == 0, "P lanes share a row");
    static_assert(M1 % KB == 0, "bins split into reduce-scatter blocks");
    static_assert(PAIRS % kNT == 0, "whole CTAs in the row pass (warp shuffles)");
    static_assert((RC * N1 / 4) % kNT == 0, "whole load rounds");
    static_assert(NK % kG == 0 && M1 % kG == 0, "mode pairs stay in one kept row");
    // bytes of each phase's shared memory
    static constexpr size_t kSmemA =
        RC * XS * 4 + RC * ZS * 8 + (size_t)A * B2 * M1 * 8;
    static constexpr size_t kSmemC =
        NK * 8 + RC * M1 * 8 + (size_t)A * B2 * M1 * 8 + RC * ZS * 8;
    static constexpr size_t kSmemTw = ((N0 + 2 * P * TS) * 8 + 15) / 16 * 16;
    // weights: block 0 holds the low kept rows, block 1 the high ones, each
    // M0 x M1 modes
    static constexpr size_t MBLK = (size_t)M0 * M1;
    static constexpr int MR = M1;                // kept modes along one line of the last axis
    __device__ static void wmap(int o, int &blk, int &local) {
        const int j = o / M1, k = o % M1;
        blk = j >= M0 ? 1 : 0;
        local = (j - blk * M0) * M1 + k;
    }
};

// Frequency of kept row j on axis 0: low rows 0..M0-1, then N0-M0..N0-1.
template <class Cf>
__device__ __forceinline__ int kept_freq(int j) {
    return j < Cf::M0 ? j : Cf::N0 - 2 * Cf::M0 + j;
}

template <typename T> struct Io;
template <> struct Io<float> {
    using W2 = float4;                               // two complex weights
    static __device__ __forceinline__ float4 load4(const float *p) {
        return __ldcs(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ void store(float *p, float v) { __stcs(p, v); }
    static __device__ __forceinline__ float2 wget(const float4 &w, int g) {
        return g == 0 ? make_float2(w.x, w.y) : make_float2(w.z, w.w);
    }
};
template <> struct Io<__half> {
    using W2 = uint2;                                // two complex weights (4 halves)
    static __device__ __forceinline__ float4 load4(const __half *p) {
        const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(p));
        const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&a.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&a.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    static __device__ __forceinline__ void store(__half *p, float v) {
        *p = __float2half_rn(v);
    }
    static __device__ __forceinline__ float2 wget(const uint2 &w, int g) {
        const unsigned u = g == 0 ? w.x : w.y;
        return __half22float2(*reinterpret_cast<const __half2 *>(&u));
    }
};

template <> struct Io<__nv_bfloat16> {
    using W2 = uint2;                                // two complex weights (4 bfloat16)
    static __device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
        const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(p));
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float v) {
        *p = __float2bfloat16_rn(v);
    }
    static __device__ __forceinline__ float2 wget(const uint2 &w, int g) {
        const unsigned u = g == 0 ? w.x : w.y;
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
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
__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}
// 16-byte asynchronous copy global -> shared through L2 only (data written by
// other CTAs of this launch must not be served from a stale L1 line)
__device__ __forceinline__ void cp_async16(void *s, const void *g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(s)), "l"(g)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void *s, const void *g) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(s)), "l"(g)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}


// Thread 0 waits until *flag != 0; gives up (sets the error word) after
// kWaitTimeoutNs or as soon as another CTA has reported an error.
__device__ bool wait_flag(const int *flag, int *err) {
    if (ld_acquire(flag) != 0) return true;
    const long long t0 = globaltimer();
    for (unsigned spin = 0;; ++spin) {
        if (ld_acquire(flag) != 0) return true;
        if (*reinterpret_cast<volatile int *>(err) != 0) return false;
        __nanosleep(64);
        if ((spin & 255u) == 255u && globaltimer() - t0 > kWaitTimeoutNs) {
            raise_dev_error(err, kDevTimeout);
            return false;
        }
    }
}

// Thread 0 counts one finished item of a phase (after a barrier of its
// group, so the group's writes are ordered before it); the item that completes
// the phase publishes every flag copy.  The count is an acquire-release atomic
// rather than a full fence plus atomic: it releases this group's writes and,
// for the last item, acquires every other item's.
__device__ void finish_item(int *counter, int total, int (*flags)[kLine]) {
    // flags points at the kFlagCopies lines of one group
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    if (old == total - 1) {
        // one fence orders everything this item acquired before all the flag
        // stores (a release on each store would cost a fence apiece)
        __threadfence();
        for (int i = 0; i < kFlagCopies; ++i) *reinterpret_cast<volatile int *>(&flags[i][0]) = 1;
    }
}

// L2 prefetch of a byte range (16-byte aligned, multiple of 16 bytes)
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

struct Tw {
    const float2 *t0;   // [N0]      W_N0^e
    const float2 *t1;   // [P][TS]   W_N1^{n1 k} / 2         (forward row pass)
    const float2 *t1i;  // [P][TS]   W_N1^{n1 k} c(k)/2 s    (inverse row pass, used conjugated)
};

// Row-pass tables of a configuration from the plan's W_N1 table: the forward
// carries the 1/2 of the real-pair split, the inverse the half-spectrum weight
// c(k)/2 and the output scale s (powers of two: every entry is exact).
template <class Cf>
__device__ __forceinline__ void fill_row_tables(const float2 *__restrict__ src, float2 *t1,
                                                float2 *t1i, float s) {
    for (int e = threadIdx.x; e < Cf::P * Cf::TS; e += kNT) {
        const int n1 = e / Cf::TS, k = e % Cf::TS;
        const float2 w = src[(n1 * k) & (Cf::N1 - 1)];
        t1[e] = make_float2(0.5f * w.x, 0.5f * w.y);
        const float h = ((k == 0 || 2 * k == Cf::N1) ? 0.5f : 1.f) * s;
        t1i[e] = make_float2(h * w.x, h * w.y);
    }
}

// ---------------------------------------------------------------------------
// Phase A: one chunk of rows of one input image -> partial kept modes
// ---------------------------------------------------------------------------
// 1. rows c, c+C, c+2C, ... of an image into shared memory (as float); every
//    load of the chunk is in flight before the first store
template <class Cf, typename T>
__device__ __forceinline__ void a_load_rows(const T *__restrict__ src, int c, float *xs) {
    constexpr int N1 = Cf::N1, RC = Cf::RC, C = Cf::C, XS = Cf::XS;
    const int tid = threadIdx.x;
    constexpr int kLoads = RC * N1 / 4 / kNT;
    float4 v[kLoads];
#pragma unroll
    for (int r = 0; r < kLoads; ++r) {
        const int e = tid + r * kNT;
        const int t = e / (N1 / 4), s = e % (N1 / 4);
        v[r] = Io<T>::load4(src + (size_t)(c + C * t) * N1 + 4 * s);
    }
#pragma unroll
    for (int r = 0; r < kLoads; ++r) {
        const int e = tid + r * kNT;
        const int t = e / (N1 / 4), s = e % (N1 / 4);
        *reinterpret_cast<float4 *>(xs + t * XS + 4 * s) = v[r];
    }
}

// 2. row DFT, bins 0..M1-1: Z[t][k] = sum_n1 W_N1^{n1 k} U[t][n1][k], U = Q-point DFT of
//    x[t][n1 + P n2] over n2.  Lanes P*g .. P*g+P-1 share rows (t, t + RC/2).
__device__ __forceinline__ float smp(const float *p) { return *p; }
__device__ __forceinline__ float smp(const __half *p) { return __half2float(*p); }
__device__ __forceinline__ float smp(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <class Cf, typename S = float, int XS = Cf::XS>
__device__ __forceinline__ void a_row_dft(const S *xs, float2 *zs, Tw tw) {
    constexpr int RC = Cf::RC, P = Cf::P, Q = Cf::Q, M1 = Cf::M1, ZS = Cf::ZS;
    constexpr int KB = Cf::KB;
    for (int pr = threadIdx.x; pr < Cf::PAIRS; pr += kNT) {
        const int t = pr / P, n1 = pr % P, t2 = t + RC / 2;
        float2 z[Q];
#pragma unroll
        for (int n2 = 0; n2 < Q; ++n2)
            z[n2] = make_float2(smp(xs + t * XS + n1 + P * n2), smp(xs + t2 * XS + n1 + P * n2));
        fft::fft_dif<Q, -1>(z);
        const float2 *twl = tw.t1 + n1 * Cf::TS;
        fft::unroll<0, M1 / KB>([&](auto kbi) {
            constexpr int kb = decltype(kbi)::value;
            // contributions of this lane for bins kb*KB .. kb*KB+KB-1 of both rows
            float2 vv[2 * KB];
            fft::unroll<0, KB>([&](auto qi) {
                constexpr int q = decltype(qi)::value;
                constexpr int k = kb * KB + q;
                float2 a, b;                      // twice the two rows' bins;
                fft::split_real_pair2<Q, k % Q>(z, a, b);   // the table holds W / 2
                const float2 w = twl[k];
                vv[q] = cmul(a, w);
                vv[KB + q] = cmul(b, w);
            });
            // reduce-scatter over the P lanes: lane l ends with element l of vv
            fft::unroll<0, fft::ilog2(P)>([&](auto ri) {
                constexpr int half = P >> (decltype(ri)::value + 1);
                const bool upper = (n1 & half) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float2 send = upper ? vv[i] : vv[i + half];
                    float2 keep = upper ? vv[i + half] : vv[i];
                    keep.x += __shfl_xor_sync(0xffffffffu, send.x, half);
                    keep.y += __shfl_xor_sync(0xffffffffu, send.y, half);
                    vv[i] = keep;
                }
            });
            const int row = n1 < KB ? t : t2;
            zs[row * ZS + kb * KB + (n1 % KB)] = vv[0];
        });
    }
}

// 3a. column DFT over the chunk, inner B2-point FFTs: t = t1 + A*t2
template <class Cf>
__device__ __forceinline__ void a_col_fft(const float2 *zs, float2 *ss) {
    constexpr int M1 = Cf::M1, ZS = Cf::ZS, A = Cf::A, B2 = Cf::B2;
    for (int u = threadIdx.x; u < A * M1; u += kNT) {
        const int t1 = u / M1, k = u % M1;
        float2 z[B2];
#pragma unroll
        for (int i = 0; i < B2; ++i) z[i] = zs[(t1 + A * i) * ZS + k];
        fft::fft_dif<B2, -1>(z);
#pragma unroll
        for (int q = 0; q < B2; ++q)
            ss[(t1 * B2 + q) * M1 + k] = z[fft::bitrev(q, fft::ilog2(B2))];
    }
}

// 3b. X_c[j][k] = W_N0^{f c} sum_t1 W_RC^{f t1} S[t1][f mod B2][k] for kept mode
//     o = j*M1 + k, f = freq of kept row j (c = 0: the chunk is the whole image)
template <class Cf>
__device__ __forceinline__ float2 a_kept_mode(const float2 *ss, int o, int c, Tw tw) {
    constexpr int N0 = Cf::N0, RC = Cf::RC, M1 = Cf::M1, A = Cf::A, B2 = Cf::B2;
    constexpr int kRcStep = N0 / RC;             // W_RC^e = W_N0^{e N0/RC}
    const int j = o / M1, k = o % M1;
    const int f = kept_freq<Cf>(j);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int t1 = 0; t1 < A; ++t1)
        cmac(acc, ss[(t1 * B2 + (f % B2)) * M1 + k],
             tw.t0[((f % RC) * t1 * kRcStep) & (N0 - 1)]);
    return c == 0 ? acc : cmul(acc, tw.t0[(f * c) & (N0 - 1)]);
}

template <class Cf, typename T, bool kCluster = false>
__device__ void phase_a(const T *__restrict__ x, float2 *__restrict__ part, int nimg, int img,
                        int c, char *smem, Tw tw) {
    constexpr int N0 = Cf::N0, N1 = Cf::N1, RC = Cf::RC, C = Cf::C;
    constexpr int XS = Cf::XS, ZS = Cf::ZS;
    constexpr int NK = Cf::NK;
    float *xs = reinterpret_cast<float *>(smem);                         // [RC][XS]
    float2 *zs = reinterpret_cast<float2 *>(smem + RC * XS * 4);         // [RC][ZS]
    float2 *ss = zs + RC * ZS;                                           // [A][B2][M1]
    const int tid = threadIdx.x;

    a_load_rows<Cf, T>(x + (size_t)img * N0 * N1, c, xs);
    __syncthreads();
    a_row_dft<Cf>(xs, zs, tw);
    __syncthreads();
    a_col_fft<Cf>(zs, ss);
    __syncthreads();

    // 3b. the chunk's partial modes.  Without a cluster they go to the workspace
    //     (the mixing sums the C partials); in a cluster of the image's C chunk-CTAs
    //     they stay in shared memory (over the x rows, no longer needed) and each
    //     CTA sums one C-th of the modes over the cluster's CTAs, writing X once.
    float2 *xpart = reinterpret_cast<float2 *>(smem);
    float2 *dst = part + ((size_t)(kCluster ? 0 : c) * nimg + img) * NK;
    for (int o = tid; o < NK; o += kNT) {
        const float2 acc = a_kept_mode<Cf>(ss, o, c, tw);
        if constexpr (kCluster)
            xpart[o] = acc;
        else
            __stcg(dst + o, acc);
    }
    if constexpr (kCluster) {
        static_assert(NK % C == 0, "mode slices");
        asm volatile("barrier.cluster.arrive.release.aligned;\n"
                     "barrier.cluster.wait.acquire.aligned;" ::: "memory");
        const uint32_t local = (uint32_t)__cvta_generic_to_shared(xpart);
        constexpr int kSlice = NK / C;           // modes this CTA reduces
        for (int o = c * kSlice + tid; o < (c + 1) * kSlice; o += kNT) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < C; ++r) {
                uint32_t remote;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                             : "=r"(remote) : "r"(local + o * 8), "r"(r));
                float2 v;
                asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                             : "=f"(v.x), "=f"(v.y) : "r"(remote) : "memory");
                acc.x += v.x;
                acc.y += v.y;
            }
            __stcg(dst + o, acc);
        }
        // no CTA may leave while another still reads its shared memory
        asm volatile("barrier.cluster.arrive.release.aligned;\n"
                     "barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
}

// ---------------------------------------------------------------------------
// Phase B: Y[b][o][mode] = sum_i X[b][i][mode] W[blk][i][o][local], X = sum of partials.
// One item: kG consecutive bins of one kept row, outputs [o0, o0+nob), the batch
// rows [b0, b0+nbb) of one batch group.  The weight slab is requested before the
// item waits for phase A of its group.  Each thread accumulates a register tile
// of BT batch rows x 2 outputs x 2 bins over every S-th input channel; the S
// lanes that share a tile then combine their sums by a shuffle reduce-scatter.
// ---------------------------------------------------------------------------
// A group of threads that runs one item: the whole CTA, or one of the
// independent streams of the tensor-core kernel (synchronised by a named barrier).
struct CtaGroup {
    int tid;
    __device__ void sync() const { __syncthreads(); }
};
struct StreamGroup {
    int tid;
    int bar;      // named barrier id (1, 2, ...), 256 threads
    __device__ void sync() const { asm volatile("bar.sync %0, 256;" ::"r"(bar) : "memory"); }
};

struct BItem {
    int pair, o0, nob, b0, nbb;
};
constexpr int kBT = 4;      // batch rows per register tile

template <class Cf, typename T, int NT, class G>
__device__ void phase_b_weights(const G &grp, const T *__restrict__ w, int cin, int cout,
                                const BItem &it, int ob, char *smem, bool packed = false) {
    using W2 = typename Io<T>::W2;
    int blk, local;
    Cf::wmap(it.pair * kG, blk, local);          // the pair is adjacent in its block
    W2 *ws = reinterpret_cast<W2 *>(smem);                   // [cin][ob]
    // element e = i * nob + o of the slab; a thread steps by NT elements, with
    // the divisions done once
    const int nob = it.nob;
    int i = grp.tid / nob, o = grp.tid - i * nob;
    const int di = NT / nob, dO = NT - di * nob;
    // the pair's two modes are adjacent in both layouts (the pair starts at an even
    // kept index: within one group of four when packed)
    const T *base = w + (((size_t)blk * cin * cout + it.o0) * Cf::MBLK + local) * 2;
    while (i < cin) {
        const T *p = packed ? w + packed_index(it.pair * kG, i, it.o0 + o, cin, cout) * 2
                            : base + (size_t)(i * cout + o) * (Cf::MBLK * 2);
        if constexpr (sizeof(W2) == 16)
            cp_async16(ws + i * ob + o, p);
        else
            cp_async8(ws + i * ob + o, p);
        i += di;
        o += dO;
        if (o >= nob) {
            o -= nob;
            ++i;
        }
    }
    cp_async_commit();
}

// lanes per tile (split of the input channels) for a given tile count
__host__ __device__ inline int b_split(int tiles, int nt) {
    int s = 1;
    while (s < 16 && tiles * s * 2 <= nt) s *= 2;
    return s;
}

template <class Cf, typename T, int S, int NT, class G>
__device__ void phase_b_tiles(const G &grp, float2 *__restrict__ Y, int cin, int cout, const BItem &it,
                              int ob, const typename Io<T>::W2 *ws, const float4 *xp,
                              int tiles) {
    using W2 = typename Io<T>::W2;
    constexpr int NK = Cf::NK;
    constexpr int V = kBT * 2 * kG;                      // values per tile
    static_assert(V % S == 0, "tile values split evenly over the lanes");
    const int mode0 = it.pair * kG;
    const int no2 = (it.nob + 1) / 2;
    // every lane of a warp runs the same number of passes (the shuffles below
    // need the whole warp); lanes past the last tile add zeros and store nothing
    const int total = tiles * S, bound = (total + 31) / 32 * 32;
    for (int u = grp.tid; u < bound; u += NT) {
        const bool active = u < total;
        const int s = u % S, tile = active ? u / S : 0;
        const int o = 2 * (tile % no2), b = kBT * (tile / no2);
        const bool o1 = o + 1 < it.nob;
        float2 vv[V];                                    // [bb][oo][g]
#pragma unroll
        for (int q = 0; q < V; ++q) vv[q] = make_float2(0.f, 0.f);
        for (int i = s; active && i < cin; i += S) {
            const W2 w0 = ws[i * ob + o];
            const W2 w1 = o1 ? ws[i * ob + o + 1] : w0;
            float2 wv[2][kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                wv[0][g] = Io<T>::wget(w0, g);
                wv[1][g] = Io<T>::wget(w1, g);
            }
#pragma unroll
            for (int bb = 0; bb < kBT; ++bb) {
                const int bi = b + bb < it.nbb ? b + bb : it.nbb - 1;
                const float4 xv = xp[bi * cin + i];
                const float2 x0 = make_float2(xv.x, xv.y), x1 = make_float2(xv.z, xv.w);
#pragma unroll
                for (int oo = 0; oo < 2; ++oo) {
                    cmac(vv[(bb * 2 + oo) * kG + 0], x0, wv[oo][0]);
                    cmac(vv[(bb * 2 + oo) * kG + 1], x1, wv[oo][1]);
                }
            }
        }
        // reduce-scatter over the S adjacent lanes of the tile: lane s ends with
        // the sums of values s*(V/S) .. s*(V/S) + V/S - 1 in vv[0 .. V/S)
        fft::unroll<0, fft::ilog2(S)>([&](auto ri) {
            constexpr int h = S >> (decltype(ri)::value + 1);
            constexpr int len = V >> (decltype(ri)::value + 1);
            const bool upper = (s & h) != 0;
#pragma unroll
            for (int q = 0; q < len; ++q) {
                const float2 send = upper ? vv[q] : vv[q + len];
                float2 keep = upper ? vv[q + len] : vv[q];
                keep.x += __shfl_xor_sync(0xffffffffu, send.x, h);
                keep.y += __shfl_xor_sync(0xffffffffu, send.y, h);
                vv[q] = keep;
            }
        });
        constexpr int per = V / S;
#pragma unroll
        for (int q = 0; q < per; ++q) {
            const int v = s * per + q;
            const int g = v % kG, oo = (v / kG) % 2, bb = v / (2 * kG);
            if (active && b + bb < it.nbb && o + oo < it.nob)
                __stcg(Y + ((size_t)(it.b0 + b + bb) * cout + it.o0 + o + oo) * NK + mode0 + g,
                       vv[q]);
        }
    }
}

// The partial modes of the item's rows into xp: xp[cc][r] = X_cc[b0*cin + r][mode0 ..
// mode0+1] for the kParts partial copies (issued, not committed)
template <class Cf, int NT, class G, int kParts = Cf::C>
__device__ __forceinline__ void phase_b_issue_parts(const G &grp, const float2 *__restrict__ part,
                                                    int cin, int nimg_in, const BItem &it,
                                                    float4 *xp) {
    constexpr int NK = Cf::NK;
    const int mode0 = it.pair * kG;
    const int nr = it.nbb * cin;                         // rows (b, i) of this item
#pragma unroll
    for (int cc = 0; cc < kParts; ++cc) {
        const float2 *src = part + ((size_t)cc * nimg_in + (size_t)it.b0 * cin) * NK + mode0;
        for (int r = grp.tid; r < nr; r += NT) cp_async16(xp + cc * nr + r, src + (size_t)r * NK);
    }
}

// byte offset of the partial modes behind the weight slab [cin][ob] in an item's
// shared memory
template <typename T>
__host__ __device__ inline size_t b_xp_offset(int cin, int ob) {
    return ((size_t)cin * ob * sizeof(typename Io<T>::W2) + 15) / 16 * 16;
}

// Given the item's weight slab and partials in shared memory (visible to the
// group): sum the partials, then the register tiles and the stores of Y.
template <class Cf, typename T, int NT, class G, int kParts = Cf::C>
__device__ void phase_b_compute(const G &grp, float2 *__restrict__ Y, int cin, int cout,
                                const BItem &it, int ob, char *smem) {
    using W2 = typename Io<T>::W2;
    constexpr int C = kParts;
    const W2 *ws = reinterpret_cast<const W2 *>(smem);                       // [cin][ob]
    float4 *xp = reinterpret_cast<float4 *>(smem + b_xp_offset<T>(cin, ob));
    const int tid = grp.tid;
    const int nr = it.nbb * cin;
    if constexpr (C > 1) {
        for (int r = tid; r < nr; r += NT) {
            float4 s = xp[r];
#pragma unroll
            for (int cc = 1; cc < C; ++cc) {
                const float4 q = xp[cc * nr + r];
                s.x += q.x; s.y += q.y; s.z += q.z; s.w += q.w;
            }
            xp[r] = s;
        }
        grp.sync();
    }
    const int nbt = (it.nbb + kBT - 1) / kBT, no2 = (it.nob + 1) / 2;
    const int tiles = nbt * no2;
    switch (b_split(tiles, NT)) {
        case 16: phase_b_tiles<Cf, T, 16, NT>(grp, Y, cin, cout, it, ob, ws, xp, tiles); break;
        case 8: phase_b_tiles<Cf, T, 8, NT>(grp, Y, cin, cout, it, ob, ws, xp, tiles); break;
        case 4: phase_b_tiles<Cf, T, 4, NT>(grp, Y, cin, cout, it, ob, ws, xp, tiles); break;
        case 2: phase_b_tiles<Cf, T, 2, NT>(grp, Y, cin, cout, it, ob, ws, xp, tiles); break;
        default: phase_b_tiles<Cf, T, 1, NT>(grp, Y, cin, cout, it, ob, ws, xp, tiles); break;
    }
}

template <class Cf, typename T, int NT, class G, int kParts = Cf::C>
__device__ void phase_b(const G &grp, const float2 *__restrict__ part, float2 *__restrict__ Y, int cin,
                        int cout, int nimg_in, const BItem &it, int ob, char *smem,
                        unsigned long long *t_loaded = nullptr) {
    float4 *xp = reinterpret_cast<float4 *>(smem + b_xp_offset<T>(cin, ob));
    phase_b_issue_parts<Cf, NT, G, kParts>(grp, part, cin, nimg_in, it, xp);
    cp_async_commit();
    cp_async_wait_all();                                 // also covers the weight slab
    grp.sync();
    if (t_loaded && grp.tid == 0) *t_loaded = (unsigned long long)globaltimer();
    phase_b_compute<Cf, T, NT, G, kParts>(grp, Y, cin, cout, it, ob, smem);
}

// ---------------------------------------------------------------------------
// Phase C: mixed modes of one output image -> one chunk of its rows
// ---------------------------------------------------------------------------
// Step 1 (given the image's kept modes ys[K0][M1] in shared memory):
// V[q][k] = Y[j][k] conj(W_N0^{f c}), q = f mod RC (distinct for the kept rows)
template <class Cf>
__device__ __forceinline__ void c_residues(const float2 *ys, float2 *vs, int c, Tw tw) {
    constexpr int N0 = Cf::N0, RC = Cf::RC, M0 = Cf::M0, M1 = Cf::M1, K0 = Cf::K0;
    for (int e = threadIdx.x; e < RC * M1; e += kNT) {
        const int q = e / M1, k = e % M1;
        int j = -1;
        if (q < M0) j = q;
        else if (q >= RC - M0) j = K0 - (RC - q);
        float2 v = make_float2(0.f, 0.f);
        if (j >= 0) v = c == 0 ? ys[j * M1 + k]
                               : cmulc(ys[j * M1 + k], tw.t0[(kept_freq<Cf>(j) * c) & (N0 - 1)]);
        vs[e] = v;
    }
}

// 2a. inner B2-point inverse FFTs over q2 (q = q1 + A q2)
template <class Cf>
__device__ __forceinline__ void c_col_ifft(const float2 *vs, float2 *ss) {
    constexpr int M1 = Cf::M1, A = Cf::A, B2 = Cf::B2;
    for (int u = threadIdx.x; u < A * M1; u += kNT) {
        const int q1 = u / M1, k = u % M1;
        float2 z[B2];
#pragma unroll
        for (int i = 0; i < B2; ++i) z[i] = vs[(q1 + A * i) * M1 + k];
        fft::fft_dif<B2, 1>(z);
#pragma unroll
        for (int r = 0; r < B2; ++r)
            ss[(q1 * B2 + r) * M1 + k] = z[fft::bitrev(r, fft::ilog2(B2))];
    }
}

// 2b. Zo[t][k] = sum_q1 W_RC^{-q1 t} S[q1][t mod B2][k]
template <class Cf>
__device__ __forceinline__ void c_col_combine(const float2 *ss, float2 *zo, Tw tw) {
    constexpr int N0 = Cf::N0, RC = Cf::RC, M1 = Cf::M1, A = Cf::A, B2 = Cf::B2, ZS = Cf::ZS;
    constexpr int kRcStep = N0 / RC;
    for (int e = threadIdx.x; e < RC * M1; e += kNT) {
        const int t = e / M1, k = e % M1;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q1 = 0; q1 < A; ++q1) {
            const float2 wv = tw.t0[(q1 * t * kRcStep) & (N0 - 1)];
            cmac(acc, ss[(q1 * B2 + (t % B2)) * M1 + k], make_float2(wv.x, -wv.y));
        }
        zo[t * ZS + k] = acc;
    }
}

// 3. rows: y[t][n1 + P n2] = s Re sum_k c_k W_N1^{-k n1} Zo[t][k] W_Q^{-k n2}, stored to
//    rows c + C t of the image at dst
template <class Cf, typename T>
__device__ __forceinline__ void c_row_store(const float2 *zo, T *__restrict__ dst, int c, Tw tw) {
    constexpr int N1 = Cf::N1, RC = Cf::RC, C = Cf::C, P = Cf::P, Q = Cf::Q;
    constexpr int M1 = Cf::M1, ZS = Cf::ZS;
    for (int pr = threadIdx.x; pr < Cf::PAIRS; pr += kNT) {
        const int t = pr / P, n1 = pr % P, t2 = t + RC / 2;
        const float2 *twl = tw.t1i + n1 * Cf::TS;
        // z[q] = Herm(ga)[q] + i Herm(gb)[q], accumulated directly: a bin k
        // (q = k mod Q) with va = c_k W^{-k n1} Zo[t][k], vb likewise for row t2,
        // adds (va + i vb)/2 at q and (conj va + i conj vb)/2 at Q - q; the
        // table entry carries c_k/2 and the output scale
        float2 z[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) z[q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < M1; ++k) {
            const float2 w = twl[k];
            const float2 va = cmulc(zo[t * ZS + k], w);
            const float2 vb = cmulc(zo[t2 * ZS + k], w);
            const int q = k % Q, qm = (Q - q) % Q;
            z[q].x += va.x - vb.y;
            z[q].y += va.y + vb.x;
            z[qm].x += va.x + vb.y;
            z[qm].y += vb.x - va.y;
        }
        fft::fft_dif<Q, 1>(z);
        T *ra = dst + (size_t)(c + C * t) * N1 + n1;
        T *rb = dst + (size_t)(c + C * t2) * N1 + n1;
#pragma unroll
        for (int n2 = 0; n2 < Q; ++n2) {
            const float2 v = z[fft::bitrev(n2, fft::ilog2(Q))];
            Io<T>::store(ra + P * n2, v.x);
            Io<T>::store(rb + P * n2, v.y);
        }
    }
}

template <class Cf, typename T>
__device__ void phase_c(const float2 *__restrict__ Y, T *__restrict__ y, int img, int c,
                        char *smem, Tw tw) {
    constexpr int N0 = Cf::N0, N1 = Cf::N1, RC = Cf::RC, M1 = Cf::M1, A = Cf::A, B2 = Cf::B2;
    constexpr int NK = Cf::NK;
    float2 *ys = reinterpret_cast<float2 *>(smem);           // [K0][M1]
    float2 *vs = ys + NK;                                    // [RC][M1] residue-ordered
    float2 *ss = vs + RC * M1;                               // [A][B2][M1]
    float2 *zo = ss + A * B2 * M1;                           // [RC][ZS]
    const int tid = threadIdx.x;
    const float2 *src = Y + (size_t)img * NK;

    // 1. the image's kept modes, all copies in flight at once
    for (int e = tid; e < NK / 2; e += kNT) cp_async16(ys + 2 * e, src + 2 * e);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    c_residues<Cf>(ys, vs, c, tw);
    __syncthreads();
    c_col_ifft<Cf>(vs, ss);
    __syncthreads();
    c_col_combine<Cf>(ss, zo, tw);
    __syncthreads();
    c_row_store<Cf, T>(zo, y + (size_t)img * N0 * N1, c, tw);
}

__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Arguments of the fused kernels (one struct for all variants; a kernel reads
// the fields it needs).
struct Args {
    const void *x;
    const void *w;
    void *y;
    float2 *part;       // [C][B*Cin][NK]
    float2 *Y;          // [B*Cout][NK]
    SyncBlock *sync;
    const float2 *tw0;  // N0 twiddles
    const float2 *tw1;  // N1 twiddles
    const float2 *tw2;  // N2 twiddles (3-D layer)
    int *err;
    fno_trace_record_t *trace;   // nullptr unless FNO_PLAN_TRACE
    size_t wbytes;               // weight tensor bytes
    unsigned wslice;             // bytes of it each phase-A item prefetches into L2
    int batch, cin, cout;
    int bg, ng;         // batch rows per group, groups
    int npairs;         // phase B: kept-mode pairs
    int ob, nob;        // phase B: outputs per item, output blocks
    int trace_b, trace_c;   // three-kernel variants: first trace record of kernel B, C
    int wpacked;            // w is in the packed mode-major layout
    int mix16;              // 16-bit layer mixing on the tensor cores: the kept modes
                            // leave kernel A as per-mode 16-bit operand images (mix16_x)
                            // and the mixed modes leave kernel B as 16-bit pairs
};

__device__ __forceinline__ unsigned long long trace_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Three-kernel variants: one trace record per CTA, written once every thread of
// the CTA is done (t_start: entry, t_ready: the wait for the previous kernel
// returned).  A no-op unless the plan traces.
// cta_record_at: the same for work item `idx` of a CTA that runs several.
__device__ __forceinline__ void cta_record_at(const Args &a, int phase, int first, int idx,
                                              unsigned long long t_start,
                                              unsigned long long t_ready,
                                              unsigned long long t_compute = 0) {
    if (!a.trace) return;
    __syncthreads();
    if (threadIdx.x != 0) return;
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    fno_trace_record_t r;
    r.item = ((unsigned)phase << 24) | ((unsigned)idx & 0xFFFFFFu);
    r.worker = smid;
    r.t_start = t_start;
    r.t_ready = t_ready;
    r.t_end = trace_now();
    r.t_compute = t_compute ? t_compute : r.t_end;
    a.trace[first + idx] = r;
}
__device__ __forceinline__ void cta_record(const Args &a, int phase, int first,
                                           unsigned long long t_start,
                                           unsigned long long t_ready,
                                           unsigned long long t_compute = 0) {
    cta_record_at(a, phase, first, (int)blockIdx.x, t_start, t_ready, t_compute);
}

// item = (pair * nob + output block) * batch blocks + batch block; a.bg = batch
// rows per block, a.ng = batch blocks
__device__ __forceinline__ BItem b_item(const Args &a, int it) {
    const int bblk = it % a.ng;
    it /= a.ng;
    BItem bi;
    bi.pair = it / a.nob;
    bi.o0 = (it % a.nob) * a.ob;
    bi.nob = min(a.ob, a.cout - bi.o0);
    bi.b0 = bblk * a.bg;
    bi.nbb = min(a.bg, a.batch - bi.b0);
    return bi;
}

// Mixing that streams the weights: one CTA per run of R adjacent kept modes
// (one line of the last axis), every output channel and batch row.  The run's
// kept modes X[b][i][r] (summed over the partial copies) go to shared memory;
// thread (o, r-pair) then walks the input channels, reading two modes of
// W[blk][i][o][local + r] per load straight from global memory (a warp reads
// 64 / R runs of R x 8 contiguous bytes) and accumulating Y[b][o][r..r+1]
// for the kMaxB batch rows in registers.
// Each weight is read once and used for every batch row with no shared-memory
// staging; for small batches this is the weight stream's own bound.
constexpr int kMixThreads = 256;
// CTAs of the streaming mixing resident per SM with up to 4 batch rows (its
// register bound; two with more rows, whose accumulators need the registers):
// a CTA is a short chain of dependent loads, so the more of them are in flight
// the better the latency is hidden (its registers alone allowed three)
#ifndef FNO_MIX_STREAM_MINB
#define FNO_MIX_STREAM_MINB 4
#endif
#ifndef FNO_MIX_STREAM_DEPTH
#define FNO_MIX_STREAM_DEPTH 8
#endif
template <class Cf, typename T, int kParts, int R, int kMaxB>
__global__ void __launch_bounds__(kMixThreads, kMaxB <= 4 ? FNO_MIX_STREAM_MINB : 2) k_mix_stream(Args a) {
    extern __shared__ __align__(16) char smem[];
    float2 *xs = reinterpret_cast<float2 *>(smem);          // [batch][cin][R]
    static_assert(Cf::MR % R == 0, "a run stays on one line of the last axis");
    const int tid = threadIdx.x;
    const int mode0 = blockIdx.x * R;
    int blk, local;
    Cf::wmap(mode0, blk, local);
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    pdl_trigger();
    pdl_wait();                                  // kernel A's kept modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    constexpr int NK = Cf::NK;
    const int nimg = a.batch * a.cin;
    for (int e = tid; e < nimg * R; e += kMixThreads) {
        const int r = e % R, row = e / R;
        float2 acc = __ldcg(a.part + (size_t)row * NK + mode0 + r);
#pragma unroll
        for (int p = 1; p < kParts; ++p) {
            const float2 v = __ldcg(a.part + ((size_t)p * nimg + row) * NK + mode0 + r);
            acc.x += v.x;
            acc.y += v.y;
        }
        xs[e] = acc;
    }
    __syncthreads();
    const T *w = static_cast<const T *>(a.w);
    const size_t istride = (size_t)a.cout * Cf::MBLK * 2;    // next input channel (elements)
    // thread (o, rp): modes r = 2 rp and 2 rp + 1 of the run, one 2-mode load a weight
    static_assert(R % 2 == 0, "mode pairs");
    constexpr int RP = R / 2;
    for (int e = tid; e < a.cout * RP; e += kMixThreads) {
        const int r = 2 * (e % RP), o = e / RP;
        float2 acc0[kMaxB], acc1[kMaxB];
#pragma unroll
        for (int b = 0; b < kMaxB; ++b) acc0[b] = acc1[b] = make_float2(0.f, 0.f);
        const T *wp = w + ((((size_t)blk * a.cin) * a.cout + o) * Cf::MBLK + local + r) * 2;
        // kWv weight pairs in flight before the first product
        constexpr int kWv = FNO_MIX_STREAM_DEPTH;
        for (int i0 = 0; i0 < a.cin; i0 += kWv) {
            float4 wv[kWv];
#pragma unroll
            for (int q = 0; q < kWv; ++q) {
                const int i = i0 + q;
                wv[q] = i < a.cin ? Storage<T>::load4(
                                        a.wpacked ? w + packed_index(mode0 + r, i, o, a.cin,
                                                                     a.cout) * 2
                                                  : wp + (size_t)i * istride)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kWv; ++q) {
                const int i = i0 + q;
                if (i >= a.cin) break;
                const float2 w0 = make_float2(wv[q].x, wv[q].y), w1 = make_float2(wv[q].z, wv[q].w);
#pragma unroll
                for (int b = 0; b < kMaxB; ++b) {
                    if (b < a.batch) {
                        const float4 x2 = *reinterpret_cast<const float4 *>(
                            &xs[(b * a.cin + i) * R + r]);
                        cmac(acc0[b], make_float2(x2.x, x2.y), w0);
                        cmac(acc1[b], make_float2(x2.z, x2.w), w1);
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kMaxB; ++b)
            if (b < a.batch)
                __stcg(reinterpret_cast<float4 *>(a.Y + ((size_t)b * a.cout + o) * NK + mode0 + r),
                       make_float4(acc0[b].x, acc0[b].y, acc1[b].x, acc1[b].y));
    }
    cta_record(a, 1, a.trace_b, t0, t1);
}

template <class Cf, typename T, int kParts, int kNTB>
__global__ void __launch_bounds__(kNTB) k_phase_b(Args a) {
    extern __shared__ __align__(16) char smem[];
    const BItem bi = b_item(a, blockIdx.x);
    const CtaGroup grp{(int)threadIdx.x};
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    // weight slab rows padded by one entry: the lanes of a warp read S input
    // channels of one output pair, which an unpadded row stride would put on
    // the same banks
    const int wstride = a.ob + 1;
    phase_b_weights<Cf, T, kNTB>(grp, static_cast<const T *>(a.w), a.cin, a.cout, bi, wstride,
                                 smem, a.wpacked != 0);
    pdl_trigger();
    pdl_wait();                                  // kernel A's partial modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    unsigned long long tl = 0;
    phase_b<Cf, T, kNTB, CtaGroup, kParts>(grp, a.part, a.Y, a.cin, a.cout, a.batch * a.cin, bi,
                                          wstride, smem, a.trace ? &tl : nullptr);
    cta_record(a, 1, a.trace_b, t0, t1, tl);
}

}  // namespace
}  // namespace fno
