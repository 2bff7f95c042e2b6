// fno_fused3d.cu -- the 3-D spectral-convolution layer (a volume N0 x N1 x N2,
// 2*M0 x 2*M1 x M2 kept modes in four corner blocks) as three kernels chained
// by programmatic dependent launch, the steps of the TurboFNO article
// (gsyq.cn/news/457482) §2.1-§2.3 with the volume's intermediates kept in
// registers, shared memory and L2.
//
//   kernel A  (volume, chunk c), the C0 chunk-CTAs of a volume form a cluster.
//     A CTA takes the planes i0 = c + C0 t (t < R0 = N0 / C0) of one input
//     volume one after another through a cp.async ring of shared-memory
//     stages.  Each plane gets the truncated 2-D transform of the 2-D kernels
//     (row DFT over the last axis keeping M2 bins, column DFT over axis 1
//     keeping 2*M1 rows, with the whole plane as one chunk), and its kept
//     modes are folded into an R0-point DFT over t held in registers:
//         P_c[r] = sum_t S(c + C0 t) W_R0^{r t}.
//     Since W_N0^{f (c + C0 t)} = W_N0^{f c} W_R0^{f t}, the axis-0 transform
//     of the volume is X[f] = sum_c W_N0^{f c} P_c[f mod R0] (one decimation-
//     in-time step); the cluster's CTAs evaluate it through distributed shared
//     memory, each for one C0-th of the plane modes, and write X once.
//   kernel B  the per-mode channel mixing.  For batches up to 16 (few rows per
//     weight) the weight-streaming kernel: one CTA per run of 8 modes of a
//     last-axis line, thread (o, r) reading W straight from global memory for
//     every batch row; otherwise the slab kernel shared with the 2-D layers.
//   kernel C  (volume, chunk c).  Z_c[r] = sum_{f = r mod R0} Y[f] conj(W_N0^{f c});
//     an R0-point inverse DFT over r gives the 2-D spectra of the planes
//     c + C0 t, and each plane's inverse (column transform back to N1 rows,
//     then the half-spectrum row transform with c(0) = 1, c(k) = 2 and the
//     1/(N0 N1 N2) scale) is stored.
#include "fno_fused_dev.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

// Kernel A's plane ring depth and its CTAs per SM: two stages and a 128-register
// bound fit four CTAs on an SM (measured 20.1 k -> 22.0 k samples/s on the
// 4 x 32-channel 64^3 layer against three stages at three CTAs)
#ifndef FNO_RING_STAGES
#define FNO_RING_STAGES 2
#endif
#ifndef FNO_A3_MIN_BLOCKS
#define FNO_A3_MIN_BLOCKS 4
#endif
template <int N0_, int N1_, int N2_, int M0_, int M1_, int M2_, int C0_, int Q_, int B2_>
struct Cfg3 {
    static constexpr int N0 = N0_, N1 = N1_, N2 = N2_, M0 = M0_, M1 = M1_, M2 = M2_;
    static constexpr int C0 = C0_;                 // chunk-CTAs per volume (one cluster)
    static constexpr int R0 = N0 / C0;             // planes per chunk: i0 = c + C0 t
    static constexpr int K0 = 2 * M0;              // kept rows on axis 0
    using Pl = Cfg<N1, N2, M1, M2, N1, Q_, B2_>;   // one plane as a single chunk
    static constexpr int NKP = Pl::NK;             // kept modes per plane, [2 M1][M2]
    static constexpr int NK = K0 * NKP;            // kept modes per volume, [2 M0][2 M1][M2]
    static constexpr int QT = NKP / kNT;           // plane modes per thread
    static constexpr int KR = K0 / R0;             // kept rows per residue mod R0
    static constexpr int kCols = NKP / C0;         // plane modes each CTA reduces
    static constexpr int kStages = FNO_RING_STAGES;   // plane ring depth
    static_assert(N0 % C0 == 0 && M0 % R0 == 0, "kept rows j0 = r + R0 m share residue r");
    static_assert(NKP % kNT == 0 && NKP % C0 == 0 && (R0 * kCols) % kNT == 0, "tiling");
    static_assert(C0 >= 2 && C0 <= 8, "portable cluster");
    static_assert(M2 % kG == 0, "mode pairs stay in one kept row");
    static_assert(Pl::C == 1, "the plane transform covers the whole plane");

    // weights: block b = h0 + 2 h1 (h_a = 1 for the high kept rows on axis a),
    // each M0 x M1 x M2 modes
    static constexpr size_t MBLK = (size_t)M0 * M1 * M2;
    static constexpr int MR = M2;                  // kept modes along one line of the last axis
    __device__ static void wmap(int o, int &blk, int &local) {
        const int j0 = o / NKP, rest = o % NKP;
        const int j1 = rest / M2, k = rest % M2;
        const int h0 = j0 >= M0 ? 1 : 0, h1 = j1 >= M1 ? 1 : 0;
        blk = h0 | (h1 << 1);
        local = ((j0 - h0 * M0) * M1 + (j1 - h1 * M1)) * M2 + k;
    }

    // shared memory: twiddles W_N1 [N1], the row tables [2][P][TS], W_N0 [N0]
    static constexpr size_t kSmemTw = ((N1 + 2 * Pl::P * Pl::TS + N0) * 8 + 15) / 16 * 16;
    template <typename T>
    static constexpr size_t stage_bytes() {
        return (size_t)N1 * Pl::template xs_of<T>() * sizeof(T);
    }
    template <typename T>
    static constexpr size_t ring_bytes() {
        // the ring also holds the chunk's residues [R0][NKP] at the end
        return kStages * stage_bytes<T>() > (size_t)R0 * NKP * 8 ? kStages * stage_bytes<T>()
                                                                : (size_t)R0 * NKP * 8;
    }
    template <typename T>
    static constexpr size_t smem_a() { return kSmemTw + ring_bytes<T>() + (size_t)N1 * Pl::ZS * 8; }
    // kernel C: twiddles, the chunk's plane spectra [R0][NKP] and one plane's
    // spectral rows [N1][ZS]
    static constexpr size_t kSmemC = kSmemTw + (size_t)R0 * NKP * 8 + (size_t)N1 * Pl::ZS * 8;
    // kernel C reads the volume's mixed modes kYRows kept rows at a time, two
    // stages over the spectra region
    static constexpr int kYRows = 4;
    static_assert(K0 % kYRows == 0 && 2 * kYRows <= R0 && (kYRows * NKP) % 2 == 0,
                  "two stages of kept rows fit over the spectra");
    static_assert(stage_bytes<float>() % 16 == 0 && stage_bytes<__half>() % 16 == 0, "align");
    static_assert((size_t)Pl::A * Pl::B2 * M2 * 8 <= stage_bytes<__half>(),
                  "the column pass works in the stage of its plane");
};

using Cfg3d64 = Cfg3<64, 64, 64, 16, 16, 16, 8, 16, 8>;

// Twiddles of the 3-D layer into shared memory: the plane transform's tables
// (W_N1 for axis 1, W_N2^{n1 k} per row lane) and W_N0 for axis 0.
template <class C3>
__device__ __forceinline__ Tw load_tw3(const Args &a, char *smem, const float2 **twa) {
    using Pl = typename C3::Pl;
    float2 *t0 = reinterpret_cast<float2 *>(smem);
    float2 *t1 = t0 + C3::N1;
    float2 *t1i = t1 + Pl::P * Pl::TS;
    float2 *ta = t1i + Pl::P * Pl::TS;
    for (int e = threadIdx.x; e < C3::N1; e += kNT) t0[e] = a.tw1[e];
    fill_row_tables<Pl>(a.tw2, t1, t1i,
                        1.0f / ((float)C3::N0 * (float)C3::N1 * (float)C3::N2));
    for (int e = threadIdx.x; e < C3::N0; e += kNT) ta[e] = a.tw0[e];
    *twa = ta;
    return Tw{t0, t1, t1i};
}

// Column inverse of one plane into its spectral rows.  Kept row j holds the
// signed frequency g = j (j < M0) or j - 2 M0; with g = g1 + 8 g2 and, for a
// 64-row plane, t = t1 + 8 t2,
//   Zo[t][k] = sum_g1 e^{+2 pi i g1 t2 / 8} sum_g2 Y[g][k] e^{+2 pi i g t1 / N0},
// 2 M0 / 8 terms in each inner sum and an 8-point inverse register FFT over g1;
// thread (t1, k) owns the eight rows t1 + 8 t2 of bin k.
template <class Pl>
__device__ __forceinline__ void plane_col_inverse(const float2 *ys, float2 *zo, Tw tw) {
    constexpr int N0 = Pl::N0, M0 = Pl::M0, M1 = Pl::M1, K0 = Pl::K0, ZS = Pl::ZS;
    constexpr int G1 = 8, T1 = N0 / G1, G2 = M0 / G1;   // g2 = -G2 .. G2 - 1
    static_assert(M0 % G1 == 0 && T1 == G1, "8 x 8 split of the plane's rows");
    for (int u = threadIdx.x; u < T1 * M1; u += kNT) {
        const int k = u % M1, t1 = u / M1;
        float2 z[G1];
#pragma unroll
        for (int g1 = 0; g1 < G1; ++g1) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int g2 = -G2; g2 < G2; ++g2) {
                const int g = g1 + G1 * g2, j = g < 0 ? g + K0 : g;
                const float2 wv = tw.t0[(g * t1) & (N0 - 1)];     // e^{-2 pi i g t1 / N0}
                cmac(acc, ys[j * M1 + k], make_float2(wv.x, -wv.y));
            }
            z[g1] = acc;
        }
        fft::fft_dif<G1, 1>(z);
#pragma unroll
        for (int t2 = 0; t2 < G1; ++t2)
            zo[(t1 + T1 * t2) * ZS + k] = z[fft::bitrev(t2, fft::ilog2(G1))];
    }
}

// The kept modes of a 64-row plane from the column pass's 8-point sums
// S[t1][q][k] = sum_t2 Z[t1 + 8 t2][k] W_8^{q t2} (ss, a_col_fft's output):
// with the frequency f = q + 8 f2,
//   X[f][k] = sum_t1 W_8^{f2 t1} (W_64^{q t1} S[t1][q][k]),
// an 8-point FFT over t1 per (q, k) after the twiddle, of whose outputs the
// kept rows need f2 = 0, 1 (f = q, q + 8) and 6, 7 (f = q - 16, q - 8).
// Thread (q, k) = (tid / 16, tid % 16) so leaves exactly the modes
// o = tid + 128 m (kept row j = q + 8 m) that it folds: m = 0..3 <-> f2 = 0,
// 1, 6, 7 -- the same sums as a_kept_mode for these four modes, in
// 8 + 8 loads and one FFT instead of 4 x 16 loads and 32 products.
template <class Pl>
__device__ __forceinline__ void plane_kept_modes(const float2 *ss, Tw tw, float2 (&v)[4]) {
    constexpr int N = Pl::N0, M1 = Pl::M1, A = Pl::A, B2 = Pl::B2;
    static_assert(N == 64 && A == 8 && B2 == 8 && Pl::K0 == 32 && Pl::M0 == 16 && M1 * A == kNT,
                  "64-row plane, 32 kept rows, one (q, k) unit per thread");
    const int q = threadIdx.x / M1, k = threadIdx.x % M1;
    float2 u[A];
#pragma unroll
    for (int t1 = 0; t1 < A; ++t1)
        u[t1] = cmul(ss[(t1 * B2 + q) * M1 + k], tw.t0[(q * t1) & (N - 1)]);   // W_64^{q t1}
    fft::fft_dif<A, -1>(u);                      // output f2 at u[bitrev(f2)]
    constexpr int lg = fft::ilog2(A);
    v[0] = u[fft::bitrev(0, lg)];
    v[1] = u[fft::bitrev(1, lg)];
    v[2] = u[fft::bitrev(6, lg)];
    v[3] = u[fft::bitrev(7, lg)];
}

// acc += v W_8^m, W_8 = e^{-2 pi i / 8}, for a compile-time m: the even
// powers are 1, -i, -1, +i (adds and swaps); the odd ones (+-1 +- i) / sqrt 2
// share s = (v.x + v.y) / sqrt 2 and d = (v.y - v.x) / sqrt 2
template <int M>
__device__ __forceinline__ void cmac_w8(float2 &acc, float2 v, float s, float d) {
    constexpr int m = M & 7;
    if constexpr (m == 0) { acc.x += v.x; acc.y += v.y; }
    else if constexpr (m == 2) { acc.x += v.y; acc.y -= v.x; }
    else if constexpr (m == 4) { acc.x -= v.x; acc.y -= v.y; }
    else if constexpr (m == 6) { acc.x -= v.y; acc.y += v.x; }
    else if constexpr (m == 1) { acc.x += s; acc.y += d; }
    else if constexpr (m == 3) { acc.x += d; acc.y -= s; }
    else if constexpr (m == 5) { acc.x -= s; acc.y -= d; }
    else { acc.x -= d; acc.y += s; }
}
// the fold of plane t's kept modes into the eight residues, P[r] += v W_8^{r t}
template <int T, int QT>
__device__ __forceinline__ void fold_w8(float2 (&acc)[8][QT], const float2 (&v)[QT]) {
    constexpr float c = 0.70710678118654752f;
#pragma unroll
    for (int q = 0; q < QT; ++q) {
        const float s = c * (v[q].x + v[q].y), d = c * (v[q].y - v[q].x);
        fft::unroll<0, 8>([&](auto ri) {
            constexpr int r = decltype(ri)::value;
            cmac_w8<r * T>(acc[r][q], v[q], s, d);
        });
    }
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float2 ld_dsmem(uint32_t local, int rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v.x), "=f"(v.y) : "r"(remote) : "memory");
    return v;
}

// Frequency of kept row j on axis 0.
template <class C3>
__device__ __forceinline__ int freq0(int j) {
    return j < C3::M0 ? j : C3::N0 - C3::K0 + j;
}

// grid: volumes x C0 CTAs, clusters of C0 along x (cluster rank = blockIdx.x % C0)
template <class C3, typename T>
__global__ void __launch_bounds__(kNT, FNO_A3_MIN_BLOCKS) k_phase_a3(Args a) {
    using Pl = typename C3::Pl;
    constexpr int N0 = C3::N0, N1 = C3::N1, N2 = C3::N2, C0 = C3::C0, R0 = C3::R0;
    constexpr int NKP = C3::NKP, QT = C3::QT, S = C3::kStages;
    constexpr size_t kStage = C3::template stage_bytes<T>();
    extern __shared__ __align__(16) char smem[];
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const float2 *twa;
    const Tw tw = load_tw3<C3>(a, smem, &twa);
    char *ring = smem + C3::kSmemTw;
    float2 *zs = reinterpret_cast<float2 *>(ring + C3::template ring_bytes<T>());   // [N1][ZS]
    const int vol = blockIdx.x / C0, c = blockIdx.x % C0;
    const T *src = static_cast<const T *>(a.x) + (size_t)vol * N0 * N1 * N2;
    pdl_trigger();                               // kernel B may start fetching weights

    // plane c + C0 t into stage t % S, rows padded to xs_of<T>() samples
    auto issue = [&](int t) {
        T *dst = reinterpret_cast<T *>(ring + (t % S) * kStage);
        const T *p = src + (size_t)(c + C0 * t) * N1 * N2;
        constexpr int kPer = 16 / (int)sizeof(T);
        constexpr int kRow = N2 / kPer;
        for (int e = threadIdx.x; e < N1 * kRow; e += kNT) {
            const int row = e / kRow, s = e % kRow;
            cp_async16(dst + row * Pl::template xs_of<T>() + s * kPer,
                       p + (size_t)row * N2 + s * kPer);
        }
    };
#pragma unroll
    for (int t = 0; t < S - 1; ++t) {
        if (t < R0) issue(t);
        cp_async_commit();
    }
    float2 acc[R0][QT];
#pragma unroll
    for (int r = 0; r < R0; ++r)
#pragma unroll
        for (int q = 0; q < QT; ++q) acc[r][q] = make_float2(0.f, 0.f);

    for (int t = 0; t < R0; ++t) {
        // the stage refilled here held plane t - 1, released by the barrier that
        // ended the previous iteration
        if (t + S - 1 < R0) issue(t + S - 1);
        cp_async_commit();
        asm volatile("cp.async.wait_group %0;" ::"n"(S - 1) : "memory");
        __syncthreads();                         // plane t is in its stage
        const T *xs = reinterpret_cast<const T *>(ring + (t % S) * kStage);
        a_row_dft<Pl, T, Pl::template xs_of<T>()>(xs, zs, tw);
        __syncthreads();
        float2 *ss = reinterpret_cast<float2 *>(ring + (t % S) * kStage);   // plane t consumed
        a_col_fft<Pl>(zs, ss);
        __syncthreads();
        float2 v[QT];
        plane_kept_modes<Pl>(ss, tw, v);
        // P_c[r] += v W_R0^{r t}: with t known at compile time in each case the
        // multipliers are the eighth roots of unity, applied as adds
        static_assert(R0 == 8, "the fold's cases are the planes t < 8");
        switch (t) {
            case 0: fold_w8<0>(acc, v); break;
            case 1: fold_w8<1>(acc, v); break;
            case 2: fold_w8<2>(acc, v); break;
            case 3: fold_w8<3>(acc, v); break;
            case 4: fold_w8<4>(acc, v); break;
            case 5: fold_w8<5>(acc, v); break;
            case 6: fold_w8<6>(acc, v); break;
            default: fold_w8<7>(acc, v); break;
        }
        __syncthreads();
    }
    const unsigned long long t_planes = a.trace ? trace_now() : 0;

    // residues to shared memory (over the ring), then the cluster's combine
    float2 *pm = reinterpret_cast<float2 *>(ring);   // [R0][NKP]
#pragma unroll
    for (int r = 0; r < R0; ++r)
#pragma unroll
        for (int q = 0; q < QT; ++q) pm[r * NKP + threadIdx.x + q * kNT] = acc[r][q];
    cluster_sync();
    const uint32_t local = smem_addr(pm);
    float2 *X = a.part + (size_t)vol * C3::NK;
    // X[f] = sum_cc W_64^{f cc} P_cc[r] for the kept rows of residue r: with
    // f = r + 8 f2 an 8-point FFT over cc after the twiddle W_64^{r cc}, whose
    // outputs f2 = 0, 1, 6, 7 are the kept rows r, r + 8, r + 16, r + 24
    static_assert(C0 == 8 && R0 == 8 && C3::KR == 4 && N0 == 64 && C3::M0 == 16,
                  "64 planes, 8 chunks, 32 kept rows");
    for (int u = threadIdx.x; u < R0 * C3::kCols; u += kNT) {
        const int r = u / C3::kCols, col = c * C3::kCols + u % C3::kCols;
        float2 v[C0];
#pragma unroll
        for (int cc = 0; cc < C0; ++cc)
            v[cc] = cmul(ld_dsmem(local + (uint32_t)(r * NKP + col) * 8, cc),
                         twa[(r * cc) & (N0 - 1)]);
        fft::fft_dif<C0, -1>(v);                 // output f2 at v[bitrev(f2)]
        constexpr int lg = fft::ilog2(C0);
        constexpr int kF2[4] = {0, 1, 6, 7};
#pragma unroll
        for (int m = 0; m < C3::KR; ++m)
            __stcg(X + (size_t)(r + R0 * m) * NKP + col, v[fft::bitrev(kF2[m], lg)]);
    }
    cluster_sync();                              // peers may still read this CTA's residues
    cta_record(a, 0, 0, t0, t0, t_planes);       // compute: the planes, tail: the combine
}

// grid: volumes x C0 CTAs
template <class C3, typename T>
__global__ void __launch_bounds__(kNT) k_phase_c3(Args a) {
    using Pl = typename C3::Pl;
    constexpr int N0 = C3::N0, N1 = C3::N1, N2 = C3::N2, C0 = C3::C0, R0 = C3::R0;
    constexpr int NKP = C3::NKP, QT = C3::QT, M2 = C3::M2;
    extern __shared__ __align__(16) char smem[];
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const float2 *twa;
    const Tw tw = load_tw3<C3>(a, smem, &twa);
    float2 *spec = reinterpret_cast<float2 *>(smem + C3::kSmemTw);   // [R0][NKP]
    float2 *zo = spec + R0 * NKP;                                    // [N1][ZS]
    __syncthreads();
    pdl_wait();                                  // kernel B's mixed modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    const int vol = blockIdx.x / C0, c = blockIdx.x % C0;
    const float2 *Yv = a.Y + (size_t)vol * C3::NK;

    // 1. Z[r] = sum_m Y[r + R0 m] conj(W_N0^{f c}) for this thread's plane modes,
    //    then the R0-point inverse DFT over r: spectra of planes c + C0 t.  The
    //    volume's kept rows come through two cp.async stages of kRows rows over
    //    the spectra region, so that the reads of a stage overlap the sums of
    //    the one before.
    constexpr int kRows = C3::kYRows, kNSt = C3::K0 / kRows;
    auto issue_y = [&](int st) {
        float2 *d = spec + (st & 1) * kRows * NKP;
        const float2 *g = Yv + (size_t)st * kRows * NKP;
        for (int e = threadIdx.x; e < kRows * NKP / 2; e += kNT) cp_async16(d + 2 * e, g + 2 * e);
    };
    issue_y(0);
    cp_async_commit();
    issue_y(1);
    cp_async_commit();
    float2 z[QT][R0];
#pragma unroll
    for (int r = 0; r < R0; ++r)
#pragma unroll
        for (int q = 0; q < QT; ++q) z[q][r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int st = 0; st < kNSt; ++st) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();                         // stage st is in its buffer
        const float2 *yb = spec + (st & 1) * kRows * NKP;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            const int j0 = st * kRows + rr;
            const float2 w = twa[(freq0<C3>(j0) * c) & (N0 - 1)];
            const float2 wc = make_float2(w.x, -w.y);
#pragma unroll
            for (int q = 0; q < QT; ++q)
                cmac(z[q][j0 % R0], yb[rr * NKP + threadIdx.x + q * kNT], wc);
        }
        __syncthreads();                         // its buffer is free again
        if (st + 2 < kNSt) issue_y(st + 2);
        cp_async_commit();
    }
#pragma unroll
    for (int q = 0; q < QT; ++q) {
        fft::fft_dif<R0, 1>(z[q]);
#pragma unroll
        for (int t = 0; t < R0; ++t)
            spec[t * NKP + threadIdx.x + q * kNT] = z[q][fft::bitrev(t, fft::ilog2(R0))];
    }
    __syncthreads();

    // 2. every plane of the chunk: column inverse, row inverse, store
    T *dst = static_cast<T *>(a.y) + (size_t)vol * N0 * N1 * N2;
    for (int t = 0; t < R0; ++t) {
        plane_col_inverse<Pl>(spec + t * NKP, zo, tw);
        __syncthreads();
        c_row_store<Pl, T>(zo, dst + (size_t)(c + C0 * t) * N1 * N2, 0, tw);
        __syncthreads();                         // zo is rewritten for the next plane
    }
    cta_record(a, 2, a.trace_c, t0, t1);
}

// ---------------------------------------------------------------------------
// Kernel A on the tensor cores (float32 storage): the row DFT of the planes
// (64 samples -> the 16 kept bins) is a 3xTF32 GEMM per pair of planes,
// D[(plane, t1)][j] = sum_n x[plane][t1][n] T[j][n] with T[j][n] = cos(2 pi k n
// / 64) (j = k < 16) or -sin (j = 16 + k): M = 128 rows (two planes), K = 64,
// in two passes as in the 2-D fp32 kernel, x [T_hi ; T_lo] (N = 64) then
// x_lo T_hi (N = 32, x_lo written over x).  TMA brings each plane's rows into
// the K-major 128-byte-swizzled operand directly (two stages of a plane pair);
// the column DFT, the kept modes and the fold into the chunk's residues over t
// stay on the SIMT cores as in k_phase_a3, and so does the cluster's axis-0
// combine.
struct Geo3A {
    static constexpr int N = 64, M2 = 16;
    static constexpr uint32_t kTile = 128u * 128u;      // one K chunk of a plane pair
    static constexpr uint32_t kPair = 2 * kTile;        // a plane pair (K = 64)
    static constexpr uint32_t kTChunk = 64u * 128u;     // [T_hi rows 0..31 | T_lo rows 0..31]
    static constexpr uint32_t kTBytes = 2 * kTChunk;
    static constexpr uint32_t kRing = 0;                // two plane-pair stages
    static constexpr uint32_t kT = kRing + 2 * kPair;
    static constexpr uint32_t kZ = kT + kTBytes;        // two planes' row spectra [N1][ZS]
    static constexpr uint32_t kTmemCols = 64;
};

template <class C3>
__global__ void __launch_bounds__(kNT, 2)
k_phase_a3_tc(const __grid_constant__ CUtensorMap xmap, Args a, const void *table) {
    using Pl = typename C3::Pl;
    using Gm = Geo3A;
    using namespace tcu;
    constexpr int N0 = C3::N0, N1 = C3::N1, C0 = C3::C0, R0 = C3::R0, NKP = C3::NKP, QT = C3::QT;
    constexpr int kPairs = R0 / 2;
    static_assert(N1 == Gm::N && C3::N2 == Gm::N && C3::M2 == Gm::M2 && R0 % 2 == 0, "64^3");
    static_assert(kNT == 128, "a warp per tensor-memory lane quarter");
    constexpr uint32_t kZBytes = (uint32_t)N1 * Pl::ZS * 8;
    constexpr uint32_t kSs = Gm::kZ + 2 * kZBytes;      // the column pass's sums
    constexpr uint32_t kTw = kSs + (uint32_t)Pl::A * Pl::B2 * Pl::M1 * 8;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_t, bar_x[2], bar_p1, bar_fin;
    __shared__ uint32_t s_tmem;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int vol = blockIdx.x / C0, c = blockIdx.x % C0;
    const float2 *twa;
    const Tw tw = load_tw3<C3>(a, base + kTw, &twa);
    // plane pair q (planes c + C0 (2q + p), p = 0, 1) into stage st: rows
    // p * 64 .. of each K chunk
    auto issue = [&](int q, int st) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(tc_smem_addr(&bar_x[st])), "r"(Gm::kPair) : "memory");
        for (int pl = 0; pl < 2; ++pl) {
            const int i0 = c + C0 * (2 * q + pl);
            const int row0 = (vol * N0 + i0) * N1;
            for (int kc = 0; kc < 2; ++kc)
                tma_load_2d(tc_smem_addr(base + Gm::kRing + st * Gm::kPair + kc * Gm::kTile +
                                         pl * (Gm::kTile / 2)),
                            &xmap, kc * 32, row0, &bar_x[st]);
        }
    };
    if (tid == 0) {
        const uint64_t *bars[5] = {&bar_t, &bar_x[0], &bar_x[1], &bar_p1, &bar_fin};
        for (const uint64_t *b : bars)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(b)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(tc_smem_addr(&bar_t)), "r"(Gm::kTBytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(tc_smem_addr(base + Gm::kT)), "l"(table), "r"(Gm::kTBytes),
                     "r"(tc_smem_addr(&bar_t)) : "memory");
        issue(0, 0);
        if (kPairs > 1) issue(1, 1);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(Gm::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    pdl_trigger();                               // kernel B may start fetching weights
    const uint32_t tmem = s_tmem;
    const uint32_t ts = tc_smem_addr(base + Gm::kT);
    float2 *ss = reinterpret_cast<float2 *>(base + kSs);
    bool ok = true;
    if (tid == 0) ok &= mbar_wait(&bar_t, 0, a.err);
    float2 acc[R0][QT];
#pragma unroll
    for (int r = 0; r < R0; ++r)
#pragma unroll
        for (int q = 0; q < QT; ++q) acc[r][q] = make_float2(0.f, 0.f);

    for (int q = 0; q < kPairs; ++q) {
        const int st = q & 1;
        char *stage = base + Gm::kRing + st * Gm::kPair;
        const uint32_t xs = tc_smem_addr(stage);
        // pass 1 (one thread): x [T_hi ; T_lo]^T into columns 0..63
        if (tid == 0) {
            ok &= mbar_wait(&bar_x[st], (uint32_t)(q >> 1), a.err);
            tc_after_sync();
            constexpr uint32_t id = idesc_tf32(64);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_tf32(tmem, desc_sw128(xs + kc * Gm::kTile + s4 * 32),
                             desc_sw128(ts + kc * Gm::kTChunk + s4 * 32), id, (kc | s4) ? 1u : 0u);
            mma_commit(&bar_p1);
        }
        ok &= mbar_wait(&bar_p1, (uint32_t)q, a.err);   // pass 1 has read the pair
        // x_lo over the pair (elementwise: the swizzled layout carries over)
        {
            float4 *xv = reinterpret_cast<float4 *>(stage);
            for (int e = tid; e < (int)(Gm::kPair / 16); e += kNT) {
                const float4 v = xv[e];
                xv[e] = make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
            }
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();
        // pass 2: x_lo T_hi^T into columns 0..31
        if (tid == 0) {
            tc_after_sync();
            constexpr uint32_t id = idesc_tf32(32);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_tf32(tmem, desc_sw128(xs + kc * Gm::kTile + s4 * 32),
                             desc_sw128(ts + kc * Gm::kTChunk + s4 * 32), id, 1u);
            mma_commit(&bar_fin);
        }
        ok &= mbar_wait(&bar_fin, (uint32_t)q, a.err);
        tc_after_sync();
        // the two planes' row spectra: lane r = (plane r / 64, row r % 64), warp
        // w reading lanes 32 w..; bins 8h .. 8h + 7 at a time (re = columns k
        // and 32 + k, im = 16 + k and 48 + k: the T_hi and T_lo halves summed)
        {
            const int r = 32 * warp + (tid & 31);
            const uint32_t la = tmem + ((uint32_t)(32 * warp) << 16);
            float2 *zs = reinterpret_cast<float2 *>(base + Gm::kZ + (r / 64) * kZBytes) +
                         (r % 64) * Pl::ZS;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float re0[8], re1[8], im0[8], im1[8];
                tmem_ld8(la + 8 * h, re0);           // cos of bins 8h .., T_hi
                tmem_ld8(la + 16 + 8 * h, im0);      // -sin, T_hi
                tmem_ld8(la + 32 + 8 * h, re1);      // cos, T_lo
                tmem_ld8(la + 48 + 8 * h, im1);      // -sin, T_lo
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    zs[8 * h + k] = ok ? make_float2(re0[k] + re1[k], im0[k] + im1[k])
                                       : make_float2(0.f, 0.f);
            }
        }
        tc_before_sync();
        __syncthreads();                         // the stage and tensor memory are free
        if (tid == 0 && q + 2 < kPairs) issue(q + 2, st);
        // each plane of the pair: column DFT, kept modes, fold into the residues
#pragma unroll
        for (int pl = 0; pl < 2; ++pl) {
            const int t = 2 * q + pl;
            const float2 *zs = reinterpret_cast<const float2 *>(base + Gm::kZ + pl * kZBytes);
            a_col_fft<Pl>(zs, ss);
            __syncthreads();
            float2 wr[R0];                       // W_R0^{r t} = W_N0^{C0 r t}
#pragma unroll
            for (int rr = 0; rr < R0; ++rr) wr[rr] = twa[(C0 * rr * t) & (N0 - 1)];
#pragma unroll
            for (int qq = 0; qq < QT; ++qq) {
                const float2 v = a_kept_mode<Pl>(ss, threadIdx.x + qq * kNT, 0, tw);
#pragma unroll
                for (int rr = 0; rr < R0; ++rr) cmac(acc[rr][qq], v, wr[rr]);
            }
            __syncthreads();                     // ss is rewritten by the next plane
        }
    }
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(Gm::kTmemCols));
    }
    // residues to shared memory (over the ring), then the cluster's combine
    float2 *pm = reinterpret_cast<float2 *>(base + Gm::kRing);   // [R0][NKP]
#pragma unroll
    for (int rr = 0; rr < R0; ++rr)
#pragma unroll
        for (int qq = 0; qq < QT; ++qq) pm[rr * NKP + threadIdx.x + qq * kNT] = acc[rr][qq];
    cluster_sync();
    const uint32_t local = smem_addr(pm);
    float2 *X = a.part + (size_t)vol * C3::NK;
    for (int u = threadIdx.x; u < R0 * C3::kCols; u += kNT) {
        const int rr = u / C3::kCols, col = c * C3::kCols + u % C3::kCols;
        float2 v[C0];
#pragma unroll
        for (int cc = 0; cc < C0; ++cc) v[cc] = ld_dsmem(local + (uint32_t)(rr * NKP + col) * 8, cc);
#pragma unroll
        for (int m = 0; m < C3::KR; ++m) {
            const int j0 = rr + R0 * m, f0 = freq0<C3>(j0);
            float2 sum = make_float2(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < C0; ++cc) cmac(sum, v[cc], twa[(f0 * cc) & (N0 - 1)]);
            __stcg(X + (size_t)j0 * NKP + col, sum);
        }
    }
    cluster_sync();                              // peers may still read this CTA's residues
    cta_record(a, 0, 0, t0, t0);
}

// shared memory of the tensor-core kernel A
template <class C3>
constexpr size_t smem_a3_tc() {
    using Pl = typename C3::Pl;
    return Geo3A::kZ + 2 * (size_t)C3::N1 * Pl::ZS * 8 + (size_t)Pl::A * Pl::B2 * Pl::M1 * 8 +
           C3::kSmemTw + 1024;
}

// ---------------------------------------------------------------------------
// Kernel C on the tensor cores (64^3 volumes, 16^3 modes per block): the row
// inverse of every plane, 16 kept bins -> 64 samples, is a 3xTF32 GEMM per
// plane computed transposed, y^T = T Zo'^T with Zo' = [Re Zo | Im Zo] (K = 32
// per row) and T[n] = s [c(k) cos(2 pi k n / 64) | -c(k) sin(...)], s =
// 1 / 64^3: M = 64 output samples, N = 64 rows, the three products
// concatenated along K, [T_hi | T_hi | T_lo] against [Zo'_hi | Zo'_lo | Zo'_hi]
// (K = 96).  Tensor-memory lane n then holds sample n of every row, so the 16
// lanes of a warp that carry data store 64 contiguous bytes of a row at a
// time.  Z_c (the sums over the volume's kept rows) and the 8-point inverse
// DFT over the residues stay in registers as in k_phase_c3; each plane's
// spectrum goes to shared memory just before its column inverse (SIMT), whose
// rows are written as the GEMM's operand.  Four CTAs of four warps per SM as
// for k_phase_c3: one operand buffer, two 64-column accumulators, a plane's
// MMAs running while the threads store the plane before and compute the next
// plane's column inverse.
struct Geo3C {
    static constexpr int N = 64, M1 = 16, K0 = 32;
    static constexpr uint32_t kRows64 = 64u * 128u;     // 64 rows x 32 fp32, swizzled
    static constexpr uint32_t kT = 0;                   // T_hi, T_lo
    static constexpr uint32_t kZ = kT + 2 * kRows64;    // Zo'_hi, Zo'_lo of a plane
    static constexpr uint32_t kSpec = kZ + 2 * kRows64; // one plane's spectrum [32][16]
    static constexpr uint32_t kTmemCols = 128;          // two plane accumulators
};

// tensor memory -> registers, shape .16x32bx2: threads 0..15 read lanes
// base .. base + 15 at columns col .. col + 15, threads 16..31 the same lanes
// at columns col + kOff ..
template <int kOff>
__device__ __forceinline__ void tmem_ld16x2(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                 "%11,%12,%13,%14,%15}, [%16], %17;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr), "n"(kOff));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <class C3>
constexpr size_t smem_c3_tc() {
    return Geo3C::kSpec + (size_t)C3::NKP * 8 + (size_t)(C3::N0 + C3::N1) * 8 + 1024;
}

// grid: volumes x C0 CTAs
template <class C3, typename T>
__global__ void __launch_bounds__(kNT, 4)
k_phase_c3_tc(Args a, const void *table) {
    using Gm = Geo3C;
    using namespace tcu;
    constexpr int NT = kNT;
    constexpr int N0 = C3::N0, N1 = C3::N1, N2 = C3::N2, C0 = C3::C0, R0 = C3::R0;
    constexpr int NKP = C3::NKP, M1 = C3::M2, QT = NKP / NT;   // M1: bins per kept row
    constexpr int G1 = 8, T1 = N1 / G1, G2 = C3::M1 / G1;      // column inverse: g = g1 + 8 g2
    static_assert(N1 == Gm::N && N2 == Gm::N && M1 == Gm::M1 && C3::M1 == Gm::M1 &&
                  2 * M1 == Gm::K0, "64^3 volumes, 16^3 modes per block");
    static_assert(NKP % NT == 0 && T1 * M1 == NT, "one column-inverse unit per thread");
    static_assert(2 * Gm::kRows64 >= (uint32_t)C3::kYRows * NKP * 8,
                  "a stage of kept rows fits over each pair of 64-row tiles");
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_t, bar_mma[2];
    __shared__ uint32_t s_tmem;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vol = blockIdx.x / C0, c = blockIdx.x % C0;
    float2 *ysp = reinterpret_cast<float2 *>(base + Gm::kSpec);            // [32][16]
    float2 *twa = ysp + NKP;                                                 // W_N0
    float2 *tw1 = twa + N0;                                                  // W_N1
    if (tid == 0) {
        const uint64_t *bars[3] = {&bar_t, &bar_mma[0], &bar_mma[1]};
        for (const uint64_t *b : bars)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(b)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(Gm::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    for (int e = tid; e < N0; e += NT) twa[e] = a.tw0[e];
    for (int e = tid; e < N1; e += NT) tw1[e] = a.tw1[e];
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    pdl_wait();                                  // kernel B's mixed modes are complete
    const unsigned long long t_ready = a.trace ? trace_now() : 0;
    const float2 *Yv = a.Y + (size_t)vol * C3::NK;

    // 1. Z[r] = sum_m Y[r + R0 m] conj(W_N0^{f c}) for this thread's plane modes,
    //    then the R0-point inverse DFT over r: spectra of planes c + C0 t, kept
    //    in registers.  The volume's kept rows come through two cp.async stages
    //    over the operand tiles (the T operand is fetched afterwards).
    constexpr int kRows = C3::kYRows, kNSt = C3::K0 / kRows;
    auto issue_y = [&](int st) {
        float2 *d = reinterpret_cast<float2 *>(base + (st & 1) * 2 * Gm::kRows64);
        const float2 *g = Yv + (size_t)st * kRows * NKP;
        for (int e = tid; e < kRows * NKP / 2; e += NT) cp_async16(d + 2 * e, g + 2 * e);
    };
    issue_y(0);
    cp_async_commit();
    issue_y(1);
    cp_async_commit();
    float2 z[QT][R0];
#pragma unroll
    for (int r = 0; r < R0; ++r)
#pragma unroll
        for (int q = 0; q < QT; ++q) z[q][r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int st = 0; st < kNSt; ++st) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();                         // stage st is in its buffer
        const float2 *yb = reinterpret_cast<const float2 *>(base + (st & 1) * 2 * Gm::kRows64);
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            const int j0 = st * kRows + rr;
            const float2 w = twa[(freq0<C3>(j0) * c) & (N0 - 1)];
            const float2 wc = make_float2(w.x, -w.y);
#pragma unroll
            for (int q = 0; q < QT; ++q) cmac(z[q][j0 % R0], yb[rr * NKP + tid + q * NT], wc);
        }
        __syncthreads();                         // its buffer is free again
        if (st + 2 < kNSt) issue_y(st + 2);
        cp_async_commit();
    }
#pragma unroll
    for (int q = 0; q < QT; ++q) fft::fft_dif<R0, 1>(z[q]);   // plane t at z[q][bitrev(t)]
    if (tid == 0) {                              // the T operand over the first stage
        fence_async_smem();
        arrive_expect_tx(&bar_t, 2 * Gm::kRows64);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(tc_smem_addr(base + Gm::kT)), "l"(table), "r"(2 * Gm::kRows64),
                     "r"(tc_smem_addr(&bar_t)) : "memory");
    }
    const unsigned long long t_spec = a.trace ? trace_now() : 0;
    bool ok = mbar_wait(&bar_t, 0, a.err);

    // 2. planes: spectrum -> column inverse (SIMT) -> Zo' operands -> MMAs -> rows out
    char *Zhi = base + Gm::kZ, *Zlo = Zhi + Gm::kRows64;
    const int k = tid % M1, t1 = tid / M1;       // this thread's column-inverse unit
    T *dst = static_cast<T *>(a.y) + (size_t)vol * N0 * N1 * N2;
    // plane t's rows from accumulator t & 1: with M = 64, sample n sits in lane
    // 32 (n / 16) + n % 16, so warp w reads samples 16 w .., lanes 0..15
    // carrying data
    // (the .16x32bx2 load: lanes 0..15 of the warp read the 16 data lanes at
    // rows 16 g .., lanes 16..31 the same lanes 32 rows further on, so every
    // lane stores and a warp's store covers two rows)
    auto drain = [&](int t) {
        const int i0 = c + C0 * t, n = 16 * warp + (lane & 15), h = lane >> 4;
        T *out = dst + (size_t)i0 * N1 * N2 + (size_t)(32 * h) * N2 + n;
        const uint32_t acc = tmem + (uint32_t)(64 * (t & 1)) + ((uint32_t)(32 * warp) << 16);
#pragma unroll
        for (int g = 0; g < N1 / 32; ++g) {
            float v[16];
            tmem_ld16x2<32>(acc + 16 * g, v);    // rows 16 g + 32 h + i
            if (!ok) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Io<T>::store(out + (size_t)(16 * g + i) * N2, v[i]);
        }
    };
#pragma unroll 1
    for (int t = 0; t < R0; ++t) {
        // the plane's spectrum from the registers (the buffer's previous plane
        // was read before the barrier that ended the last iteration)
        fft::unroll<0, R0>([&](auto ri) {
            constexpr int r = decltype(ri)::value;
            if (fft::bitrev(t, fft::ilog2(R0)) == r) {
#pragma unroll
                for (int q = 0; q < QT; ++q) ysp[tid + q * NT] = z[q][r];
            }
        });
        __syncthreads();
        // Zo[t1 + 8 t2][k] = sum_g1 e^{+2 pi i g1 t2 / 8} sum_g2 Y[g][k] e^{+2 pi i g t1 / 64}
        float2 zc[G1];
#pragma unroll
        for (int g1 = 0; g1 < G1; ++g1) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int g2 = -G2; g2 < G2; ++g2) {
                const int g = g1 + G1 * g2, j = g < 0 ? g + 2 * C3::M1 : g;   // kept row of g
                const float2 wv = tw1[(g * t1) & (N1 - 1)];   // e^{-2 pi i g t1 / 64}
                cmac(acc, ysp[j * M1 + k], make_float2(wv.x, -wv.y));
            }
            zc[g1] = acc;
        }
        fft::fft_dif<G1, 1>(zc);
        if (t > 0) ok &= mbar_wait(&bar_mma[(t - 1) & 1], (uint32_t)((t - 1) >> 1), a.err);
        tc_after_sync();
#pragma unroll
        for (int t2 = 0; t2 < G1; ++t2) {
            const float2 v = zc[fft::bitrev(t2, fft::ilog2(G1))];
            const int row = t1 + T1 * t2;
            const uint32_t ore = sw_off(row, k), oim = sw_off(row, M1 + k);
            *reinterpret_cast<float *>(Zhi + ore) = v.x;
            *reinterpret_cast<float *>(Zhi + oim) = v.y;
            *reinterpret_cast<float *>(Zlo + ore) = tf32_lo(v.x);
            *reinterpret_cast<float *>(Zlo + oim) = tf32_lo(v.y);
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();                         // the operands are written, the spectrum
                                                 // read; plane t - 2's accumulator drained
        if (tid == 0) {
            tc_after_sync();
            const uint32_t d = tmem + (uint32_t)(64 * (t & 1));
            const uint32_t zh = tc_smem_addr(Zhi), zl = tc_smem_addr(Zlo);
            const uint32_t th = tc_smem_addr(base + Gm::kT), tl = th + Gm::kRows64;
            constexpr uint32_t id = idesc_tf32(64, 64);    // M = 64 samples, N = 64 rows
#pragma unroll
            for (int s = 0; s < Gm::K0 / 8; ++s) {
                mma_tf32(d, desc_sw128(th + s * 32), desc_sw128(zh + s * 32), id, s ? 1u : 0u);
                mma_tf32(d, desc_sw128(th + s * 32), desc_sw128(zl + s * 32), id, 1u);
                mma_tf32(d, desc_sw128(tl + s * 32), desc_sw128(zh + s * 32), id, 1u);
            }
            mma_commit(&bar_mma[t & 1]);
        }
        if (t > 0) drain(t - 1);
        tc_before_sync();
    }
    ok &= mbar_wait(&bar_mma[(R0 - 1) & 1], (uint32_t)((R0 - 1) >> 1), a.err);
    tc_after_sync();
    drain(R0 - 1);
    tc_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(Gm::kTmemCols));
    }
    cta_record(a, 2, a.trace_c, t0, t_ready, t_spec);  // compute: the planes' spectra, tail: the planes
}

// Host: the row-DFT operand for 64 samples and 16 bins, per K chunk [T_hi |
// T_lo] with T[j][n] = cos(2 pi k n / 64) (j = k < 16) or -sin (j = 16 + k),
// split in double (T_hi as stored is read at tf32 precision; T_lo is the rest)
void make_table_a3(std::vector<unsigned char> &img) {
    using Gm = Geo3A;
    using tcu::sw_off;
    using tcu::tf32_lo;
    img.assign(Gm::kTBytes, 0);
    const double two_pi = 2.0 * M_PI;
    for (int j = 0; j < 2 * Gm::M2; ++j)
        for (int n = 0; n < Gm::N; ++n) {
            const int k = j % Gm::M2;
            const double ang = two_pi * (double)k * (double)n / (double)Gm::N;
            const double v = j < Gm::M2 ? std::cos(ang) : -std::sin(ang);
            const float hi = (float)v;
            const float lo = (float)(v - (double)(hi - tf32_lo(hi)));
            const uint32_t chunk = (uint32_t)(n / 32) * Gm::kTChunk;
            memcpy(&img[chunk + sw_off(j, n % 32)], &hi, 4);
            memcpy(&img[chunk + sw_off(2 * Gm::M2 + j, n % 32)], &lo, 4);
        }
}

// Host: kernel C's row-inverse operands T_hi and T_lo, two 64-row tiles (k < 16: s c(k) cos(2 pi k n / 64), 16 + k: -s c(k) sin(...), s =
// 1 / 64^3), split in double
void make_table_c3(std::vector<unsigned char> &img) {
    using Gm = Geo3C;
    using tcu::sw_off;
    using tcu::tf32_lo;
    img.assign(2 * Gm::kRows64, 0);
    const double two_pi = 2.0 * M_PI, s = 1.0 / ((double)Gm::N * Gm::N * Gm::N);
    for (int n = 0; n < Gm::N; ++n)
        for (int k = 0; k < Gm::M1; ++k) {
            const double ck = (k == 0 || 2 * k == Gm::N) ? 1.0 : 2.0;
            const double ang = two_pi * (double)k * (double)n / (double)Gm::N;
            const double v[2] = {s * ck * std::cos(ang), -s * ck * std::sin(ang)};
            for (int h = 0; h < 2; ++h) {
                const float hi = (float)v[h];
                const float lo = (float)(v[h] - (double)(hi - tf32_lo(hi)));
                memcpy(&img[sw_off(n, h * Gm::M1 + k)], &hi, 4);
                memcpy(&img[sw_off(Gm::N + n, h * Gm::M1 + k)], &lo, 4);
            }
        }
}

// ---------------------------------------------------------------------------
// Kernel B of the float32 3-D layer with the weights streamed by TMA (batch up
// to 4, up to 32 channels each way, weights in the standard layout).  One
// persistent CTA per SM walks the runs of kR = 16 kept modes along the last
// axis, run it = blockIdx.x, blockIdx.x + gridDim.x, ...  A producer warp
// brings a run's weights W[blk][i][o][local .. local + 15] through a ring of
// stages as boxes of 16 input channels x Cout x 16 modes (one 4-D TMA load,
// 64 KB for 32 outputs), starting before kernel A has finished: the weights
// do not depend on it.  The 8 compute warps, thread (o, mode pair), fetch the
// run's kept modes of every batch row from L2 (cp.async, the next run's
// during the current run's products), accumulate from shared memory and
// store the mixed modes.
namespace mixtma {
#ifndef FNO_MIX_TMA_I
#define FNO_MIX_TMA_I 16
#endif
#ifndef FNO_MIX_TMA_STAGES
#define FNO_MIX_TMA_STAGES 3
#endif
constexpr int kR = 16;                           // kept modes a run
constexpr int kI = FNO_MIX_TMA_I;                // input channels a stage
constexpr int kStages = FNO_MIX_TMA_STAGES;
constexpr int kCompute = 256;                    // threads of the 8 compute warps
constexpr int kThreads = kCompute + 32;          // and the producer warp
constexpr int kMaxC = 32, kMaxB = 4;
constexpr uint32_t kStageBytes = (uint32_t)kR * 8 * kMaxC * kI;        // 64 KB
constexpr uint32_t kXsBytes = (uint32_t)kMaxB * kMaxC * kR * 8;        // one run's kept modes
constexpr size_t kSmem = (size_t)kStages * kStageBytes + 2 * kXsBytes + 1024;   // + alignment
static_assert(kCompute == kMaxC * kR / 2, "one thread per (output, mode pair)");
}  // namespace mixtma

// A 4-D tile load; the weights are a stream read once a forward, so with
// FNO_MIX_TMA_EVICT_FIRST their lines are marked first to go from L2 (the kept
// and mixed modes that the other kernels read back stay)
#ifndef FNO_MIX_TMA_EVICT_FIRST
#define FNO_MIX_TMA_EVICT_FIRST 1
#endif
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar) {
#if FNO_MIX_TMA_EVICT_FIRST
    const uint64_t pol = tcu::l2_evict_first_policy();
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
                   "r"(tcu::tc_smem_addr(bar)), "l"(pol) : "memory");
#else
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5}], [%6];"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
                   "r"(tcu::tc_smem_addr(bar)) : "memory");
#endif
}

template <class C3>
__global__ void __launch_bounds__(mixtma::kThreads, 1)
k_mix_tma(const __grid_constant__ CUtensorMap wmap, Args a) {
    using namespace mixtma;
    using tcu::tc_smem_addr;
    constexpr int NK = C3::NK, kRuns = NK / kR;
    static_assert(NK % kR == 0 && C3::MR % kR == 0, "a run stays on one line of the last axis");
    extern __shared__ __align__(1024) char smem_raw[];
    // the stages start on a 1024-byte boundary (TMA destinations)
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    float2 *xs = reinterpret_cast<float2 *>(smem + kStages * kStageBytes);   // [2][batch][cin][kR]
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    const int tid = threadIdx.x, warp = tid >> 5;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int cin = a.cin, cout = a.cout, nb = a.batch;
    const int ib = cin < kI ? cin : kI;          // input channels of a box
    const int nst = (cin + kI - 1) / kI;         // stages a run
    const uint32_t box = (uint32_t)kR * 8 * cout * ib;
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&full[st])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                         ::"r"(tc_smem_addr(&empty[st])), "r"(kCompute));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_trigger();                               // kernel C may set itself up
    if (warp == kCompute / 32) {                 // the producer
        if ((tid & 31) == 0) {
            // a TMA destination must be aligned: check rather than issue a bad copy
            bool ok = (tc_smem_addr(smem) & 1023u) == 0;
            if (!ok) raise_dev_error(a.err, kDevBounds);
            int k = 0;
            for (int it = blockIdx.x; it < kRuns && ok; it += gridDim.x) {
                int blk, local;
                C3::wmap(it * kR, blk, local);
                for (int st = 0; st < nst && ok; ++st, ++k) {
                    const int sl = k % kStages;
                    if (k >= kStages) ok &= tcu::mbar_wait(&empty[sl], (uint32_t)(k / kStages - 1), a.err);
                    if (!ok) break;
                    tcu::arrive_expect_tx(&full[sl], box);
                    tma_load_4d(tc_smem_addr(smem + sl * kStageBytes), &wmap, 2 * local, 0, st * kI,
                                blk, &full[sl]);
                }
            }
        }
        return;
    }
    // thread (o, mode pair r, r + 1)
    const int o = tid / (kR / 2), r = 2 * (tid % (kR / 2));
    const bool act = o < cout;
    auto load_x = [&](int it, int buf) {
        float2 *d = xs + buf * (kXsBytes / 8);
        for (int e = tid; e < nb * cin * (kR / 2); e += kCompute) {
            const int row = e / (kR / 2), pr = e % (kR / 2);   // row = b * cin + i
            cp_async16(d + row * kR + 2 * pr, a.part + (size_t)row * NK + (size_t)it * kR + 2 * pr);
        }
    };
    pdl_wait();                                  // kernel A's kept modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    if ((int)blockIdx.x < kRuns) load_x(blockIdx.x, 0);
    cp_async_commit();
    bool ok = true;
    int k = 0, n = 0;
    for (int it = blockIdx.x; it < kRuns; it += gridDim.x, ++n) {
        if (it + (int)gridDim.x < kRuns) load_x(it + gridDim.x, (n + 1) & 1);
        cp_async_commit();
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");   // this run's kept modes
        const float2 *x = xs + (n & 1) * (kXsBytes / 8);
        float2 acc0[kMaxB], acc1[kMaxB];
#pragma unroll
        for (int b = 0; b < kMaxB; ++b) acc0[b] = acc1[b] = make_float2(0.f, 0.f);
        for (int st = 0; st < nst; ++st, ++k) {
            const int sl = k % kStages;
            ok &= tcu::mbar_wait(&full[sl], (uint32_t)(k / kStages), a.err);
            if (act) {
                const float *ws = reinterpret_cast<const float *>(smem + sl * kStageBytes);
                const int i1 = cin - st * kI < kI ? cin - st * kI : kI;
                for (int ii = 0; ii < i1; ++ii) {
                    const int i = st * kI + ii;
                    const float4 w = *reinterpret_cast<const float4 *>(
                        ws + ((size_t)(ii * cout + o) * kR + r) * 2);
                    const float2 w0 = make_float2(w.x, w.y), w1 = make_float2(w.z, w.w);
#pragma unroll
                    for (int b = 0; b < kMaxB; ++b) {
                        if (b < nb) {
                            const float4 x2 = *reinterpret_cast<const float4 *>(&x[(b * cin + i) * kR + r]);
                            cmac(acc0[b], make_float2(x2.x, x2.y), w0);
                            cmac(acc1[b], make_float2(x2.z, x2.w), w1);
                        }
                    }
                }
            }
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_addr(&empty[sl]))
                         : "memory");
        }
        if (act) {
#pragma unroll
            for (int b = 0; b < kMaxB; ++b)
                if (b < nb)
                    __stcg(reinterpret_cast<float4 *>(a.Y + ((size_t)b * cout + o) * NK +
                                                      (size_t)it * kR + r),
                           make_float4(acc0[b].x, acc0[b].y, acc1[b].x, acc1[b].y));
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");   // xs[n & 1] is read
    }
    (void)ok;
    if (a.trace) {
        asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
        if (tid == 0) {
            unsigned smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            fno_trace_record_t rec;
            rec.item = (1u << 24) | ((unsigned)blockIdx.x & 0xFFFFFFu);
            rec.worker = smid;
            rec.t_start = t0;
            rec.t_ready = t1;
            rec.t_end = trace_now();
            rec.t_compute = rec.t_end;
            a.trace[a.trace_b + blockIdx.x] = rec;
        }
    }
}

// Host: the weights of a 3-D float32 layer as a 4-D tensor map, [blk][i][o][mode
// (re, im)], boxes of 16 modes x Cout x min(16, Cin) x 1 block
template <class C3>
bool encode_wmap(CUtensorMap *map, const void *w, int cin, int cout) {
    using namespace mixtma;
    tcu::EncodeTiled fn = tcu::encoder();
    if (!fn) return false;
    const cuuint64_t e = 4, run = (cuuint64_t)C3::MBLK * 2;   // floats of one (blk, i, o)
    const cuuint64_t dims[4] = {run, (cuuint64_t)cout, (cuuint64_t)cin, 4};
    const cuuint64_t strides[3] = {run * e, run * e * cout, run * e * cout * cin};
    const cuuint32_t boxd[4] = {(cuuint32_t)kR * 2, (cuuint32_t)cout,
                                (cuuint32_t)(cin < kI ? cin : kI), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(w), dims, strides, boxd,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef FNO_MIX_STREAM
#define FNO_MIX_STREAM 1
#endif
#ifndef FNO_MIX_TMA
#define FNO_MIX_TMA 1
#endif
#ifndef FNO_STREAM_R
#define FNO_STREAM_R 16
#endif
template <class C3>
struct Pdl3 {
    static int batch_block(int64_t batch, int cin) {
        int bb = (int)batch;
        while (bb > 1 && (size_t)bb * cin * 16 > kXpBudget) bb = (bb + 1) / 2;
        return bb;
    }
    static int out_block(fno_dtype_t dt, int cin, int cout) {
        const size_t w2 = dt == FNO_F32 ? 16 : 8;
        int ob = cout;
        while (ob > 1 && (size_t)cin * ob * w2 > kWsBudget) ob = (ob + 1) / 2;
        return ob;
    }
    static size_t smem_b(fno_dtype_t dt, int cin, int ob, int bb) {
        const size_t w2 = dt == FNO_F32 ? 16 : 8;
        return ((size_t)cin * ob * w2 + 15) / 16 * 16 + (size_t)bb * cin * 16;
    }
    static constexpr int kStreamR = FNO_STREAM_R;   // modes per CTA of the streaming mixing
    template <typename T>
    static void *stream_kernel(int64_t batch) {
        if (batch <= 4) return reinterpret_cast<void *>(&k_mix_stream<C3, T, 1, kStreamR, 4>);
        if (batch <= 8) return reinterpret_cast<void *>(&k_mix_stream<C3, T, 1, kStreamR, 8>);
        return reinterpret_cast<void *>(&k_mix_stream<C3, T, 1, kStreamR, 16>);
    }
    template <typename T>
    static cudaError_t init(Plan &p) {
        const int ob = out_block(p.dtype, p.cin, p.cout), bb = batch_block(p.batch, p.cin);
        cudaError_t e = raise_smem_limit(k_phase_a3<C3, T>, (int)C3::template smem_a<T>());
        // float32, on request: the row DFT of kernel A on the tensor cores (TMA
        // plane pairs; slower than the register FFTs on the 4 x 32-channel
        // layer, 202 against 173 us a forward)
        p.fused_tca = false;
        std::vector<unsigned char> img;          // the tensor-core kernels' operands
        if constexpr (std::is_same<T, float>::value) {
            if (e == cudaSuccess && (p.flags & FNO_PLAN_TENSOR_EXTRA) &&
                !(p.flags & FNO_PLAN_SIMT_TRANSFORM) && tcu::encoder()) {
                p.fused_tca = true;
                e = raise_smem_limit(k_phase_a3_tc<C3>, (int)smem_a3_tc<C3>());
                make_table_a3(img);
            }
        }
        // kernel C's row inverse on the tensor cores unless the SIMT transforms
        // are asked for
        p.fused_tcc = !(p.flags & FNO_PLAN_SIMT_TRANSFORM);
        if (e == cudaSuccess && p.fused_tcc) {
            e = raise_smem_limit(k_phase_c3_tc<C3, T>, (int)smem_c3_tc<C3>());
            std::vector<unsigned char> imc;
            make_table_c3(imc);
            p.fused_table_c = img.size();
            img.insert(img.end(), imc.begin(), imc.end());
        }
        if (e == cudaSuccess && !img.empty()) {
            e = cudaMalloc(&p.fused_tables, img.size());
            if (e == cudaSuccess)
                e = cudaMemcpy(p.fused_tables, img.data(), img.size(), cudaMemcpyHostToDevice);
        }
        if (e == cudaSuccess)
            e = raise_smem_limit(k_phase_b<C3, T, 1, kNT>, smem_b(p.dtype, p.cin, ob + 1, bb));
        if (e == cudaSuccess)
            e = raise_smem_limit(k_phase_c3<C3, T>, (int)C3::kSmemC);
        p.fused_bb = bb;
        p.fused_ob = ob;
        p.fused_smem = smem_b(p.dtype, p.cin, ob + 1, bb);   // padded slab rows
        p.fused_grid = 0;
        // small batches: the weight-streaming mixing (each weight serves few rows)
        p.fused_bstream = 0;
        const size_t xs = (size_t)p.batch * p.cin * kStreamR * 8;   // the run's kept modes
        if (FNO_MIX_STREAM && p.batch <= 16 && p.cout * kStreamR <= 4 * kMixThreads &&
            xs <= (64u << 10)) {
            p.fused_bstream = kStreamR;
            if (e == cudaSuccess) e = raise_smem_limit(stream_kernel<T>(p.batch), xs);
        }
        // float32, batch <= 4, <= 32 channels, standard weight layout: the
        // weights streamed by TMA into one persistent CTA per SM (fused_grid CTAs)
        if constexpr (std::is_same<T, float>::value) {
            if (FNO_MIX_TMA && e == cudaSuccess && p.fused_bstream && p.batch <= mixtma::kMaxB &&
                p.cin <= mixtma::kMaxC && p.cout <= mixtma::kMaxC &&
                !(p.flags & FNO_PLAN_PACKED_WEIGHTS) && !(p.flags & FNO_PLAN_SIMT_MIX) &&
                tcu::encoder()) {
                p.fused_grid = std::min(p.num_sms, (int)(C3::NK / mixtma::kR));
                e = raise_smem_limit(k_mix_tma<C3>, mixtma::kSmem);
            }
        }
        if (e == cudaSuccess && (p.flags & FNO_PLAN_TRACE)) {
            const size_t nB = p.fused_grid      ? (size_t)p.fused_grid
                              : p.fused_bstream ? (size_t)(C3::NK / p.fused_bstream)
                                                : (size_t)(C3::NK / kG) * ((p.cout + ob - 1) / ob) *
                                                      ((p.batch + bb - 1) / bb);
            p.trace_records = (size_t)p.batch * (p.cin + p.cout) * C3::C0 + nB;
            e = cudaMalloc(&p.trace, p.trace_records * sizeof(fno_trace_record_t));
        }
        return e;
    }
    template <typename T>
    static cudaError_t forward(const Plan &p, Args a, cudaStream_t s) {
        a.bg = p.fused_bb;
        a.ng = (int)((p.batch + a.bg - 1) / a.bg);
        a.ob = p.fused_ob;
        a.nob = (p.cout + a.ob - 1) / a.ob;
        a.npairs = C3::NK / kG;
        a.trace = p.trace;
        a.trace_b = (int)(p.batch * p.cin * C3::C0);
        a.trace_c = a.trace_b + (p.fused_grid      ? p.fused_grid
                                 : p.fused_bstream ? C3::NK / p.fused_bstream
                                                   : a.npairs * a.nob * a.ng);
        cudaLaunchAttribute cl;
        cl.id = cudaLaunchAttributeClusterDimension;
        cl.val.clusterDim.x = C3::C0;
        cl.val.clusterDim.y = 1;
        cl.val.clusterDim.z = 1;
        cudaLaunchConfig_t ca = {};
        ca.gridDim = dim3((unsigned)(p.batch * p.cin * C3::C0));
        ca.blockDim = dim3(kNT);
        ca.dynamicSmemBytes = C3::template smem_a<T>();
        ca.stream = s;
        ca.attrs = &cl;
        ca.numAttrs = 1;
        cudaError_t e = cudaSuccess;
        bool done_a = false;
        if constexpr (std::is_same<T, float>::value) {
            if (p.fused_tca) {
                // the input as rows of N2 samples, boxes of 32 samples x one plane
                CUtensorMap xmap;
                if (!tcu::encode_rows_tiled(&xmap, a.x, (int64_t)p.batch * p.cin * C3::N0 * C3::N1,
                                            C3::N2, sizeof(float), 32, tcu::tma_type<float>(),
                                            C3::N1))
                    return cudaErrorInvalidValue;
                ca.dynamicSmemBytes = smem_a3_tc<C3>();
                e = cudaLaunchKernelEx(&ca, k_phase_a3_tc<C3>, xmap, a,
                                       static_cast<const void *>(p.fused_tables));
                done_a = true;
            }
        }
        if (!done_a) e = cudaLaunchKernelEx(&ca, k_phase_a3<C3, T>, a);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kNT);
        cfg.stream = s;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        bool done_b = false;
        if constexpr (std::is_same<T, float>::value) {
            if (p.fused_grid) {
                CUtensorMap wmap;
                if (!encode_wmap<C3>(&wmap, a.w, p.cin, p.cout)) return cudaErrorInvalidValue;
                cfg.gridDim = dim3((unsigned)p.fused_grid);
                cfg.blockDim = dim3(mixtma::kThreads);
                cfg.dynamicSmemBytes = mixtma::kSmem;
                e = cudaLaunchKernelEx(&cfg, k_mix_tma<C3>, wmap, a);
                done_b = true;
            }
        }
        if (done_b) {
        } else if (p.fused_bstream) {
            cfg.gridDim = dim3((unsigned)(C3::NK / p.fused_bstream));
            cfg.blockDim = dim3(kMixThreads);
            cfg.dynamicSmemBytes = (size_t)p.batch * p.cin * p.fused_bstream * 8;
            if (p.batch <= 4)
                e = cudaLaunchKernelEx(&cfg, k_mix_stream<C3, T, 1, kStreamR, 4>, a);
            else if (p.batch <= 8)
                e = cudaLaunchKernelEx(&cfg, k_mix_stream<C3, T, 1, kStreamR, 8>, a);
            else
                e = cudaLaunchKernelEx(&cfg, k_mix_stream<C3, T, 1, kStreamR, 16>, a);
        } else {
            cfg.gridDim = dim3((unsigned)(a.npairs * a.nob * a.ng));
            cfg.blockDim = dim3(kNT);
            cfg.dynamicSmemBytes = p.fused_smem;
            e = cudaLaunchKernelEx(&cfg, k_phase_b<C3, T, 1, kNT>, a);
        }
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3((unsigned)(p.batch * p.cout * C3::C0));
        if (p.fused_tcc) {
            cfg.blockDim = dim3(kNT);
            cfg.dynamicSmemBytes = smem_c3_tc<C3>();
            const void *tab = static_cast<const char *>(p.fused_tables) + p.fused_table_c;
            e = cudaLaunchKernelEx(&cfg, k_phase_c3_tc<C3, T>, a, tab);
        } else {
            cfg.blockDim = dim3(kNT);
            cfg.dynamicSmemBytes = C3::kSmemC;
            e = cudaLaunchKernelEx(&cfg, k_phase_c3<C3, T>, a);
        }
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

bool fused3d_match(const Geom &g, fno_dtype_t dtype) {
    using C3 = Cfg3d64;
    return g.d == 3 && (dtype == FNO_F32 || dtype == FNO_F16 || dtype == FNO_BF16) &&
           g.n[0] == C3::N0 &&
           g.n[1] == C3::N1 && g.n[2] == C3::N2 && g.m[0] == C3::M0 && g.m[1] == C3::M1 &&
           g.m[2] == C3::M2;
}

bool fused3d_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout) {
    using C3 = Cfg3d64;
    if (!fused3d_match(g, dtype)) return false;
    const size_t w2 = dtype == FNO_F32 ? 16 : 8;
    // grids fit in x; one output's weight slab and one batch row of modes fit
    // the mixing item's shared memory
    return batch * (int64_t)(cin > cout ? cin : cout) * C3::C0 < (1ll << 31) &&
           (int64_t)(C3::NK / kG) * cout * batch < (1ll << 31) &&
           (size_t)cin * w2 <= kWsBudget && (size_t)cin * 16 <= kXpBudget;
}

size_t fused3d_workspace_bytes(const Geom &g, int64_t batch, int cin, int cout) {
    return align256((size_t)batch * cin * g.nkept * sizeof(float2)) +
           align256((size_t)batch * cout * g.nkept * sizeof(float2));
}

cudaError_t fused3d_plan_init(Plan &p) {
    return with_storage(p.dtype, [&](auto t) { return Pdl3<Cfg3d64>::init<decltype(t)>(p); });
}

cudaError_t fused3d_forward_modes(const Plan &p, const void *x, int64_t nimg, float2 *out,
                                  cudaStream_t s) {
    using C3 = Cfg3d64;
    Args a{};
    a.x = x;
    a.part = out;
    a.tw0 = p.tw[0];
    a.tw1 = p.tw[1];
    a.tw2 = p.tw[2];
    a.err = p.dev_err;
    return with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        cudaLaunchAttribute cl;
        cl.id = cudaLaunchAttributeClusterDimension;
        cl.val.clusterDim.x = C3::C0;
        cl.val.clusterDim.y = 1;
        cl.val.clusterDim.z = 1;
        cudaLaunchConfig_t ca = {};
        ca.gridDim = dim3((unsigned)(nimg * C3::C0));
        ca.blockDim = dim3(kNT);
        ca.dynamicSmemBytes = C3::template smem_a<T>();
        ca.stream = s;
        ca.attrs = &cl;
        ca.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&ca, k_phase_a3<C3, T>, a);
        return e != cudaSuccess ? e : cudaGetLastError();
    });
}

cudaError_t fused3d_forward(const Plan &p, const Buffers &b, cudaStream_t s) {
    Args a{};
    a.x = b.x;
    a.w = b.w;
    a.y = b.y;
    a.part = static_cast<float2 *>(b.ws);
    a.Y = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) +
                                     align256((size_t)p.batch * p.cin * p.g.nkept * sizeof(float2)));
    a.tw0 = p.tw[0];
    a.tw1 = p.tw[1];
    a.tw2 = p.tw[2];
    a.err = p.dev_err;
    a.batch = (int)p.batch;
    a.cin = p.cin;
    a.cout = p.cout;
    a.wpacked = (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0;
    return with_storage(p.dtype,
                        [&](auto t) { return Pdl3<Cfg3d64>::forward<decltype(t)>(p, a, s); });
}

}  // namespace fno
