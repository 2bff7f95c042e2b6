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
//   phase A  (image, row chunk)           x rows -> partial kept modes   (HBM read)
//   phase B  (mode pair, o block, b block) sum partials, mix with W -> Y (L2 + W)
//   phase C  (image, row chunk)           Y -> output rows              (HBM write)
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
//
// Shared-memory layouts are chosen so that the 32 lanes of a warp touch 32
// distinct banks (padded row strides, bin index fastest); loads of the
// mixing and inverse phases are issued as cp.async copies all at once, and
// the weights of a mixing item are fetched before it waits for phase A.
#include <new>
#include <vector>

#include "fno_fused_dev.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

// ---------------------------------------------------------------------------
// The persistent kernel
// ---------------------------------------------------------------------------

// Work items of group g, in ticket order: A(0), A(1), B(0), A(2), B(1), C(0),
// ..., so that while a group mixes, the next one transforms and the previous
// one runs its inverse.
struct Item {
    int phase;          // 0: A, 1: B, 2: C, -1: none left
    int g, idx;
    int ticket;
};

template <class Cf>
__device__ Item decode_ticket(const Args &a, int t) {
    const int t0 = t;
    for (int st = 0; st < a.ng + 2; ++st) {
        if (st < a.ng) {
            const int n = min(a.bg, a.batch - st * a.bg) * a.cin * Cf::C;
            if (t < n) return Item{0, st, t, t0};
            t -= n;
        }
        if (st >= 1 && st - 1 < a.ng) {
            const int n = a.npairs * a.nob;
            if (t < n) return Item{1, st - 1, t, t0};
            t -= n;
        }
        if (st >= 2) {
            const int g = st - 2;
            const int n = min(a.bg, a.batch - g * a.bg) * a.cout * Cf::C;
            if (t < n) return Item{2, g, t, t0};
            t -= n;
        }
    }
    return Item{-1, 0, 0, t0};
}

// Trace stamps of one item, written by the thread that runs its serial part.
struct TraceStamp {
    unsigned long long t_start = 0, t_ready = 0, t_compute = 0;
    __device__ void start(const Args &a) { if (a.trace) t_start = trace_now(); }
    __device__ void ready(const Args &a) { if (a.trace) t_ready = trace_now(); }
    __device__ void computed(const Args &a) { if (a.trace) t_compute = trace_now(); }
    __device__ void end(const Args &a, const Item &it, unsigned worker) const {
        if (!a.trace) return;
        fno_trace_record_t r;
        r.item = ((unsigned)it.phase << 24) | ((unsigned)it.g << 16) | (unsigned)it.idx;
        r.worker = worker;
        r.t_start = t_start;
        r.t_ready = t_ready ? t_ready : t_start;
        r.t_compute = t_compute ? t_compute : r.t_ready;
        r.t_end = trace_now();
        a.trace[it.ticket] = r;
    }
};

template <class Cf, typename T>
__global__ void __launch_bounds__(kNT)
k_fused2d(Args a) {
    extern __shared__ __align__(16) char smem[];
    __shared__ Item s_item;
    __shared__ int s_ok;
    float2 *tw0 = reinterpret_cast<float2 *>(smem);
    float2 *tw1 = tw0 + Cf::N0;
    float2 *tw1i = tw1 + Cf::P * Cf::TS;
    char *work = smem + Cf::kSmemTw;
    const int tid = threadIdx.x;
    for (int e = tid; e < Cf::N0; e += kNT) tw0[e] = a.tw0[e];
    fill_row_tables<Cf>(a.tw1, tw1, tw1i, 1.0f / ((float)Cf::N0 * (float)Cf::N1));
    const Tw tw{tw0, tw1, tw1i};
    const int nimg_in = a.batch * a.cin;
    // thread 0 claims one ticket ahead: the atomic's round trip overlaps the
    // current item.  A held ticket is always larger than its holder's current
    // item and every dependency points to smaller tickets, so the smallest
    // unfinished ticket can always run: no deadlock.
    int next_ticket = 0;
    if (tid == 0) next_ticket = atomicAdd(&a.sync->ticket[0], 1);
    for (;;) {
        if (tid == 0) {
            s_item = decode_ticket<Cf>(a, next_ticket);
            if (s_item.phase >= 0) next_ticket = atomicAdd(&a.sync->ticket[0], 1);
        }
        __syncthreads();
        const Item it = s_item;
        __syncthreads();
        if (it.phase < 0) break;
        const int nbg = min(a.bg, a.batch - it.g * a.bg);     // batch rows of the group
        TraceStamp ts;
        if (tid == 0) ts.start(a);
        if (it.phase == 0) {
            const int img = it.g * a.bg * a.cin + it.idx / Cf::C;
            // the weights are read by the mixing items: bring them into L2 meanwhile
            if (tid == 0 && a.wslice) {
                const size_t off = (size_t)it.ticket * a.wslice;
                if (off < a.wbytes)
                    prefetch_l2(static_cast<const char *>(a.w) + off,
                                (unsigned)min((size_t)a.wslice, a.wbytes - off));
            }
            phase_a<Cf, T>(static_cast<const T *>(a.x), a.part, nimg_in, img, it.idx % Cf::C,
                           work, tw);
            __syncthreads();
            if (tid == 0) ts.computed(a);
            if (tid == 0)
                finish_item(&a.sync->done_a[it.g][0], nbg * a.cin * Cf::C, a.sync->flag_a[it.g]);
        } else if (it.phase == 1) {
            BItem bi;
            bi.pair = it.idx / a.nob;
            bi.o0 = (it.idx % a.nob) * a.ob;
            bi.nob = min(a.ob, a.cout - bi.o0);
            bi.b0 = it.g * a.bg;
            bi.nbb = nbg;
            // the weights do not depend on phase A: request them first
            phase_b_weights<Cf, T, kNT>(CtaGroup{tid}, static_cast<const T *>(a.w), a.cin, a.cout, bi,
                                        a.ob, work, a.wpacked != 0);
            if (tid == 0)
                s_ok = wait_flag(&a.sync->flag_a[it.g][blockIdx.x % kFlagCopies][0], a.err);
            if (tid == 0) ts.ready(a);
            __syncthreads();
            if (s_ok) phase_b<Cf, T, kNT>(CtaGroup{tid}, a.part, a.Y, a.cin, a.cout, nimg_in, bi, a.ob, work);
            else cp_async_wait_all();
            __syncthreads();
            if (tid == 0) ts.computed(a);
            if (tid == 0)
                finish_item(&a.sync->done_b[it.g][0], a.npairs * a.nob, a.sync->flag_b[it.g]);
        } else {
            if (tid == 0)
                s_ok = wait_flag(&a.sync->flag_b[it.g][blockIdx.x % kFlagCopies][0], a.err);
            if (tid == 0) ts.ready(a);
            __syncthreads();
            if (s_ok) {
                const int img = it.g * a.bg * a.cout + it.idx / Cf::C;
                phase_c<Cf, T>(a.Y, static_cast<T *>(a.y), img, it.idx % Cf::C, work, tw);
            }
        }
        __syncthreads();
        if (tid == 0) ts.end(a, it, blockIdx.x);
    }
    // the last CTA to leave resets the counters and flags for the next launch
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(&a.sync->exited[0], 1);
        if (prev == (int)gridDim.x - 1) {
            a.sync->ticket[0] = 0;
            for (int g = 0; g < a.ng; ++g) {
                a.sync->done_a[g][0] = 0;
                a.sync->done_b[g][0] = 0;
                for (int i = 0; i < kFlagCopies; ++i) {
                    a.sync->flag_a[g][i][0] = 0;
                    a.sync->flag_b[g][i][0] = 0;
                }
            }
            __threadfence();
            a.sync->exited[0] = 0;
        }
    }
}

// ---------------------------------------------------------------------------
// Three-kernel variant: phase A, B and C as separate grids chained by
// programmatic dependent launch.  Every CTA runs one item, so the hardware
// block scheduler replaces the ticket queue and its atomics.  Kernel B (C) is
// launched while kernel A (B) still runs; its CTAs become resident once every
// CTA of the previous grid has started, fetch what does not depend on it (the
// weight slab, the twiddles) and then wait in griddepcontrol.wait until the
// previous grid has finished and its writes are visible.  The first kernel of
// a forward is an ordinary launch, so it is ordered after whatever the stream
// ran before (e.g. the producer of x).
// ---------------------------------------------------------------------------

template <class Cf>
__device__ __forceinline__ Tw load_twiddles(const Args &a, char *smem) {
    float2 *tw0 = reinterpret_cast<float2 *>(smem);
    float2 *tw1 = tw0 + Cf::N0;
    float2 *tw1i = tw1 + Cf::P * Cf::TS;
    for (int e = threadIdx.x; e < Cf::N0; e += kNT) tw0[e] = a.tw0[e];
    fill_row_tables<Cf>(a.tw1, tw1, tw1i, 1.0f / ((float)Cf::N0 * (float)Cf::N1));
    return Tw{tw0, tw1, tw1i};
}

template <class Cf, typename T, bool kCluster>
__global__ void __launch_bounds__(kNT) k_phase_a(Args a) {
    extern __shared__ __align__(16) char smem[];
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const Tw tw = load_twiddles<Cf>(a, smem);
    __syncthreads();
    pdl_trigger();
    const int item = blockIdx.x;                 // image * C + chunk
    phase_a<Cf, T, kCluster>(static_cast<const T *>(a.x), a.part, a.batch * a.cin, item / Cf::C,
                             item % Cf::C, smem + Cf::kSmemTw, tw);
    cta_record(a, 0, 0, t0, t0);
}

template <class Cf, typename T>
__global__ void __launch_bounds__(kNT) k_phase_c(Args a) {
    extern __shared__ __align__(16) char smem[];
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const Tw tw = load_twiddles<Cf>(a, smem);
    __syncthreads();
    pdl_wait();                                  // kernel B's mixed modes are complete
    pdl_trigger();                               // a dependent kernel may set itself up
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    const int item = blockIdx.x;
    phase_c<Cf, T>(a.Y, static_cast<T *>(a.y), item / Cf::C, item % Cf::C, smem + Cf::kSmemTw, tw);
    cta_record(a, 2, a.trace_c, t0, t1);
}


// ---------------------------------------------------------------------------
// Kernel A of the three-kernel path on the tensor cores for 16-bit 256 x 256
// layers: a CTA transforms whole input images, so the kept modes leave it
// complete (no partial copies).  One persistent CTA per SM takes the images
// blockIdx.x, blockIdx.x + gridDim.x, ...: as soon as an image's MMAs have
// read its tile, the next image's tile is requested into the same buffer and
// lands while the current image's column work runs.
//
// TMA brings an image into shared memory as M tiles of 128 rows, K-major with
// the 128-byte swizzle.  The row DFT of bins 0..M1-1 is the GEMM
// Z = X . T^T, T[j][n] = cos(2 pi j n / N1) (j < M1) and -sin(...) (j >= M1),
// on tcgen05 with the accumulator in tensor memory, one kind::f16 pass (the
// 16-bit tolerance class is 1e-2; fp32 images have their own pipelined kernel
// below).  The column DFT over the N0 rows, kept rows only, runs on the SIMT
// cores in two steps: with rows t = t1 + T1 t2 and the signed frequencies
// g = g1 + G1 g2 (G1 = M0, T1 = N0 / G1),
//   F[t1][g1][k] = sum_t2 Z[t1 + T1 t2][k] e^{-2 pi i g1 t2 / G1}   (register FFTs)
//   X[g][k]      = sum_t1 W_N0^{g t1} F[t1][g mod G1][k]             (T1 terms).
// ---------------------------------------------------------------------------
namespace tca {

constexpr int NT = 256;
template <typename T> struct Shape;
template <> struct Shape<__half> {         // 256 x 256, 32 x 32 modes
    static constexpr int N0 = 256, N1 = 256, M0 = 32, M1 = 32, kE = 64;
    static constexpr int kMinBlocks = 1;
};
template <> struct Shape<__nv_bfloat16> : Shape<__half> {};

template <typename T>
struct Geo {
    using S = Shape<T>;
    static constexpr int N0 = S::N0, N1 = S::N1, M0 = S::M0, M1 = S::M1, kE = S::kE;
    static constexpr int KC = N1 / kE;                  // K chunks of 128 bytes
    static constexpr int MT = N0 / 128;                 // M tiles
    static constexpr int N = 2 * M1;                    // MMA N: bins, re then im
    static constexpr int K0 = 2 * M0, NK = K0 * M1;
    static constexpr int G1 = M0, T1 = N0 / G1;         // column DFT split
    static constexpr uint32_t kTile = 16384;            // 128 rows x 128 bytes
    static constexpr uint32_t kXBytes = (uint32_t)MT * KC * kTile;
    static constexpr uint32_t kTChunk = (uint32_t)N * 128;
    static constexpr uint32_t kTBytes = KC * kTChunk;
    // Z planes (re, im) [N0][M1], columns XOR-swizzled by the row; the column
    // sums F [T1][G1][M1] go over them
    static constexpr uint32_t kZBytes = (uint32_t)N0 * M1 * 4 * 2;
    static constexpr uint32_t kFBytes = (uint32_t)T1 * G1 * M1 * 8;
    static constexpr uint32_t kT = kXBytes;             // offsets from a 1024-aligned base
    static constexpr uint32_t kZ = kT + kTBytes;
    static constexpr uint32_t kSmem = kZ + (kZBytes > kFBytes ? kZBytes : kFBytes) + 1024;
    static constexpr uint32_t kTmemCols = MT * N <= 32 ? 32 : (MT * N <= 64 ? 64 : 128);
    static_assert(T1 * 32 == NT && M1 == 32 && K0 == 2 * G1, "warp t1, lane k");
    static_assert(kSmem + 1024 <= 232448, "image tile, table and Z planes fit one CTA");
};

// The kernel is warp-specialised.  Warp 8 (one elected thread) is the
// producer: it loads each image as two 128-row M tiles (64 KiB each, four TMA
// boxes), issues a tile's row-DFT MMAs as soon as the tile has landed into one
// of two tensor-memory accumulators, and requests the next image's tile into
// the same buffer as soon as those MMAs have read it.  Warps 0-7 (the
// consumers) take an accumulator once both tiles' MMAs are done, copy Z out of
// tensor memory, release the accumulator, and run the column DFT.  So the next
// image's loads and row DFT proceed under this image's column work.
constexpr int kNTA = NT + 32;            // consumers + producer warp

// named barrier of the 256 consumer threads (barrier 0 is the whole CTA's)
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(NT) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kNTA, Shape<T>::kMinBlocks)
k_phase_a_tc(const __grid_constant__ CUtensorMap xmap, Args a, const void *tables, int nimg) {
    using Gm = Geo<T>;
    using namespace tcu;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    // full[t]: tile t landed; empty[t]: its MMAs are done (the buffer may be
    // refilled); acc[b]: accumulator b holds an image's Z; free_[b]: the
    // consumers have copied accumulator b out (256 arrivals)
    __shared__ __align__(8) uint64_t bar_t, full[2], empty[2], acc[2], free_[2];
    __shared__ uint32_t s_tmem;
    static_assert(Gm::MT == 2, "two M tiles");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr uint32_t kTileBytes = Gm::KC * Gm::kTile;        // one M tile of the image
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_t)));
        for (int i = 0; i < 2; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&empty[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&acc[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem_addr(&free_[i])),
                         "r"(NT));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(2 * Gm::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    pdl_trigger();
    const uint32_t tmem = s_tmem;
    const uint32_t xs = tc_smem_addr(base), ts = tc_smem_addr(base + Gm::kT);

    if (warp == NT / 32) {
        // ----- producer -----
        if (lane == 0) {
            // the input is read once: its lines leave L2 first, so the kept modes
            // this kernel writes (and the mixing reads next) stay resident
            const uint64_t pol = l2_evict_first_policy();
            auto load_tile = [&](int img, int t) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             ::"r"(tc_smem_addr(&full[t])), "r"(kTileBytes) : "memory");
                for (int kc = 0; kc < Gm::KC; ++kc)
                    tma_load_2d_hint(xs + (t * Gm::KC + kc) * Gm::kTile, &xmap, kc * Gm::kE,
                                     img * Gm::N0 + 128 * t, &full[t], pol);
            };
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         ::"r"(tc_smem_addr(&bar_t)), "r"(Gm::kTBytes) : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(ts), "l"(tables), "r"(Gm::kTBytes), "r"(tc_smem_addr(&bar_t))
                         : "memory");
            if ((int)blockIdx.x < nimg) {
                load_tile(blockIdx.x, 0);
                load_tile(blockIdx.x, 1);
            }
            bool ok = mbar_wait(&bar_t, 0, a.err);
            constexpr uint32_t id = idesc_f16(Gm::N, std::is_same<T, __nv_bfloat16>::value);
            uint32_t it = 0;
            for (int img = blockIdx.x; img < nimg; img += gridDim.x, ++it) {
                const uint32_t b = it & 1;
                if (it >= 2) ok &= mbar_wait(&free_[b], ((it - 2) >> 1) & 1, a.err);
                tc_after_sync();
                for (int t = 0; t < Gm::MT; ++t) {
                    ok &= mbar_wait(&full[t], it & 1, a.err);
                    tc_after_sync();
                    const uint32_t d = tmem + b * Gm::kTmemCols + t * Gm::N;
                    for (int kc = 0; kc < Gm::KC && ok; ++kc)
#pragma unroll
                        for (int s4 = 0; s4 < 4; ++s4)
                            mma_f16(d, desc_sw128(xs + (t * Gm::KC + kc) * Gm::kTile + s4 * 32),
                                    desc_sw128(ts + kc * Gm::kTChunk + s4 * 32), id,
                                    (kc | s4) ? 1u : 0u);
                    mma_commit(&empty[t]);
                }
                mma_commit(&acc[b]);
                const int next = img + (int)gridDim.x;
                for (int t = 0; t < Gm::MT; ++t) {
                    ok &= mbar_wait(&empty[t], it & 1, a.err);
                    if (next < nimg) load_tile(next, t);
                }
            }
        }
    } else {
        // ----- consumers: warp t1, lane k of the column DFT -----
        // Z as complex rows [t][32 bins], the bin index XOR-swizzled by the row
        float2 *Zc = reinterpret_cast<float2 *>(base + Gm::kZ);
        float2 *F = reinterpret_cast<float2 *>(base + Gm::kZ);
        bool ok = true;
        uint32_t it = 0;
        for (int img = blockIdx.x; img < nimg; img += gridDim.x, ++it) {
            const unsigned long long t0 = a.trace ? trace_now() : 0;
            const uint32_t b = it & 1;
            ok &= mbar_wait(&acc[b], (it >> 1) & 1, a.err);
            tc_after_sync();
            const unsigned long long t_z = a.trace ? trace_now() : 0;   // the row DFT is done
            // Z from tensor memory: warp w reads the lanes 32 (w % 4).. of M tile w / 4,
            // all 64 columns (bins re, then im) of its row
            {
                const int t = warp >> 2;
                const int row = 128 * t + 32 * (warp & 3) + lane;
                const uint32_t tbase = tmem + ((uint32_t)(32 * (warp & 3)) << 16) +
                                       b * Gm::kTmemCols + t * Gm::N;
#pragma unroll
                for (int g = 0; g < Gm::M1 / 16; ++g) {
                    float re[16], im[16];
                    tmem_ld16(tbase + 16 * g, re);
                    tmem_ld16(tbase + Gm::M1 + 16 * g, im);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int k = 16 * g + q;
                        Zc[row * Gm::M1 + (k ^ (row & 31))] =
                            ok ? make_float2(re[q], im[q]) : make_float2(0.f, 0.f);
                    }
                }
            }
            tc_before_sync();
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_addr(&free_[b]))
                         : "memory");
            consumer_sync();
            // F[t1][g1][k]: G1-point FFT over t2 of Z[t1 + T1 t2][k], warp t1, lane k
            float2 z[Gm::G1];
#pragma unroll
            for (int t2 = 0; t2 < Gm::G1; ++t2) {
                const int r = warp + Gm::T1 * t2;
                z[t2] = Zc[r * Gm::M1 + (lane ^ (r & 31))];
            }
            fft::fft_dif<Gm::G1, -1>(z);
            consumer_sync();                     // Z is read: F goes over it
#pragma unroll
            for (int g1 = 0; g1 < Gm::G1; ++g1)
                F[(warp * Gm::G1 + g1) * Gm::M1 + lane] = z[fft::bitrev(g1, fft::ilog2(Gm::G1))];
            consumer_sync();
            // kept modes in pairs: low row j (g = j) and high row j + 32 (g = j - 32)
            // share F[t1][j][k]; with P[t1] = W_N0^{j t1} F[t1][j][k],
            //   X[j][k] = sum_t1 P[t1],  X[j + 32][k] = sum_t1 P[t1] e^{+2 pi i t1 / 8}
            // (W_N0^{-32 t1} = e^{+2 pi i t1 / 8}, a compile-time constant)
            static_assert(Gm::K0 == 2 * Gm::G1 && Gm::T1 == 8, "pairs of kept rows, 8 terms");
            const size_t gstride = (size_t)a.batch * a.cin * 8;         // words per group
            uint32_t *xg = reinterpret_cast<uint32_t *>(a.part) + (size_t)img * 8;
            float2 *dst = a.part + (size_t)img * Gm::NK;
#pragma unroll
            for (int pq = 0; pq < Gm::G1 / 8; ++pq) {
                const int j = warp + 8 * pq;
                float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
                fft::unroll<0, Gm::T1>([&](auto tt) {
                    constexpr int t1 = decltype(tt)::value;
                    const float2 f = F[(t1 * Gm::G1 + j) * Gm::M1 + lane];
                    const float2 P = fft::cmul(f, __ldg(a.tw0 + ((j * t1) & (Gm::N0 - 1))));
                    lo = fft::cadd(lo, P);
                    hi = fft::cadd(hi, fft::twiddle<t1, Gm::T1, +1>(P));
                });
                const int o_lo = j * Gm::M1 + lane, o_hi = (j + Gm::G1) * Gm::M1 + lane;
                if (a.mix16) {
                    // 16-bit (re, im) pairs in group o / 8 of the mixing's input:
                    // [group][image][8 modes], a warp's 32 modes fill four 32-byte pieces
                    uint32_t ulo, uhi;
                    if constexpr (std::is_same<T, __half>::value) {
                        const __half2 h0 = __floats2half2_rn(lo.x, lo.y);
                        const __half2 h1 = __floats2half2_rn(hi.x, hi.y);
                        memcpy(&ulo, &h0, 4);
                        memcpy(&uhi, &h1, 4);
                    } else {
                        const __nv_bfloat162 h0 = __floats2bfloat162_rn(lo.x, lo.y);
                        const __nv_bfloat162 h1 = __floats2bfloat162_rn(hi.x, hi.y);
                        memcpy(&ulo, &h0, 4);
                        memcpy(&uhi, &h1, 4);
                    }
                    const int64_t xwords = (int64_t)Gm::NK * a.batch * a.cin;
                    const int64_t ilo = (o_lo >> 3) * gstride + (o_lo & 7) + (int64_t)img * 8;
                    const int64_t ihi = (o_hi >> 3) * gstride + (o_hi & 7) + (int64_t)img * 8;
                    if (in_bounds(ilo, xwords, a.err)) xg[ilo - (int64_t)img * 8] = ulo;
                    if (in_bounds(ihi, xwords, a.err)) xg[ihi - (int64_t)img * 8] = uhi;
                } else {
                    __stcg(dst + o_lo, lo);
                    __stcg(dst + o_hi, hi);
                }
            }
            consumer_sync();                     // F is read: the next Z goes over it
            if (a.trace && tid == 0) {
                unsigned smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                fno_trace_record_t r;
                r.item = (0u << 24) | ((unsigned)img & 0xFFFFFFu);
                r.worker = smid;
                r.t_start = t0;
                r.t_ready = t_z;
                r.t_compute = t_z;
                r.t_end = trace_now();
                a.trace[img] = r;
            }
        }
    }
    tc_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(2 * Gm::kTmemCols));
    }
}

// ---------------------------------------------------------------------------
// Kernel A on the tensor cores for fp32 128 x 128 layers (16 x 16 modes), a
// pipeline over the image's four 32-column K chunks.  Each chunk has its own
// TMA barrier; pass 1 multiplies the chunk by [T_hi; T_lo] (N = 64: columns
// 0..31 of the accumulator take x T_hi, 32..63 x T_lo) as soon as it lands,
// then, while the next chunk's pass 1 runs, the threads overwrite the chunk
// with its tf32 remainder x_lo and pass 2 adds x_lo T_hi into columns 0..31.
// Z = the two column halves summed; the column DFT and the kept modes follow
// on the SIMT cores as in the 16-bit kernel.  Two CTAs per SM.
// ---------------------------------------------------------------------------
struct Geo32 {
    static constexpr int N0 = 128, N1 = 128, M0 = 16, M1 = 16, K0 = 32, NK = K0 * M1;
    static constexpr int KC = 4;                        // K chunks of 32 fp32 (128 bytes)
    static constexpr int B2 = 8, R1 = N0 / B2;          // column DFT: r = r1 + 16 r2
    static constexpr uint32_t kTile = 16384;            // one K chunk of the image
    static constexpr uint32_t kXBytes = KC * kTile;
    static constexpr uint32_t kTChunk = 64 * 128;       // [T_hi rows 0..31 | T_lo rows 0..31]
    static constexpr uint32_t kTBytes = KC * kTChunk;
    // Z planes (then the column sums over them) [N0][M1], bin k of row r at
    // column k ^ (r % 16): conflict-free both for a warp of rows and for a warp
    // of (row pair, bins); they go over the image's last K chunk
    static constexpr int ZS = M1;
    static constexpr uint32_t kZBytes = (uint32_t)N0 * ZS * 4 * 2;
    static constexpr uint32_t kZOff = 3 * kTile;
    static_assert(M1 == 16 && kZOff + kZBytes <= kXBytes, "Z planes fit over chunk 3");
    static constexpr uint32_t kT = kXBytes;
    static constexpr uint32_t kTw = kT + kTBytes;
    static constexpr uint32_t kSmem = kTw + N0 * 8 + 1024;
    static constexpr uint32_t kTmemCols = 64;
};

// One persistent CTA (two per SM) walks images img = blockIdx.x + k gridDim.x.
// An image's four K chunks arrive by TMA; the row spectra (Z, then the column
// sums over them in place) go over chunk 3 once the second pass has read it,
// so the next image's chunks 0..2 are requested as soon as the row DFT is done
// and chunk 3 once the kept modes are written: the loads of one image land
// under the column work of the one before.
__global__ void __launch_bounds__(NT, 2)
k_phase_a_tc32(const __grid_constant__ CUtensorMap xmap, Args a, const void *tables, int nimg) {
    using Gm = Geo32;
    using namespace tcu;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_t, bar_fin, bar_x[Gm::KC], bar_p1[Gm::KC];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5;
    float2 *tw = reinterpret_cast<float2 *>(base + Gm::kTw);
    auto issue = [&](int img, int kc) {          // chunk kc of image img (thread 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(tc_smem_addr(&bar_x[kc])), "r"(Gm::kTile) : "memory");
        tma_load_2d(tc_smem_addr(base + kc * Gm::kTile), &xmap, kc * 32, img * Gm::N0,
                    &bar_x[kc]);
    };
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_t)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_fin)));
        for (int kc = 0; kc < Gm::KC; ++kc) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_x[kc])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_p1[kc])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(tc_smem_addr(&bar_t)), "r"(Gm::kTBytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(tc_smem_addr(base + Gm::kT)), "l"(tables), "r"(Gm::kTBytes),
                     "r"(tc_smem_addr(&bar_t)) : "memory");
        if ((int)blockIdx.x < nimg)
            for (int kc = 0; kc < Gm::KC; ++kc) issue(blockIdx.x, kc);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(Gm::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    for (int e = tid; e < Gm::N0; e += NT) tw[e] = a.tw0[e];
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    pdl_trigger();
    const uint32_t tmem = s_tmem;
    const uint32_t xs = tc_smem_addr(base), ts = tc_smem_addr(base + Gm::kT);
    bool ok = true;
    if (tid == 0) ok &= mbar_wait(&bar_t, 0, a.err);
    uint32_t it = 0;
    for (int img = blockIdx.x; img < nimg; img += gridDim.x, ++it) {
        const unsigned long long t0 = a.trace ? trace_now() : 0;
        const int nxt = img + (int)gridDim.x;
        // pass 1 (one thread): x [T_hi; T_lo]^T into columns 0..63, each K chunk
        // as it lands
        if (tid == 0) {
            constexpr uint32_t id = idesc_tf32(64);
            for (int kc = 0; kc < Gm::KC; ++kc) {
                ok &= mbar_wait(&bar_x[kc], it, a.err);
                tc_after_sync();
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_tf32(tmem, desc_sw128(xs + kc * Gm::kTile + s4 * 32),
                             desc_sw128(ts + kc * Gm::kTChunk + s4 * 32), id,
                             (kc | s4) ? 1u : 0u);
            }
            mma_commit(&bar_p1[0]);
        }
        ok &= mbar_wait(&bar_p1[0], it, a.err);                // pass 1 has read the image
        // x_lo over the image (elementwise: the swizzled layout carries over)
        {
            float4 *xv = reinterpret_cast<float4 *>(base);
            for (int e = tid; e < (int)(Gm::kXBytes / 16); e += NT) {
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
            for (int kc = 0; kc < Gm::KC; ++kc)
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_tf32(tmem, desc_sw128(xs + kc * Gm::kTile + s4 * 32),
                             desc_sw128(ts + kc * Gm::kTChunk + s4 * 32), id, 1u);
        }
        if (tid == 0) mma_commit(&bar_fin);
        ok &= mbar_wait(&bar_fin, it, a.err);
        tc_after_sync();
        const unsigned long long t_z = a.trace ? trace_now() : 0;   // the row DFT is done
        // Z planes from tensor memory over chunk 3: warps w and w + 4 read
        // the same lanes, the first the re, the second the im bins, each summing
        // the T_hi and T_lo column halves
        float *zr = reinterpret_cast<float *>(base + Gm::kZOff);
        float *zi = zr + Gm::N0 * Gm::ZS;
        {
            const int half = warp >> 2, row = 32 * (warp & 3) + (tid & 31);
            const uint32_t lanes = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
            float v[16], u[16];
            tmem_ld16(lanes + half * Gm::M1, v);
            tmem_ld16(lanes + 32 + half * Gm::M1, u);
            float *dz = half ? zi : zr;
#pragma unroll
            for (int q = 0; q < 16; ++q) dz[row * Gm::ZS + (q ^ (row & 15))] = ok ? v[q] + u[q] : 0.f;
        }
        tc_before_sync();
        __syncthreads();
        // chunks 0..2 and tensor memory are free: most of the next image
        if (tid == 0 && nxt < nimg)
            for (int kc = 0; kc < Gm::KC - 1; ++kc) issue(nxt, kc);
        // column DFT in place: thread (r1, k) replaces Z rows r1 + R1 r2 of bin
        // k by S[r1][q][k] = the B2-point DFT over r2 (row r1 + R1 q)
        for (int u = tid; u < Gm::R1 * Gm::M1; u += NT) {
            const int r1 = u / Gm::M1, k = u % Gm::M1;
            float2 z[Gm::B2];
#pragma unroll
            const int kc = k ^ r1;                        // rows r1 + R1 r2: r % 16 = r1
            for (int r2 = 0; r2 < Gm::B2; ++r2) {
                const int r = r1 + Gm::R1 * r2;
                z[r2] = make_float2(zr[r * Gm::ZS + kc], zi[r * Gm::ZS + kc]);
            }
            fft::fft_dif<Gm::B2, -1>(z);
#pragma unroll
            for (int q = 0; q < Gm::B2; ++q) {
                const int r = r1 + Gm::R1 * q;
                const float2 sv = z[fft::bitrev(q, fft::ilog2(Gm::B2))];
                zr[r * Gm::ZS + kc] = sv.x;
                zi[r * Gm::ZS + kc] = sv.y;
            }
        }
        __syncthreads();
        // kept modes: X[j][k] = sum_r1 W_N0^{f r1} S[r1][f mod B2][k]
        float2 *dst = a.part + (size_t)img * Gm::NK;
        for (int o = tid; o < Gm::NK; o += NT) {
            const int j = o / Gm::M1, k = o % Gm::M1;
            const int f = j < Gm::M0 ? j : Gm::N0 - Gm::K0 + j;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int r1 = 0; r1 < Gm::R1; ++r1) {
                const int r = r1 + Gm::R1 * (f % Gm::B2);
                cmac(acc, make_float2(zr[r * Gm::ZS + (k ^ r1)], zi[r * Gm::ZS + (k ^ r1)]),
                     tw[(f * r1) & (Gm::N0 - 1)]);
            }
            __stcg(dst + o, acc);
        }
        fence_async_smem();
        __syncthreads();
        // chunk 3 is free: the rest of the next image
        if (tid == 0 && nxt < nimg) issue(nxt, Gm::KC - 1);
        if (a.trace) cta_record_at(a, 0, 0, img, t0, t0, t_z);
    }
    tc_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(Gm::kTmemCols));
    }
}

// Host: kernel A's fp32 operand image, per K chunk [T_hi | T_lo] with T[j][n] =
// cos(2 pi k n / 128) (j = k < 16) or -sin (j = 16 + k), split in double.
void make_table32(std::vector<unsigned char> &img) {
    using Gm = Geo32;
    using tcu::sw_off;
    using tcu::tf32_lo;
    img.assign(Gm::kTBytes, 0);
    const double two_pi = 2.0 * M_PI;
    for (int j = 0; j < 2 * Gm::M1; ++j)
        for (int n = 0; n < Gm::N1; ++n) {
            const int k = j % Gm::M1;
            const double ang = two_pi * (double)k * (double)n / (double)Gm::N1;
            const double v = j < Gm::M1 ? std::cos(ang) : -std::sin(ang);
            const float hi = (float)v;
            const float lo = (float)(v - (double)(hi - tf32_lo(hi)));
            const uint32_t chunk = (uint32_t)(n / 32) * Gm::kTChunk;
            memcpy(&img[chunk + sw_off(j, n % 32)], &hi, 4);
            memcpy(&img[chunk + sw_off(2 * Gm::M1 + j, n % 32)], &lo, 4);
        }
}

// Host: the 16-bit twiddle operand in its swizzled shared-memory image,
// computed in double and rounded once.
template <typename T>
void make_table(std::vector<unsigned char> &img) {
    using Gm = Geo<T>;
    using tcu::sw_off16;
    img.assign(Gm::kTBytes, 0);
    const double two_pi = 2.0 * M_PI;
    for (int j = 0; j < Gm::N; ++j)
        for (int n = 0; n < Gm::N1; ++n) {
            const int k = j % Gm::M1;
            const double ang = two_pi * (double)k * (double)n / (double)Gm::N1;
            const double v = j < Gm::M1 ? std::cos(ang) : -std::sin(ang);
            const uint32_t chunk = (uint32_t)(n / Gm::kE) * Gm::kTChunk;
            const uint32_t off = chunk + sw_off16(j, n % Gm::kE);
            const T h = std::is_same<T, __half>::value ? T(__float2half_rn((float)v))
                                                       : T(__float2bfloat16_rn((float)v));
            memcpy(&img[off], &h, 2);
        }
}

// ---------------------------------------------------------------------------
// Kernel C on the tensor cores for fp32 128 x 128 layers (16 x 16 modes per
// block): one CTA inverts a whole output image, two CTAs per SM.
//   1. column inverse on the SIMT cores.  The kept rows are the signed
//      frequencies g = -16 .. 15; with g = g1 + 8 g2 (g1 = 0..7, g2 = -2..1) and
//      t = t1 + 16 t2, Zo[t][k] = sum_g V[g][k] e^{+2 pi i g t / 128} becomes
//      U[g1][t1][k] = sum_g2 V[g1 + 8 g2][k] e^{+2 pi i (g1 + 8 g2) t1 / 128}
//      (four terms) followed by 8-point inverse register FFTs over g1 for
//      every (t1, k);
//   2. row inverse as the GEMM y = Zo' . T^T with Zo' = [Re Zo | Im Zo] (K = 32)
//      and T[n] = s [c(k) cos(2 pi k n / 128) | -c(k) sin(...)], s = 1/128^2, in
//      three kind::tf32 passes (Zo_hi T_hi + Zo_hi T_lo + Zo_lo T_hi, hi/lo the
//      tf32 head of a float and the exact remainder), N = 128 outputs in tensor
//      memory;
//   3. the 128 x 128 tile leaves through four swizzled 32-column staging boxes
//      (over the operands, free once the MMAs completed) by TMA stores.
// ---------------------------------------------------------------------------
// kFused: the two column steps in one pass per thread (no U buffer in shared
// memory, three CTAs per SM) -- for layers with many output images; the
// two-pass form spreads the column inverse over more independent work per CTA
// and is faster when there are at most two CTAs per SM anyway.
template <bool kFused>
struct GeoC32 {
    static constexpr int N0 = 128, N1 = 128, M0 = 16, M1 = 16, K0 = 32, NK = K0 * M1;
    static constexpr int G1 = 8, T1 = N0 / G1;          // g = g1 + 8 g2, t = t1 + 16 t2
    static constexpr uint32_t kTile = 16384;            // 128 rows x 128 bytes
    static constexpr uint32_t kT = 0;                   // T hi, T lo (B operands)
    static constexpr uint32_t kTBytes = 2 * kTile;
    static constexpr uint32_t kA = kT + kTBytes;        // Zo' hi, Zo' lo (A operands)
    static constexpr uint32_t kS = kA + 2 * kTile;      // U[G1][T1][M1] (two-pass form)
    static constexpr uint32_t kY = kS + (kFused ? 0 : G1 * T1 * M1 * 8);
    static constexpr uint32_t kTw = kY + NK * 8;
    static constexpr uint32_t kSmem = kTw + N0 * 8 + 1024;
    static constexpr uint32_t kStage = 0;               // 4 output boxes over T and A
    static constexpr uint32_t kTmemCols = 128;
    static_assert(kS >= 4 * kTile, "staging boxes fit over the operands");
};

template <bool kFused>
__global__ void __launch_bounds__(NT, kFused ? 3 : 2)
k_phase_c_tc32(const __grid_constant__ CUtensorMap ymap, Args a, const void *table) {
    using Gm = GeoC32<kFused>;
    using namespace tcu;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_t, bar_mma;
    __shared__ uint32_t s_tmem;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int img = blockIdx.x;
    float2 *ys = reinterpret_cast<float2 *>(base + Gm::kY);
    float2 *tw = reinterpret_cast<float2 *>(base + Gm::kTw);
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_t)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_mma)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(tc_smem_addr(&bar_t)), "r"(Gm::kTBytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(tc_smem_addr(base + Gm::kT)), "l"(table), "r"(Gm::kTBytes),
                     "r"(tc_smem_addr(&bar_t)) : "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(Gm::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    for (int e = tid; e < Gm::N0; e += NT) tw[e] = a.tw0[e];
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    pdl_wait();                                  // kernel B's mixed modes are complete
    pdl_trigger();                               // a dependent kernel may set itself up
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    const float2 *src = a.Y + (size_t)img * Gm::NK;
    for (int e = tid; e < Gm::NK / 2; e += NT) cp_async16(ys + 2 * e, src + 2 * e);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    char *Ahi = base + Gm::kA, *Alo = Ahi + Gm::kTile;
    // Zo[t][k] split into the tf32 head and remainder, written as the K-major
    // operands: columns 0..15 the real parts, 16..31 the imaginary
    auto put = [&](int t, int k, float2 v) {
        const uint32_t ore = sw_off(t, k), oim = sw_off(t, Gm::M1 + k);
        *reinterpret_cast<float *>(Ahi + ore) = v.x;
        *reinterpret_cast<float *>(Ahi + oim) = v.y;
        *reinterpret_cast<float *>(Alo + ore) = tf32_lo(v.x);
        *reinterpret_cast<float *>(Alo + oim) = tf32_lo(v.y);
    };
    if constexpr (kFused) {
        // thread (t1, k): the eight U[g1] (four-term sums, kept row j holds g = j
        // for j < 16, j - 32 above), then the 8-point inverse FFT over g1
        for (int u = tid; u < Gm::T1 * Gm::M1; u += NT) {
            const int k = u % Gm::M1, t1 = u / Gm::M1;
            float2 z[Gm::G1];
#pragma unroll
            for (int g1 = 0; g1 < Gm::G1; ++g1) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int g2 = -2; g2 < 2; ++g2) {
                    const int g = g1 + 8 * g2, j = g < 0 ? g + Gm::K0 : g;
                    const float2 wv = tw[(g * t1) & (Gm::N0 - 1)];   // e^{-2 pi i g t1 / 128}
                    cmac(acc, ys[j * Gm::M1 + k], make_float2(wv.x, -wv.y));
                }
                z[g1] = acc;
            }
            fft::fft_dif<Gm::G1, 1>(z);
#pragma unroll
            for (int t2 = 0; t2 < Gm::G1; ++t2)
                put(t1 + Gm::T1 * t2, k, z[fft::bitrev(t2, fft::ilog2(Gm::G1))]);
        }
    } else {
        float2 *S = reinterpret_cast<float2 *>(base + Gm::kS);
        // 1. U[g1][t1][k0..k0+3]: kept row j holds g = j (j < 16) or j - 32
        for (int u = tid; u < Gm::G1 * Gm::T1 * (Gm::M1 / 4); u += NT) {
            const int k0 = 4 * (u % (Gm::M1 / 4)), t1 = (u / (Gm::M1 / 4)) % Gm::T1;
            const int g1 = u / (Gm::M1 / 4 * Gm::T1);
            float2 acc[4];
    #pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
    #pragma unroll
            for (int g2 = -2; g2 < 2; ++g2) {
                const int g = g1 + 8 * g2, j = g < 0 ? g + Gm::K0 : g;
                const float2 wv = tw[(g * t1) & (Gm::N0 - 1)];        // e^{-2 pi i g t1 / 128}
                const float2 wc = make_float2(wv.x, -wv.y);
                const float4 *y4 = reinterpret_cast<const float4 *>(ys + j * Gm::M1 + k0);
                const float4 p0 = y4[0], p1 = y4[1];
                cmac(acc[0], make_float2(p0.x, p0.y), wc);
                cmac(acc[1], make_float2(p0.z, p0.w), wc);
                cmac(acc[2], make_float2(p1.x, p1.y), wc);
                cmac(acc[3], make_float2(p1.z, p1.w), wc);
            }
            float4 *d = reinterpret_cast<float4 *>(S + (g1 * Gm::T1 + t1) * Gm::M1 + k0);
            d[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
            d[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
        }
        __syncthreads();
        // 2. Zo[t1 + 16 t2][k] = sum_g1 e^{+2 pi i g1 t2 / 8} U[g1][t1][k], split into the
        //    tf32 head and remainder and written as the K-major operands: columns
        //    0..15 the real parts, 16..31 the imaginary
        for (int u = tid; u < Gm::T1 * Gm::M1; u += NT) {
            const int k = u % Gm::M1, t1 = u / Gm::M1;
            float2 z[Gm::G1];
    #pragma unroll
            for (int g1 = 0; g1 < Gm::G1; ++g1) z[g1] = S[(g1 * Gm::T1 + t1) * Gm::M1 + k];
            fft::fft_dif<Gm::G1, 1>(z);
    #pragma unroll
            for (int t2 = 0; t2 < Gm::G1; ++t2) {
                const float2 v = z[fft::bitrev(t2, fft::ilog2(Gm::G1))];
                put(t1 + Gm::T1 * t2, k, v);
            }
        }
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();
    bool ok = mbar_wait(&bar_t, 0, a.err);
    if (tid == 0) {
        tc_after_sync();
        constexpr uint32_t id = idesc_tf32(Gm::N1);
        const uint32_t ah = tc_smem_addr(Ahi), al = tc_smem_addr(Alo);
        const uint32_t th = tc_smem_addr(base + Gm::kT), tl = th + Gm::kTile;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            mma_tf32(tmem, desc_sw128(ah + s * 32), desc_sw128(th + s * 32), id, s ? 1u : 0u);
            mma_tf32(tmem, desc_sw128(ah + s * 32), desc_sw128(tl + s * 32), id, 1u);
            mma_tf32(tmem, desc_sw128(al + s * 32), desc_sw128(th + s * 32), id, 1u);
        }
        mma_commit(&bar_mma);
    }
    ok &= mbar_wait(&bar_mma, 0, a.err);
    tc_after_sync();
    const unsigned long long t_m = a.trace ? trace_now() : 0;
    // 3. warp w reads lanes 32 (w % 4).. of tensor memory (the image rows), the two
    //    warp halves columns 0..63 and 64..127, into boxes 2h and 2h + 1
    {
        const int half = warp >> 2, lrow = 32 * (warp & 3) + (tid & 31);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * half + 16 * g, v);
            char *box = base + Gm::kStage + (2 * half + (g >> 1)) * Gm::kTile;
            const int col0 = 16 * (g & 1);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float4 *>(box + sw_off(lrow, col0 + 4 * q)) =
                    ok ? make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3])
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();
    if (tid == 0) {
        for (int b = 0; b < 4; ++b)
            tma_store_2d(&ymap, 32 * b, img * Gm::N0,
                         tc_smem_addr(base + Gm::kStage + b * Gm::kTile));
        bulk_commit();
        bulk_wait_read();                        // the staging boxes may be released
    }
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(Gm::kTmemCols));
    }
    cta_record(a, 2, a.trace_c, t0, t1, t_m);   // compute: the row-inverse MMAs are done
}

// Host: the fp32 inverse row-DFT operand, [hi, lo][n][k] (k < 16: cos, else
// -sin), with c(k) and the output scale 1/128^2 folded in, computed in double.
void make_table_c32(std::vector<unsigned char> &img) {
    using Gm = GeoC32<false>;
    using tcu::sw_off;
    using tcu::tf32_lo;
    img.assign(Gm::kTBytes, 0);
    const double two_pi = 2.0 * M_PI, s = 1.0 / ((double)Gm::N0 * (double)Gm::N1);
    for (int n = 0; n < Gm::N1; ++n)
        for (int k = 0; k < Gm::M1; ++k) {
            const double ck = (k == 0 || 2 * k == Gm::N1) ? 1.0 : 2.0;
            const double ang = two_pi * (double)k * (double)n / (double)Gm::N1;
            const double v[2] = {s * ck * std::cos(ang), -s * ck * std::sin(ang)};
            for (int h = 0; h < 2; ++h) {
                const float hi = (float)v[h];
                const float lo = (float)(v[h] - (double)(hi - tf32_lo(hi)));
                const uint32_t off = sw_off(n, h * Gm::M1 + k);
                memcpy(&img[off], &hi, 4);
                memcpy(&img[Gm::kTile + off], &lo, 4);
            }
        }
}

}  // namespace tca

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// 128 x 128 grid, 16 x 16 modes per block: chunks of 32 strided rows,
// 16-point row FFTs (8 partial sums per bin), 8-point column FFTs.
using Cfg128 = Cfg<128, 128, 16, 16, 32, 16, 8>;

bool is_cfg128(const Geom &g) {
    return g.d == 2 && g.n[0] == 128 && g.n[1] == 128 && g.m[0] == 16 && g.m[1] == 16;
}

struct BShape {
    int ob;     // outputs per phase-B item
    int bg;     // batch rows per group
};

// Batch groups of about batch/kTargetGroups rows; outputs per phase-B item so
// that the weight slab fits kWsBudget and the group's partials fit kXpBudget.
BShape b_shape(fno_dtype_t dt, int64_t batch, int cin, int cout) {
    const size_t w2 = dt == FNO_F32 ? 16 : 8;
    BShape s;
    s.ob = cout;
    while (s.ob > 1 && (size_t)cin * s.ob * w2 > kWsBudget) s.ob = (s.ob + 1) / 2;
    s.bg = (int)((batch + kTargetGroups - 1) / kTargetGroups);
    while (s.bg > 1 && (size_t)Cfg128::C * s.bg * cin * 16 > kXpBudget) s.bg = (s.bg + 1) / 2;
    while ((batch + s.bg - 1) / s.bg > kMaxGroups) ++s.bg;
    return s;
}

size_t smem_bytes(fno_dtype_t dt, int cin, const BShape &s) {
    const size_t w2 = dt == FNO_F32 ? 16 : 8;
    const size_t b = ((size_t)cin * s.ob * w2 + 15) / 16 * 16 + (size_t)Cfg128::C * s.bg * cin * 16;
    size_t m = Cfg128::kSmemA > Cfg128::kSmemC ? Cfg128::kSmemA : Cfg128::kSmemC;
    m = m > b ? m : b;
    return Cfg128::kSmemTw + m;
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
    return reinterpret_cast<void *>(&k_fused2d<Cfg128, T>);
}

// ----- tensor-core variant: host side -----
using tcu::encoder;
using tcu::EncodeTiled;


// Self-test of the two bounded waits the fused kernels use.  which 0: thread 0
// waits on a flag word that nothing sets (the form CTAs use to wait for a
// phase of another CTA); which 1: thread 0 waits on phase 0 of an mbarrier
// that nothing arrives on (the form the tensor-core kernels use for TMA and
// MMA completion).  Each wait must give up within its limit, set the error
// word to the time-out code and return, leaving the context usable.
__global__ void k_wait_check(const int *never_set, int *err, int which) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    if (which == 0) {
        wait_flag(never_set, err);
    } else {
        const uint32_t a = tcu::tc_smem_addr(&bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tcu::mbar_wait(&bar, 0, err);
        asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(a) : "memory");
    }
}

}  // namespace

cudaError_t launch_wait_check(const Plan &p, int which, cudaStream_t s) {
    // the flag is a word of the error line that no kernel writes
    const int *never_set = p.dev_err + kLine / 2;
    k_wait_check<<<1, 32, 0, s>>>(never_set, p.dev_err, which);
    return cudaGetLastError();
}

size_t fused_sync_bytes() { return kSyncBytes; }

// 256 x 256 grid, 32 x 32 modes per block: chunks of 64 strided rows, 32-point
// row FFTs (8 partial sums per bin), 8-point column FFTs; the four chunk-CTAs
// of an image reduce their partial modes in a cluster.
using Cfg256 = Cfg<256, 256, 32, 32, 64, 32, 8>;

bool is_cfg256(const Geom &g) {
    return g.d == 2 && g.n[0] == 256 && g.n[1] == 256 && g.m[0] == 32 && g.m[1] == 32;
}

// Three-kernel variant, per shape: whether phase A reduces its partials in a
// cluster, and the kernels' shared memory.
// Whether kernel A runs on the tensor cores for this shape and storage type:
// fp32 128 x 128 (16 x 16 modes) and 16-bit 256 x 256 (32 x 32 modes).
template <class Cf>
bool tca_shape(fno_dtype_t dt) {
    if (dt == FNO_F32)
        return Cf::N0 == 128 && Cf::N1 == 128 && Cf::M0 == 16 && Cf::M1 == 16;
    return Cf::N0 == 256 && Cf::N1 == 256 && Cf::M0 == 32 && Cf::M1 == 32;
}

#ifndef FNO_PDL_XP_BUDGET
#define FNO_PDL_XP_BUDGET (64u << 10)
#endif
constexpr size_t kPdlXpBudget = FNO_PDL_XP_BUDGET;   // kernel B's partial modes (bytes)
// kernel B's weight slab in the three-kernel variants: a whole output block
// per item where it fits (64 -> 64 channels in one item: 256 items of 80 KB on
// the FNO layer, one wave, instead of 1024 items over the four output blocks;
// FNO stack 468 -> 459 us)
#ifndef FNO_PDL_WS_BUDGET
#define FNO_PDL_WS_BUDGET (64u << 10)
#endif
constexpr size_t kPdlWsBudget = FNO_PDL_WS_BUDGET;

// ---------------------------------------------------------------------------
// Kernel B of the float32 128 x 128 layer with the weights brought in by TMA
// (up to 64 channels each way, up to 16 samples, weights in the standard
// layout, kernel A leaving one copy of the kept modes): one CTA per run of
// kR = 4 kept modes of a kept row.  Thread 0 requests the run's whole weight
// block W[blk][i][o][local .. local + 3] (Cin x Cout x 4 modes, up to 128 KB)
// as 4-D TMA boxes of 16 input channels before the CTA waits for kernel A --
// the weights do not depend on it -- and the kept modes of every batch row
// follow from L2 once kernel A is complete; thread (batch group, o, mode
// pair) accumulates its rows from shared memory.
#ifndef FNO_MIX_TMA_EVICT_FIRST
#define FNO_MIX_TMA_EVICT_FIRST 1
#endif
namespace mix2d {
constexpr int kR = 4;                            // kept modes a CTA
constexpr int kI = 16;                           // input channels a box
constexpr int kThreads = 512;
constexpr int kMaxC = 64, kMaxB = 16, kRows = 4; // batch rows a thread
constexpr uint32_t kWBytes = (uint32_t)kMaxC * kMaxC * kR * 8;   // 128 KB
constexpr uint32_t kXBytes = (uint32_t)kMaxB * kMaxC * kR * 8;   // 32 KB
constexpr size_t kSmem = (size_t)kWBytes + kXBytes + 1024;       // + alignment
// batch groups for cout outputs: kNT / (2 cout) >= 4, so kMaxB rows need at
// most kRows rows a thread
static_assert(kThreads / (2 * kMaxC) * kRows >= kMaxB, "rows per thread");
}  // namespace mix2d

template <class Cf>
__global__ void __launch_bounds__(mix2d::kThreads, 1)
k_mix_tma2d(const __grid_constant__ CUtensorMap wmap, Args a) {
    using namespace mix2d;
    using tcu::tc_smem_addr;
    constexpr int NK = Cf::NK;
    static_assert(NK % kR == 0 && Cf::M1 % kR == 0, "a run stays on one kept row");
    extern __shared__ __align__(1024) char smem_raw[];
    // the boxes start on a 1024-byte boundary (TMA destinations)
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    const float *ws = reinterpret_cast<const float *>(smem);            // [i][o][kR] complex
    float2 *xs = reinterpret_cast<float2 *>(smem + kWBytes);            // [b][i][kR]
    __shared__ __align__(8) uint64_t bar_w;
    const int tid = threadIdx.x;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int cin = a.cin, cout = a.cout, nb = a.batch;
    const int mode0 = blockIdx.x * kR;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_w)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // a TMA destination must be aligned: check rather than issue a bad copy
        if ((tc_smem_addr(smem) & 1023u) != 0) {
            raise_dev_error(a.err, kDevBounds);
        } else {
            int blk, local;
            Cf::wmap(mode0, blk, local);
            const int ib = cin < kI ? cin : kI, nbox = (cin + kI - 1) / kI;
            const uint32_t boxb = (uint32_t)kR * 8 * cout * ib;
            tcu::arrive_expect_tx(&bar_w, boxb * nbox);
#if FNO_MIX_TMA_EVICT_FIRST
            // the weights are read once a forward: their lines go first from L2
            const uint64_t pol = tcu::l2_evict_first_policy();
            for (int k = 0; k < nbox; ++k)
                asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::"
                             "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
                             ::"r"(tc_smem_addr(smem + k * boxb)), "l"(&wmap), "r"(2 * local),
                               "r"(0), "r"(k * kI), "r"(blk), "r"(tc_smem_addr(&bar_w)), "l"(pol)
                             : "memory");
#else
            for (int k = 0; k < nbox; ++k)
                asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::"
                             "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
                             ::"r"(tc_smem_addr(smem + k * boxb)), "l"(&wmap), "r"(2 * local),
                               "r"(0), "r"(k * kI), "r"(blk), "r"(tc_smem_addr(&bar_w))
                             : "memory");
#endif
        }
    }
    __syncthreads();
    pdl_trigger();                               // kernel C may set itself up
    pdl_wait();                                  // kernel A's kept modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    for (int e = tid; e < nb * cin * (kR / 2); e += kThreads) {
        const int row = e / (kR / 2), h = e % (kR / 2);   // row = b * cin + i
        cp_async16(xs + row * kR + 2 * h, a.part + (size_t)row * NK + mode0 + 2 * h);
    }
    cp_async_commit();
    cp_async_wait_all();
    const bool ok = tcu::mbar_wait(&bar_w, 0, a.err);
    __syncthreads();
    // thread (bg, o, mp): mode pair mp fastest, then the output, then the batch
    // group; rows b = bg, bg + nbg, ...
    const int nbg = kThreads / (2 * cout);
    const int mp = tid & 1, o = (tid >> 1) % cout, bg = (tid >> 1) / cout;
    if (ok && bg < nbg) {
        float2 acc0[kRows], acc1[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) acc0[q] = acc1[q] = make_float2(0.f, 0.f);
        for (int i = 0; i < cin; ++i) {
            const float4 w = *reinterpret_cast<const float4 *>(ws + ((size_t)i * cout + o) * 8 + 4 * mp);
            const float2 w0 = make_float2(w.x, w.y), w1 = make_float2(w.z, w.w);
#pragma unroll
            for (int q = 0; q < kRows; ++q) {
                const int b = bg + nbg * q;
                if (b < nb) {
                    const float4 x2 =
                        *reinterpret_cast<const float4 *>(&xs[((size_t)b * cin + i) * kR + 2 * mp]);
                    cmac(acc0[q], make_float2(x2.x, x2.y), w0);
                    cmac(acc1[q], make_float2(x2.z, x2.w), w1);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int b = bg + nbg * q;
            if (b < nb)
                __stcg(reinterpret_cast<float4 *>(a.Y + ((size_t)b * cout + o) * NK + mode0 + 2 * mp),
                       make_float4(acc0[q].x, acc0[q].y, acc1[q].x, acc1[q].y));
        }
    }
    cta_record(a, 1, a.trace_b, t0, t1);
}

// Host: the weights of a float32 2-D layer as a 4-D tensor map, [blk][i][o][mode
// (re, im)], boxes of kR modes x Cout x min(16, Cin) x 1 block
template <class Cf>
bool encode_wmap2d(CUtensorMap *map, const void *w, int cin, int cout) {
    using namespace mix2d;
    tcu::EncodeTiled fn = tcu::encoder();
    if (!fn) return false;
    const cuuint64_t e = 4, run = (cuuint64_t)Cf::MBLK * 2;   // floats of one (blk, i, o)
    const cuuint64_t dims[4] = {run, (cuuint64_t)cout, (cuuint64_t)cin, 2};
    const cuuint64_t strides[3] = {run * e, run * e * cout, run * e * cout * cin};
    const cuuint32_t boxd[4] = {(cuuint32_t)kR * 2, (cuuint32_t)cout,
                                (cuuint32_t)(cin < kI ? cin : kI), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(w), dims, strides, boxd,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifndef FNO_MIX_TMA2D
#define FNO_MIX_TMA2D 1
#endif

template <class Cf, class CfC = Cf>
struct Pdl {
    static constexpr bool kCluster = Cf::N0 >= 256;
    static constexpr int kParts = kCluster ? 1 : Cf::C;
    // threads of a kernel-B CTA: the 128 x 128 items are small enough that
    // splitting each over 8 warps shortens the path after kernel A (measured:
    // 23.4 -> 22.3 us on the 8 x 32-channel workload); 4 warps elsewhere
    static constexpr int kBThreads = Cf::N0 == 128 ? 256 : 128;
    // (no CUDA call: sizes are reported before any device work; a plan whose
    // driver lacks the tensor-map encoder fails at creation)
    // Whether kernel A runs on the tensor cores: by default for the shapes that
    // have a tensor-core kernel (FNO_PLAN_SIMT_TRANSFORM opts out)
    static bool use_tca(fno_dtype_t dt, uint32_t flags) {
        if (!tca_shape<Cf>(dt)) return false;
        return (flags & FNO_PLAN_SIMT_TRANSFORM) == 0;
    }
    // Whether kernel C runs on the tensor cores: 16-bit 256 x 256 together with
    // kernel A; fp32 128 x 128 by default (FNO_PLAN_SIMT_TRANSFORM opts out)
    static bool use_tcc(fno_dtype_t dt, uint32_t flags) {
        if (!tca_shape<CfC>(dt) || (flags & FNO_PLAN_SIMT_TRANSFORM)) return false;
        return dt == FNO_F32 ? true : use_tca(dt, flags);
    }
    // partial copies of the kept modes kernel A leaves (one from the tensor-core kernel)
    static int parts(fno_dtype_t dt, uint32_t flags) { return use_tca(dt, flags) ? 1 : kParts; }
    static int batch_block(int64_t batch, int cin, int np) {
        int bb = (int)batch;
        while (bb > 1 && (size_t)np * bb * cin * 16 > kPdlXpBudget) bb = (bb + 1) / 2;
        return bb;
    }
    static size_t smem_b(fno_dtype_t dt, int cin, int ob, int bb, int np) {
        const size_t w2 = dt == FNO_F32 ? 16 : 8;
        return ((size_t)cin * ob * w2 + 15) / 16 * 16 + (size_t)np * bb * cin * 16;
    }
    // the mixing runs on the tensor cores (kernel A then writes 16-bit operand
    // images of the kept modes, kernel B 16-bit mixed modes)
    static bool mix16(const Geom &g, fno_dtype_t dt, int64_t batch, int cin, int cout,
                      uint32_t flags) {
        return dt != FNO_F32 && use_tca(dt, flags) && parts(dt, flags) == 1 &&
               !(flags & FNO_PLAN_SIMT_MIX) &&
               mixtc_supported(g.d, dt, batch, cin, cout, Cf::M1, g.nkept);
    }
    static size_t part_bytes(const Geom &g, int64_t batch, int cin, int cout, fno_dtype_t dt,
                             uint32_t flags) {
        const size_t f32 = (size_t)parts(dt, flags) * batch * cin * g.nkept * sizeof(float2);
        const size_t x16 = mix16(g, dt, batch, cin, cout, flags)
                               ? mixtc_x_bytes(batch, cin, g.nkept) : 0;
        return f32 > x16 ? f32 : x16;
    }
    template <typename T, int NP>
    static void *kernel_b() {
        return reinterpret_cast<void *>(&k_phase_b<Cf, T, NP, kBThreads>);
    }

    template <typename T>
    static cudaError_t init(Plan &p) {
        const size_t w2 = p.dtype == FNO_F32 ? 16 : 8;
        p.fused_tca = use_tca(p.dtype, p.flags);
        const int np = parts(p.dtype, p.flags);
        int ob = p.cout;
        while (ob > 1 && (size_t)p.cin * ob * w2 > kPdlWsBudget) ob = (ob + 1) / 2;
        const int bb = batch_block(p.batch, p.cin, np);
        const size_t sa = Cf::kSmemTw + Cf::kSmemA, sc = CfC::kSmemTw + CfC::kSmemC;
        const size_t sb = smem_b(p.dtype, p.cin, ob + 1, bb, np);   // padded slab rows
        cudaError_t e = raise_smem_limit(k_phase_a<Cf, T, kCluster>, (int)sa);
        if (e == cudaSuccess)
            e = raise_smem_limit(np == 1 ? kernel_b<T, 1>() : kernel_b<T, kParts>(), (int)sb);
        if (e == cudaSuccess)
            e = raise_smem_limit(k_phase_c<CfC, T>, (int)sc);
        if constexpr (!std::is_same<T, float>::value || Cf::N0 == 128) {
            // the 16-bit inverse kernel reads the tensor-core mixing's 16-bit output
            p.fused_tcc = use_tcc(p.dtype, p.flags) &&
                          (p.dtype == FNO_F32 ||
                           mix16(p.g, p.dtype, p.batch, p.cin, p.cout, p.flags));
            if (e == cudaSuccess && (p.fused_tca || p.fused_tcc) && !tcu::encoder())
                e = cudaErrorNotSupported;
            std::vector<unsigned char> img, imgc;
            if (e == cudaSuccess && p.fused_tca) {
                if constexpr (std::is_same<T, float>::value) {
                    e = raise_smem_limit(tca::k_phase_a_tc32, (int)tca::Geo32::kSmem);
                    tca::make_table32(img);
                } else {
                    e = raise_smem_limit(tca::k_phase_a_tc<T>, (int)tca::Geo<T>::kSmem);
                    tca::make_table<T>(img);
                }
            }
            if (e == cudaSuccess && p.fused_tcc) {
                if constexpr (std::is_same<T, float>::value) {
                    // the one-pass form where the output images fill more than
                    // two CTAs per SM
                    p.fused_c1pass = p.batch * p.cout > 2 * (int64_t)p.num_sms;
                    e = p.fused_c1pass
                            ? raise_smem_limit(tca::k_phase_c_tc32<true>,
                                               (int)tca::GeoC32<true>::kSmem)
                            : raise_smem_limit(tca::k_phase_c_tc32<false>,
                                               (int)tca::GeoC32<false>::kSmem);
                    tca::make_table_c32(imgc);
                } else {
                    // the persistent two-GEMM inverse (fno_inv16.cu)
                    e = inv16_init(p.dtype);
                    inv16_make_tables(p.dtype, imgc);
                }
            }
            if (e == cudaSuccess && (p.fused_tca || p.fused_tcc)) {
                const size_t off_c = (img.size() + 255) & ~size_t(255);
                e = cudaMalloc(&p.fused_tables, off_c + imgc.size());
                if (e == cudaSuccess && !img.empty())
                    e = cudaMemcpy(p.fused_tables, img.data(), img.size(),
                                   cudaMemcpyHostToDevice);
                if (e == cudaSuccess && !imgc.empty())
                    e = cudaMemcpy(static_cast<char *>(p.fused_tables) + off_c, imgc.data(),
                                   imgc.size(), cudaMemcpyHostToDevice);
                p.fused_table_c = off_c;
            }
        }
        p.fused_bb = bb;
        p.fused_ob = ob;
        p.fused_smem = sb;             // kernel B's; A and C use their fixed sizes
        p.fused_grid = 0;
        // tensor-core mixing where the kept modes arrive reduced (one copy)
        p.fused_mixtc = mix16(p.g, p.dtype, p.batch, p.cin, p.cout, p.flags);
        if (e == cudaSuccess && p.fused_mixtc) e = mixtc_init(p.dtype);
        // fp32, on request: the 3xTF32 tensor-core mixing where kernel A writes
        // one reduced copy of the kept modes and the weights are in the
        // standard layout
        p.fused_mixtf32 = false;
        if constexpr (std::is_same<T, float>::value)
            p.fused_mixtf32 = (p.flags & FNO_PLAN_TENSOR_EXTRA) && p.fused_tca &&
                              !(p.flags & (FNO_PLAN_SIMT_MIX | FNO_PLAN_PACKED_WEIGHTS)) &&
                              mixtf32_supported(p.batch, p.cin, p.cout, Cf::M1, p.g.nkept);
        if (e == cudaSuccess && p.fused_mixtf32) e = mixtf32_init();
        // fp32 128 x 128 with one copy of the kept modes: the mixing fed by TMA
        // (fused_grid CTAs, one per run of kept modes) where a run's weights are
        // at least 64 KB; with smaller blocks (the 8 x 32-channel layer) the slab
        // kernel measured as fast or faster (7.1 against 8.3 us a launch)
        if constexpr (std::is_same<T, float>::value && Cf::N0 == 128) {
            if (FNO_MIX_TMA2D && e == cudaSuccess && p.fused_tca && !p.fused_mixtf32 &&
                !(p.flags & (FNO_PLAN_SIMT_MIX | FNO_PLAN_PACKED_WEIGHTS)) &&
                p.batch <= mix2d::kMaxB && p.cin <= mix2d::kMaxC && p.cout <= mix2d::kMaxC &&
                p.cin * p.cout >= 2048 && tcu::encoder()) {
                p.fused_grid = Cf::NK / mix2d::kR;
                e = raise_smem_limit(k_mix_tma2d<Cf>, mix2d::kSmem);
            }
        }
        p.mix_image = p.fused_mixtc && (p.flags & FNO_PLAN_PACKED_WEIGHTS) &&
                      mixtc_image_layout(p.cin, p.cout);
        p.fused_bstream = 0;

        if (e == cudaSuccess && (p.flags & FNO_PLAN_TRACE)) {
            const size_t nB = p.fused_mixtc     ? (size_t)mixtc_items(p.g.nkept)
                              : p.fused_mixtf32 ? (size_t)(p.g.nkept / 2)
                              : p.fused_grid    ? (size_t)p.fused_grid
                                                : (size_t)(p.g.nkept / kG) * ((p.cout + ob - 1) / ob) *
                                                      ((p.batch + bb - 1) / bb);
            const size_t nA = (size_t)p.batch * p.cin * (p.fused_tca ? 1 : Cf::C);
            const size_t nC = (size_t)p.batch * p.cout * (p.fused_tcc ? 1 : CfC::C);
            p.trace_records = nA + nC + nB;
            e = cudaMalloc(&p.trace, p.trace_records * sizeof(fno_trace_record_t));
        }
        return e;
    }
    // kernel A alone over nimg images (an ordinary launch; the register-FFT
    // kernel, whose partial-copy count the backward pass's workspace assumes)
    template <typename T>
    static cudaError_t forward_a(const Args &a, int64_t nimg, cudaStream_t s) {
        cudaLaunchAttribute cl;
        cl.id = cudaLaunchAttributeClusterDimension;
        cl.val.clusterDim.x = Cf::C;
        cl.val.clusterDim.y = 1;
        cl.val.clusterDim.z = 1;
        cudaLaunchConfig_t ca = {};
        ca.gridDim = dim3((unsigned)(nimg * Cf::C));
        ca.blockDim = dim3(kNT);
        ca.dynamicSmemBytes = Cf::kSmemTw + Cf::kSmemA;
        ca.stream = s;
        ca.attrs = kCluster ? &cl : nullptr;
        ca.numAttrs = kCluster ? 1 : 0;
        cudaError_t e = cudaLaunchKernelEx(&ca, k_phase_a<Cf, T, kCluster>, a);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    // mixed_only: kernels A and B alone (the caller inverts the mixed modes)
    template <typename T>
    static cudaError_t forward(const Plan &p, Args a, cudaStream_t s, bool mixed_only = false) {
        a.bg = p.fused_bb;
        a.ng = (int)((p.batch + a.bg - 1) / a.bg);
        a.ob = p.fused_ob;
        a.nob = (p.cout + a.ob - 1) / a.ob;
        a.npairs = (int)(p.g.nkept / kG);
        const int nA = (int)p.batch * p.cin * (p.fused_tca ? 1 : Cf::C);
        const int nB = p.fused_mixtc     ? mixtc_items(p.g.nkept)
                       : p.fused_mixtf32 ? (int)(p.g.nkept / 2)
                       : p.fused_grid    ? p.fused_grid
                                         : a.npairs * a.nob * a.ng;
        const int nC = (int)p.batch * p.cout * (p.fused_tcc ? 1 : CfC::C);
        a.trace = p.trace;
        a.trace_b = nA;
        a.trace_c = nA + nB;
        cudaError_t e = cudaSuccess;
        bool done_a = false;
        if constexpr (!std::is_same<T, float>::value || Cf::N0 == 128) {
            if (p.fused_tca) {
                CUtensorMap xmap;
                if constexpr (std::is_same<T, float>::value) {
                    using Gm = tca::Geo32;
                    if (!tcu::encode_rows_tiled(&xmap, a.x, (int64_t)p.batch * p.cin * Gm::N0,
                                                Gm::N1, sizeof(T), 32, tcu::tma_type<T>()))
                        return cudaErrorInvalidValue;
                    // persistent: two CTAs per SM walk the images
                    const int grid = nA < 2 * p.num_sms ? nA : 2 * p.num_sms;
                    tca::k_phase_a_tc32<<<grid, tca::NT, Gm::kSmem, s>>>(xmap, a, p.fused_tables,
                                                                         nA);
                } else {
                    using Gm = tca::Geo<T>;
                    if (!tcu::encode_rows_tiled(&xmap, a.x, (int64_t)p.batch * p.cin * Gm::N0,
                                                Gm::N1, sizeof(T), Gm::kE, tcu::tma_type<T>()))
                        return cudaErrorInvalidValue;
                    // persistent: one CTA per SM walks the images
                    const int grid = nA < p.num_sms ? nA : p.num_sms;
                    tca::k_phase_a_tc<T><<<grid, tca::kNTA, Gm::kSmem, s>>>(xmap, a, p.fused_tables,
                                                                           nA);
                }
                e = cudaGetLastError();
                done_a = true;
            }
        }
        if (!done_a) {
            cudaLaunchAttribute cl;
            cl.id = cudaLaunchAttributeClusterDimension;
            cl.val.clusterDim.x = Cf::C;
            cl.val.clusterDim.y = 1;
            cl.val.clusterDim.z = 1;
            cudaLaunchConfig_t ca = {};
            ca.gridDim = dim3(nA);
            ca.blockDim = dim3(kNT);
            ca.dynamicSmemBytes = Cf::kSmemTw + Cf::kSmemA;
            ca.stream = s;
            ca.attrs = kCluster ? &cl : nullptr;
            ca.numAttrs = kCluster ? 1 : 0;
            e = cudaLaunchKernelEx(&ca, k_phase_a<Cf, T, kCluster>, a);
        }
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(kNT);
        cfg.stream = s;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (p.fused_mixtc) {
            MixTcArgs m;
            m.X = a.part;
            m.w = a.w;
            m.Y = a.Y;
            m.err = a.err;
            m.trace = a.trace;
            m.trace_first = nA;
            m.batch = (int)p.batch;
            m.cin = p.cin;
            m.cout = p.cout;
            m.m0 = Cf::M0;
            m.m1 = Cf::M1;
            m.mblk = (int)Cf::MBLK;
            m.nk = Cf::NK;
            m.packed = p.mix_image ? 2 : a.wpacked;
            m.num_sms = p.num_sms;
            e = mixtc_launch(p.dtype, m, s);
        } else if (p.fused_mixtf32) {
            MixTf32Args m;
            m.X = a.part;
            m.w = static_cast<const float *>(a.w);
            m.Y = a.Y;
            m.err = a.err;
            m.trace = a.trace;
            m.trace_first = nA;
            m.batch = (int)p.batch;
            m.cin = p.cin;
            m.cout = p.cout;
            m.m0 = Cf::M0;
            m.m1 = Cf::M1;
            m.nk = Cf::NK;
            e = mixtf32_launch(m, s);
        } else if (p.fused_grid) {
            if constexpr (std::is_same<T, float>::value && Cf::N0 == 128) {
                CUtensorMap wmap;
                if (!encode_wmap2d<Cf>(&wmap, a.w, p.cin, p.cout)) return cudaErrorInvalidValue;
                cfg.gridDim = dim3((unsigned)p.fused_grid);
                cfg.blockDim = dim3(mix2d::kThreads);
                cfg.dynamicSmemBytes = mix2d::kSmem;
                e = cudaLaunchKernelEx(&cfg, k_mix_tma2d<Cf>, wmap, a);
            }
        } else {
            cfg.gridDim = dim3(nB);
            cfg.blockDim = dim3(kBThreads);
            cfg.dynamicSmemBytes = p.fused_smem;
            if (p.fused_tca)
                e = cudaLaunchKernelEx(&cfg, k_phase_b<Cf, T, 1, kBThreads>, a);
            else
                e = cudaLaunchKernelEx(&cfg, k_phase_b<Cf, T, kParts, kBThreads>, a);
        }
        if (e != cudaSuccess) return e;
        if (mixed_only) return cudaGetLastError();
        cfg.gridDim = dim3(nC);
        cfg.blockDim = dim3(kNT);
        if constexpr (std::is_same<T, float>::value && CfC::N0 == 128) {
            if (p.fused_tcc) {
                using Gc = tca::GeoC32<false>;
                CUtensorMap ymap;
                if (!tcu::encode_rows_tiled(&ymap, a.y, (int64_t)p.batch * p.cout * Gc::N0,
                                            Gc::N1, sizeof(float), 32, tcu::tma_type<float>()))
                    return cudaErrorInvalidValue;
                cfg.blockDim = dim3(tca::NT);
                const void *tab = static_cast<const char *>(p.fused_tables) + p.fused_table_c;
                if (p.fused_c1pass) {
                    cfg.dynamicSmemBytes = tca::GeoC32<true>::kSmem;
                    e = cudaLaunchKernelEx(&cfg, tca::k_phase_c_tc32<true>, ymap, a, tab);
                } else {
                    cfg.dynamicSmemBytes = Gc::kSmem;
                    e = cudaLaunchKernelEx(&cfg, tca::k_phase_c_tc32<false>, ymap, a, tab);
                }
                if (e != cudaSuccess) return e;
                return cudaGetLastError();
            }
        }
        if constexpr (!std::is_same<T, float>::value) {
            if (p.fused_tcc) {
                Inv16Args ia;
                ia.Y = a.Y;
                ia.y = a.y;
                ia.err = a.err;
                ia.trace = a.trace;
                ia.trace_first = a.trace_c;
                const void *tab = static_cast<const char *>(p.fused_tables) + p.fused_table_c;
                return inv16_launch(p.dtype, ia, tab, p.batch * p.cout, p.num_sms, s);
            }
        }
        cfg.dynamicSmemBytes = CfC::kSmemTw + CfC::kSmemC;
        e = cudaLaunchKernelEx(&cfg, k_phase_c<CfC, T>, a);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
};

using Pdl128 = Pdl<Cfg128>;

enum Variant { kVarNone, kVarPdl128, kVarPdl256, kVarPersistent128, kVarPdl3d, kVarOne1d };

// Which fused kernel(s) a description runs on.
Variant variant(const Geom &g, fno_dtype_t dtype, uint32_t flags) {
    if (dtype != FNO_F32 && dtype != FNO_F16 && dtype != FNO_BF16) return kVarNone;
    if (g.d == 1) return kVarOne1d;
    if (fused3d_match(g, dtype)) return kVarPdl3d;
    if (is_cfg256(g)) return kVarPdl256;
    if (!is_cfg128(g)) return kVarNone;
    if ((flags & FNO_PLAN_PERSISTENT) && dtype != FNO_BF16) return kVarPersistent128;
    return kVarPdl128;
}

bool fused_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout,
                     uint32_t flags) {
    const Variant v = variant(g, dtype, flags);
    if (v == kVarNone) return false;
    if (v == kVarPdl3d) return fused3d_supported(g, dtype, batch, cin, cout);
    if (v == kVarOne1d) return fused1d_supported(g, dtype, batch, cin, cout);
    const int C = v == kVarPdl256 ? Cfg256::C : Cfg128::C;
    if (batch * (int64_t)cin * C >= (1 << 30) || batch * (int64_t)cout * C >= (1 << 30))
        return false;
    if (v == kVarPersistent128)
        return smem_bytes(dtype, cin, b_shape(dtype, batch, cin, cout)) <= 200 * 1024;
    // three-kernel variants: a weight slab of one output and one batch row must fit
    const size_t w2 = dtype == FNO_F32 ? 16 : 8;
    return (size_t)cin * w2 <= kWsBudget && (size_t)cin * 16 * Pdl128::kParts <= kXpBudget;
}

size_t fused_workspace_bytes(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout,
                             uint32_t flags) {
    const Variant v = variant(g, dtype, flags);
    if (v == kVarPdl3d) return fused3d_workspace_bytes(g, batch, cin, cout);
    if (v == kVarOne1d) return 0;
    if (v == kVarPersistent128) return layout(g, batch, cin, cout).total;
    const size_t part = v == kVarPdl256 ? Pdl<Cfg256>::part_bytes(g, batch, cin, cout, dtype, flags)
                                        : Pdl128::part_bytes(g, batch, cin, cout, dtype, flags);
    const size_t y = (size_t)batch * cout * g.nkept * sizeof(float2);
    return ((part + 255) & ~size_t(255)) + ((y + 255) & ~size_t(255));
}

int fused_kernel_count(const Geom &g, fno_dtype_t dtype, int64_t, int, int, uint32_t flags) {
    const Variant v = variant(g, dtype, flags);
    return (v == kVarPdl128 || v == kVarPdl256 || v == kVarPdl3d) ? 3 : 1;
}

int fused_modes_parts(const Geom &g, fno_dtype_t dtype, uint32_t flags) {
    switch (variant(g, dtype, flags)) {
        case kVarPdl128: return Pdl128::kParts;
        case kVarPdl256: return Pdl<Cfg256>::kParts;
        case kVarPdl3d: return 1;
        default: return 0;
    }
}

cudaError_t fused_forward_modes(const Plan &p, const void *x, int64_t nimg, float2 *parts,
                                cudaStream_t s) {
    const Variant v = variant(p.g, p.dtype, p.flags);
    if (v == kVarPdl3d) return fused3d_forward_modes(p, x, nimg, parts, s);
    if (v != kVarPdl128 && v != kVarPdl256) return cudaErrorInvalidValue;
    Args a{};
    a.x = x;
    a.part = parts;
    a.tw0 = p.tw[0];
    a.tw1 = p.tw[1];
    a.err = p.dev_err;
    a.batch = (int)nimg;      // images = batch * cin
    a.cin = 1;
    return with_storage(p.dtype, [&](auto t) {
        using T = decltype(t);
        return v == kVarPdl256 ? Pdl<Cfg256>::forward_a<T>(a, nimg, s)
                               : Pdl128::forward_a<T>(a, nimg, s);
    });
}

cudaError_t fused_plan_init(Plan &p) {
    const Variant v = variant(p.g, p.dtype, p.flags);
    if (v == kVarPdl3d) return fused3d_plan_init(p);
    if (v == kVarOne1d) return cudaSuccess;
    if (v == kVarPdl128)
        return with_storage(p.dtype, [&](auto t) { return Pdl128::init<decltype(t)>(p); });
    if (v == kVarPdl256)
        return with_storage(p.dtype, [&](auto t) { return Pdl<Cfg256>::init<decltype(t)>(p); });

    const BShape bs = b_shape(p.dtype, p.batch, p.cin, p.cout);
    const size_t smem = smem_bytes(p.dtype, p.cin, bs);
    void *fn = p.dtype == FNO_F32 ? kernel_ptr<float>() : kernel_ptr<__half>();
    cudaError_t e = raise_smem_limit(fn, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kNT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    p.fused_grid = p.num_sms * per_sm;
    p.fused_smem = smem;
    p.fused_ob = bs.ob;
    p.fused_bb = bs.bg;
    if (p.flags & FNO_PLAN_TRACE) {
        const int ng = (int)((p.batch + bs.bg - 1) / bs.bg);
        p.trace_records = (size_t)p.batch * (p.cin + p.cout) * Cfg128::C +
                          (size_t)ng * (p.g.nkept / kG) * ((p.cout + bs.ob - 1) / bs.ob);
        e = cudaMalloc(&p.trace, p.trace_records * sizeof(fno_trace_record_t));
        if (e != cudaSuccess) return e;
    }
    return cudaMemset(p.sync, 0, kSyncBytes);
}

void fused_plan_release(Plan &p) {
    if (p.fused_tables) cudaFree(p.fused_tables);
    if (p.trace) cudaFree(p.trace);
    p.fused_tables = nullptr;
    p.trace = nullptr;
}

bool fused_mixed_available(const Plan &p) {
    // the mixed modes in float32 (the 16-bit tensor-core mixing writes its own
    // 16-bit layout for the inverse kernel that reads it)
    return p.path == kPathFused && variant(p.g, p.dtype, p.flags) == kVarPdl128 &&
           !p.fused_mixtc && !p.trace;
}

cudaError_t fused_forward_mixed(const Plan &p, const Buffers &b, const float2 **Y,
                                cudaStream_t s) {
    if (!fused_mixed_available(p)) return cudaErrorInvalidValue;
    const size_t part = Pdl128::part_bytes(p.g, p.batch, p.cin, p.cout, p.dtype, p.flags);
    Args a{};
    a.x = b.x;
    a.w = b.w;
    a.y = nullptr;
    a.wpacked = (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0;
    a.part = static_cast<float2 *>(b.ws);
    a.Y = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) + ((part + 255) & ~size_t(255)));
    a.tw0 = p.tw[0];
    a.tw1 = p.tw[1];
    a.err = p.dev_err;
    a.batch = (int)p.batch;
    a.cin = p.cin;
    a.cout = p.cout;
    *Y = a.Y;
    return with_storage(p.dtype, [&](auto t) {
        return Pdl128::forward<decltype(t)>(p, a, s, true);
    });
}

void inverse_row_operand_tf32(std::vector<unsigned char> &img) { tca::make_table_c32(img); }

cudaError_t fused_forward(const Plan &p, const Buffers &b, cudaStream_t s) {
    const Variant v = variant(p.g, p.dtype, p.flags);
    if (v == kVarPdl3d) return fused3d_forward(p, b, s);
    if (v == kVarOne1d) return fused1d_forward(p, b, s);

    if (v == kVarPdl128 || v == kVarPdl256) {
        const size_t part = v == kVarPdl256
                                ? Pdl<Cfg256>::part_bytes(p.g, p.batch, p.cin, p.cout, p.dtype, p.flags)
                                : Pdl128::part_bytes(p.g, p.batch, p.cin, p.cout, p.dtype, p.flags);
        Args a{};
        a.x = b.x;
        a.w = b.w;
        a.y = b.y;
        a.wpacked = (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0;
        a.mix16 = p.fused_mixtc ? 1 : 0;
        a.part = static_cast<float2 *>(b.ws);
        a.Y = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) + ((part + 255) & ~size_t(255)));
        a.tw0 = p.tw[0];
        a.tw1 = p.tw[1];
        a.err = p.dev_err;
        a.batch = (int)p.batch;
        a.cin = p.cin;
        a.cout = p.cout;
        return with_storage(p.dtype, [&](auto t) {
            using T = decltype(t);
            return v == kVarPdl256 ? Pdl<Cfg256>::forward<T>(p, a, s)
                                   : Pdl128::forward<T>(p, a, s);
        });
    }
    const Layout l = layout(p.g, p.batch, p.cin, p.cout);
    Args a{};
    a.x = b.x;
    a.w = b.w;
    a.y = b.y;
    a.wpacked = (p.flags & FNO_PLAN_PACKED_WEIGHTS) ? 1 : 0;
    a.part = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) + l.part_off);
    a.Y = reinterpret_cast<float2 *>(static_cast<char *>(b.ws) + l.y_off);
    a.sync = reinterpret_cast<SyncBlock *>(p.sync);
    a.tw0 = p.tw[0];
    a.tw1 = p.tw[1];
    a.err = p.dev_err;
    a.trace = p.trace;
    a.batch = (int)p.batch;
    a.cin = p.cin;
    a.cout = p.cout;
    a.bg = p.fused_bb;
    a.ng = (int)((p.batch + a.bg - 1) / a.bg);
    a.npairs = (int)(p.g.nkept / kG);
    a.ob = p.fused_ob;
    a.nob = (p.cout + a.ob - 1) / a.ob;
    {
        // phase-A tickets are the first ones of each batch group's A segment;
        // spread the weight bytes over the first nA tickets in 16-byte units
        const size_t nA = (size_t)p.batch * p.cin * Cfg128::C;
        a.wbytes = p.weight_bytes;
        a.wslice = kWeightPrefetch ? (unsigned)(((p.weight_bytes + nA - 1) / nA + 15) / 16 * 16) : 0u;
    }
    const int total = (int)p.batch * (p.cin + p.cout) * Cfg128::C + a.ng * a.npairs * a.nob;
    const int grid = p.fused_grid < total ? p.fused_grid : total;
    if (p.dtype == FNO_F32)
        k_fused2d<Cfg128, float><<<grid, kNT, p.fused_smem, s>>>(a);
    else
        k_fused2d<Cfg128, __half><<<grid, kNT, p.fused_smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace fno
