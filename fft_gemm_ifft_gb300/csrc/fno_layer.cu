// fno_layer.cu -- the output half of an FNO layer (128 x 128 grid, 16 x 16
// kept modes per block; activations in float32 or a 16-bit storage type,
// arithmetic in float32): the inverse transform of the mixed modes, the 1x1
// linear of the layer's input, bias and GELU, without writing the spectral
// branch out.
//
// The layer is the one of the TurboFNO article (gsyq.cn/news/457482, §5):
// out = GELU(K(x) + W x + b), K(x) the spectral convolution (truncated forward
// real FFT, per-mode mixing, zero-padded inverse real FFT).  The inverse real
// DFT of the mixed modes Y[j][k] (kept rows j <-> frequency g(j) = j or j - 32,
// kept columns k < 16) is
//   K(x)[t][n] = s sum_k c(k) Re( Z[t][k] e^{+2 pi i k n / 128} ),
//   Z[t][k]    = sum_j Y[j][k] e^{+2 pi i g(j) t / 128},
// with s = 1 / 128^2, c(0) = 1 and c(k) = 2 otherwise (the Hermitian half;
// the imaginary part of the k = 0 column drops out as in any real inverse).
// For one image row t and all output channels o the row step and the 1x1
// linear are one GEMM with concatenated K:
//   D[n][o] = sum_{k' < 32} T[n][k'] Zr[o][k']  +  sum_i x[i][t][n] W[o][i],
// T[n][k] = s c(k) cos(2 pi k n / 128), T[n][16 + k] = -s c(k) sin(...),
// Zr[o][k] = Re Z_o[t][k], Zr[o][16 + k] = Im Z_o[t][k].
//
// Kernel 1 (k_colinv) computes Z for every (batch, channel) image -- the
// column step -- and stores it split for 3xTF32 as rows [b][t][hi, lo][o][32]
// (hi = the value, lo = its remainder below tf32), so that one image row's
// coefficients for all channels are one contiguous 128-byte-wide box: the
// B operand [Zr_hi; Zr_lo] stacked along N.
// Kernel 2 (k_layer_gemm) walks tiles (b, t) of 128 pixels persistently, one
// CTA per SM, with specialised warps as the 1x1-linear kernel
// (fno_pointwise.cu): a load warp brings the tile's activations [C][128] and
// its coefficients Zr (a 128-byte-swizzled box = the K-major B operand) into a
// ring of slots by TMA; 8 transposer warps move the activations one K chunk
// of 32 channels at a time into the K-major A operand (3xTF32: hi = the value,
// lo = its exact remainder below tf32) and split Zr; an MMA warp issues the
// spectral K chunk (A = T, a constant operand) and the channel chunks into one
// of two tensor-memory accumulators and hands the slot back to the load warp
// when the tile's MMAs are done; 8 epilogue warps apply bias and GELU to a
// finished accumulator and store it, under the next tiles' transposes and
// MMAs.  The spectral branch never reaches global memory.
#include "fno_layer.cuh"

#include <type_traits>

#include "fno_fft.cuh"
#include "fno_gelu.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

constexpr int kN0 = 128;        // grid rows and columns
constexpr int kM1 = 16;         // kept columns
constexpr int kK0 = 32;         // kept rows (two blocks of 16)
constexpr int kZW = 2 * kM1;    // a row's coefficients: 16 real parts, then 16 imaginary

__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Kernel 1: Z[b][t][h][o][k | 16 + k] = Re | Im sum_j Y[b][o][j][k] e^{+2 pi i g(j) t / 128},
// h = 0 the value, h = 1 its remainder below tf32.
// One CTA per image; thread (t1, k), t1 < 16: the eight partial sums
// U[g1] = sum_{g2 = -2..1} Y[g1 + 8 g2][k] e^{+2 pi i (g1 + 8 g2) t1 / 128}
// (the kept frequencies g = g1 + 8 g2 run over -16..15), then the 8-point
// inverse DFT over g1 gives Z[t1 + 16 t2][k] for t2 < 8.
// ---------------------------------------------------------------------------
constexpr int kColThreads = 256;

__global__ void __launch_bounds__(kColThreads) k_colinv(const float2 *__restrict__ Y,
                                                        const float2 *__restrict__ tw,
                                                        float *__restrict__ Z, int width) {
    __shared__ __align__(16) float2 ys[kK0 * kM1];
    __shared__ float2 tws[kN0];
    const int tid = threadIdx.x, img = blockIdx.x;
    if (tid < kN0) tws[tid] = tw[tid];
    grid_wait();                                  // the mixing kernel's modes are complete
    grid_trigger();                               // the GEMM kernel may set itself up
    reinterpret_cast<float4 *>(ys)[tid] =
        reinterpret_cast<const float4 *>(Y + (size_t)img * kK0 * kM1)[tid];
    __syncthreads();
    const int k = tid % kM1, t1 = tid / kM1;
    float2 z[8];
#pragma unroll
    for (int g1 = 0; g1 < 8; ++g1) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int g2 = -2; g2 < 2; ++g2) {
            const int g = g1 + 8 * g2, j = g < 0 ? g + kK0 : g;
            const float2 w = tws[(g * t1) & (kN0 - 1)];           // e^{-2 pi i g t1 / 128}
            fft::cmac(acc, ys[j * kM1 + k], make_float2(w.x, -w.y));
        }
        z[g1] = acc;
    }
    fft::fft_dif<8, 1>(z);
    const int b = img / width, o = img % width;
#pragma unroll
    for (int t2 = 0; t2 < 8; ++t2) {
        const float2 v = z[fft::bitrev(t2, 3)];
        float *row = Z + (((size_t)b * kN0 + t1 + 16 * t2) * 2 * width + o) * kZW;
        row[k] = v.x;
        row[kM1 + k] = v.y;
        row[(size_t)width * kZW + k] = tcu::tf32_lo(v.x);
        row[(size_t)width * kZW + kM1 + k] = tcu::tf32_lo(v.y);
    }
}

// ---------------------------------------------------------------------------
// Kernel 2: the GEMM per image row.
// ---------------------------------------------------------------------------
constexpr int kTWarps = 4;                // warps 0..3 move the activations into tensor memory
constexpr int kEWarps = 16;               // warps 4..19 run the epilogue (GELU-bound)
constexpr int kWarps = kTWarps + kEWarps;
constexpr int kCompute = 32 * kWarps;
constexpr int kThreads = kCompute + 96;   // + a load warp and two MMA warps
constexpr int kRows = 128;                // M: the pixels of one image row
constexpr uint32_t kTile = 16384;         // 128 rows x 128 bytes
constexpr int kTmemCols = 512;

// Shared-memory map (offsets from a 1024-aligned base) and tensor-memory
// columns for C channels in and out.  B operands hold hi and lo stacked along
// N (rows 0..C-1 hi, C..2C-1 lo), so that x_hi [B_hi; B_lo] is one MMA of
// N = 2C and x_lo B_hi one of N = C: an MMA of N <= 128 costs about the same
// on these tensor cores whatever N is, and 3xTF32 then takes two per K step.
template <int C, typename T>
struct Lay {
    static constexpr int kKC = C / 32;                          // K chunks of the 1x1 linear
    static constexpr uint32_t kHalf = (uint32_t)C * 128;        // C rows x 128 bytes
    static constexpr uint32_t kW = 0;                           // W chunk c: [hi; lo] at c * 2 kHalf
    static constexpr uint32_t kX = 2 * kKC * kHalf;             // ring: activations [C][128]
    static constexpr uint32_t kXBytes = (uint32_t)(C * kRows * sizeof(T));
    static constexpr int kNX = 4;
    static constexpr uint32_t kZ = kX + kNX * kXBytes;           // ring: Zr [hi; lo] (one box)
    static constexpr uint32_t kZBytes = 2 * kHalf;
    static constexpr int kNZ = 4;
    static constexpr uint32_t kAlloc = kZ + kNZ * kZBytes + 1024;
    static constexpr uint32_t kLimit = 227u * 1024u;
    static constexpr uint32_t kStatic = 1024;                   // barriers, biases (bound)
    // tensor memory: accumulator b at columns [b 2C, b 2C + 2C) (the hi half,
    // then the lo half), T hi / lo, and three A chunk buffers (hi, lo): chunk
    // q may be written once chunk q - 3's MMAs are done, so that a transpose
    // has a whole tile's MMAs to hide under
    static constexpr uint32_t kTc = 4 * C;                      // T hi, T lo: 32 columns each
    static constexpr uint32_t kAc = kTc + 64;                   // A buffer a: kAc + 64 a (hi, lo)
    static constexpr int kNA = 3;
    static_assert(C == 32 || C == 64, "32 or 64 channels");
    static_assert(kAlloc + kStatic <= kLimit, "shared memory");
    static_assert(kAc + 64 * kNA <= kTmemCols, "tensor memory");
};

struct GParams {
    const float *W, *bias;
    const void *table;
    void *out;                 // [batch][C][128 * 128], storage type
    int64_t ntiles;            // batch x 128 image rows
    int gelu;
    int *err;
};

__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_addr(bar))
                     : "memory");
}
// the same with relaxed semantics: orders no earlier memory accesses (an
// epilogue warp hands its accumulator back after tcgen05.wait::ld, without
// waiting for the global stores of the tile before)
__device__ __forceinline__ void warp_arrive_relaxed(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];"
                     ::"r"(tc_smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

template <int C, typename T>
__global__ void __launch_bounds__(kThreads, 1)
k_layer_gemm(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap zmap,
             const GParams p) {
    using L = Lay<C, T>;
    // 16-bit activations are exact in tf32: no remainder operand, and the
    // channel part needs only a_hi [W_hi; W_lo]
    constexpr bool kLo = std::is_same<T, float>::value;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    // x_full / x_empty: the activation slots (loaded / transposed);
    // z_full / z_empty: the coefficient slots (loaded / read by the MMAs);
    // a_full / a_empty: the A chunk buffers in tensor memory (written /
    // consumed; chunk q of the CTA's sequence, q = j * kKC + c, uses buffer
    // q % kNA); acc_full / acc_empty: the two accumulators
    __shared__ __align__(8) uint64_t x_full[L::kNX], x_empty[L::kNX], z_full[L::kNZ],
        z_empty[L::kNZ], a_full[L::kNA], a_empty[L::kNA], acc_full[2], acc_empty[2];
    __shared__ uint32_t s_tmem;
    __shared__ __align__(16) float s_bias[C];
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        auto init = [](uint64_t *b, uint32_t count) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem_addr(b)),
                         "r"(count));
        };
        for (int k = 0; k < L::kNX; ++k) {
            init(&x_full[k], 1);
            init(&x_empty[k], kTWarps);
        }
        for (int k = 0; k < L::kNZ; ++k) {
            init(&z_full[k], 1);
            init(&z_empty[k], 1);
        }
        for (int k = 0; k < L::kNA; ++k) {
            init(&a_full[k], kTWarps);
            init(&a_empty[k], 1);
        }
        for (int k = 0; k < 2; ++k) {
            init(&acc_full[k], 1);
            init(&acc_empty[k], kEWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    grid_trigger();
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;

    const int64_t nt =
        p.ntiles > (int64_t)blockIdx.x ? (p.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto xslot = [&](int64_t j) { return base + L::kX + (uint32_t)(j % L::kNX) * L::kXBytes; };
    auto zslot = [&](int64_t j) { return base + L::kZ + (uint32_t)(j % L::kNZ) * L::kZBytes; };
    auto acol = [&](int64_t q) { return tmem + L::kAc + 64u * (uint32_t)(q % L::kNA); };

    if (warp == kWarps) {
        // ---- load warp: tile j's activations and coefficients
        if ((tid & 31) == 0) {
            const uint64_t pol = l2_evict_first_policy();       // both are read once
            grid_wait();                                         // Z comes from kernel 1
            for (int64_t j = 0; j < nt; ++j) {
                const int64_t tg = blockIdx.x + j * gridDim.x;   // = b * 128 + t
                const int b = (int)(tg / kN0), t = (int)(tg % kN0);
                const int sx = (int)(j % L::kNX), sz = (int)(j % L::kNZ);
                if (j >= L::kNX) mbar_wait(&x_empty[sx], (uint32_t)(j / L::kNX - 1), p.err);
                arrive_expect_tx(&x_full[sx], L::kXBytes);
                tma_load_2d_hint(tc_smem_addr(xslot(j)), &xmap, t * kRows, b * C, &x_full[sx], pol);
                if (j >= L::kNZ) mbar_wait(&z_empty[sz], (uint32_t)(j / L::kNZ - 1), p.err);
                arrive_expect_tx(&z_full[sz], L::kZBytes);
                tma_load_2d_hint(tc_smem_addr(zslot(j)), &zmap, 0, (int)(tg * 2 * C), &z_full[sz],
                                 pol);
            }
        }
    } else if (warp > kWarps) {
        // ---- MMA warps: warp kWarps + 1 + (j % 2) takes tile j (accumulator
        // j % 2), so that one warp's waits and commits overlap the other's
        // issue (the tensor pipe queues few MMAs); per tile the spectral chunk
        // (with channel chunk 0), then the other channel chunks; per K step
        // A_hi [B_hi; B_lo] (N = 2C) and A_lo B_hi (N = C).  A commit tracks
        // the MMAs of its own thread, and the two warps share no accumulator.
        if ((tid & 31) == 0) {
            constexpr uint32_t id2 = idesc_tf32(2 * C), id1 = idesc_tf32(C);
            const uint32_t w0 = tc_smem_addr(base + L::kW);
            const uint32_t t_hi = tmem + L::kTc, t_lo = t_hi + 32;
            for (int64_t j = warp - (kWarps + 1); j < nt; j += 2) {
                const int buf = (int)(j & 1), sz = (int)(j % L::kNZ);
                const uint32_t zb = tc_smem_addr(zslot(j));
                const uint32_t d = tmem + (uint32_t)buf * 2 * C;
                if (j >= 2) mbar_wait(&acc_empty[buf], (uint32_t)((j - 2) >> 1), p.err);
                mbar_wait(&z_full[sz], (uint32_t)(j / L::kNZ), p.err);
                for (int c = 0; c < L::kKC; ++c) {
                    const int64_t q = j * L::kKC + c;
                    const int ab = (int)(q % L::kNA);
                    mbar_wait(&a_full[ab], (uint32_t)(q / L::kNA), p.err);
                    tc_after_sync();
                    if (c == 0) {
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t zd = desc_sw128(zb + 32 * s);
                            mma_tf32_ts(d, t_hi + 8 * s, zd, id2, s ? 1u : 0u);
                            mma_tf32_ts(d, t_lo + 8 * s, zd, id1, 1u);
                        }
                    }
                    const uint32_t a_hi = acol(q), a_lo = a_hi + 32;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t wd = desc_sw128(w0 + (uint32_t)c * 2 * L::kHalf + 32 * s);
                        mma_tf32_ts(d, a_hi + 8 * s, wd, id2, 1u);
                        if constexpr (kLo) mma_tf32_ts(d, a_lo + 8 * s, wd, id1, 1u);
                    }
                    if (c == 0) mma_commit(&z_empty[sz]);           // Zr has been read
                    if (c == L::kKC - 1) mma_commit(&acc_full[buf]);
                    mma_commit(&a_empty[ab]);
                }
            }
        }
    } else {
        // ---- compute warps, set-up: W as the K-major B operand, chunk c of 32
        // inputs = [hi; lo] (rows = outputs); the biases
        for (int e = tid; e < C * C; e += kCompute) {
            const float w = p.W[e];
            const int o = e / C, i = e % C;
            char *ch = base + L::kW + (uint32_t)(i / 32) * 2 * L::kHalf;
            *reinterpret_cast<float *>(ch + sw_off(o, i % 32)) = w;
            *reinterpret_cast<float *>(ch + L::kHalf + sw_off(o, i % 32)) = tf32_lo(w);
        }
        for (int o = tid; o < C; o += kCompute) s_bias[o] = p.bias[o];
        fence_async_smem();
        compute_sync();
        // thread -> pixel row = tensor-memory lane: warp w works on the lane
        // quarter w % 4
        const int row = 32 * (warp & 3) + (tid & 31);
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        if (warp < kTWarps) {
            // the constant A operand T (the inverse row DFT, hi and lo) into
            // tensor memory: thread = one row's 32 columns
            {
                const char *tab = static_cast<const char *>(p.table);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float hi[16], lo[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const uint32_t off = sw_off(row, 16 * half + u);
                        hi[u] = *reinterpret_cast<const float *>(tab + off);
                        lo[u] = *reinterpret_cast<const float *>(tab + kTile + off);
                    }
                    tmem_st16(tmem + lane_base + L::kTc + 16 * half, hi);
                    tmem_st16(tmem + lane_base + L::kTc + 32 + 16 * half, lo);
                }
            }
            // ---- transposer warps: chunk q of 32 channels into A buffer q % kNA
            // once chunk q - kNA's MMAs are done; thread = the chunk's 32
            // channels of its pixel, i.e. 32 columns of its lane
            for (int64_t j = 0; j < nt; ++j) {
                mbar_wait(&x_full[j % L::kNX], (uint32_t)(j / L::kNX), p.err);
                const T *X = reinterpret_cast<const T *>(xslot(j));
                for (int c = 0; c < L::kKC; ++c) {
                    const int64_t q = j * L::kKC + c;
                    if (q >= L::kNA) {
                        mbar_wait(&a_empty[q % L::kNA], (uint32_t)(q / L::kNA - 1), p.err);
                        tc_after_sync();
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int i0 = 32 * c + 16 * half;
                        float v[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) v[u] = Storage<T>::load(X + (i0 + u) * kRows + row);
                        const uint32_t a = acol(q) + lane_base + 16 * half;
                        tmem_st16(a, v);
                        if constexpr (kLo) {
                            float lo[16];
#pragma unroll
                            for (int u = 0; u < 16; ++u) lo[u] = tf32_lo(v[u]);
                            tmem_st16(a + 32, lo);
                        }
                    }
                    tmem_st_wait();
                    tc_before_sync();
                    warp_arrive(&a_full[q % L::kNA]);
                }
                warp_arrive(&x_empty[j % L::kNX]);               // the activations are read
            }
        } else {
            // ---- epilogue warps: hi half + lo half of accumulator j % 2, bias,
            // GELU, stored straight out (a warp writes 128 consecutive bytes of
            // one output channel per store); thread (row, part) takes C / 4 outputs
            constexpr int kOut = C / 4;
            const int o0 = ((warp - kTWarps) >> 2) * kOut;
            for (int64_t j = 0; j < nt; ++j) {
                const int buf = (int)(j & 1);
                float v[kOut];
                mbar_wait(&acc_full[buf], (uint32_t)(j >> 1), p.err);
                tc_after_sync();
                const uint32_t ta = tmem + lane_base + (uint32_t)buf * 2 * C + (uint32_t)o0;
                if constexpr (kOut == 16) {
                    float u[16], w[16];
                    tmem_ld16(ta, u);
                    tmem_ld16(ta + C, w);
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] = u[q] + w[q];
                } else {
                    float u[8], w[8];
                    tmem_ld8(ta, u);
                    tmem_ld8(ta + C, w);
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = u[q] + w[q];
                }
                tc_before_sync();
                warp_arrive_relaxed(&acc_empty[buf]);
                const int64_t tg = blockIdx.x + j * gridDim.x;
                const int64_t b = tg / kN0, t = tg % kN0;
                T *op = static_cast<T *>(p.out) + (b * C + o0) * (int64_t)(kN0 * kN0) + t * kRows + row;
#pragma unroll
                for (int q4 = 0; q4 < kOut / 4; ++q4) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(&s_bias[o0 + 4 * q4]);
                    float r[4] = {v[4 * q4] + b4.x, v[4 * q4 + 1] + b4.y, v[4 * q4 + 2] + b4.z,
                                  v[4 * q4 + 3] + b4.w};
                    if (p.gelu) {
                        gelu_erf2(r[0], r[1]);
                        gelu_erf2(r[2], r[3]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        Storage<T>::store(op + (int64_t)(4 * q4 + q) * (kN0 * kN0), r[q]);
                }
            }
        }
    }
    tc_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
    }
}

template <int C, typename T>
cudaError_t launch_gemm(const LayerOutArgs &a, int num_sms, cudaStream_t s) {
    using L = Lay<C, T>;
    const int64_t npix = (int64_t)kN0 * kN0;
    CUtensorMap xmap, zmap;
    if (!encode_rows_plain(&xmap, a.x, a.batch * C, npix, sizeof(T), kRows, C, tma_type<T>()) ||
        !encode_rows_tiled(&zmap, a.Z, a.batch * kN0 * 2 * C, kZW, 4, kZW,
                           CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2 * C))
        return cudaErrorInvalidValue;
    GParams gp;
    gp.out = a.out;
    gp.W = a.W;
    gp.bias = a.bias;
    gp.table = a.table;
    gp.ntiles = a.batch * kN0;
    gp.gelu = a.gelu;
    gp.err = a.err;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(gp.ntiles, std::max(num_sms, 1)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_layer_gemm<C, T>, xmap, zmap, gp);
}

}  // namespace

bool layer_out_supported(int width, int64_t batch) {
    if (!tcu::encoder()) return false;
    // Z's rows are addressed as one 32-bit TMA coordinate
    return (width == 32 || width == 64) && batch >= 1 &&
           batch * kN0 * 2 * width < ((int64_t)1 << 31);
}

size_t layer_out_z_bytes(int64_t batch, int width) {
    return (size_t)batch * kN0 * 2 * width * kZW * sizeof(float);
}

cudaError_t layer_out_init(fno_dtype_t dt, int width) {
    return with_storage(dt, [&](auto t) {
        using T = decltype(t);
        return width == 32 ? raise_smem_limit(k_layer_gemm<32, T>, Lay<32, T>::kAlloc)
                           : raise_smem_limit(k_layer_gemm<64, T>, Lay<64, T>::kAlloc);
    });
}

cudaError_t layer_out_launch(const LayerOutArgs &a, int num_sms, cudaStream_t s) {
    if (a.batch < 1) return cudaSuccess;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.batch * a.width));
    cfg.blockDim = dim3(kColThreads);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_colinv, a.Y, a.tw, a.Z, a.width);
    if (e != cudaSuccess) return e;
    e = with_storage(a.dtype, [&](auto t) {
        using T = decltype(t);
        return a.width == 32 ? launch_gemm<32, T>(a, num_sms, s) : launch_gemm<64, T>(a, num_sms, s);
    });
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace fno
