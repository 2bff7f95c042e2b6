// fno_head.cu -- the projection head of the FNO stack as one persistent
// tensor-core kernel (activations and output in float32 or a 16-bit storage
// type, arithmetic in float32).
//
// The head is the two-layer 1x1 projection of the TurboFNO article's model
// (gsyq.cn/news/457482, §5): out = P2 GELU(W a + b) + c2 per pixel, W of
// hidden x cin, P2 of cout2 x hidden.  One tile = 128 pixels of one image; its
// hidden activations are the GEMM D[p][o] = sum_i a[i][p] W[o][i] (M = 128
// pixels, N = hidden, K = cin) in 3xTF32 (hi = the value, lo = its remainder
// below tf32: a_hi W_hi + a_hi W_lo + a_lo W_hi).
//
// One CTA per SM walks the tiles with specialised warps:
// * a load warp brings the activations [cin][128] into a ring by TMA;
// * 4 transposer warps (one per tensor-memory lane quarter; thread = pixel =
//   lane) write a tile's channels, 32 at a time, as tensor-memory columns
//   (hi and lo) -- the A operand -- into one of three chunk buffers;
// * two MMA warps take alternate tiles, each into its own accumulator, so that
//   one warp's waits overlap the other's issue;
// * 16 epilogue warps (4 per lane quarter, a quarter of the hidden units each)
//   add the bias, apply the GELU two values at a time, accumulate the second
//   projection and sum the four parts of a pixel through shared memory into a
//   staging tile;
// * a store warp writes each staging tile out by TMA (the epilogue warps
//   synchronise with one another, and a barrier would wait for their own
//   global stores).
// Every wait is bounded (a time-out sets the plan's error word).
#include "fno_head.cuh"

#include <algorithm>
#include <type_traits>

#include "fno_gelu.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

constexpr int kTWarps = 4;                // warps 0..3: activations into tensor memory
constexpr int kEWarps = 16;               // warps 4..19: the epilogue
constexpr int kWarps = kTWarps + kEWarps;
constexpr int kCompute = 32 * kWarps;
constexpr int kThreads = kCompute + 128;  // + a load warp, two MMA warps, a store warp
constexpr int kRows = 128;                // M: pixels per tile
constexpr int kTmemCols = 512;
constexpr int kNA = 3;                    // A chunk buffers in tensor memory

// Shared memory (offsets from a 1024-aligned base): W chunk c (32 inputs) =
// [hi: H rows x 128 B][lo: H rows x 128 B]; the bias as one more K chunk
// (row o: bias_hi, bias_lo, then zeros), multiplied by a constant A of ones
// in tensor memory so that the accumulator starts at the bias; the
// activation ring; the partial
// second projections of parts 1..3 per tile parity; the output staging tiles
// [2][C2][128]; bias, P2, c2.
template <int C, int H, int C2, typename T>
struct Lay {
    static constexpr int kKC = C / 32;
    static constexpr uint32_t kWHalf = (uint32_t)H * 128;
    static constexpr uint32_t kW = 0;
    static constexpr uint32_t kBias = 2 * kKC * kWHalf;
    static constexpr uint32_t kX = kBias + kWHalf;
    static constexpr uint32_t kXBytes = (uint32_t)(C * kRows * sizeof(T));
    static constexpr uint32_t kRedBytes = 2u * 3u * C2 * kRows * 4;
    static constexpr uint32_t kOutBytes =
        ((uint32_t)(2 * C2 * kRows * sizeof(T)) + 1023u) & ~1023u;   // staging, storage type
    static constexpr uint32_t kParBytes = ((uint32_t)(H + C2 * H + C2) * 4 + 15) & ~15u;
    static constexpr uint32_t kLimit = 227u * 1024u;
    static constexpr uint32_t kStatic = 1024;
    static constexpr int kNXFit =
        (int)((kLimit - kStatic - 1024 - kX - kRedBytes - kOutBytes - kParBytes) / kXBytes);
    static constexpr int kNX = kNXFit < 4 ? kNXFit : 4;
    static constexpr uint32_t kRed = kX + kNX * kXBytes;
    static constexpr uint32_t kOut = kRed + kRedBytes;
    static constexpr uint32_t kPar = kOut + kOutBytes;
    static constexpr uint32_t kAlloc = kPar + kParBytes + 1024;
    static constexpr uint32_t kAc = 2 * H;          // A buffer a at columns kAc + 64 a
    static constexpr uint32_t kOnes = kAc + 64 * kNA;   // 16 columns: 1, 1, 0 ...
    static_assert(C == 32 || C == 64, "32 or 64 inputs");
    static_assert(H == 64 || H == 128, "64 or 128 hidden units");
    static_assert(kNX >= 2, "two activation slots");
    static_assert(kAlloc + kStatic <= kLimit, "shared memory");
    static_assert(kOnes + 16 <= kTmemCols, "tensor memory");
};

struct KParams {
    const float *W, *bias, *P2, *c2;
    void *out;
    int cout2;
    int64_t npix, ptiles, ntiles;
    int *err;
};

__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_addr(bar))
                     : "memory");
}
// relaxed: orders no earlier memory accesses (an epilogue warp hands its
// accumulator back after tcgen05.wait::ld without waiting for its stores)
__device__ __forceinline__ void warp_arrive_relaxed(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];"
                     ::"r"(tc_smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}
// the four epilogue warps of one tensor-memory lane quarter
__device__ __forceinline__ void quarter_sync(int quarter) {
    asm volatile("bar.sync %0, 128;" ::"r"(2 + quarter) : "memory");
}

template <int C, int H, int C2, typename T>
__global__ void __launch_bounds__(kThreads, 1)
k_head(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap omap,
       const KParams p) {
    using L = Lay<C, H, C2, T>;
    // 16-bit activations are exact in tf32: no remainder operand or product
    constexpr bool kLo = std::is_same<T, float>::value;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    // x_full / x_empty: the activation slots; a_full / a_empty: the A chunk
    // buffers (chunk q = j * kKC + c in buffer q % kNA); acc_full / acc_empty:
    // the two accumulators; o_full / o_empty: the two output staging tiles
    __shared__ __align__(8) uint64_t x_full[L::kNX], x_empty[L::kNX], a_full[kNA],
        a_empty[kNA], acc_full[2], acc_empty[2], o_full[2], o_empty[2];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5;
    float *s_bias = reinterpret_cast<float *>(base + L::kPar);
    float *s_p2 = s_bias + H;                    // [C2][H]
    float *s_c2 = s_p2 + C2 * H;

    if (tid == 0) {
        auto init = [](uint64_t *b, uint32_t count) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem_addr(b)),
                         "r"(count));
        };
        for (int k = 0; k < L::kNX; ++k) {
            init(&x_full[k], 1);
            init(&x_empty[k], kTWarps);
        }
        for (int k = 0; k < kNA; ++k) {
            init(&a_full[k], kTWarps);
            init(&a_empty[k], 1);
        }
        for (int k = 0; k < 2; ++k) {
            init(&acc_full[k], 1);
            init(&acc_empty[k], kEWarps);
            init(&o_full[k], 4);
            init(&o_empty[k], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;

    const int64_t nt =
        p.ntiles > (int64_t)blockIdx.x ? (p.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto xslot = [&](int64_t j) { return base + L::kX + (uint32_t)(j % L::kNX) * L::kXBytes; };
    auto acol = [&](int64_t q) { return tmem + L::kAc + 64u * (uint32_t)(q % kNA); };

    if (warp == kWarps) {
        // ---- load warp
        if ((tid & 31) == 0) {
            const uint64_t pol = l2_evict_first_policy();       // read once
            asm volatile("griddepcontrol.wait;" ::: "memory");  // the last layer's output
            for (int64_t j = 0; j < nt; ++j) {
                const int64_t tg = blockIdx.x + j * gridDim.x;
                const int b = (int)(tg / p.ptiles), p0 = (int)((tg % p.ptiles) * kRows);
                const int sx = (int)(j % L::kNX);
                if (j >= L::kNX) mbar_wait(&x_empty[sx], (uint32_t)(j / L::kNX - 1), p.err);
                arrive_expect_tx(&x_full[sx], L::kXBytes);
                tma_load_2d_hint(tc_smem_addr(xslot(j)), &xmap, p0, b * C, &x_full[sx], pol);
            }
        }
    } else if (warp == kWarps + 3) {
        // ---- store warp: staging tile j % 2 -> out[b][0..cout2)[p0..p0+128)
        if ((tid & 31) == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // nothing earlier reads out
            for (int64_t j = 0; j < nt; ++j) {
                const int buf = (int)(j & 1);
                mbar_wait(&o_full[buf], (uint32_t)(j >> 1), p.err);
                const int64_t tg = blockIdx.x + j * gridDim.x;
                const int b = (int)(tg / p.ptiles), p0 = (int)((tg % p.ptiles) * kRows);
                tma_store_2d(&omap, p0, b * p.cout2,
                             tc_smem_addr(base + L::kOut + (uint32_t)(buf * C2 * kRows * sizeof(T))));
                bulk_commit();
                bulk_wait_read();
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                             ::"r"(tc_smem_addr(&o_empty[buf])) : "memory");
            }
            bulk_wait_all();
        }
    } else if (warp > kWarps) {
        // ---- MMA warps: warp kWarps + 1 + (j % 2) takes tile j into
        // accumulator j % 2: first ones x [bias_hi, bias_lo] (the bias in every
        // row), then per K step a_hi W_hi, a_hi W_lo, a_lo W_hi (N = H)
        if ((tid & 31) == 0) {
            constexpr uint32_t idesc = idesc_tf32(H);
            const uint32_t w0 = tc_smem_addr(base + L::kW);
            const uint64_t bias_desc = desc_sw128(tc_smem_addr(base + L::kBias));
            for (int64_t j = warp - (kWarps + 1); j < nt; j += 2) {
                const int buf = (int)(j & 1);
                const uint32_t d = tmem + (uint32_t)buf * H;
                if (j >= 2) mbar_wait(&acc_empty[buf], (uint32_t)((j - 2) >> 1), p.err);
                for (int c = 0; c < L::kKC; ++c) {
                    const int64_t q = j * L::kKC + c;
                    const int ab = (int)(q % kNA);
                    mbar_wait(&a_full[ab], (uint32_t)(q / kNA), p.err);
                    tc_after_sync();
                    const uint32_t a_hi = acol(q), a_lo = a_hi + 32;
                    const uint32_t wh = w0 + (uint32_t)c * 2 * L::kWHalf, wl = wh + L::kWHalf;
                    if (c == 0) mma_tf32_ts(d, tmem + L::kOnes, bias_desc, idesc, 0u);
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        mma_tf32_ts(d, a_hi + 8 * s, desc_sw128(wh + 32 * s), idesc, 1u);
                        mma_tf32_ts(d, a_hi + 8 * s, desc_sw128(wl + 32 * s), idesc, 1u);
                        if constexpr (kLo)
                            mma_tf32_ts(d, a_lo + 8 * s, desc_sw128(wh + 32 * s), idesc, 1u);
                    }
                    if (c == L::kKC - 1) mma_commit(&acc_full[buf]);
                    mma_commit(&a_empty[ab]);
                }
            }
        }
    } else {
        // ---- compute warps, set-up: W as the K-major B operand (rows = hidden
        // units), hi and lo; bias, P2, c2
        for (int e = tid; e < H * C; e += kCompute) {
            const float w = p.W[e];
            const int o = e / C, i = e % C;
            char *ch = base + L::kW + (uint32_t)(i / 32) * 2 * L::kWHalf;
            *reinterpret_cast<float *>(ch + sw_off(o, i % 32)) = w;
            *reinterpret_cast<float *>(ch + L::kWHalf + sw_off(o, i % 32)) = tf32_lo(w);
        }
        for (int e = tid; e < H * 32; e += kCompute) {
            const int o = e / 32, k = e % 32;
            const float b = p.bias[o];
            *reinterpret_cast<float *>(base + L::kBias + sw_off(o, k)) =
                k == 0 ? b : (k == 1 ? tf32_lo(b) : 0.f);
        }
        for (int e = tid; e < C2 * H; e += kCompute) {
            const int c = e / H;
            s_p2[e] = c < p.cout2 ? p.P2[e] : 0.f;
        }
        for (int c = tid; c < C2; c += kCompute) s_c2[c] = c < p.cout2 ? p.c2[c] : 0.f;
        fence_async_smem();
        compute_sync();
        const int quarter = warp & 3, row = 32 * quarter + (tid & 31);
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        if (warp < kTWarps) {
            // the constant ones operand (columns kOnes, kOnes + 1 = 1, the rest 0)
            {
                float one[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) one[u] = u < 2 ? 1.f : 0.f;
                tmem_st16(tmem + lane_base + L::kOnes, one);
            }
            // ---- transposer warps: chunk q into A buffer q % kNA once chunk
            // q - kNA's MMAs are done; thread = its pixel's 32 channels of the chunk
            for (int64_t j = 0; j < nt; ++j) {
                mbar_wait(&x_full[j % L::kNX], (uint32_t)(j / L::kNX), p.err);
                const T *X = reinterpret_cast<const T *>(xslot(j));
                for (int c = 0; c < L::kKC; ++c) {
                    const int64_t q = j * L::kKC + c;
                    if (q >= kNA) {
                        mbar_wait(&a_empty[q % kNA], (uint32_t)(q / kNA - 1), p.err);
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
                    warp_arrive(&a_full[q % kNA]);
                }
                warp_arrive(&x_empty[j % L::kNX]);
            }
        } else {
            // ---- epilogue warps: part = a quarter of the hidden units
            constexpr int kOut = H / 4;
            const int part = (warp - kTWarps) >> 2, o0 = part * kOut;
            float *red = reinterpret_cast<float *>(base + L::kRed);   // [2][3][C2][128]
            for (int64_t j = 0; j < nt; ++j) {
                const int buf = (int)(j & 1);
                mbar_wait(&acc_full[buf], (uint32_t)(j >> 1), p.err);
                tc_after_sync();
                const uint32_t ta = tmem + lane_base + (uint32_t)buf * H + (uint32_t)o0;
                // the second projection as pairs (two partial sums per output,
                // packed f32x2 fused multiply-adds)
                unsigned long long acc2[C2];
#pragma unroll
                for (int c = 0; c < C2; ++c) acc2[c] = gelu2_detail::splat(0.f);
                // 16 columns at a time; the accumulator goes back after the last load
#pragma unroll
                for (int g = 0; g < kOut / 16; ++g) {
                    float v[16];
                    tmem_ld16(ta + 16 * g, v);
                    if (g == kOut / 16 - 1) {
                        tc_before_sync();
                        warp_arrive_relaxed(&acc_empty[buf]);
                    }
                    const int ob = o0 + 16 * g;
#pragma unroll
                    for (int q = 0; q < 16; q += 4) {
                        gelu_erf2(v[q], v[q + 1]);
                        gelu_erf2(v[q + 2], v[q + 3]);
                        const unsigned long long h01 = gelu2_detail::pk(v[q], v[q + 1]);
                        const unsigned long long h23 = gelu2_detail::pk(v[q + 2], v[q + 3]);
#pragma unroll
                        for (int c = 0; c < C2; ++c) {
                            const float4 w4 = *reinterpret_cast<const float4 *>(s_p2 + c * H + ob + q);
                            acc2[c] = gelu2_detail::fma2(gelu2_detail::pk(w4.x, w4.y), h01, acc2[c]);
                            acc2[c] = gelu2_detail::fma2(gelu2_detail::pk(w4.z, w4.w), h23, acc2[c]);
                        }
                    }
                }
                float acc[C2];
#pragma unroll
                for (int c = 0; c < C2; ++c) {
                    float a0, a1;
                    gelu2_detail::upk(acc2[c], a0, a1);
                    acc[c] = a0 + a1;
                }
                // the four parts of a pixel: parts 1..3 leave their sums, part 0
                // adds them (a buffer per tile parity: a warp runs at most one
                // tile ahead of its quarter's barrier)
                float *rb = red + (size_t)buf * 3 * C2 * kRows;
                if (part > 0) {
#pragma unroll
                    for (int c = 0; c < C2; ++c) rb[((part - 1) * C2 + c) * kRows + row] = acc[c];
                }
                quarter_sync(quarter);
                if (part == 0) {
                    // the staging tile [cout2][128] of this parity is free once
                    // tile j - 2 has been read out
                    if (j >= 2) mbar_wait(&o_empty[buf], (uint32_t)((j - 2) >> 1), p.err);
                    T *ob = reinterpret_cast<T *>(base + L::kOut) + buf * C2 * kRows;
#pragma unroll
                    for (int c = 0; c < C2; ++c) {
                        if (c < p.cout2) {
                            float r = s_c2[c] + acc[c];
#pragma unroll
                            for (int k = 0; k < 3; ++k) r += rb[(k * C2 + c) * kRows + row];
                            Storage<T>::store(ob + c * kRows + row, r);
                        }
                    }
                    fence_async_smem();
                    warp_arrive(&o_full[buf]);
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

struct Pick {
    const void *fn;
    uint32_t smem;
    int cin;
};
template <int C, int H, int C2, typename T>
Pick make_pick() {
    return {(const void *)k_head<C, H, C2, T>, Lay<C, H, C2, T>::kAlloc, C};
}
template <typename T>
Pick pick_t(int cin, int hidden, int cout2) {
    const bool c1 = cout2 <= 1;
    if (cin <= 32) {
        if (hidden <= 64) return c1 ? make_pick<32, 64, 1, T>() : make_pick<32, 64, 8, T>();
        return c1 ? make_pick<32, 128, 1, T>() : make_pick<32, 128, 8, T>();
    }
    if (hidden <= 64) return c1 ? make_pick<64, 64, 1, T>() : make_pick<64, 64, 8, T>();
    return c1 ? make_pick<64, 128, 1, T>() : make_pick<64, 128, 8, T>();
}
Pick pick(fno_dtype_t dt, int cin, int hidden, int cout2) {
    return with_storage(dt, [&](auto t) { return pick_t<decltype(t)>(cin, hidden, cout2); });
}

}  // namespace

bool head_supported(fno_dtype_t dt, int cin, int hidden, int cout2, int64_t npix) {
    if ((dt != FNO_F32 && dt != FNO_F16 && dt != FNO_BF16) || !tcu::encoder()) return false;
    return (cin == 32 || cin == 64) && (hidden == 64 || hidden == 128) && cout2 >= 1 &&
           cout2 <= 8 && npix > 0 && npix % kRows == 0 && npix < ((int64_t)1 << 31);
}

cudaError_t head_init(fno_dtype_t dt, int cin, int hidden, int cout2) {
    const Pick k = pick(dt, cin, hidden, cout2);
    return raise_smem_limit(k.fn, k.smem);
}

cudaError_t head_launch(const HeadArgs &a, int num_sms, cudaStream_t s) {
    const Pick k = pick(a.dtype, a.cin, a.hidden, a.cout2);
    const size_t eb = a.dtype == FNO_F32 ? 4 : 2;
    const CUtensorMapDataType ty =
        a.dtype == FNO_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                           : (a.dtype == FNO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    CUtensorMap xmap, omap;
    if (!tcu::encode_rows_plain(&xmap, a.a, a.batch * a.cin, a.npix, eb, kRows, a.cin, ty) ||
        !tcu::encode_rows_plain(&omap, a.out, a.batch * a.cout2, a.npix, eb, kRows, a.cout2, ty))
        return cudaErrorInvalidValue;
    KParams kp;
    kp.W = a.W;
    kp.bias = a.bias;
    kp.P2 = a.P2;
    kp.c2 = a.c2;
    kp.out = a.out;
    kp.cout2 = a.cout2;
    kp.npix = a.npix;
    kp.ptiles = a.npix / kRows;
    kp.ntiles = a.batch * kp.ptiles;
    kp.err = a.err;
    if (kp.ntiles < 1) return cudaSuccess;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(kp.ntiles, std::max(num_sms, 1)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = k.smem;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    void *args[] = {&xmap, &omap, &kp};
    return cudaLaunchKernelExC(&cfg, k.fn, args);
}

}  // namespace fno
