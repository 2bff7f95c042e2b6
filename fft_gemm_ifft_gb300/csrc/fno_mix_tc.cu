// fno_mix_tc.cu -- the per-mode channel mixing on the tensor cores, for 16-bit
// storage (fp16 / bfloat16 operands, float32 accumulation).
//
// The mixing of the TurboFNO article (gsyq.cn/news/457482) §2.2, Y[b,o,k] =
// sum_i X[b,i,k] W[i,o,k], is per mode k a complex (B x Cin) . (Cin x Cout)
// product.  Written in real-block form with the output channels on the M side,
//
//     [Yr]   [ Wr^T  -Wi^T ] [Xr]
//     [Yi] = [ Wi^T   Wr^T ] [Xi]      (M = 2 Cout rows, K = 2 Cin, N = batch)
//
// it is one tcgen05.mma chain (kind::f16, M = 128, K = 128 in 8 steps of 16)
// per mode, accumulating in tensor memory.  A CTA takes a run of kRun (two or
// four) adjacent modes of one kept row (adjacent in the weight tensor too): it
// builds the run's 128 x 128 real-block weight operands in shared memory (128-
// byte swizzle, K-major) from 8- or 16-byte loads of the weights -- before
// waiting for the forward-transform kernel, since they do not depend on it --
// then the operands [Xr; Xi]^T (N rows = batch) from the kept modes, issues
// one chain per mode into its own column range of tensor memory, and writes Y
// for the run's modes of every (b, o) as one contiguous piece through a
// shared-memory staging tile.  Channel counts up to 64 are zero-padded to the
// tile.
//
// Weights packed as operand images (plans with FNO_PLAN_PACKED_WEIGHTS and 64
// input and output channels): fno_spectral_conv_pack_weights writes, once per
// weight update, each kept mode's [Wr^T; Wi^T] as two 64 x 64 tiles in the
// swizzled K-major layout above (16 KiB a mode, the size of the mode's weights).
// A CTA then fetches a mode with one bulk copy into the middle of a 24 KiB slot
// [-Wi^T | Wr^T | Wi^T] and negates Wi^T into the first third: K chunk 0 of the
// real-block operand is the slot from its second tile (rows Wr^T, then Wi^T),
// chunk 1 the slot from its start (rows -Wi^T, then Wr^T).
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "fno_fused_dev.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

#ifndef FNO_MIX_THREADS
#define FNO_MIX_THREADS 256
#endif
constexpr int kMT = FNO_MIX_THREADS;      // threads (256 or 512)
// Runs of two modes fit two CTAs on an SM (97 KB of shared memory each against
// 193 KB for four); behind the persistent 16-bit forward transform, which
// leaves no SM to an early mixing CTA, that measured 275 -> 266 us on the
// 32 x 64-channel 256^2 fp16 layer.
#ifndef FNO_MIX_RUN
#define FNO_MIX_RUN 2
#endif
constexpr int kRun = FNO_MIX_RUN;         // modes per CTA (2 or 4)
static_assert(kRun == 2 || kRun == 4, "modes per CTA");
constexpr int kCh = 64;                   // channel tile (Cin, Cout <= 64)
constexpr uint32_t kAChunk = 128 * 128;   // 128 rows x 128 bytes (64 elements of K)
constexpr uint32_t kAMode = 2 * kAChunk;  // one mode's weight operand (K = 128)
constexpr int kMaxB = 64;                 // batch rows (N) per CTA
constexpr uint32_t kBChunk = kMaxB * 128;
constexpr uint32_t kBMode = 2 * kBChunk;
constexpr uint32_t kOffB = kRun * kAMode;                 // weight operands, 32 KiB a mode
constexpr uint32_t kSmem = kOffB + kRun * kBMode + 1024;  // + X operands, 16 KiB a mode + align
constexpr uint32_t kTmemCols = kRun * 64;                  // kRun x N (N <= 64)
// operand-image weights: a 24 KiB slot per mode
constexpr uint32_t kHalfTile = 64 * 128;                   // 64 rows x 128 bytes
constexpr uint32_t kASlot = 3 * kHalfTile;
constexpr uint32_t kOffBImg = kRun * kASlot;
constexpr uint32_t kSmemImg = kOffBImg + kRun * kBMode + 1024;
constexpr uint32_t kImgMode = 2 * kHalfTile;               // packed bytes per mode (16-bit)
// the drain's staging tile (batch x 64 outputs x kRun modes, complex float) goes
// over the weight and X operands once the MMAs are done
static_assert((uint32_t)kMaxB * kCh * kRun * 8 <= kRun * kASlot + kRun * kBMode, "staging fits");

template <typename T> struct Bits;
template <> struct Bits<__half> {
    static constexpr bool kBf16 = false;
    static __device__ __forceinline__ unsigned short from(float v) {
        return __half_as_ushort(__float2half_rn(v));
    }
};
template <> struct Bits<__nv_bfloat16> {
    static constexpr bool kBf16 = true;
    static __device__ __forceinline__ unsigned short from(float v) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
};

template <typename T, bool kImg>
__global__ void __launch_bounds__(kMT, kRun == 2 ? 2 : 1) k_mix_tc(MixTcArgs a) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    constexpr uint32_t kB0 = kImg ? kOffBImg : kOffB;        // X operands
    __shared__ __align__(8) uint64_t bar, bar_w;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int mode0 = blockIdx.x * kRun;
    const int nbp = (a.batch + 15) / 16 * 16;                // N: batch padded to 16
    // kept row j and bin k of mode0; weight block and local index
    const int j = mode0 / a.m1, k = mode0 % a.m1;
    const int blk = j >= a.m0 ? 1 : 0;
    const int local0 = (j - blk * a.m0) * a.m1 + k;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_w)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if constexpr (kImg) {
            // the run's weight images: kRun contiguous 16 KiB pieces, each into the
            // middle third of its slot (independent of kernel A); a run beyond the
            // packed tensor is an error, recorded, and nothing is copied (the
            // barrier is released without bytes)
            const bool inside = mode0 >= 0 && mode0 + kRun <= a.nk;
            if (!inside) raise_dev_error(a.err, kDevBounds);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         ::"r"(tc_smem_addr(&bar_w)), "r"(inside ? kRun * kImgMode : 0u)
                         : "memory");
            const char *src = static_cast<const char *>(a.w) + (size_t)mode0 * kImgMode;
            for (int r = 0; r < kRun && inside; ++r)
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                             " [%0], [%1], %2, [%3];"
                             ::"r"(tc_smem_addr(base + r * kASlot + kHalfTile)),
                               "l"(src + (size_t)r * kImgMode), "r"(kImgMode),
                               "r"(tc_smem_addr(&bar_w)) : "memory");
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    bool ok = true;
    if constexpr (kImg) {
        // every thread waits on bar_w: it must be initialised first
        __syncthreads();
        // -Wi^T into the first third of each slot (a sign flip of every 16-bit value)
        ok = mbar_wait(&bar_w, 0, a.err);
        for (int e = tid; e < (int)(kRun * kHalfTile / 16); e += kMT) {
            const int r = e / (kHalfTile / 16), q = e % (kHalfTile / 16);
            const uint4 v = reinterpret_cast<const uint4 *>(base + r * kASlot + 2 * kHalfTile)[q];
            reinterpret_cast<uint4 *>(base + r * kASlot)[q] =
                make_uint4(v.x ^ 0x80008000u, v.y ^ 0x80008000u, v.z ^ 0x80008000u,
                           v.w ^ 0x80008000u);
        }
    }
    // 1. zero the operands where the channel counts leave padding
    if (!kImg && (a.cin < kCh || a.cout < kCh)) {
        for (int e = tid; e < (int)(kRun * kAMode / 16); e += kMT)
            reinterpret_cast<uint4 *>(base)[e] = make_uint4(0, 0, 0, 0);
        __syncthreads();
    }
    // 2. weight operands of the four modes (independent of kernel A)
    using U = unsigned short;
    const T *w = static_cast<const T *>(a.w);
    // a unit = one output o and eight consecutive input channels: eight 16-byte
    // loads (four modes each), then per mode and quadrant one 16-byte store of
    // eight consecutive K elements (conflict-free under the swizzle)
    for (int un = tid; !kImg && un < kCh * (kCh / 8); un += kMT) {
        const int o = un % kCh, i0 = 8 * (un / kCh);
        if (o >= a.cout || i0 >= a.cin) continue;
        // the run's kRun modes of one (i, o): kRun x 4 bytes, contiguous in both layouts
        using WV = std::conditional_t<kRun == 4, uint4, uint2>;
        WV q[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            q[t] = WV{};
            if (i0 + t < a.cin)
                q[t] = __ldg(reinterpret_cast<const WV *>(
                    a.packed ? w + packed_index(mode0, i0 + t, o, a.cin, a.cout) * 2
                             : w + ((((size_t)blk * a.cin + i0 + t) * a.cout + o) * a.mblk +
                                    local0) * 2));
        }
#pragma unroll
        for (int r = 0; r < kRun; ++r) {
            // element t of mode r: re = half 2r, im = half 2r + 1 of q[t]
            U re[8], im[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint32_t word = reinterpret_cast<const uint32_t *>(&q[t])[r];
                re[t] = (U)(word & 0xFFFF);
                im[t] = (U)(word >> 16);
            }
            auto pack = [](const U (&v)[8], bool negate) {
                uint4 p;
                const uint32_t m = negate ? 0x80008000u : 0u;
                p.x = ((uint32_t)v[0] | ((uint32_t)v[1] << 16)) ^ m;
                p.y = ((uint32_t)v[2] | ((uint32_t)v[3] << 16)) ^ m;
                p.z = ((uint32_t)v[4] | ((uint32_t)v[5] << 16)) ^ m;
                p.w = ((uint32_t)v[6] | ((uint32_t)v[7] << 16)) ^ m;
                return p;
            };
            char *A = base + r * kAMode;
            // row o: [Wr | -Wi], row 64 + o: [Wi | Wr]; K columns i0.. and 64 + i0..
            *reinterpret_cast<uint4 *>(A + sw_off16(o, i0)) = pack(re, false);
            *reinterpret_cast<uint4 *>(A + kAChunk + sw_off16(o, i0)) = pack(im, true);
            *reinterpret_cast<uint4 *>(A + sw_off16(kCh + o, i0)) = pack(im, false);
            *reinterpret_cast<uint4 *>(A + kAChunk + sw_off16(kCh + o, i0)) = pack(re, false);
        }
    }
    pdl_trigger();
    pdl_wait();                                  // kernel A's kept modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    // 3. X operands: row n = batch index, K columns [Xr(i) | Xi(i)].  A unit is
    //    one batch row and eight input channels: sixteen 16-byte loads, then per
    //    mode two 16-byte stores
    for (int un = tid; un < nbp * (kCh / 8); un += kMT) {
        const int bb = un / (kCh / 8), i0 = 8 * (un % (kCh / 8));
        constexpr int kV = kRun / 2;                     // float4 per (b, i): two modes each
        float4 v[8 * kV];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
#pragma unroll
            for (int h = 0; h < kV; ++h) v[kV * t + h] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (bb < a.batch && i0 + t < a.cin) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    a.X + ((size_t)bb * a.cin + i0 + t) * a.nk + mode0);
#pragma unroll
                for (int h = 0; h < kV; ++h) v[kV * t + h] = __ldcg(src + h);
            }
        }
#pragma unroll
        for (int r = 0; r < kRun; ++r) {
            uint32_t pr[4], pi[4];
#pragma unroll
            for (int t2 = 0; t2 < 4; ++t2) {
                float xr[2], xi[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 &u4 = v[kV * (2 * t2 + h) + r / 2];
                    xr[h] = (r & 1) ? u4.z : u4.x;
                    xi[h] = (r & 1) ? u4.w : u4.y;
                }
                pr[t2] = (uint32_t)Bits<T>::from(xr[0]) | ((uint32_t)Bits<T>::from(xr[1]) << 16);
                pi[t2] = (uint32_t)Bits<T>::from(xi[0]) | ((uint32_t)Bits<T>::from(xi[1]) << 16);
            }
            char *B = base + kB0 + r * kBMode;
            *reinterpret_cast<uint4 *>(B + sw_off16(bb, i0)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
            *reinterpret_cast<uint4 *>(B + kBChunk + sw_off16(bb, i0)) =
                make_uint4(pi[0], pi[1], pi[2], pi[3]);
        }
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        const uint32_t idesc = idesc_f16(nbp, Bits<T>::kBf16);
#pragma unroll
        for (int r = 0; r < kRun && ok; ++r) {
            const uint32_t bm = tc_smem_addr(base + kB0 + r * kBMode);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                // K chunk c of the real-block weight operand
                const uint32_t am =
                    kImg ? tc_smem_addr(base + r * kASlot + (c == 0 ? kHalfTile : 0u))
                         : tc_smem_addr(base + r * kAMode + c * kAChunk);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(tmem + r * nbp, desc_sw128(am + s * 32),
                            desc_sw128(bm + c * kBChunk + s * 32), idesc, (c | s) ? 1u : 0u);
            }
        }
        mma_commit(&bar);
    }
    ok &= mbar_wait(&bar, 0, a.err);
    tc_after_sync();
    // 4. tensor memory -> staging [b][o][4 modes] complex (over the weight operands,
    //    which the finished MMAs no longer read)
    float *stage = reinterpret_cast<float *>(base);
    {
        const int m = 32 * (warp & 3) + (tid & 31);          // D row: o (re) or 64 + o (im)
        const int o = m % kCh, part = m / kCh;
        // each group of four warps drains kPer of the run's modes
        constexpr int kPer = kRun / (kMT / 128);
        static_assert(kPer >= 1 && kPer * (kMT / 128) == kRun, "modes per warp group");
        for (int r = kPer * (warp >> 2); r < kPer * (warp >> 2) + kPer; ++r) {
            for (int g = 0; g < nbp / 16; ++g) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + r * nbp + 16 * g, v);
                if (o < a.cout) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int b = 16 * g + q;
                        if (b < a.batch)
                            stage[(((size_t)b * kCh + o) * kRun + r) * 2 + part] = ok ? v[q] : 0.f;
                    }
                }
            }
        }
    }
    tc_before_sync();
    __syncthreads();
    // 5. Y for the run's modes of every (b, o): kRun x 8 contiguous bytes
    for (int e = tid; e < a.batch * a.cout; e += kMT) {
        const int b = e / a.cout, o = e % a.cout;
        const float4 *s4 = reinterpret_cast<const float4 *>(stage + ((size_t)b * kCh + o) * kRun * 2);
        float4 *dst = reinterpret_cast<float4 *>(a.Y + ((size_t)b * a.cout + o) * a.nk + mode0);
#pragma unroll
        for (int h = 0; h < kRun / 2; ++h) __stcg(dst + h, s4[h]);
    }
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
    }
    if (a.trace) {
        __syncthreads();
        if (tid == 0) {
            unsigned smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            fno_trace_record_t rec;
            rec.item = (1u << 24) | (blockIdx.x & 0xFFFFFFu);
            rec.worker = smid;
            rec.t_start = t0;
            rec.t_ready = t1;
            rec.t_compute = rec.t_end = trace_now();
            a.trace[a.trace_first + blockIdx.x] = rec;
        }
    }
}

}  // namespace

bool mixtc_supported(int d, fno_dtype_t dtype, int64_t batch, int cin, int cout, int m1,
                     int64_t nkept) {
    return d == 2 && (dtype == FNO_F16 || dtype == FNO_BF16) && cin <= kCh && cout <= kCh &&
           batch >= 1 && batch <= kMaxB && m1 % kRun == 0 && nkept % kRun == 0;
}

int mixtc_items(int64_t nkept) { return (int)(nkept / kRun); }

cudaError_t mixtc_init(fno_dtype_t dtype) {
    return with_storage(dtype, [&](auto t) {
        using T = decltype(t);
        if constexpr (std::is_same<T, float>::value) {
            return cudaErrorInvalidValue;
        } else {
            cudaError_t e = raise_smem_limit(k_mix_tc<T, false>, (int)kSmem);
            return e != cudaSuccess ? e : raise_smem_limit(k_mix_tc<T, true>, (int)kSmemImg);
        }
    });
}

cudaError_t mixtc_launch(fno_dtype_t dtype, const MixTcArgs &args, cudaStream_t s) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(args.nk / kRun));
    cfg.blockDim = dim3(kMT);
    cfg.dynamicSmemBytes = args.packed == 2 ? kSmemImg : kSmem;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return with_storage(dtype, [&](auto t) {
        using T = decltype(t);
        if constexpr (std::is_same<T, float>::value) {
            return cudaErrorInvalidValue;
        } else {
            cudaError_t e = args.packed == 2 ? cudaLaunchKernelEx(&cfg, k_mix_tc<T, true>, args)
                                             : cudaLaunchKernelEx(&cfg, k_mix_tc<T, false>, args);
            return e != cudaSuccess ? e : cudaGetLastError();
        }
    });
}

namespace {

// One thread per 16-byte piece of the packed images: mode kk, tile (0: Wr^T,
// 1: Wi^T), row o, physical piece p of the swizzled row (logical columns
// i = 8 ((p ^ o) & 7) .. + 7).  Zero outside cin x cout.
template <typename T>
__global__ void __launch_bounds__(256)
k_pack_image(const T *__restrict__ w, uint4 *__restrict__ wp, int cin, int cout, int m0, int m1,
             int mblk, int nk) {
    const int64_t total = (int64_t)nk * 2 * kCh * 8;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(idx & 7);
        const int o = (int)((idx >> 3) % kCh);
        const int tile = (int)((idx >> 3) / kCh % 2);
        const int kk = (int)(idx / (16 * kCh));
        const int jr = kk / m1, k = kk % m1;
        const int blk = jr >= m0 ? 1 : 0;
        const int local = (jr - blk * m0) * m1 + k;
        const int i0 = 8 * ((p ^ o) & 7);
        unsigned short v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u;
            v[u] = 0;
            if (i < cin && o < cout) {
                const T val = w[((((size_t)blk * cin + i) * cout + o) * mblk + local) * 2 + tile];
                memcpy(&v[u], &val, 2);
            }
        }
        uint4 q;
        q.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
        q.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
        q.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
        q.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
        wp[idx] = q;
    }
}

}  // namespace

bool mixtc_image_layout(int cin, int cout) { return cin == kCh && cout == kCh; }

cudaError_t mixtc_pack_image(fno_dtype_t dtype, const void *w, void *wp, int cin, int cout,
                             int m0, int m1, int mblk, int nk, int num_sms, cudaStream_t s) {
    const int64_t pieces = (int64_t)nk * 2 * kCh * 8;
    const int grid = (int)std::min<int64_t>((pieces + 255) / 256, (int64_t)num_sms * 16);
    return with_storage(dtype, [&](auto t) {
        using T = decltype(t);
        if constexpr (std::is_same<T, float>::value) {
            return cudaErrorInvalidValue;
        } else {
            k_pack_image<T><<<grid, 256, 0, s>>>(static_cast<const T *>(w),
                                                 static_cast<uint4 *>(wp), cin, cout, m0, m1,
                                                 mblk, nk);
            return cudaGetLastError();
        }
    });
}

}  // namespace fno
