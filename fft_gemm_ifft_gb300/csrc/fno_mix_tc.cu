// fno_mix_tc.cu -- the per-mode channel mixing on the tensor cores, for 16-bit
// storage (fp16 / bfloat16 operands, float32 accumulation): kernel B of the
// 16-bit 256 x 256 layer.
//
// The mixing of the TurboFNO article (gsyq.cn/news/457482) §2.2, Y[b,o,k] =
// sum_i X[b,i,k] W[i,o,k], is per mode k a complex (B x Cin) . (Cin x Cout)
// product.  Written in real-block form with the output channels on the M side,
//
//     [Yr]   [ Wr^T  -Wi^T ] [Xr]
//     [Yi] = [ Wi^T   Wr^T ] [Xi]      (M = 2 Cout rows, K = 2 Cin, N = batch)
//
// it is one tcgen05.mma chain (kind::f16, M = 128, K = 128 in 8 steps of 16)
// per mode, accumulating in tensor memory.
//
// The kept modes arrive from the forward-transform kernel, and the mixed modes
// leave for the inverse, in layouts chosen so that every global access moves
// whole 32-byte sectors (the layer's two all-to-all exchanges are transposes
// between an image-major and a mode-major order; done with 2- to 16-byte
// pieces they cost one L2 request per piece):
//   X: [group of 8 kept modes][image b * Cin + i][8 modes] of 16-bit (re, im)
//      pairs -- a group is one contiguous block of B * Cin * 32 bytes;
//   Y: [image b * Cout + o][kept mode] of 16-bit (re, im) pairs -- a group's 8
//      modes are 32 contiguous bytes of every image.
// A CTA takes one group: one bulk copy brings its X block, the threads
// transpose it in shared memory into the 8 modes' operands [Xr | Xi] (rows =
// batch, K = input channels, the 128-byte-swizzled K-major layout), the modes'
// weight operands pass through a ring of three slots, one MMA chain per mode
// accumulates into its own tensor-memory columns, and the results are staged
// so that each image's 8 modes leave as one 32-byte piece.
//
// Weights.  With FNO_PLAN_PACKED_WEIGHTS and 64 input and output channels,
// fno_spectral_conv_pack_weights has written each kept mode's [Wr^T; Wi^T] once
// (per weight update) as two 64 x 64 tiles in the swizzled layout (16 KiB a
// mode, the mode's own bytes): a slot [-Wi^T | Wr^T | Wi^T] receives the image
// in its last two thirds by one bulk copy and the threads negate Wi^T into the
// first third; K chunk 0 of the real block is then the slot from its second
// tile (rows Wr^T, then Wi^T) and chunk 1 the slot from its start (rows -Wi^T,
// then Wr^T).  Otherwise (weights in the standard or the mode-major layout) the
// threads build each slot from 4-byte weight loads.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "fno_fused_dev.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

constexpr int kMT = 256;                  // threads
constexpr int kGrp = 8;                   // kept modes per CTA (one group)
constexpr int kCh = 64;                   // channel tile (Cin, Cout <= 64)
constexpr int kMaxN = 32;                 // batch rows (N) per CTA
constexpr int kSlots = 3;                 // weight ring
constexpr uint32_t kHalfTile = 64 * 128;  // 64 rows x 128 bytes
constexpr uint32_t kASlot = 3 * kHalfTile;          // [-Wi^T | Wr^T | Wi^T]
constexpr uint32_t kImgMode = 2 * kHalfTile;        // packed bytes per mode
constexpr uint32_t kXMode = 2 * kMaxN * 128;        // a mode's X operand: [Re | Im] x 32 rows
// shared memory: the raw X block (B * Cin images x 32 bytes), later the Y
// staging (B * Cout images x 9 words: a padded row keeps the drain free of
// bank conflicts); the 8 X operands; the weight ring
constexpr uint32_t kStageRow = 9;                   // words per staged image
constexpr uint32_t kRawBytes = kCh * kMaxN * kStageRow * 4;   // >= B * Cin * 32 as well
constexpr uint32_t kOffXop = (kRawBytes + 1023) / 1024 * 1024;
constexpr uint32_t kOffW = kOffXop + kGrp * kXMode;
constexpr uint32_t kSmem = kOffW + kSlots * kASlot + 1024;
constexpr uint32_t kTmemCols = 256;                 // kGrp modes x N (<= 32)
static_assert(kSmem <= 232448 - 512, "one CTA per SM");
static_assert((uint32_t)kCh * kMaxN * 32 <= kRawBytes, "raw X block fits");

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

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(tc_smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(tc_smem_addr(bar)), "r"(bytes) : "memory");
}

template <typename T, bool kImg>
__global__ void __launch_bounds__(kMT, 1) k_mix_tc(MixTcArgs a) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_x, bar_w[kSlots], bar_m[kSlots];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int grp = blockIdx.x, mode0 = grp * kGrp;
    const int nbp = (a.batch + 15) / 16 * 16;                // N: batch padded to 16
    const int nimg_in = a.batch * a.cin, nimg_out = a.batch * a.cout;
    const uint32_t sb = tc_smem_addr(base);
    const bool inside = mode0 >= 0 && mode0 + kGrp <= a.nk;    // the group lies in the tensors
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_x)));
        for (int s = 0; s < kSlots; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_w[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_m[s])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!inside) raise_dev_error(a.err, kDevBounds);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // every thread waits on the barriers: they must be initialised first
    __syncthreads();
    // The packed weight image of mode r into the last two thirds of slot r % kSlots
    // (thread 0; nothing is copied for a group outside the tensors).
    auto fetch_w = [&](int r) {
        const int s = r % kSlots;
        expect_tx(&bar_w[s], inside ? kImgMode : 0u);
        if (inside)
            bulk_g2s(sb + kOffW + s * kASlot + kHalfTile,
                     static_cast<const char *>(a.w) + (size_t)(mode0 + r) * kImgMode, kImgMode,
                     &bar_w[s]);
    };
    // Slot r % kSlots = [-Wi^T | Wr^T | Wi^T] of mode r from the weight tensor
    // (all threads; element (o, i) of each tile).
    auto build_w = [&](int r) {
        char *slot = base + kOffW + (r % kSlots) * kASlot;
        const int kk = mode0 + r, j = kk / a.m1, k = kk % a.m1;
        const int blk = j >= a.m0 ? 1 : 0;
        const int local = (j - blk * a.m0) * a.m1 + k;
        const T *w = static_cast<const T *>(a.w);
        for (int e = tid; e < kCh * kCh; e += kMT) {
            const int o = e % kCh, i = e / kCh;
            uint32_t word = 0;
            if (inside && i < a.cin && o < a.cout) {
                const T *p = a.packed ? w + packed_index(kk, i, o, a.cin, a.cout) * 2
                                      : w + ((((size_t)blk * a.cin + i) * a.cout + o) * a.mblk +
                                             local) * 2;
                word = __ldg(reinterpret_cast<const unsigned int *>(p));
            }
            const unsigned short re = (unsigned short)(word & 0xFFFF);
            const unsigned short im = (unsigned short)(word >> 16);
            const uint32_t off = sw_off16(o, i);
            *reinterpret_cast<unsigned short *>(slot + off) = im ^ 0x8000;
            *reinterpret_cast<unsigned short *>(slot + kHalfTile + off) = re;
            *reinterpret_cast<unsigned short *>(slot + 2 * kHalfTile + off) = im;
        }
    };
    // 1. the first weight slots (independent of kernel A)
    if constexpr (kImg) {
        if (tid == 0)
            for (int r = 0; r < kSlots; ++r) fetch_w(r);
    }
    pdl_trigger();
    pdl_wait();                                  // kernel A's kept modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    // 2. the group's X block: B * Cin images x 32 bytes, one bulk copy
    const uint32_t xblock = (uint32_t)nimg_in * 32;
    if (tid == 0) {
        expect_tx(&bar_x, inside ? xblock : 0u);
        if (inside)
            bulk_g2s(sb, static_cast<const char *>(a.X) + (size_t)grp * xblock, xblock, &bar_x);
    }
    if (a.cin < kCh) {
        // input columns beyond cin stay zero in every X operand
        for (int e = tid; e < (int)(kGrp * kXMode / 16); e += kMT)
            reinterpret_cast<uint4 *>(base + kOffXop)[e] = make_uint4(0, 0, 0, 0);
        __syncthreads();                         // zeroing before the transpose writes
    }
    bool ok = mbar_wait(&bar_x, 0, a.err);
    // 3. transpose: image (b, i) holds 8 modes (re, im); mode r's operand gets
    //    Re in chunk 0 and Im in chunk 1 at row b, column i.  A warp takes 32
    //    consecutive images, so each of its 2-byte stores fills 64 contiguous bytes.
    for (int img = tid; img < nimg_in; img += kMT) {
        const uint4 *src = reinterpret_cast<const uint4 *>(base + (size_t)img * 32);
        const uint4 p0 = src[0], p1 = src[1];
        const uint32_t v[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        const uint32_t off = sw_off16(img / a.cin, img % a.cin);
#pragma unroll
        for (int r = 0; r < kGrp; ++r) {
            char *xo = base + kOffXop + r * kXMode;
            *reinterpret_cast<unsigned short *>(xo + off) = (unsigned short)(v[r] & 0xFFFF);
            *reinterpret_cast<unsigned short *>(xo + nbp * 128 + off) =
                (unsigned short)(v[r] >> 16);
        }
    }
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = idesc_f16(nbp, Bits<T>::kBf16);
    // 4. one chain per mode.  Packed images: slot r % kSlots is refilled with
    //    mode r + kSlots by thread 0 as soon as mode r's MMAs have read it.
    //    Built slots: every thread waits for the slot's previous MMAs first.
    for (int r = 0; r < kGrp; ++r) {
        const int s = r % kSlots;
        char *slot = base + kOffW + s * kASlot;
        if constexpr (kImg) {
            ok &= mbar_wait(&bar_w[s], (r / kSlots) & 1, a.err);
            for (int e = tid; e < (int)(kHalfTile / 16); e += kMT) {   // -Wi^T, exact
                const uint4 v = reinterpret_cast<const uint4 *>(slot + 2 * kHalfTile)[e];
                reinterpret_cast<uint4 *>(slot)[e] =
                    make_uint4(v.x ^ 0x80008000u, v.y ^ 0x80008000u, v.z ^ 0x80008000u,
                               v.w ^ 0x80008000u);
            }
        } else {
            if (r >= kSlots) {
                ok &= mbar_wait(&bar_m[s], ((r - kSlots) / kSlots) & 1, a.err);
                tc_after_sync();
            }
            build_w(r);
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();                         // slot (and, at r = 0, the X operands) ready
        if (tid == 0) {
            tc_after_sync();
            if (ok) {
                const uint32_t bm = sb + kOffXop + r * kXMode;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint32_t am = sb + kOffW + s * kASlot + (c == 0 ? kHalfTile : 0u);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        mma_f16(tmem + r * nbp, desc_sw128(am + q * 32),
                                desc_sw128(bm + c * nbp * 128 + q * 32), idesc,
                                (c | q) ? 1u : 0u);
                }
            }
            mma_commit(&bar_m[s]);
            if constexpr (kImg) {
                if (r + kSlots < kGrp) {
                    ok &= mbar_wait(&bar_m[s], (r / kSlots) & 1, a.err);
                    fetch_w(r + kSlots);
                }
            }
        }
    }
    // every chain is done once the last commit of each slot has arrived
    for (int r = kGrp - kSlots; r < kGrp; ++r)
        ok &= mbar_wait(&bar_m[r % kSlots], (r / kSlots) & 1, a.err);
    tc_after_sync();
    // 5. tensor memory -> staging: D row m = o (re) or 64 + o (im), column b;
    //    staged image row (b * Cout + o) of 9 words, word r = mode r (re, im)
    uint32_t *stage = reinterpret_cast<uint32_t *>(base);
    {
        const int m = 32 * (warp & 3) + lane;
        const int o = m % kCh, part = m / kCh;
        for (int r = warp >> 2; r < kGrp; r += 2) {              // warps 0-3 even modes, 4-7 odd
            for (int g = 0; g < nbp / 16; ++g) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + r * nbp + 16 * g, v);
                if (o < a.cout) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int b = 16 * g + q;
                        if (b < a.batch)
                            reinterpret_cast<unsigned short *>(
                                stage + ((size_t)b * a.cout + o) * kStageRow + r)[part] =
                                Bits<T>::from(ok ? v[q] : 0.f);
                    }
                }
            }
        }
    }
    tc_before_sync();
    __syncthreads();
    // 6. Y: each image's 8 modes as one 32-byte piece
    for (int img = tid; img < nimg_out && inside; img += kMT) {
        const uint32_t *sv = stage + (size_t)img * kStageRow;
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint32_t *>(a.Y) +
                                               (size_t)img * a.nk + mode0);
        dst[0] = make_uint4(sv[0], sv[1], sv[2], sv[3]);
        dst[1] = make_uint4(sv[4], sv[5], sv[6], sv[7]);
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

bool mixtc_supported(int d, fno_dtype_t dtype, int64_t batch, int cin, int cout, int m1,
                     int64_t nkept) {
    return d == 2 && (dtype == FNO_F16 || dtype == FNO_BF16) && cin <= kCh && cout <= kCh &&
           batch >= 1 && batch <= kMaxN && m1 % kGrp == 0 && nkept % kGrp == 0;
}

int mixtc_items(int64_t nkept) { return (int)(nkept / kGrp); }

size_t mixtc_x_bytes(int64_t batch, int cin, int64_t nkept) {
    return (size_t)nkept * batch * cin * 4;
}

cudaError_t mixtc_init(fno_dtype_t dtype) {
    return with_storage(dtype, [&](auto t) {
        using T = decltype(t);
        if constexpr (std::is_same<T, float>::value) {
            return cudaErrorInvalidValue;
        } else {
            cudaError_t e = raise_smem_limit(k_mix_tc<T, false>, (int)kSmem);
            return e != cudaSuccess ? e : raise_smem_limit(k_mix_tc<T, true>, (int)kSmem);
        }
    });
}

cudaError_t mixtc_launch(fno_dtype_t dtype, const MixTcArgs &args, cudaStream_t s) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(args.nk / kGrp));
    cfg.blockDim = dim3(kMT);
    cfg.dynamicSmemBytes = kSmem;
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
