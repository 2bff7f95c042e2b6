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
//   Y: [group of 8 kept modes][image b * Cout + o][8 modes] of 16-bit (re, im)
//      pairs, the same layout; the inverse gathers an image's 256 group rows
//      with one three-dimensional TMA load.
// A CTA takes half a group (4 modes; two CTAs per SM): the threads read each
// image's 16 bytes of the run with coalesced loads and transpose them in
// shared memory into the 4 modes' operands [Xr | Xi] (rows = batch, K = input
// channels, the 128-byte-swizzled K-major layout), the modes' weight operands
// pass through a ring of three slots, one MMA chain per mode accumulates into
// its own tensor-memory columns, and the results are staged so that each
// image's 4 modes leave as one 16-byte piece.
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

constexpr int kMT = 512;                  // threads
constexpr int kGrp = 8;                   // kept modes per group of the X / Y layout
constexpr int kRun = 4;                   // kept modes per work unit: half a group
constexpr int kCh = 64;                   // channel tile (Cin, Cout <= 64)
constexpr int kMaxN = 32;                 // batch rows (N)
constexpr uint32_t kHalfTile = 64 * 128;  // 64 rows x 128 bytes
constexpr uint32_t kASlot = 3 * kHalfTile;          // [-Wi^T | Wr^T | Wi^T]
constexpr uint32_t kImgMode = 2 * kHalfTile;        // packed bytes per mode
constexpr uint32_t kXMode = 2 * kMaxN * 128;        // a mode's X operand: [Re | Im] x 32 rows
constexpr uint32_t kXUnit = kRun * kXMode;          // a unit's X operands
// shared memory (one persistent CTA per SM): two buffers of a unit's X
// operands (the next unit's are transposed in while the current one's MMAs
// run), the unit's four weight slots, and the Y staging (B * Cout images x 5
// words: a padded row keeps the drain free of bank conflicts)
constexpr uint32_t kStageRow = kRun + 1;            // words per staged image
constexpr uint32_t kOffW = 2 * kXUnit;
constexpr uint32_t kOffStage = kOffW + kRun * kASlot;
constexpr uint32_t kStageBytes = (uint32_t)kMaxN * kCh * kStageRow * 4;
constexpr uint32_t kSmem = kOffStage + kStageBytes + 1024;
constexpr uint32_t kTmemCols = 256;                 // two units x kRun modes x N (<= 32)
static_assert(kSmem + 256 <= 232448, "one CTA per SM");

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
    __shared__ __align__(8) uint64_t bar_w[kRun], bar_m[2];
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nbp = (a.batch + 15) / 16 * 16;                // N: batch padded to 16
    const int nimg_in = a.batch * a.cin, nimg_out = a.batch * a.cout;
    const int nunits = a.nk / kRun;
    const uint32_t sb = tc_smem_addr(base);
    if (tid == 0) {
        for (int s = 0; s < kRun; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_w[s])));
        for (int s = 0; s < 2; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar_m[s])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // both X operand buffers start at zero: rows past the batch and columns past
    // cin are never written and must not hold stale bits (NaN times zero)
    for (int e = tid; e < (int)(2 * kXUnit / 16); e += kMT)
        reinterpret_cast<uint4 *>(base)[e] = make_uint4(0, 0, 0, 0);
    // every thread waits on the barriers: they must be initialised first
    __syncthreads();
    auto slot_at = [&](int r) -> char * { return base + kOffW + r * kASlot; };
    // the packed weight images of unit u's modes into the last two thirds of
    // the four slots (thread 0)
    auto fetch_w = [&](int u) {
        const bool in = u >= 0 && (u + 1) * kRun <= a.nk;
        if (!in) raise_dev_error(a.err, kDevBounds);
        for (int r = 0; r < kRun; ++r) {
            expect_tx(&bar_w[r], in ? kImgMode : 0u);
            if (in)
                bulk_g2s(tc_smem_addr(slot_at(r) + kHalfTile),
                         static_cast<const char *>(a.w) + ((size_t)u * kRun + r) * kImgMode,
                         kImgMode, &bar_w[r]);
        }
    };
    // slot r = [-Wi^T | Wr^T | Wi^T] of kept mode kk from the weight tensor
    // (all threads; element (o, i) of each tile)
    auto build_w = [&](int r, int kk) {
        char *slot = slot_at(r);
        const int j = kk / a.m1, k = kk % a.m1;
        const int blk = j >= a.m0 ? 1 : 0;
        const int local = (j - blk * a.m0) * a.m1 + k;
        const T *w = static_cast<const T *>(a.w);
        for (int e = tid; e < kCh * kCh; e += kMT) {
            const int o = e % kCh, i = e / kCh;
            uint32_t word = 0;
            if (i < a.cin && o < a.cout) {
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
    // unit u's kept modes: image (b, i) holds the unit's 4 modes (re, im) as 16
    // contiguous bytes of its group row; all of a thread's loads are in flight
    // before the transpose writes mode r's Re (chunk 0) and Im (chunk 1) at row
    // b, column i of X operand buffer xo.  A warp takes 32 consecutive images:
    // each of its 2-byte stores fills 64 contiguous bytes.
    auto load_x = [&](int u, char *xo) {
        const int grp = u / 2, half = u % 2;
        const char *xg = static_cast<const char *>(a.X) + (size_t)grp * nimg_in * 32 + half * 16;
        constexpr int kPer = 4;
        for (int img0 = 0; img0 < nimg_in; img0 += kPer * kMT) {
            uint4 v[kPer];
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int img = img0 + q * kMT + tid;
                const int64_t word = ((int64_t)grp * nimg_in + img) * kGrp + half * kRun + 3;
                v[q] = img < nimg_in && in_bounds(word, (int64_t)a.nk * nimg_in, a.err)
                           ? __ldcg(reinterpret_cast<const uint4 *>(xg + (size_t)img * 32))
                           : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int img = img0 + q * kMT + tid;
                if (img >= nimg_in) break;
                const uint32_t off = sw_off16(img / a.cin, img % a.cin);
                const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int r = 0; r < kRun; ++r) {
                    char *m = xo + r * kXMode;
                    *reinterpret_cast<unsigned short *>(m + off) = (unsigned short)(w4[r] & 0xFFFF);
                    *reinterpret_cast<unsigned short *>(m + nbp * 128 + off) =
                        (unsigned short)(w4[r] >> 16);
                }
            }
        }
    };
    const uint32_t tmem = s_tmem;
    const uint32_t idesc = idesc_f16(nbp, Bits<T>::kBf16);
    uint32_t *stage = reinterpret_cast<uint32_t *>(base + kOffStage);
    bool ok = true;
    // the first unit's weights (independent of kernel A), then its kept modes
    const int u0 = blockIdx.x;
    if constexpr (kImg) {
        if (tid == 0 && u0 < nunits) fetch_w(u0);
    }
    pdl_trigger();
    pdl_wait();                                  // kernel A's kept modes are complete
    if (u0 < nunits) load_x(u0, base);
    fence_async_smem();
    uint32_t it = 0;
    for (int u = u0; u < nunits; u += gridDim.x, ++it) {
        const unsigned long long t0 = a.trace ? trace_now() : 0;
        const int nxt = u + (int)gridDim.x;
        char *xo = base + (it & 1) * kXUnit;
        const uint32_t tb = tmem + (it & 1) * (kTmemCols / 2);
        // a. the unit's weight slots: packed images arrive and Wi^T is negated
        //    into each slot's first third, or the slots are built from the weights
        for (int r = 0; r < kRun; ++r) {
            char *slot = slot_at(r);
            if constexpr (kImg) {
                ok &= mbar_wait(&bar_w[r], it & 1, a.err);
                for (int e = tid; e < (int)(kHalfTile / 16); e += kMT) {   // exact sign flip
                    const uint4 v = reinterpret_cast<const uint4 *>(slot + 2 * kHalfTile)[e];
                    reinterpret_cast<uint4 *>(slot)[e] =
                        make_uint4(v.x ^ 0x80008000u, v.y ^ 0x80008000u, v.z ^ 0x80008000u,
                                   v.w ^ 0x80008000u);
                }
            } else {
                build_w(r, u * kRun + r);
            }
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();                         // slots, X operands, staging reads done
        const unsigned long long t1 = a.trace ? trace_now() : 0;
        // b. one chain per mode into this unit's half of tensor memory; thread 0
        //    then refills the slots with the next unit's images once they are read
        if (tid == 0) {
            tc_after_sync();
            if (ok) {
                for (int r = 0; r < kRun; ++r) {
                    const uint32_t am0 = tc_smem_addr(slot_at(r));
                    const uint32_t bm = tc_smem_addr(xo + r * kXMode);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t am = am0 + (c == 0 ? kHalfTile : 0u);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            mma_f16(tb + r * nbp, desc_sw128(am + q * 32),
                                    desc_sw128(bm + c * nbp * 128 + q * 32), idesc,
                                    (c | q) ? 1u : 0u);
                    }
                }
            }
            mma_commit(&bar_m[it & 1]);
            if constexpr (kImg) {
                if (nxt < nunits) {
                    ok &= mbar_wait(&bar_m[it & 1], (it >> 1) & 1, a.err);
                    fetch_w(nxt);
                }
            }
        }
        // c. the next unit's kept modes into the other X buffer (its previous
        //    unit's MMAs were waited for in the previous iteration)
        if (nxt < nunits) load_x(nxt, base + ((it + 1) & 1) * kXUnit);
        fence_async_smem();
        // d. tensor memory -> staging: D row m = o (re) or 64 + o (im), column b;
        //    staged image row (b * Cout + o) of 5 words, word r = mode r (re, im)
        ok &= mbar_wait(&bar_m[it & 1], (it >> 1) & 1, a.err);
        tc_after_sync();
        const unsigned long long t2 = a.trace ? trace_now() : 0;
        {
            const int m = 32 * (warp & 3) + lane;
            const int o = m % kCh, part = m / kCh;
            // warps w, w + 4, ... share tensor-memory lanes: each group of four warps
            // drains its own modes
            for (int r = warp >> 2; r < kRun; r += kMT / 128) {
                for (int g = 0; g < nbp / 16; ++g) {
                    float v[16];
                    tmem_ld16(tb + ((uint32_t)(32 * (warp & 3)) << 16) + r * nbp + 16 * g, v);
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
        // e. Y in the group layout: each image's 4 modes as one 16-byte piece of
        //    its 32-byte group row, so a warp's 32 consecutive images fill 1 KiB
        {
            const int grp = u / 2, half = u % 2;
            uint32_t *yg = static_cast<uint32_t *>(a.Y) + (size_t)grp * nimg_out * kGrp + half * kRun;
            for (int img = tid; img < nimg_out; img += kMT) {
                const uint32_t *sv = stage + (size_t)img * kStageRow;
                const int64_t word = ((int64_t)grp * nimg_out + img) * kGrp + half * kRun + 3;
                if (in_bounds(word, (int64_t)a.nk * nimg_out, a.err))
                    *reinterpret_cast<uint4 *>(yg + (size_t)img * kGrp) =
                        make_uint4(sv[0], sv[1], sv[2], sv[3]);
            }
        }
        if (a.trace) {
            __syncthreads();
            if (tid == 0) {
                unsigned smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                fno_trace_record_t rec;
                rec.item = (1u << 24) | ((unsigned)u & 0xFFFFFFu);
                rec.worker = smid;
                rec.t_start = t0;
                rec.t_ready = t1;
                rec.t_compute = t2;
                rec.t_end = trace_now();
                a.trace[a.trace_first + u] = rec;
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

int mixtc_items(int64_t nkept) { return (int)(nkept / kRun); }

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
    const int nunits = args.nk / kRun;
    cfg.gridDim = dim3((unsigned)(nunits < args.num_sms ? nunits : args.num_sms));
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
