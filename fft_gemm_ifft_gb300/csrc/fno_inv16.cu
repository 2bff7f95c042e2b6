// fno_inv16.cu -- kernel C of the 16-bit 256 x 256 layer (32 x 32 modes per
// corner block): the zero-padded inverse real FFT of the TurboFNO article
// (gsyq.cn/news/457482) §2.3 / §3.3, as two tensor-core GEMMs per output image
// in one persistent kernel.
//
// For an output image (b, o) the mixed modes V[j][k] (16-bit (re, im) pairs from
// the tensor-core mixing, stored in groups of 8 modes [group][image][8] and
// gathered by one TMA load per image; kept row j = 0..63 with
// the signed frequency g = j for j < 32 and j - 64 otherwise, bin k = 0..31)
// give
//   column inverse  Zo[t][k] = sum_j V[j][k] e^{+2 pi i g t / 256}     (t = 0..255)
//   row inverse     y[t][n]  = (1 / 256^2) sum_k c(k) Re(Zo[t][k] e^{+2 pi i k n / 256})
// with c(0) = 1 and c(k) = 2 for the other kept bins.  Both are real GEMMs on
// tcgen05 (kind::f16: fp16 or bf16 operands, the storage type of the layer, float32
// accumulation in tensor memory):
//   GEMM 1  D1[t][n] = sum_kappa E[t][kappa] B1[n][kappa]          M = 256, N = 64, K = 128
//           E = [cos(2 pi g t / 256) | sin(2 pi g t / 256)]  (kappa = j, then 64 + j)
//           B1[k]      = [ Vr[.][k] | -Vi[.][k] ]   (column k < 32 of D1 = Re Zo)
//           B1[32 + k] = [ Vi[.][k] |  Vr[.][k] ]   (column 32 + k     = Im Zo)
//   GEMM 2  D2[t][n] = sum_q A2[t][q] T[n][q]                        M = 256, N = 256, K = 64
//           A2 = [Re Zo' | Im Zo'], Zo' = Zo / 256 (exact: a power of two)
//           T[n] = [c(k) cos(2 pi k n / 256) | -c(k) sin(2 pi k n / 256)]
//   and y = D2 / 256, rounded once to the storage type.
// D1 leaves tensor memory as the K-major operand A2 (each thread writes its row's
// 64 values as eight 16-byte pieces), D2 leaves it through a ring of four
// 128 x 64 staging boxes that TMA stores write out while the threads drain
// the next box, so an image's output streams to HBM under the next image's
// loads and GEMMs.  One CTA per SM walks the images; the mixed modes of the
// next image are fetched by one bulk copy as soon as the current image's have
// been turned into its operand.
#include <cmath>
#include <cstring>
#include <type_traits>
#include <vector>

#include "fno_fused.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

constexpr int kN = 256, kM = 32, kK0 = 64, kNK = kK0 * kM;   // grid, modes, kept rows
constexpr int kThreads = 256;
constexpr uint32_t kTile = 16384;                 // 128 rows x 128 bytes
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kOffE = 0;                     // [tile 2][chunk 2] GEMM-1 A, 64 KiB
constexpr uint32_t kOffT = kOffE + 4 * kTile;     // GEMM-2 B: 256 rows x 128 B, 32 KiB
constexpr uint32_t kOffB1 = kOffT + 2 * kTile;    // GEMM-1 B: [chunk 2][64 rows], 16 KiB
constexpr uint32_t kOffA2 = kOffB1 + kTile;       // GEMM-2 A: [tile 2], 32 KiB
constexpr uint32_t kOffY = kOffA2 + 2 * kTile;    // mixed modes of one image, 16-bit pairs, 8 KiB
constexpr uint32_t kYBytes = kNK * 4;
constexpr uint32_t kOffS = kOffY + kYBytes;       // staging ring: 4 boxes of 128 x 64, 64 KiB
constexpr uint32_t kSmem = kOffS + 4 * kTile + 1024;
constexpr uint32_t kTablesBytes = 6 * kTile;      // E then T, as they sit in shared memory
constexpr uint32_t kTmemCols = 512;
static_assert(kSmem <= 232448 - 256, "one CTA per SM");

template <typename T> struct Kind;
template <> struct Kind<__half> { static constexpr bool kBf16 = false; };
template <> struct Kind<__nv_bfloat16> { static constexpr bool kBf16 = true; };

template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
    uint32_t u;
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(lo, hi);
        memcpy(&u, &h, 4);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        memcpy(&u, &h, 4);
    }
    return u;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(tc_smem_addr(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(tc_smem_addr(bar)) : "memory");
}

// 64 consecutive accumulator columns of this thread's lane, times `scale`,
// rounded to T and written as one 128-byte K-major row of a swizzled tile.
template <typename T>
__device__ __forceinline__ void drain_row64(uint32_t taddr, float scale, bool ok, char *tile,
                                            int row) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        float v[16];
        tmem_ld16(taddr + 16 * g, v);
        uint32_t pk[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            pk[q] = ok ? pack_pair<T>(v[2 * q] * scale, v[2 * q + 1] * scale) : 0u;
        *reinterpret_cast<uint4 *>(tile + sw_off16(row, 16 * g)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(tile + sw_off16(row, 16 * g + 8)) =
            make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
k_inv16(const __grid_constant__ CUtensorMap ymap, const __grid_constant__ CUtensorMap gmap,
        Inv16Args a, const void *tables, int nimg) {
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_t, bar_y, bar_m1, bar_m2a, bar_m2b;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = tc_smem_addr(base);
    const uint32_t *ys = reinterpret_cast<const uint32_t *>(base + kOffY);   // (re, im) pairs
    if (tid == 0) {
        uint64_t *bars[5] = {&bar_t, &bar_y, &bar_m1, &bar_m2a, &bar_m2b};
        for (int i = 0; i < 5; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(bars[i])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // both constant operands in their swizzled images, one bulk copy
        bulk_load(sbase + kOffE, tables, kTablesBytes, &bar_t);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");   // kernel B's mixed modes are complete
    // an image's mixed modes: its row of each of the 256 groups of 8 modes, one
    // TMA load that lands them in kept-mode order
    auto load_y = [&](int img) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(tc_smem_addr(&bar_y)), "r"(kYBytes) : "memory");
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%2, %3, %4}], [%5];"
                     ::"r"(sbase + kOffY), "l"(&gmap), "r"(0), "r"(img), "r"(0),
                       "r"(tc_smem_addr(&bar_y)) : "memory");
    };
    if (tid == 0 && (int)blockIdx.x < nimg) load_y(blockIdx.x);
    bool ok = mbar_wait(&bar_t, 0, a.err);
    constexpr uint32_t id1 = idesc_f16(64, Kind<T>::kBf16);
    constexpr uint32_t id2 = idesc_f16(256, Kind<T>::kBf16);
    const int half = warp >> 2;                  // warps w and w + 4 share TMEM lanes
    const int lrow = 32 * (warp & 3) + lane;     // this thread's row of a 128-row tile
    const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t it = 0, round = 0;
    for (int img = blockIdx.x; img < nimg; img += gridDim.x, ++it) {
        const long long t0 = a.trace ? tc_globaltimer() : 0;
        ok &= mbar_wait(&bar_y, it, a.err);
        const long long t1 = a.trace ? tc_globaltimer() : 0;
        // 1. GEMM-1 B operand from the mixed modes: thread (k, group of 8 kept rows)
        {
            const int k = lane, j0 = 8 * warp;
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = ys[(j0 + u) * kM + k];
            uint32_t re[4], nim[4], im[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                re[q] = __byte_perm(v[2 * q], v[2 * q + 1], 0x5410);   // low halves
                im[q] = __byte_perm(v[2 * q], v[2 * q + 1], 0x7632);   // high halves
                nim[q] = im[q] ^ 0x80008000u;        // sign flip of both halves (exact)
            }
            char *b1 = base + kOffB1;
            constexpr uint32_t kChunk = 64 * 128;
            *reinterpret_cast<uint4 *>(b1 + sw_off16(k, j0)) = make_uint4(re[0], re[1], re[2], re[3]);
            *reinterpret_cast<uint4 *>(b1 + kChunk + sw_off16(k, j0)) =
                make_uint4(nim[0], nim[1], nim[2], nim[3]);
            *reinterpret_cast<uint4 *>(b1 + sw_off16(32 + k, j0)) =
                make_uint4(im[0], im[1], im[2], im[3]);
            *reinterpret_cast<uint4 *>(b1 + kChunk + sw_off16(32 + k, j0)) =
                make_uint4(re[0], re[1], re[2], re[3]);
        }
        fence_async_smem();
        tc_before_sync();
        __syncthreads();                         // B1 written, the Y buffer is read
        tc_after_sync();
        if (tid == 0) {
            const int next = img + (int)gridDim.x;
            if (next < nimg) load_y(next);       // the next image's modes land under this one
            if (ok) {
                for (int t = 0; t < 2; ++t)
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            mma_f16(tmem + 64 * t,
                                    desc_sw128(sbase + kOffE + (2 * t + c) * kTile + 32 * s),
                                    desc_sw128(sbase + kOffB1 + c * 8192 + 32 * s), id1,
                                    (c | s) ? 1u : 0u);
            }
            mma_commit(&bar_m1);
        }
        ok &= mbar_wait(&bar_m1, it, a.err);
        tc_after_sync();
        // 2. D1 -> A2 = Zo / 256 in the storage type (warps 0-3 tile 0, 4-7 tile 1)
        drain_row64<T>(tmem + tlane + 64 * half, 1.f / kN, ok, base + kOffA2 + half * kTile,
                       lrow);
        fence_async_smem();
        tc_before_sync();
        __syncthreads();
        tc_after_sync();
        if (tid == 0) {
            if (ok) {
                for (int t = 0; t < 2; ++t) {
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_f16(tmem + 256 * t, desc_sw128(sbase + kOffA2 + t * kTile + 32 * s),
                                desc_sw128(sbase + kOffT + 32 * s), id2, s ? 1u : 0u);
                    mma_commit(t == 0 ? &bar_m2a : &bar_m2b);
                }
            } else {
                mma_commit(&bar_m2a);
                mma_commit(&bar_m2b);
            }
        }
        // 3. D2 -> staging ring -> TMA stores.  Round r of a tile: half h drains the
        //    64-column block 2h + r into slot 2h + r; the slot was last used two
        //    rounds ago, whose store group must have finished reading it.
        for (int t = 0; t < 2; ++t) {
            ok &= mbar_wait(t == 0 ? &bar_m2a : &bar_m2b, it, a.err);
            tc_after_sync();
            for (int r = 0; r < 2; ++r, ++round) {
                if (tid == 0 && round >= 2)
                    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                __syncthreads();
                const int cb = 2 * half + r;
                drain_row64<T>(tmem + tlane + 256 * t + 64 * cb, 1.f / kN, ok,
                               base + kOffS + cb * kTile, lrow);
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    for (int h = 0; h < 2; ++h) {
                        const int c2 = 2 * h + r;
                        tma_store_2d(&ymap, 64 * c2, img * kN + 128 * t,
                                     sbase + kOffS + c2 * kTile);
                    }
                    bulk_commit();
                }
            }
        }
        tc_before_sync();
        if (a.trace) {                           // one record per image, once its stores are issued
            __syncthreads();
            if (tid == 0) {
                unsigned smid;
                asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
                fno_trace_record_t rec;
                rec.item = (2u << 24) | ((unsigned)img & 0xFFFFFFu);
                rec.worker = smid;
                rec.t_start = (uint64_t)t0;
                rec.t_ready = (uint64_t)t1;
                rec.t_compute = rec.t_end = (uint64_t)tc_globaltimer();
                a.trace[a.trace_first + img] = rec;
            }
        }
    }
    if (tid == 0) bulk_wait_all();               // the output has left shared memory
    tc_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
    }
}

}  // namespace

size_t inv16_tables_bytes() { return kTablesBytes; }

// E (GEMM-1 A) and T (GEMM-2 B) in their swizzled shared-memory images,
// computed in double and rounded once to the storage type.
void inv16_make_tables(fno_dtype_t dtype, std::vector<unsigned char> &img) {
    img.assign(kTablesBytes, 0);
    const double two_pi = 2.0 * M_PI;
    auto put = [&](size_t off, double v) {
        if (dtype == FNO_F16) {
            const __half h = __float2half_rn((float)v);
            memcpy(&img[off], &h, 2);
        } else {
            const __nv_bfloat16 h = __float2bfloat16_rn((float)v);
            memcpy(&img[off], &h, 2);
        }
    };
    // E: row t, kappa = j (cos) or 64 + j (sin); tile t / 128, chunk kappa / 64
    for (int t = 0; t < kN; ++t)
        for (int j = 0; j < kK0; ++j) {
            const int g = j < kM ? j : j - kK0;
            const double ang = two_pi * (double)g * (double)t / (double)kN;
            const size_t tile = (size_t)(t / 128) * 2;
            put(kOffE + (tile + 0) * kTile + sw_off16(t % 128, j), std::cos(ang));
            put(kOffE + (tile + 1) * kTile + sw_off16(t % 128, j), std::sin(ang));
        }
    // T: row n, q = k (c(k) cos) or 32 + k (-c(k) sin)
    for (int n = 0; n < kN; ++n)
        for (int k = 0; k < kM; ++k) {
            const double ck = k == 0 ? 1.0 : 2.0;
            const double ang = two_pi * (double)k * (double)n / (double)kN;
            put(kOffT + sw_off16(n, k), ck * std::cos(ang));
            put(kOffT + sw_off16(n, kM + k), -ck * std::sin(ang));
        }
}

cudaError_t inv16_init(fno_dtype_t dtype) {
    if (dtype == FNO_F16) return raise_smem_limit(k_inv16<__half>, (int)kSmem);
    if (dtype == FNO_BF16) return raise_smem_limit(k_inv16<__nv_bfloat16>, (int)kSmem);
    return cudaErrorInvalidValue;
}

// Launch after kernel B with programmatic dependent launch; one CTA per SM
// (at most one per output image).
cudaError_t inv16_launch(fno_dtype_t dtype, const Inv16Args &a, const void *tables,
                         int64_t nimg, int num_sms, cudaStream_t s) {
    CUtensorMap ymap, gmap;
    const size_t eb = 2;
    if (!encode_rows_tiled(&ymap, a.y, nimg * kN, kN, eb, 64,
                           dtype == FNO_F16 ? tma_type<__half>() : tma_type<__nv_bfloat16>()))
        return cudaErrorInvalidValue;
    if (!encode_group_gather(&gmap, a.Y, 8, nimg, kNK / 8)) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nimg < num_sms ? nimg : num_sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (dtype == FNO_F16)
        e = cudaLaunchKernelEx(&cfg, k_inv16<__half>, ymap, gmap, a, tables, (int)nimg);
    else
        e = cudaLaunchKernelEx(&cfg, k_inv16<__nv_bfloat16>, ymap, gmap, a, tables, (int)nimg);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace fno
