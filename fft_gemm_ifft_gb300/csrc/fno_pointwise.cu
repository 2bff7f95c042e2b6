// fno_pointwise.cu -- the 1x1 linears of the FNO stack on the tensor cores.
//
// The stack is the model the TurboFNO article (gsyq.cn/news/457482) runs in
// its §5 tasks: a 1x1 lift, layers whose pointwise branch is a 1x1 linear with
// bias added to the spectral branch before the GELU, and a two-layer 1x1
// projection head with a GELU between.  A 1x1 linear over a channels-first
// tile is the dense GEMM D[p][o] = sum_i a[i][p] W[o][i]: M = 128 pixels,
// N = the output channels, K = the input channels, in 3xTF32 (hi*hi + hi*lo +
// lo*hi, hi = the value read at tf32 precision, lo = the exact remainder).
//
// One persistent CTA per SM walks the tiles (b, 128 pixels) with specialised
// warps handing work over through mbarriers; every global access is a TMA
// copy, so that no thread's synchronisation waits on its own loads or stores:
// * a load warp brings the activations [cin][128 pixels] into a ring of
//   two to four shared-memory stages, that many tiles ahead;
// * 16 compute warps (thread = one pixel row and a quarter of the channels:
//   kParts = 4 threads per pixel row; 8 compute warps measured slower)
//   transpose and split a tile's activations into the K-major 128-byte-
//   swizzled A operand, then run the previous tile's epilogue: a layer adds
//   bias and spectral branch and applies the GELU in place in the branch
//   tile; the head applies bias and GELU per hidden unit and sums the second
//   projection over the four threads of a pixel;
// * an MMA warp issues each tile's chains into one of two tensor-memory
//   accumulators, so that they run under the previous tile's epilogue;
// * a store warp (layers) writes each finished branch tile out with one TMA
//   store and refills it with the spectral branch of the tile two ahead.
// The kernel is launched as a programmatic dependent of the preceding one:
// barriers, tensor memory and the weights are set up under that kernel's
// tail, and the load and store warps wait for it before their first copy
// (so the weights, biases and head parameters must not come from a kernel
// that lets its dependents start early; the layer kernels do not write them).
#include "fno_pointwise.cuh"

#include "fno_gelu.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

constexpr int kCompute = 512;            // compute threads: kParts per pixel row of a tile
constexpr int kWarps = kCompute / 32;
constexpr int kParts = kWarps / 4;       // compute warps sharing one tensor-memory lane quarter
constexpr int kThreads = kCompute + 96;  // + the load, MMA and store warps
constexpr int kRows = 128;               // M: pixels per tile
constexpr uint32_t kChunk = 16384;       // 128 rows x 128 bytes = 32 fp32 of K
constexpr int kMaxC2 = 8;                // head outputs

constexpr uint32_t align1k(uint32_t v) { return (v + 1023u) & ~1023u; }

// Shared-memory map (offsets from a 1024-aligned base).  KC = K chunks of 32
// input channels, NG = groups of 16 output channels.
template <int KC, int NG, bool HEAD, int C2, typename T>
struct Lay {
    static constexpr int kN = 16 * NG;
    static constexpr int kK = 32 * KC;
    static constexpr uint32_t kLimit = 227u * 1024u;
    static constexpr uint32_t kWChunk = (uint32_t)kN * 128;     // n rows x 128 bytes
    static constexpr uint32_t kW = 0, kWlo = KC * kWChunk;      // B operand, hi then lo
    static constexpr uint32_t kA = 2 * KC * kWChunk;            // A operand, hi then lo
    static constexpr uint32_t kAlo = kA + KC * kChunk;
    static constexpr uint32_t kX = kA + 2 * KC * kChunk;        // ring of [cin][128] tiles
    static constexpr uint32_t kXBytes = align1k((uint32_t)(kK * kRows * sizeof(T)));
    static constexpr uint32_t kSBytes = align1k((uint32_t)(kN * kRows * sizeof(T)));
    // the kernel's static shared memory (biases, head weights and partial
    // sums, barriers), bounded from above; it comes in whole kilobytes ahead
    // of the 1024-aligned dynamic part
    static constexpr uint32_t kStatic =
        align1k(4u * (kN + (HEAD ? C2 * kN + 2 * (kParts - 1) * C2 * kRows : 1) + C2) + 512);
    // as many activation stages (at most four) as the shared memory holds
    // beside the operands and, for a layer, two branch tiles
    static constexpr uint32_t kFixed = kX + (HEAD ? 0u : 2 * kSBytes) + 1024 + kStatic;
    static constexpr int kNX =
        (int)((kLimit - kFixed) / kXBytes) < 4 ? (int)((kLimit - kFixed) / kXBytes) : 4;
    static constexpr uint32_t kS = kX + kNX * kXBytes;          // layer: 2 x [n][128]
    static constexpr uint32_t kAlloc = kS + (HEAD ? 0u : 2 * kSBytes) + 1024;
    static_assert(kNX >= 2, "two activation stages");
    static constexpr uint32_t kCols = 2 * kN;                   // two accumulators
    static_assert(kAlloc + kStatic <= kLimit, "shared memory");
};

struct KParams {
    const float *W, *bias, *P2, *c2;
    void *out;                 // head: [batch][cout2][npix]
    int cin, n, cout2, gelu, has_add;
    int64_t npix, ptiles, ntiles;
    int *err;
};

// mbarrier arrival of one elected lane per warp (the warp's earlier shared-
// memory writes and tensor-memory loads are ordered before it by the caller)
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_addr(bar))
                     : "memory");
}
__device__ __forceinline__ void thread_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_addr(bar)) : "memory");
}
// barrier of the compute warps alone
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

template <int KC, int NG, bool HEAD, int C2, typename T>
__global__ void __launch_bounds__(kThreads, 1)
k_pointwise_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap,
               const __grid_constant__ CUtensorMap omap, const KParams p) {
    using L = Lay<KC, NG, HEAD, C2, T>;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    // x_full / x_empty: activation stages; a_full / a_empty: the A operand;
    // acc_full / acc_empty: the two accumulators; s_full / s_done: the two
    // branch tiles (loaded or free / written by the epilogue)
    __shared__ __align__(8) uint64_t x_full[L::kNX], x_empty[L::kNX], a_full, a_empty,
        acc_full[2], acc_empty[2], s_full[2], s_done[2];
    __shared__ uint32_t s_tmem;
    __shared__ __align__(16) float s_bias[L::kN];        // read as float4
    __shared__ float s_p2[HEAD ? C2 * L::kN : 1], s_c2[C2];
    // head: the partial second projections of parts 1.. of a pixel, two tiles
    __shared__ float s_red[HEAD ? 2 * (kParts - 1) * C2 * kRows : 1];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int cin = p.cin, n = p.n;

    if (tid == 0) {
        auto init = [](uint64_t *b, uint32_t count) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem_addr(b)),
                         "r"(count));
        };
        for (int k = 0; k < L::kNX; ++k) {
            init(&x_full[k], 1);
            init(&x_empty[k], kWarps);
        }
        init(&a_full, kWarps);
        init(&a_empty, 1);
        for (int k = 0; k < 2; ++k) {
            init(&acc_full[k], 1);
            init(&acc_empty[k], kWarps);
            init(&s_full[k], 1);
            init(&s_done[k], kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(L::kCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // the kernel that follows may start its own set-up
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;

    // this CTA's tiles: blockIdx.x + j * gridDim.x, j < nt
    const int64_t nt =
        p.ntiles > (int64_t)blockIdx.x ? (p.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto tile_at = [&](int64_t j, int &c0, int &b) {
        const int64_t t = blockIdx.x + j * gridDim.x;
        b = (int)(t / p.ptiles);
        c0 = (int)((t % p.ptiles) * kRows);
    };
    auto s_tile = [&](int buf) { return base + L::kS + buf * L::kSBytes; };
    const bool has_add = !HEAD && p.has_add;

    if (warp == kWarps) {
        // ---- load warp: activation stages, kNX tiles ahead
        if ((tid & 31) == 0) {
            const uint64_t pol = l2_evict_first_policy();   // every tile is read once
            const uint32_t x_tx = (uint32_t)(cin * kRows * sizeof(T));
            auto issue_x = [&](int64_t j) {                 // tile j -> stage j % kNX
                int c0, b;
                tile_at(j, c0, b);
                const int st = (int)(j % L::kNX);
                arrive_expect_tx(&x_full[st], x_tx);
                tma_load_2d_hint(tc_smem_addr(base + L::kX + st * L::kXBytes), &xmap, c0,
                                 b * cin, &x_full[st], pol);
            };
            // the activations may come from the preceding kernel
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int64_t j = 0; j < L::kNX && j < nt; ++j) issue_x(j);
            for (int64_t j = 0; j + L::kNX < nt; ++j) {
                // stage j % kNX is free once tile j has been transposed
                const int st = (int)(j % L::kNX);
                mbar_wait(&x_empty[st], (uint32_t)(j / L::kNX), p.err);
                issue_x(j + L::kNX);
            }
        }
    } else if (warp == kWarps + 1) {
        // ---- MMA warp: tile j's 3xTF32 chains into accumulator j % 2
        if ((tid & 31) == 0) {
            constexpr uint32_t idesc = idesc_tf32(L::kN);
            const uint32_t ah = tc_smem_addr(base + L::kA), al = tc_smem_addr(base + L::kAlo);
            const uint32_t wh = tc_smem_addr(base + L::kW), wl = tc_smem_addr(base + L::kWlo);
            const int ksteps = (cin + 7) / 8;                 // K = 8 per tf32 MMA
            for (int64_t j = 0; j < nt; ++j) {
                const int buf = (int)(j & 1);
                mbar_wait(&a_full, (uint32_t)j, p.err);
                if (j >= 2) mbar_wait(&acc_empty[buf], (uint32_t)((j - 2) >> 1), p.err);
                tc_after_sync();
                const uint32_t d = tmem + (uint32_t)buf * L::kN;
                for (int k = 0; k < ksteps; ++k) {
                    const uint32_t ao = (k >> 2) * kChunk + (k & 3) * 32,
                                   bo = (k >> 2) * L::kWChunk + (k & 3) * 32;
                    mma_tf32(d, desc_sw128(ah + ao), desc_sw128(wh + bo), idesc, k ? 1u : 0u);
                    mma_tf32(d, desc_sw128(ah + ao), desc_sw128(wl + bo), idesc, 1u);
                    mma_tf32(d, desc_sw128(al + ao), desc_sw128(wh + bo), idesc, 1u);
                }
                mma_commit(&acc_full[buf]);
                mma_commit(&a_empty);
            }
        }
    } else if (warp == kWarps + 2) {
        // ---- store warp (layers): tile j's output leaves branch tile j % 2,
        // which then takes tile j + 2's spectral branch (or is merely free)
        if (!HEAD && (tid & 31) == 0) {
            const uint64_t pol = l2_evict_first_policy();
            const uint32_t s_tx = (uint32_t)(n * kRows * sizeof(T));
            auto ready_s = [&](int64_t j) {
                const int buf = (int)(j & 1);
                if (has_add) {
                    int c0, b;
                    tile_at(j, c0, b);
                    arrive_expect_tx(&s_full[buf], s_tx);
                    tma_load_2d_hint(tc_smem_addr(s_tile(buf)), &smap, c0, b * n, &s_full[buf],
                                     pol);
                } else {
                    thread_arrive(&s_full[buf]);
                }
            };
            // the spectral branch comes from the preceding kernel, and the
            // output may still be read by one before it
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int64_t j = 0; j < 2 && j < nt; ++j) ready_s(j);
            for (int64_t j = 0; j < nt; ++j) {
                const int buf = (int)(j & 1);
                mbar_wait(&s_done[buf], (uint32_t)(j >> 1), p.err);
                int c0, b;
                tile_at(j, c0, b);
                tma_store_2d(&omap, c0, b * n, tc_smem_addr(s_tile(buf)));
                bulk_commit();
                if (j + 2 < nt) {
                    bulk_wait_read();                        // the tile has been read out
                    ready_s(j + 2);
                }
            }
            bulk_wait_all();                                // the stores have landed
        }
    } else {
        // ---- compute warps: thread -> (pixel row, part); warps w, w+4, w+8,
        // w+12 share tensor-memory lanes
        const int row = 32 * (warp & 3) + (tid & 31), part = warp >> 2;
        // the weights, hi and lo, as the B operand (N rows = outputs, K =
        // inputs), zero past n outputs and cin inputs; every load in flight
        // before the first store (the activations are on their way meanwhile)
        {
            constexpr int kPer = (L::kN * L::kK + kCompute - 1) / kCompute;
            float w[kPer];
#pragma unroll
            for (int r = 0; r < kPer; ++r) {
                const int e = tid + r * kCompute, o = e / L::kK, i = e % L::kK;
                w[r] = (e < L::kN * L::kK && o < n && i < cin) ? p.W[(int64_t)o * cin + i] : 0.f;
            }
#pragma unroll
            for (int r = 0; r < kPer; ++r) {
                const int e = tid + r * kCompute, o = e / L::kK, i = e % L::kK;
                if (e < L::kN * L::kK) {
                    const uint32_t off = (uint32_t)(i / 32) * L::kWChunk + sw_off(o, i % 32);
                    *reinterpret_cast<float *>(base + L::kW + off) = w[r];
                    *reinterpret_cast<float *>(base + L::kWlo + off) = tf32_lo(w[r]);
                }
            }
        }
        for (int o = tid; o < L::kN; o += kCompute) s_bias[o] = o < n ? p.bias[o] : 0.f;
        if constexpr (HEAD) {
            for (int e = tid; e < C2 * L::kN; e += kCompute) {
                const int c = e / L::kN, o = e % L::kN;
                s_p2[e] = (c < p.cout2 && o < n) ? p.P2[(int64_t)c * n + o] : 0.f;
            }
            for (int c = tid; c < C2; c += kCompute) s_c2[c] = c < p.cout2 ? p.c2[c] : 0.f;
        }
        compute_sync();                               // biases and head weights are in place
        constexpr int kPerT = L::kK / kParts;                 // input channels per thread
        const int i0 = part * kPerT;
        for (int64_t j = 0; j <= nt; ++j) {
            if (j < nt) {
                // tile j: activations into the A operand (free once tile j - 1's
                // MMAs are done)
                const int st = (int)(j % L::kNX);
                mbar_wait(&x_full[st], (uint32_t)(j / L::kNX), p.err);
                if (j >= 1) mbar_wait(&a_empty, (uint32_t)(j - 1), p.err);
                const T *X = reinterpret_cast<const T *>(base + L::kX + st * L::kXBytes);
#pragma unroll
                for (int i4 = 0; i4 < kPerT / 4; ++i4) {
                    const int i = i0 + 4 * i4;
                    float v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        v[q] = (i + q < cin) ? Storage<T>::load(X + (i + q) * kRows + row) : 0.f;
                    const uint32_t off = (uint32_t)(i / 32) * kChunk + sw_off(row, i % 32);
                    *reinterpret_cast<float4 *>(base + L::kA + off) =
                        make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<float4 *>(base + L::kAlo + off) =
                        make_float4(tf32_lo(v[0]), tf32_lo(v[1]), tf32_lo(v[2]), tf32_lo(v[3]));
                }
                fence_async_smem();
                warp_arrive(&x_empty[st]);
                warp_arrive(&a_full);
            }
            if (j >= 1) {
                // tile j - 1: the epilogue, under tile j's MMAs
                const int64_t jj = j - 1;
                const int buf = (int)(jj & 1);
                mbar_wait(&acc_full[buf], (uint32_t)(jj >> 1), p.err);
                tc_after_sync();
                const uint32_t lane_addr =
                    tmem + (uint32_t)buf * L::kN + ((uint32_t)(32 * (warp & 3)) << 16);
                if constexpr (!HEAD) {
                    T *S = reinterpret_cast<T *>(s_tile(buf));
                    // groups part, part + kParts, ... of 16 outputs
                    constexpr int kG = (NG + kParts - 1) / kParts;
                    float v[kG][16];
#pragma unroll
                    for (int gg = 0; gg < kG; ++gg) {
                        const int g = part + kParts * gg;
                        if (g < NG && 16 * g < n) tmem_ld16(lane_addr + 16 * g, v[gg]);
                    }
                    tc_before_sync();
                    warp_arrive(&acc_empty[buf]);
                    mbar_wait(&s_full[buf], (uint32_t)(jj >> 1), p.err);
#pragma unroll
                    for (int gg = 0; gg < kG; ++gg) {
                        const int g = part + kParts * gg;
                        if (g < NG && 16 * g < n) {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const float4 b4 =
                                    *reinterpret_cast<const float4 *>(&s_bias[16 * g + 4 * q4]);
                                const float bq[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                                for (int q1 = 0; q1 < 4; ++q1) {
                                    const int q = 4 * q4 + q1;
                                    T *sp = S + (16 * g + q) * kRows + row;
                                    float r = v[gg][q] + bq[q1];
                                    if (has_add) r += Storage<T>::load(sp);
                                    if (p.gelu) r = gelu_erf(r);
                                    Storage<T>::store(sp, r);
                                }
                            }
                        }
                    }
                    fence_async_smem();
                    warp_arrive(&s_done[buf]);
                } else {
                    float hacc[C2];
#pragma unroll
                    for (int c = 0; c < C2; ++c) hacc[c] = 0.f;
#pragma unroll
                    for (int gg = 0; gg < (NG + kParts - 1) / kParts; ++gg) {
                        const int g = part + kParts * gg;
                        if (g < NG && 16 * g < n) {
                            float v[16];
                            tmem_ld16(lane_addr + 16 * g, v);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const float4 b4 =
                                    *reinterpret_cast<const float4 *>(&s_bias[16 * g + 4 * q4]);
                                const float bq[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const int o = 16 * g + 4 * q4 + q;
                                    const float h = gelu_erf(v[4 * q4 + q] + bq[q]);
#pragma unroll
                                    for (int c = 0; c < C2; ++c)
                                        hacc[c] = fmaf(s_p2[c * L::kN + o], h, hacc[c]);
                                }
                            }
                        }
                    }
                    tc_before_sync();
                    warp_arrive(&acc_empty[buf]);
                    // the kParts threads of a pixel sum their partial second
                    // projections (a buffer per tile parity: a warp is at most
                    // one tile ahead of another)
                    float *red = s_red + buf * (kParts - 1) * C2 * kRows;
                    if (part > 0) {
#pragma unroll
                        for (int c = 0; c < C2; ++c)
                            red[((part - 1) * C2 + c) * kRows + row] = hacc[c];
                    }
                    compute_sync();
                    int c0, b;
                    tile_at(jj, c0, b);
                    const int64_t px = c0 + row;
                    if (part == 0 && px < p.npix) {
                        // the head's only global stores: one value per pixel and output
                        T *op = static_cast<T *>(p.out) + (int64_t)b * p.cout2 * p.npix + px;
#pragma unroll
                        for (int c = 0; c < C2; ++c) {
                            if (c < p.cout2) {
                                float v = s_c2[c] + hacc[c];
#pragma unroll
                                for (int qq = 0; qq < kParts - 1; ++qq)
                                    v += red[(qq * C2 + c) * kRows + row];
                                Storage<T>::store(op + (int64_t)c * p.npix, v);
                            }
                        }
                    }
                }
            }
        }
    }
    tc_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(L::kCols));
    }
}

struct Pick {
    const void *fn;
    uint32_t smem;
};
template <int KC, int NG, bool HEAD, int C2, typename T>
Pick make_pick() {
    return {(const void *)k_pointwise_tc<KC, NG, HEAD, C2, T>, Lay<KC, NG, HEAD, C2, T>::kAlloc};
}
// layers and the lift: n <= 64; the head: n <= 128, one or up to eight outputs
template <typename T>
Pick pick(int cin, int cout2, bool head) {
    const bool k1 = cin <= 32;
    if (head) {
        if (cout2 <= 1) return k1 ? make_pick<1, 8, true, 1, T>() : make_pick<2, 8, true, 1, T>();
        return k1 ? make_pick<1, 8, true, kMaxC2, T>() : make_pick<2, 8, true, kMaxC2, T>();
    }
    return k1 ? make_pick<1, 4, false, 1, T>() : make_pick<2, 4, false, 1, T>();
}
Pick pick_dt(fno_dtype_t dt, int cin, int cout2, bool head) {
    return with_storage(dt, [&](auto t) { return pick<decltype(t)>(cin, cout2, head); });
}

}  // namespace

bool pointwise_supported(fno_dtype_t dt, int cin, int n, int cout2, bool head, int64_t npix) {
    if (!tcu::encoder()) return false;
    const size_t eb = dt == FNO_F32 ? 4 : 2;
    if (cin < 1 || cin > 64 || n < 16 || n % 16 != 0 || n > (head ? 128 : 64)) return false;
    if (head && (cout2 < 1 || cout2 > kMaxC2)) return false;
    return npix > 0 && (npix * (int64_t)eb) % 16 == 0 && npix < ((int64_t)1 << 31);
}

cudaError_t pointwise_init(fno_dtype_t dt, int cin, int n, int cout2, bool head) {
    (void)n;
    const Pick k = pick_dt(dt, cin, cout2, head);
    return raise_smem_limit(k.fn, k.smem);
}

cudaError_t pointwise_launch(fno_dtype_t dt, const PointwiseArgs &a, int num_sms,
                             cudaStream_t s) {
    const Pick k = pick_dt(dt, a.cin, a.cout2, a.head != 0);
    const size_t eb = dt == FNO_F32 ? 4 : 2;
    const CUtensorMapDataType ty =
        dt == FNO_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                      : (dt == FNO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    CUtensorMap xmap, smap, omap;
    if (!tcu::encode_rows_plain(&xmap, a.a, a.batch * a.cin, a.npix, eb, kRows, a.cin, ty))
        return cudaErrorInvalidValue;
    smap = omap = xmap;
    if (!a.head && a.add &&
        !tcu::encode_rows_plain(&smap, a.add, a.batch * a.n, a.npix, eb, kRows, a.n, ty))
        return cudaErrorInvalidValue;
    if (!a.head &&
        !tcu::encode_rows_plain(&omap, a.out, a.batch * a.n, a.npix, eb, kRows, a.n, ty))
        return cudaErrorInvalidValue;
    KParams kp;
    kp.W = a.W;
    kp.bias = a.bias;
    kp.P2 = a.P2;
    kp.c2 = a.c2;
    kp.out = a.out;
    kp.cin = a.cin;
    kp.n = a.n;
    kp.cout2 = a.head ? a.cout2 : 0;
    kp.gelu = a.gelu;
    kp.has_add = !a.head && a.add != nullptr;
    kp.npix = a.npix;
    kp.ptiles = (a.npix + kRows - 1) / kRows;
    kp.ntiles = a.batch * kp.ptiles;
    kp.err = a.err;
    if (kp.ntiles < 1) return cudaSuccess;
    const unsigned grid = (unsigned)std::min<int64_t>(kp.ntiles, std::max(num_sms, 1));
    // programmatic dependent launch: the set-up (weights, barriers, tensor
    // memory) overlaps the preceding kernel's tail; the load and store warps
    // wait for it before their first copy
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = k.smem;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    void *args[] = {&xmap, &smap, &omap, &kp};
    return cudaLaunchKernelExC(&cfg, k.fn, args);
}

}  // namespace fno
