// fno_mix_tf32.cu -- the per-mode channel mixing on the tensor cores for
// float32 storage: kernel B of the fp32 128 x 128 three-kernel layer.
//
// The mixing of the TurboFNO article (gsyq.cn/news/457482) §2.2, Y[b,o,k] =
// sum_i X[b,i,k] W[i,o,k], is per kept mode k a complex (B x Cin) . (Cin x Cout)
// product.  With the output channels on the M side and both weight parts
// stacked in one operand,
//
//     A = [ Wr^T ]  (M = 2 Cout rows, K = Cin),   D1 = A Xr,   D2 = A Xi,
//         [ Wi^T ]
//
// the real-block product needs only A, read twice:
//
//     Yr = Wr^T Xr - Wi^T Xi = D1[top] - D2[bottom],
//     Yi = Wi^T Xr + Wr^T Xi = D1[bottom] + D2[top],
//
// so a mode's weight operand holds each weight once (no negated or repeated
// copy).  Each product is 3xTF32 (hi*hi + hi*lo + lo*hi, hi = the value at tf32
// precision, lo = the exact remainder) on kind::tf32 tcgen05.mma with M = 128,
// N = the batch rows (padded to the MMA's granularity), accumulating in tensor
// memory.  With 32 output channels two modes share the M = 128 rows and their
// kept modes sit side by side on N (the product's off-diagonal blocks are not
// read).
//
// One CTA per pair of adjacent kept modes (the pair is adjacent in the kept
// order of the modes X and Y are indexed by, and in its weight block, so each
// (i, o) weight pair is one 16-byte load and each image's pair of kept modes
// one 16-byte load).  The weights are read into registers before the kernel
// waits for the forward transform (programmatic dependent launch); then the
// kept modes are split into the B operands, each mode group's A operand is
// written from the registers, one thread issues the two MMA chains, and the
// rows of the bottom half hand their products to the top half through shared
// memory, which combines and stores Y.
#include "fno_fused.cuh"

#include "fno_fused_dev.cuh"
#include "fno_tc.cuh"

namespace fno {
namespace {

using namespace tcu;

constexpr int kMT = 512;                     // threads: four warps per lane quarter
constexpr uint32_t kAChunk = 128u * 128u;    // 128 rows x 128 bytes (32 fp32 of K)

__host__ __device__ constexpr int groups_of(int cout) { return 128 / (2 * cout); }
// tensor memory: per mode group D1 and D2, at most 32 columns each
__host__ __device__ constexpr uint32_t tmem_cols(int cout) { return groups_of(cout) == 1 ? 128u : 64u; }

// batch rows of one mode on N (the MMA's N = G * nb is a multiple of 16)
__host__ __device__ inline int rows_per_mode(int cout, int batch) {
    return groups_of(cout) == 1 ? (batch <= 16 ? 16 : 32) : (batch <= 8 ? 8 : 16);
}

// shared memory: per mode group the A operand (hi, lo), then per mode group
// the B operand [Xr ; Xi] (2n rows x K, hi then lo: one MMA chain gives D1 in
// columns 0..n-1 and D2 in n..2n-1 of the group's accumulator); the top/bottom
// exchange reuses the A operands once the MMAs are done
struct MixLayout {
    int kc, g, ngrp, nb, n;
    uint32_t a_bytes, b_chunk, b_group, total;
};
__host__ __device__ inline MixLayout mix_layout(int cin, int cout, int batch) {
    MixLayout m;
    m.kc = cin / 32;
    m.g = groups_of(cout);
    m.ngrp = 2 / m.g;
    m.nb = rows_per_mode(cout, batch);
    m.n = m.g * m.nb;
    m.a_bytes = 2u * m.kc * kAChunk;                 // one group's A (hi + lo)
    m.b_chunk = (uint32_t)(2 * m.n) * 128u;          // rows: Xr (n), then Xi (n)
    m.b_group = 2u * m.kc * m.b_chunk;               // hi, then lo
    m.total = m.ngrp * (m.a_bytes + m.b_group) + 1024u;
    return m;
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[8]) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = __uint_as_float(r[i]);
        v[i + 4] = 0.f;
    }
}

// fp32 element (row, k) of a K-major operand of `rows` rows, 128-byte swizzle,
// K chunks of 32
__device__ __forceinline__ uint32_t op_off(int row, int k, uint32_t chunk_bytes) {
    return (uint32_t)(k >> 5) * chunk_bytes + sw_off(row, k & 31);
}
__device__ __forceinline__ void put_split(char *hi, char *lo, uint32_t off, float v) {
    *reinterpret_cast<float *>(hi + off) = v;
    *reinterpret_cast<float *>(lo + off) = tf32_lo(v);
}

template <int CIN, int COUT>
__global__ void __launch_bounds__(kMT, 1) k_mix_tf32(const MixTf32Args a) {
    constexpr int G = groups_of(COUT), NGRP = 2 / G, KC = CIN / 32;
    constexpr int kW = CIN * COUT / kMT;                  // weight pairs per thread
    static_assert(CIN * COUT % kMT == 0 && 2 * COUT * G == 128, "tiling");
    const MixLayout L = mix_layout(CIN, COUT, a.batch);
    const int nb = L.nb, n = L.n;
    extern __shared__ __align__(1024) char smem_raw[];
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    char *A = base;                                       // group gi: A + gi * a_bytes
    char *B = base + NGRP * L.a_bytes;                    // group gi: B + gi * b_group
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    const unsigned long long t0 = a.trace ? trace_now() : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u = blockIdx.x, k0 = 2 * u;                 // the pair's first kept mode
    // the pair's weight block and position in it (kept row j: the low rows
    // first, then the high ones; the pair starts at an even column)
    const int j = k0 / a.m1, c = k0 % a.m1;
    const int blk = j >= a.m0 ? 1 : 0;
    const int local = (j - blk * a.m0) * a.m1 + c;
    const size_t mblk = (size_t)a.m0 * a.m1;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem_addr(&bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    constexpr uint32_t kTmemCols = tmem_cols(COUT);
    // The weights do not come from the forward transform: the A operands are
    // written while it finishes.  W[blk][i][o][local .. local + 1] = (re, im,
    // re, im) of the pair; lanes take consecutive i, so a warp writes whole
    // swizzled rows.  Rows of group gi: (g, h, o) = W_h[i][o] of mode g
    // (G == 2) or of mode gi (G == 1).
    {
        float4 wv[kW];
#pragma unroll
        for (int r = 0; r < kW; ++r) {
            const int e = tid + r * kMT, i = e % CIN, o = e / CIN;
            wv[r] = __ldg(reinterpret_cast<const float4 *>(
                a.w + ((((size_t)blk * CIN + i) * COUT + o) * mblk + local) * 2));
        }
#pragma unroll
        for (int q = 0; q < kW; ++q) {
            const int e = tid + q * kMT, i = e % CIN, oo = e / CIN;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                char *Ah = A + (G == 1 ? m : 0) * L.a_bytes, *Al = Ah + KC * kAChunk;
                const int rowbase = G == 1 ? 0 : m * 2 * COUT;
                const float wr = m ? wv[q].z : wv[q].x, wi = m ? wv[q].w : wv[q].y;
                put_split(Ah, Al, op_off(rowbase + oo, i, kAChunk), wr);
                put_split(Ah, Al, op_off(rowbase + COUT + oo, i, kAChunk), wi);
            }
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");   // kernel A's kept modes are complete
    const unsigned long long t1 = a.trace ? trace_now() : 0;
    // tensor memory only now: a CTA waiting for kernel A holds none of it
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(tc_smem_addr(&s_tmem)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }

    // the kept modes of the pair as the B operands [Xr ; Xi], rows = batch
    // (zero past it): G == 1, group m holds mode m; G == 2, group 0 holds mode
    // m at rows m * nb
    for (int e = tid; e < nb * CIN; e += kMT) {
        const int b = e / CIN, i = e % CIN;
        const float4 x = b < a.batch ? __ldcg(reinterpret_cast<const float4 *>(
                                           a.X + ((size_t)b * CIN + i) * a.nk + k0))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int row = G == 1 ? b : m * nb + b;
            char *bh = B + (G == 1 ? m : 0) * L.b_group, *bl = bh + KC * L.b_chunk;
            put_split(bh, bl, op_off(row, i, L.b_chunk), m ? x.z : x.x);
            put_split(bh, bl, op_off(n + row, i, L.b_chunk), m ? x.w : x.y);
        }
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        const uint32_t idesc = idesc_tf32(2 * n);         // N = [Xr ; Xi] rows
#pragma unroll
        for (int gi = 0; gi < NGRP; ++gi) {
            // descriptors of K step 0; a step adds its byte offset / 16
            const char *Ah = A + gi * L.a_bytes, *bh = B + gi * L.b_group;
            const uint64_t dah = desc_sw128(tc_smem_addr(Ah)),
                           dal = desc_sw128(tc_smem_addr(Ah + KC * kAChunk));
            const uint64_t dbh = desc_sw128(tc_smem_addr(bh)),
                           dbl = desc_sw128(tc_smem_addr(bh + KC * L.b_chunk));
            const uint32_t d = tmem + (uint32_t)(gi * 2 * n);
#pragma unroll
            for (int ks = 0; ks < CIN / 8; ++ks) {
                const uint64_t ao = ((ks >> 2) * kAChunk + (ks & 3) * 32) >> 4,
                               bo = ((ks >> 2) * L.b_chunk + (ks & 3) * 32) >> 4;
                mma_tf32(d, dah + ao, dbh + bo, idesc, ks ? 1u : 0u);
                mma_tf32(d, dah + ao, dbl + bo, idesc, 1u);
                mma_tf32(d, dal + ao, dbh + bo, idesc, 1u);
            }
        }
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0u, a.err);
    tc_after_sync();

    // epilogue: row r of D is TMEM lane r; warps w, w + 4, w + 8 and w + 12
    // share a lane quarter and take one quarter of the n columns each
    const int r = 32 * (warp & 3) + lane, cq = warp >> 2;
    const int g = r / (2 * COUT), h = (r / COUT) & 1, o = r % COUT;
    constexpr int kQ = 8;                                 // n / 4 <= 8 columns a warp
    const int nq = n / 4, c0 = cq * nq;
    const uint32_t la = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    float d1[NGRP][kQ], d2[NGRP][kQ];
#pragma unroll
    for (int gi = 0; gi < NGRP; ++gi) {
        const uint32_t col = la + (uint32_t)(gi * 2 * n + c0);
        if (nq == 8) {
            tmem_ld8(col, d1[gi]);
            tmem_ld8(col + n, d2[gi]);
        } else {
            tmem_ld4(col, d1[gi]);
            tmem_ld4(col + n, d2[gi]);
        }
        if (!ok) {
#pragma unroll
            for (int q = 0; q < kQ; ++q) d1[gi][q] = d2[gi][q] = 0.f;
        }
    }
    // the bottom rows (Wi^T X) hand their columns to the top rows (Wr^T X) of
    // the same mode and output channel; the exchange reuses the A operands
    float2 *E = reinterpret_cast<float2 *>(A);            // [gi][g * COUT + o][n]
    if (h == 1) {
#pragma unroll
        for (int gi = 0; gi < NGRP; ++gi)
#pragma unroll
            for (int q = 0; q < kQ; ++q)
                if (q < nq)
                    E[(gi * G * COUT + g * COUT + o) * n + c0 + q] =
                        make_float2(d1[gi][q], d2[gi][q]);
    }
    tc_before_sync();
    __syncthreads();
    if (h == 0) {
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const int col = c0 + q, b = col % nb;
            if (q < nq && col / nb == g && b < a.batch) {
                float yr[NGRP], yi[NGRP];
#pragma unroll
                for (int gi = 0; gi < NGRP; ++gi) {
                    const float2 ex = E[(gi * G * COUT + g * COUT + o) * n + col];
                    yr[gi] = d1[gi][q] - ex.y;
                    yi[gi] = ex.x + d2[gi][q];
                }
                float2 *yp = a.Y + ((size_t)b * COUT + o) * a.nk + k0;
                if constexpr (G == 1)
                    __stcg(reinterpret_cast<float4 *>(yp), make_float4(yr[0], yi[0], yr[1], yi[1]));
                else
                    __stcg(yp + g, make_float2(yr[0], yi[0]));
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
    if (a.trace && tid == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        fno_trace_record_t rec;
        rec.item = (1u << 24) | (unsigned)u;
        rec.worker = smid;
        rec.t_start = t0;
        rec.t_ready = t1;
        rec.t_end = trace_now();
        rec.t_compute = rec.t_end;
        a.trace[a.trace_first + u] = rec;
    }
}

template <int CIN, int COUT>
const void *kernel_for() {
    return reinterpret_cast<const void *>(&k_mix_tf32<CIN, COUT>);
}
const void *pick(int cin, int cout) {
    if (cin == 64) return cout == 64 ? kernel_for<64, 64>() : kernel_for<64, 32>();
    return cout == 64 ? kernel_for<32, 64>() : kernel_for<32, 32>();
}

}  // namespace

bool mixtf32_supported(int64_t batch, int cin, int cout, int m1, int64_t nkept) {
    const bool ch = (cin == 32 || cin == 64) && (cout == 32 || cout == 64);
    const int64_t maxb = groups_of(cout == 64 ? 64 : 32) == 1 ? 32 : 16;
    return ch && batch >= 1 && batch <= maxb && m1 % 2 == 0 && nkept % 2 == 0;
}

cudaError_t mixtf32_init() {
    // the largest layout: 64 input channels, 32 batch rows of one mode
    const MixLayout L = mix_layout(64, 64, 32);
    for (int ci : {32, 64})
        for (int co : {32, 64}) {
            const cudaError_t e = raise_smem_limit(pick(ci, co), L.total);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t mixtf32_launch(const MixTf32Args &a, cudaStream_t s) {
    if (!mixtf32_supported(a.batch, a.cin, a.cout, a.m1, a.nk)) return cudaErrorInvalidValue;
    const MixLayout L = mix_layout(a.cin, a.cout, a.batch);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.nk / 2));
    cfg.blockDim = dim3(kMT);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    MixTf32Args arg = a;
    void *args[] = {&arg};
    return cudaLaunchKernelExC(&cfg, pick(a.cin, a.cout), args);
}

}  // namespace fno
