// fno_tc.cuh -- tcgen05 building blocks shared by the tensor-core kernels:
// the 128-byte-swizzled K-major operand layout for 32-bit elements, its
// shared-memory descriptor, the tf32 instruction descriptor, the 3xTF32 split,
// MMA issue / commit, tensor-memory loads and a bounded mbarrier wait.
#pragma once

#include <cuda.h>

#include <cstring>

#include "fno_internal.cuh"

namespace fno {
namespace tcu {

__device__ __forceinline__ uint32_t tc_smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ long long tc_globaltimer() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
constexpr long long kTcWaitTimeoutNs = 500000000;   // bounded device waits: 0.5 s

// byte offset of (row, col) in a chunk of rows x 32 fp32 stored K-major with
// the 128-byte swizzle (8-row atoms of 1024 bytes, 16-byte pieces permuted by
// row % 8); the chunk must start on a 1024-byte boundary
__host__ __device__ inline uint32_t sw_off(int row, int col) {
    const uint32_t b = (uint32_t)col * 4, r = row & 7, j = b >> 4;
    return (uint32_t)(row >> 3) * 1024 + r * 128 + ((j ^ r) << 4) + (b & 15);
}
__host__ __device__ inline float tf32_lo(float v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    u &= 0xFFFFE000u;
    float h;
    memcpy(&h, &u, 4);
    return v - h;
}
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// instruction descriptor: D f32, A/B tf32, K-major, M = 128 (or m)
__host__ __device__ constexpr uint32_t idesc_tf32(int n, int m = 128) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(tc_smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// Bounded wait for the phase `n` (0, 1, 2, ...) of an mbarrier; on time-out the
// error word is set and the caller goes on (its results are then discarded).
__device__ inline bool mbar_wait(uint64_t *bar, uint32_t n, int *err) {
    const uint32_t a = tc_smem_addr(bar), parity = n & 1;
    uint32_t done = 0;
    long long t0 = 0;
    for (uint32_t spin = 0;; ++spin) {
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     "selp.u32 %0, 1, 0, p;\n}" : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
        if (spin == 0) t0 = tc_globaltimer();
        if ((spin & 1023u) == 1023u) {
            if (*reinterpret_cast<volatile int *>(err) != 0) return false;
            if (tc_globaltimer() - t0 > kTcWaitTimeoutNs) {
                raise_dev_error(err, kDevTimeout);
                return false;
            }
        }
    }
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                 "%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// registers -> tensor memory: lane = the thread's lane in its quarter, 16
// consecutive columns (the caller waits with tmem_st_wait before handing the
// columns to the tensor cores)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,"
                 "%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                   "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                   "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                   "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                   "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                   "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// D (tensor memory) += A (tensor memory, M = 128 lanes x K columns) x B
// (shared-memory descriptor), kind::tf32
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}"
                 ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// byte offset of (row, col) in a chunk of rows x 64 16-bit elements stored
// K-major with the 128-byte swizzle (same atoms as above, 8 elements per
// 16-byte piece)
__host__ __device__ inline uint32_t sw_off16(int row, int col) {
    const uint32_t b = (uint32_t)col * 2, r = row & 7, j = b >> 4;
    return (uint32_t)(row >> 3) * 1024 + r * 128 + ((j ^ r) << 4) + (b & 15);
}
// instruction descriptor: D f32, A/B f16 (bf16 = false) or bf16, K-major, M = 128
__host__ __device__ constexpr uint32_t idesc_f16(int n, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(tc_smem_addr(bar)) : "memory");
}

// An L2 policy that marks the lines it touches first to go (a stream read once)
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int c0,
                                                 int c1, uint64_t *bar, uint64_t policy) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(tc_smem_addr(bar)), "l"(policy)
                 : "memory");
}

// shared -> global tile store (bulk group); the source must stay untouched
// until bulk_wait_read() returns
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int c0, int c1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(map), "r"(c0), "r"(c1), "r"(src) : "memory");
}
__device__ __forceinline__ void arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(tc_smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ----- host: TMA tensor maps -----
typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's cuTensorMapEncodeTiled through the runtime's entry-point query
// (no link against the driver library); nullptr if unavailable.
inline EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(ptr);
        else
            cudaGetLastError();
    }
    return fn;
}

template <typename T> inline CUtensorMapDataType tma_type();
template <> inline CUtensorMapDataType tma_type<float>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT32; }
template <> inline CUtensorMapDataType tma_type<__half>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT16; }
template <> inline CUtensorMapDataType tma_type<__nv_bfloat16>() {
    return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// A (rows x cols) row-major matrix read in boxes of box_cols (128 bytes) x
// box_rows (128 unless given) rows with the 128-byte swizzle.
inline bool encode_rows_tiled(CUtensorMap *map, const void *ptr, int64_t rows, int cols,
                              size_t elem, int box_cols, CUtensorMapDataType type,
                              int box_rows = 128) {
    EncodeTiled fn = encoder();
    if (!fn || box_rows < 1 || box_rows > 256) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * elem};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A (rows x cols) row-major matrix read or written in plain (unswizzled) boxes
// of box_cols x box_rows elements; the box lands in shared memory as box_rows
// dense rows of box_cols elements.
inline bool encode_rows_plain(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols,
                              size_t elem, int box_cols, int box_rows, CUtensorMapDataType type) {
    EncodeTiled fn = encoder();
    if (!fn || box_cols > 256 || box_rows > 256 || box_rows < 1) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * elem};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A gather map for groups of 32-bit words laid out [group][row][w words]: one
// box = w words of one row from each of `groups` groups (TMA boxes hold at most
// 256 entries per dimension).
inline bool encode_group_gather(CUtensorMap *map, const void *ptr, int w, int64_t rows,
                                int groups) {
    EncodeTiled fn = encoder();
    if (!fn || groups > 256 || w > 256) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)w, (cuuint64_t)rows, (cuuint64_t)groups};
    const cuuint64_t strides[2] = {(cuuint64_t)w * 4, (cuuint64_t)rows * w * 4};
    const cuuint32_t box[3] = {(cuuint32_t)w, 1, (cuuint32_t)groups};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcu
}  // namespace fno
