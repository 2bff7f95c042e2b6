// fno_fused.cu -- fused layer kernels (placeholder: no shape is fused yet).
#include "fno_fused.cuh"

namespace fno {

bool fused_supported(const Geom &, fno_dtype_t, int64_t, int, int) { return false; }
size_t fused_workspace_bytes(const Geom &, fno_dtype_t, int64_t, int, int) { return 0; }
int fused_kernel_count(const Geom &, fno_dtype_t, int64_t, int, int) { return 0; }
cudaError_t fused_plan_init(Plan &) { return cudaSuccess; }
void fused_plan_release(Plan &) {}
cudaError_t fused_forward(const Plan &, const Buffers &, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace fno
