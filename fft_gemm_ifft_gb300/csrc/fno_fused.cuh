// fno_fused.cuh -- host-side entry points of the fused layer kernels.
#pragma once

#include "fno_internal.cuh"

namespace fno {

// Bytes of plan-owned device memory the fused kernels keep their counters in.
size_t fused_sync_bytes();
// True when the fused path handles this description.
bool fused_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout,
                     uint32_t flags);
size_t fused_workspace_bytes(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin,
                             int cout, uint32_t flags);
int fused_kernel_count(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout,
                       uint32_t flags);
// Plan-time set-up (tables, attributes); called once from plan creation.
cudaError_t fused_plan_init(Plan &p);
void fused_plan_release(Plan &p);
cudaError_t fused_forward(const Plan &p, const Buffers &b, cudaStream_t s);

}  // namespace fno
