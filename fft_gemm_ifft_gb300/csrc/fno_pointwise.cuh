// fno_pointwise.cuh -- the FNO stack's 1x1 linears on the tensor cores, with
// every activation tile moved by TMA (fno_pointwise.cu).
#pragma once

#include "fno_internal.cuh"

namespace fno {

// One 1x1 linear over channels-first activations [batch][cin][npix]:
//   layer:  out[b][o][p] = act(sum_i W[o][i] a[b][i][p] + bias[o] (+ add[b][o][p]))
//   head:   out[b][c][p] = c2[c] + sum_o P2[c][o] GELU(sum_i W[o][i] a[b][i][p] + bias[o])
// a, add and out in the storage type; W, bias, P2, c2 float32.
struct PointwiseArgs {
    const void *a;
    const float *W;            // [n][cin]
    const float *bias;         // [n]
    const void *add;           // layer: [batch][n][npix] or nullptr
    const float *P2, *c2;      // head: [cout2][n], [cout2]
    void *out;
    int cin, n, cout2;
    int64_t batch, npix;
    int gelu;                  // layer: apply GELU
    int head;
    int *err;
};

// Whether the TMA + tensor-core kernel handles this linear (else the caller
// runs the register-tiled SIMT kernels).
bool pointwise_supported(fno_dtype_t dt, int cin, int n, int cout2, bool head, int64_t npix);
// Plan-time: raise the shared-memory limit of the kernel the launch will use.
cudaError_t pointwise_init(fno_dtype_t dt, int cin, int n, int cout2, bool head);
cudaError_t pointwise_launch(fno_dtype_t dt, const PointwiseArgs &a, int num_sms,
                             cudaStream_t s);

}  // namespace fno
