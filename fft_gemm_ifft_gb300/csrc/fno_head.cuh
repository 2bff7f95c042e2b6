// fno_head.cuh -- the FNO stack's projection head as one persistent
// tensor-core kernel (fno_head.cu): activations and output in float32, fp16
// or bfloat16, parameters and arithmetic in float32; 32 or 64 input
// channels, 64 or 128 hidden units and up to 8 outputs.
#pragma once

#include "fno_internal.cuh"

namespace fno {

// out[b][c][p] = c2[c] + sum_o P2[c][o] GELU(sum_i W[o][i] a[b][i][p] + bias[o])
struct HeadArgs {
    const void *a;             // [batch][cin][npix], storage type
    const float *W, *bias;     // [hidden][cin], [hidden]
    const float *P2, *c2;      // [cout2][hidden], [cout2]
    void *out;                 // [batch][cout2][npix], storage type
    int cin, hidden, cout2;
    int64_t batch, npix;
    fno_dtype_t dtype;
    int *err;
};

bool head_supported(fno_dtype_t dt, int cin, int hidden, int cout2, int64_t npix);
cudaError_t head_init(fno_dtype_t dt, int cin, int hidden, int cout2);
// A programmatic dependent of the preceding kernel (the last layer).
cudaError_t head_launch(const HeadArgs &a, int num_sms, cudaStream_t s);

}  // namespace fno
