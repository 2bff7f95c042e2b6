// fno_layer.cuh -- the output half of an FNO layer in two kernels
// (fno_layer.cu): the inverse transform's column step, then the inverse row
// DFT and the layer's 1x1 linear as ONE tensor-core GEMM per image row, with
// bias and GELU, for 128 x 128 layers with 16 x 16 modes (activations in
// float32 or a 16-bit storage type; the coefficients and sums in float32).
#pragma once

#include "fno_internal.cuh"

namespace fno {

struct LayerOutArgs {
    const float2 *Y;       // mixed modes, [batch * width][32 kept rows][16 kept columns]
    const float2 *tw;      // tw[j] = exp(-2 pi i j / 128), j < 128
    float *Z;              // workspace: [batch][128 rows][hi, lo][width][32] (layer_out_z_bytes)
    const void *x;         // the layer's input, [batch][width][128 * 128], storage type
    const float *W;        // 1x1 linear, [width][width] (out, in)
    const float *bias;     // [width]
    void *out;             // [batch][width][128 * 128], storage type
    const void *table;     // the inverse row-DFT operand (inverse_row_operand_tf32)
    int64_t batch;
    fno_dtype_t dtype;     // storage type of x and out
    int width;
    int gelu;              // apply the GELU (every layer but the last)
    int *err;
};

// Whether the two kernels handle this layer: 128 x 128, 16 x 16 modes
// (checked by the caller), width 32 or 64.
bool layer_out_supported(int width, int64_t batch);
size_t layer_out_z_bytes(int64_t batch, int width);
// Plan-time: raise the shared-memory limit of the GEMM kernel.
cudaError_t layer_out_init(fno_dtype_t dt, int width);
// Launches the column step (a programmatic dependent of the mixing kernel)
// and the GEMM kernel (a programmatic dependent of the column step).
cudaError_t layer_out_launch(const LayerOutArgs &a, int num_sms, cudaStream_t s);

}  // namespace fno
