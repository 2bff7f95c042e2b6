// fno_fused.cuh -- host-side entry points of the fused layer kernels.
#pragma once

#include <vector>

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

// Kept modes of nimg images by the forward-transform kernel of the
// three-kernel path alone (used by the backward pass).  fused_modes_parts
// returns how many partial copies that kernel writes ([parts][nimg][|K|]
// complex float, summed by the reader), or 0 when the plan's variant has no
// such kernel.
int fused_modes_parts(const Geom &g, fno_dtype_t dtype, uint32_t flags);
cudaError_t fused_forward_modes(const Plan &p, const void *x, int64_t nimg, float2 *parts,
                                cudaStream_t s);
cudaError_t fused3d_forward_modes(const Plan &p, const void *x, int64_t nimg, float2 *out,
                                  cudaStream_t s);

// The 128 x 128 layer (16 x 16 modes) up to its mixed modes: the
// forward-transform and mixing kernels of the three-kernel path alone, for a
// caller that runs its own inverse (the FNO layer's fused output, fno_layer.cu).
// True when the plan runs that path and leaves the mixed modes in float32.
bool fused_mixed_available(const Plan &p);
// Launches the two kernels; *Y = the mixed modes in the workspace,
// [batch * cout][32 kept rows][16 kept columns] complex float.
cudaError_t fused_forward_mixed(const Plan &p, const Buffers &b, const float2 **Y,
                                cudaStream_t s);
// The inverse row-DFT operand of the float32 128-point inverse: 128 rows of
// [s c(k) cos(2 pi k n / 128) | -s c(k) sin(...)], k < 16, s = 1/128^2, as the
// 128-byte-swizzled K-major tf32 operand, hi then lo (2 x 16 KB).
void inverse_row_operand_tf32(std::vector<unsigned char> &img);

// Tensor-core mixing (kernel B of the three-kernel 2-D path) for 16-bit
// storage: four adjacent modes per CTA, real-block complex GEMMs on tcgen05.
struct MixTcArgs {
    const void *X;                // kept modes: [group of 8 modes][batch * cin][8] 16-bit
                                  // (re, im) pairs, as kernel A writes them (mixtc_x_bytes)
    const void *w;                // weights (2, cin, cout, m0, m1) interleaved complex
    void *Y;                      // mixed modes: [group of 8 modes][batch * cout][8] 16-bit
                                  // (re, im) pairs, as kernel C gathers them
    int *err;
    fno_trace_record_t *trace;    // nullptr unless tracing: one record per run of 4 modes
    int trace_first;
    int batch, cin, cout, m0, m1, mblk, nk;
    int packed;                   // w packed: 1 mode-major groups of four, 2 operand images
    int num_sms;                  // persistent grid: at most one CTA per SM
};
bool mixtc_supported(int d, fno_dtype_t dtype, int64_t batch, int cin, int cout, int m1,
                     int64_t nkept);
// Bytes of the kept modes in the tensor-core mixing's input layout: kept mode
// kk of image img = b * cin + i is the 16-bit (re, im) pair at byte
// ((kk / 8) * batch * cin + img) * 32 + (kk % 8) * 4.
size_t mixtc_x_bytes(int64_t batch, int cin, int64_t nkept);
int mixtc_items(int64_t nkept);
cudaError_t mixtc_init(fno_dtype_t dtype);
cudaError_t mixtc_launch(fno_dtype_t dtype, const MixTcArgs &args, cudaStream_t s);
// Packed weights as the mixing kernel's operand images (MixTcArgs.packed = 2):
// offered for 64 input and 64 output channels, where the images take exactly
// the bytes of the weights.
bool mixtc_image_layout(int cin, int cout);
cudaError_t mixtc_pack_image(fno_dtype_t dtype, const void *w, void *wp, int cin, int cout,
                             int m0, int m1, int mblk, int nk, int num_sms, cudaStream_t s);

// Tensor-core mixing for float32 storage (kernel B of the fp32 128 x 128
// three-kernel layer, fno_mix_tf32.cu): one CTA per pair of kept modes, the
// complex products in 3xTF32 on tcgen05.
struct MixTf32Args {
    const float2 *X;              // kept modes [batch * cin][nk] (one reduced copy)
    const float *w;               // weights (2, cin, cout, m0, m1) interleaved complex
    float2 *Y;                    // mixed modes [batch * cout][nk]
    int *err;
    fno_trace_record_t *trace;    // nullptr unless tracing: one record per pair
    int trace_first;
    int batch, cin, cout, m0, m1, nk;
};
bool mixtf32_supported(int64_t batch, int cin, int cout, int m1, int64_t nkept);
cudaError_t mixtf32_init();
cudaError_t mixtf32_launch(const MixTf32Args &a, cudaStream_t s);

// Kernel C of the 16-bit 256 x 256 layer (fno_inv16.cu): the column and row
// inverse DFTs of each output image as two tcgen05 GEMMs, persistent.
struct Inv16Args {
    const void *Y;                // mixed modes [nimg][64 kept rows][32 bins], 16-bit (re, im)
    void *y;                      // output images [nimg][256][256], storage type
    int *err;
    fno_trace_record_t *trace;    // nullptr unless tracing: one record per image
    int trace_first;
};
size_t inv16_tables_bytes();
void inv16_make_tables(fno_dtype_t dtype, std::vector<unsigned char> &img);
cudaError_t inv16_init(fno_dtype_t dtype);
cudaError_t inv16_launch(fno_dtype_t dtype, const Inv16Args &a, const void *tables,
                         int64_t nimg, int num_sms, cudaStream_t s);

// The 1-D layer's kernel (one cluster per sample).
bool fused1d_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout);
cudaError_t fused1d_forward(const Plan &p, const Buffers &b, cudaStream_t s);

// The 3-D layer's kernels (64 x 64 x 64, 16 x 16 x 16 modes per corner block).
bool fused3d_match(const Geom &g, fno_dtype_t dtype);
bool fused3d_supported(const Geom &g, fno_dtype_t dtype, int64_t batch, int cin, int cout);
size_t fused3d_workspace_bytes(const Geom &g, int64_t batch, int cin, int cout);
cudaError_t fused3d_plan_init(Plan &p);
cudaError_t fused3d_forward(const Plan &p, const Buffers &b, cudaStream_t s);

}  // namespace fno
