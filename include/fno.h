/*
 * fno.h -- C ABI of the GB300 (sm_103a) Fourier Neural Operator library.
 *
 * The library computes the FNO spectral-convolution layer described in the
 * TurboFNO article (gsyq.cn/news/457482):
 *   §2.1  a real forward FFT over the spatial axes of a channels-first real
 *         tensor (unnormalised, kernel e^{-2 pi i k.n/N});
 *   §2.2  truncation to the retained low-frequency modes and a per-mode
 *         complex contraction over the input channels with a learned complex
 *         weight per mode (plain complex product, no conjugation);
 *   §2.3  zero-padding of the discarded modes and an inverse real FFT back to
 *         the grid (scale 1/prod(N)),
 * fused on the device so that the intermediates stay on chip or in L2 (§3.4).
 * §4.3 of the article exposes the fused layer as a C function of a shared
 * library taking raw device pointers; this header is that boundary.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - No entry point throws, aborts or prints; each returns fno_status_t.
 *  - Device pointers are caller-owned.  The library never frees them and never
 *    keeps them beyond the call.
 *  - fno_stream_t is a cudaStream_t (NULL = the legacy default stream).  All
 *    device work is enqueued asynchronously on that stream.
 *  - Tensors are dense, row-major (last axis contiguous), with no padding.
 *  - Complex values are interleaved (re, im) pairs of the storage type.
 *
 * Kept modes (the "corner blocks").  For spatial extents N_0..N_{d-1} and
 * per-block modes m_0..m_{d-1}:
 *  - on each full axis a < d-1 the kept rows are the low rows 0..m_a-1 and
 *    the high rows N_a-m_a..N_a-1 (negative frequencies -m_a..-1);
 *  - on the last (half-spectrum) axis the kept bins are 0..m_{d-1}-1.
 * A weight block is one choice of low/high per full axis; block
 * beta = sum_a hi_a * 2^a (axis 0 varies fastest): 1 block in 1-D, 2 in 2-D
 * (low rows, high rows), 4 in 3-D ((lo,lo), (hi,lo), (lo,hi), (hi,hi)).
 * In the inverse, bins 0 and N_{d-1}/2 of the half axis carry weight 1 and
 * every other bin weight 2, and the real part is taken (the convention of a
 * real inverse FFT applied to a zero-filled half spectrum).
 */
#ifndef FNO_H_
#define FNO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FNO_MAX_NDIM 3

typedef enum fno_status_e {
    FNO_OK = 0,
    FNO_ERR_INVALID_ARG = 1,     /* a null pointer, a bad rank/extent/modes/channels     */
    FNO_ERR_UNSUPPORTED = 2,     /* valid shape this build does not handle               */
    FNO_ERR_MISALIGNED = 3,      /* a device pointer is not 16-byte aligned              */
    FNO_ERR_OUT_OF_MEMORY = 4,   /* plan-owned device or host memory could not be had    */
    FNO_ERR_CUDA = 5,            /* a CUDA runtime call or kernel launch failed          */
    FNO_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait gave up                   */
    FNO_ERR_DEVICE_BOUNDS = 7,   /* a device index check failed (index-checking build)   */
    FNO_ERR_ALIASING = 8         /* the output overlaps an input or the workspace        */
} fno_status_t;

typedef enum fno_dtype_e {
    FNO_F32 = 0,   /* float32 storage, float32 arithmetic                                 */
    FNO_F16 = 1,   /* IEEE half storage (x, w, y), float32 accumulation                   */
    FNO_BF16 = 2   /* bfloat16 storage (x, w, y), float32 accumulation                    */
} fno_dtype_t;

typedef void *fno_stream_t;                 /* a cudaStream_t                            */
typedef struct fno_plan_s *fno_plan_t;      /* opaque spectral-convolution plan          */
typedef struct fno_model_s *fno_model_t;    /* opaque FNO-stack plan                     */

/* Plan flags. */
#define FNO_PLAN_DEFAULT 0u
/* Run the layer as separate per-axis transform, mixing and inverse kernels
 * through the workspace instead of the fused path (the "separate kernels"
 * ablation of the article's §5.2 note).  Results agree with the fused path
 * within rounding.                                                           */
#define FNO_PLAN_UNFUSED 1u
/* Record a timeline of the fused kernels' work items (read back with
 * fno_plan_get_trace): the persistent kernel's queue items, or one record per
 * CTA of each kernel of the three-kernel variants (2-D and 3-D layers).
 * Costs a few timer reads, a barrier and a store per item.                  */
#define FNO_PLAN_TRACE 2u
/* Bit 4u is unused; a plan with it set is rejected (FNO_ERR_INVALID_ARG).
 * The tensor-core kernels are the default wherever they exist, and
 * FNO_PLAN_SIMT_TRANSFORM / FNO_PLAN_SIMT_MIX select the SIMT kernels.       */
/* Run the float32 / fp16 128x128 layer as ONE persistent kernel with a work
 * queue instead of three kernels chained by programmatic dependent launch
 * (the default).  FNO_PLAN_TRACE records only this variant.               */
#define FNO_PLAN_PERSISTENT 8u
/* Also prepare the plan for fno_spectral_conv_backward: the plan then holds
 * an internal plan of the adjoint layer (Cin and Cout swapped) and reports a
 * workspace size that covers the backward call as well.                    */
#define FNO_PLAN_BACKWARD 16u
/* Mix with the SIMT kernel where the tensor-core mixing kernel would run
 * (2-D fp16 / bf16 layers with at most 64 channels and 64 samples; the
 * tensor-core kernel is the default there), and, for the float32 64x64x64
 * layer with at most 4 samples and 32 channels and the float32 128x128 layer
 * with at most 16 samples and 64 channels, with the SIMT kernels that load W
 * themselves instead of the kernels fed by TMA boxes of weights.  An
 * ablation switch.                                                          */
#define FNO_PLAN_SIMT_MIX 32u
/* Run the transforms on the register-FFT kernels instead of the tensor-core
 * kernels that are the default for these shapes: for the 16-bit 256x256
 * layer (32x32 modes) the forward transform (a kind::f16 tcgen05 GEMM per
 * image) and the inverse (a kind::tf32 GEMM per image); for the float32
 * 128x128 layer (16x16 modes) the forward transform and the inverse (3xTF32
 * GEMMs per image, TMA loads and stores); for the 64x64x64 layer (16x16x16
 * modes per block) the inverse's row transform (a 3xTF32 GEMM per pair of
 * planes).  An ablation switch.                                             */
#define FNO_PLAN_SIMT_TRANSFORM 64u
/* The weights passed to fno_spectral_conv_forward are in the packed layout
 * written by fno_spectral_conv_pack_weights (weights are parameters: pack once
 * per update, use many times).  Packed, every mixing kernel reads a mode's (or
 * a group of four modes') Cin x Cout weights as one contiguous run instead of
 * pieces strided by the mode count; the tensor-core mixing of the 64-channel
 * 16-bit 2-D layers reads them as ready operand images.  Requires
 * |K| % 4 == 0; not combinable with FNO_PLAN_BACKWARD.                      */
#define FNO_PLAN_PACKED_WEIGHTS 128u
/* Also run the tensor-core variants that are not the default because they
 * measured slower on the workloads (each matches the oracle like the default;
 * ignored where none applies):
 *  - the mixing of the float32 128x128 three-kernel layer: per pair of kept
 *    modes one CTA, the complex products in 3xTF32 on kind::tf32
 *    tcgen05.mma, [Wr^T ; Wi^T] as the one weight operand (fno_mix_tf32.cu),
 *    for 32 or 64 input and output channels, batch <= 32 (64 outputs) or
 *    <= 16 (32 outputs), weights in the standard layout;
 *  - the forward transform of the float32 64^3 layer: the row DFT of each
 *    pair of planes as a 3xTF32 GEMM, the planes brought in by TMA
 *    (k_phase_a3_tc in fno_fused3d.cu).
 * The products involved are small; the kernels are bound by the latency of
 * their loads and by their SIMT steps, not by arithmetic.                   */
#define FNO_PLAN_TENSOR_EXTRA 256u
/* FNO stack (fno_model_plan) only: run each layer as the spectral
 * convolution's three kernels, which write the spectral branch out, followed
 * by the 1x1-linear kernel that adds it (bias, sum, GELU).  The default for
 * float32 128x128 layers with 16x16 modes and 32 or 64 channels instead runs
 * the forward transform and the mixing, a column-step kernel, and ONE
 * tensor-core GEMM per image row whose K concatenates the inverse row DFT's
 * coefficients and the input channels (3xTF32), so that the spectral branch
 * never reaches global memory.  Both match the oracle; an ablation switch.
 * fno_spectral_conv_plan accepts and ignores it.                             */
#define FNO_PLAN_SPLIT_LAYER 512u

/* One work item of the fused kernel, as recorded under FNO_PLAN_TRACE.
 * Times are the GPU's global nanosecond timer.                              */
typedef struct fno_trace_record_s {
    uint32_t item;      /* phase << 24 | batch group << 16 | index in the phase-group
                           (phase 0: forward transform, 1: mixing, 2: inverse); in
                           the three-kernel variants phase << 24 | CTA index     */
    uint32_t worker;    /* which CTA / stream ran it (three-kernel variants: the SM) */
    uint64_t t_start;   /* processing began                                       */
    uint64_t t_ready;   /* its inputs were available (loads landed, waits over)   */
    uint64_t t_compute; /* its arithmetic was done                                */
    uint64_t t_end;     /* its outputs were issued and the item counted done      */
} fno_trace_record_t;

/* Human-readable name of a status code; never NULL. */
const char *fno_status_string(fno_status_t status);

/* Library version as major*10000 + minor*100 + patch. */
int fno_version(void);

/* -------------------------------------------------------------------------
 * Spectral convolution (one layer).
 * ------------------------------------------------------------------------- */

/* Validate a layer description and report its memory needs without touching
 * the GPU (no CUDA call is made).  The layer is the one of the TurboFNO
 * article §2.1-§2.3 (forward real FFT, kept modes, per-mode mixing, inverse
 * real FFT); its sizes are fixed here, ahead of any call, as §2.3 and §3.3
 * ask of the fused module (compile-time output size).
 *   ndim          1, 2 or 3
 *   n[ndim]       spatial extents, 2 <= N <= 4096 (any length: extents
 *                 that are not powers of two, and shapes without a fused
 *                 kernel, run on the separate per-axis kernels)
 *   modes[ndim]   per-block modes; 1 <= m_a and 2 m_a <= N_a on full axes,
 *                 1 <= m_{d-1} <= N_{d-1}/2 + 1 on the last axis
 *   batch, cin, cout  >= 1
 *   dtype         FNO_F32, FNO_F16 or FNO_BF16
 *   flags         FNO_PLAN_* bits
 * Outputs (each may be NULL):
 *   workspace_bytes  device scratch the forward call needs (caller-owned)
 *   weight_bytes     size of w: nblk*cin*cout*prod(m)*2*sizeof(storage)
 * Returns FNO_OK, FNO_ERR_INVALID_ARG or FNO_ERR_UNSUPPORTED.             */
fno_status_t fno_spectral_conv_query(int ndim, const int64_t *n, const int32_t *modes,
                                     int64_t batch, int32_t cin, int32_t cout,
                                     fno_dtype_t dtype, uint32_t flags,
                                     size_t *workspace_bytes, size_t *weight_bytes);

/* Create a plan on the current CUDA device (TurboFNO §2.3, §3.3: every size
 * and table fixed before the first forward, so the forward is a fixed launch
 * sequence that a CUDA graph can hold).  Arguments as in
 * fno_spectral_conv_query.  The plan computes its twiddle tables on the host
 * in double precision, rounds them once to float and copies them to
 * plan-owned device memory; it synchronises the device once, here, and is
 * immutable afterwards.  *plan is set to NULL on failure.
 * Errors: INVALID_ARG, UNSUPPORTED, OUT_OF_MEMORY, CUDA.                  */
fno_status_t fno_spectral_conv_plan(fno_plan_t *plan, int ndim, const int64_t *n,
                                    const int32_t *modes, int64_t batch, int32_t cin,
                                    int32_t cout, fno_dtype_t dtype, uint32_t flags);

/* The layer on a non-periodic domain (TurboFNO §2.3: the input is zero-padded
 * so that the transform sees no wrap-around, and the output is cropped back
 * to the original size; §3.3: the crop is a guarded store in the inverse's
 * final stage, not an extra copy or kernel).
 *   n[ndim]    extents of x and y (1 <= n[a] <= 4096)
 *   pad[ndim]  zeros appended after the last sample of each axis (>= 0);
 *              the transform of axis a runs over L_a = n[a] + pad[a] <= 4096
 *              points and `modes` are counted on L (2 m_a <= L_a on full
 *              axes, m_{d-1} <= L_{d-1}/2 + 1); NULL or all zeros is the
 *              periodic layer of fno_spectral_conv_plan
 * x stays (batch, cin, n...) and y (batch, cout, n...): the forward reads x
 * as if extended with zeros and writes only the first n[a] samples of the
 * inverse along each axis (scale 1/prod(L)).  A padded plan runs on the
 * separate per-axis kernels (FNO_PLAN_UNFUSED is implied) and takes the
 * weights of the L-sized layer; FNO_PLAN_BACKWARD is not supported with
 * padding (FNO_ERR_UNSUPPORTED).  Other arguments, ownership and errors as in
 * fno_spectral_conv_query / fno_spectral_conv_plan; the plan is used with
 * fno_spectral_conv_workspace_size, _kernel_count, _forward,
 * _pack_weights and fno_plan_destroy like any other.                       */
fno_status_t fno_spectral_conv_query_padded(int ndim, const int64_t *n, const int64_t *pad,
                                            const int32_t *modes, int64_t batch, int32_t cin,
                                            int32_t cout, fno_dtype_t dtype, uint32_t flags,
                                            size_t *workspace_bytes, size_t *weight_bytes);
fno_status_t fno_spectral_conv_plan_padded(fno_plan_t *plan, int ndim, const int64_t *n,
                                           const int64_t *pad, const int32_t *modes,
                                           int64_t batch, int32_t cin, int32_t cout,
                                           fno_dtype_t dtype, uint32_t flags);

/* Bytes of device workspace fno_spectral_conv_forward needs for this plan:
 * the kept modes handed between the fused kernel's phases (TurboFNO §3.4
 * keeps them on chip; here they pass through an L2-resident buffer). */
fno_status_t fno_spectral_conv_workspace_size(fno_plan_t plan, size_t *bytes);

/* Number of kernels one forward call launches for this plan (TurboFNO §1
 * and §3.4 speak of one fused kernel and of three kernels per forward; the
 * §5.2 note times the separate-kernels arrangement). */
fno_status_t fno_spectral_conv_kernel_count(fno_plan_t plan, int *count);

/* y = SpectralConv(x; w), enqueued on `stream`: TurboFNO §2.1 (forward real
 * FFT, truncated), §2.2 (per-mode complex mixing), §2.3 / §3.3 (zero-padded
 * inverse real FFT), fused as §3.4 describes, behind the raw-pointer C
 * function of §4.3.
 *   x          device, (batch, cin, N_0..N_{d-1}) storage dtype
 *   w          device, (nblk, cin, cout, m_0..m_{d-1}) complex storage dtype,
 *              block order as described at the top of this header
 *   y          device, (batch, cout, N_0..N_{d-1}) storage dtype; fully
 *              overwritten; must not overlap x, w or the workspace
 *   workspace  device, at least fno_spectral_conv_workspace_size bytes, or
 *              NULL when that size is 0; its contents on entry are ignored
 *              and on exit are unspecified.
 * Calls that may run at the same time on the GPU (different streams) need
 * their own plan and their own workspace: the fused kernel keeps its work-
 * queue counters in plan-owned device memory and resets them at the end of
 * every call.  Calls on one stream, or stream-ordered, may share both.
 * Every pointer must be 16-byte aligned (FNO_ERR_MISALIGNED otherwise).
 * The call makes no allocation and no host synchronisation, so it may be
 * captured in a CUDA graph.  Its first kernel is ordered after the work
 * already on `stream` like any launch; its later kernels use programmatic
 * dependent launch among themselves.  Launch failures return FNO_ERR_CUDA; faults
 * detected inside kernels are reported by fno_plan_get_device_error.        */
fno_status_t fno_spectral_conv_forward(fno_plan_t plan, const void *x, const void *w,
                                       void *y, void *workspace, fno_stream_t stream);

/* y = SpectralConv(x; w) for callers that cannot allocate GPU memory.
 * The pages on the FNO layer have no counterpart to this call; it exists for
 * callers that may not call cudaMalloc (code running under another
 * framework's allocator, or with a device memory budget fixed at start-up)
 * and therefore can create neither a plan nor a workspace.
 *   ndim, n, modes, batch, cin, cout, dtype   as in fno_spectral_conv_query
 *   x, w, y   device pointers, layouts as in fno_spectral_conv_forward
 * No plan, no workspace: the intermediates live in a fixed 16 MiB scratch
 * array in device memory that the library reserves on every GPU that loads it,
 * held until the process exits; the twiddle tables live in another such array.
 * Shapes whose intermediates need more than 16 MiB (the workspace that
 * fno_spectral_conv_query reports under FNO_PLAN_UNFUSED) are rejected with
 * FNO_ERR_UNSUPPORTED before anything is enqueued.
 * The call allocates nothing.  Its first call on a device looks up the device
 * addresses of those arrays and fills the twiddle tables with a synchronous
 * copy (with that device current), so that first call should come before any
 * stream capture.  Every call shares the one scratch array, which keeps the
 * last call's contents; none of it has to start at zero.  Calls that overlap
 * on the GPU (different streams) race on the scratch and give wrong results;
 * calls on one stream are safe.  The looked-up addresses are kept for the life
 * of the process: after a cudaDeviceReset of a device (which discards the
 * arrays) this call must not be used on that device again.  Runs the
 * separate-kernels path (the kernels of FNO_PLAN_UNFUSED).  Errors:
 * INVALID_ARG, UNSUPPORTED, MISALIGNED, ALIASING (y overlaps x or w, or an
 * operand lies inside the library's scratch array), CUDA.                   */
fno_status_t fno_spectral_conv_forward_static(int ndim, const int64_t *n,
                                              const int32_t *modes, int64_t batch,
                                              int32_t cin, int32_t cout, fno_dtype_t dtype,
                                              const void *x, const void *w, void *y,
                                              fno_stream_t stream);

/* Re-lay the learned weights out once per weight update (TurboFNO §2.2: one
 * complex Cin x Cout weight per mode; §3.2: the GEMM stage takes its weights
 * in the tensor-core operand layout rather than the framework's).
 * Write w (nblk, Cin, Cout, m...) in the packed layout of the plan; same size
 * as w.  Kept modes are numbered in the order of the layer's kept-mode index:
 * axis by axis, low rows then high rows on full axes.  Two layouts:
 *  - the tensor-core mixing's operand images, for 2-D fp16 / bf16 layers with
 *    Cin = Cout = 64 whose mixing runs on the tensor cores (the 256 x 256,
 *    32 x 32-mode layer): per kept mode k, 16 KiB = two 64 x 64 tiles of the
 *    storage type, Wr^T then Wi^T (row o, column i holds W[i][o]), each row
 *    128 bytes whose eight 16-byte pieces are permuted by p -> p ^ (o % 8)
 *    (the 128-byte swizzle of the tensor cores' shared-memory operands); a
 *    mixing CTA reads a mode's weights with one bulk copy;
 *  - otherwise mode-major groups of four: w_packed[(q * Cin + i) * Cout + o][r]
 *    = W of kept mode k = 4 q + r, interleaved complex.
 * For plans made with FNO_PLAN_PACKED_WEIGHTS.  Asynchronous on `stream`.
 * Errors: INVALID_ARG (NULL, plan without the flag), MISALIGNED, ALIASING
 * (w and w_packed overlap), CUDA.                                           */
fno_status_t fno_spectral_conv_pack_weights(fno_plan_t plan, const void *w, void *w_packed,
                                            fno_stream_t stream);

/* Gradients of the layer for a real loss L, given dy = dL/dy (B, Cout, N...)
 * in the storage dtype: the backward of the autograd function that TurboFNO
 * §4.3 wraps around the fused layer.  The pages define only the forward pass; this is its
 * derivative, with dz = dL/dRe(z) + i dL/dIm(z) for a complex z:
 *   dY = c(k_last) / prod(N) * (truncated forward DFT of dy),
 *   dx = the layer applied to dy with the weights W'[blk][o][i] =
 *        conj(W[blk][i][o]) (Cout -> Cin): the fused forward path of the
 *        adjoint plan, after one kernel writes W' into the workspace;
 *   dw[blk][i][o][l] = sum_b dY[b][o][k] conj(X[b][i][k]), X the truncated
 *        forward DFT of x (dense per-axis DFT kernels plus one reduction
 *        kernel over the batch), same layout and dtype as w.
 * dx (B, Cin, N...) or dw may be NULL to skip it (not both); x is needed only
 * for dw, w only for dx.  The plan must have been made with
 * FNO_PLAN_BACKWARD; the workspace is the plan's (fno_spectral_conv_workspace_size).
 * Asynchronous on `stream`; no allocation.  Errors: INVALID_ARG (NULL
 * handle, missing flag, missing operand), MISALIGNED, ALIASING (an output
 * overlaps an input, the other output or the workspace), CUDA.              */
fno_status_t fno_spectral_conv_backward(fno_plan_t plan, const void *x, const void *w,
                                        const void *dy, void *dx, void *dw, void *workspace,
                                        fno_stream_t stream);

/* Copy the trace of the plan's last forward call (FNO_PLAN_TRACE) to host
 * memory (the per-phase timeline TurboFNO §1 reads from a kernel launch
 * trace): up to `capacity` records, ordered by ticket (three-kernel variants:
 * kernel A's CTAs, then B's, then C's); *count receives the number of records
 * the call produced.  Synchronises the device.  Returns FNO_ERR_INVALID_ARG if
 * the plan was made without FNO_PLAN_TRACE or runs a path that records none
 * (separate kernels, the 1-D kernel).                                       */
fno_status_t fno_plan_get_trace(fno_plan_t plan, fno_trace_record_t *records, size_t capacity,
                                size_t *count);

/* Synchronise `stream`, then read and clear the plan's device error word
 * (TurboFNO §6.1 traces a crash to an unchecked device index; faults found on
 * the device are reported here instead of trapping).  FNO_ERR_DEVICE_BOUNDS
 * comes from the index-checking build of the library (libfno_bounds.so,
 * compiled with FNO_DEBUG_BOUNDS), whose kernels check the global-memory
 * indices of the separate-kernels path and of the 16-bit 256 x 256 fused
 * path, record a failure here and skip the access.
 * Returns FNO_OK, FNO_ERR_DEVICE_TIMEOUT, FNO_ERR_DEVICE_BOUNDS or CUDA.   */
fno_status_t fno_plan_get_device_error(fno_plan_t plan, fno_stream_t stream);

/* Self-test of the bounded device waits (the waits of the fused kernels of
 * TurboFNO §3.4 between their phases).  Launches one CTA on `stream` that
 * waits for something no one will do -- which = 0: a flag word in the plan's
 * memory that no kernel writes (the wait CTAs of one launch use for each
 * other's phases); which = 1: phase 0 of an mbarrier nothing arrives on (the
 * wait of the tensor-core kernels for TMA and MMA completion).  The wait gives
 * up after its limit (0.5 s), sets the plan's device error word and returns,
 * so the next fno_plan_get_device_error returns FNO_ERR_DEVICE_TIMEOUT and the
 * context stays usable.  Asynchronous; no allocation.  Errors: INVALID_ARG
 * (NULL plan, `which` not 0 or 1), CUDA (launch failed).                    */
fno_status_t fno_plan_check_bounded_wait(fno_plan_t plan, int which, fno_stream_t stream);

/* Release the plan and its device memory (the plan of TurboFNO §2.3).  NULL is accepted (no-op).  The
 * caller must make sure no work that uses the plan is still running.       */
fno_status_t fno_plan_destroy(fno_plan_t plan);

/* -------------------------------------------------------------------------
 * FNO forward stack (2-D grid), the workload of the article's §5 tasks:
 *   a_0     = Lift x + lift_b                         (1x1, cin_lift -> width)
 *   t_l     = SpectralConv_l(a_l) + Pw_l a_l + pw_b_l (l = 0 .. nlayers-1)
 *   a_{l+1} = GELU(t_l) for l < nlayers-1, t_l for the last layer
 *   out     = Proj2 GELU(Proj1 a_L + proj1_b) + proj2_b
 * GELU is the exact form v/2 (1 + erf(v / sqrt 2)).  1x1 linear weights are
 * (out, in) row-major float32.
 * ------------------------------------------------------------------------- */
typedef struct fno_model_desc_s {
    int64_t batch;       /* B                                                   */
    int32_t cin_lift;    /* input channels (3: field + two coordinates)         */
    int32_t width;       /* hidden channels of the spectral layers              */
    int32_t nlayers;     /* number of spectral layers                           */
    int32_t hidden;      /* projection hidden width                             */
    int32_t cout;        /* output channels                                     */
    int64_t h, w;        /* grid                                                */
    int32_t modes[2];    /* per-block modes (rows, half-axis bins)              */
    fno_dtype_t dtype;   /* storage of x, activations, spec_w and out: FNO_F32,
                            FNO_F16 or FNO_BF16 (arithmetic float32 throughout;
                            the 1x1 weights and biases stay float32)           */
    uint32_t flags;      /* FNO_PLAN_* bits, applied to every spectral layer    */
} fno_model_desc_t;

typedef struct fno_model_params_s {
    const float *lift_w;   /* (width, cin_lift)                                  */
    const float *lift_b;   /* (width)                                            */
    const void *spec_w;    /* nlayers x (2, width, width, m0, m1) complex, in the
                              storage dtype (interleaved re, im)                */
    const float *pw_w;     /* nlayers x (width, width)                           */
    const float *pw_b;     /* nlayers x (width)                                  */
    const float *proj1_w;  /* (hidden, width)                                    */
    const float *proj1_b;  /* (hidden)                                           */
    const float *proj2_w;  /* (cout, hidden)                                     */
    const float *proj2_b;  /* (cout)                                             */
} fno_model_params_t;

/* Validate the description and create the stack's plan (one spectral plan
 * shared by the layers; TurboFNO §2.1 runs the layer inside a multi-layer
 * operator, §5 on 128 x 128 tasks).  Errors as for fno_spectral_conv_plan; also
 * INVALID_ARG for an unknown dtype, UNSUPPORTED for cout > 8,
 * batch > 65535, or h*w not a multiple of 4.  The 1x1 linears run on the
 * tensor cores (3xTF32) for float32 storage where the channel counts fit one
 * tile, else as register-tiled float32 GEMMs.                               */
fno_status_t fno_model_plan(fno_model_t *model, const fno_model_desc_t *desc);

/* Device workspace bytes fno_forward needs (activations + layer scratch;
 * TurboFNO §2.1). */
fno_status_t fno_model_workspace_size(fno_model_t model, size_t *bytes);

/* Number of kernels one fno_forward call launches (TurboFNO §2.1 counts the
 * launches of a multi-layer operator). */
fno_status_t fno_model_kernel_count(fno_model_t model, int *count);

/* out = FNO(x), enqueued on `stream` (TurboFNO §2.1: the spectral layer inside
 * an FNO; §2.3: capturable as one CUDA graph).
 *   x    device, (batch, cin_lift, h, w) in the storage dtype
 *   p    host struct of device pointers (all 16-byte aligned)
 *   out  device, (batch, cout, h, w) in the storage dtype; must not overlap
 *        the inputs
 *   workspace  device, fno_model_workspace_size bytes
 * No allocation, no host synchronisation (graph-capturable).               */
fno_status_t fno_forward(fno_model_t model, const void *x, const fno_model_params_t *p,
                         void *out, void *workspace, fno_stream_t stream);

/* Synchronise `stream`, read and clear the device error word of the stack
 * (as fno_plan_get_device_error, TurboFNO §6.1). */
fno_status_t fno_model_get_device_error(fno_model_t model, fno_stream_t stream);

/* Release the stack's plan; NULL is accepted (TurboFNO §2.1). */
fno_status_t fno_model_destroy(fno_model_t model);

#ifdef __cplusplus
}
#endif

#endif /* FNO_H_ */
