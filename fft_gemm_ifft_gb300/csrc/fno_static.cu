// fno_static.cu -- a forward call for callers that cannot allocate GPU memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or allocator hooks, code that must not change the
// device's memory footprint after start-up, or a host that hands us only the
// input and output buffers.  fno_spectral_conv_forward_static serves them: it
// needs no plan and no workspace.  The intermediates of the layer live in one
// file-scope __device__ array of kStaticScratchBytes, and the twiddle tables in
// another; every GPU that loads this library holds both until the process
// exits.  The computation is the separate-kernels path of the library (one
// kernel per transform axis plus the mixing kernel), the same kernels that
// fno_spectral_conv_forward runs under FNO_PLAN_UNFUSED.
//
// In host code the names of these arrays are host-side stand-ins, not device
// addresses.  The first call on a device therefore looks up their device
// addresses with cudaGetSymbolAddress (with that device current) and fills the
// twiddle tables with a synchronous copy; later calls on that device reuse the
// addresses.  That first call should come before any stream capture.  The
// cached state assumes the device's context lives as long as the process: a
// caller that runs cudaDeviceReset reloads the module (new, zeroed arrays) and
// must not call this entry point on that device afterwards.
#include <cmath>
#include <mutex>
#include <vector>

#include "fno_internal.cuh"

namespace fno {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;     // 16 MiB
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxStaticN = 1024;
// twiddle tables for N = 2, 4, ..., 1024 back to back: the table of N starts at
// entry N - 2 and holds exp(-2 pi i j / N), j < N
constexpr int kTwEntries = 2 * kMaxStaticN - 2;

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];
static __device__ __align__(256) float2 g_twiddles[kTwEntries];

struct DeviceState {
    bool ready = false;
    void *scratch = nullptr;      // device address of g_scratch
    float2 *twiddles = nullptr;   // device address of g_twiddles
    int num_sms = 0;
};
std::mutex g_mu;
DeviceState g_state[kMaxDevices];

// Once per device, with that device current: device addresses of the arrays,
// twiddle tables computed in double and rounded once to float.
fno_status_t setup(int dev, DeviceState **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_state[dev];
    if (!st.ready) {
        void *scratch = nullptr, *tw = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_scratch) != cudaSuccess ||
            cudaGetSymbolAddress(&tw, g_twiddles) != cudaSuccess) {
            cudaGetLastError();
            return FNO_ERR_CUDA;
        }
        std::vector<float2> host(kTwEntries);
        for (int64_t n = 2; n <= kMaxStaticN; n *= 2)
            for (int64_t j = 0; j < n; ++j) {
                const double ang = -2.0 * M_PI * (double)j / (double)n;
                host[n - 2 + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
        int sms = 0;
        if (cudaMemcpyToSymbol(g_twiddles, host.data(), sizeof(float2) * kTwEntries) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return FNO_ERR_CUDA;
        }
        st.scratch = scratch;
        st.twiddles = static_cast<float2 *>(tw);
        st.num_sms = sms;
        st.ready = true;
    }
    *out = &st;
    return FNO_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

}  // namespace
}  // namespace fno

using namespace fno;

extern "C" fno_status_t fno_spectral_conv_forward_static(
    int ndim, const int64_t *n, const int32_t *modes, int64_t batch, int32_t cin,
    int32_t cout, fno_dtype_t dtype, const void *x, const void *w, void *y,
    fno_stream_t stream) {
    size_t weight_bytes = 0;
    fno_status_t st = fno_spectral_conv_query(ndim, n, modes, batch, cin, cout, dtype,
                                              FNO_PLAN_UNFUSED, nullptr, &weight_bytes);
    if (st != FNO_OK) return st;
    if (!x || !w || !y) return FNO_ERR_INVALID_ARG;
    // the static twiddle tables cover power-of-two extents up to kMaxStaticN
    for (int a = 0; a < ndim; ++a)
        if (n[a] > kMaxStaticN || (n[a] & (n[a] - 1)) != 0) return FNO_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return FNO_ERR_MISALIGNED;

    Plan p{};
    Geom &g = p.g;
    g.d = ndim;
    g.nkept = g.npix = g.ntr = g.nblk = g.mblk = 1;
    for (int a = 0; a < ndim; ++a) {
        g.n[a] = g.ext[a] = n[a];
        g.ntr *= n[a];
        g.m[a] = modes[a];
        g.kdim[a] = a < ndim - 1 ? 2 * (int64_t)modes[a] : modes[a];
        if (a < ndim - 1) g.nblk *= 2;
        g.nkept *= g.kdim[a];
        g.npix *= n[a];
        g.mblk *= modes[a];
    }
    // the layer's intermediates must fit the static scratch array
    if (unfused_workspace_bytes(g, batch, cin, cout) > kStaticScratchBytes)
        return FNO_ERR_UNSUPPORTED;
    const size_t eb = dtype == FNO_F32 ? 4 : 2;
    const size_t xb = (size_t)batch * cin * g.npix * eb, yb = (size_t)batch * cout * g.npix * eb;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, weight_bytes)) return FNO_ERR_ALIASING;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FNO_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FNO_ERR_UNSUPPORTED;
    DeviceState *ds = nullptr;
    st = setup(dev, &ds);
    if (st != FNO_OK) return st;
    // no operand may lie inside the library's own scratch array
    if (overlaps(y, yb, ds->scratch, kStaticScratchBytes) ||
        overlaps(x, xb, ds->scratch, kStaticScratchBytes) ||
        overlaps(w, weight_bytes, ds->scratch, kStaticScratchBytes))
        return FNO_ERR_ALIASING;

    p.batch = batch;
    p.cin = cin;
    p.cout = cout;
    p.dtype = dtype;
    p.flags = FNO_PLAN_UNFUSED;
    p.device = dev;
    p.path = kPathUnfused;
    p.num_sms = ds->num_sms;
    for (int a = 0; a < ndim; ++a) p.tw[a] = ds->twiddles + (n[a] - 2);
    // nothing in the scratch has to start at zero: every intermediate of the
    // sequence is written in full before it is read
    Buffers b{x, w, y, ds->scratch};
    if (unfused_forward(p, b, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FNO_ERR_CUDA;
    }
    return FNO_OK;
}
