// s5_noalloc.cu -- a forward entry point that allocates nothing and needs no
// workspace from its caller.
//
// Some callers cannot call cudaMalloc where they run the layer: a plugin
// inside a host application that owns all device memory and exposes no
// allocator, a latency-critical loop that must never enter the allocator
// (cudaMalloc can synchronise the device and take driver locks), or an
// embedded deployment whose memory budget is fixed up front.  s5_forward needs
// a caller-provided workspace for the carries its chunked scan passes between
// tiles; this variant keeps that scratch in a fixed, file-scope device array
// instead.  The paper has no counterpart: this is a deployment convenience.
#include <cstdint>
#include <mutex>

#include "s5_simt.cuh"

namespace {

// Carry scratch of the chunked scan (header, flags, per-tile aggregates).
// Every GPU that loads the library holds these bytes until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[S5_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_ptr[64] = {nullptr};   // device address of the array, per device
int g_num_sms[64] = {0};

bool aligned16(const void *p) { return (reinterpret_cast<std::uintptr_t>(p) & 15u) == 0; }

// The array's name in host code is a host-side stand-in, not a device
// address; the device address is looked up once per device, with that device
// current, and cached.
s5_status device_scratch(void **ptr, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return S5_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return S5_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return S5_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_num_sms[dev] = n;
    }
    *ptr = g_scratch_ptr[dev];
    *num_sms = g_num_sms[dev];
    return S5_OK;
}

}  // namespace

extern "C" s5_status s5_forward_noalloc(const float *lambda_bar, const float *b_bar,
                                        const float *c_tilde, const float *d, const void *u,
                                        s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                                        s5_dtype proj_dtype, int B, int L, int H, int P,
                                        const float *x0, float *x_last, s5_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B < 0 || L < 0 || H < 1 || P < 1) return S5_ERR_INVALID_ARGUMENT;
    const bool dt_ok = (u_dtype == S5_F32 || u_dtype == S5_BF16) &&
                       (y_dtype == S5_F32 || y_dtype == S5_BF16) &&
                       (proj_dtype == S5_F32 || proj_dtype == S5_BF16);
    if (!dt_ok) return S5_ERR_INVALID_ARGUMENT;
    const void *params[] = {lambda_bar, b_bar, c_tilde, d};
    for (const void *p : params)
        if (!p || !aligned16(p)) return S5_ERR_INVALID_ARGUMENT;
    if ((x0 && !aligned16(x0)) || (x_last && !aligned16(x_last))) return S5_ERR_INVALID_ARGUMENT;
    const size_t need = s5_workspace_size(B, L, H, P);
    if (need == 0 || need > S5_NOALLOC_SCRATCH_BYTES) return S5_ERR_INVALID_ARGUMENT;
    if ((long long)B * L == 0) {
        if (!x_last || B == 0) return S5_OK;
        const size_t bytes = sizeof(float) * 2 * (size_t)B * P;
        cudaError_t e = x0 ? cudaMemcpyAsync(x_last, x0, bytes, cudaMemcpyDeviceToDevice, st)
                           : cudaMemsetAsync(x_last, 0, bytes, st);
        return e == cudaSuccess ? S5_OK : S5_ERR_CUDA;
    }
    if (!u || !y || !aligned16(u) || !aligned16(y)) return S5_ERR_INVALID_ARGUMENT;

    const int T = s5::simt_tile_tokens(H, P, false);
    if (T == 0) return S5_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    int sms = 0;
    s5_status s = device_scratch(&scratch, &sms);
    if (s != S5_OK) return s;

    const long long nchunks = (L + T - 1) / T;
    const long long ntiles = nchunks * B;
    // The array keeps the previous call's contents: the header (counters,
    // epoch, status) and the carry flags must start at zero, so they are
    // cleared on the caller's stream before the launch.
    const size_t clear = 256 + s5::align256(sizeof(unsigned int) * (size_t)ntiles);
    if (cudaMemsetAsync(scratch, 0, clear, st) != cudaSuccess) return S5_ERR_CUDA;

    s5::SimtArgs a;
    a.lambda_bar = reinterpret_cast<const float2 *>(lambda_bar);
    a.w = reinterpret_cast<const float2 *>(b_bar);
    a.c_tilde = reinterpret_cast<const float2 *>(c_tilde);
    a.d = d;
    a.u = u;
    a.y = y;
    a.x0 = reinterpret_cast<const float2 *>(x0);
    a.x_last = reinterpret_cast<float2 *>(x_last);
    a.g = nullptr;
    a.B = B;
    a.L = L;
    a.H = H;
    a.P = P;
    a.T = T;
    a.nchunks = (int)nchunks;
    a.nseg = s5::simt_nseg(P);
    a.ntiles = ntiles;
    a.ws = s5::ws_layout(scratch, ntiles, P);
    cudaError_t e = s5::launch_forward_simt(a, u_dtype == S5_BF16, y_dtype == S5_BF16, false, st,
                                            sms);
    return e == cudaSuccess ? S5_OK : S5_ERR_CUDA;
}
