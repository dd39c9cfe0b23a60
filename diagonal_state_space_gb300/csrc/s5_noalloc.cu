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

#include "s5_internal.cuh"

namespace {

// Carry scratch of the chunked scan (header, flags, per-tile aggregates and
// carries, the tensor-core path's weight images).  A __device__ array starts
// zeroed, which is all a workspace needs before its first use: every later
// launch tags what it writes with a new epoch, so nothing is cleared between
// calls.  Every GPU that loads the library holds these bytes until the
// process exits.
__device__ __align__(1024) unsigned char g_noalloc_scratch[S5_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_ptr[64] = {nullptr};   // device address of the array, per device

// The array's name in host code is a host-side stand-in, not a device
// address; the device address is looked up once per device, with that device
// current, and cached.
s5_status device_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return s5::cuda_failure(e);
    if (dev < 0 || dev >= 64) return S5_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return s5::cuda_failure(e);
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return S5_OK;
}

}  // namespace

// s5_forward on the library's own scratch: the same argument checks, the same
// choice of kernel (the tensor-core kernel for bf16 u, y and projections at
// H = P = 128, the CUDA-core kernel otherwise) and the same error reporting.
extern "C" s5_status s5_forward_noalloc(const float *lambda_bar, const float *b_bar,
                                        const float *c_tilde, const float *d, const void *u,
                                        s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                                        s5_dtype proj_dtype, int B, int L, int H, int P,
                                        const float *x0, float *x_last, s5_stream_t stream) {
    if (B < 0 || L < 0 || H < 1 || P < 1) return S5_ERR_INVALID_ARGUMENT;
    const size_t need = s5_workspace_size(B, L, H, P);
    if (need == 0 || need > S5_NOALLOC_SCRATCH_BYTES) return S5_ERR_INVALID_ARGUMENT;
    void *scratch = nullptr;
    const s5_status s = device_scratch(&scratch);
    if (s != S5_OK) return s;
    return s5_forward(lambda_bar, b_bar, c_tilde, d, u, u_dtype, y, y_dtype, proj_dtype, B, L, H, P,
                      x0, x_last, scratch, S5_NOALLOC_SCRATCH_BYTES, stream);
}
